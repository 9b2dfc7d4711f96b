"""The multi-rank host logic of bench.py on CPU: world_size 2 over gloo.

With data-parallel attention every rank runs an independent replica of the
rank workload (no collective on the data path); the only cross-rank steps are
the barrier and the max over ranks of the measured time, and rank 0 reports
the whole-job throughput."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        ms = 10.0 + 5.0 * rank          # rank 1 is the slower one
        slowest = bench.reduce_max(ms, w)
        gbs = bench.job_throughput_gbs(w, 1e9, slowest)
        q.put((r, w, lr, slowest, gbs))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_timing_and_whole_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r, w, lr, slowest, gbs) in enumerate(res):
        assert (r, w, lr) == (rank, 2, rank)
        assert slowest == 15.0                       # max over ranks, on every rank
        assert gbs == pytest.approx(2 * 1e9 / 15e-3 / 1e9)  # both replicas' bytes / slowest time


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.job_throughput_gbs(1, 2e9, 1000.0) == pytest.approx(2.0)


def test_e2e_chunk_bounds():
    """The e2e step's copy chunks: the input chunks start with layer 0 alone
    and grow, the output chunks mirror them and end with the last layer
    alone, both covering every layer once."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.e2e_chunk_bounds(61) == ([0, 1, 2, 4, 7, 12, 20, 32, 52, 61],
                                          [0, 9, 29, 41, 49, 54, 57, 59, 60, 61])
    for layers in range(1, 130):
        ins, outs = bench.e2e_chunk_bounds(layers)
        for b in (ins, outs):
            assert b[0] == 0 and b[-1] == layers
            assert all(x < y for x, y in zip(b, b[1:]))
        assert ins[1] == 1 and outs[-2] == layers - 1
        widths = [y - x for x, y in zip(ins, ins[1:])]
        assert all(w1 <= w2 for w1, w2 in zip(widths[:-2], widths[1:-1]))  # growing, bar the last
