"""KV-load-aware placement of requests on data-parallel attention ranks (host
only, no GPU): the oracle pinned to list-scheduling facts, the library's
mla_place_requests / mla_place_one equal to the oracle, and simulated ranks
over gloo."""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
from oracle import placement as op  # noqa: E402

# DP-attention rank capacity on 8 x H200 in the pages' arithmetic: 35.9 GB of
# KV per GPU at 70,272 B per token [dp-attention-expert-parallel-mla-kv-
# replication (inferenceinterviews.com), "A strong answer"]
H200_DP_RANK_TOKENS = 35_900_000_000 // 70_272


def _mla():
    import mla_latent_cache_decode_gb300 as mla
    try:
        mla.get_lib()
    except ImportError as e:
        pytest.skip(f"libmla not built: {e}")
    return mla


# ------------------------------------------------------------------ oracle pins

def _graham_tight(m):
    """2m+1 jobs: two each of 2m-1 .. m+1, three of m.  Decreasing-order list
    scheduling ends at 4m-1; the optimum is 3m (Graham 1969)."""
    jobs = []
    for v in range(2 * m - 1, m, -1):
        jobs += [v, v]
    return jobs + [m, m, m]


@pytest.mark.parametrize("m", [2, 3])
def test_oracle_graham_tight_instance_against_exhaustive_optimum(m):
    jobs = _graham_tight(m)
    _, load = op.place(jobs, m)
    assert max(load) == 4 * m - 1
    assert op.optimal_max_load(jobs, m) == 3 * m


@pytest.mark.parametrize("m", [4, 5, 8])
def test_oracle_graham_tight_instance_larger(m):
    _, load = op.place(_graham_tight(m), m)
    assert max(load) == 4 * m - 1 and sum(load) == sum(_graham_tight(m))


def test_oracle_within_graham_bound_of_the_optimum():
    rng = np.random.default_rng(7)
    for _ in range(60):
        m = int(rng.integers(2, 4))
        jobs = [int(x) for x in rng.integers(1, 50, size=int(rng.integers(1, 8)))]
        _, load = op.place(jobs, m)
        opt = op.optimal_max_load(jobs, m)
        assert opt <= max(load) <= (4 / 3 - 1 / (3 * m)) * opt + 1e-9, (jobs, m)


def test_oracle_closed_forms():
    # fewer requests than ranks: each alone, the longest on rank 0
    rank_of, load = op.place([5, 9, 1], 4)
    assert rank_of == [1, 0, 2] and load == [9, 5, 1, 0]
    # equal lengths: counts differ by at most one, the extra on the low ranks
    rank_of, load = op.place([7] * 11, 4)
    assert load == [21, 21, 21, 14]
    assert [rank_of.count(r) for r in range(4)] == [3, 3, 3, 2]
    # nothing to place
    assert op.place([], 3) == ([], [0, 0, 0])


def test_oracle_capacity():
    rank_of, load = op.place([10, 6, 6, 3], 2, capacity_tokens=9)
    assert rank_of == [-1, 0, 1, 0] and load == [9, 6]
    assert max(load) <= 9
    assert op.place_one([4, 2, 2], 3) == 1
    assert op.place_one([4, 2, 2], 3, capacity_tokens=4) == -1
    assert op.place_one([0], 5) == 0


# ------------------------------------------------------------------ library = oracle

def _cases():
    rng = np.random.default_rng(20261202)
    yield "node batch 159 x 4096 on 8 ranks", [4096] * 159, 8, 0
    yield "6 long users + 100 short on 8 ranks", [131072] * 6 + [int(x) for x in rng.integers(512, 8193, 100)], 8, 0
    yield "256 x U[512, 8192] on 8 ranks", [int(x) for x in rng.integers(512, 8193, 256)], 8, 0
    yield "long contexts at the H200 DP-rank capacity", [int(x) for x in rng.integers(50_000, 400_000, 24)], 8, H200_DP_RANK_TOKENS
    yield "many ties", [int(x) for x in rng.integers(1, 4, 1000)], 7, 0
    yield "zero-length requests", [0, 3, 0, 3], 2, 0
    yield "one rank", [5, 1, 7], 1, 0
    yield "empty", [], 3, 0


@pytest.mark.parametrize("name,tokens,ranks,cap", list(_cases()), ids=[c[0] for c in _cases()])
def test_library_equals_oracle(name, tokens, ranks, cap):
    mla = _mla()
    rank_of, load = mla.place_requests(tokens, ranks, cap)
    ref_of, ref_load = op.place(tokens, ranks, cap)
    assert rank_of.tolist() == ref_of
    assert load.tolist() == ref_load
    placed = [t for t, r in zip(tokens, ref_of) if r >= 0]
    assert sum(load) == sum(placed)
    if cap:
        assert max(load) <= cap


def test_library_place_one_equals_oracle():
    mla = _mla()
    rng = np.random.default_rng(3)
    for _ in range(200):
        ranks = int(rng.integers(1, 9))
        loads = [int(x) for x in rng.integers(0, 20, ranks)]
        t = int(rng.integers(0, 30))
        cap = int(rng.choice([0, 25, 40]))
        assert mla.place_one(loads, t, cap) == op.place_one(loads, t, cap)


def test_library_rejects_bad_arguments():
    mla = _mla()
    for args in (([1, -2], 2, 0), ([1], 0, 0), ([1], 2, -1)):
        with pytest.raises(mla.MlaError):
            mla.place_requests(*args)
    with pytest.raises(mla.MlaError):
        mla.place_one([1, -1], 3)


# ------------------------------------------------------------------ simulated ranks (gloo)

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import mla_latent_cache_decode_gb300 as mla
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank sees the same arrivals and places them identically; each
        # then keeps only its own requests and reports what it holds
        tokens = [131072] * 3 + [int(x) for x in np.random.default_rng(11).integers(512, 8193, 40)]
        rank_of, load = mla.place_requests(tokens, world)
        mine = [t for t, r in zip(tokens, rank_of) if r == rank]
        held = torch.tensor([sum(mine)], dtype=torch.int64)
        all_held = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(all_held, held)
        slowest = held.clone()
        dist.all_reduce(slowest, op=dist.ReduceOp.MAX)
        q.put((rank, [int(x.item()) for x in all_held], int(slowest.item()), load.tolist(),
               sum(tokens)))
    finally:
        dist.destroy_process_group()


def test_two_simulated_ranks_agree_on_loads():
    torch = pytest.importorskip("torch")
    _mla()
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, held, slowest, load, total in res:
        assert held == load                       # what the ranks hold is the plan's loads
        assert sum(held) == total                 # every request somewhere, once
        assert slowest == max(load)               # the lockstepped step waits for this rank
    # the three long requests are not all on one rank
    assert max(res[0][3]) < 3 * 131072
