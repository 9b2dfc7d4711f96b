"""GPU parity of the few-head kernel (1 to 32 heads: a tensor-parallel rank's
share of the 128 heads) against the fp64 oracle, through the C ABI.

Same bar as the 128-head path: rel-L2 <= 5e-3 and max-abs <= 1e-2 * max|ref|
for the bf16 output, lse within 2e-3.  Every host layer poisons the rows no
request owns (and page tails) with NaN, so a read past a sequence end shows
up as a non-finite output.
"""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from gpu_helpers import assert_close, assert_lse_close, dev, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mla():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import mla_latent_cache_decode_gb300 as m
    return m


def run_few(mla, d, heads, planned=False, ws=None):
    """Decode one host layer (no append) with `heads` heads; torch results."""
    cache = dev_bf16(d["cache"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B = d["q"].shape[0]
    out = torch.full((B, heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, heads), float("nan"), dtype=torch.float32, device="cuda")
    q = dev_bf16(d["q"])
    bt = dev(d["block_table"], torch.int32)
    sl = dev(d["seq_lens"], torch.int32)
    if ws is None:
        ws = mla.make_workspace(B, heads)
    if planned:
        mla.mla_decode_plan(sl, bt, d["cache"].shape[1], ws, num_heads=heads, dev_status=status)
        mla.mla_decode_planned(q, cache, bt, sl, d["softmax_scale"], out, lse, workspace=ws,
                               dev_status=status)
    else:
        mla.mla_decode(q, cache, bt, sl, d["softmax_scale"], out, lse, workspace=ws,
                       dev_status=status)
    torch.cuda.synchronize()
    return out, lse, int(status.item())


def oracle_few(d):
    return oracle.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], d["softmax_scale"])


def host_layer(lens, block_size, heads, seed, q_kind="sharp", pool_factor=1.3):
    w = mi.custom_workload(lens, block_size=block_size, append=False, pool_factor=pool_factor)
    return mi.make_host_layer(w, np.random.default_rng(seed), q_kind=q_kind, num_heads=heads)


@pytest.mark.parametrize("heads", [1, 2, 8, 15, 16, 17, 24, 31, 32])
@pytest.mark.parametrize("planned", [False, True])
def test_every_head_count_against_oracle(mla, heads, planned):
    """Both padded widths (16 and 32) and head counts that fill them partly:
    the pad heads read other requests' q rows (or zeros past the end of q)
    and must change nothing."""
    d = host_layer([1, 17, 64, 65, 200, 1500, 4100], 64, heads, 100 + heads)
    out, lse, st = run_few(mla, d, heads, planned)
    assert st == 0
    ref, ref_lse = oracle_few(d)
    assert_close(host_f64(out), ref, f"{heads} heads")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("block_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("heads", [16, 32])
def test_block_sizes_ragged(mla, block_size, heads):
    """Pages shorter than a tile (one box per page and chunk) and longer (one
    box per tile), with tails of every residue mod 16."""
    lens = [1, 31, 32, 33, 63, 64, 65, 127, 129, 255, 257, 600, 1023, 1500]
    d = host_layer(lens, block_size, heads, block_size + heads)
    out, lse, st = run_few(mla, d, heads)
    assert st == 0
    ref, ref_lse = oracle_few(d)
    assert_close(host_f64(out), ref, f"BS={block_size} heads={heads}")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_zero_length_requests_and_empty_batch(mla):
    d = host_layer([5, 5, 5, 130, 5], 16, 16, 7, pool_factor=2)
    d["seq_lens"] = np.array([0, 5, 0, 130, 0], np.int32)
    out, lse, st = run_few(mla, d, 16)
    assert st == 0
    ref, ref_lse = oracle_few(d)
    o = host_f64(out)
    for b in (0, 2, 4):
        assert (o[b] == 0).all() and torch.isinf(lse[b]).all()
    assert_close(o[[1, 3]], ref[[1, 3]])
    assert_lse_close(lse.cpu().numpy(), ref_lse)
    d["seq_lens"] = np.zeros(5, np.int32)
    out, lse, st = run_few(mla, d, 16)
    assert st == 0 and (host_f64(out) == 0).all() and torch.isinf(lse).all()


@pytest.mark.parametrize("heads", [16, 32])
def test_one_token_contexts_bit_exact(mla, heads):
    """One token: its probability is exactly 1, so every head's output is the
    token's kv_c row, bit for bit."""
    d = host_layer([1] * 37, 16, heads, 8, pool_factor=3.0)
    out, lse, st = run_few(mla, d, heads)
    assert st == 0
    got = host_bits(out)
    for b in range(37):
        row = mi.gather_rows(d["cache"], d["block_table"], b, 1, 16)[0]
        assert np.array_equal(got[b], np.broadcast_to(row[:512], got[b].shape))


@pytest.mark.parametrize("heads", [16, 32])
def test_long_request_split_over_every_sm(mla, heads):
    """One request of 20,000 tokens spread over all the ranges (split partials
    and the few-head combine) beside short ones."""
    d = host_layer([20000, 3, 70, 1], 64, heads, 9, pool_factor=1.1)
    for planned in (False, True):
        out, lse, st = run_few(mla, d, heads, planned)
        assert st == 0
        ref, ref_lse = oracle_few(d)
        assert_close(host_f64(out), ref, f"long + short, {heads} heads")
        assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_many_short_requests(mla):
    """700 requests: ranges of many segments (walked past the plan's cached
    records), each loading its q into the next of two buffers."""
    rng = np.random.default_rng(13)
    lens = rng.integers(1, 40, size=700).tolist()
    d = host_layer(lens, 16, 16, 14, q_kind="normal", pool_factor=1.2)
    out, lse, st = run_few(mla, d, 16)
    assert st == 0
    ref, ref_lse = oracle_few(d)
    assert_close(host_f64(out), ref, "700 short requests")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_block_permutation_bit_exact_and_repeatable(mla):
    d = host_layer([300, 1000, 77, 2048], 32, 16, 15, pool_factor=1.7)
    out0, lse0, _ = run_few(mla, d, 16)
    out0b, lse0b, _ = run_few(mla, d, 16)
    assert torch.equal(out0.view(torch.int16), out0b.view(torch.int16)) and torch.equal(lse0, lse0b)
    NB = d["cache"].shape[0]
    perm = np.random.default_rng(10).permutation(NB)
    d2 = dict(d)
    d2["cache"] = np.empty_like(d["cache"])
    d2["cache"][perm] = d["cache"]
    d2["block_table"] = np.where(d["block_table"] >= 0, perm[np.maximum(d["block_table"], 0)],
                                 -1).astype(np.int32)
    out1, lse1, _ = run_few(mla, d2, 16)
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16)) and torch.equal(lse0, lse1)


def test_repeated_bit_identical(mla):
    """Thirty decodes of a layer whose ranges hold long runs of tiles and
    several segments: every output finite and equal bit for bit to the first
    (a race between the roles shows up as a repeat that differs)."""
    rng = np.random.default_rng(16)
    lens = rng.integers(200, 6000, size=48).tolist()
    d = host_layer(lens, 64, 16, 17)
    first = None
    for rep in range(30):
        out, lse, st = run_few(mla, d, 16)
        assert st == 0
        assert bool(torch.isfinite(out.float()).all()), f"run {rep}: non-finite output"
        if first is None:
            first = (out, lse)
            ref, ref_lse = oracle_few(d)
            assert_close(host_f64(out), ref, "48 requests")
            assert_lse_close(lse.cpu().numpy(), ref_lse)
        else:
            assert torch.equal(out.view(torch.int16), first[0].view(torch.int16)), f"run {rep}"
            assert torch.equal(lse, first[1]), f"run {rep} lse"


def test_partial_then_combine_equals_planned(mla):
    d = host_layer([9000, 3, 70, 1, 2500], 64, 16, 18)
    B, H = 5, 16
    q, cache = dev_bf16(d["q"]), dev_bf16(d["cache"])
    bt, sl = dev(d["block_table"], torch.int32), dev(d["seq_lens"], torch.int32)
    ws = mla.make_workspace(B, H)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_decode_plan(sl, bt, 64, ws, num_heads=H, dev_status=status)
    outs = []
    for split_calls in (False, True):
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
        args = (q, cache, bt, sl, d["softmax_scale"], out, lse)
        if split_calls:
            mla.mla_decode_partial(*args, workspace=ws, dev_status=status)
            mla.mla_combine_planned(ws, B, out, lse, num_heads=H)
        else:
            mla.mla_decode_planned(*args, workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append((out, lse))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])


def test_bad_block_id_is_flagged_not_faulted(mla):
    d = host_layer([40, 40], 16, 16, 19, pool_factor=1.0)
    d["block_table"] = d["block_table"].copy()
    d["block_table"][1, 1] = 10_000_000
    out, lse, st = run_few(mla, d, 16)
    assert st == 5
    ref, _ = oracle.decode(d["q"][:1], d["cache"], d["block_table"][:1], d["seq_lens"][:1],
                           d["softmax_scale"])
    assert_close(host_f64(out)[:1], ref, "request without the bad entry")


def test_fused_append_needs_all_heads(mla):
    d = host_layer([40, 40], 16, 16, 20, pool_factor=1.5)
    B = 2
    out = torch.empty((B, 16, 512), dtype=torch.bfloat16, device="cuda")
    kv_new = torch.zeros((B, 576), dtype=torch.bfloat16, device="cuda")
    ws = mla.make_workspace(B, 16)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_append_planned(dev_bf16(d["q"]), dev_bf16(d["cache"]), kv_new,
                                      dev(d["block_table"], torch.int32),
                                      dev(d["seq_lens"], torch.int32), d["softmax_scale"], out,
                                      workspace=ws)
    assert e.value.status == 2  # MLA_ERR_UNSUPPORTED


def test_graph_captured_layers_equal_eager(mla):
    """Plan + three layers captured in a CUDA graph on a side stream give the
    eager bits, replay after replay."""
    lens = [700, 64, 1500, 33, 4096, 129]
    w = mi.custom_workload(lens, block_size=64, layers=3, append=False, pool_factor=1.5)
    bt = mi.make_block_table(mi.rng_for(0, 0, 21), lens, 64, w.num_blocks())
    layers = [mi.make_device_layer(w, l, "cuda", q_kind="sharp", num_heads=16, block_table=bt)
              for l in range(3)]
    B, H = len(lens), 16
    ws = mla.make_workspace(B, H)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda") for _ in layers]
    lses = [torch.empty((B, H), dtype=torch.float32, device="cuda") for _ in layers]
    side = torch.cuda.Stream()
    sh = side.cuda_stream

    def step():
        d0 = layers[0]
        mla.mla_decode_plan(d0["seq_lens"], d0["block_table"], 64, ws, num_heads=H,
                            dev_status=status, stream=sh, num_blocks=w.num_blocks())
        for dl, out, lse in zip(layers, outs, lses):
            mla.mla_decode_planned(dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"],
                                   dl["softmax_scale"], out, lse, workspace=ws,
                                   dev_status=status, stream=sh)

    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    eager = [(o.clone(), l.clone()) for o, l in zip(outs, lses)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    for rep in range(3):
        for o in outs:
            o.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for (eo, el), o, l in zip(eager, outs, lses):
            assert torch.equal(o.view(torch.int16), eo.view(torch.int16)), f"replay {rep}"
            assert torch.equal(l, el), f"replay {rep} lse"
    for dl, o, l in zip(layers, outs, lses):
        ref, ref_lse = oracle.decode(mi.to_bits(dl["q"]), mi.to_bits(dl["cache"]), bt,
                                     np.array(lens, np.int32), dl["softmax_scale"])
        assert_close(host_f64(o), ref, "graph layer")
        assert_lse_close(l.cpu().numpy(), ref_lse)


def test_tp_rank_full_size_sampled(mla):
    """The node batch under TP = 8 attention, as the benchmark times it: 159
    requests x 4096 tokens, 16 heads, pages of 64, in the benchmark's launch
    configuration; sampled requests against the oracle (their rows gathered
    on the device, so the oracle reads only those)."""
    lens = [4096] * 159
    w = mi.custom_workload(lens, block_size=64, append=False, pool_factor=1.0)
    dl = mi.make_device_layer(w, 0, "cuda", q_kind="normal", num_heads=16)
    B, H = 159, 16
    ws = mla.make_workspace(B, H)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    mla.mla_decode(dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"], dl["softmax_scale"],
                   out, lse, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    reqs = [0, 79, 158]
    nblk = 4096 // 64
    bt_host = dl["block_table_host"]
    rows = torch.stack([dl["cache"][torch.as_tensor(bt_host[b, :nblk], device="cuda").long()]
                        for b in reqs])                    # [3, 64 pages, 64, 576]
    cache_s = mi.to_bits(rows.reshape(len(reqs) * nblk, 64, 576))
    bt_s = np.arange(len(reqs) * nblk, dtype=np.int32).reshape(len(reqs), nblk)
    ref, ref_lse = oracle.decode(mi.to_bits(dl["q"])[reqs], cache_s, bt_s,
                                 np.full(len(reqs), 4096, np.int32), dl["softmax_scale"])
    assert_close(host_f64(out)[reqs], ref, "TP rank sampled")
    assert_lse_close(lse.cpu().numpy()[reqs], ref_lse)
