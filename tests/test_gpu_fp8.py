"""GPU parity of the FP8 (E4M3) latent cache path against the FP8 oracle.

The FP8 cache holds one byte per latent element, 576 bytes per token per
layer [MLA 的 TP 切分 (10100.com), opening paragraph and section 5.1]; the
format, scale and rounding readings are stated in oracle/mla_oracle_fp8.c.
The oracle reads the bytes exactly (fp64), so the only error of the GPU path
is its own arithmetic, the same as for the bf16 cache: the bar is the bf16
path's (rel-L2 <= 5e-3, max-abs <= 1e-2 max|ref|, lse within 2e-3), and the
quantising append is bit-exact.
"""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from gpu_helpers import assert_close, assert_lse_close, dev, dev_bf16, host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mla():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import mla_latent_cache_decode_gb300 as m
    return m


def _dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def _host_u8(t):
    return t.detach().contiguous().cpu().numpy()


def _decode_fp8_layer(mla, d, *, append, planned, kv_scale):
    cache8 = _dev_u8(d["cache8"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B = d["q"].shape[0]
    out = torch.full((B, 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, 128), float("nan"), dtype=torch.float32, device="cuda")
    q, bt, sl = dev_bf16(d["q"]), dev(d["block_table"], torch.int32), dev(d["seq_lens"], torch.int32)
    ws = mla.make_workspace(B)
    if planned:
        mla.mla_decode_plan(sl, bt, d["cache8"].shape[1], ws, dev_status=status,
                            num_blocks=d["cache8"].shape[0])
        mla.mla_decode_fp8_planned(q, cache8, bt, sl, d["softmax_scale"], out, lse,
                                   kv_scale=kv_scale, workspace=ws, dev_status=status,
                                   kv_new=dev_bf16(d["kv_new"]) if append else None)
    else:
        if append:
            mla.mla_cache_append_fp8(dev_bf16(d["kv_new"]), dev(d["slot_mapping"], torch.int64),
                                     cache8, kv_scale=kv_scale, dev_status=status)
        mla.mla_decode_fp8(q, cache8, bt, sl, d["softmax_scale"], out, lse, kv_scale=kv_scale,
                           workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    return cache8, out, lse, int(status.item())


def _oracle_fp8_layer(d, *, append, kv_scale):
    cache8 = d["cache8"].copy()
    if append:
        oracle.append_fp8(d["kv_new"], d["slot_mapping"], cache8, kv_scale)
    out, lse = oracle.decode_fp8(d["q"], cache8, d["block_table"], d["seq_lens"],
                                 d["softmax_scale"], kv_scale)
    return cache8, out, lse


# ----------------------------------------------------------------------------- append

@pytest.mark.parametrize("kv_scale", [1.0, 0.37, 4.0])
def test_fp8_append_bit_exact(mla, kv_scale):
    rng = np.random.default_rng(71)
    T = 300
    x = rng.standard_normal((T, 576)).astype(np.float32)
    x[0, :64] *= 1e-4                      # subnormal codes and underflow to zero
    x[1, :64] *= 1e3                       # saturation at +-448 * kv_scale
    x[2, :8] = [0.0, -0.0, 448.0, -448.0, 464.0, 2.0 ** -10, -2.0 ** -10, 1.0625]
    kv = mi.f32_to_bf16_bits(x)
    NB, BS = 40, 16
    cache0 = np.full((NB, BS, 576), 0x5A, np.uint8)
    slots = rng.permutation(NB * BS)[:T].astype(np.int64)
    slots[7] = -1
    ref = cache0.copy()
    oracle.append_fp8(kv, slots, ref, kv_scale)
    cache8 = _dev_u8(cache0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append_fp8(dev_bf16(kv), dev(slots, torch.int64), cache8, kv_scale=kv_scale,
                             dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(_host_u8(cache8), ref)


def test_fp8_append_flags_out_of_range_slot(mla):
    kv = dev_bf16(mi.f32_to_bf16_bits(np.ones((2, 576), np.float32)))
    cache8 = torch.zeros((4, 16, 576), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append_fp8(kv, torch.tensor([3, 64], dtype=torch.int64, device="cuda"), cache8,
                             dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5                        # MLA_ERR_DEVICE_RANGE
    c = _host_u8(cache8).reshape(-1, 576)
    assert np.all(c[3] == 0x38) and np.all(np.delete(c, 3, axis=0) == 0)


# ----------------------------------------------------------------------------- decode

def test_fp8_one_token_returns_every_code_exactly(mla):
    """A 1-token context gives p = 1, so out = value(code) * kv_scale exactly.
    Request 0's row holds code c at dim c and at dim 511 - c, so every finite
    code is dequantised in both byte positions of a pair; request 1 reads the
    row reversed.  (NaN codes mark rows that are never read: one in a live row
    would make every score of that token NaN.)"""
    NB, BS = 4, 16
    row = np.concatenate([np.arange(256), np.arange(255, -1, -1), np.arange(64)]).astype(np.uint8)
    row[(row & 0x7F) == 0x7F] = 0x38
    cache8 = np.full((NB, BS, 576), 0x38, np.uint8)
    cache8[2, 0] = row
    cache8[3, 0] = row[::-1]
    q = mi.make_queries(np.random.default_rng(5), 2, kind="sharp")
    d = dict(q=q, cache8=cache8, block_table=np.array([[2], [3]], np.int32),
             seq_lens=np.array([1, 1], np.int32), softmax_scale=mi.SOFTMAX_SCALE)
    for kv_scale in (1.0, 0.5):
        _, out, _, st = _decode_fp8_layer(mla, d, append=False, planned=False, kv_scale=kv_scale)
        assert st == 0
        got = host_f64(out)
        for b, r in enumerate((row, row[::-1])):
            want = oracle.e4m3_value(r[:512]) * kv_scale
            assert np.array_equal(got[b], np.broadcast_to(want, got[b].shape)), (b, kv_scale)


@pytest.mark.parametrize("q_kind", ["normal", "sharp"])
@pytest.mark.parametrize("planned", [False, True])
@pytest.mark.parametrize("kv_scale", [1.0, 0.37])
def test_fp8_config1_after_append(mla, q_kind, planned, kv_scale):
    w = mi.workload(1)
    d = mi.make_host_layer_fp8(w, mi.rng_for(1, 0, 5), q_kind=q_kind)
    cache_g, out, lse, st = _decode_fp8_layer(mla, d, append=True, planned=planned,
                                              kv_scale=kv_scale)
    assert st == 0
    cache_r, ref, ref_lse = _oracle_fp8_layer(d, append=True, kv_scale=kv_scale)
    assert np.array_equal(_host_u8(cache_g), cache_r), "appended FP8 rows"
    assert_close(host_f64(out), ref, f"fp8 config1 {q_kind}")
    assert_lse_close(lse.cpu().numpy(), ref_lse, "fp8 config1 lse")


@pytest.mark.parametrize("block_size", [16, 32, 64, 128, 256])
def test_fp8_block_sizes_ragged(mla, block_size):
    lens = [1, 63, 64, 65, 200, 513, 1000]
    w = mi.custom_workload(lens, block_size=block_size, append=True, pool_factor=1.3)
    d = mi.make_host_layer_fp8(w, np.random.default_rng(block_size), q_kind="sharp")
    _, out, lse, st = _decode_fp8_layer(mla, d, append=True, planned=True, kv_scale=1.0)
    assert st == 0
    _, ref, ref_lse = _oracle_fp8_layer(d, append=True, kv_scale=1.0)
    assert_close(host_f64(out), ref, f"fp8 block {block_size}")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_fp8_repeat_bit_identical(mla):
    w = mi.custom_workload([4096, 17, 1500, 64], block_size=64, append=False, pool_factor=1.2)
    d = mi.make_host_layer_fp8(w, np.random.default_rng(3), q_kind="sharp")
    runs = [_decode_fp8_layer(mla, d, append=False, planned=False, kv_scale=0.5)[1]
            for _ in range(5)]
    for r in runs[1:]:
        assert torch.equal(r.view(torch.int16), runs[0].view(torch.int16))


def _device_fp8(w, layer, q_kind="normal", block_table=None):
    dl = mi.make_device_layer_fp8(w, layer, "cuda", q_kind=q_kind, block_table=block_table)
    host = dict(q=mi.to_bits(dl["q"]), cache8=_host_u8(dl["cache8"]),
                block_table=dl["block_table_host"], seq_lens=dl["seq_lens"].cpu().numpy(),
                kv_new=mi.to_bits(dl["kv_new"]), slot_mapping=dl["slot_mapping"].cpu().numpy(),
                softmax_scale=dl["softmax_scale"])
    return dl, host


def _oracle_fp8_sample(host, reqs, kv_scale):
    cache8 = host["cache8"].copy()
    oracle.append_fp8(host["kv_new"], host["slot_mapping"], cache8, kv_scale)
    return oracle.decode_fp8(host["q"][reqs], cache8, host["block_table"][reqs],
                             host["seq_lens"][reqs], host["softmax_scale"], kv_scale)


@pytest.mark.parametrize("cfg,reqs", [(2, [0, 31, 63]), (4, [0, 3, 7]), (5, [0, 100, 255])])
def test_fp8_full_size_configs_sampled(mla, cfg, reqs):
    w = mi.workload(cfg)
    kv_scale = 0.75
    dl, host = _device_fp8(w, 0, q_kind="sharp" if cfg != 5 else "normal")
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((w.batch, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.batch, 128), dtype=torch.float32, device="cuda")
    mla.mla_decode_plan(dl["seq_lens"], dl["block_table"], w.block_size, ws, dev_status=status,
                        num_blocks=w.num_blocks())
    mla.mla_decode_fp8_planned(dl["q"], dl["cache8"], dl["block_table"], dl["seq_lens"],
                               dl["softmax_scale"], out, lse, kv_scale=kv_scale, workspace=ws,
                               dev_status=status, kv_new=dl["kv_new"])
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse = _oracle_fp8_sample(host, reqs, kv_scale)
    assert_close(host_f64(out)[reqs], ref, f"fp8 config {cfg}")
    assert_lse_close(lse.cpu().numpy()[reqs], ref_lse)


def test_fp8_config3_dp_rank_layers_sampled(mla):
    """The DP-rank workload with an FP8 cache as the benchmark runs it: one
    plan, then per layer the fused quantising append and the decode; three
    layers (each with its own cache) checked on sampled requests, and the
    appended rows byte-exact."""
    w = mi.workload(3)
    bt = mi.make_block_table(mi.rng_for(3, 0, 1), w.seq_lens, w.block_size, w.num_blocks())
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    reqs = [0, 9, 19]
    for layer in range(3):
        dl, host = _device_fp8(w, layer, block_table=bt)
        if layer == 0:
            mla.mla_decode_plan(dl["seq_lens"], dl["block_table"], w.block_size, ws,
                                dev_status=status, num_blocks=w.num_blocks())
        out = torch.empty((w.batch, 128, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.batch, 128), dtype=torch.float32, device="cuda")
        mla.mla_decode_fp8_planned(dl["q"], dl["cache8"], dl["block_table"], dl["seq_lens"],
                                   dl["softmax_scale"], out, lse, kv_scale=1.0, workspace=ws,
                                   dev_status=status, kv_new=dl["kv_new"])
        torch.cuda.synchronize()
        ref, ref_lse = _oracle_fp8_sample(host, reqs, 1.0)
        assert_close(host_f64(out)[reqs], ref, f"fp8 config3 layer {layer}")
        assert_lse_close(lse.cpu().numpy()[reqs], ref_lse)
        rows = _host_u8(dl["cache8"]).reshape(-1, 576)[host["slot_mapping"]]
        assert np.array_equal(rows, oracle.quantize_rows(host["kv_new"], 1.0))
    assert int(status.item()) == 0


@pytest.mark.parametrize("lens", [[700, 64, 1500, 33, 4096, 129],
                                  [700, 64, 1500, 33, 4096, 129, 2000, 517, 3000, 90] * 4])
def test_fp8_graph_step_equals_eager(mla, lens):
    """A two-layer FP8 step captured in a CUDA graph (plan, then per layer the
    fused quantising append, the decode and its combine, which is launched as
    a programmatic dependent of the decode) gives the same bits as the same
    calls run eagerly, replay after replay, and matches the oracle on sampled
    requests."""
    w = mi.custom_workload(lens, block_size=64, layers=2, append=True, pool_factor=1.5,
                           name="fp8_graph_check")
    bt = mi.make_block_table(mi.rng_for(w.config_id, 0, 1), w.seq_lens, w.block_size,
                             w.num_blocks())
    kv_scale = 0.75
    layers = []
    for layer in range(w.layers):
        dl, host = _device_fp8(w, layer, q_kind="sharp", block_table=bt)
        layers.append((dl, host, dl["cache8"].clone()))
    B = w.batch
    ws = mla.make_workspace(B)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.empty((B, 128, 512), dtype=torch.bfloat16, device="cuda") for _ in layers]
    lses = [torch.empty((B, 128), dtype=torch.float32, device="cuda") for _ in layers]
    side = torch.cuda.Stream()
    sh = side.cuda_stream

    def step():
        d0 = layers[0][0]
        mla.mla_decode_plan(d0["seq_lens"], d0["block_table"], w.block_size, ws,
                            dev_status=status, stream=sh, num_blocks=w.num_blocks())
        for (dl, _, _), out, lse in zip(layers, outs, lses):
            mla.mla_decode_fp8_planned(dl["q"], dl["cache8"], dl["block_table"], dl["seq_lens"],
                                       dl["softmax_scale"], out, lse, kv_scale=kv_scale,
                                       workspace=ws, dev_status=status, kv_new=dl["kv_new"],
                                       stream=sh)

    def reset_caches():
        for dl, _, pristine in layers:
            dl["cache8"].copy_(pristine)

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
        reset_caches()
        for o in outs:
            o.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for (eo, el), o, l in zip(eager, outs, lses):
            assert torch.equal(o.view(torch.int16), eo.view(torch.int16)), f"replay {rep}"
            assert torch.equal(l, el), f"replay {rep} lse"
    reqs = [0, 2, 4]
    for (dl, host, _), o, l in zip(layers, outs, lses):
        ref, ref_lse = _oracle_fp8_sample(host, reqs, kv_scale)
        assert_close(host_f64(o)[reqs], ref, "fp8 graph step")
        assert_lse_close(l.cpu().numpy()[reqs], ref_lse)


def test_fp8_host_validation(mla):
    q = torch.zeros((1, 128, 576), dtype=torch.bfloat16, device="cuda")
    cache8 = torch.zeros((4, 16, 576), dtype=torch.uint8, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, 128, 512), dtype=torch.bfloat16, device="cuda")
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(mla.MlaError):
            mla.mla_decode_fp8(q, cache8, bt, sl, 0.1, out, kv_scale=bad)
    q16 = torch.zeros((1, 16, 576), dtype=torch.bfloat16, device="cuda")
    out16 = torch.empty((1, 16, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mla.MlaError):
        mla.mla_decode_fp8(q16, cache8, bt, sl, 0.1, out16)
