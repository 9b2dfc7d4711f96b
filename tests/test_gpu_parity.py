"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases compare every output element; the full-size workloads (in the
launch configuration the benchmark times) compare sampled requests the oracle
can compute.  Bar: rel-L2 <= 5e-3 and max-abs <= 1e-2 * max|ref| for the bf16
output, lse within 2e-3, append bit-exact.
"""
import math

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from gpu_helpers import (assert_close, assert_lse_close, dev, dev_bf16, host_bits, host_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mla():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import mla_latent_cache_decode_gb300 as m
    return m


def run_layer(mla, d, *, append=True, planned=False, heads=128):
    """Append (optional) + decode one host layer on the GPU; returns torch results."""
    cache = dev_bf16(d["cache"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if append:
        mla.mla_cache_append(dev_bf16(d["kv_new"]), dev(d["slot_mapping"], torch.int64), cache,
                             dev_status=status)
    B = d["q"].shape[0]
    out = torch.full((B, heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, heads), float("nan"), dtype=torch.float32, device="cuda")
    q = dev_bf16(d["q"])
    bt = dev(d["block_table"], torch.int32)
    sl = dev(d["seq_lens"], torch.int32)
    ws = mla.make_workspace(B)
    if planned:
        mla.mla_decode_plan(sl, bt, d["cache"].shape[1], ws, dev_status=status)
        mla.mla_decode_planned(q, cache, bt, sl, d["softmax_scale"], out, lse, workspace=ws,
                               dev_status=status)
    else:
        mla.mla_decode(q, cache, bt, sl, d["softmax_scale"], out, lse, workspace=ws,
                       dev_status=status)
    torch.cuda.synchronize()
    return cache, out, lse, int(status.item())


def oracle_layer(d, append=True):
    cache = d["cache"].copy()
    if append:
        oracle.append(d["kv_new"], d["slot_mapping"], cache)
    out, lse = oracle.decode(d["q"], cache, d["block_table"], d["seq_lens"], d["softmax_scale"])
    return cache, out, lse


# ----------------------------------------------------------------------------- append

def test_append_bit_exact(mla):
    w = mi.workload(1)
    d = mi.make_host_layer(w, mi.rng_for(1))
    cache, *_ = run_layer(mla, d)
    ref_cache, _, _ = oracle_layer(d)
    assert np.array_equal(host_bits(cache), ref_cache)


def test_append_skips_minus_one_and_flags_out_of_range(mla):
    rng = np.random.default_rng(5)
    cache_h = mi.f32_to_bf16_bits(rng.standard_normal((6, 16, 576), dtype=np.float32))
    kv = mi.f32_to_bf16_bits(rng.standard_normal((5, 576), dtype=np.float32))
    slots = np.array([3, -1, 95, 96, 40], np.int64)   # 96 = 6*16 is outside the pool
    cache = dev_bf16(cache_h)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append(dev_bf16(kv), dev(slots, torch.int64), cache, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    ref = cache_h.copy()
    ok = slots.copy()
    ok[3] = -1
    oracle.append(kv, ok, ref)
    assert np.array_equal(host_bits(cache), ref)


def test_append_many_tokens(mla):
    rng = np.random.default_rng(6)
    NB, BS, T = 300, 64, 5000
    cache_h = mi.f32_to_bf16_bits(rng.standard_normal((NB, BS, 576), dtype=np.float32))
    kv = mi.f32_to_bf16_bits(rng.standard_normal((T, 576), dtype=np.float32))
    slots = rng.permutation(NB * BS)[:T].astype(np.int64)
    cache = dev_bf16(cache_h)
    mla.mla_cache_append(dev_bf16(kv), dev(slots, torch.int64), cache)
    torch.cuda.synchronize()
    oracle.append(kv, slots, cache_h)
    assert np.array_equal(host_bits(cache), cache_h)


# ----------------------------------------------------------------------------- config 1

@pytest.mark.parametrize("q_kind", ["normal", "sharp"])
@pytest.mark.parametrize("planned", [False, True])
def test_config1_after_append(mla, q_kind, planned):
    w = mi.workload(1)
    d = mi.make_host_layer(w, mi.rng_for(1), q_kind=q_kind)
    cache, out, lse, st = run_layer(mla, d, planned=planned)
    assert st == 0
    ref_cache, ref, ref_lse = oracle_layer(d)
    assert np.array_equal(host_bits(cache), ref_cache)
    assert_close(host_f64(out), ref, f"config1 {q_kind}")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("q_kind", ["normal", "sharp"])
def test_config1_before_append_lengths_1_17_64_200(mla, q_kind):
    w = mi.workload(1)
    d = mi.make_host_layer(w, mi.rng_for(1), q_kind=q_kind)
    d["seq_lens"] = np.array(w.extra["pre_append_lens"], np.int32)
    _, out, lse, st = run_layer(mla, d, append=False)
    assert st == 0
    _, ref, ref_lse = oracle_layer(d, append=False)
    assert_close(host_f64(out), ref, f"config1 pre-append {q_kind}")
    assert_lse_close(lse.cpu().numpy(), ref_lse)
    # 1-token context: output is exactly the kv_c part of the only row
    row0 = mi.gather_rows(d["cache"], d["block_table"], 0, 1, 16)[0]
    got0 = host_bits(out)[0]
    assert np.array_equal(got0, np.broadcast_to(row0[:512], got0.shape))


# ----------------------------------------------------------------------------- invariants

def test_one_token_contexts_bit_exact(mla):
    w = mi.custom_workload([1] * 37, block_size=16, append=False, pool_factor=3.0)
    d = mi.make_host_layer(w, np.random.default_rng(8), q_kind="sharp")
    _, out, lse, st = run_layer(mla, d, append=False)
    assert st == 0
    got = host_bits(out)
    for b in range(37):
        row = mi.gather_rows(d["cache"], d["block_table"], b, 1, 16)[0]
        assert np.array_equal(got[b], np.broadcast_to(row[:512], got[b].shape))


def test_block_permutation_bit_exact_and_repeatable(mla):
    w = mi.custom_workload([300, 1000, 77, 2048], block_size=32, append=False, pool_factor=1.7)
    d = mi.make_host_layer(w, np.random.default_rng(9), q_kind="sharp")
    _, out0, lse0, _ = run_layer(mla, d, append=False)
    _, out0b, lse0b, _ = run_layer(mla, d, append=False)
    assert torch.equal(out0.view(torch.int16), out0b.view(torch.int16)) and torch.equal(lse0, lse0b)
    NB = d["cache"].shape[0]
    perm = np.random.default_rng(10).permutation(NB)
    d2 = dict(d)
    d2["cache"] = np.empty_like(d["cache"])
    d2["cache"][perm] = d["cache"]
    d2["block_table"] = np.where(d["block_table"] >= 0, perm[np.maximum(d["block_table"], 0)],
                                 -1).astype(np.int32)
    _, out1, lse1, _ = run_layer(mla, d2, append=False)
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16)) and torch.equal(lse0, lse1)


# ----------------------------------------------------------------------------- edge cases

def test_empty_batch_is_a_noop(mla):
    q = torch.empty((0, 128, 576), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((4, 16, 576), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    sl = torch.zeros((0,), dtype=torch.int32, device="cuda")
    out = torch.empty((0, 128, 512), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    mla.mla_decode(q, cache, bt, sl, 0.1, out, workspace=ws)
    torch.cuda.synchronize()


def test_zero_length_requests(mla):
    lens = [0, 5, 0, 130, 0]
    w = mi.custom_workload([max(L, 1) for L in lens], block_size=16, append=False, pool_factor=2)
    d = mi.make_host_layer(w, np.random.default_rng(11))
    d["seq_lens"] = np.array(lens, np.int32)
    _, out, lse, st = run_layer(mla, d, append=False)
    assert st == 0
    _, ref, ref_lse = oracle_layer(d, append=False)
    o = host_f64(out)
    for b in (0, 2, 4):
        assert (o[b] == 0).all()
    assert_close(o[[1, 3]], ref[[1, 3]])
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_all_empty_batch(mla):
    w = mi.custom_workload([1, 1, 1], block_size=16, append=False, pool_factor=2)
    d = mi.make_host_layer(w, np.random.default_rng(12))
    d["seq_lens"] = np.zeros(3, np.int32)
    _, out, lse, st = run_layer(mla, d, append=False)
    assert st == 0 and (host_f64(out) == 0).all() and torch.isinf(lse).all()


@pytest.mark.parametrize("block_size", [16, 32, 64, 128, 256])
def test_block_sizes_ragged(mla, block_size):
    lens = [1, 31, 32, 33, 63, 64, 65, 127, 129, 255, 257, 600, 1023, 1500]
    w = mi.custom_workload(lens, block_size=block_size, append=True, pool_factor=1.3)
    d = mi.make_host_layer(w, np.random.default_rng(block_size), q_kind="sharp")
    cache, out, lse, st = run_layer(mla, d)
    assert st == 0
    ref_cache, ref, ref_lse = oracle_layer(d)
    assert np.array_equal(host_bits(cache), ref_cache)
    assert_close(host_f64(out), ref, f"BS={block_size}")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_many_short_requests(mla):
    rng = np.random.default_rng(13)
    lens = rng.integers(1, 40, size=700).tolist()
    w = mi.custom_workload(lens, block_size=16, append=True, pool_factor=1.2)
    d = mi.make_host_layer(w, rng)
    cache, out, lse, st = run_layer(mla, d)
    assert st == 0
    _, ref, ref_lse = oracle_layer(d)
    assert_close(host_f64(out), ref, "700 short requests")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_one_long_request_among_short(mla):
    lens = [9000, 3, 70, 1]
    w = mi.custom_workload(lens, block_size=64, append=True, pool_factor=1.1)
    d = mi.make_host_layer(w, np.random.default_rng(14), q_kind="sharp")
    cache, out, lse, st = run_layer(mla, d)
    assert st == 0
    _, ref, ref_lse = oracle_layer(d)
    assert_close(host_f64(out), ref, "long + short")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_bad_block_id_is_flagged_not_faulted(mla):
    w = mi.custom_workload([40, 40], block_size=16, append=False, pool_factor=1.0)
    d = mi.make_host_layer(w, np.random.default_rng(15))
    d["block_table"] = d["block_table"].copy()
    d["block_table"][1, 1] = 10_000_000
    _, out, lse, st = run_layer(mla, d, append=False)
    assert st == 5
    _, ref, _ = oracle_layer(dict(d, q=d["q"][:1], block_table=d["block_table"][:1],
                                  seq_lens=d["seq_lens"][:1]), append=False)
    assert_close(host_f64(out)[:1], ref, "request without the bad entry")


def test_seq_len_longer_than_table_is_flagged(mla):
    w = mi.custom_workload([40], block_size=16, append=False, pool_factor=1.0)
    d = mi.make_host_layer(w, np.random.default_rng(16))
    d["seq_lens"] = np.array([10_000], np.int32)
    _, out, lse, st = run_layer(mla, d, append=False)
    assert st == 5


@pytest.mark.parametrize("budget_ms", [1, 5])
def test_bounded_wait_times_out_and_context_survives(mla, budget_ms):
    # a wait on a barrier nothing arrives at gives up after its budget and
    # reports MLA_ERR_DEVICE_TIMEOUT; the other warp's wait (the decode's own,
    # 100 ms budget) is ended by the abort flag well before its budget; the
    # kernel returns and the context stays usable
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(2, dtype=torch.int64, device="cuda")
    mla.selftest_wait_timeout(budget_ms * 1_000_000, status, elapsed)
    torch.cuda.synchronize()
    assert int(status.item()) == 6
    e0, e1 = (int(x) for x in elapsed.cpu())
    assert budget_ms * 1_000_000 <= e0 < 90_000_000, e0
    assert budget_ms * 1_000_000 <= e1 < 90_000_000, e1  # under its own 100 ms
    w = mi.workload(1)
    d = mi.make_host_layer(w, mi.rng_for(1))
    cache, out, lse, st = run_layer(mla, d)
    assert st == 0
    ref_cache, ref, ref_lse = oracle_layer(d)
    assert np.array_equal(host_bits(cache), ref_cache)
    assert_close(host_f64(out), ref, "decode after the timeout check")


def test_host_validation_errors(mla):
    q = torch.zeros((1, 128, 576), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((4, 16, 576), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    sl = torch.ones((1,), dtype=torch.int32, device="cuda")
    out = torch.empty((1, 128, 512), dtype=torch.bfloat16, device="cuda")
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode(q, cache, bt, sl, 0.1, out, workspace=small)
    assert e.value.status == 3
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode(q, cache, bt, sl, 0.1, out, max_seq_len=65)
    assert e.value.status == 1
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode(q, cache, bt, sl, float("inf"), out)
    assert e.value.status == 1
    for bad_scale in (0.0, -0.1, float("nan")):
        with pytest.raises(mla.MlaError) as e:
            mla.mla_decode(q, cache, bt, sl, bad_scale, out)
        assert e.value.status == 1


# ----------------------------------------------------------------------------- combine

def test_combine_against_oracle(mla):
    rng = np.random.default_rng(17)
    counts = [3, 1, 0, 5, 2]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    W, H = int(offs[-1]), 128
    o = rng.standard_normal((W, H, 512)).astype(np.float32)
    l = (rng.standard_normal((W, H)) * 3).astype(np.float32)
    l[4, :7] = -np.inf
    out = torch.empty((5, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((5, H), dtype=torch.float32, device="cuda")
    mla.mla_combine(dev(o, torch.float32), dev(l, torch.float32), dev(offs, torch.int32), out, lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.combine(o.astype(np.float64), l.astype(np.float64), offs)
    got = host_f64(out)
    assert (got[2] == 0).all() and torch.isinf(lse[2]).all()
    keep = [0, 1, 3, 4]
    assert_close(got[keep], ref[keep], "combine")
    assert_lse_close(lse.cpu().numpy()[keep], ref_lse[keep])


# ----------------------------------------------------------------------------- full-size workloads

def _device_layer_and_host(w, layer, q_kind="normal", block_table=None):
    dl = mi.make_device_layer(w, layer, "cuda", q_kind=q_kind, block_table=block_table)
    host = dict(q=mi.to_bits(dl["q"]), cache=mi.to_bits(dl["cache"]),
                block_table=dl["block_table_host"], seq_lens=dl["seq_lens"].cpu().numpy(),
                kv_new=mi.to_bits(dl["kv_new"]), slot_mapping=dl["slot_mapping"].cpu().numpy(),
                softmax_scale=dl["softmax_scale"])
    return dl, host


def _oracle_sample(host, reqs, heads=None):
    cache = host["cache"].copy()
    oracle.append(host["kv_new"], host["slot_mapping"], cache)
    q = host["q"][reqs]
    if heads is not None:
        q = q[:, heads]
    return oracle.decode(q, cache, host["block_table"][reqs], host["seq_lens"][reqs],
                         host["softmax_scale"])


def _gpu_layer(mla, dl, ws, status, planned):
    B = dl["q"].shape[0]
    out = torch.empty((B, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, 128), dtype=torch.float32, device="cuda")
    mla.mla_cache_append(dl["kv_new"], dl["slot_mapping"], dl["cache"], dev_status=status)
    fn = mla.mla_decode_planned if planned else mla.mla_decode
    fn(dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"], dl["softmax_scale"], out, lse,
       workspace=ws, dev_status=status)
    return out, lse


@pytest.mark.parametrize("q_kind", ["normal", "sharp"])
def test_config2_layer_b64x4096_sampled(mla, q_kind):
    w = mi.workload(2)
    dl, host = _device_layer_and_host(w, 0, q_kind)
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _gpu_layer(mla, dl, ws, status, planned=False)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    reqs = [0, 17, 40, 63]
    ref, ref_lse = _oracle_sample(host, reqs)
    assert_close(host_f64(out)[reqs], ref, f"config2 {q_kind}")
    assert_lse_close(lse.cpu().numpy()[reqs], ref_lse)


def test_config4_skewed_sampled(mla):
    w = mi.workload(4)
    dl, host = _device_layer_and_host(w, 0, "sharp")
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _gpu_layer(mla, dl, ws, status, planned=False)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    heads = [0, 37, 64, 127]
    ref, ref_lse = _oracle_sample(host, [0], heads)     # the 131072-token request
    assert_close(host_f64(out)[0, heads], ref[0], "config4 long request")
    assert_lse_close(lse.cpu().numpy()[0, heads], ref_lse[0])
    ref, ref_lse = _oracle_sample(host, [1, 7])
    assert_close(host_f64(out)[[1, 7]], ref, "config4 short requests")


@pytest.mark.parametrize("q_kind", ["normal", "sharp"])
def test_config4_every_short_request_repeated(mla, q_kind):
    """Ranges holding several segments (split and unsplit, the last of a
    range among them), run ten times: every short request against the oracle
    once, then each repeat bit-identical to the first.  A race between the
    pipeline's roles shows up as a repeat that differs, or as garbage in a
    block of heads."""
    w = mi.workload(4)
    dl, host = _device_layer_and_host(w, 0, q_kind)
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _gpu_layer(mla, dl, ws, status, planned=False)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    reqs = list(range(1, w.batch))
    ref, ref_lse = _oracle_sample(host, reqs)
    assert_close(host_f64(out)[reqs], ref, f"config4 {q_kind} short requests")
    assert_lse_close(lse.cpu().numpy()[reqs], ref_lse)
    first = out.clone()
    for rep in range(9):
        out2 = torch.empty_like(out)
        lse2 = torch.empty_like(lse)
        mla.mla_decode(dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"],
                       dl["softmax_scale"], out2, lse2, workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out2.view(torch.int16), first.view(torch.int16)), f"repeat {rep}"
        assert torch.equal(lse2, lse), f"repeat {rep} lse"


def test_config2_layer_repeated_bit_identical(mla):
    """A 64 x 4096 layer decoded thirty times: every output finite and equal
    bit for bit to the first.  Its ranges hold long runs of tiles, where the
    S MMAs two tiles on overwrite the tensor-memory buffer that P V reads P
    from; an S issued before that P V has finished shows up as a few heads of
    non-finite or changing output (P read from raw fp32 S bits)."""
    w = mi.workload(2)
    dl = mi.make_device_layer(w, 0, "cuda", q_kind="sharp")
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append(dl["kv_new"], dl["slot_mapping"], dl["cache"], dev_status=status)
    first = None
    for rep in range(30):
        out = torch.full((w.batch, 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        mla.mla_decode(dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"],
                       dl["softmax_scale"], out, None, workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert bool(torch.isfinite(out.float()).all()), f"run {rep}: non-finite output"
        if first is None:
            first = out
        else:
            assert torch.equal(out.view(torch.int16), first.view(torch.int16)), f"run {rep} differs"


@pytest.mark.parametrize("cfg", [4, 2])
def test_partial_then_combine_equals_planned(mla, cfg):
    """mla_decode_partial + mla_combine_planned is exactly mla_decode_planned:
    on config 4 (8 requests) the planned form also runs the separate combine,
    on config 2 (64 requests) it merges inside the decode kernel, with the
    same arithmetic."""
    w = mi.workload(cfg)
    dl, host = _device_layer_and_host(w, 0, "sharp")
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append(dl["kv_new"], dl["slot_mapping"], dl["cache"], dev_status=status)
    mla.mla_decode_plan(dl["seq_lens"], dl["block_table"], w.block_size, ws, dev_status=status)
    outs = []
    for split_calls in (False, True):
        out = torch.empty((w.batch, 128, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.batch, 128), dtype=torch.float32, device="cuda")
        args = (dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"], dl["softmax_scale"], out, lse)
        if split_calls:
            mla.mla_decode_partial(*args, workspace=ws, dev_status=status)
            mla.mla_combine_planned(ws, w.batch, out, lse)
        else:
            mla.mla_decode_planned(*args, workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append((out, lse))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])


def test_fused_append_config1_against_oracle(mla):
    """mla_decode_append_planned: the cache after it equals the oracle's append
    with the decode step's slot mapping, and the outputs match the oracle."""
    w = mi.workload(1)
    for q_kind in ("normal", "sharp"):
        d = mi.make_host_layer(w, mi.rng_for(1), q_kind=q_kind)
        cache = dev_bf16(d["cache"])
        q, kv = dev_bf16(d["q"]), dev_bf16(d["kv_new"])
        bt, sl = dev(d["block_table"], torch.int32), dev(d["seq_lens"], torch.int32)
        B = d["q"].shape[0]
        out = torch.full((B, 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, 128), float("nan"), dtype=torch.float32, device="cuda")
        ws = mla.make_workspace(B)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        mla.mla_decode_plan(sl, bt, w.block_size, ws, dev_status=status)
        mla.mla_decode_append_planned(q, cache, kv, bt, sl, d["softmax_scale"], out, lse,
                                      workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref_cache, ref, ref_lse = oracle_layer(d)
        assert np.array_equal(host_bits(cache), ref_cache)
        assert_close(host_f64(out), ref, f"fused append config1 {q_kind}")
        assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("workload_id", [4, 5])
def test_fused_append_equals_separate_append(mla, workload_id):
    """The fused path gives the same bits as mla_cache_append + mla_decode_planned
    (split and unsplit requests, one and several segments per range)."""
    w = mi.workload(workload_id)
    res = []
    for fused in (False, True):
        dl = mi.make_device_layer(w, 0, "cuda", q_kind="sharp")
        ws = mla.make_workspace(w.batch)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        mla.mla_decode_plan(dl["seq_lens"], dl["block_table"], w.block_size, ws, dev_status=status)
        out = torch.empty((w.batch, 128, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.batch, 128), dtype=torch.float32, device="cuda")
        args = (dl["q"], dl["cache"])
        if fused:
            mla.mla_decode_append_planned(dl["q"], dl["cache"], dl["kv_new"], dl["block_table"],
                                          dl["seq_lens"], dl["softmax_scale"], out, lse,
                                          workspace=ws, dev_status=status)
        else:
            mla.mla_cache_append(dl["kv_new"], dl["slot_mapping"], dl["cache"], dev_status=status)
            mla.mla_decode_planned(dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"],
                                   dl["softmax_scale"], out, lse, workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        res.append((out, lse, dl["cache"].view(torch.int16).clone()))
        del dl, args
    assert torch.equal(res[0][2], res[1][2]), "caches differ"
    assert torch.equal(res[0][0].view(torch.int16), res[1][0].view(torch.int16))
    assert torch.equal(res[0][1], res[1][1])


def test_fused_append_skips_empty_requests(mla):
    lens = [0, 5, 0, 130, 1]
    w = mi.custom_workload([max(L, 1) for L in lens], block_size=16, append=True, pool_factor=2)
    d = mi.make_host_layer(w, np.random.default_rng(31))
    d["seq_lens"] = np.array(lens, np.int32)
    cache = dev_bf16(d["cache"])
    B = len(lens)
    out = torch.empty((B, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, 128), dtype=torch.float32, device="cuda")
    bt, sl = dev(d["block_table"], torch.int32), dev(d["seq_lens"], torch.int32)
    ws = mla.make_workspace(B)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_decode_plan(sl, bt, 16, ws, dev_status=status)
    mla.mla_decode_append_planned(dev_bf16(d["q"]), cache, dev_bf16(d["kv_new"]), bt, sl,
                                  d["softmax_scale"], out, lse, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    slots = np.array([mi.slot_of(d["block_table"], b, L - 1, 16) if L > 0 else -1
                      for b, L in enumerate(lens)], np.int64)
    ref_cache = d["cache"].copy()
    oracle.append(d["kv_new"], slots, ref_cache)
    assert np.array_equal(host_bits(cache), ref_cache)
    got = host_f64(out)
    ro, rl = oracle.decode(d["q"], ref_cache, d["block_table"], d["seq_lens"], d["softmax_scale"])
    assert_close(got, ro, "fused append with empty requests")
    assert_lse_close(lse.cpu().numpy(), rl)


def test_config5_mixed_fragmented_sampled(mla):
    w = mi.workload(5)
    bt = mi.make_block_table(mi.rng_for(5, 0, 1), w.seq_lens, w.block_size, w.num_blocks())
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = np.array(w.seq_lens)
    reqs = sorted({int(lens.argmin()), int(lens.argmax()), 0, 100, 255})
    for layer in range(w.layers):
        dl, host = _device_layer_and_host(w, layer, block_table=bt)
        if layer == 0:
            seq = dl["seq_lens"]
            mla.mla_decode_plan(seq, dl["block_table"], w.block_size, ws, dev_status=status,
                                num_blocks=w.num_blocks())
        out, lse = _gpu_layer(mla, dl, ws, status, planned=True)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        if layer in (0, w.layers - 1):
            ref, ref_lse = _oracle_sample(host, reqs)
            assert_close(host_f64(out)[reqs], ref, f"config5 layer {layer}")
            assert_lse_close(lse.cpu().numpy()[reqs], ref_lse)
        del dl, host


def test_config3_dp_rank_61_layers_sampled(mla):
    """The benchmark's launch configuration: one plan per step, then per layer
    the fused append + planned decode, each layer with its own cache, shared
    table; sampled requests against the oracle, and the appended rows."""
    w = mi.workload(3)
    bt = mi.make_block_table(mi.rng_for(3, 0, 1), w.seq_lens, w.block_size, w.num_blocks())
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sample_layers = {0, 29, 60}
    reqs = [0, 11, 19]
    for layer in range(w.layers):
        dl = mi.make_device_layer(w, layer, "cuda", block_table=bt)
        if layer == 0:
            mla.mla_decode_plan(dl["seq_lens"], dl["block_table"], w.block_size, ws,
                                dev_status=status, num_blocks=w.num_blocks())
        host = None
        if layer in sample_layers:
            host = dict(q=mi.to_bits(dl["q"]), cache=mi.to_bits(dl["cache"]), block_table=bt,
                        seq_lens=dl["seq_lens"].cpu().numpy(), kv_new=mi.to_bits(dl["kv_new"]),
                        slot_mapping=dl["slot_mapping"].cpu().numpy(),
                        softmax_scale=dl["softmax_scale"])
        out = torch.empty((w.batch, 128, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.batch, 128), dtype=torch.float32, device="cuda")
        mla.mla_decode_append_planned(dl["q"], dl["cache"], dl["kv_new"], dl["block_table"],
                                      dl["seq_lens"], dl["softmax_scale"], out, lse,
                                      workspace=ws, dev_status=status)
        if host is not None:
            torch.cuda.synchronize()
            ref, ref_lse = _oracle_sample(host, reqs)
            assert_close(host_f64(out)[reqs], ref, f"config3 layer {layer}")
            assert_lse_close(lse.cpu().numpy()[reqs], ref_lse)
            slots = host["slot_mapping"]
            got_rows = mi.to_bits(dl["cache"]).reshape(-1, 576)[slots]
            assert np.array_equal(got_rows, host["kv_new"]), f"config3 layer {layer} appended rows"
        del dl
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("lens", [[700, 64, 1500, 33, 4096, 129],
                                  [700, 64, 1500, 33, 4096, 129, 2000, 517, 3000, 90] * 4])
def test_graph_captured_step_equals_eager(mla, lens):
    """A step captured in a CUDA graph (plan + per-layer fused append and
    decode, on a side stream, as the benchmark runs it) gives the same bits as
    the same calls run eagerly, replay after replay; its outputs match the
    oracle on sampled requests.  With six requests the decode is launched
    normally and its combine as a programmatic dependent of it; with forty
    the decode is the programmatic dependent (of the previous layer's
    combine) and the combine is launched normally."""
    w = mi.custom_workload(lens, block_size=64, layers=2, append=True,
                           pool_factor=1.5, name="graph_check")
    bt = mi.make_block_table(mi.rng_for(w.config_id, 0, 1), w.seq_lens, w.block_size,
                             w.num_blocks())
    layers = []
    for l in range(w.layers):
        dl, host = _device_layer_and_host(w, l, q_kind="sharp", block_table=bt)
        layers.append((dl, host, dl["cache"].clone()))  # pristine cache for each run
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
            mla.mla_decode_append_planned(dl["q"], dl["cache"], dl["kv_new"], dl["block_table"],
                                          dl["seq_lens"], dl["softmax_scale"], out, lse,
                                          workspace=ws, dev_status=status, stream=sh)

    def reset_caches():
        for dl, _, pristine in layers:
            dl["cache"].copy_(pristine)

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
    reqs = np.array([0, 2, 4])
    for (dl, host, _), o, l in zip(layers, outs, lses):
        ref, ref_lse = _oracle_sample(host, reqs)
        assert_close(host_f64(o)[reqs], ref, "graph step")
        assert_lse_close(l.cpu().numpy()[reqs], ref_lse)


def _read_plan(ws, batch):
    """The plan in the workspace, parsed with the layout documented next to
    the planner (all offsets 256-byte aligned)."""
    raw = ws.cpu().numpy().view(np.uint8)
    a256 = lambda x: (x + 255) & ~255
    hdr = raw[:32].view(np.int32)
    U, P, Pm = int(hdr[0]), int(hdr[1]), int(hdr[2])
    o = a256(32)
    seq = raw[o:o + 4 * batch].view(np.int32); o = a256(o + 4 * batch)
    prefix = raw[o:o + 4 * (batch + 1)].view(np.int32); o = a256(o + 4 * (batch + 1))
    rstart = raw[o:o + 4 * (Pm + 1)].view(np.int32); o = a256(o + 4 * (Pm + 1))
    o = a256(o + 4 * (Pm + 1))            # range_first
    o = a256(o + 8 * (batch + 1))         # cost_prefix
    o = a256(o + 4 * 2 * batch)           # counters
    segc = raw[o:o + 4 * Pm].view(np.int32); o = a256(o + 4 * Pm)
    recs = raw[o:o + 32 * 4 * Pm].view(np.int32).reshape(Pm, 4, 8); o = a256(o + 32 * 4 * Pm)
    split = raw[o:o + 16 * batch].view(np.int32).reshape(batch, 4)
    return dict(U=U, P=P, Pm=Pm, seq=seq, prefix=prefix, rstart=rstart, segc=segc, recs=recs,
                split=split)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_plan_invariants(mla, cfg):
    """The planner's ranges tile the units; every range's segment records,
    every request's split record and the partial slots follow from the
    ranges; and the ranges' modelled costs (2 per unit, 7 per request start,
    a start counted in the range holding the request's first unit) are
    balanced: the targets are C/P apart and a boundary lands within a start's
    cost or a unit of its target, so no two ranges differ by more than
    2 x (7 + 2)."""
    _check_plan(mla, mi.workload(cfg))


@pytest.mark.parametrize("lens", [[4864], [3000], [4864, 64, 1], [64] * 40 + [2560],
                                  [1600, 1, 1, 1, 1, 1600, 1, 1, 1, 1, 1600]],
                         ids=["76units", "47units", "76units+2", "40x1+40units", "3x25units+8x1"])
def test_plan_invariants_crowded(mla, lens):
    """Workloads with about as many units as split ranges, where the cost
    targets leave some ranges empty and the planner's fix-up moves the
    boundaries (over several 32-boundary chunks): the same invariants."""
    _check_plan(mla, mi.custom_workload(lens, block_size=64, append=False, pool_factor=1.5))


def _check_plan(mla, w):
    dl = mi.make_device_layer(w, 0, "cuda")
    ws = mla.make_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_decode_plan(dl["seq_lens"], dl["block_table"], w.block_size, ws, dev_status=status,
                        num_blocks=dl["cache"].shape[0])
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    pl = _read_plan(ws, w.batch)
    unit = 64
    bt = dl["block_table"].cpu().numpy()
    seq = dl["seq_lens"].cpu().numpy().astype(np.int64)
    units = (seq + unit - 1) // unit
    assert np.array_equal(pl["seq"], seq)
    assert np.array_equal(pl["prefix"], np.concatenate([[0], np.cumsum(units)]))
    U, P, R = pl["U"], pl["P"], pl["rstart"].astype(np.int64)
    assert U == units.sum() and P == min(U, pl["Pm"])
    assert R[0] == 0 and R[P] == U and np.all(np.diff(R[:P + 1]) > 0) and np.all(R[P:] == U)
    starts = pl["prefix"][:-1][units > 0]
    cost = []
    for p in range(P):
        r0, r1 = R[p], R[p + 1]
        segs = []
        for b in range(w.batch):
            Ub, Ue = pl["prefix"][b], pl["prefix"][b + 1]
            u0, u1 = max(r0, Ub), min(r1, Ue)
            if u0 < u1:
                slot = (2 * p + (1 if r0 < Ub else 0)) if (Ub < r0 or Ue > r1) else -1
                segs.append((b, (u0 - Ub) * unit, min((u1 - Ub) * unit, seq[b]), slot))
        assert pl["segc"][p] == len(segs)
        for i, sgm in enumerate(segs[:4]):
            assert tuple(pl["recs"][p, i, :4]) == sgm, (p, i)
            b, t0, t1 = sgm[0], sgm[1], sgm[2]
            row0 = (int(bt[b, t0 // w.block_size]) * w.block_size + t0 % w.block_size
                    if w.block_size >= unit and t0 < t1 else -1)
            assert pl["recs"][p, i, 4] == row0, (p, i, "row0")
        cost.append(2 * (r1 - r0) + 7 * int(((starts >= r0) & (starts < r1)).sum()))
    for b in range(w.batch):
        if units[b] == 0:
            continue
        Ub, Ue = pl["prefix"][b], pl["prefix"][b + 1]
        p0 = int(np.searchsorted(R[:P], Ub, side="right") - 1)
        p1 = int(np.searchsorted(R[:P], Ue - 1, side="right") - 1)
        assert tuple(pl["split"][b, :3]) == (p0, p1, 1 if R[p0] < Ub else 0), b
    if U >= 8 * P:  # ranges of several units
        assert max(cost) - min(cost) <= 2 * (7 + 2), (min(cost), max(cost))


# ------------------------------------------------------------ absorption GEMMs

def _absorb_inputs(B, seed):
    rng = np.random.default_rng(seed)

    def bf16(shape, s=1.0):
        return mi.f32_to_bf16_bits((rng.standard_normal(shape) * s).astype(np.float32))
    return dict(q_nope=bf16((B, 128, 128)), q_pe=bf16((B, 128, 64)),
                w_uk=bf16((128, 128, 512), 128 ** -0.5), w_uv=bf16((128, 512, 128), 512 ** -0.5),
                out=bf16((B, 128, 512)))


@pytest.mark.parametrize("B", [1, 20, 64, 200])
def test_absorb_q_matches_oracle(mla, B):
    """q[b,h,:512] = q_nope[b,h] . W_UK[h] within the parity bar (fp32 sums, bf16
    out); q[b,h,512:] = q_pe[b,h] bit for bit."""
    x = _absorb_inputs(B, 100 + B)
    q = torch.empty((B, 128, 576), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_absorb_q(dev_bf16(x["q_nope"]), dev_bf16(x["q_pe"]), dev_bf16(x["w_uk"]), q,
                     dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.absorb_q(x["q_nope"], x["q_pe"], x["w_uk"])
    assert_close(host_f64(q)[:, :, :512], ref[:, :, :512], f"absorbed q B={B}")
    assert np.array_equal(host_bits(q)[:, :, 512:], x["q_pe"])


@pytest.mark.parametrize("B", [1, 20, 64, 200])
def test_absorb_out_matches_oracle(mla, B):
    """o[b,h] = out[b,h] . W_UV[h] within the parity bar."""
    x = _absorb_inputs(B, 200 + B)
    o = torch.empty((B, 128, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_absorb_out(dev_bf16(x["out"]), dev_bf16(x["w_uv"]), o, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(host_f64(o), oracle.absorb_out(x["out"], x["w_uv"]), f"absorbed out B={B}")


def test_absorbed_layer_chain_matches_oracle(mla):
    """q_nope, q_pe -> mla_absorb_q -> mla_decode -> mla_absorb_out against the
    oracle's absorb_q -> decode -> absorb_out on the same inputs."""
    lens = [1, 70, 513, 1500]
    w = mi.custom_workload(lens, block_size=64, append=False, pool_factor=1.5)
    dl = mi.make_device_layer(w, 0, "cuda")
    B = len(lens)
    x = _absorb_inputs(B, 300)
    q = torch.empty((B, 128, 576), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((B, 128, 512), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((B, 128, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_absorb_q(dev_bf16(x["q_nope"]), dev_bf16(x["q_pe"]), dev_bf16(x["w_uk"]), q,
                     dev_status=status)
    mla.mla_decode(q, dl["cache"], dl["block_table"], dl["seq_lens"], dl["softmax_scale"], out,
                   workspace=mla.make_workspace(B), dev_status=status)
    mla.mla_absorb_out(out, dev_bf16(x["w_uv"]), o, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    q_ref = oracle.absorb_q(x["q_nope"], x["q_pe"], x["w_uk"])
    q_ref_bits = mi.f32_to_bf16_bits(q_ref.astype(np.float32))
    out_ref, _ = oracle.decode(q_ref_bits, host_bits(dl["cache"]), dl["block_table_host"],
                               np.array(lens, np.int32), dl["softmax_scale"])
    assert_close(host_f64(o), oracle.absorb_out(out_ref, x["w_uv"]), "absorbed layer")


# ------------------------------------------------------------ fewer heads (a TP rank)

@pytest.mark.parametrize("heads", [1, 16, 64])
@pytest.mark.parametrize("planned", [False, True])
def test_fewer_heads_against_oracle(mla, heads, planned):
    """A tensor-parallel rank's share of the heads (16 at TP = 8) over the same
    cache: the library pads q to 128 heads in its workspace; only the caller's
    heads come back, and they match the oracle."""
    lens = [1, 17, 64, 200, 1500]
    w = mi.custom_workload(lens, block_size=64, append=False, pool_factor=1.5)
    dl = mi.make_device_layer(w, 0, "cuda", q_kind="sharp", num_heads=heads)
    B = len(lens)
    out = torch.full((B, heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, heads), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = mla.make_workspace(B, heads)
    if planned:
        mla.mla_decode_plan(dl["seq_lens"], dl["block_table"], w.block_size, ws, num_heads=heads,
                            dev_status=status)
        mla.mla_decode_planned(dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"],
                               dl["softmax_scale"], out, lse, workspace=ws, dev_status=status)
    else:
        mla.mla_decode(dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"],
                       dl["softmax_scale"], out, lse, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse = oracle.decode(host_bits(dl["q"]), host_bits(dl["cache"]), dl["block_table_host"],
                                 np.array(lens, np.int32), dl["softmax_scale"])
    assert_close(host_f64(out), ref, f"{heads} heads")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


# ------------------------------------------------------------ a plan made for other arguments

@pytest.mark.parametrize("case", ["unplanned", "other_heads", "other_batch", "other_page"])
def test_mismatched_plan_is_reported(mla, case):
    """mla_decode_planned with a workspace whose plan was made for other
    arguments (or never made) reports MLA_ERR_DEVICE_PLAN: the decode checks
    the plan's header before reading it, and the combine stays within the
    workspace.  A correctly planned call on the same workspace then gives the
    oracle's result."""
    lens = [300, 1000, 77, 2048]
    w = mi.custom_workload(lens, block_size=64, append=False, pool_factor=1.5)
    heads = 16 if case == "other_heads" else 128
    dl = mi.make_device_layer(w, 0, "cuda", q_kind="sharp", num_heads=heads)
    B = len(lens)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.full((max(mla.mla_decode_workspace_size(B, 128), mla.mla_decode_workspace_size(B, 16),
                         mla.mla_decode_workspace_size(B + 1, 128)),), 0x5A, dtype=torch.uint8,
                    device="cuda")   # never planned: a byte pattern
    if case == "other_heads":     # planned for 128 heads, decoded with 16
        mla.mla_decode_plan(dl["seq_lens"], dl["block_table"], 64, ws, num_heads=128,
                            dev_status=status)
    elif case == "other_batch":   # planned for one more request
        sl = torch.cat([dl["seq_lens"], dl["seq_lens"][:1]])
        bt = torch.cat([dl["block_table"], dl["block_table"][:1]])
        mla.mla_decode_plan(sl, bt, 64, ws, dev_status=status)
    elif case == "other_page":    # the same rows seen as pages of 32
        bt32 = torch.repeat_interleave(dl["block_table"], 2, dim=1)
        mla.mla_decode_plan(dl["seq_lens"], bt32, 32, ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out = torch.full((B, heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, heads), float("nan"), dtype=torch.float32, device="cuda")
    args = (dl["q"], dl["cache"], dl["block_table"], dl["seq_lens"], dl["softmax_scale"], out, lse)
    mla.mla_decode_planned(*args, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 7   # MLA_ERR_DEVICE_PLAN
    status.zero_()
    mla.mla_decode_plan(dl["seq_lens"], dl["block_table"], 64, ws, num_heads=heads,
                        dev_status=status)
    mla.mla_decode_planned(*args, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, ref_lse = oracle.decode(host_bits(dl["q"]), host_bits(dl["cache"]), dl["block_table_host"],
                                 np.array(lens, np.int32), dl["softmax_scale"])
    assert_close(host_f64(out), ref, case)
    assert_lse_close(lse.cpu().numpy(), ref_lse)
