"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test is chosen so that a plausible slip in the oracle (a dropped rope term,
a wrong value range, a transposed operand, a paging index swap, a sign or scale
error, a wrong merge weight) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from oracle import nonabsorbed

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _layer(seq_lens, block_size=16, heads=8, q_kind="normal", seed=0, pool=1.5):
    w = mi.custom_workload(seq_lens, block_size=block_size, append=False, pool_factor=pool)
    d = mi.make_host_layer(w, np.random.default_rng(seed), q_kind=q_kind, num_heads=heads)
    return w, d


# ----------------------------------------------------------------- the non-absorbed form

@pytest.mark.parametrize("heads,lens", [(16, [1, 5, 33]), (128, [3, 2])])
def test_matches_nonabsorbed_mha(heads, lens):
    """W_UV[h] @ oracle(absorbed q) equals explicit-K/V multi-head attention.

    W_UK has entries in {-1,0,1} and q_nope in {-1,0,1}/8, so the absorbed query
    q_lat = W_UK[h]^T q_nope is exact in bfloat16 and both sides see the same
    numbers; the remaining difference is fp64 rounding.
    """
    rng = np.random.default_rng(7)
    dn, dv, BS = 128, 128, 16
    w = mi.custom_workload(lens, block_size=BS, append=False, pool_factor=2.0)
    NB = w.num_blocks()
    bt = mi.make_block_table(rng, lens, BS, NB)
    cache = mi.f32_to_bf16_bits(rng.standard_normal((NB, BS, 576), dtype=np.float32))
    mi.poison_unused(cache, bt, lens, BS)
    B = len(lens)
    w_uk = rng.choice([-1.0, 0.0, 1.0], p=[0.02, 0.96, 0.02], size=(heads, dn, 512))
    w_uv = rng.standard_normal((heads, dv, 512))
    q_nope = rng.choice([-1.0, 0.0, 1.0], size=(B, heads, dn)) / 8.0
    q_pe_bits = mi.f32_to_bf16_bits(rng.standard_normal((B, heads, 64), dtype=np.float32))
    q_pe = oracle.bf16_bits_to_f64(q_pe_bits)
    q_lat = np.einsum("hik,bhi->bhk", w_uk, q_nope)
    q_lat_bits = mi.f32_to_bf16_bits(q_lat.astype(np.float32))
    assert np.array_equal(oracle.bf16_bits_to_f64(q_lat_bits), q_lat), "absorbed q not exact"
    q_bits = np.concatenate([q_lat_bits, q_pe_bits], axis=2)
    scale = 1.0 / math.sqrt(192.0)
    out, lse = oracle.decode(q_bits, cache, bt, np.array(lens, np.int32), scale)
    for b, L in enumerate(lens):
        rows = oracle.bf16_bits_to_f64(mi.gather_rows(cache, bt, b, L, BS))
        ref = nonabsorbed.mha_nonabsorbed(q_nope[b], q_pe[b], w_uk, w_uv, rows, scale)
        got = np.einsum("hik,hk->hi", w_uv, out[b])
        err = np.abs(got - ref).max() / np.abs(ref).max()
        assert err < 1e-10, (b, err)


@pytest.mark.parametrize("heads", [8, 128])
def test_absorption_chain_matches_nonabsorbed_mha(heads):
    """absorb_out(decode(absorb_q(q_nope, q_pe, W_UK)), W_UV) equals explicit-K/V
    multi-head attention with keys [W_UK[h]^T c ; k_rope] and values
    W_UV[h]^T c.  W_UK and q_nope are chosen so that the absorbed query is
    exact in bfloat16 (entries in {-1,0,1} and {-1,0,1}/8); W_UV is any
    bfloat16 array.  A transposed weight, a dropped rope copy or a wrong
    contraction index in either absorption fails this by orders of magnitude."""
    rng = np.random.default_rng(17)
    lens, BS = [4, 29], 16
    w = mi.custom_workload(lens, block_size=BS, append=False, pool_factor=2.0)
    NB = w.num_blocks()
    bt = mi.make_block_table(rng, lens, BS, NB)
    cache = mi.f32_to_bf16_bits(rng.standard_normal((NB, BS, 576), dtype=np.float32))
    mi.poison_unused(cache, bt, lens, BS)
    B = len(lens)
    w_uk_f = rng.choice([-1.0, 0.0, 1.0], p=[0.02, 0.96, 0.02], size=(heads, 128, 512))
    q_nope_f = rng.choice([-1.0, 0.0, 1.0], size=(B, heads, 128)) / 8.0
    w_uk = mi.f32_to_bf16_bits(w_uk_f.astype(np.float32))
    q_nope = mi.f32_to_bf16_bits(q_nope_f.astype(np.float32))
    q_pe = mi.f32_to_bf16_bits(rng.standard_normal((B, heads, 64), dtype=np.float32))
    w_uv = mi.f32_to_bf16_bits(rng.standard_normal((heads, 512, 128), dtype=np.float32))
    q = oracle.absorb_q(q_nope, q_pe, w_uk)
    q_bits = mi.f32_to_bf16_bits(q.astype(np.float32))
    assert np.array_equal(oracle.bf16_bits_to_f64(q_bits), q), "absorbed q not exact in bf16"
    scale = 1.0 / math.sqrt(192.0)
    out, _ = oracle.decode(q_bits, cache, bt, np.array(lens, np.int32), scale)
    o = oracle.absorb_out(out, w_uv)
    for b, L in enumerate(lens):
        rows = oracle.bf16_bits_to_f64(mi.gather_rows(cache, bt, b, L, BS))
        ref = nonabsorbed.mha_nonabsorbed(q_nope_f[b], oracle.bf16_bits_to_f64(q_pe[b]), w_uk_f,
                                          oracle.bf16_bits_to_f64(w_uv).transpose(0, 2, 1),
                                          rows, scale)
        err = np.abs(o[b] - ref).max() / np.abs(ref).max()
        assert err < 1e-10, (b, err)


def test_matches_textbook_attention_per_head():
    """Each (b, h) equals softmax(scale K q) V with K = rows, V = rows[:, :512]."""
    w, d = _layer([1, 9, 40], heads=4, q_kind="sharp", seed=3)
    out, lse = oracle.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], mi.SOFTMAX_SCALE)
    for b, L in enumerate(w.seq_lens):
        rows = oracle.bf16_bits_to_f64(mi.gather_rows(d["cache"], d["block_table"], b, L, 16))
        for h in range(4):
            q = oracle.bf16_bits_to_f64(d["q"][b, h])
            ref = nonabsorbed.softmax_attention(q, rows, rows[:, :512], mi.SOFTMAX_SCALE)
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------- closed forms

def test_two_token_closed_form_golden():
    with open(os.path.join(GOLDEN, "two_token_closed_form.json")) as f:
        g = json.load(f)
    q = np.zeros((1, 1, 576), np.float32)
    for k, v in g["q"].items():
        q[0, 0, int(k)] = v
    cache = np.zeros((1, 2, 576), np.float32)
    for t, r in enumerate(g["rows"]):
        for k, v in r.items():
            cache[0, t, int(k)] = v
    out, lse = oracle.decode(mi.f32_to_bf16_bits(q), mi.f32_to_bf16_bits(cache),
                             np.array([[0]], np.int32), np.array([2], np.int32),
                             g["softmax_scale"])
    expect = np.zeros(512)
    for k, v in g["expected_out"].items():
        expect[int(k)] = v
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-14, atol=1e-15)
    assert abs(lse[0, 0] - g["expected_lse"]) < 1e-14


def test_one_token_context_returns_kv_c_exactly():
    w, d = _layer([1, 1, 1], heads=8, q_kind="sharp")
    out, lse = oracle.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], mi.SOFTMAX_SCALE)
    for b in range(3):
        row = oracle.bf16_bits_to_f64(mi.gather_rows(d["cache"], d["block_table"], b, 1, 16))[0]
        for h in range(8):
            assert np.array_equal(out[b, h], row[:512])
            q = oracle.bf16_bits_to_f64(d["q"][b, h])
            assert abs(lse[b, h] - mi.SOFTMAX_SCALE * float(q @ row)) < 1e-12


def test_zero_query_gives_mean_of_kv_c():
    w, d = _layer([1, 7, 50], heads=2)
    q = np.zeros_like(d["q"])
    out, lse = oracle.decode(q, d["cache"], d["block_table"], d["seq_lens"], mi.SOFTMAX_SCALE)
    for b, L in enumerate(w.seq_lens):
        rows = oracle.bf16_bits_to_f64(mi.gather_rows(d["cache"], d["block_table"], b, L, 16))
        mean = rows[:, :512].sum(axis=0) / L
        np.testing.assert_allclose(out[b, 0], mean, rtol=1e-12, atol=1e-14)
        assert abs(lse[b, 0] - math.log(L)) < 1e-12


def test_dominant_logit_selects_its_row():
    """q = 64 * c_k makes token k's score exceed every other by hundreds."""
    w, d = _layer([30], heads=1)
    rows = mi.gather_rows(d["cache"], d["block_table"], 0, 30, 16)
    k = 11
    qf = mi.bf16_bits_to_f32(rows[k]) * 64.0
    q = mi.f32_to_bf16_bits(qf)[None, None]
    out, _ = oracle.decode(q, d["cache"], d["block_table"], d["seq_lens"], 1.0)
    np.testing.assert_allclose(out[0, 0], oracle.bf16_bits_to_f64(rows[k])[:512], rtol=0, atol=1e-12)


def test_rope_dims_enter_scores_but_not_values():
    """Changing only dims 512..575 of a row moves the scores, never out of span(kv_c)."""
    w, d = _layer([2], heads=1, q_kind="sharp", seed=5)
    out0, lse0 = oracle.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], 1.0)
    cache2 = d["cache"].copy()
    blk = d["block_table"][0, 0]
    cache2[blk, 1, 512:] = mi.f32_to_bf16_bits(np.full(64, 3.0, np.float32))
    out1, lse1 = oracle.decode(d["q"], cache2, d["block_table"], d["seq_lens"], 1.0)
    assert lse1[0, 0] != lse0[0, 0]
    rows = oracle.bf16_bits_to_f64(mi.gather_rows(cache2, d["block_table"], 0, 2, 16))
    # out must be a convex combination of the two kv_c rows with the new weights
    p = oracle.probs(d["q"], cache2, d["block_table"], d["seq_lens"], 0, 0, 1.0)
    np.testing.assert_allclose(out1[0, 0], p @ rows[:, :512], rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------- invariants

def test_softmax_rows_sum_to_one():
    w, d = _layer([1, 17, 64, 200], heads=4, q_kind="sharp")
    for b in range(4):
        for h in range(4):
            p = oracle.probs(d["q"], d["cache"], d["block_table"], d["seq_lens"], b, h,
                             mi.SOFTMAX_SCALE)
            assert abs(p.sum() - 1.0) < 1e-12 and (p >= 0).all()


def test_invariant_to_physical_block_order():
    w, d = _layer([5, 33, 64], heads=4, seed=11)
    out0, lse0 = oracle.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], 0.1)
    rng = np.random.default_rng(99)
    NB = d["cache"].shape[0]
    perm = rng.permutation(NB)            # new physical index of old block i is perm[i]
    cache2 = np.empty_like(d["cache"])
    cache2[perm] = d["cache"]
    bt2 = np.where(d["block_table"] >= 0, perm[np.maximum(d["block_table"], 0)], -1).astype(np.int32)
    out1, lse1 = oracle.decode(d["q"], cache2, bt2, d["seq_lens"], 0.1)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_page_size_does_not_change_result():
    """The same logical rows stored with pages of 16 and of 64 give identical results."""
    lens = [7, 70, 130]
    w, d = _layer(lens, block_size=16, heads=3, seed=2)
    w64 = mi.custom_workload(lens, block_size=64, append=False, pool_factor=1.0)
    NB64 = w64.num_blocks()
    bt64 = mi.make_block_table(np.random.default_rng(4), lens, 64, NB64)
    cache64 = np.full((NB64, 64, 576), mi.BF16_NAN, np.uint16)
    for b, L in enumerate(lens):
        rows = mi.gather_rows(d["cache"], d["block_table"], b, L, 16)
        for t in range(L):
            cache64[bt64[b, t // 64], t % 64] = rows[t]
    o16, l16 = oracle.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], 0.07)
    o64, l64 = oracle.decode(d["q"], cache64, bt64, d["seq_lens"], 0.07)
    assert np.array_equal(o16, o64) and np.array_equal(l16, l64)


def test_query_scale_tradeoff():
    """(2q, scale/2) gives the same scores exactly, so the same result."""
    w, d = _layer([9, 21], heads=3, q_kind="sharp")
    q2 = mi.f32_to_bf16_bits(mi.bf16_bits_to_f32(d["q"]) * 2.0)
    o1, l1 = oracle.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], 0.3)
    o2, l2 = oracle.decode(q2, d["cache"], d["block_table"], d["seq_lens"], 0.15)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_poisoned_rows_are_never_read():
    """NaN in every unowned row (pool holes and tails) leaves the result finite."""
    w, d = _layer([3, 16, 17, 31], heads=2, pool=3.0)
    assert np.isnan(mi.bf16_bits_to_f32(d["cache"])).any()
    out, lse = oracle.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], 0.1)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_empty_range_and_bad_table():
    w, d = _layer([4], heads=1)
    out, lse = oracle.decode_range(d["q"], d["cache"], d["block_table"], [2], [2], 0.1)
    assert (out == 0).all() and lse[0, 0] == -np.inf
    bad = d["block_table"].copy()
    bad[0, 0] = d["cache"].shape[0]
    with pytest.raises(ValueError):
        oracle.decode(d["q"], d["cache"], bad, d["seq_lens"], 0.1)


# ----------------------------------------------------------------- combine

@pytest.mark.parametrize("nsplit", [1, 2, 5])
def test_combine_of_split_ranges_equals_whole(nsplit):
    lens = [1, 40, 200]
    w, d = _layer(lens, heads=4, q_kind="sharp", seed=21)
    full_o, full_l = oracle.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], 0.08)
    parts_o, parts_l, offs = [], [], [0]
    for b, L in enumerate(lens):
        cuts = np.linspace(0, L, nsplit + 1).round().astype(int)
        for s in range(nsplit):
            tb = np.zeros(len(lens), np.int32)
            te = np.zeros(len(lens), np.int32)
            tb[b], te[b] = cuts[s], cuts[s + 1]
            o, l = oracle.decode_range(d["q"], d["cache"], d["block_table"], tb, te, 0.08)
            parts_o.append(o[b])
            parts_l.append(l[b])
        offs.append(offs[-1] + nsplit)
    co, cl = oracle.combine(np.stack(parts_o), np.stack(parts_l), np.array(offs, np.int32))
    np.testing.assert_allclose(co, full_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(cl, full_l, rtol=1e-13, atol=1e-13)


def test_combine_weights_by_lse():
    """Two partials with lse 0 and ln 3 mix 1:3 (hand-derived)."""
    o = np.zeros((2, 1, 512))
    o[0, 0, :] = 1.0
    o[1, 0, :] = -1.0
    out, lse = oracle.combine(o, np.array([[0.0], [math.log(3.0)]]), np.array([0, 2], np.int32))
    np.testing.assert_allclose(out[0, 0], np.full(512, -0.5), rtol=1e-15)
    assert abs(lse[0, 0] - math.log(4.0)) < 1e-15


# ----------------------------------------------------------------- append and layout facts

def test_append_copies_rows_bit_exact_and_skips_minus_one():
    w = mi.workload(1)
    d = mi.make_host_layer(w, mi.rng_for(1))
    cache = d["cache"].copy()
    slots = d["slot_mapping"].copy()
    slots[2] = -1
    before = cache.copy()
    oracle.append(d["kv_new"], slots, cache)
    bs = w.block_size
    for b in range(4):
        blk, row = divmod(int(d["slot_mapping"][b]), bs)
        if b == 2:
            assert np.array_equal(cache[blk, row], before[blk, row])
        else:
            assert np.array_equal(cache[blk, row], d["kv_new"][b])
    changed = (cache != before).any(axis=2).sum()
    assert changed == 3
    with pytest.raises(ValueError):
        oracle.append(d["kv_new"][:1], np.array([cache.shape[0] * bs], np.int64), cache)


def test_page_facts_pin_layout_constants():
    with open(os.path.join(GOLDEN, "page_facts.json")) as f:
        g = json.load(f)
    row = g["latent_row_dims"]
    assert oracle.ROW == row["value"] == row["kv_c"] + row["k_rope"] == mi.ROW
    assert oracle.VDIM == row["kv_c"]
    per_tok = g["bf16_bytes_per_token_61_layers"]
    assert per_tok["layers"] * oracle.ROW * per_tok["bytes_per_elem"] == per_tok["value"]
    # the rank's share of the node batch reads ~5.7 GB per step (and TP=8 reads 8x that)
    dp = g["dp_attention_cache_read_per_gpu_gb"]
    share = dp["seqs_per_node"] / dp["gpus"] * dp["context"] * per_tok["value"] / 1e9
    assert round(share, 1) == dp["value"]
    assert abs(share / 4.8 - dp["ms_at_4p8_tbs"]) < 0.05
    tp = g["tp8_cache_read_per_gpu_gb"]
    assert round(tp["seqs"] * tp["context"] * per_tok["value"] / 1e9, 1) == tp["value"]
    # the 61-layer, 20 x 4096 workload reads exactly 20 * 4096 * 70272 bytes of cache per step
    w3 = mi.workload(3)
    assert w3.cache_bytes_per_layer_read() * w3.layers == 20 * 4096 * per_tok["value"]
    assert g["fp8_bytes_per_token_per_layer"]["value"] == oracle.ROW
    r = g["rope_is_shared_not_per_head"]
    assert r["num_heads"] * r["rope_dim"] == r["per_head_rope_total_if_not_shared"]
    assert oracle.ROW - oracle.VDIM == r["rope_dim"]


def test_inputs_module_recipe():
    """Config 1 recipe: page 16, pool with spare blocks, NaN in unowned rows and the append slot."""
    w = mi.workload(1)
    assert w.extra["pre_append_lens"] == [1, 17, 64, 200] and w.seq_lens == [2, 18, 65, 201]
    d = mi.make_host_layer(w, mi.rng_for(1))
    assert d["cache"].shape[1] == 16 and d["cache"].shape[0] > w.blocks_needed()
    blk, row = np.divmod(d["slot_mapping"], 16)
    assert (d["cache"][blk, row] == mi.BF16_NAN).all()
    bits = mi.f32_to_bf16_bits(np.array([1.0, 1.00390625, 1.01171875, -2.5], np.float32))
    assert list(bits) == [0x3F80, 0x3F80, 0x3F82, 0xC020]  # ties round to even
