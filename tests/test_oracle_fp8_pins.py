"""Pins of the FP8 (E4M3) cache oracle to facts outside itself (CPU only).

The pages fix that an FP8 latent cache holds 576 bytes per token per layer
[MLA 的 TP 切分 (10100.com), opening paragraph and section 5.1]; the format
(OCP E4M3), the per-layer scale and the rounding are readings of the pages,
stated in the oracle's header.  Each pin below would fail on a plausible
mistake: a wrong exponent bias or subnormal scale, a NaN or saturation code,
ties rounded up instead of to even, a dropped kv_scale, or a decode that does
not read the bytes as the bf16 oracle reads the same values.
"""
import math

import numpy as np
import pytest

import mla_inputs as mi
import oracle

torch = pytest.importorskip("torch")


def test_all_256_codes_against_the_format_and_a_library_routine():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_value(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2      # 0x7F and 0xFF only
    assert np.array_equal(got[~nan], lib[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(lib[~nan]))
    # special values of the format, by hand
    assert got[0x00] == 0.0 and got[0x80] == 0.0 and math.copysign(1, got[0x80]) < 0
    assert got[0x01] == 2.0 ** -9                 # smallest subnormal: 2^-6 * 1/8
    assert got[0x07] == 7 * 2.0 ** -9             # largest subnormal
    assert got[0x08] == 2.0 ** -6                 # smallest normal
    assert got[0x38] == 1.0                       # exponent field 7 = bias
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0   # largest finite: 2^8 * 1.75
    assert np.all(np.diff(got[:0x7F]) > 0)        # non-negative codes increase with value


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_value(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_ties_go_to_the_even_code_and_off_ties_to_the_nearest():
    pos = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    for c in range(0x7E):
        lo, hi = pos[c], pos[c + 1]
        mid = np.float32((lo + hi) / 2)           # at most 5 significant bits: exact in fp32
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(np.array([mid]))[0] == even, (c, lo, hi)
        assert oracle.e4m3_encode(-np.array([mid]))[0] == 0x80 | even
        eps = (hi - lo) / 16
        assert oracle.e4m3_encode(np.array([lo + eps], np.float32))[0] == c
        assert oracle.e4m3_encode(np.array([hi - eps], np.float32))[0] == c + 1


def test_saturation_nan_and_tiny_values():
    enc = lambda v: int(oracle.e4m3_encode(np.array([v], np.float32))[0])
    assert enc(448.0) == 0x7E and enc(449.0) == 0x7E and enc(1e30) == 0x7E
    assert enc(float("inf")) == 0x7E and enc(-500.0) == 0xFE and enc(-float("inf")) == 0xFE
    assert enc(float("nan")) == 0x7F
    assert enc(2.0 ** -10) == 0x00                # halfway to the smallest subnormal: even (0)
    assert enc(1.5 * 2.0 ** -10) == 0x01
    assert enc(-1e-30) == 0x80                    # sign kept on underflow


def test_encode_agrees_with_the_library_conversion_in_range():
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0)])
    x = x[np.abs(x) < 448].astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), lib)


def test_quantize_rows_applies_the_scale_in_fp32():
    rng = np.random.default_rng(9)
    # values that are exactly code * 2^k are stored exactly under kv_scale = 2^k
    codes = rng.integers(0, 0x7F, size=2000).astype(np.uint8) | (rng.integers(0, 2, 2000) << 7).astype(np.uint8)
    for k in (-3, 0, 2):
        x = (oracle.e4m3_value(codes) * 2.0 ** k).astype(np.float32)
        bits = mi.f32_to_bf16_bits(x)             # exact: at most 4 significant bits
        assert np.array_equal(mi.bf16_bits_to_f32(bits), x)
        got = oracle.quantize_rows(bits, 2.0 ** k)
        zero = oracle.e4m3_value(codes) == 0
        assert np.array_equal(got[~zero], codes[~zero])
    # a non-power-of-two scale: the nearest code to fp32(x) * fp32(1/s)
    x = rng.standard_normal(4096).astype(np.float32) * 3
    bits = mi.f32_to_bf16_bits(x)
    s = np.float32(0.37)
    got = oracle.quantize_rows(bits, float(s))
    y = mi.bf16_bits_to_f32(bits) * (np.float32(1) / s)
    back = oracle.e4m3_value(got)
    # nearest: no other finite code is closer to y
    pos = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    best = np.min(np.abs(np.abs(y.astype(np.float64))[:, None] - pos[None, :]), axis=1)
    assert np.allclose(np.abs(np.abs(y) - np.abs(back)), best, rtol=0, atol=0)


def _fp8_layer(seed, lens, block_size, heads=128, q_kind="sharp"):
    rng = np.random.default_rng(seed)
    w = mi.custom_workload(lens, block_size=block_size, append=False, pool_factor=1.25)
    bt = mi.make_block_table(rng, w.seq_lens, block_size, w.num_blocks())
    codes = rng.integers(0, 256, size=(w.num_blocks(), block_size, mi.ROW)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38          # no NaN codes in live rows
    q = mi.make_queries(rng, len(lens), num_heads=heads, kind=q_kind)
    return codes, bt, np.array(lens, np.int32), q


def test_fp8_decode_equals_the_bf16_oracle_on_the_same_values():
    codes, bt, sl, q = _fp8_layer(10, [1, 5, 64, 131], 16)
    vals = oracle.e4m3_value(codes)
    cache16 = mi.f32_to_bf16_bits(vals.astype(np.float32))   # exact: e4m3 values fit bf16
    assert np.array_equal(mi.bf16_bits_to_f32(cache16).astype(np.float64), vals)
    ref, ref_lse = oracle.decode(q, cache16, bt, sl, mi.SOFTMAX_SCALE)
    got, got_lse = oracle.decode_fp8(q, codes, bt, sl, mi.SOFTMAX_SCALE)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
    assert np.max(np.abs(got_lse - ref_lse)) <= 1e-12


def test_fp8_decode_scale_multiplies_every_row_element():
    codes, bt, sl, q = _fp8_layer(11, [3, 40, 77], 16)
    for s in (0.25, 0.37):
        vals = oracle.e4m3_value(codes) * s
        got, got_lse = oracle.decode_fp8(q, codes, bt, sl, mi.SOFTMAX_SCALE, kv_scale=s)
        # brute force in numpy over the same values
        qv = mi.bf16_bits_to_f32(q).astype(np.float64)
        for b, L in enumerate(sl):
            rows = np.stack([vals[bt[b, t // 16], t % 16] for t in range(L)])
            sc = mi.SOFTMAX_SCALE * qv[b] @ rows.T
            p = np.exp(sc - sc.max(axis=1, keepdims=True))
            ref = (p / p.sum(axis=1, keepdims=True)) @ rows[:, :512]
            lse = sc.max(axis=1) + np.log(p.sum(axis=1))
            assert np.max(np.abs(got[b] - ref)) <= 1e-12 * np.max(np.abs(ref))
            assert np.max(np.abs(got_lse[b] - lse)) <= 1e-12


def test_fp8_decode_one_token_returns_its_values():
    codes, bt, sl, q = _fp8_layer(12, [1, 1], 16)
    got, _ = oracle.decode_fp8(q, codes, bt, sl, mi.SOFTMAX_SCALE, kv_scale=0.5)
    for b in range(2):
        assert np.array_equal(got[b], np.broadcast_to(
            oracle.e4m3_value(codes[bt[b, 0], 0, :512]) * 0.5, got[b].shape))


def test_fp8_append_places_quantised_rows_and_skips():
    rng = np.random.default_rng(13)
    cache = np.full((4, 16, mi.ROW), 0x55, np.uint8)
    kv = mi.f32_to_bf16_bits(rng.standard_normal((3, mi.ROW)).astype(np.float32))
    slots = np.array([5, -1, 63], np.int64)
    before = cache.copy()
    oracle.append_fp8(kv, slots, cache, kv_scale=0.5)
    assert np.array_equal(cache[0, 5], oracle.quantize_rows(kv[0], 0.5))
    assert np.array_equal(cache[3, 15], oracle.quantize_rows(kv[2], 0.5))
    mask = np.ones(cache.shape[:2], bool)
    mask[0, 5] = mask[3, 15] = False
    assert np.array_equal(cache[mask], before[mask])
    with pytest.raises(ValueError):
        oracle.append_fp8(kv, np.array([0, 1, 64], np.int64), cache)
