"""Oracle for the MLA latent-cache decode step (fp64, CPU).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library never imports, links or calls it, and this package imports
nothing from the product package: the two share only the seeded inputs made by
``mla_inputs``.

``mla_oracle.c`` is the plain definition of absorbed-form attention over the
shared 576-wide latent (see its header for the passages it follows);
``mla_oracle_fp8.c`` the same over an FP8 (E4M3) cache, with the format's
encode and decode written from its definition;
``nonabsorbed.py`` is an independent numpy restatement of the *non-absorbed*
128-head attention, used to pin it.  Every function here takes numpy arrays of
raw bfloat16 bit patterns (``uint16``) for q / cache rows and returns fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

ROW = 576     # 512 kv_c + 64 k_rope
VDIM = 512    # kv_lora_rank, the value width

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_SRC_FP8 = os.path.join(_HERE, "mla_oracle_fp8.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmla_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable C11 + OpenMP, no ISA flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    srcs = [_SRC, _SRC_FP8]
    if force or not os.path.exists(_LIB_PATH) or any(
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(f) for f in srcs):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp] + srcs + ["-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_decode_range.argtypes = [P, P, i64, i32, P, i32, P, P, i32, i32, f64, P, P]
        lib.oracle_decode_range.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [P, P, i64, i32, P, i32, P, i32, i32, f64, P, P]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_probs.argtypes = [P, P, i64, i32, P, i32, P, i32, i32, i32, f64, P]
        lib.oracle_probs.restype = ctypes.c_int
        lib.oracle_append.argtypes = [P, P, i64, P, i64, i32]
        lib.oracle_append.restype = ctypes.c_int
        lib.oracle_combine.argtypes = [P, P, P, i32, i32, P, P]
        lib.oracle_combine.restype = None
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = f64
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quantize_rows.argtypes = [P, i64, ctypes.c_float, P]
        lib.oracle_quantize_rows.restype = None
        lib.oracle_append_fp8.argtypes = [P, P, i64, ctypes.c_float, P, i64]
        lib.oracle_append_fp8.restype = ctypes.c_int
        lib.oracle_decode_fp8.argtypes = [P, P, f64, i64, i32, P, i32, P, i32, i32, f64, P, P]
        lib.oracle_decode_fp8.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def decode(q, cache, block_table, seq_lens, softmax_scale):
    """Absorbed-form decode over tokens [0, seq_lens[b]) of every request.

    q: uint16 [B, H, 576]; cache: uint16 [NB, BS, 576]; block_table: int32
    [B, max_blocks]; seq_lens: int32 [B].  Returns (out fp64 [B, H, 512],
    lse fp64 [B, H]).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    return decode_range(q, cache, block_table, np.zeros_like(seq_lens), seq_lens, softmax_scale)


def decode_range(q, cache, block_table, t_begin, t_end, softmax_scale):
    """Attention of every (request, head) over tokens [t_begin[b], t_end[b])."""
    lib = _load()
    q, qp = _c(q, np.uint16)
    cache, cp = _c(cache, np.uint16)
    bt, btp = _c(block_table, np.int32)
    tb, tbp = _c(t_begin, np.int32)
    te, tep = _c(t_end, np.int32)
    B, H, row = q.shape
    assert row == ROW and cache.shape[2] == ROW and bt.shape[0] == B
    NB, BS = cache.shape[0], cache.shape[1]
    out = np.zeros((B, H, VDIM), np.float64)
    lse = np.zeros((B, H), np.float64)
    rc = lib.oracle_decode_range(qp, cp, NB, BS, btp, bt.shape[1], tbp, tep, B, H,
                                 float(softmax_scale), out.ctypes.data_as(ctypes.c_void_p),
                                 lse.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"oracle_decode_range: bad input (code {rc})")
    return out, lse


def probs(q, cache, block_table, seq_lens, b, h, softmax_scale):
    """Softmax weights p_t (fp64 [seq_lens[b]]) of request b, head h."""
    lib = _load()
    q, qp = _c(q, np.uint16)
    cache, cp = _c(cache, np.uint16)
    bt, btp = _c(block_table, np.int32)
    sl, slp = _c(seq_lens, np.int32)
    p = np.zeros(int(sl[b]), np.float64)
    rc = lib.oracle_probs(qp, cp, cache.shape[0], cache.shape[1], btp, bt.shape[1], slp,
                          q.shape[1], int(b), int(h), float(softmax_scale),
                          p.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("oracle_probs: bad block table")
    return p


def append(kv_new, slot_mapping, cache):
    """Copy rows of kv_new (uint16 [T, 576]) into cache (uint16 [NB, BS, 576], in place)."""
    lib = _load()
    kv, kvp = _c(kv_new, np.uint16)
    sm, smp = _c(slot_mapping, np.int64)
    assert cache.dtype == np.uint16 and cache.flags.c_contiguous
    rc = lib.oracle_append(kvp, smp, kv.shape[0], cache.ctypes.data_as(ctypes.c_void_p),
                           cache.shape[0], cache.shape[1])
    if rc != 0:
        raise ValueError("oracle_append: slot out of range")
    return cache


def combine(o_partial, lse_partial, split_offsets):
    """Merge split partials (fp64 [W, H, 512], [W, H]) by request offsets [B+1]."""
    lib = _load()
    o, op = _c(o_partial, np.float64)
    l, lp = _c(lse_partial, np.float64)
    so, sop = _c(split_offsets, np.int32)
    B = so.shape[0] - 1
    H = o.shape[1]
    out = np.zeros((B, H, VDIM), np.float64)
    lse = np.zeros((B, H), np.float64)
    lib.oracle_combine(op, lp, sop, B, H, out.ctypes.data_as(ctypes.c_void_p),
                       lse.ctypes.data_as(ctypes.c_void_p))
    return out, lse


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to fp64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def absorb_q(q_nope, q_pe, w_uk) -> np.ndarray:
    """The absorbed query in fp64: q[b,h,0:512] = sum_i q_nope[b,h,i] W_UK[h,i,:],
    q[b,h,512:576] = q_pe[b,h,:].  Each head's non-rotary query is projected
    into the latent space, the rotary dims are shared as they are
    [dp-attention-expert-parallel-mla-kv-replication (inferenceinterviews.com),
    "A strong answer"; MLA 的 TP 切分 (10100.com), section 一].

    q_nope [B,H,128], q_pe [B,H,64], w_uk [H,128,512]: bfloat16 bit patterns.
    Returns [B,H,576] fp64."""
    qn = bf16_bits_to_f64(q_nope)
    w = bf16_bits_to_f64(w_uk)
    lat = np.einsum("bhi,hik->bhk", qn, w)
    return np.concatenate([lat, bf16_bits_to_f64(q_pe)], axis=2)


def absorb_out(out, w_uv) -> np.ndarray:
    """The head's value output in fp64: o[b,h,:] = sum_k out[b,h,k] W_UV[h,k,:]
    (same passages as absorb_q).  out [B,H,512]: fp64 values, or bfloat16 bit
    patterns (uint16); w_uv [H,512,128]: bfloat16 bit patterns.  Returns
    [B,H,128] fp64."""
    out = np.asarray(out)
    o = bf16_bits_to_f64(out) if out.dtype == np.uint16 else out.astype(np.float64)
    return np.einsum("bhk,hkj->bhj", o, bf16_bits_to_f64(w_uv))


# ----------------------------------------------------------------------------- FP8 cache

def e4m3_value(codes) -> np.ndarray:
    """fp64 value of E4M3 codes (uint8 array), from the format's definition."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_value(int(x)) for x in c.ravel()],
                    np.float64).reshape(c.shape)


def e4m3_encode(values) -> np.ndarray:
    """E4M3 codes of fp32 values: nearest, ties to the even code, saturating
    to +-448, NaN -> 0x7F."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    return np.array([lib.oracle_e4m3_encode(float(x)) for x in v.ravel()],
                    np.uint8).reshape(v.shape)


def quantize_rows(bf16_bits, kv_scale=1.0) -> np.ndarray:
    """FP8 codes of bf16 values: encode(fp32(x) * fp32(1 / kv_scale))."""
    lib = _load()
    x, xp = _c(bf16_bits, np.uint16)
    out = np.zeros(x.shape, np.uint8)
    lib.oracle_quantize_rows(xp, x.size, float(kv_scale), out.ctypes.data_as(ctypes.c_void_p))
    return out


def append_fp8(kv_new, slot_mapping, cache8, kv_scale=1.0):
    """Quantise rows of kv_new (uint16 bf16 bits [T, 576]) into the FP8 cache
    (uint8 [NB, BS, 576], in place)."""
    lib = _load()
    kv, kvp = _c(kv_new, np.uint16)
    sm, smp = _c(slot_mapping, np.int64)
    assert cache8.dtype == np.uint8 and cache8.flags.c_contiguous
    rc = lib.oracle_append_fp8(kvp, smp, kv.shape[0], float(kv_scale),
                               cache8.ctypes.data_as(ctypes.c_void_p),
                               cache8.shape[0] * cache8.shape[1])
    if rc != 0:
        raise ValueError("oracle_append_fp8: slot out of range")
    return cache8


def decode_fp8(q, cache8, block_table, seq_lens, softmax_scale, kv_scale=1.0):
    """Absorbed-form decode over an FP8 cache: row elements value(code) * kv_scale.

    q: uint16 bf16 bits [B, H, 576]; cache8: uint8 [NB, BS, 576]; block_table
    int32 [B, max_blocks]; seq_lens int32 [B].  Returns (out fp64 [B, H, 512],
    lse fp64 [B, H])."""
    lib = _load()
    q, qp = _c(q, np.uint16)
    cache8, cp = _c(cache8, np.uint8)
    bt, btp = _c(block_table, np.int32)
    sl, slp = _c(seq_lens, np.int32)
    B, H, row = q.shape
    assert row == ROW and cache8.shape[2] == ROW and bt.shape[0] == B
    out = np.zeros((B, H, VDIM), np.float64)
    lse = np.zeros((B, H), np.float64)
    rc = lib.oracle_decode_fp8(qp, cp, float(kv_scale), cache8.shape[0], cache8.shape[1], btp,
                               bt.shape[1], slp, B, H, float(softmax_scale),
                               out.ctypes.data_as(ctypes.c_void_p),
                               lse.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"oracle_decode_fp8: bad block table (code {rc})")
    return out, lse
