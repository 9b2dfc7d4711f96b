"""Python binding of libmla (MLA latent-cache decode on GB300 / sm_103a).

Argument marshalling only: each function below checks dtypes/shapes of the
PyTorch tensors it is given, passes raw device pointers, sizes and the current
CUDA stream to the C ABI declared in include/mla.h, and raises MlaError on a
non-zero status.  Every step of the computation runs in the library's CUDA
kernels; there is no other implementation to fall back to: the first call
raises ImportError if the compiled library is missing.

Functions carry the C names: mla_cache_append, mla_decode_plan, mla_decode,
mla_decode_planned, mla_combine, mla_decode_workspace_size.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmla.so")

ROW_DIM = 576
KV_LORA_RANK = 512
ROPE_DIM = 64
NUM_HEADS = 128

STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARGUMENT", 2: "MLA_ERR_UNSUPPORTED",
          3: "MLA_ERR_WORKSPACE_TOO_SMALL", 4: "MLA_ERR_CUDA", 5: "MLA_ERR_DEVICE_RANGE",
          6: "MLA_ERR_DEVICE_TIMEOUT", 7: "MLA_ERR_DEVICE_PLAN"}
EXPORTED = ("mla_status_string", "mla_last_error_detail", "mla_abi_version", "mla_cache_append",
            "mla_decode_workspace_size", "mla_decode_plan", "mla_decode", "mla_decode_planned",
            "mla_combine", "mla_decode_noalloc", "mla_decode_partial", "mla_combine_planned",
            "mla_decode_append_planned", "mla_place_requests", "mla_place_one", "mla_absorb_q",
            "mla_absorb_out", "mla_selftest_wait_timeout", "mla_cache_append_fp8",
            "mla_decode_fp8", "mla_decode_fp8_planned")


class MlaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS.get(status, status)}: {detail}")
        self.status = status
        self.detail = detail


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmla is not built ({LIB_PATH} missing): run "
                          "`python -m mla_latent_cache_decode_gb300.build` first")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_last_error_detail.argtypes = []
    lib.mla_last_error_detail.restype = ctypes.c_char_p
    lib.mla_abi_version.argtypes = []
    lib.mla_abi_version.restype = ctypes.c_int
    lib.mla_cache_append.argtypes = [P, P, i64, P, i64, i32, P, P]
    lib.mla_cache_append.restype = ctypes.c_int
    lib.mla_decode_workspace_size.argtypes = [i32, i32]
    lib.mla_decode_workspace_size.restype = sz
    lib.mla_decode_plan.argtypes = [P, P, i32, i32, i32, i32, i64, P, sz, P, P]
    lib.mla_decode_plan.restype = ctypes.c_int
    dec = [P, P, i64, i32, P, i32, P, i32, i32, i32, f32, P, P, P, sz, P, P]
    lib.mla_decode.argtypes = dec
    lib.mla_decode.restype = ctypes.c_int
    lib.mla_decode_planned.argtypes = dec
    lib.mla_decode_planned.restype = ctypes.c_int
    lib.mla_decode_partial.argtypes = [P, P, P, i64, i32, P, i32, P, i32, i32, i32, f32, P, P, P,
                                       sz, P, P]
    lib.mla_decode_partial.restype = ctypes.c_int
    lib.mla_combine_planned.argtypes = [P, sz, i32, i32, P, P, P]
    lib.mla_combine_planned.restype = ctypes.c_int
    lib.mla_decode_append_planned.argtypes = [P, P, P, i64, i32, P, i32, P, i32, i32, i32, f32,
                                              P, P, P, sz, P, P]
    lib.mla_decode_append_planned.restype = ctypes.c_int
    lib.mla_combine.argtypes = [P, P, P, i32, i32, P, P, P]
    lib.mla_combine.restype = ctypes.c_int
    lib.mla_decode_noalloc.argtypes = [P, P, i64, i32, P, i32, P, i32, i32, i32, f32, P, P, P, P]
    lib.mla_decode_noalloc.restype = ctypes.c_int
    lib.mla_place_requests.argtypes = [P, i32, i32, i64, P, P, P]
    lib.mla_place_requests.restype = ctypes.c_int
    lib.mla_place_one.argtypes = [P, i32, i64, i64, P]
    lib.mla_place_one.restype = ctypes.c_int
    lib.mla_absorb_q.argtypes = [P, P, P, i32, i32, P, P, P]
    lib.mla_absorb_q.restype = ctypes.c_int
    lib.mla_absorb_out.argtypes = [P, P, i32, i32, P, P, P]
    lib.mla_absorb_out.restype = ctypes.c_int
    lib.mla_cache_append_fp8.argtypes = [P, P, i64, P, i64, i32, f32, P, P]
    lib.mla_cache_append_fp8.restype = ctypes.c_int
    lib.mla_decode_fp8.argtypes = [P, P, i64, i32, P, i32, P, i32, i32, i32, f32, f32, P, P, P, sz,
                                   P, P]
    lib.mla_decode_fp8.restype = ctypes.c_int
    lib.mla_decode_fp8_planned.argtypes = [P, P, P, i64, i32, P, i32, P, i32, i32, i32, f32, f32,
                                           P, P, P, sz, P, P]
    lib.mla_decode_fp8_planned.restype = ctypes.c_int
    lib.mla_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P, P, P]
    lib.mla_selftest_wait_timeout.restype = ctypes.c_int
    return lib


_lib = None


def get_lib():
    """The loaded libmla (loaded on first use; raises ImportError if not built)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def __getattr__(name):
    if name == "lib":
        return get_lib()
    raise AttributeError(name)


def _check(status: int):
    if status != 0:
        raise MlaError(status, get_lib().mla_last_error_detail().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need(t, dtype, ndim, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: need contiguous CUDA {dtype} with {ndim} dims, got "
                         f"{t.dtype} {tuple(t.shape)} on {t.device}")


def mla_decode_workspace_size(batch: int, num_heads: int = NUM_HEADS) -> int:
    return int(get_lib().mla_decode_workspace_size(batch, num_heads))


def make_workspace(batch: int, num_heads: int = NUM_HEADS, device=None):
    """A workspace tensor of the size mla_decode needs on the current device."""
    import torch
    n = mla_decode_workspace_size(batch, num_heads)
    if n == 0:
        raise MlaError(4, "cannot size the workspace (no CUDA device?)")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def mla_cache_append(kv_new, slot_mapping, cache, dev_status=None, stream=None):
    """cache[slot // BS, slot % BS, :] = kv_new[i] for every slot != -1 (bit-exact)."""
    import torch
    _need(kv_new, torch.bfloat16, 2, "kv_new")
    _need(slot_mapping, torch.int64, 1, "slot_mapping")
    _need(cache, torch.bfloat16, 3, "cache")
    if kv_new.shape[1] != ROW_DIM or cache.shape[2] != ROW_DIM:
        raise ValueError("rows must be 576 wide")
    if slot_mapping.shape[0] != kv_new.shape[0]:
        raise ValueError("slot_mapping and kv_new disagree on the token count")
    _check(get_lib().mla_cache_append(_ptr(kv_new), _ptr(slot_mapping), kv_new.shape[0], _ptr(cache),
                                cache.shape[0], cache.shape[1], _ptr(dev_status),
                                _stream(stream)))


def mla_decode_plan(seq_lens, block_table, block_size, workspace, num_heads=NUM_HEADS,
                    dev_status=None, stream=None, num_blocks=None):
    """Split-KV plan for these lengths.  With num_blocks (the cache pool's block
    count) the plan also records where every worker's first tile lies in the
    cache (the plan then depends on block_table too: re-plan when it changes)."""
    import torch
    _need(seq_lens, torch.int32, 1, "seq_lens")
    _need(block_table, torch.int32, 2, "block_table")
    table = _ptr(block_table) if num_blocks else None
    _check(get_lib().mla_decode_plan(_ptr(seq_lens), table, seq_lens.shape[0], num_heads,
                                     block_table.shape[1], block_size, int(num_blocks or 0),
                                     _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _ptr(dev_status), _stream(stream)))


def _check_decode_tensors(q, cache, block_table, seq_lens, out, lse):
    """dtype, layout and shape checks shared by every decode entry point: the C
    ABI sees raw pointers, so a mismatched out, lse, seq_lens or block_table
    would otherwise be read or written past its end on the device."""
    import torch
    _need(q, torch.bfloat16, 3, "q")
    _need(cache, torch.bfloat16, 3, "cache")
    _need(block_table, torch.int32, 2, "block_table")
    _need(seq_lens, torch.int32, 1, "seq_lens")
    _need(out, torch.bfloat16, 3, "out")
    if lse is not None:
        _need(lse, torch.float32, 2, "lse")
    B, H, row = q.shape
    if row != ROW_DIM or cache.shape[2] != ROW_DIM or tuple(out.shape) != (B, H, KV_LORA_RANK):
        raise ValueError("shape mismatch: q [B,H,576], cache [NB,BS,576], out [B,H,512]")
    if seq_lens.shape[0] != B or block_table.shape[0] != B:
        raise ValueError("seq_lens / block_table batch mismatch")
    if lse is not None and tuple(lse.shape) != (B, H):
        raise ValueError(f"lse must be [B, H] = [{B}, {H}], got {tuple(lse.shape)}")
    return B, H


def _decode(fn, q, cache, block_table, seq_lens, softmax_scale, out, lse, workspace,
            max_seq_len, dev_status, stream):
    B, H = _check_decode_tensors(q, cache, block_table, seq_lens, out, lse)
    if max_seq_len is None:
        max_seq_len = block_table.shape[1] * cache.shape[1]
    _check(fn(_ptr(q), _ptr(cache), cache.shape[0], cache.shape[1], _ptr(block_table),
              block_table.shape[1], _ptr(seq_lens), B, H, int(max_seq_len), float(softmax_scale),
              _ptr(out), _ptr(lse), _ptr(workspace),
              workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)))
    return out


def mla_decode(q, cache, block_table, seq_lens, softmax_scale, out, lse=None, workspace=None,
               max_seq_len=None, dev_status=None, stream=None):
    """Absorbed-form MLA decode: out[b,h] = softmax(scale * q[b,h] . rows) @ rows[:, :512]."""
    if workspace is None:
        workspace = make_workspace(q.shape[0], q.shape[1], q.device)
    return _decode(get_lib().mla_decode, q, cache, block_table, seq_lens, softmax_scale, out, lse,
                   workspace, max_seq_len, dev_status, stream)


def mla_decode_planned(q, cache, block_table, seq_lens, softmax_scale, out, lse=None,
                       workspace=None, max_seq_len=None, dev_status=None, stream=None):
    """mla_decode reusing the plan mla_decode_plan wrote into `workspace`."""
    return _decode(get_lib().mla_decode_planned, q, cache, block_table, seq_lens, softmax_scale, out,
                   lse, workspace, max_seq_len, dev_status, stream)


def _with_kv_new(entry, kv_new, q):
    import torch
    if kv_new is not None:
        _need(kv_new, torch.bfloat16, 2, "kv_new")
        if tuple(kv_new.shape) != (q.shape[0], ROW_DIM):
            raise ValueError("kv_new must be [B, 576]")

    def fn(qp, cp, nb, bs, btp, mb, slp, B, H, msl, sc, op, lp, wp, wb, dsp, st):
        return entry(qp, cp, _ptr(kv_new), nb, bs, btp, mb, slp, B, H, msl, sc, op, lp, wp, wb,
                     dsp, st)
    return fn


def mla_decode_partial(q, cache, block_table, seq_lens, softmax_scale, out, lse=None,
                       workspace=None, max_seq_len=None, dev_status=None, stream=None,
                       kv_new=None):
    """The decode kernel of mla_decode_planned alone (split requests leave partials);
    with kv_new, each request's new row is stored first (as mla_decode_append_planned)."""
    return _decode(_with_kv_new(get_lib().mla_decode_partial, kv_new, q), q, cache, block_table,
                   seq_lens, softmax_scale, out, lse, workspace, max_seq_len, dev_status, stream)


def mla_decode_append_planned(q, cache, kv_new, block_table, seq_lens, softmax_scale, out,
                              lse=None, workspace=None, max_seq_len=None, dev_status=None,
                              stream=None):
    """Store kv_new[b] at position seq_lens[b]-1 of request b, then mla_decode_planned, in
    one decode kernel (plus the split combine)."""
    if kv_new is None:
        raise ValueError("kv_new is required")
    return _decode(_with_kv_new(get_lib().mla_decode_append_planned, kv_new, q), q, cache,
                   block_table, seq_lens, softmax_scale, out, lse, workspace, max_seq_len,
                   dev_status, stream)


def mla_combine_planned(workspace, batch, out, lse=None, num_heads=None, stream=None):
    """Merge the partials mla_decode_partial left in `workspace` into out / lse
    (num_heads: out's head count unless given)."""
    import torch
    _need(out, torch.bfloat16, 3, "out")
    if num_heads is None:
        num_heads = out.shape[1]
    if lse is not None:
        _need(lse, torch.float32, 2, "lse")
    _check(get_lib().mla_combine_planned(_ptr(workspace),
                                         workspace.numel() * workspace.element_size(), int(batch),
                                         num_heads, _ptr(out), _ptr(lse), _stream(stream)))
    return out


def mla_combine(o_partial, lse_partial, split_offsets, out, lse=None, stream=None):
    """Log-sum-exp merge of split partials (fp32 [W,H,512], [W,H]) into out bf16 [B,H,512]."""
    import torch
    _need(o_partial, torch.float32, 3, "o_partial")
    _need(lse_partial, torch.float32, 2, "lse_partial")
    _need(split_offsets, torch.int32, 1, "split_offsets")
    _need(out, torch.bfloat16, 3, "out")
    B = split_offsets.shape[0] - 1
    H = o_partial.shape[1]
    if o_partial.shape[2] != KV_LORA_RANK or tuple(out.shape) != (B, H, KV_LORA_RANK):
        raise ValueError("shape mismatch")
    _check(get_lib().mla_combine(_ptr(o_partial), _ptr(lse_partial), _ptr(split_offsets), B, H,
                           _ptr(out), _ptr(lse), _stream(stream)))
    return out


def mla_decode_noalloc(q, cache, block_table, seq_lens, softmax_scale, out, lse=None,
                       max_seq_len=None, dev_status=None, stream=None):
    """mla_decode without a workspace, for callers that cannot allocate device
    memory: the library's fixed 16 MiB scratch array stands in for it (128
    heads, batch <= 8192; make a first call per device at set-up; calls must
    not overlap on the GPU)."""
    B, H = _check_decode_tensors(q, cache, block_table, seq_lens, out, lse)
    if max_seq_len is None:
        max_seq_len = block_table.shape[1] * cache.shape[1]
    _check(get_lib().mla_decode_noalloc(
        _ptr(q), _ptr(cache), cache.shape[0], cache.shape[1], _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, H, int(max_seq_len), float(softmax_scale),
        _ptr(out), _ptr(lse), _ptr(dev_status), _stream(stream)))
    return out


def mla_cache_append_fp8(kv_new, slot_mapping, cache8, kv_scale=1.0, dev_status=None,
                         stream=None):
    """Quantise each bf16 row of kv_new into the FP8 (E4M3) cache at its slot
    (code nearest to x / kv_scale, ties to even, saturating to 448)."""
    import torch
    _need(kv_new, torch.bfloat16, 2, "kv_new")
    _need(slot_mapping, torch.int64, 1, "slot_mapping")
    _need(cache8, torch.uint8, 3, "cache8")
    if kv_new.shape[1] != ROW_DIM or cache8.shape[2] != ROW_DIM:
        raise ValueError("rows must be 576 wide")
    if slot_mapping.shape[0] != kv_new.shape[0]:
        raise ValueError("slot_mapping and kv_new disagree on the token count")
    _check(get_lib().mla_cache_append_fp8(_ptr(kv_new), _ptr(slot_mapping), kv_new.shape[0],
                                          _ptr(cache8), cache8.shape[0], cache8.shape[1],
                                          float(kv_scale), _ptr(dev_status), _stream(stream)))


def mla_decode_fp8(q, cache8, block_table, seq_lens, softmax_scale, out, lse=None,
                   kv_scale=1.0, workspace=None, max_seq_len=None, dev_status=None, stream=None):
    """Absorbed-form MLA decode over an FP8 (E4M3) cache: row elements are
    value(code) * kv_scale (plans, decodes, merges)."""
    return _decode_fp8(get_lib().mla_decode_fp8, None, q, cache8, block_table, seq_lens,
                       softmax_scale, out, lse, kv_scale, workspace, max_seq_len, dev_status,
                       stream)


def mla_decode_fp8_planned(q, cache8, block_table, seq_lens, softmax_scale, out, lse=None,
                           kv_scale=1.0, workspace=None, max_seq_len=None, dev_status=None,
                           stream=None, kv_new=None):
    """mla_decode_fp8 with the plan already in `workspace`; with kv_new (bf16 [B, 576]) each
    request's new row is quantised into the cache first, inside the decode kernel."""
    return _decode_fp8(get_lib().mla_decode_fp8_planned, kv_new, q, cache8, block_table,
                       seq_lens, softmax_scale, out, lse, kv_scale, workspace, max_seq_len,
                       dev_status, stream)


def _decode_fp8(fn, kv_new, q, cache8, block_table, seq_lens, softmax_scale, out, lse, kv_scale,
                workspace, max_seq_len, dev_status, stream):
    import torch
    _need(q, torch.bfloat16, 3, "q")
    _need(cache8, torch.uint8, 3, "cache8")
    _need(block_table, torch.int32, 2, "block_table")
    _need(seq_lens, torch.int32, 1, "seq_lens")
    _need(out, torch.bfloat16, 3, "out")
    if lse is not None:
        _need(lse, torch.float32, 2, "lse")
    B, H, row = q.shape
    if row != ROW_DIM or cache8.shape[2] != ROW_DIM or tuple(out.shape) != (B, H, KV_LORA_RANK):
        raise ValueError("shape mismatch: q [B,H,576], cache8 [NB,BS,576], out [B,H,512]")
    if seq_lens.shape[0] != B or block_table.shape[0] != B:
        raise ValueError("seq_lens / block_table batch mismatch")
    if lse is not None and tuple(lse.shape) != (B, H):
        raise ValueError(f"lse must be [B, H] = [{B}, {H}], got {tuple(lse.shape)}")
    if kv_new is not None:
        _need(kv_new, torch.bfloat16, 2, "kv_new")
        if tuple(kv_new.shape) != (B, ROW_DIM):
            raise ValueError("kv_new must be [B, 576]")
    if workspace is None:
        workspace = make_workspace(B, H, q.device)
    if max_seq_len is None:
        max_seq_len = block_table.shape[1] * cache8.shape[1]
    args = [_ptr(q), _ptr(cache8)]
    if kv_new is not None or fn is get_lib().mla_decode_fp8_planned:
        args.append(_ptr(kv_new))
    args += [cache8.shape[0], cache8.shape[1], _ptr(block_table), block_table.shape[1],
             _ptr(seq_lens), B, H, int(max_seq_len), float(softmax_scale), float(kv_scale),
             _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
             _ptr(dev_status), _stream(stream)]
    _check(fn(*args))
    return out


def place_requests(kv_tokens, ranks: int, capacity_tokens: int = 0):
    """KV-load-aware placement of requests on `ranks` DP attention ranks
    (mla_place_requests; host only).  kv_tokens: cached tokens per request.
    Returns (rank_of int32 [n], -1 where no rank can hold the request within
    capacity_tokens; rank_load int64 [ranks])."""
    import numpy as np
    t = np.ascontiguousarray(kv_tokens, dtype=np.int64)
    if t.ndim != 1:
        raise ValueError("kv_tokens must be 1-D")
    rank_of = np.empty(t.shape[0], np.int32)
    rank_load = np.empty(int(ranks), np.int64)
    unplaced = ctypes.c_int32(0)
    _check(get_lib().mla_place_requests(t.ctypes.data if t.size else None, t.shape[0], int(ranks),
                                        int(capacity_tokens),
                                        rank_of.ctypes.data if t.size else None,
                                        rank_load.ctypes.data, ctypes.byref(unplaced)))
    return rank_of, rank_load


def place_one(rank_load, kv_tokens: int, capacity_tokens: int = 0) -> int:
    """The rank a new request of kv_tokens cached tokens goes to, given the
    ranks' loads (mla_place_one; host only), or -1 if none can hold it."""
    import numpy as np
    lo = np.ascontiguousarray(rank_load, dtype=np.int64)
    rank = ctypes.c_int32(0)
    _check(get_lib().mla_place_one(lo.ctypes.data, lo.shape[0], int(capacity_tokens),
                                   int(kv_tokens), ctypes.byref(rank)))
    return rank.value


def mla_absorb_q(q_nope, q_pe, w_uk, q, dev_status=None, stream=None):
    """q[b,h,0:512] = q_nope[b,h] . W_UK[h]; q[b,h,512:576] = q_pe[b,h] (mla_absorb_q).
    dev_status: optional device int32 [1], set to MLA_ERR_DEVICE_TIMEOUT if a wait runs out."""
    import torch
    _need(q_nope, torch.bfloat16, 3, "q_nope")
    _need(q_pe, torch.bfloat16, 3, "q_pe")
    _need(w_uk, torch.bfloat16, 3, "w_uk")
    _need(q, torch.bfloat16, 3, "q")
    B, H = q_nope.shape[0], q_nope.shape[1]
    if (tuple(q_nope.shape) != (B, H, 128) or tuple(q_pe.shape) != (B, H, 64)
            or tuple(w_uk.shape) != (H, 128, 512) or tuple(q.shape) != (B, H, ROW_DIM)):
        raise ValueError("shapes: q_nope [B,H,128], q_pe [B,H,64], w_uk [H,128,512], q [B,H,576]")
    _check(get_lib().mla_absorb_q(_ptr(q_nope), _ptr(q_pe), _ptr(w_uk), B, H, _ptr(q),
                                  _ptr(dev_status), _stream(stream)))
    return q


def mla_absorb_out(out, w_uv, o, dev_status=None, stream=None):
    """o[b,h] = out[b,h] . W_UV[h] (mla_absorb_out).  dev_status as for mla_absorb_q."""
    import torch
    _need(out, torch.bfloat16, 3, "out")
    _need(w_uv, torch.bfloat16, 3, "w_uv")
    _need(o, torch.bfloat16, 3, "o")
    B, H = out.shape[0], out.shape[1]
    if (tuple(out.shape) != (B, H, 512) or tuple(w_uv.shape) != (H, 512, 128)
            or tuple(o.shape) != (B, H, 128)):
        raise ValueError("shapes: out [B,H,512], w_uv [H,512,128], o [B,H,128]")
    _check(get_lib().mla_absorb_out(_ptr(out), _ptr(w_uv), B, H, _ptr(o), _ptr(dev_status),
                                    _stream(stream)))
    return o


def selftest_wait_timeout(budget_ns: int, dev_status, elapsed_ns, stream=None):
    """Runs the device check of the bounded waits (mla_selftest_wait_timeout):
    dev_status int32 [1] receives MLA_ERR_DEVICE_TIMEOUT, elapsed_ns int64 [2]
    each warp's wait time in ns.  Asynchronous on `stream`."""
    import torch
    _need(dev_status, torch.int32, 1, "dev_status")
    _need(elapsed_ns, torch.int64, 1, "elapsed_ns")
    if elapsed_ns.shape[0] < 2:
        raise ValueError("elapsed_ns needs 2 entries")
    _check(get_lib().mla_selftest_wait_timeout(int(budget_ns), _ptr(dev_status), _ptr(elapsed_ns),
                                               _stream(stream)))
