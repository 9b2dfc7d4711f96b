"""C-ABI library checks that need no GPU: it loads, exports every declared
symbol, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mla_latent_cache_decode_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(mla_\w+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_binding_names_match_header():
    import mla_latent_cache_decode_gb300 as mla
    assert set(mla.EXPORTED) == set(declared_functions())


def test_status_strings_and_version(lib):
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_abi_version.restype = ctypes.c_int
    assert lib.mla_abi_version() == 4
    names = [lib.mla_status_string(i).decode() for i in range(8)]
    assert names[0] == "MLA_OK" and names[6] == "MLA_ERR_DEVICE_TIMEOUT"
    assert names[7] == "MLA_ERR_DEVICE_PLAN"
    assert lib.mla_status_string(99).decode() == "MLA_ERR_UNKNOWN"


def test_host_validation_before_any_launch(lib):
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.mla_decode.argtypes = [P, P, i64, i32, P, i32, P, i32, i32, i32, f32, P, P, P, sz, P, P]
    lib.mla_decode.restype = ctypes.c_int
    lib.mla_last_error_detail.restype = ctypes.c_char_p
    lib.mla_cache_append.argtypes = [P, P, i64, P, i64, i32, P, P]
    lib.mla_cache_append.restype = ctypes.c_int
    lib.mla_combine.argtypes = [P, P, P, i32, i32, P, P, P]
    lib.mla_combine.restype = ctypes.c_int
    args = lambda batch, heads, bs: (None, None, 1, bs, None, 1, None, batch, heads, 1, 0.1,
                                     None, None, None, 0, None, None)
    assert lib.mla_decode(*args(-1, 128, 64)) == 1
    assert lib.mla_decode(*args(2, 129, 64)) == 2         # more heads than 128
    assert b"num_heads" in lib.mla_last_error_detail()
    assert lib.mla_decode(*args(2, 0, 64)) == 2
    assert lib.mla_decode(*args(2, 16, 64)) == 1          # a TP rank's 16 heads: past the
                                                          # head check, then null pointers
    assert lib.mla_decode(*args(2, 128, 48)) == 2         # unsupported page size
    assert lib.mla_decode(*args(2, 128, 0)) == 1
    assert lib.mla_decode(*args(0, 128, 64)) == 0         # empty batch: valid no-op
    assert lib.mla_decode(*args(2, 128, 64)) == 1         # null pointers
    assert lib.mla_cache_append(None, None, 0, None, 1, 16, None, None) == 0
    assert lib.mla_cache_append(None, None, 3, None, 1, 16, None, None) == 1
    assert lib.mla_cache_append(None, None, -1, None, 1, 16, None, None) == 1
    assert lib.mla_combine(None, None, None, 0, 128, None, None, None) == 0
    assert lib.mla_combine(None, None, None, 2, 128, None, None, None) == 1


def test_wait_selftest_host_validation(lib):
    P = ctypes.c_void_p
    lib.mla_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P, P, P]
    lib.mla_selftest_wait_timeout.restype = ctypes.c_int
    lib.mla_last_error_detail.restype = ctypes.c_char_p
    st, el = ctypes.c_int32(0), (ctypes.c_uint64 * 2)()
    pst, pel = ctypes.addressof(st), ctypes.addressof(el)
    assert lib.mla_selftest_wait_timeout(0, pst, pel, None) == 1           # budget below 1 us
    assert b"budget_ns" in lib.mla_last_error_detail()
    assert lib.mla_selftest_wait_timeout(2_000_000_000, pst, pel, None) == 1  # above 1 s
    assert lib.mla_selftest_wait_timeout(1_000_000, None, pel, None) == 1
    assert lib.mla_selftest_wait_timeout(1_000_000, pst, None, None) == 1
    assert lib.mla_selftest_wait_timeout(1_000_000, pst + 1, pel, None) == 1  # misaligned
    assert st.value == 0  # nothing launched


def test_absorption_host_validation(lib):
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.mla_absorb_q.argtypes = [P, P, P, i32, i32, P, P, P]
    lib.mla_absorb_q.restype = ctypes.c_int
    lib.mla_absorb_out.argtypes = [P, P, i32, i32, P, P, P]
    lib.mla_absorb_out.restype = ctypes.c_int
    lib.mla_last_error_detail.restype = ctypes.c_char_p
    assert lib.mla_absorb_q(None, None, None, 0, 128, None, None, None) == 0     # empty batch: no-op
    assert lib.mla_absorb_q(None, None, None, -1, 128, None, None, None) == 1
    assert lib.mla_absorb_q(None, None, None, 4, 64, None, None, None) == 2      # heads other than 128
    assert lib.mla_absorb_q(None, None, None, 4, 128, None, None, None) == 1     # null pointers
    assert b"null" in lib.mla_last_error_detail()
    assert lib.mla_absorb_q(16, 32, 48, 4, 128, 72, None, None) == 1             # misaligned
    assert lib.mla_absorb_out(None, None, 0, 128, None, None, None) == 0
    assert lib.mla_absorb_out(None, None, 4, 128, None, None, None) == 1
    assert lib.mla_absorb_out(None, None, 4, 100, None, None, None) == 2


def test_partial_entry_points_take_few_or_all_heads(lib):
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.mla_decode_partial.argtypes = [P, P, P, i64, i32, P, i32, P, i32, i32, i32, f32, P, P, P,
                                       sz, P, P]
    lib.mla_decode_partial.restype = ctypes.c_int
    lib.mla_combine_planned.argtypes = [P, sz, i32, i32, P, P, P]
    lib.mla_combine_planned.restype = ctypes.c_int
    # the split form takes the few-head kernel's 1 to 32 heads or the pair
    # kernel's 128; 33 to 127 go through mla_decode(_planned), padded to 128
    assert lib.mla_decode_partial(None, None, None, 1, 64, None, 1, None, 2, 64, 1, 0.1, None,
                                  None, None, 0, None, None) == 2
    assert lib.mla_combine_planned(None, 0, 2, 64, None, None, None) == 2
    # 16 heads pass the head check and stop at the null pointers ...
    assert lib.mla_decode_partial(None, None, None, 1, 64, None, 1, None, 2, 16, 1, 0.1, None,
                                  None, None, 0, None, None) == 1
    assert lib.mla_combine_planned(None, 0, 2, 16, None, None, None) == 1
    # ... but the fused append needs all 128
    kv_new = ctypes.c_void_p(256)
    assert lib.mla_decode_partial(None, None, kv_new, 1, 64, None, 1, None, 2, 16, 1, 0.1, None,
                                  None, None, 0, None, None) == 2
    lib.mla_decode_workspace_size.argtypes = [i32, i32]
    lib.mla_decode_workspace_size.restype = sz
    assert lib.mla_decode_workspace_size(4, 129) == 0


def test_noalloc_host_validation(lib):
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.mla_decode_noalloc.argtypes = [P, P, i64, i32, P, i32, P, i32, i32, i32, f32, P, P, P, P]
    lib.mla_decode_noalloc.restype = ctypes.c_int
    lib.mla_last_error_detail.restype = ctypes.c_char_p
    call = lambda batch, heads: lib.mla_decode_noalloc(None, None, 1, 64, None, 1, None, batch,
                                                       heads, 64, 0.1, None, None, None, None)
    assert call(8193, 128) == 1                      # beyond the fixed scratch's batch limit
    assert b"MLA_NOALLOC_MAX_BATCH" in lib.mla_last_error_detail()
    assert call(4, 16) == 2                          # only the kernel's 128 heads
    assert b"num_heads" in lib.mla_last_error_detail()
    assert call(-1, 128) == 1
    assert call(0, 128) == 0                         # empty batch: valid no-op, nothing touched
