"""mla_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (a host framework that owns all device memory and gives a plugin
only its inputs and outputs, or a serving path that must not touch the
allocator mid-step).  It uses the library's fixed scratch array instead of a
workspace, so its results must match mla_decode's within the parity tolerance,
also on a second call right after the first (the scratch keeps the previous
call's contents and must not leak into the next result).

Collected last on purpose, and self-contained so it also passes alone in a
fresh process.
"""
import ctypes

import numpy as np
import pytest

import mla_inputs as mi
from gpu_helpers import assert_close, assert_lse_close, dev, dev_bf16, host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _inputs(lens, block_size, seed, q_kind):
    w = mi.custom_workload(lens, block_size=block_size, append=False, pool_factor=1.3)
    d = mi.make_host_layer(w, np.random.default_rng(seed), q_kind=q_kind)
    return dict(q=dev_bf16(d["q"]), cache=dev_bf16(d["cache"]),
                bt=dev(d["block_table"], torch.int32), sl=dev(d["seq_lens"], torch.int32),
                scale=d["softmax_scale"], B=len(lens))


def _noalloc_via_c_abi(lib, x, out, lse, status, heads=128):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.mla_decode_noalloc(
        ctypes.c_void_p(x["q"].data_ptr()), ctypes.c_void_p(x["cache"].data_ptr()),
        x["cache"].shape[0], x["cache"].shape[1], ctypes.c_void_p(x["bt"].data_ptr()),
        x["bt"].shape[1], ctypes.c_void_p(x["sl"].data_ptr()), x["B"], heads,
        x["bt"].shape[1] * x["cache"].shape[1], ctypes.c_float(x["scale"]),
        ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()) if lse is not None else None,
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream))


def test_noalloc_matches_mla_decode_on_two_calls_in_a_row():
    assert torch.cuda.is_available()
    import mla_latent_cache_decode_gb300 as mla
    lib = mla.get_lib()
    cases = [_inputs([2, 18, 65, 201, 4096, 1], 16, 31, "sharp"),
             _inputs([9000, 7, 300, 1200, 64, 129, 1, 3333], 64, 32, "normal")]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    results = []
    for x in cases:   # two calls in a row, different batch and lengths
        out = torch.full((x["B"], 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((x["B"], 128), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc_via_c_abi(lib, x, out, lse, status)
        assert rc == 0, mla.get_lib().mla_last_error_detail()
        results.append((out, lse))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for x, (out, lse) in zip(cases, results):
        ref = torch.empty((x["B"], 128, 512), dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.empty((x["B"], 128), dtype=torch.float32, device="cuda")
        mla.mla_decode(x["q"], x["cache"], x["bt"], x["sl"], x["scale"], ref, ref_lse)
        torch.cuda.synchronize()
        assert_close(host_f64(out), host_f64(ref), "noalloc vs mla_decode")
        assert_lse_close(lse.cpu().numpy(), ref_lse.cpu().numpy())


def test_noalloc_rejects_batch_beyond_its_scratch():
    import mla_latent_cache_decode_gb300 as mla
    lib = mla.get_lib()
    rc = lib.mla_decode_noalloc(None, None, 1, 64, None, 1, None, 8193, 128, 64,
                                ctypes.c_float(0.1), None, None, None, None)
    assert rc == 1
    assert b"MLA_NOALLOC_MAX_BATCH" in lib.mla_last_error_detail()


def test_noalloc_rejects_other_head_counts_on_the_host():
    """Only the kernel's 128 heads: a tensor-parallel rank's 16 heads would need
    q padded into a workspace, which this entry point does not have."""
    import mla_latent_cache_decode_gb300 as mla
    lib = mla.get_lib()
    x = _inputs([5, 70], 16, 33, "normal")
    out = torch.empty((x["B"], 128, 512), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc_via_c_abi(lib, x, out, None, status, heads=16) == 2
    assert b"num_heads" in lib.mla_last_error_detail()
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_noalloc_without_lse_and_at_an_intermediate_batch():
    """lse = NULL, and a 4096-request batch holding one long-context request:
    the fixed scratch then holds fewer split ranges than mla_decode's workspace
    (one per SM pair), so the plans differ; the results agree within the
    tolerance, and out written with lse = NULL equals out written with it."""
    import mla_latent_cache_decode_gb300 as mla
    lib = mla.get_lib()
    rng = np.random.default_rng(4096)
    lens = rng.integers(1, 100, size=4096).tolist()
    lens[1234] = 30000
    x = _inputs(lens, 32, 34, "sharp")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_nolse = torch.full((x["B"], 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _noalloc_via_c_abi(lib, x, out_nolse, None, status) == 0, lib.mla_last_error_detail()
    out = torch.full_like(out_nolse, float("nan"))
    lse = torch.full((x["B"], 128), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc_via_c_abi(lib, x, out, lse, status) == 0, lib.mla_last_error_detail()
    ref = torch.empty_like(out)
    ref_lse = torch.empty_like(lse)
    mla.mla_decode(x["q"], x["cache"], x["bt"], x["sl"], x["scale"], ref, ref_lse,
                   dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out_nolse.view(torch.int16), out.view(torch.int16))
    assert_close(host_f64(out), host_f64(ref), "noalloc vs mla_decode, 4096 requests")
    assert_close(host_f64(out[1234]), host_f64(ref[1234]), "the 30000-token request")
    assert_lse_close(lse.cpu().numpy(), ref_lse.cpu().numpy())


def test_maximum_batch_against_oracle():
    """The largest batch the library documents (MLA_NOALLOC_MAX_BATCH = 8192
    requests of 1-24 tokens, page 16): mla_decode with a workspace and
    mla_decode_noalloc, whose 16 MiB scratch then holds only ~62 of the split
    ranges, both against the oracle on sampled requests and against each
    other everywhere."""
    import mla_latent_cache_decode_gb300 as mla
    import oracle
    lib = mla.get_lib()
    B = 8192
    rng = np.random.default_rng(8192)
    lens = rng.integers(1, 25, size=B).tolist()
    w = mi.custom_workload(lens, block_size=16, append=True, pool_factor=1.2)
    dl = mi.make_device_layer(w, 0, "cuda", q_kind="sharp")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache0 = mi.to_bits(dl["cache"])   # the oracle's input: the cache before any GPU work
    mla.mla_cache_append(dl["kv_new"], dl["slot_mapping"], dl["cache"], dev_status=status)
    x = dict(q=dl["q"], cache=dl["cache"], bt=dl["block_table"], sl=dl["seq_lens"],
             scale=dl["softmax_scale"], B=B)
    out = torch.full((B, 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, 128), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode(x["q"], x["cache"], x["bt"], x["sl"], x["scale"], out, lse, dev_status=status)
    out_na = torch.full_like(out, float("nan"))
    lse_na = torch.full_like(lse, float("nan"))
    rc = _noalloc_via_c_abi(lib, x, out_na, lse_na, status)
    assert rc == 0, lib.mla_last_error_detail()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(host_f64(out_na), host_f64(out), "noalloc vs mla_decode at 8192 requests")
    assert_lse_close(lse_na.cpu().numpy(), lse.cpu().numpy())
    arr = np.array(lens)
    reqs = sorted({0, 1, B // 2, B - 1, int(arr.argmin()), int(arr.argmax())}
                  | set(rng.choice(B, 26, replace=False).tolist()))
    oracle.append(mi.to_bits(dl["kv_new"]), dl["slot_mapping"].cpu().numpy(), cache0)
    ref, ref_lse = oracle.decode(mi.to_bits(dl["q"][reqs]), cache0, dl["block_table_host"][reqs],
                                 arr[reqs].astype(np.int32), dl["softmax_scale"])
    for name, o, l in (("mla_decode", out, lse), ("noalloc", out_na, lse_na)):
        assert_close(host_f64(o)[reqs], ref, f"{name} at 8192 requests")
        assert_lse_close(l.cpu().numpy()[reqs], ref_lse)
