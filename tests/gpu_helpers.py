"""Helpers shared by the GPU tests: moving seeded host inputs to the device and
comparing device results with the oracle at the stated tolerance."""
from __future__ import annotations

import numpy as np

# Parity bar for bf16 cache / fp32 accumulation: rel-L2 <= 5e-3 and
# max-abs <= 1e-2 * max|ref| over the compared outputs.  lse is fp32: its
# error is fp32 rounding of a 576-term dot product and of log(sum): 2e-3
# absolute covers it with a wide margin (the observed error is ~1e-5).
REL_L2 = 5e-3
MAX_ABS_FRAC = 1e-2
LSE_ABS = 2e-3


def dev_bf16(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def dev(a, dtype, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device).to(dtype)


def host_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300)
    assert rel <= REL_L2 and mx <= MAX_ABS_FRAC, f"{what}: rel-L2 {rel:.3e}, max-abs/max|ref| {mx:.3e}"
    return rel, mx


def assert_lse_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    inf = np.isinf(ref)
    assert np.array_equal(np.isinf(got), inf), f"{what}: -inf pattern differs"
    if (~inf).any():
        err = np.abs(got[~inf] - ref[~inf]).max()
        assert err <= LSE_ABS, f"{what}: lse error {err:.3e}"
