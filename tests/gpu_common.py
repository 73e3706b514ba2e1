"""Helpers shared by the GPU parity tests: move seeded workloads to the
device, run the library through its C ABI binding, and compare with the
oracle under the stated tolerances."""
import numpy as np
import pytest
import torch

# max |out - ref| <= OUT_ATOL + OUT_RTOL * |ref| and |lse - ref| <= LSE_ATOL
OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 2e-3


def cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return torch.device("cuda:0")


def load_lib():
    from context_packed_thd_gb300 import build
    build.build()
    import context_packed_thd_gb300 as cp
    return cp


def new_err(dev):
    return torch.zeros(2, dtype=torch.int32, device=dev)


def assert_attn_matches(out, lse, ref_out, ref_lse, what=""):
    """out: bf16 [n, Hq, d]; lse: fp32 [Hq, n]; refs float64 numpy."""
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    pad = np.isneginf(ref_lse)                         # [Hq, n]
    assert np.array_equal(np.isneginf(l), pad), f"{what}: pad-row pattern differs"
    pad_rows = pad.all(axis=0)
    if pad_rows.any():
        assert np.all(o[pad_rows] == 0.0), f"{what}: pad rows not zero"
    fin = ~pad
    dl = np.abs(l[fin] - ref_lse[fin])
    assert dl.size == 0 or dl.max() <= LSE_ATOL, f"{what}: max |dLSE| = {dl.max():.3e}"
    err = np.abs(o - ref_out)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} outputs out of tolerance; worst excess "
                           f"{(err - bound).max():.3e}, max |dout| {err.max():.3e}")
    return float(err.max()), float(dl.max()) if dl.size else 0.0
