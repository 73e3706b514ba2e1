"""thd_causal_attn_fwd_static_scratch: the attention entry point for callers
that cannot allocate device memory (a host framework that owns every
allocation, a plugin that must not call cudaMalloc in the middle of a step).
It keeps its scratch in a fixed array inside the library instead of a
caller workspace.

The GPU test calls it twice in a row through the C ABI, on two different
slices (the second call finds the first call's leftovers in the shared
array), and checks each result against the regular entry point's under the
same tolerances as the other attention tests. This file sorts last so that a
run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from gpu_common import LSE_ATOL, OUT_ATOL, OUT_RTOL, cuda_or_skip, load_lib, new_err

SCRATCH_LIMIT = -10


def _static_call(cp, idx, q, k, v, cu, cup, out, lse, err):
    t_local, hq, d = q.shape
    T, hkv, _ = k.shape
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return cp.lib.thd_causal_attn_fwd_static_scratch(
        p(idx), t_local, p(q), p(k), p(v), T, p(cu), p(cup), cu.numel() - 1, hq, hkv, d, 0.0, p(out), p(lse), p(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _slice(cp, cfg, strategy, rank, dev):
    inp = W.make_attn_inputs(cfg, strategy)
    lay = inp.layout
    cu = torch.from_numpy(lay.cu_seqlens).to(dev)
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    idx = cp.cp_partition_index(strategy, cup, lay.T, cfg.cp, rank)
    return idx, cp.cp_reorder(q, idx), k, v, cu, cup


def test_static_scratch_limit_rejected_on_host():
    """A slice too large for the built-in array is refused before anything
    runs on a device (no GPU needed)."""
    cp = load_lib()
    rc = cp.lib.thd_causal_attn_fwd_static_scratch(None, 10_000_000, None, None, None, 10_000_000, None, None, 1,
                                                   8, 8, 128, 0.0, None, None, None, None)
    assert rc == SCRATCH_LIMIT
    assert "scratch" in cp.cpthd_status_string(rc)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point():
    dev = cuda_or_skip()
    cp = load_lib()
    cases = [
        (W.CONFIG_BY_NAME["t8192_mha16"], "dcs", 1),               # one head, two row tiles per CTA
        (W.CONFIG_BY_NAME["t32768_lognormal_gqa32x8"], "nlb", 5),  # two heads of one KV head per CTA
    ]
    for cfg, strategy, rank in cases:
        idx, q_loc, k, v, cu, cup = _slice(cp, cfg, strategy, rank, dev)
        ref_out, ref_lse = cp.thd_causal_attn_fwd(idx, q_loc, k, v, cu, cup)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        err = new_err(dev)
        rc = _static_call(cp, idx, q_loc, k, v, cu, cup, out, lse, err)
        assert rc == 0, cp.cpthd_status_string(rc)
        torch.cuda.synchronize()
        assert err.cpu().tolist() == [0, 0]
        o, r = out.float().cpu().numpy(), ref_out.float().cpu().numpy()
        assert np.all(np.abs(o - r) <= OUT_ATOL + OUT_RTOL * np.abs(r)), f"{cfg.name}: output differs"
        l, rl = lse.cpu().numpy(), ref_lse.cpu().numpy()
        assert np.array_equal(np.isneginf(l), np.isneginf(rl))
        fin = np.isfinite(rl)
        assert np.all(np.abs(l[fin] - rl[fin]) <= LSE_ATOL), f"{cfg.name}: LSE differs"
