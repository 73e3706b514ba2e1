"""thd_causal_attn_fwd_static_scratch: the attention entry point for callers
that cannot allocate device memory (a host framework that owns every
allocation, a plugin that must not call cudaMalloc in the middle of a step).
It keeps its scratch in a fixed array inside the library instead of a
caller workspace.

The GPU test calls it twice in a row through the C ABI, on two different
slices (the second call finds the first call's leftovers in the shared
array), and checks that each result equals the regular entry point's bit for
bit (both run the same kernels). This file sorts last so that a
run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import workloads as W
from gpu_common import cuda_or_skip, load_lib, new_err

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


def test_static_scratch_host_checks_match_workspace_entry_point():
    """The same host checks, in the same order, as thd_causal_attn_fwd: shape
    arguments first (also for an empty slice), then the head dim, then the
    scratch limit. Fake pointers: every call here returns before a launch."""
    cp = load_lib()
    f = cp.lib.thd_causal_attn_fwd_static_scratch
    g = cp.lib.thd_causal_attn_fwd
    p = ctypes.c_void_p(256)

    def both(t_local, T, num_docs, hq, hkv, d):
        a = f(p, t_local, p, p, p, T, p, None, num_docs, hq, hkv, d, 0.0, p, p, None, None)
        b = g(p, t_local, p, p, p, T, p, None, num_docs, hq, hkv, d, 0.0, p, p, None, 0, None, None)
        return a, b

    assert both(0, -1, 1, 2, 2, 64) == (-1, -1)             # negative T, empty slice
    assert both(0, 8, -1, 2, 2, 64) == (-1, -1)             # negative document count
    assert both(0, 8, 1, 65536 * 2, 2, 64) == (-3, -3)     # too many query heads
    assert both(4, 8, 1, 3, 2, 64) == (-3, -3)              # GQA mismatch
    assert both(4, 8, 1, 2, 2, 96) == (-3, -3)              # head dim
    assert both(2 ** 31, 2 ** 31 - 1, 1, 2, 2, 64) == (-1, -1)  # t_local beyond int32: invalid, not a scratch limit
    assert both(0, 8, 1, 2, 2, 64) == (0, 0)                # empty slice: nothing to do


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
        # both entry points run the same kernels on the same inputs: the
        # results are identical, bit for bit
        assert torch.equal(out, ref_out), f"{cfg.name}: output differs"
        assert torch.equal(lse, ref_lse), f"{cfg.name}: LSE differs"
