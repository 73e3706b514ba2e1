"""Failure detection of the attention forward's pipeline: every wait is
bounded, and a wait that cannot complete ends the kernel with
CPTHD_ERR_TIMEOUT recorded in err, instead of a hang.

The tests load a test-only build of the library (CPTHD_WAIT_TEST, built
apart from libcpthd.so by build.build_wait_test): its waits give up after
5 ms, and it withholds one signal, chosen with cpthd_wait_test_mode:

  1. the data-relay warp withholds its arrivals for key block 1, so the MMA
     issuer's wait for P(1) never completes (a wait inside one CTA);
  2. the pieces of items cut between CTAs never raise their hand-off flags,
     so the CTA that merges an item's pieces waits in vain (a wait on
     another CTA).

Every CTA whose wait runs out must raise its abort flag, drain its copies
and MMAs, free its tensor memory and return. Each test checks that the call
ends within a few seconds, that err reads CPTHD_ERR_TIMEOUT, and that the
regular library then runs the same slice correctly in the same process (the
aborted CTAs released their tensor memory, and the context is still usable).
"""
import ctypes
import time

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import partition as P
import workloads as W
from gpu_common import assert_attn_matches, cuda_or_skip, load_lib, new_err

TIMEOUT = -9


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _run_until_timeout(cp, dev, mode, idx, q_loc, k, v, T, cu, cup, num_docs, hq, hkv, dd):
    """One forward call of the test build with failure `mode`; returns err."""
    from context_packed_thd_gb300 import build
    test_lib = ctypes.CDLL(build.build_wait_test())
    test_lib.thd_causal_attn_fwd.argtypes = cp.lib.thd_causal_attn_fwd.argtypes
    test_lib.thd_causal_attn_fwd.restype = ctypes.c_int
    test_lib.cpthd_wait_test_mode.argtypes = [ctypes.c_int]
    test_lib.cpthd_wait_test_mode.restype = ctypes.c_int
    assert test_lib.cpthd_wait_test_mode(mode) == 0
    t_local = q_loc.shape[0]
    out = torch.zeros_like(q_loc)
    lse = torch.zeros((hq, t_local), dtype=torch.float32, device=dev)
    ws = torch.empty(cp.thd_causal_attn_workspace_size(t_local, hq, hkv, dd), dtype=torch.uint8, device=dev)
    err = new_err(dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = test_lib.thd_causal_attn_fwd(_p(idx), t_local, _p(q_loc), _p(k), _p(v), T, _p(cu), _p(cup), num_docs,
                                      hq, hkv, dd, 0.0, _p(out), _p(lse), _p(ws), ws.numel(), _p(err),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 10.0, elapsed
    return err.cpu().tolist()


@pytest.mark.gpu
def test_withheld_arrival_ends_in_timeout_status():
    dev = cuda_or_skip()
    cp = load_lib()
    cfg = W.CONFIG_BY_NAME["t8192_mha16"]
    inp = W.make_attn_inputs(cfg, "dcs")
    lay = inp.layout
    cu = torch.from_numpy(lay.cu_seqlens).to(dev)
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    idx = cp.cp_partition_index("dcs", cup, lay.T, cfg.cp, 0)
    q_loc = cp.cp_reorder(q, idx)
    err = _run_until_timeout(cp, dev, 1, idx, q_loc, k, v, lay.T, cu, cup, lay.num_docs, cfg.hq, cfg.hkv, cfg.d)
    assert err[0] == TIMEOUT, err

    # the regular library, same process, same slice: correct results
    err2 = new_err(dev)
    out2, lse2 = cp.thd_causal_attn_fwd(idx, q_loc, k, v, cu, cup, err=err2)
    torch.cuda.synchronize()
    assert err2.cpu().tolist() == [0, 0]
    ref_idx = np.asarray(P.partition_index("dcs", lay.cu_seqlens_padded.tolist(), cfg.cp, 0), dtype=np.int64)
    ro, rl = A.attention_fwd(inp.q[torch.from_numpy(ref_idx)], inp.k, inp.v, lay.cu_seqlens,
                             lay.cu_seqlens_padded, ref_idx)
    assert_attn_matches(out2, lse2, ro, rl, "after the timeout")


@pytest.mark.gpu
def test_withheld_piece_flags_end_in_timeout_status():
    """One 16384-token document as one slice (cp_size 1), one head, d 128:
    the items are long, so the CTAs take equal shares of the work and items
    are cut into pieces; with the pieces' flags withheld, every merging CTA's
    flag wait runs out."""
    dev = cuda_or_skip()
    cp = load_lib()
    hq = hkv = 1
    dd = 128
    lay = W.make_layout([16384], 1)
    q_h, k_h, v_h = W.make_qkv_logical(47, 16384, hq, hkv, dd)
    cu = torch.from_numpy(lay.cu_seqlens).to(dev)
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    idx = cp.cp_partition_index("nlb", cup, lay.T, 1, 0)
    q_loc = cp.cp_reorder(q, idx)
    err = _run_until_timeout(cp, dev, 2, idx, q_loc, k, v, lay.T, cu, cup, lay.num_docs, hq, hkv, dd)
    assert err[0] == TIMEOUT, err

    err2 = new_err(dev)
    out2, lse2 = cp.thd_causal_attn_fwd(idx, q_loc, k, v, cu, cup, err=err2)
    torch.cuda.synchronize()
    assert err2.cpu().tolist() == [0, 0]
    ref_idx = np.arange(lay.T, dtype=np.int64)
    ro, rl = A.attention_fwd(q_h, k_h, v_h, lay.cu_seqlens, lay.cu_seqlens_padded, ref_idx)
    assert_attn_matches(out2, lse2, ro, rl, "after the flag timeout")
