"""Failure detection of the attention forward's pipeline: every wait is
bounded, and a wait that cannot complete ends the kernel with
CPTHD_ERR_TIMEOUT recorded in err, instead of a hang.

The test loads a test-only build of the library (CPTHD_WAIT_TEST, built
apart from libcpthd.so by build.build_wait_test): its waits give up after
5 ms, and its data-relay warp withholds the arrivals for key block 1, so the
MMA issuer's wait for P(1) never completes. Every CTA with more than one key
block must then raise its abort flag, drain its copies and MMAs, free its
tensor memory and return. The test checks that the call ends within a few
seconds, that err reads CPTHD_ERR_TIMEOUT, and that the regular library
then runs the same slice correctly in the same process (the aborted CTAs
released their tensor memory, and the context is still usable).
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


@pytest.mark.gpu
def test_withheld_arrival_ends_in_timeout_status():
    dev = cuda_or_skip()
    cp = load_lib()
    from context_packed_thd_gb300 import build
    test_lib = ctypes.CDLL(build.build_wait_test())
    test_lib.thd_causal_attn_fwd.argtypes = cp.lib.thd_causal_attn_fwd.argtypes
    test_lib.thd_causal_attn_fwd.restype = ctypes.c_int

    cfg = W.CONFIG_BY_NAME["t8192_mha16"]
    inp = W.make_attn_inputs(cfg, "dcs")
    lay = inp.layout
    cu = torch.from_numpy(lay.cu_seqlens).to(dev)
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    idx = cp.cp_partition_index("dcs", cup, lay.T, cfg.cp, 0)
    q_loc = cp.cp_reorder(q, idx)
    t_local = q_loc.shape[0]
    out = torch.zeros_like(q_loc)
    lse = torch.zeros((cfg.hq, t_local), dtype=torch.float32, device=dev)
    ws = torch.empty(cp.thd_causal_attn_workspace_size(t_local, cfg.hq, cfg.hkv, cfg.d), dtype=torch.uint8,
                     device=dev)
    err = new_err(dev)
    torch.cuda.synchronize()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    t0 = time.perf_counter()
    rc = test_lib.thd_causal_attn_fwd(p(idx), t_local, p(q_loc), p(k), p(v), lay.T, p(cu), p(cup), lay.num_docs,
                                      cfg.hq, cfg.hkv, cfg.d, 0.0, p(out), p(lse), p(ws), ws.numel(), p(err),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert err.cpu().tolist()[0] == TIMEOUT, err.cpu().tolist()
    assert elapsed < 10.0, elapsed

    # the regular library, same process, same slice: correct results
    err2 = new_err(dev)
    out2, lse2 = cp.thd_causal_attn_fwd(idx, q_loc, k, v, cu, cup, err=err2)
    torch.cuda.synchronize()
    assert err2.cpu().tolist() == [0, 0]
    ref_idx = np.asarray(P.partition_index("dcs", lay.cu_seqlens_padded.tolist(), cfg.cp, 0), dtype=np.int64)
    ro, rl = A.attention_fwd(inp.q[torch.from_numpy(ref_idx)], inp.k, inp.v, lay.cu_seqlens,
                             lay.cu_seqlens_padded, ref_idx)
    assert_attn_matches(out2, lse2, ro, rl, "after the timeout")
