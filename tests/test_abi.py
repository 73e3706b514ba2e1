"""The C ABI without a GPU: libcpthd.so loads, exports every entry point
include/cpthd.h declares, and its host-only calls validate their arguments
(no kernel is launched by any call in this file)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names += re.findall(r"CPTHD_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def cp():
    from context_packed_thd_gb300 import build
    build.build()
    import context_packed_thd_gb300 as cp
    return cp


def test_every_declared_symbol_is_exported(cp):
    names = _declared()
    assert {"cp_partition_index", "cp_restore_index", "cp_reorder", "cp_reorder_multi", "thd_causal_attn_fwd",
            "thd_causal_attn_workspace_size", "cp_local_tokens", "cpthd_status_string"} <= set(names)
    raw = ctypes.CDLL(cp.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_binding_names_match_abi(cp):
    for n in _declared():
        assert callable(getattr(cp, n)), n


def test_local_tokens(cp):
    assert cp.cp_local_tokens("dcs", 132, 2) == 66
    assert cp.cp_local_tokens("nlb", 131072, 16) == 8192
    assert cp.cp_local_tokens("mirrored", 128, 2) == 64
    with pytest.raises(cp.CpthdError) as e:
        cp.cp_local_tokens("mirrored", 132, 4)      # divisible by 4, not by 8
    assert e.value.status == -2
    with pytest.raises(cp.CpthdError) as e:
        cp.cp_local_tokens("nlb", 130, 4)
    assert e.value.status == -2
    with pytest.raises(cp.CpthdError) as e:
        cp.cp_local_tokens("nlb", 128, 0)
    assert e.value.status == -1
    with pytest.raises(cp.CpthdError):
        cp.cp_local_tokens(7, 128, 2)


def test_status_strings(cp):
    for s in range(0, -10, -1):
        assert cp.cpthd_status_string(s) not in ("", "unknown status")
    assert cp.cpthd_status_string(-99) == "unknown status"


def test_host_validation_launches_nothing(cp):
    L = cp.lib
    st = cp._i32
    # rank out of range, bad cp_size, null offsets: rejected on the host
    assert L.cp_partition_index(0, ctypes.c_void_p(16), 1, 8, 2, 5, ctypes.c_void_p(16), None, None) == -1
    assert L.cp_partition_index(0, None, 1, 8, 2, 0, ctypes.c_void_p(16), None, None) == -1
    assert L.cp_partition_index(1, ctypes.c_void_p(16), 1, 9, 2, 0, ctypes.c_void_p(16), None, None) == -2
    # reorder: too many tensors, negative rows
    assert L.cp_reorder(ctypes.c_void_p(16), -1, 16, ctypes.c_void_p(16), 4, ctypes.c_void_p(16), None, None) == -1
    # fused partition + gather: rank out of range, NLB with T % cp != 0, missing index output
    vp = ctypes.c_void_p
    srcs = (vp * 1)(vp(16)); dsts = (vp * 1)(vp(16)); rb = (ctypes.c_int64 * 1)(16)
    pr = L.cp_partition_reorder_multi
    assert pr(0, vp(16), 1, 8, 2, 2, 1, srcs, dsts, rb, vp(16), None, None) == -1
    assert pr(1, vp(16), 1, 9, 2, 0, 1, srcs, dsts, rb, vp(16), None, None) == -2
    assert pr(1, vp(16), 1, 8, 2, 0, 1, srcs, dsts, rb, None, None, None) == -1
    assert pr(0, None, 1, 8, 2, 0, 1, srcs, dsts, rb, vp(16), None, None) == -1
    # attention: unsupported head dim, GQA mismatch, missing workspace
    f = L.thd_causal_attn_fwd
    p = ctypes.c_void_p(256)
    assert f(p, 4, p, p, p, 8, p, None, 1, 2, 2, 96, 0.0, p, p, p, 1 << 20, None, None) == -3
    assert f(p, 4, p, p, p, 8, p, None, 1, 3, 2, 64, 0.0, p, p, p, 1 << 20, None, None) == -3
    assert f(p, 4, p, p, p, 8, p, None, 1, 2, 2, 64, 0.0, p, p, None, 0, None, None) == -4
    # plan / planned run: same host checks as the one-call forward
    pl = L.thd_causal_attn_plan
    assert pl(p, 4, 8, p, None, 1, 3, 2, p, 1 << 20, None, None) == -3        # GQA mismatch
    assert pl(p, 4, 8, p, None, 1, 2, 2, None, 0, None, None) == -4           # missing workspace
    assert pl(p, 4, 8, None, None, 1, 2, 2, p, 1 << 20, None, None) == -1     # missing offsets
    assert pl(p, 4, 8, p, None, 1, 2, 2, vp(260), 1 << 20, None, None) == -4  # workspace not 256-B aligned
    assert pl(None, 0, 8, None, None, 1, 2, 2, None, 0, None, None) == 0
    fp = L.thd_causal_attn_fwd_planned
    assert fp(4, p, p, p, 8, 2, 2, 96, 0.0, p, p, p, 1 << 20, None, None) == -3
    assert fp(4, p, p, p, 8, 2, 2, 64, 0.0, p, p, None, 0, None, None) == -4
    assert fp(4, vp(264), p, p, 8, 2, 2, 64, 0.0, p, p, p, 1 << 20, None, None) == -3  # q not 16-B aligned
    assert fp(4, p, None, p, 8, 2, 2, 64, 0.0, p, p, p, 1 << 20, None, None) == -1
    assert fp(0, None, None, None, 8, 2, 2, 64, 0.0, None, None, None, 0, None, None) == 0
    # plan from the partition formulas: rank out of range, T not divisible,
    # GQA mismatch, missing workspace, missing offsets; T = 0 is empty
    pp = L.thd_causal_attn_plan_partition
    assert pp(0, 8, p, p, 1, 2, 2, 2, 2, p, 1 << 20, None, None) == -1
    assert pp(1, 9, p, p, 1, 2, 0, 2, 2, p, 1 << 20, None, None) == -2
    assert pp(0, 8, p, p, 1, 2, 0, 3, 2, p, 1 << 20, None, None) == -3
    assert pp(0, 8, p, p, 1, 2, 0, 2, 2, None, 0, None, None) == -4
    assert pp(0, 8, None, None, 1, 2, 0, 2, 2, p, 1 << 20, None, None) == -1
    assert pp(7, 8, p, p, 1, 2, 0, 2, 2, p, 1 << 20, None, None) == -1
    assert pp(0, 0, None, None, 1, 2, 0, 2, 2, None, 0, None, None) == 0
    # empty slice: nothing to do
    assert f(None, 0, None, None, None, 8, None, None, 1, 2, 2, 64, 0.0, None, None, None, 0, None, None) == 0


def test_workspace_size(cp):
    a = cp.thd_causal_attn_workspace_size(128, 8, 8, 128)
    b = cp.thd_causal_attn_workspace_size(257, 8, 8, 128)      # 256-row groups (one head, two row tiles)
    c = cp.thd_causal_attn_workspace_size(128, 32, 8, 128)     # 128-row groups (two heads, one row tile)
    e = cp.thd_causal_attn_workspace_size(129, 32, 8, 128)
    assert 0 < a < b and 0 < c < e
    assert cp.thd_causal_attn_workspace_size(0, 8, 8, 128) >= 0


def test_host_validation_restore_multi_reorder_backward(cp):
    """Host checks of the remaining entry points: each call returns its
    status before any launch or device call (no GPU needed)."""
    L = cp.lib
    vp = ctypes.c_void_p
    p = vp(256)
    # restore index: T not divisible, negative document count, missing offsets / output
    assert L.cp_restore_index(1, p, 1, 9, 2, p, None, None) == -2
    assert L.cp_restore_index(0, p, -1, 8, 2, p, None, None) == -1
    assert L.cp_restore_index(0, None, 1, 8, 2, p, None, None) == -1
    assert L.cp_restore_index(0, p, 1, 8, 2, None, None, None) == -1
    # multi-tensor gather: tensor count out of [1, 8], missing arrays, negative row width,
    # missing index list while rows are to be copied
    srcs = (vp * 9)(*([p] * 9)); dsts = (vp * 9)(*([p] * 9)); rb = (ctypes.c_int64 * 9)(*([16] * 9))
    rm = L.cp_reorder_multi
    assert rm(0, srcs, dsts, rb, 8, p, 4, None, None) == -1
    assert rm(9, srcs, dsts, rb, 8, p, 4, None, None) == -1
    assert rm(1, None, dsts, rb, 8, p, 4, None, None) == -1
    neg = (ctypes.c_int64 * 1)(-16)
    assert rm(1, srcs, dsts, neg, 8, p, 4, None, None) == -1
    assert rm(1, srcs, dsts, rb, 8, None, 4, None, None) == -1
    assert rm(1, srcs, dsts, rb, 8, p, 0, None, None) == 0  # nothing to gather
    # backward: negative rows, head dim, GQA mismatch, too many query tiles, missing dK/dV
    bw = L.thd_causal_attn_bwd
    args = lambda t_local, hq, hkv, d, dk: (p, t_local, p, p, p, p, p, p, 8, p, None, 1, hq, hkv, d, 0.0, p, dk, p,
                                             p, 1 << 20, None, None)
    assert bw(*args(-1, 2, 2, 64, p)) == -1
    assert bw(*args(4, 2, 2, 96, p)) == -3
    assert bw(*args(4, 3, 2, 64, p)) == -3
    assert bw(*args(2048 * 128 + 1, 2, 2, 64, p)) == -3
    assert bw(*args(4, 2, 2, 64, None)) == -1
    # every host check returns before dK/dV are zeroed: a misaligned pointer or
    # a missing workspace is reported with nothing queued on the stream (the
    # fake pointers here would fault if a memset were queued on them)
    mis = lambda t_local, q, ws, nbytes: (p, t_local, q, p, p, p, p, p, 8, p, None, 1, 2, 2, 64, 0.0, p, p, p, ws,
                                          nbytes, None, None)
    assert bw(*mis(4, vp(264), p, 1 << 20)) == -3
    assert bw(*mis(4, p, None, 0, )) == -4
    assert bw(*mis(4, p, vp(260), 1 << 20)) == -4
    assert bw(*mis(4, p, p, 16)) == -4
    size = ctypes.c_size_t(0)
    assert L.thd_causal_attn_bwd_workspace_size(-1, 2, 2, 64, ctypes.byref(size)) == -1
    assert L.thd_causal_attn_bwd_workspace_size(256, 2, 2, 64, ctypes.byref(size)) == 0 and size.value > 0
