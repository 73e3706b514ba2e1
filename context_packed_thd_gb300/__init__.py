"""Python binding of libcpthd (context-parallel causal attention over packed THD).

The functions keep the C ABI's names (include/cpthd.h) and only marshal
arguments: torch tensors in, device pointers and the current CUDA stream out.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback. Importing the package builds libcpthd.so in-tree when
it is missing or stale (nvcc, sm_103a) and fails loudly when it cannot.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

__all__ = [
    "DUAL_CHUNK_SWAP", "NO_LOAD_BALANCE", "PACKED_MIRRORED", "CpthdError", "LIB_PATH", "lib",
    "cpthd_status_string", "cp_local_tokens", "cp_partition_index", "cp_restore_index", "cp_reorder",
    "cp_reorder_multi",
    "cp_partition_reorder_multi",
    "thd_causal_attn_workspace_size", "thd_causal_attn_fwd", "thd_causal_attn_plan", "thd_causal_attn_fwd_planned",
    "thd_causal_attn_plan_partition",
    "thd_causal_attn_fwd_static_scratch",
    "thd_causal_attn_bwd_workspace_size", "thd_causal_attn_bwd",
    "get_batch_on_this_cp_rank", "strategy_code",
]

DUAL_CHUNK_SWAP = 0
NO_LOAD_BALANCE = 1
PACKED_MIRRORED = 2

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcpthd.so")


def _load_library():
    """Load libcpthd.so, building it in-tree with nvcc on first use. There is
    no fallback: without the library (or nvcc to build it) the import fails."""
    from . import build as _build
    try:
        _build.build()
    except _build.NvccMissing as e:  # a prebuilt library may still be there
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libcpthd.so is missing and could not be built: {e}") from e
    except RuntimeError as e:       # a compile or link error never falls back to a stale library
        raise ImportError(f"building libcpthd.so failed: {e}") from e
    return ctypes.CDLL(LIB_PATH)


lib = _load_library()

_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

lib.cpthd_status_string.argtypes = [_i32]
lib.cpthd_status_string.restype = ctypes.c_char_p
lib.cp_local_tokens.argtypes = [_i32, _i64, _i32, ctypes.POINTER(_i64)]
lib.cp_local_tokens.restype = _i32
lib.cp_partition_index.argtypes = [_i32, _vp, _i32, _i64, _i32, _i32, _vp, _vp, _vp]
lib.cp_partition_index.restype = _i32
lib.cp_restore_index.argtypes = [_i32, _vp, _i32, _i64, _i32, _vp, _vp, _vp]
lib.cp_restore_index.restype = _i32
lib.cp_reorder.argtypes = [_vp, _i64, _i64, _vp, _i64, _vp, _vp, _vp]
lib.cp_reorder.restype = _i32
lib.cp_reorder_multi.argtypes = [_i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_i64), _i64, _vp,
                                 _i64, _vp, _vp]
lib.cp_reorder_multi.restype = _i32
lib.cp_partition_reorder_multi.argtypes = [_i32, _vp, _i32, _i64, _i32, _i32, _i32, ctypes.POINTER(_vp),
                                           ctypes.POINTER(_vp), ctypes.POINTER(_i64), _vp, _vp, _vp]
lib.cp_partition_reorder_multi.restype = _i32
lib.thd_causal_attn_workspace_size.argtypes = [_i64, _i32, _i32, _i32, ctypes.POINTER(_sz)]
lib.thd_causal_attn_workspace_size.restype = _i32
lib.thd_causal_attn_fwd.argtypes = [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32, _f32, _vp,
                                    _vp, _vp, _sz, _vp, _vp]
lib.thd_causal_attn_fwd.restype = _i32
lib.thd_causal_attn_plan.argtypes = [_vp, _i64, _i64, _vp, _vp, _i32, _i32, _i32, _vp, _sz, _vp, _vp]
lib.thd_causal_attn_plan.restype = _i32
lib.thd_causal_attn_fwd_planned.argtypes = [_i64, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _sz,
                                            _vp, _vp]
lib.thd_causal_attn_fwd_planned.restype = _i32
lib.thd_causal_attn_plan_partition.argtypes = [_i32, _i64, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _sz, _vp,
                                               _vp]
lib.thd_causal_attn_plan_partition.restype = _i32
lib.thd_causal_attn_bwd_workspace_size.argtypes = [_i64, _i32, _i32, _i32, ctypes.POINTER(_sz)]
lib.thd_causal_attn_bwd_workspace_size.restype = _i32
lib.thd_causal_attn_bwd.argtypes = [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32,
                                    _f32, _vp, _vp, _vp, _vp, _sz, _vp, _vp]
lib.thd_causal_attn_bwd.restype = _i32
lib.thd_causal_attn_fwd_static_scratch.argtypes = [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32,
                                                   _f32, _vp, _vp, _vp, _vp]
lib.thd_causal_attn_fwd_static_scratch.restype = _i32


class CpthdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {cpthd_status_string(status)} (status {status})")


def cpthd_status_string(status: int) -> str:
    return lib.cpthd_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != 0:
        raise CpthdError(status, where)


def strategy_code(strategy) -> int:
    if isinstance(strategy, str):
        s = strategy.lower()
        if s in ("dcs", "dual_chunk_swap"):
            return DUAL_CHUNK_SWAP
        if s in ("nlb", "no_load_balance"):
            return NO_LOAD_BALANCE
        if s in ("mirrored", "packed_mirrored"):
            return PACKED_MIRRORED
        raise ValueError(f"unknown strategy {strategy!r}")
    return int(strategy)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libcpthd takes CUDA tensors only")


def cp_local_tokens(strategy, T: int, cp_size: int) -> int:
    out = _i64(0)
    _check(lib.cp_local_tokens(strategy_code(strategy), int(T), int(cp_size), ctypes.byref(out)), "cp_local_tokens")
    return int(out.value)


def cp_partition_index(strategy, cu_seqlens_padded: torch.Tensor, T: int, cp_size: int, rank: int,
                       out: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """int32 physical indices owned by ``rank`` (rank = -1: all ranks, rank-major)."""
    _need_cuda(cu_seqlens_padded, out, err)
    assert cu_seqlens_padded.dtype == torch.int32 and cu_seqlens_padded.is_contiguous()
    n = cp_local_tokens(strategy, T, cp_size) * (cp_size if rank < 0 else 1)
    if out is None:
        out = torch.empty(n, dtype=torch.int32, device=cu_seqlens_padded.device)
    assert out.numel() >= n and out.dtype == torch.int32
    _check(lib.cp_partition_index(strategy_code(strategy), _ptr(cu_seqlens_padded), cu_seqlens_padded.numel() - 1,
                                  int(T), int(cp_size), int(rank), _ptr(out), _ptr(err), _stream(stream)),
           "cp_partition_index")
    return out


def cp_restore_index(strategy, cu_seqlens_padded: torch.Tensor, T: int, cp_size: int,
                     out: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """int32 [T]: row of the rank-major all-gathered buffer holding each physical slot."""
    _need_cuda(cu_seqlens_padded, out, err)
    assert cu_seqlens_padded.dtype == torch.int32 and cu_seqlens_padded.is_contiguous()
    if out is None:
        out = torch.empty(int(T), dtype=torch.int32, device=cu_seqlens_padded.device)
    assert out.numel() >= T and out.dtype == torch.int32
    _check(lib.cp_restore_index(strategy_code(strategy), _ptr(cu_seqlens_padded), cu_seqlens_padded.numel() - 1,
                                int(T), int(cp_size), _ptr(out), _ptr(err), _stream(stream)), "cp_restore_index")
    return out


def cp_reorder(src: torch.Tensor, idx: torch.Tensor, out: Optional[torch.Tensor] = None,
               err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[i] = src[idx[i]] along dim 0, bit exact."""
    _need_cuda(src, idx, out, err)
    assert src.is_contiguous() and idx.dtype == torch.int32 and idx.is_contiguous()
    if out is None:
        out = torch.empty((idx.numel(),) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    rb = int(src[0].numel() * src.element_size()) if src.dim() > 1 else src.element_size()
    _check(lib.cp_reorder(_ptr(src), src.shape[0], rb, _ptr(idx), idx.numel(), _ptr(out), _ptr(err),
                          _stream(stream)), "cp_reorder")
    return out


def cp_reorder_multi(srcs: Sequence[torch.Tensor], idx: torch.Tensor, outs=None,
                     err: Optional[torch.Tensor] = None, stream=None):
    """Gather several tensors (same row count) by one index list in one launch."""
    srcs = list(srcs)
    _need_cuda(idx, err, *srcs)
    n = len(srcs)
    rows = srcs[0].shape[0]
    assert all(s.shape[0] == rows and s.is_contiguous() for s in srcs)
    if outs is None:
        outs = [torch.empty((idx.numel(),) + tuple(s.shape[1:]), dtype=s.dtype, device=s.device) for s in srcs]
    sp = (_vp * n)(*[s.data_ptr() for s in srcs])
    dp = (_vp * n)(*[o.data_ptr() for o in outs])
    rb = (_i64 * n)(*[int(s[0].numel() * s.element_size()) if s.dim() > 1 else s.element_size() for s in srcs])
    _check(lib.cp_reorder_multi(n, sp, dp, rb, rows, _ptr(idx), idx.numel(), _ptr(err), _stream(stream)),
           "cp_reorder_multi")
    return outs


def cp_partition_reorder_multi(strategy, cu_seqlens_padded: torch.Tensor, T: int, cp_size: int, rank: int,
                               srcs: Sequence[torch.Tensor], outs=None, idx_out: Optional[torch.Tensor] = None,
                               err: Optional[torch.Tensor] = None, stream=None):
    """The rank's partition index and every tensor of ``srcs`` (T rows each)
    gathered by it, in one launch. Returns (idx int32 [T/cp_size], outs)."""
    srcs = list(srcs)
    _need_cuda(cu_seqlens_padded, idx_out, err, *srcs)
    assert cu_seqlens_padded.dtype == torch.int32 and cu_seqlens_padded.is_contiguous()
    assert all(s.shape[0] == T and s.is_contiguous() for s in srcs)
    n_loc = cp_local_tokens(strategy, T, cp_size)
    if idx_out is None:
        idx_out = torch.empty(n_loc, dtype=torch.int32, device=cu_seqlens_padded.device)
    assert idx_out.numel() >= n_loc and idx_out.dtype == torch.int32
    if outs is None:
        outs = [torch.empty((n_loc,) + tuple(s.shape[1:]), dtype=s.dtype, device=s.device) for s in srcs]
    n = len(srcs)
    sp = (_vp * n)(*[s.data_ptr() for s in srcs])
    dp = (_vp * n)(*[o.data_ptr() for o in outs])
    rb = (_i64 * n)(*[int(s[0].numel() * s.element_size()) if s.dim() > 1 else s.element_size() for s in srcs])
    _check(lib.cp_partition_reorder_multi(strategy_code(strategy), _ptr(cu_seqlens_padded),
                                          cu_seqlens_padded.numel() - 1, int(T), int(cp_size), int(rank), n, sp, dp,
                                          rb, _ptr(idx_out), _ptr(err), _stream(stream)),
           "cp_partition_reorder_multi")
    return idx_out, outs


def thd_causal_attn_workspace_size(t_local: int, Hq: int, Hkv: int, d: int) -> int:
    out = _sz(0)
    _check(lib.thd_causal_attn_workspace_size(int(t_local), int(Hq), int(Hkv), int(d), ctypes.byref(out)),
           "thd_causal_attn_workspace_size")
    return int(out.value)


def thd_causal_attn_fwd(q_slice_idx: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        cu_seqlens: torch.Tensor, cu_seqlens_padded: Optional[torch.Tensor] = None,
                        softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                        lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        err: Optional[torch.Tensor] = None, stream=None):
    """Causal THD attention of a rank's query slice q [t_local, Hq, d] against
    the full k, v [T, Hkv, d]. Returns (out bf16 [t_local, Hq, d], lse fp32 [Hq, t_local])."""
    _need_cuda(q_slice_idx, q, k, v, cu_seqlens, cu_seqlens_padded, out, lse, workspace, err)
    t_local, Hq, d = q.shape
    T, Hkv, _ = k.shape
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16 and t.is_contiguous()
    assert q_slice_idx.dtype == torch.int32 and q_slice_idx.numel() == t_local
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, t_local), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(thd_causal_attn_workspace_size(t_local, Hq, Hkv, d), dtype=torch.uint8,
                                device=q.device)
    _check(lib.thd_causal_attn_fwd(_ptr(q_slice_idx), t_local, _ptr(q), _ptr(k), _ptr(v), T, _ptr(cu_seqlens),
                                   _ptr(cu_seqlens_padded), cu_seqlens.numel() - 1, Hq, Hkv, d,
                                   float(softmax_scale) if softmax_scale else 0.0, _ptr(out), _ptr(lse),
                                   _ptr(workspace), workspace.numel(), _ptr(err), _stream(stream)),
           "thd_causal_attn_fwd")
    return out, lse


def thd_causal_attn_plan(q_slice_idx: torch.Tensor, T: int, cu_seqlens: torch.Tensor,
                         cu_seqlens_padded: Optional[torch.Tensor], Hq: int, Hkv: int,
                         workspace: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None, stream=None):
    """Row-group metadata of a query slice (the first half of
    thd_causal_attn_fwd). Returns the workspace holding the plan; pass it to
    thd_causal_attn_fwd_planned for every attention over this slice."""
    _need_cuda(q_slice_idx, cu_seqlens, cu_seqlens_padded, workspace, err)
    assert q_slice_idx.dtype == torch.int32
    t_local = q_slice_idx.numel()
    if workspace is None:
        workspace = torch.empty(thd_causal_attn_workspace_size(t_local, Hq, Hkv, 128), dtype=torch.uint8,
                                device=q_slice_idx.device)
    _check(lib.thd_causal_attn_plan(_ptr(q_slice_idx), t_local, int(T), _ptr(cu_seqlens), _ptr(cu_seqlens_padded),
                                    cu_seqlens.numel() - 1, int(Hq), int(Hkv), _ptr(workspace), workspace.numel(),
                                    _ptr(err), _stream(stream)), "thd_causal_attn_plan")
    return workspace


def thd_causal_attn_plan_partition(strategy, T: int, cu_seqlens: torch.Tensor,
                                   cu_seqlens_padded: Optional[torch.Tensor], cp_size: int, rank: int, Hq: int,
                                   Hkv: int, workspace: Optional[torch.Tensor] = None,
                                   err: Optional[torch.Tensor] = None, stream=None):
    """The plan of rank ``rank``'s slice under ``strategy`` with the row slots
    computed from the partition formulas (no index list needed). Returns the
    workspace, as thd_causal_attn_plan does for the same slice."""
    _need_cuda(cu_seqlens, cu_seqlens_padded, workspace, err)
    code = strategy_code(strategy)
    t_local = cp_local_tokens(code, T, cp_size)
    if workspace is None:
        workspace = torch.empty(thd_causal_attn_workspace_size(t_local, Hq, Hkv, 128), dtype=torch.uint8,
                                device=cu_seqlens.device)
    _check(lib.thd_causal_attn_plan_partition(code, int(T), _ptr(cu_seqlens), _ptr(cu_seqlens_padded),
                                              cu_seqlens.numel() - 1, int(cp_size), int(rank), int(Hq), int(Hkv),
                                              _ptr(workspace), workspace.numel(), _ptr(err), _stream(stream)),
           "thd_causal_attn_plan_partition")
    return workspace


def thd_causal_attn_fwd_planned(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, workspace: torch.Tensor,
                                softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                                lse: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None,
                                stream=None):
    """The attention kernel alone, against a plan written by
    thd_causal_attn_plan for the same slice, T, Hq and Hkv. Returns
    (out bf16 [t_local, Hq, d], lse fp32 [Hq, t_local])."""
    _need_cuda(q, k, v, workspace, out, lse, err)
    t_local, Hq, d = q.shape
    T, Hkv, _ = k.shape
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16 and t.is_contiguous()
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, t_local), dtype=torch.float32, device=q.device)
    _check(lib.thd_causal_attn_fwd_planned(t_local, _ptr(q), _ptr(k), _ptr(v), T, Hq, Hkv, d,
                                           float(softmax_scale) if softmax_scale else 0.0, _ptr(out), _ptr(lse),
                                           _ptr(workspace), workspace.numel(), _ptr(err), _stream(stream)),
           "thd_causal_attn_fwd_planned")
    return out, lse


def thd_causal_attn_fwd_static_scratch(q_slice_idx: torch.Tensor, q: torch.Tensor, k: torch.Tensor,
                                       v: torch.Tensor, cu_seqlens: torch.Tensor,
                                       cu_seqlens_padded: Optional[torch.Tensor] = None,
                                       softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                                       lse: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None,
                                       stream=None):
    """thd_causal_attn_fwd for callers that cannot allocate device memory: the
    library's built-in scratch array replaces the workspace. Pass ``out`` and
    ``lse`` to keep the call itself free of allocations (when they are None
    this convenience wrapper creates them with torch)."""
    _need_cuda(q_slice_idx, q, k, v, cu_seqlens, cu_seqlens_padded, out, lse, err)
    t_local, Hq, d = q.shape
    T, Hkv, _ = k.shape
    for t in (q, k, v):
        assert t.dtype == torch.bfloat16 and t.is_contiguous()
    assert q_slice_idx.dtype == torch.int32 and q_slice_idx.numel() == t_local
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, t_local), dtype=torch.float32, device=q.device)
    _check(lib.thd_causal_attn_fwd_static_scratch(
        _ptr(q_slice_idx), t_local, _ptr(q), _ptr(k), _ptr(v), T, _ptr(cu_seqlens), _ptr(cu_seqlens_padded),
        cu_seqlens.numel() - 1, Hq, Hkv, d, float(softmax_scale) if softmax_scale else 0.0, _ptr(out), _ptr(lse),
        _ptr(err), _stream(stream)), "thd_causal_attn_fwd_static_scratch")
    return out, lse


def thd_causal_attn_bwd_workspace_size(t_local: int, Hq: int, Hkv: int, d: int) -> int:
    out = _sz(0)
    _check(lib.thd_causal_attn_bwd_workspace_size(int(t_local), int(Hq), int(Hkv), int(d), ctypes.byref(out)),
           "thd_causal_attn_bwd_workspace_size")
    return int(out.value)


def thd_causal_attn_bwd(q_slice_idx: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        out: torch.Tensor, dout: torch.Tensor, lse: torch.Tensor, cu_seqlens: torch.Tensor,
                        cu_seqlens_padded: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
                        dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
                        dv: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        err: Optional[torch.Tensor] = None, stream=None):
    """Gradients of sum(dout * out) for a rank's slice. Returns fp32
    (dq [t_local, Hq, d], dk [T, Hkv, d], dv [T, Hkv, d]); dk/dv hold this
    rank's contribution."""
    _need_cuda(q_slice_idx, q, k, v, out, dout, lse, cu_seqlens, cu_seqlens_padded, dq, dk, dv, workspace, err)
    t_local, Hq, d = q.shape
    T, Hkv, _ = k.shape
    for t in (q, k, v, out, dout):
        assert t.dtype == torch.bfloat16 and t.is_contiguous()
    assert lse.dtype == torch.float32 and lse.is_contiguous()
    if dq is None:
        dq = torch.empty((t_local, Hq, d), dtype=torch.float32, device=q.device)
    if dk is None:
        dk = torch.empty((T, Hkv, d), dtype=torch.float32, device=q.device)
    if dv is None:
        dv = torch.empty((T, Hkv, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(thd_causal_attn_bwd_workspace_size(t_local, Hq, Hkv, d), dtype=torch.uint8,
                                device=q.device)
    _check(lib.thd_causal_attn_bwd(_ptr(q_slice_idx), t_local, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout),
                                   _ptr(lse), T, _ptr(cu_seqlens), _ptr(cu_seqlens_padded), cu_seqlens.numel() - 1,
                                   Hq, Hkv, d, float(softmax_scale) if softmax_scale else 0.0, _ptr(dq), _ptr(dk),
                                   _ptr(dv), _ptr(workspace), workspace.numel(), _ptr(err), _stream(stream)),
           "thd_causal_attn_bwd")
    return dq, dk, dv


def get_batch_on_this_cp_rank(cu_seqlens_padded: torch.Tensor, *tensors: torch.Tensor, cp_size: int, rank: int,
                              strategy=DUAL_CHUNK_SWAP, err: Optional[torch.Tensor] = None):
    """Slice THD tensors (input_ids, labels, position_ids, activations ...)
    to ``rank``'s tokens in one reorder launch. Returns (idx, [slices])."""
    T = int(tensors[0].shape[0])
    idx = cp_partition_index(strategy, cu_seqlens_padded, T, cp_size, rank, err=err)
    outs = cp_reorder_multi(tensors, idx, err=err) if tensors else []
    return idx, outs
