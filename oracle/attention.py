"""Causal packed-THD attention oracle, float64.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

What is computed (TransformerEngine PR #3221): causal self-attention without a
sliding window, window_size=(-1, 0) ("Scope and constraints"), over a THD
buffer whose documents stay isolated through cu_seqlens / cu_seqlens_padded
("What changed": logical document boundaries are preserved through THD
metadata). One rank's query slice (the rows ``idx`` of the physical buffer,
as produced by either partition) attends to the full K/V buffer, which is
what the all-gather of K/V over cp_group gives every rank.

For a local row i with physical index p = idx[i]:
  j    = the document with cu_seqlens_padded[j] <= p < cu_seqlens_padded[j+1]
  pos  = p - cu_seqlens_padded[j]
  the row is a pad slot when pos >= L_j = cu_seqlens[j+1] - cu_seqlens[j]
  keys = physical slots cu_seqlens_padded[j] + u for u = 0..pos
  s_u  = scale * <q[i, h], k[key_u, h // (Hq/Hkv)]>
  lse  = ln sum_u exp(s_u)
  out  = sum_u exp(s_u - lse) * v[key_u, h // (Hq/Hkv)]

Readings where the pages are silent: scale defaults to 1/sqrt(d); query head h
uses KV head h // (Hq/Hkv); LSE is the natural logarithm, laid out
[Hq, rows]; a pad row has out = 0 and lse = -inf. Inputs are bf16 values
converted exactly to float64.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


def _f64(x) -> np.ndarray:
    """bf16/fp32 torch tensor or numpy array -> float64 numpy (exact)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", dtype=torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def locate_rows(idx, cu_seqlens, cu_seqlens_padded):
    """Per local row: document j, position pos, and whether the row is a real
    token (pos < L_j) or a pad slot."""
    idx = np.asarray(idx, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cup = np.asarray(cu_seqlens_padded, dtype=np.int64)
    j = np.searchsorted(cup, idx, side="right") - 1
    pos = idx - cup[j]
    L = cu[1:] - cu[:-1]
    valid = pos < L[j]
    return j, pos, valid


def attention_fwd(q_local, k, v, cu_seqlens, cu_seqlens_padded, idx,
                  scale: Optional[float] = None, rows: Optional[Sequence[int]] = None,
                  block_rows: int = 1024):
    """Oracle forward for one rank's query slice.

    q_local: [T_loc, Hq, d]; k, v: [T, Hkv, d]; idx: the rank's physical
    indices [T_loc]. ``rows`` optionally selects a subset of local rows.
    Returns (out [n, Hq, d] float64, lse [Hq, n] float64) for the selected rows
    in the order given.
    """
    Q = _f64(q_local)
    K = _f64(k)
    V = _f64(v)
    idx = np.asarray(idx, dtype=np.int64)
    Hq, d = Q.shape[1], Q.shape[2]
    Hkv = K.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    sel = np.arange(idx.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    n = sel.shape[0]
    out = np.zeros((n, Hq, d), dtype=np.float64)
    lse = np.full((Hq, n), -np.inf, dtype=np.float64)
    if n == 0:
        return out, lse
    cup = np.asarray(cu_seqlens_padded, dtype=np.int64)
    j, pos, valid = locate_rows(idx[sel], cu_seqlens, cu_seqlens_padded)

    for doc in np.unique(j[valid]):
        members = np.nonzero(valid & (j == doc))[0]          # positions within ``sel``
        start = int(cup[doc])
        for b0 in range(0, members.shape[0], block_rows):
            mb = members[b0:b0 + block_rows]
            p = pos[mb]                                        # [m]
            nk = int(p.max()) + 1
            keys = np.arange(nk)
            allowed = keys[None, :] <= p[:, None]              # causal within the document
            for h in range(Hq):
                kvh = h // g
                qh = Q[sel[mb], h, :]                          # [m, d]
                kh = K[start:start + nk, kvh, :]               # [nk, d]
                vh = V[start:start + nk, kvh, :]
                s = scale * (qh @ kh.T)                        # [m, nk]
                s = np.where(allowed, s, -np.inf)
                mx = s.max(axis=1, keepdims=True)
                e = np.exp(s - mx)
                z = e.sum(axis=1, keepdims=True)
                lse[h, mb] = (mx + np.log(z))[:, 0]
                out[mb, h, :] = (e / z) @ vh
    return out, lse


def attention_bruteforce(q_local, k, v, cu_seqlens, cu_seqlens_padded, idx, scale: Optional[float] = None):
    """Per-pair scalar loops over the definition, for tiny inputs only."""
    Q = _f64(q_local).tolist()
    K = _f64(k).tolist()
    V = _f64(v).tolist()
    cu = [int(x) for x in cu_seqlens]
    cup = [int(x) for x in cu_seqlens_padded]
    T_loc = len(Q)
    Hq = len(Q[0]) if T_loc else 0
    d = len(Q[0][0]) if T_loc else 0
    Hkv = len(K[0]) if K else 1
    g = Hq // Hkv if Hkv else 1
    if scale is None:
        scale = 1.0 / math.sqrt(d) if d else 1.0
    out = [[[0.0] * d for _ in range(Hq)] for _ in range(T_loc)]
    lse = [[-math.inf] * T_loc for _ in range(Hq)]
    for i in range(T_loc):
        p = int(idx[i])
        doc = None
        for jj in range(len(cup) - 1):
            if cup[jj] <= p < cup[jj + 1]:
                doc = jj
                break
        if doc is None:
            raise IndexError("index outside the buffer")
        pos = p - cup[doc]
        if pos >= cu[doc + 1] - cu[doc]:
            continue                                           # pad row
        for h in range(Hq):
            kvh = h // g
            s = []
            for u in range(pos + 1):
                key = cup[doc] + u
                acc = 0.0
                for e in range(d):
                    acc += Q[i][h][e] * K[key][kvh][e]
                s.append(scale * acc)
            mx = max(s)
            z = 0.0
            for su in s:
                z += math.exp(su - mx)
            l = mx + math.log(z)
            lse[h][i] = l
            for e in range(d):
                acc = 0.0
                for u in range(pos + 1):
                    acc += math.exp(s[u] - l) * V[cup[doc] + u][kvh][e]
                out[i][h][e] = acc
    return np.array(out, dtype=np.float64).reshape(T_loc, Hq, d), np.array(lse, dtype=np.float64).reshape(Hq, T_loc)


def unmasked_pairs(idx, cu_seqlens, cu_seqlens_padded) -> int:
    """Number of allowed (query, key) pairs of a query slice, per head:
    sum over real rows of (pos + 1)."""
    j, pos, valid = locate_rows(idx, cu_seqlens, cu_seqlens_padded)
    return int((pos[valid] + 1).sum())


def attention_bwd(q_local, k, v, cu_seqlens, cu_seqlens_padded, idx, dout, scale: Optional[float] = None,
                  block_rows: int = 1024):
    """Oracle backward of ``attention_fwd`` for one rank's query slice.

    The forward is recomputed here in float64 (out and lse from the
    definition), then, for every allowed pair (i, u) of a row i with keys u:
      P    = exp(s - lse_i)
      D_i  = <dout_i, out_i>
      dV_u += P dout_i
      dS   = P (<dout_i, v_u> - D_i)
      dQ_i += scale dS k_u,   dK_u += scale dS q_i
    (the gradients of sum(dout * out) with respect to q, k, v). K/V heads
    collect the gradients of every query head of their group. dK and dV cover
    the whole buffer [T, Hkv, d] and hold this rank's contribution only (the
    part a reduce-scatter over CP ranks would sum; TE PR: backward reuses the
    forward's layout).
    Returns (dq [T_loc, Hq, d], dk [T, Hkv, d], dv [T, Hkv, d]) float64.
    """
    Q = _f64(q_local)
    K = _f64(k)
    V = _f64(v)
    dO = _f64(dout)
    idx = np.asarray(idx, dtype=np.int64)
    T_loc, Hq, d = Q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.zeros_like(Q)
    dk = np.zeros_like(K)
    dv = np.zeros_like(V)
    if T_loc == 0:
        return dq, dk, dv
    cup = np.asarray(cu_seqlens_padded, dtype=np.int64)
    j, pos, valid = locate_rows(idx, cu_seqlens, cu_seqlens_padded)
    for doc in np.unique(j[valid]):
        members = np.nonzero(valid & (j == doc))[0]
        start = int(cup[doc])
        for b0 in range(0, members.shape[0], block_rows):
            mb = members[b0:b0 + block_rows]
            p = pos[mb]
            nk = int(p.max()) + 1
            allowed = np.arange(nk)[None, :] <= p[:, None]
            for h in range(Hq):
                kvh = h // g
                qh = Q[mb, h, :]
                kh = K[start:start + nk, kvh, :]
                vh = V[start:start + nk, kvh, :]
                doh = dO[mb, h, :]
                s = scale * (qh @ kh.T)
                s = np.where(allowed, s, -np.inf)
                mx = s.max(axis=1, keepdims=True)
                e = np.exp(s - mx)
                P = e / e.sum(axis=1, keepdims=True)                 # exp(s - lse)
                out = P @ vh
                D = (doh * out).sum(axis=1, keepdims=True)
                dP = doh @ vh.T
                dS = P * (dP - D)                                   # zero where not allowed (P = 0)
                dq[mb, h, :] += scale * (dS @ kh)
                dk[start:start + nk, kvh, :] += scale * (dS.T @ qh)
                dv[start:start + nk, kvh, :] += P.T @ doh
    return dq, dk, dv
