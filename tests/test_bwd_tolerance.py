"""The backward's element-wise tolerance (tests/gpu_common.bwd_term_magnitudes)
checked on the CPU, so that the GPU tests' bound is neither vacuous nor too
tight: the backward is emulated in numpy with the roundings the GPU applies
(P and dS to bf16 before the tensor-core products, the forward's output O to
bf16 before D = rowsum(dO * O)), and

* the emulated gradients stay within BWD_C * M of the float64 oracle;
* the bound is not loose by orders of magnitude (some entry uses a
  noticeable part of it);
* a planted mistake (one key block left out of the sums) breaks it.
"""
import math

import numpy as np
import torch

from oracle import attention as A
import workloads as W
from gpu_common import bwd_term_magnitudes

BWD_C = 2.0 ** -6


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _emulated_bwd(q, k, v, lay, idx, dout, drop_block=None):
    """The GPU's arithmetic, restated with its bf16 roundings (one document
    per pack here, all rows valid)."""
    Q, K, V, dO = (t.double().numpy() for t in (q, k, v, dout))
    T_loc, hq, d = Q.shape
    scale = 1.0 / math.sqrt(d)
    cup = lay.cu_seqlens_padded.astype(np.int64)
    dq, dk, dv = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    j = np.searchsorted(cup, idx, side="right") - 1
    for doc in np.unique(j):
        mb = np.nonzero(j == doc)[0]
        start = int(cup[doc])
        p = idx[mb] - start
        nk = int(p.max()) + 1
        allowed = np.arange(nk)[None, :] <= p[:, None]
        if drop_block is not None:
            allowed[:, drop_block * 128:(drop_block + 1) * 128] = False
        for h in range(hq):
            kvh = h // (hq // K.shape[1])
            qh, doh = Q[mb, h], dO[mb, h]
            kh, vh = K[start:start + nk, kvh], V[start:start + nk, kvh]
            s = np.where(allowed, scale * (qh @ kh.T), -np.inf)
            e = np.exp(s - s.max(axis=1, keepdims=True))
            P = e / e.sum(axis=1, keepdims=True)
            Pb = _bf16(P)
            O = _bf16(Pb @ vh)                           # forward: bf16 P in P V, bf16 output
            D = (doh * O).sum(axis=1, keepdims=True)
            dS = _bf16(Pb * (doh @ vh.T - D))             # dK/dV pass form: P from bf16, dS to bf16
            dq[mb, h] += scale * (dS @ kh)
            dk[start:start + nk, kvh] += scale * (dS.T @ qh)
            dv[start:start + nk, kvh] += Pb.T @ doh
    return dq, dk, dv


def _case():
    lay = W.make_layout([700], 1)
    q, k, v = W.make_qkv_logical(31, 700, 2, 2, 64)
    idx = np.arange(700, dtype=np.int64)
    dout = W.randn_bf16(31, 6, (700, 2, 64))
    return lay, q, k, v, idx, dout


def test_emulated_gpu_roundings_stay_within_bound():
    lay, q, k, v, idx, dout = _case()
    ref = A.attention_bwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
    mag = bwd_term_magnitudes(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
    emu = _emulated_bwd(q, k, v, lay, idx, dout)
    worst = 0.0
    for e, r, m in zip(emu, ref, mag):
        ratio = np.abs(e - r) / (BWD_C * m)
        assert np.all(ratio <= 1.0)
        worst = max(worst, float(ratio.max()))
    # the bound is a worst case; random roundings use part of it, not 1e-4 of it
    assert worst > 0.02, worst


def test_planted_mistake_breaks_bound():
    lay, q, k, v, idx, dout = _case()
    ref = A.attention_bwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
    mag = bwd_term_magnitudes(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
    bad = _emulated_bwd(q, k, v, lay, idx, dout, drop_block=2)
    assert any(np.any(np.abs(e - r) > BWD_C * m) for e, r, m in zip(bad, ref, mag))


def test_magnitudes_bound_the_gradients():
    """|grad| <= M entrywise (M sums the magnitudes of the grad's own terms)."""
    lay, q, k, v, idx, dout = _case()
    ref = A.attention_bwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
    mag = bwd_term_magnitudes(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
    for r, m in zip(ref, mag):
        assert np.all(np.abs(r) <= m * (1 + 1e-12) + 1e-300)
