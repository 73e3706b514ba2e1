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


def bwd_term_magnitudes(q_local, k, v, cu_seqlens, cu_seqlens_padded, idx, dout, scale=None, block_rows=512):
    """Per-element error scale of the GPU backward (test tolerance helper).

    The GPU rounds three quantities to bf16 on the way to its fp32 gradients:
    P (before dV += P^T dO, and inside dS in the dK/dV pass), dS (before
    dQ += dS K and dK += dS^T Q), and the forward's output O (which gives
    D = rowsum(dO * O)). bf16 keeps 8 significant bits, so each rounding is
    at most 2^-8 relative. Following every term of every gradient through
    those roundings:
      |d dV[k]| <= 2^-8 sum_q P[q,k] |dO[q]|
      |d dS[q,k]| <= 2^-7 |dS[q,k]| + P[q,k] |d D_q|,
      |d D_q| <= 2^-7 sum_e |dO[q,e]| (P |V|)[q,e]        (bf16 P in P V, bf16 O)
      |d dQ[q]| <= scale sum_k |d dS[q,k]| |K[k]|
      |d dK[k]| <= scale sum_q |d dS[q,k]| |Q[q]|
    This returns M_q, M_k, M_v with |error| <= 2^-7 M elementwise (the fp32
    accumulations and ex2.approx add terms orders of magnitude below):
      M_v = P^T |dO|,
      M_q = scale (|dS| |K| + e_D * P |K|),   M_k = scale (|dS|^T |Q| + P^T (e_D * |Q|)),
      e_D[q] = sum_e |dO[q,e]| (P |V|)[q,e].
    P and dS are the exact float64 values of the definition (per document,
    causal, max-shifted softmax), as in oracle.attention.attention_bwd."""
    import math
    f64 = lambda t: t.detach().to("cpu", dtype=torch.float64).numpy() if isinstance(t, torch.Tensor) \
        else np.asarray(t, dtype=np.float64)  # noqa: E731
    Q, K, V, dO = f64(q_local), f64(k), f64(v), f64(dout)
    idx = np.asarray(idx, dtype=np.int64)
    hq, d = Q.shape[1], Q.shape[2]
    g = hq // K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    mq, mk, mv = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cup = np.asarray(cu_seqlens_padded, dtype=np.int64)
    j = np.searchsorted(cup, idx, side="right") - 1
    pos = idx - cup[j]
    valid = pos < (cu[1:] - cu[:-1])[j]
    for doc in np.unique(j[valid]):
        members = np.nonzero(valid & (j == doc))[0]
        start = int(cup[doc])
        for b0 in range(0, members.shape[0], block_rows):
            mb = members[b0:b0 + block_rows]
            p = pos[mb]
            nk = int(p.max()) + 1
            allowed = np.arange(nk)[None, :] <= p[:, None]
            for h in range(hq):
                kvh = h // g
                qh, doh = Q[mb, h, :], dO[mb, h, :]
                kh, vh = K[start:start + nk, kvh, :], V[start:start + nk, kvh, :]
                s = np.where(allowed, scale * (qh @ kh.T), -np.inf)
                e = np.exp(s - s.max(axis=1, keepdims=True))
                P = e / e.sum(axis=1, keepdims=True)
                D = (doh * (P @ vh)).sum(axis=1, keepdims=True)
                aS = np.abs(P * (doh @ vh.T - D))
                e_d = (np.abs(doh) * (P @ np.abs(vh))).sum(axis=1, keepdims=True)
                mv[start:start + nk, kvh, :] += P.T @ np.abs(doh)
                mq[mb, h, :] += scale * (aS @ np.abs(kh) + e_d * (P @ np.abs(kh)))
                mk[start:start + nk, kvh, :] += scale * (aS.T @ np.abs(qh) + P.T @ (e_d * np.abs(qh)))
    return mq, mk, mv
