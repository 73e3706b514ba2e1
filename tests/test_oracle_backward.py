"""Pins for the backward oracle (no GPU): central finite differences of
sum(dout * out) through the forward oracle; autograd through torch's float64
scaled_dot_product_attention(is_causal=True) for one document with
cp_size 1; and the CP decomposition -- per-rank dQ scattered back and per-rank
dK/dV summed equal the cp_size 1 gradients."""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import partition as P
import workloads as W


def _loss(q, k, v, lay, idx, dout, scale):
    out, _ = A.attention_fwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, scale=scale)
    return float((out * dout).sum())


def test_finite_differences():
    rng = np.random.default_rng(0)
    lay = W.make_layout([3, 4], 2)          # pads included (padded lengths 4, 4)
    T = lay.T; hq, hkv, d = 4, 2, 3
    q = rng.standard_normal((T, hq, d)); k = rng.standard_normal((T, hkv, d)); v = rng.standard_normal((T, hkv, d))
    idx = np.arange(T)
    dout = rng.standard_normal((T, hq, d))
    dq, dk, dv = A.attention_bwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout, scale=0.8)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            xp = x.copy(); xp[pos] += eps
            xm = x.copy(); xm[pos] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], lay, idx, dout, 0.8)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], lay, idx, dout, 0.8)
            num[pos] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=2e-7, err_msg=name)


@pytest.mark.parametrize("S", [1, 9, 130])
def test_single_doc_matches_sdpa_autograd(S):
    rng = np.random.default_rng(S)
    d = 16
    q = torch.tensor(rng.standard_normal((S, 2, d)), requires_grad=True)
    k = torch.tensor(rng.standard_normal((S, 2, d)), requires_grad=True)
    v = torch.tensor(rng.standard_normal((S, 2, d)), requires_grad=True)
    dout = rng.standard_normal((S, 2, d))
    out = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None], v.permute(1, 0, 2)[None], is_causal=True)
    out = out[0].permute(1, 0, 2)
    (out * torch.tensor(dout)).sum().backward()
    dq, dk, dv = A.attention_bwd(q.detach(), k.detach(), v.detach(), [0, S], [0, S], np.arange(S), dout)
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("strategy", ["dcs", "nlb", "mirrored"])
def test_cp_decomposition(strategy):
    cfg = W.CONFIG_BY_NAME["tiny"]
    inp = W.make_attn_inputs(cfg, strategy)
    lay = inp.layout
    T = lay.T
    rng = np.random.default_rng(5)
    dout_full = rng.standard_normal((T, cfg.hq, cfg.d))
    fq, fk, fv = A.attention_bwd(inp.q, inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded, np.arange(T), dout_full)
    dq = np.zeros_like(fq); dk = np.zeros_like(fk); dv = np.zeros_like(fv)
    for r in range(cfg.cp):
        idx = np.asarray(P.partition_index(strategy, lay.cu_seqlens_padded.tolist(), cfg.cp, r))
        q_r, k_r, v_r = A.attention_bwd(inp.q[torch.from_numpy(idx)], inp.k, inp.v, lay.cu_seqlens,
                                        lay.cu_seqlens_padded, idx, dout_full[idx])
        dq[idx] = q_r
        dk += k_r
        dv += v_r
    np.testing.assert_allclose(dq, fq, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk, fk, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv, fv, rtol=0, atol=1e-10)
