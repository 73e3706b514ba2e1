"""GPU attention backward (dQ, dK, dV) vs the float64 oracle.

The GPU backward rounds P and dS to bf16 for the tensor cores and uses the
forward's bf16 output for rowsum(dO * O); its results are compared per
tensor with a norm-relative bound: max |x - ref| <= BWD_TOL * max |ref| (the
bf16 rounding of P and dS is 2^-9 relative, and sums over many keys of mixed
sign keep that order relative to the largest entries), plus pad / untouched
entries exactly zero.
"""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import partition as P
import workloads as W
from gpu_common import cuda_or_skip, load_lib, new_err

pytestmark = pytest.mark.gpu
BWD_TOL = 2e-2


def _rank_bwd(cp, inp, strategy, cpsize, r, dev, dout_phys, err):
    lay = inp.layout
    cu = torch.from_numpy(lay.cu_seqlens).to(dev)
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    idx = cp.cp_partition_index(strategy, cup, lay.T, cpsize, r, err=err)
    q_loc = cp.cp_reorder(q, idx, err=err)
    dout = cp.cp_reorder(dout_phys.to(dev), idx, err=err)
    out, lse = cp.thd_causal_attn_fwd(idx, q_loc, k, v, cu, cup, err=err)
    dq, dk, dv = cp.thd_causal_attn_bwd(idx, q_loc, k, v, out, dout, lse, cu, cup, err=err)
    return idx.cpu().numpy().astype(np.int64), dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy(), dout.cpu()


def _structural_zero(lay, idx):
    """Rows of dq that are pad slots, and keys of dk/dv no query of the slice
    reaches: these must be exactly zero."""
    j, pos, valid = A.locate_rows(idx, lay.cu_seqlens, lay.cu_seqlens_padded)
    reached = np.zeros(lay.T, dtype=bool)
    cup = lay.cu_seqlens_padded.astype(np.int64)
    for jj, pp, vv in zip(j, pos, valid):
        if vv:
            reached[cup[jj]:cup[jj] + pp + 1] = True
    return ~valid, ~reached


def _check(name, got, ref, zero_rows):
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    rel = err / scale if scale > 0 else err
    cos = float((got * ref).sum() / (np.linalg.norm(got) * np.linalg.norm(ref) + 1e-30))
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    assert rel <= BWD_TOL, f"{name}: max|d| / max|ref| = {rel:.3e} (cos {cos:.6f})"
    assert np.all(got[zero_rows] == 0), f"{name}: nonzero in rows that must be zero"
    return rel


@pytest.mark.parametrize("name,strategy,ranks", [
    ("tiny", "dcs", [0, 1]), ("tiny", "nlb", [0, 1]), ("tiny", "mirrored", [0, 1]),
    ("t8192_mha16", "dcs", [0, 3]), ("t8192_mha16", "nlb", [0, 3]), ("t8192_mha16", "mirrored", [1]),
    ("t32768_lognormal_gqa32x8", "nlb", [7]),
])
def test_backward_matches_oracle(name, strategy, ranks):
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME[name]
    inp = W.make_attn_inputs(cfg, strategy)
    lay = inp.layout
    dout_phys = W.randn_bf16(cfg.seed, 6, (lay.T, cfg.hq, cfg.d))
    err = new_err(dev)
    for r in ranks:
        idx, dq, dk, dv, dout = _rank_bwd(cp, inp, strategy, cfg.cp, r, dev, dout_phys, err)
        ref = A.attention_bwd(inp.q[torch.from_numpy(idx)], inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded,
                              idx, dout)
        zq, zk = _structural_zero(lay, idx)
        rels = [_check(f"{name}/{strategy}/r{r}/{n}", g, e, z)
                for n, g, e, z in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, (zq, zk, zk))]
        print(f"{name}/{strategy}/rank{r}: max|d|/max|ref| dq {rels[0]:.2e} dk {rels[1]:.2e} dv {rels[2]:.2e}")
    assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("case", [
    dict(lengths=[300], pad=1, hq=2, hkv=2, d=128, cp=1),                  # ragged tail
    dict(lengths=[1, 0, 5, 0, 130, 1, 2], pad=1, hq=4, hkv=1, d=64, cp=1),  # empty, one-token docs, GQA 4
    dict(lengths=[37, 91, 250, 3], pad=8, hq=6, hkv=2, d=128, cp=4),       # pads, GQA 3
])
def test_backward_edge_cases(case):
    dev = cuda_or_skip(); cp = load_lib()
    lay = W.make_layout(case["lengths"], case["pad"])
    total = int(sum(case["lengths"]))
    q, k, v = W.make_qkv_logical(77, total, case["hq"], case["hkv"], case["d"])
    if lay.T != total:
        q, k, v = (W.to_physical(t, lay, 0) for t in (q, k, v))
    cfg = W.Config("edge", 77, tuple(case["lengths"]), case["hq"], case["hkv"], case["d"], case["cp"], ("dcs",),
                   case["pad"])
    inp = W.AttnInputs(cfg, "dcs", lay, q, k, v)
    dout_phys = W.randn_bf16(77, 6, (lay.T, case["hq"], case["d"]))
    err = new_err(dev)
    for s in ("dcs", "nlb"):
        if s == "dcs" and any(int(x) % (2 * case["cp"]) for x in np.diff(lay.cu_seqlens_padded)):
            continue
        if s == "nlb" and lay.T % case["cp"]:
            continue
        for r in range(case["cp"]):
            idx, dq, dk, dv, dout = _rank_bwd(cp, inp, s, case["cp"], r, dev, dout_phys, err)
            ref = A.attention_bwd(q[torch.from_numpy(idx)], k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
            zq, zk = _structural_zero(lay, idx)
            for n, g, e, z in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, (zq, zk, zk)):
                _check(f"{case}/{s}/r{r}/{n}", g, e, z)
    assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("seed", [201, 202, 203, 204])
def test_backward_random_packs(seed):
    """Seeded random packs (empty and one-token documents included, DCS
    padding, cp_size 1-8, GQA group sizes 1-4, d = 64 or 128): every rank of
    both partitions against the oracle."""
    dev = cuda_or_skip(); cp = load_lib()
    rng = np.random.default_rng(seed)
    cpsize = int(rng.choice([1, 2, 4, 8]))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 3, 4]))
    dd = int(rng.choice([64, 128]))
    lay = W.random_layout(rng, int(rng.integers(1, 16)), 500, 2 * cpsize, allow_empty=True)
    total = int(lay.cu_seqlens[-1])
    if total == 0:
        pytest.skip("empty pack")
    q, k, v = W.make_qkv_logical(seed, total, hq, hkv, dd)
    if lay.T != total:
        q, k, v = (W.to_physical(t, lay, 0) for t in (q, k, v))
    cfg = W.Config("random", seed, tuple(np.diff(lay.cu_seqlens).tolist()), hq, hkv, dd, cpsize, ("dcs", "nlb"),
                   2 * cpsize)
    inp = W.AttnInputs(cfg, "dcs", lay, q, k, v)
    dout_phys = W.randn_bf16(seed, 6, (lay.T, hq, dd))
    err = new_err(dev)
    for s in ("dcs", "nlb"):
        for r in range(cpsize):
            idx, dq, dk, dv, dout = _rank_bwd(cp, inp, s, cpsize, r, dev, dout_phys, err)
            ref = A.attention_bwd(q[torch.from_numpy(idx)], k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
            zq, zk = _structural_zero(lay, idx)
            for n, g, e, z in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, (zq, zk, zk)):
                _check(f"seed {seed}/{s}/r{r}/{n}", g, e, z)
    assert err.cpu().tolist() == [0, 0]
