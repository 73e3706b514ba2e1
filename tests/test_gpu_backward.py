"""GPU attention backward (dQ, dK, dV) vs the float64 oracle.

Tolerance, element by element: |x - ref| <= BWD_C * M, where M is the
per-element error scale of tests/gpu_common.bwd_term_magnitudes: the sum of
the magnitudes of the terms that make up that gradient entry, weighted by the
bf16 roundings the GPU applies (P, dS, and the forward's output inside
D = rowsum(dO * O), each at most 2^-8 relative: bf16 keeps 8 significant
bits). The worst case of those roundings is 2^-7 M; BWD_C = 2^-6 leaves a
factor 2 for the fp32 accumulations and ex2.approx (orders of magnitude
smaller). Pad query rows of dQ and keys no
query of the slice reaches (dK, dV) must be exactly zero.

Cases: every element of the tiny, T=8192 and lognormal slices listed below,
edge cases, seeded random packs, one query head (all its dQ rows and all
its dK/dV keys) of the 131072-token DualChunkSwap rank 3 computed with all
eight heads, the slice the backward is benchmarked on, a pack with sharp
scores and a large dO (large per-query terms), an empty slice, and the
largest slice the backward takes (2048 query tiles).
"""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import partition as P
import workloads as W
from gpu_common import bwd_term_magnitudes, cuda_or_skip, load_lib, new_err

pytestmark = pytest.mark.gpu
BWD_C = 2.0 ** -6


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


def _check(name, got, ref, mag, zero_rows):
    """Element-wise |got - ref| <= BWD_C * mag; exact zeros where required.
    Returns the largest |got - ref| / (BWD_C * mag) (1.0 = at the bound)."""
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    assert np.all(got[zero_rows] == 0), f"{name}: nonzero in rows that must be zero"
    err = np.abs(got - ref)
    bound = BWD_C * mag
    bad = err > bound
    scale = np.abs(ref).max()
    assert not bad.any(), (f"{name}: {int(bad.sum())} entries beyond the element bound; worst excess "
                           f"{(err - bound).max():.3e}, max|d| / max|ref| = {err.max() / max(scale, 1e-30):.3e}")
    nz = bound > 0
    return float((err[nz] / bound[nz]).max()) if nz.any() else 0.0


def _compare(label, cp_out, q_loc, k, v, lay, idx, dout, heads=None):
    """Oracle gradients and error scales of the slice (optionally of some
    heads only, MHA), checked against the GPU's."""
    dq, dk, dv = cp_out
    if heads is not None:
        sel = list(heads)
        q_loc, k, v, dout = q_loc[:, sel], k[:, sel], v[:, sel], dout[:, sel]
        dq, dk, dv = dq[:, sel], dk[:, sel], dv[:, sel]
    ref = A.attention_bwd(q_loc, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
    mag = bwd_term_magnitudes(q_loc, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, dout)
    zq, zk = _structural_zero(lay, idx)
    ratios = [_check(f"{label}/{n}", g, e, m, z)
              for n, g, e, m, z in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, mag, (zq, zk, zk))]
    print(f"{label}: max |d| / bound  dq {ratios[0]:.3f} dk {ratios[1]:.3f} dv {ratios[2]:.3f}")
    return ratios


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
        _compare(f"{name}/{strategy}/rank{r}", (dq, dk, dv), inp.q[torch.from_numpy(idx)], inp.k, inp.v, lay, idx,
                 dout)
    assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("case", [
    dict(lengths=[300], pad=1, hq=2, hkv=2, d=128, cp=1),                  # ragged tail
    dict(lengths=[1, 0, 5, 0, 130, 1, 2], pad=1, hq=4, hkv=1, d=64, cp=1),  # empty, one-token docs, GQA 4
    dict(lengths=[37, 91, 250, 3], pad=8, hq=6, hkv=2, d=128, cp=4),       # pads, GQA 3
    dict(lengths=[517, 1, 260, 900], pad=4, hq=16, hkv=1, d=64, cp=2),     # 16 query heads per KV head
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
            _compare(f"{case}/{s}/r{r}", (dq, dk, dv), q[torch.from_numpy(idx)], k, v, lay, idx, dout)
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
            _compare(f"seed {seed}/{s}/r{r}", (dq, dk, dv), q[torch.from_numpy(idx)], k, v, lay, idx, dout)
    assert err.cpu().tolist() == [0, 0]


def test_backward_long_context_rank_one_head():
    """The benchmarked slice: rank 3 of the 131072-token document under
    DualChunkSwap (cp_size 16), run on the GPU with all eight heads. With
    Hq = Hkv the heads are independent, so head 0's dQ (all 8192 rows) and
    dK/dV (all 131072 keys) are checked against the oracle run on head 0's
    inputs alone; the dK/dV pass's key tiles here collect up to 64 query
    tiles each."""
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME["long131072_h8"]
    inp = W.make_attn_inputs(cfg, "dcs")
    lay = inp.layout
    dout_phys = W.randn_bf16(cfg.seed, 6, (lay.T, cfg.hq, cfg.d))
    err = new_err(dev)
    idx, dq, dk, dv, dout = _rank_bwd(cp, inp, "dcs", cfg.cp, 3, dev, dout_phys, err)
    assert err.cpu().tolist() == [0, 0]
    _compare("long131072_h8/dcs/rank3/head0", (dq, dk, dv), inp.q[torch.from_numpy(idx)], inp.k, inp.v, lay, idx,
             dout, heads=[0])


def test_backward_sharp_scores_and_large_dout():
    """Scores six times sharper than the N(0,1) inputs give (Q scaled by 6
    before its bf16 rounding) and dO twenty times larger, so |s| reaches the
    hundreds and |LSE| and |D| the tens. The dK/dV pass takes the per-query
    terms lse * log2(e) / (scale log2(e)) and D into its score MMAs as sums of
    three bf16 terms; a split that kept fewer bits, or a wrong sign, breaks
    the element bound here. Both partitions, both ranks, GQA 2/1, d = 128,
    two documents."""
    dev = cuda_or_skip(); cp = load_lib()
    lengths = (700, 1300)
    lay = W.make_layout(list(lengths), 1)
    q, k, v = W.make_qkv_logical(91, sum(lengths), 2, 1, 128)
    q = (q.float() * 6).to(torch.bfloat16)
    cfg = W.Config("sharp", 91, lengths, 2, 1, 128, 2, ("dcs",), 1)
    inp = W.AttnInputs(cfg, "dcs", lay, q, k, v)
    dout_phys = (W.randn_bf16(91, 6, (lay.T, 2, 128)).float() * 20).to(torch.bfloat16)
    err = new_err(dev)
    for s in ("dcs", "nlb"):
        for r in range(2):
            idx, dq, dk, dv, dout = _rank_bwd(cp, inp, s, 2, r, dev, dout_phys, err)
            _compare(f"sharp/{s}/r{r}", (dq, dk, dv), q[torch.from_numpy(idx)], k, v, lay, idx, dout)
    assert err.cpu().tolist() == [0, 0]


def test_empty_slice():
    """A rank slice of no rows (t_local = 0) against a nonempty K/V buffer:
    the forward returns empty outputs without error, and the backward's
    contribution to dK and dV is all zeros (the buffers are pre-filled with
    garbage to see that every entry is written)."""
    dev = cuda_or_skip(); cp = load_lib()
    lay = W.make_layout([300], 1)
    _, k, v = W.make_qkv_logical(5, 300, 2, 2, 64)
    k, v = k.to(dev), v.to(dev)
    cu = torch.from_numpy(lay.cu_seqlens).to(dev)
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    idx = torch.empty(0, dtype=torch.int32, device=dev)
    q_loc = torch.empty((0, 2, 64), dtype=torch.bfloat16, device=dev)
    err = new_err(dev)
    out, lse = cp.thd_causal_attn_fwd(idx, q_loc, k, v, cu, cup, err=err)
    assert tuple(out.shape) == (0, 2, 64) and tuple(lse.shape) == (2, 0)
    dk = torch.full((300, 2, 64), 7.0, dtype=torch.float32, device=dev)
    dv = torch.full((300, 2, 64), -3.0, dtype=torch.float32, device=dev)
    dq, dk, dv = cp.thd_causal_attn_bwd(idx, q_loc, k, v, out, torch.empty_like(q_loc), lse, cu, cup, dk=dk, dv=dv,
                                        err=err)
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]
    assert tuple(dq.shape) == (0, 2, 64)
    assert bool((dk == 0).all()) and bool((dv == 0).all())


def test_backward_largest_slice():
    """The largest slice the backward takes: 2048 query tiles (t_local =
    262,144 rows), the capacity of the dK/dV pass's per-item tile lists
    (16-bit entries: tile index and a full-tile bit). 512 documents of 512
    tokens, one head, d = 64, cp_size 1; every element of dQ, dK and dV
    against the oracle. One more tile is refused on the host."""
    dev = cuda_or_skip(); cp = load_lib()
    lengths = [512] * 512
    lay = W.make_layout(lengths, 1)
    q, k, v = W.make_qkv_logical(303, lay.T, 1, 1, 64)
    cfg = W.Config("max_tiles", 303, tuple(lengths), 1, 1, 64, 1, ("nlb",), 1)
    inp = W.AttnInputs(cfg, "nlb", lay, q, k, v)
    dout_phys = W.randn_bf16(303, 6, (lay.T, 1, 64))
    err = new_err(dev)
    idx, dq, dk, dv, dout = _rank_bwd(cp, inp, "nlb", 1, 0, dev, dout_phys, err)
    assert idx.shape[0] == 2048 * 128
    assert err.cpu().tolist() == [0, 0]
    _compare("largest slice", (dq, dk, dv), q[torch.from_numpy(idx)], k, v, lay, idx, dout)
    too_many = 2048 * 128 + 1
    with pytest.raises(cp.CpthdError, match="status -"):
        cp.thd_causal_attn_bwd(torch.zeros(too_many, dtype=torch.int32, device=dev),
                               torch.zeros((too_many, 1, 64), dtype=torch.bfloat16, device=dev),
                               torch.zeros((too_many, 1, 64), dtype=torch.bfloat16, device=dev),
                               torch.zeros((too_many, 1, 64), dtype=torch.bfloat16, device=dev),
                               torch.zeros((too_many, 1, 64), dtype=torch.bfloat16, device=dev),
                               torch.zeros((too_many, 1, 64), dtype=torch.bfloat16, device=dev),
                               torch.zeros((1, too_many), dtype=torch.float32, device=dev),
                               torch.tensor([0, too_many], dtype=torch.int32, device=dev))
