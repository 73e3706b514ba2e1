"""GPU attention forward vs the float64 oracle.

Tolerances: max |out - ref| <= 1e-2 + 1e-2 |ref| (bf16 output) and
|lse - ref| <= 2e-3; pad rows must be exactly out = 0, lse = -inf.

* tiny (2 docs, d = 64) and T = 8192 (16 docs, MHA 16x128): every row of
  every rank, both strategies.
* T = 32768 lognormal GQA 32/8, 48 padded docs GQA 32/8 and the single
  131072-token document: every rank under the strategies the workload names,
  at full size, on sampled rows (first/last rows, rows at chunk and tile
  boundaries, random rows) that the oracle computes one by one; and every
  row of one rank of the lognormal (both strategies) and padded packs.
* DualChunkSwap as two launches per rank (one per owned chunk, the pages'
  two attention steps): every row against the oracle and the one launch.
* long work items cut into pieces at the CTAs' share boundaries (one long
  document, few heads): every row, and bit-identical repeated runs.
* edge cases: ragged tails, empty and one-token documents, pad rows, GQA
  group sizes, custom scale, arbitrary row order of the query slice, and
  device-checked malformed offsets.
"""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import partition as P
import workloads as W
from gpu_common import assert_attn_matches, cuda_or_skip, load_lib, new_err

pytestmark = pytest.mark.gpu


class DevInputs:
    def __init__(self, inp, dev):
        self.inp = inp
        lay = inp.layout
        self.cu = torch.from_numpy(lay.cu_seqlens).to(dev)
        self.cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
        self.q = inp.q.to(dev)
        self.k = inp.k.to(dev)
        self.v = inp.v.to(dev)


def _run_rank(cp, d, strategy, cpsize, r, err, scale=None):
    lay = d.inp.layout
    idx = cp.cp_partition_index(strategy, d.cup, lay.T, cpsize, r, err=err)
    q_loc = cp.cp_reorder(d.q, idx, err=err)
    out, lse = cp.thd_causal_attn_fwd(idx, q_loc, d.k, d.v, d.cu, d.cup, softmax_scale=scale, err=err)
    return idx, out, lse


def _sample_rows(lay, ref_idx, cpsize, rng, n_random=40):
    """Rows at the ends, at tile (128) boundaries and at DualChunkSwap chunk
    boundaries (cu_seqlens_padded / cp_size), plus random rows."""
    n = len(ref_idx)
    rows = {0, n - 1}
    for b in range(128, n, 128):
        rows.update({b - 1, b})
    loc = lay.cu_seqlens_padded // cpsize
    for x in loc[1:-1][:64]:
        rows.update({int(x) - 1, int(x)})
    rows.update(rng.integers(0, n, size=n_random).tolist())
    rows = sorted(r for r in rows if 0 <= r < n)
    if len(rows) > 160:
        rows = sorted(rng.choice(rows, size=160, replace=False).tolist() + [0, n - 1])
    return np.unique(np.asarray(rows, dtype=np.int64))


@pytest.mark.parametrize("name", ["tiny", "t8192_mha16"])
@pytest.mark.parametrize("strategy", ["dcs", "nlb", "mirrored"])
def test_small_configs_all_rows(name, strategy):
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME[name]
    inp = W.make_attn_inputs(cfg, strategy)
    d = DevInputs(inp, dev)
    lay = inp.layout
    err = new_err(dev)
    for r in range(cfg.cp):
        idx, out, lse = _run_rank(cp, d, strategy, cfg.cp, r, err)
        ref_idx = np.asarray(P.partition_index(strategy, lay.cu_seqlens_padded.tolist(), cfg.cp, r))
        assert np.array_equal(idx.cpu().numpy(), ref_idx)
        ro, rl = A.attention_fwd(inp.q[torch.from_numpy(ref_idx)], inp.k, inp.v, lay.cu_seqlens,
                                 lay.cu_seqlens_padded, ref_idx)
        assert_attn_matches(out, lse, ro, rl, f"{name}/{strategy}/rank{r}")
    assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("name,strategy", [
    ("t32768_lognormal_gqa32x8", "dcs"), ("t32768_lognormal_gqa32x8", "nlb"),
    ("t32768_lognormal_gqa32x8", "mirrored"),
    ("padded48_gqa32x8", "dcs"),
    ("long131072_h8", "dcs"), ("long131072_h8", "nlb"),
])
def test_full_size_sampled_rows(name, strategy):
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME[name]
    inp = W.make_attn_inputs(cfg, strategy)
    d = DevInputs(inp, dev)
    lay = inp.layout
    rng = np.random.default_rng(cfg.seed + 17)
    err = new_err(dev)
    for r in range(cfg.cp):
        idx, out, lse = _run_rank(cp, d, strategy, cfg.cp, r, err)
        ref_idx = np.asarray(P.partition_index(strategy, lay.cu_seqlens_padded.tolist(), cfg.cp, r))
        rows = _sample_rows(lay, ref_idx, cfg.cp, rng, n_random=24 if cfg.cp > 8 else 40)
        q_loc = inp.q[torch.from_numpy(ref_idx)]
        ro, rl = A.attention_fwd(q_loc, inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded, ref_idx, rows=rows)
        rows_t = torch.from_numpy(rows).to(dev)
        assert_attn_matches(out[rows_t], lse[:, rows_t], ro, rl, f"{name}/{strategy}/rank{r}")
        # properties of every row: finite outputs, lse >= max score bound is
        # implied by the sampled check; here: no NaN anywhere, pads exact
        assert not torch.isnan(out.float()).any()
        assert not torch.isnan(lse).any()
    assert err.cpu().tolist() == [0, 0]


def _custom(lengths, pad_multiple, hq, hkv, dd, seed):
    lay = W.make_layout(lengths, pad_multiple)
    total = int(sum(lengths))
    q, k, v = W.make_qkv_logical(seed, total, hq, hkv, dd)
    if lay.T != total:
        q, k, v = (W.to_physical(t, lay, 0) for t in (q, k, v))
    cfg = W.Config("custom", seed, tuple(lengths), hq, hkv, dd, 1, ("dcs",), pad_multiple)
    return W.AttnInputs(cfg, "dcs", lay, q, k, v)


@pytest.mark.parametrize("case", [
    dict(lengths=[300], pad=1, hq=2, hkv=2, d=128, cp=1),                  # ragged tail: 3 tiles, last has 44 rows
    dict(lengths=[1, 0, 5, 0, 130, 1, 2], pad=1, hq=4, hkv=1, d=64, cp=1),  # empty and one-token docs, GQA 4
    dict(lengths=[37, 91, 250, 3], pad=8, hq=6, hkv=2, d=128, cp=4),       # pad rows, GQA 3
    dict(lengths=[129, 127, 128, 256, 1], pad=2, hq=2, hkv=2, d=64, cp=1),  # docs at tile edges, pads
    dict(lengths=[700, 53, 1200], pad=16, hq=8, hkv=8, d=128, cp=8),       # several ranks, chunk < tile
    dict(lengths=[517, 1, 260, 900], pad=4, hq=32, hkv=1, d=64, cp=2),     # one KV head for 32 query heads
    dict(lengths=[2000, 3, 1500], pad=2, hq=5, hkv=5, d=128, cp=1),        # odd head count, one rank
])
def test_edge_cases(case):
    dev = cuda_or_skip(); cp = load_lib()
    inp = _custom(case["lengths"], case["pad"], case["hq"], case["hkv"], case["d"], 99)
    d = DevInputs(inp, dev)
    lay = inp.layout
    err = new_err(dev)
    for s in ("dcs", "nlb"):
        if s == "dcs" and any(int(x) % (2 * case["cp"]) for x in np.diff(lay.cu_seqlens_padded)):
            continue
        if s == "nlb" and lay.T % case["cp"]:
            continue
        for r in range(case["cp"]):
            idx, out, lse = _run_rank(cp, d, s, case["cp"], r, err)
            ref_idx = np.asarray(P.partition_index(s, lay.cu_seqlens_padded.tolist(), case["cp"], r))
            ro, rl = A.attention_fwd(inp.q[torch.from_numpy(ref_idx)], inp.k, inp.v, lay.cu_seqlens,
                                     lay.cu_seqlens_padded, ref_idx)
            assert_attn_matches(out, lse, ro, rl, f"{case}/{s}/rank{r}")
    assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("n_docs", [4095, 5000])
def test_many_short_documents(n_docs):
    """Thousands of 1-6 token documents: a row group holds dozens of
    documents, so the metadata's interval lists are long; every row of every
    rank against the oracle."""
    dev = cuda_or_skip(); cp = load_lib()
    rng = np.random.default_rng(n_docs)
    lengths = rng.integers(1, 7, size=n_docs).tolist()
    inp = _custom(lengths, 4, 4, 2, 64, 17)
    d = DevInputs(inp, dev)
    lay = inp.layout
    err = new_err(dev)
    for s in ("dcs", "nlb"):
        for r in range(2):
            idx, out, lse = _run_rank(cp, d, s, 2, r, err)
            ref_idx = np.asarray(P.partition_index(s, lay.cu_seqlens_padded.tolist(), 2, r))
            ro, rl = A.attention_fwd(inp.q[torch.from_numpy(ref_idx)], inp.k, inp.v, lay.cu_seqlens,
                                     lay.cu_seqlens_padded, ref_idx)
            assert_attn_matches(out, lse, ro, rl, f"{n_docs} docs/{s}/rank{r}")
    assert err.cpu().tolist() == [0, 0]


def test_custom_scale_and_permuted_rows():
    """Any row order of the query slice works (the slice index travels with
    the rows), and an explicit softmax scale is honoured."""
    dev = cuda_or_skip(); cp = load_lib()
    inp = _custom([333, 90, 611], 1, 4, 2, 128, 5)
    d = DevInputs(inp, dev)
    lay = inp.layout
    perm = np.random.default_rng(1).permutation(lay.T).astype(np.int32)
    idx = torch.from_numpy(perm).to(dev)
    q_loc = cp.cp_reorder(d.q, idx)
    out, lse = cp.thd_causal_attn_fwd(idx, q_loc, d.k, d.v, d.cu, None, softmax_scale=0.2)
    ro, rl = A.attention_fwd(inp.q[torch.from_numpy(perm.astype(np.int64))], inp.k, inp.v, lay.cu_seqlens,
                             lay.cu_seqlens_padded, perm, scale=0.2)
    assert_attn_matches(out, lse, ro, rl, "permuted")


@pytest.mark.parametrize("hq,hkv,strategy", [(16, 16, "dcs"), (32, 8, "nlb"), (32, 8, "dcs")])
def test_plan_once_run_many(hq, hkv, strategy):
    """One plan serves several attentions over the same slice (as the layers
    of a step do): each planned run is bit-identical to the one-call forward
    on the same inputs, for both head dims and for grids of one wave (MHA,
    2048 rows) and of several waves (GQA 32/8, ordered groups)."""
    dev = cuda_or_skip(); cp = load_lib()
    lengths = [2500, 700, 1800, 1, 3191]          # 8192 tokens, 8208 once padded to multiples of 2 * cp_size
    cpsize = 4
    runs = []
    for dd, seed in ((128, 11), (64, 12), (128, 13)):
        inp = _custom(lengths, 2 * cpsize, hq, hkv, dd, seed)
        runs.append(DevInputs(inp, dev))
    lay = runs[0].inp.layout
    for r in range(cpsize):
        err = new_err(dev)
        idx = cp.cp_partition_index(strategy, runs[0].cup, lay.T, cpsize, r, err=err)
        ws = cp.thd_causal_attn_plan(idx, lay.T, runs[0].cu, runs[0].cup, hq, hkv, err=err)
        for d in runs:
            q_loc = cp.cp_reorder(d.q, idx, err=err)
            o1, l1 = cp.thd_causal_attn_fwd_planned(q_loc, d.k, d.v, ws, err=err)
            o2, l2 = cp.thd_causal_attn_fwd(idx, q_loc, d.k, d.v, d.cu, d.cup, err=err)
            assert torch.equal(o1, o2) and torch.equal(l1, l2), (strategy, r, d.q.shape)
        assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("name", ["t8192_mha16", "t32768_lognormal_gqa32x8"])
def test_plan_from_partition_formulas_equals_plan_from_list(name):
    """thd_causal_attn_plan_partition (row slots from the partition formulas)
    writes the same workspace bytes as thd_causal_attn_plan given the index
    list, for every strategy and rank, and the attention run on either plan
    is identical."""
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME[name]
    for s in ("dcs", "nlb", "mirrored"):
        strat = "dcs" if s == "dcs" else "nlb"      # the mirrored split runs on the unpadded buffer
        inp = W.make_attn_inputs(cfg, strat)
        d = DevInputs(inp, dev)
        lay = inp.layout
        if s == "mirrored" and lay.T % (2 * cfg.cp) != 0:
            continue
        err = new_err(dev)
        tl = cp.cp_local_tokens(s, lay.T, cfg.cp)
        nb = cp.thd_causal_attn_workspace_size(tl, cfg.hq, cfg.hkv, cfg.d)
        for r in range(cfg.cp):
            ws_list = torch.zeros(nb, dtype=torch.uint8, device=dev)
            ws_form = torch.zeros(nb, dtype=torch.uint8, device=dev)
            idx = cp.cp_partition_index(s, d.cup, lay.T, cfg.cp, r, err=err)
            cp.thd_causal_attn_plan(idx, lay.T, d.cu, d.cup, cfg.hq, cfg.hkv, workspace=ws_list, err=err)
            cp.thd_causal_attn_plan_partition(s, lay.T, d.cu, d.cup, cfg.cp, r, cfg.hq, cfg.hkv, workspace=ws_form,
                                              err=err)
            assert torch.equal(ws_list, ws_form), (name, s, r)
            if r in (0, cfg.cp - 1):
                q_loc = cp.cp_reorder(d.q, idx, err=err)
                o1, l1 = cp.thd_causal_attn_fwd_planned(q_loc, d.k, d.v, ws_form, err=err)
                o2, l2 = cp.thd_causal_attn_fwd(idx, q_loc, d.k, d.v, d.cu, d.cup, err=err)
                assert torch.equal(o1, o2) and torch.equal(l1, l2), (name, s, r)
        assert err.cpu().tolist() == [0, 0], (name, s)


def test_plan_from_partition_checks_divisibility():
    """Under DualChunkSwap a padded length that is not a multiple of
    2*cp_size is recorded by the plan itself (no index list was built)."""
    dev = cuda_or_skip(); cp = load_lib()
    cu = torch.tensor([0, 12, 24], dtype=torch.int32, device=dev)   # 12 % (2 * 2) == 0, fine
    cup = torch.tensor([0, 12, 24], dtype=torch.int32, device=dev)
    err = new_err(dev)
    cp.thd_causal_attn_plan_partition("dcs", 24, cu, cup, 2, 0, 2, 2, err=err)
    assert err.cpu().tolist() == [0, 0]
    cu = torch.tensor([0, 10, 24], dtype=torch.int32, device=dev)   # 10 % 4 != 0
    err = new_err(dev)
    cp.thd_causal_attn_plan_partition("dcs", 24, cu, cu, 2, 0, 2, 2, err=err)
    assert err.cpu().tolist()[0] == -2


@pytest.mark.parametrize("seed", [101, 102, 103, 104, 105, 106, 107, 122, 124])
def test_random_packs_every_row(seed):
    """Seeded random packs (empty and one-token documents included, DCS
    padding, cp_size 1-8, GQA group sizes 1-4, d = 64 or 128), every rank of
    every partition that the pack allows, every row against the oracle."""
    dev = cuda_or_skip(); cp = load_lib()
    rng = np.random.default_rng(seed)
    cpsize = int(rng.choice([1, 2, 4, 8]))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 3, 4]))
    dd = int(rng.choice([64, 128]))
    lay = W.random_layout(rng, int(rng.integers(1, 24)), 700, 2 * cpsize, allow_empty=True)
    total = int(lay.cu_seqlens[-1])
    if total == 0:
        pytest.skip("empty pack")
    q, k, v = W.make_qkv_logical(seed, total, hq, hkv, dd)
    if lay.T != total:
        q, k, v = (W.to_physical(t, lay, 0) for t in (q, k, v))
    cu = torch.from_numpy(lay.cu_seqlens).to(dev)
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    strategies = ["dcs", "nlb"] + (["mirrored"] if lay.T % (2 * cpsize) == 0 else [])
    err = new_err(dev)
    for s in strategies:
        for r in range(cpsize):
            idx = cp.cp_partition_index(s, cup, lay.T, cpsize, r, err=err)
            q_loc = cp.cp_reorder(qd, idx, err=err)
            out, lse = cp.thd_causal_attn_fwd(idx, q_loc, kd, vd, cu, cup, err=err)
            ref_idx = np.asarray(P.partition_index(s, lay.cu_seqlens_padded.tolist(), cpsize, r), dtype=np.int64)
            assert np.array_equal(idx.cpu().numpy(), ref_idx)
            ro, rl = A.attention_fwd(q[torch.from_numpy(ref_idx)], k, v, lay.cu_seqlens, lay.cu_seqlens_padded,
                                     ref_idx)
            assert_attn_matches(out, lse, ro, rl, f"seed {seed}/{s}/rank{r}")
    assert err.cpu().tolist() == [0, 0]


def test_plan_on_side_stream_beside_the_gather():
    """The order a caller overlaps the path in: partition index, then the
    gather on the current stream and the plan on a side stream (the plan
    needs only the index), then the planned attention after both; checked
    against the oracle on every rank of both strategies, with the slices run
    back to back through one workspace."""
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME["t8192_mha16"]
    side = torch.cuda.Stream()
    rng = np.random.default_rng(7)
    for s in ("dcs", "nlb"):
        inp = W.make_attn_inputs(cfg, s)
        d = DevInputs(inp, dev)
        lay = inp.layout
        err = new_err(dev)
        tl = cp.cp_local_tokens(s, lay.T, cfg.cp)
        ws = torch.empty(cp.thd_causal_attn_workspace_size(tl, cfg.hq, cfg.hkv, cfg.d), dtype=torch.uint8,
                         device=dev)
        results = []
        main = torch.cuda.current_stream()
        for r in range(cfg.cp):
            idx = cp.cp_partition_index(s, d.cup, lay.T, cfg.cp, r, err=err)
            side.wait_stream(main)
            with torch.cuda.stream(side):
                cp.thd_causal_attn_plan(idx, lay.T, d.cu, d.cup, cfg.hq, cfg.hkv, workspace=ws, err=err)
            q_loc = cp.cp_reorder(d.q, idx, err=err)
            main.wait_stream(side)
            out, lse = cp.thd_causal_attn_fwd_planned(q_loc, d.k, d.v, ws, err=err)
            results.append((idx, out.clone(), lse.clone()))
        torch.cuda.synchronize()
        for r, (idx, out, lse) in enumerate(results):
            ref_idx = np.asarray(P.partition_index(s, lay.cu_seqlens_padded, cfg.cp, r), dtype=np.int64)
            assert np.array_equal(idx.cpu().numpy(), ref_idx)
            rows = _sample_rows(lay, ref_idx, cfg.cp, rng)
            ro, rl = A.attention_fwd(inp.q[torch.from_numpy(ref_idx)], inp.k, inp.v, lay.cu_seqlens,
                                     lay.cu_seqlens_padded, ref_idx, rows=rows)
            rows_t = torch.from_numpy(rows).to(dev)
            assert_attn_matches(out[rows_t], lse[:, rows_t], ro, rl, f"{s}/rank{r}")
        assert err.cpu().tolist() == [0, 0]


def test_both_layouts_agree_per_token():
    """Matched inputs: the DualChunkSwap (padded) and NO_LOAD_BALANCE
    (unpadded) runs give each real token the same result within tolerance."""
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME["t8192_mha16"]
    res = {}
    for s in ("dcs", "nlb"):
        inp = W.make_attn_inputs(cfg, s)
        d = DevInputs(inp, dev)
        lay = inp.layout
        full_o = torch.zeros((lay.T, cfg.hq, cfg.d), dtype=torch.float32)
        for r in range(cfg.cp):
            idx, out, lse = _run_rank(cp, d, s, cfg.cp, r, new_err(dev))
            full_o[idx.cpu().long()] = out.float().cpu()
        res[s] = full_o[torch.from_numpy(W.physical_slots(lay))] if s == "dcs" else full_o
    assert (res["dcs"] - res["nlb"]).abs().max().item() <= 2e-2


def test_malformed_offsets_recorded():
    dev = cuda_or_skip(); cp = load_lib()
    inp = _custom([40, 24], 8, 2, 2, 64, 3)
    d = DevInputs(inp, dev)
    idx = torch.arange(inp.layout.T, dtype=torch.int32, device=dev)
    # actual length 41 > padded length 40 for document 0
    bad_cu = torch.tensor([0, 41, 65], dtype=torch.int32, device=dev)
    err = new_err(dev)
    cp.thd_causal_attn_fwd(idx, d.q, d.k, d.v, bad_cu, d.cup, err=err)
    assert err.cpu().tolist() == [-8, 0]
    # padded offsets ending short of T
    err = new_err(dev)
    short = torch.tensor([0, 40, 60], dtype=torch.int32, device=dev)
    cp.thd_causal_attn_fwd(idx, d.q, d.k, d.v, torch.tensor([0, 40, 60], dtype=torch.int32, device=dev), short,
                           err=err)
    assert err.cpu().tolist()[0] in (-6, -7)


def _dcs_halves(lay, cpsize):
    """Local rows of a DualChunkSwap rank's first owned chunk of every
    document, and of its second: the two attention steps per rank of the
    pages' design (one per owned chunk)."""
    lcu = lay.cu_seqlens_padded.astype(np.int64) // cpsize
    halves = [[], []]
    for j in range(lay.num_docs):
        c = (lcu[j + 1] - lcu[j]) // 2
        halves[0].append(np.arange(lcu[j], lcu[j] + c))
        halves[1].append(np.arange(lcu[j] + c, lcu[j + 1]))
    return [np.concatenate(h).astype(np.int64) for h in halves]


@pytest.mark.parametrize("name,ranks", [("t8192_mha16", [0, 1, 2, 3]), ("t32768_lognormal_gqa32x8", [6]),
                                        ("padded48_gqa32x8", [1])])
def test_dcs_two_launches_match_oracle(name, ranks):
    """A DualChunkSwap rank run as two launches, one per owned chunk (each
    launch gets that chunk's rows of every document and their slots): every
    row of both launches against the oracle, and against the one-launch
    result of the same rank, with the device checks clean."""
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME[name]
    inp = W.make_attn_inputs(cfg, "dcs")
    d = DevInputs(inp, dev)
    lay = inp.layout
    halves = _dcs_halves(lay, cfg.cp)
    err = new_err(dev)
    for r in ranks:
        idx, out1, lse1 = _run_rank(cp, d, "dcs", cfg.cp, r, err)
        ref_idx = np.asarray(P.partition_index("dcs", lay.cu_seqlens_padded.tolist(), cfg.cp, r), dtype=np.int64)
        assert np.array_equal(np.sort(np.concatenate(halves)), np.arange(len(ref_idx)))
        q_loc = cp.cp_reorder(d.q, idx, err=err)
        for h, rows in enumerate(halves):
            rows_t = torch.from_numpy(rows).to(dev)
            idx_h = idx[rows_t].contiguous()
            out_h, lse_h = cp.thd_causal_attn_fwd(idx_h, q_loc[rows_t].contiguous(), d.k, d.v, d.cu, d.cup, err=err)
            ro, rl = A.attention_fwd(inp.q[torch.from_numpy(ref_idx[rows])], inp.k, inp.v, lay.cu_seqlens,
                                     lay.cu_seqlens_padded, ref_idx[rows])
            assert_attn_matches(out_h, lse_h, ro, rl, f"{name}/rank{r}/launch{h}")
            assert_attn_matches(out_h, lse_h, out1[rows_t].float().cpu().numpy(),
                                lse1[:, rows_t].cpu().numpy().astype(np.float64), f"{name}/rank{r}/launch{h} vs one")
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("name,strategy,rank", [
    ("t32768_lognormal_gqa32x8", "dcs", 5), ("t32768_lognormal_gqa32x8", "nlb", 4),
    ("padded48_gqa32x8", "dcs", 2),
])
def test_full_size_rank_every_row(name, strategy, rank):
    """Every row of one full-size rank slice against the oracle (the other
    ranks of these workloads are checked on sampled rows above)."""
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME[name]
    inp = W.make_attn_inputs(cfg, strategy)
    d = DevInputs(inp, dev)
    lay = inp.layout
    err = new_err(dev)
    idx, out, lse = _run_rank(cp, d, strategy, cfg.cp, rank, err)
    ref_idx = np.asarray(P.partition_index(strategy, lay.cu_seqlens_padded.tolist(), cfg.cp, rank), dtype=np.int64)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    ro, rl = A.attention_fwd(inp.q[torch.from_numpy(ref_idx)], inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded,
                             ref_idx)
    assert_attn_matches(out, lse, ro, rl, f"{name}/{strategy}/rank{rank}")
    assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("permute", [False, True])
def test_more_document_runs_than_shared_memory_holds(permute):
    """About 10,000 one- and two-token documents in one slice (cp_size 1):
    more document runs than the plan keeps in shared memory (4096), so the
    group blocks walk the tile cut through the global run list; with the
    slice's rows permuted, nearly every row is a run of its own. Every row
    against the oracle, and the planned run bit-identical to the one call."""
    dev = cuda_or_skip(); cp = load_lib()
    rng = np.random.default_rng(10000 + int(permute))
    lengths = rng.integers(1, 3, size=10000).tolist()
    inp = _custom(lengths, 1, 4, 2, 64, 23)
    d = DevInputs(inp, dev)
    lay = inp.layout
    order = rng.permutation(lay.T) if permute else np.arange(lay.T)
    idx = torch.from_numpy(order.astype(np.int32)).to(dev)
    err = new_err(dev)
    q_loc = cp.cp_reorder(d.q, idx, err=err)
    out, lse = cp.thd_causal_attn_fwd(idx, q_loc, d.k, d.v, d.cu, d.cup, err=err)
    ws = cp.thd_causal_attn_plan(idx, lay.T, d.cu, d.cup, 4, 2, err=err)
    o2, l2 = cp.thd_causal_attn_fwd_planned(q_loc, d.k, d.v, ws, err=err)
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]
    assert torch.equal(out, o2) and torch.equal(lse, l2)
    ref_idx = order.astype(np.int64)
    ro, rl = A.attention_fwd(inp.q[torch.from_numpy(ref_idx)], inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded,
                             ref_idx)
    assert_attn_matches(out, lse, ro, rl, f"10000 documents, permuted={permute}")


@pytest.mark.parametrize("hq,hkv,dd", [(1, 1, 64), (2, 1, 128)])
def test_long_items_cut_into_pieces_every_row(hq, hkv, dd):
    """One 16384-token document as a single slice (cp_size 1) under one or two
    query heads: the work items (one per 128- or 256-row group) are long
    (65 key blocks on average), so the CTAs take equal shares of the work
    and most items are cut into pieces whose partial results one CTA
    combines (up to five pieces here). Every row against the oracle, and one
    plan run three times: bit-identical results each time (the pieces are
    combined in a fixed order, and the hand-off flags are lowered again
    after every launch)."""
    dev = cuda_or_skip(); cp = load_lib()
    inp = _custom([16384], 1, hq, hkv, dd, 31 + dd)
    d = DevInputs(inp, dev)
    lay = inp.layout
    err = new_err(dev)
    idx = cp.cp_partition_index("nlb", d.cup, lay.T, 1, 0, err=err)
    ws = cp.thd_causal_attn_plan(idx, lay.T, d.cu, d.cup, hq, hkv, err=err)
    q_loc = cp.cp_reorder(d.q, idx, err=err)
    outs = [cp.thd_causal_attn_fwd_planned(q_loc, d.k, d.v, ws, err=err) for _ in range(3)]
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    ref_idx = np.arange(lay.T, dtype=np.int64)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    ro, rl = A.attention_fwd(inp.q, inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded, ref_idx)
    assert_attn_matches(outs[0][0], outs[0][1], ro, rl, f"one document, Hq {hq}, d {dd}")


@pytest.mark.parametrize("total", [1024, 16384])
def test_running_max_jumps_every_block(total):
    """Scores that rise by about 10 (in units of log2) from one key block to
    the next: the keys of block b are b * gamma times a direction every
    query shares, plus small N(0,1) noise. Each new block then raises every
    row's running max by more than the softmax's rescale threshold (8), so
    O is rescaled in TMEM at every block (the path the two-half P V release
    has to order before the block's first P V). 1024 tokens run as whole items
    from the counter; 16384 tokens make the plan cut items into pieces, whose
    merge combines partial results of very different maxima. One head,
    d = 128, cp_size 1, every row against the oracle."""
    dev = cuda_or_skip(); cp = load_lib()
    d_ = 128
    lay = W.make_layout([total], 1)
    q0, k0, v = W.make_qkv_logical(55, total, 1, 1, d_)
    scale = 1.0 / np.sqrt(d_)
    gamma = 10.0 / (scale * d_ * 0.25 * np.log2(np.e))  # log2 step per block with directions of 0.5
    blk = torch.arange(total, dtype=torch.float32) // 128
    q = (0.5 + 0.05 * q0.float()).to(torch.bfloat16)
    k = (0.5 * gamma * blk[:, None, None] + 0.05 * k0.float()).to(torch.bfloat16)
    cfg = W.Config("jumps", 55, (total,), 1, 1, d_, 1, ("nlb",), 1)
    inp = W.AttnInputs(cfg, "nlb", lay, q, k, v)
    d = DevInputs(inp, dev)
    err = new_err(dev)
    idx = cp.cp_partition_index("nlb", d.cup, lay.T, 1, 0, err=err)
    q_loc = cp.cp_reorder(d.q, idx, err=err)
    out, lse = cp.thd_causal_attn_fwd(idx, q_loc, d.k, d.v, d.cu, d.cup, err=err)
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]
    ref_idx = np.arange(lay.T, dtype=np.int64)
    ro, rl = A.attention_fwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, ref_idx)
    # the premise: the rows' maxima rise by more than the threshold per block
    assert float(rl[0, -1] - rl[0, 127]) * np.log2(np.e) > 8.0 * (total // 128 - 1)
    assert_attn_matches(out, lse, ro, rl, f"running max jumps, {total} tokens")
