"""Pins for the attention oracle (no GPU).

Each pin is independent of the oracle's own code path:
* a hand-worked two-token example (tests/golden/attention_tiny.json);
* a per-pair scalar brute force on tiny packs (within 1e-12);
* cp_size = 1 with one document reduces to textbook causal attention, checked
  against torch's scaled_dot_product_attention(is_causal=True) in float64;
* per-rank outputs scattered back by their index lists equal the cp_size = 1
  result (the full-vs-CP equality the TE PR's CP2 tests and torchtitan's
  loss comparison at CP degree 8 rely on);
* document independence: permuting documents permutes outputs, and changing
  one document's values leaves the others' outputs unchanged;
* closed forms: Q = 0 gives lse = ln(pos + 1) and out = the prefix mean of V;
  V = 1 gives out = 1; pad rows give out = 0 and lse = -inf;
* the GQA head map against K/V replicated with repeat_interleave.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import partition as P
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "attention_tiny.json")


def _rank_inputs(inp, strategy, cp, r):
    cup = inp.layout.cu_seqlens_padded
    idx = np.asarray(P.partition_index(strategy, cup.tolist(), cp, r), dtype=np.int64)
    q_loc = inp.q[torch.from_numpy(idx)]
    return idx, q_loc


def test_hand_worked_golden():
    g = json.load(open(GOLDEN))
    q = np.array(g["q"]); k = np.array(g["k"]); v = np.array(g["v"])
    idx = np.arange(q.shape[0])
    out, lse = A.attention_fwd(q, k, v, g["cu_seqlens"], g["cu_seqlens_padded"], idx, scale=g["scale"])
    np.testing.assert_allclose(out, np.array(g["out"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.array(g["lse"]), rtol=0, atol=1e-14)
    out2, lse2 = A.attention_bruteforce(q, k, v, g["cu_seqlens"], g["cu_seqlens_padded"], idx, scale=g["scale"])
    np.testing.assert_allclose(out2, np.array(g["out"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse2, np.array(g["lse"]), rtol=0, atol=1e-14)


@pytest.mark.parametrize("strategy", ["dcs", "nlb"])
def test_tiny_config_bruteforce(strategy):
    cfg = W.CONFIG_BY_NAME["tiny"]
    inp = W.make_attn_inputs(cfg, strategy)
    for r in range(cfg.cp):
        idx, q_loc = _rank_inputs(inp, strategy, cfg.cp, r)
        lay = inp.layout
        o1, l1 = A.attention_fwd(q_loc, inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded, idx)
        # the brute force is slow: check two heads' worth on a 16-dim slice of
        # the head dimension would change the scores, so use the full rows but
        # only a subset of rows
        rows = np.linspace(0, idx.shape[0] - 1, 9).astype(np.int64)
        o2, l2 = A.attention_bruteforce(q_loc[torch.from_numpy(rows)], inp.k, inp.v,
                                        lay.cu_seqlens, lay.cu_seqlens_padded, idx[rows])
        np.testing.assert_allclose(o1[rows], o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l1[:, rows], l2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_random_packs_bruteforce(seed):
    rng = np.random.default_rng(seed)
    cp = int(rng.choice([1, 2, 3]))
    lay = W.random_layout(rng, int(rng.integers(1, 5)), 13, 2 * cp, allow_empty=True)
    hkv = int(rng.choice([1, 2])); g = int(rng.choice([1, 2, 3])); hq = hkv * g; d = 4
    T = lay.T
    q = torch.from_numpy(rng.standard_normal((T, hq, d)))
    k = torch.from_numpy(rng.standard_normal((T, hkv, d)))
    v = torch.from_numpy(rng.standard_normal((T, hkv, d)))
    for strategy in ["dcs", "nlb"]:
        if strategy == "nlb" and T % cp:
            continue
        for r in range(cp):
            idx = np.asarray(P.partition_index(strategy, lay.cu_seqlens_padded.tolist(), cp, r))
            ql = q[torch.from_numpy(idx)] if idx.size else q[:0]
            o1, l1 = A.attention_fwd(ql, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, scale=0.7)
            o2, l2 = A.attention_bruteforce(ql, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, scale=0.7)
            np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
            np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("S,d", [(1, 8), (7, 16), (300, 64)])
def test_single_doc_cp1_is_textbook_causal(S, d):
    rng = np.random.default_rng(S)
    q = torch.from_numpy(rng.standard_normal((S, 3, d)))
    k = torch.from_numpy(rng.standard_normal((S, 3, d)))
    v = torch.from_numpy(rng.standard_normal((S, 3, d)))
    out, _ = A.attention_fwd(q, k, v, [0, S], [0, S], np.arange(S))
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None], v.permute(1, 0, 2)[None], is_causal=True)
    ref = ref[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("name", ["tiny", "t8192_mha16"])
@pytest.mark.parametrize("strategy", ["dcs", "nlb"])
def test_cp_scatter_equals_full(name, strategy):
    cfg = W.CONFIG_BY_NAME[name]
    inp = W.make_attn_inputs(cfg, strategy)
    lay = inp.layout
    T = lay.T
    # keep the heavier config cheap: two heads
    q, k, v = inp.q, inp.k, inp.v
    if name != "tiny":
        q, k, v = q[:, :2], k[:, :2], v[:, :2]
    full_o, full_l = A.attention_fwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, np.arange(T))
    back_o = np.zeros_like(full_o); back_l = np.zeros_like(full_l)
    for r in range(cfg.cp):
        idx = np.asarray(P.partition_index(strategy, lay.cu_seqlens_padded.tolist(), cfg.cp, r))
        o, l = A.attention_fwd(q[torch.from_numpy(idx)], k, v, lay.cu_seqlens, lay.cu_seqlens_padded, idx)
        back_o[idx] = o; back_l[:, idx] = l
    np.testing.assert_allclose(back_o, full_o, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(back_l), np.isinf(full_l))
    fin = np.isfinite(full_l)
    np.testing.assert_allclose(back_l[fin], full_l[fin], rtol=0, atol=1e-12)


def test_same_tokens_same_outputs_under_both_layouts():
    """The padded (DualChunkSwap) and unpadded (NO_LOAD_BALANCE) layouts of the
    same logical tokens give the same per-token results."""
    cfg = W.CONFIG_BY_NAME["tiny"]
    a = W.make_attn_inputs(cfg, "dcs"); b = W.make_attn_inputs(cfg, "nlb")
    oa, la = A.attention_fwd(a.q, a.k, a.v, a.layout.cu_seqlens, a.layout.cu_seqlens_padded, np.arange(a.layout.T))
    ob, lb = A.attention_fwd(b.q, b.k, b.v, b.layout.cu_seqlens, b.layout.cu_seqlens_padded, np.arange(b.layout.T))
    slots = W.physical_slots(a.layout)
    np.testing.assert_allclose(oa[slots], ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(la[:, slots], lb, rtol=0, atol=1e-12)


def test_document_permutation_and_independence():
    rng = np.random.default_rng(11)
    lengths = [5, 9, 3, 12]
    lay = W.make_layout(lengths)
    T = lay.T; hq = 2; d = 8
    q = rng.standard_normal((T, hq, d)); k = rng.standard_normal((T, hq, d)); v = rng.standard_normal((T, hq, d))
    o, l = A.attention_fwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, np.arange(T))
    # permute documents
    perm = [2, 0, 3, 1]
    cu = lay.cu_seqlens
    seg = [np.arange(cu[j], cu[j + 1]) for j in range(4)]
    order = np.concatenate([seg[j] for j in perm])
    lay2 = W.make_layout([lengths[j] for j in perm])
    o2, l2 = A.attention_fwd(q[order], k[order], v[order], lay2.cu_seqlens, lay2.cu_seqlens_padded, np.arange(T))
    np.testing.assert_allclose(o2, o[order], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l[:, order], rtol=0, atol=1e-12)
    # change document 1 only
    k3 = k.copy(); v3 = v.copy(); q3 = q.copy()
    k3[seg[1]] += 5.0; v3[seg[1]] -= 2.0; q3[seg[1]] *= 3.0
    o3, l3 = A.attention_fwd(q3, k3, v3, lay.cu_seqlens, lay.cu_seqlens_padded, np.arange(T))
    others = np.concatenate([seg[0], seg[2], seg[3]])
    np.testing.assert_array_equal(o3[others], o[others])
    np.testing.assert_array_equal(l3[:, others], l[:, others])
    assert not np.allclose(o3[seg[1]], o[seg[1]])


def test_zero_queries_closed_form():
    """Q = 0: every allowed score is 0, so lse = ln(pos + 1) and out is the
    mean of V over the document prefix."""
    lay = W.make_layout([6, 1, 10], 4)
    T = lay.T; rng = np.random.default_rng(3)
    q = np.zeros((T, 2, 4)); k = rng.standard_normal((T, 1, 4)); v = rng.standard_normal((T, 1, 4))
    o, l = A.attention_fwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, np.arange(T))
    cup = lay.cu_seqlens_padded; L = lay.lengths
    for j in range(3):
        for pos in range(int(L[j])):
            row = cup[j] + pos
            for h in range(2):
                assert abs(l[h, row] - math.log(pos + 1)) < 1e-13
                np.testing.assert_allclose(o[row, h], v[cup[j]:cup[j] + pos + 1, 0].mean(axis=0), atol=1e-13)
        for pos in range(int(L[j]), int(cup[j + 1] - cup[j])):
            row = cup[j] + pos
            assert np.all(o[row] == 0) and np.all(np.isneginf(l[:, row]))


def test_unit_values_closed_form():
    lay = W.make_layout([4, 11], 1)
    T = lay.T; rng = np.random.default_rng(4)
    q = rng.standard_normal((T, 2, 8)) * 3; k = rng.standard_normal((T, 2, 8)) * 3; v = np.ones((T, 2, 8))
    o, _ = A.attention_fwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, np.arange(T))
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-13)


def test_single_key_lse_is_score():
    rng = np.random.default_rng(5)
    lay = W.make_layout([1, 1, 1])
    q = rng.standard_normal((3, 1, 8)); k = rng.standard_normal((3, 1, 8)); v = rng.standard_normal((3, 1, 8))
    o, l = A.attention_fwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, np.arange(3), scale=0.5)
    for i in range(3):
        assert abs(l[0, i] - 0.5 * float(q[i, 0] @ k[i, 0])) < 1e-14
        np.testing.assert_array_equal(o[i, 0], v[i, 0])


def test_gqa_head_map_against_replicated_kv():
    rng = np.random.default_rng(6)
    lay = W.make_layout([7, 12])
    T = lay.T
    q = torch.from_numpy(rng.standard_normal((T, 6, 8)))
    k = torch.from_numpy(rng.standard_normal((T, 2, 8)))
    v = torch.from_numpy(rng.standard_normal((T, 2, 8)))
    o1, l1 = A.attention_fwd(q, k, v, lay.cu_seqlens, lay.cu_seqlens_padded, np.arange(T))
    kr = k.repeat_interleave(3, dim=1); vr = v.repeat_interleave(3, dim=1)
    o2, l2 = A.attention_fwd(q, kr, vr, lay.cu_seqlens, lay.cu_seqlens_padded, np.arange(T))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_rows_subset_matches_full():
    cfg = W.CONFIG_BY_NAME["tiny"]
    inp = W.make_attn_inputs(cfg, "dcs")
    lay = inp.layout
    idx = np.asarray(P.partition_index("dcs", lay.cu_seqlens_padded.tolist(), 2, 1))
    ql = inp.q[torch.from_numpy(idx)]
    o, l = A.attention_fwd(ql, inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded, idx)
    rows = [5, 0, 33, 65]
    o2, l2 = A.attention_fwd(ql, inp.k, inp.v, lay.cu_seqlens, lay.cu_seqlens_padded, idx, rows=rows)
    np.testing.assert_allclose(o2, o[rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l[:, rows], rtol=0, atol=1e-13)


def test_pair_count_closed_form():
    S = 1000
    assert A.unmasked_pairs(np.arange(S), [0, S], [0, S]) == S * (S + 1) // 2
    cfg = W.CONFIG_BY_NAME["tiny"]
    for s in ("dcs", "nlb"):
        lay = W.layout_for(cfg, s)
        tot = sum(A.unmasked_pairs(P.partition_index(s, lay.cu_seqlens_padded.tolist(), 2, r),
                                   lay.cu_seqlens, lay.cu_seqlens_padded) for r in range(2))
        assert tot == 37 * 38 // 2 + 91 * 92 // 2
