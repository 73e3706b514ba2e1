"""Pins for the partition oracle (no GPU).

The oracle's loop construction is checked against (i) hand-worked cases in
tests/golden/partition_cases.json, (ii) an independent ownership-marking
construction, (iii) the invariants the pages imply: disjoint per-rank slices
that cover every physical token once, equal local lengths (TransformerEngine
PR #3221, "Scope and constraints"), (iv) special cases: cp_size = 1 is the
identity, NO_LOAD_BALANCE concatenated rank-major is the identity, and for
one document DualChunkSwap is the head-tail split (torchtitan PR #2144,
"Summary").
"""
import json
import os

import numpy as np
import pytest

from oracle import partition as P
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "partition_cases.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["note"][:40])
def test_hand_worked_cases(case):
    cp = case["cp_size"]
    for r in range(cp):
        got = P.partition_index(case["strategy"], case["cu_seqlens_padded"], cp, r)
        assert got == case["ranks"][r]


@pytest.mark.parametrize("case", _golden()["errors"], ids=lambda c: c["why"][:40])
def test_hand_worked_errors(case):
    with pytest.raises(P.PartitionError):
        P.partition_index(case["strategy"], case["cu_seqlens_padded"], case["cp_size"], 0)


def _owner_marking(cup, cp):
    """Independent construction: label every physical slot with the rank that
    owns its chunk, then list each rank's slots in increasing physical order
    (chunk r precedes chunk 2cp-1-r inside a document, and documents are in
    pack order, so the owned slots of a rank are increasing)."""
    T = cup[-1]
    owner = np.full(T, -1, dtype=np.int64)
    for j in range(len(cup) - 1):
        s, e = cup[j], cup[j + 1]
        c = (e - s) // (2 * cp)
        for t in range(s, e):
            chunk = (t - s) // c
            owner[t] = chunk if chunk < cp else 2 * cp - 1 - chunk
    return [np.nonzero(owner == r)[0].tolist() for r in range(cp)]


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("seed", range(6))
def test_dcs_matches_owner_marking(cp, seed):
    rng = np.random.default_rng(seed + 100 * cp)
    lay = W.random_layout(rng, n_docs=int(rng.integers(1, 7)), max_len=60, pad_multiple=2 * cp,
                          allow_empty=True)
    cup = lay.cu_seqlens_padded.tolist()
    expect = _owner_marking(cup, cp)
    for r in range(cp):
        assert P.dual_chunk_swap_indices(cup, cp, r) == expect[r]


@pytest.mark.parametrize("strategy", ["dcs", "nlb"])
@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
def test_disjoint_cover_equal_lengths(strategy, cp):
    rng = np.random.default_rng(7 * cp)
    for _ in range(5):
        if strategy == "dcs":
            lay = W.random_layout(rng, int(rng.integers(1, 9)), 80, 2 * cp, allow_empty=True)
        else:
            lay = W.random_layout(rng, int(rng.integers(1, 9)), 80, 1)
            extra = (-lay.T) % cp
            if extra:
                lay = W.make_layout(list(lay.lengths[:-1]) + [int(lay.lengths[-1]) + extra])
        cup = lay.cu_seqlens_padded.tolist()
        T = cup[-1]
        lists = [P.partition_index(strategy, cup, cp, r) for r in range(cp)]
        n = P.local_tokens(strategy, T, cp)
        assert all(len(x) == n for x in lists)
        flat = sorted(i for x in lists for i in x)
        assert flat == list(range(T))


@pytest.mark.parametrize("strategy", ["dcs", "nlb"])
def test_cp1_identity(strategy):
    lay = W.make_layout([5, 9, 1], 2)
    cup = lay.cu_seqlens_padded.tolist()
    assert P.partition_index(strategy, cup, 1, 0) == list(range(cup[-1]))


def test_nlb_rank_major_concat_is_identity():
    cup = [0, 7, 20, 24]
    cat = []
    for r in range(4):
        cat += P.partition_index("nlb", cup, 4, r)
    assert cat == list(range(24))


@pytest.mark.parametrize("cp", [1, 2, 4, 8, 16])
def test_single_document_is_head_tail(cp):
    """torchtitan's head-tail balancer: one sequence of length S split into
    2*cp equal pieces, rank r keeps pieces r and 2cp-1-r (numpy array_split
    does the splitting here, independently of the oracle's index arithmetic)."""
    S = 2 * cp * 5
    pieces = np.array_split(np.arange(S), 2 * cp)
    for r in range(cp):
        expect = np.concatenate([pieces[r], pieces[2 * cp - 1 - r]]).tolist()
        assert P.dual_chunk_swap_indices([0, S], cp, r) == expect


@pytest.mark.parametrize("cp", [2, 4, 8])
def test_local_prefix_is_cup_over_cp(cp):
    """The rank-local layout is documents in pack order, each holding
    P_j / cp of its slots: splitting a rank's list at cup/cp gives, for
    document j, exactly the slots of that document it owns."""
    lay = W.make_layout([3, 17, 40, 8], 2 * cp)
    cup = lay.cu_seqlens_padded.tolist()
    lcu = P.local_cu_seqlens_padded(cup, cp)
    for r in range(cp):
        lst = P.dual_chunk_swap_indices(cup, cp, r)
        for j in range(len(cup) - 1):
            part = lst[lcu[j]:lcu[j + 1]]
            assert all(cup[j] <= x < cup[j + 1] for x in part)
            assert len(part) == (cup[j + 1] - cup[j]) // cp


def test_every_config_partitions():
    for cfg in W.CONFIGS:
        for s in cfg.strategies:
            lay = W.layout_for(cfg, s)
            cup = lay.cu_seqlens_padded.tolist()
            T = cup[-1]
            n = P.local_tokens(s, T, cfg.cp)
            seen = np.zeros(T, dtype=np.int64)
            for r in range(cfg.cp):
                lst = P.partition_index(s, cup, cfg.cp, r)
                assert len(lst) == n
                seen[np.asarray(lst)] += 1
            assert (seen == 1).all()


def _restore_cases():
    return _golden()["restore"]["cases"]


@pytest.mark.parametrize("case", _restore_cases(), ids=lambda c: c["note"][:40])
def test_restore_hand_worked(case):
    assert P.restore_index(case["strategy"], case["cu_seqlens_padded"], case["cp_size"]) == case["restore"]


@pytest.mark.parametrize("strategy", ["dcs", "nlb", "mirrored"])
@pytest.mark.parametrize("cp", [1, 2, 3, 4])
def test_restore_round_trip(strategy, cp):
    """Gathering every rank's slice rank-major and then reading it through the
    restore index gives back the token order; for NO_LOAD_BALANCE the restore
    index is the identity (no K/V reorder)."""
    rng = np.random.default_rng(31 * cp)
    for _ in range(4):
        pad = 2 * cp if strategy == "dcs" else 1
        lay = W.random_layout(rng, int(rng.integers(1, 6)), 50, pad, allow_empty=True)
        cup = lay.cu_seqlens_padded.tolist()
        mult = 2 * cp if strategy == "mirrored" else cp
        if cup[-1] % mult:
            continue
        x = rng.integers(0, 1 << 30, size=cup[-1])
        gathered = np.concatenate([x[P.partition_index(strategy, cup, cp, r)] for r in range(cp)])
        restore = P.restore_index(strategy, cup, cp)
        assert np.array_equal(gathered[restore], x)
        if strategy == "nlb":
            assert restore == list(range(cup[-1]))


@pytest.mark.parametrize("cp", [1, 2, 4, 8])
def test_mirrored_is_head_tail_of_whole_buffer(cp):
    T = 2 * cp * 7
    pieces = np.array_split(np.arange(T), 2 * cp)
    cup = [0, 3, 10, T]          # document boundaries do not matter
    for r in range(cp):
        expect = np.concatenate([pieces[r], pieces[2 * cp - 1 - r]]).tolist()
        assert P.partition_index("mirrored", cup, cp, r) == expect
