"""The seeded workload recipe: shapes and constraints of the five packed
workloads (no GPU)."""
import numpy as np

import workloads as W


def test_composition_recipe():
    c = W.CONFIG_BY_NAME["t8192_mha16"]
    L = np.array(c.lengths)
    assert L.sum() == 8192 and len(L) == 16
    assert (L >= 64).all() and not (L % (2 * c.cp) == 0).any()
    assert c.lengths == (251, 863, 630, 269, 491, 469, 271, 1771, 378, 1002, 612, 209, 101, 196, 427, 252)


def test_lognormal_recipe():
    c = W.CONFIG_BY_NAME["t32768_lognormal_gqa32x8"]
    assert sum(c.lengths) == 32768
    assert all(64 <= x <= 16384 for x in c.lengths[:-1])
    assert c.lengths == (15765, 159, 3111, 1161, 1302, 1651, 272, 1624, 862, 6861)


def test_padded_recipe():
    c = W.CONFIG_BY_NAME["padded48_gqa32x8"]
    assert len(c.lengths) == 48 and all(256 <= x <= 4096 for x in c.lengths)
    lay = W.layout_for(c, "dcs")
    P = np.diff(lay.cu_seqlens_padded)
    assert (P % 16 == 0).all() and (P >= lay.lengths).all()
    assert lay.T == 120272


def test_layouts_and_matched_inputs():
    c = W.CONFIG_BY_NAME["tiny"]
    a = W.make_attn_inputs(c, "dcs"); b = W.make_attn_inputs(c, "nlb")
    assert a.layout.T == 132 and b.layout.T == 128
    slots = W.physical_slots(a.layout)
    assert (a.q[slots] == b.q).all() and (a.k[slots] == b.k).all()
    pad = np.setdiff1d(np.arange(132), slots)
    assert (a.q[pad] == 0).all()


def test_determinism():
    x1 = W.randn_bf16(5, 1, (3, 4)); x2 = W.randn_bf16(5, 1, (3, 4))
    assert (x1.view(-1) == x2.view(-1)).all()
