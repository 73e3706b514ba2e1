"""Pins for the reorder oracle (no GPU): numpy take against a byte loop,
and the round trip of scattering per-rank results back by their index
lists, which must reproduce the source bit for bit."""
import numpy as np
import pytest

from oracle import partition as P
from oracle import reorder as R
import workloads as W


@pytest.mark.parametrize("row_bytes", [1, 3, 8, 16, 24, 130])
def test_take_equals_byte_loop(row_bytes):
    rng = np.random.default_rng(row_bytes)
    n = 37
    src = rng.integers(0, 256, size=(n, row_bytes), dtype=np.uint8)
    idx = rng.integers(0, n, size=50)
    got = R.reorder(src, idx)
    assert got.tobytes() == R.reorder_loop(src.tobytes(), row_bytes, idx.tolist())


@pytest.mark.parametrize("strategy", ["dcs", "nlb"])
def test_scatter_back_round_trip(strategy):
    cfg = W.CONFIG_BY_NAME["t8192_mha16"]
    lay = W.layout_for(cfg, strategy)
    ids, labels, pos = W.make_ids_logical(cfg.seed, lay)
    ids = W.to_physical(ids, lay, -1).numpy()
    T = lay.T
    back = np.zeros_like(ids)
    for r in range(cfg.cp):
        idx = P.partition_index(strategy, lay.cu_seqlens_padded.tolist(), cfg.cp, r)
        part = R.reorder(ids, idx)
        back[np.asarray(idx)] = part
    assert back.tobytes() == ids.tobytes()


def test_bf16_bits_preserved():
    import torch
    x = W.randn_bf16(9, 1, (20, 4, 8))
    raw = x.view(torch.int16).numpy()
    raw[3, 0, 0] = np.int16(0x7fc1)          # a NaN payload must survive the copy
    idx = [3, 3, 0, 19]
    got = R.reorder(raw, idx)
    assert got.tobytes() == b"".join(raw[i].tobytes() for i in idx)


def test_out_of_range_index_rejected():
    with pytest.raises(IndexError):
        R.reorder(np.zeros((4, 2)), [0, 4])
