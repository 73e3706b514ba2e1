"""GPU reorder vs the oracle's byte gather: bit exact for every row width
and alignment path, the multi-tensor launch, the int64 id tensors of every
workload, the full-size activation reorders (sampled rows), and the
out-of-range index check."""
import numpy as np
import pytest
import torch

from oracle import partition as P
from oracle import reorder as R
import workloads as W
from gpu_common import cuda_or_skip, load_lib, new_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("row_bytes", [1, 2, 3, 4, 8, 12, 16, 48, 200, 512, 8192, 16400])
def test_reorder_widths(row_bytes):
    dev = cuda_or_skip(); cp = load_lib()
    rng = np.random.default_rng(row_bytes)
    n_src, n = 517, 333
    src = rng.integers(0, 256, size=(n_src, row_bytes), dtype=np.uint8)
    idx = rng.integers(0, n_src, size=n).astype(np.int32)
    err = new_err(dev)
    got = cp.cp_reorder(torch.from_numpy(src).to(dev), torch.from_numpy(idx).to(dev), err=err).cpu().numpy()
    assert got.tobytes() == R.reorder(src, idx).tobytes()
    assert err.cpu().tolist() == [0, 0]


def test_reorder_unaligned_base():
    dev = cuda_or_skip(); cp = load_lib()
    rng = np.random.default_rng(0)
    raw = torch.from_numpy(rng.integers(0, 256, size=64 * 40 + 3, dtype=np.uint8)).to(dev)
    src = raw[3:3 + 64 * 40].view(64, 40)          # base pointer 3 bytes past an allocation
    idx = torch.from_numpy(rng.integers(0, 64, size=50).astype(np.int32)).to(dev)
    got = cp.cp_reorder(src, idx).cpu().numpy()
    assert got.tobytes() == R.reorder(src.cpu().numpy(), idx.cpu().numpy()).tobytes()


@pytest.mark.parametrize("cfg", W.CONFIGS, ids=lambda c: c.name)
def test_ids_reorder_multi(cfg):
    dev = cuda_or_skip(); cp = load_lib()
    for s in cfg.strategies:
        lay = W.layout_for(cfg, s)
        ids, labels, pos = W.make_ids_logical(cfg.seed, lay)
        phys = [W.to_physical(t, lay, -1) for t in (ids, labels, pos)]
        dev_t = [t.to(dev) for t in phys]
        cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
        err = new_err(dev)
        for r in range(cfg.cp):
            idx, outs = cp.get_batch_on_this_cp_rank(cup, *dev_t, cp_size=cfg.cp, rank=r, strategy=s, err=err)
            ref_idx = P.partition_index(s, lay.cu_seqlens_padded.tolist(), cfg.cp, r)
            for o, src in zip(outs, phys):
                assert o.cpu().numpy().tobytes() == R.reorder(src.numpy(), ref_idx).tobytes()
        assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("name", ["padded48_gqa32x8", "long131072_h8"])
def test_activation_reorder_full_size(name):
    """[T, 4096] / [T, 8192] bf16 activations at full size for every rank:
    every row of the library's gather equals, bit for bit (compared on the
    device as int16 bit patterns), the source rows that the oracle's index
    list names, gathered by torch's index_select."""
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME[name]
    s = cfg.strategies[0]
    lay = W.layout_for(cfg, s)
    act = W.make_activations(cfg.seed, lay.T, cfg.act_width, device="cuda:0")
    bits = act.view(torch.int16)
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    err = new_err(dev)
    out = None
    for r in range(cfg.cp):
        ref_idx = np.asarray(P.partition_index(s, lay.cu_seqlens_padded.tolist(), cfg.cp, r), dtype=np.int64)
        idx = cp.cp_partition_index(s, cup, lay.T, cfg.cp, r, err=err)
        out = cp.cp_reorder(act, idx, out=out, err=err)
        want = torch.index_select(bits, 0, torch.from_numpy(ref_idx).to(dev))
        assert torch.equal(out.view(torch.int16), want), f"{name}: rank {r} differs"
    assert err.cpu().tolist() == [0, 0]


def test_reorder_index_out_of_range_recorded():
    dev = cuda_or_skip(); cp = load_lib()
    src = torch.arange(40, dtype=torch.int64, device=dev).view(10, 4)
    idx = torch.tensor([1, 12, 3, -1], dtype=torch.int32, device=dev)
    out = torch.full((4, 4), 7, dtype=torch.int64, device=dev)
    err = new_err(dev)
    cp.cp_reorder(src, idx, out=out, err=err)
    e = err.cpu().tolist()
    assert e[0] == -7 and e[1] in (1, 3)
    o = out.cpu()
    assert o[0].tolist() == [4, 5, 6, 7] and o[2].tolist() == [12, 13, 14, 15]
    assert o[1].tolist() == [7] * 4 and o[3].tolist() == [7] * 4
