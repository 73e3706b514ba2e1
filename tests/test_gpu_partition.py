"""GPU partition index vs the oracle: bit exact, every workload, every rank,
both strategies; rank = -1 gives all ranks rank-major; device-side checks of
malformed offsets land in the error word."""
import numpy as np
import pytest
import torch

from oracle import partition as P
import workloads as W
from gpu_common import cuda_or_skip, load_lib, new_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", W.CONFIGS, ids=lambda c: c.name)
def test_partition_every_config(cfg):
    dev = cuda_or_skip(); cp = load_lib()
    for s in cfg.strategies:
        lay = W.layout_for(cfg, s)
        cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
        err = new_err(dev)
        for r in range(cfg.cp):
            got = cp.cp_partition_index(s, cup, lay.T, cfg.cp, r, err=err).cpu().numpy()
            ref = np.asarray(P.partition_index(s, lay.cu_seqlens_padded.tolist(), cfg.cp, r), dtype=np.int32)
            assert np.array_equal(got, ref), (s, r)
        allr = cp.cp_partition_index(s, cup, lay.T, cfg.cp, -1, err=err).cpu().numpy()
        ref = np.concatenate([P.partition_index(s, lay.cu_seqlens_padded.tolist(), cfg.cp, r)
                              for r in range(cfg.cp)]).astype(np.int32)
        assert np.array_equal(allr, ref)
        assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("cpsize", [1, 2, 3, 5, 8])
def test_partition_random_packs(cpsize):
    dev = cuda_or_skip(); cp = load_lib()
    rng = np.random.default_rng(cpsize)
    for _ in range(8):
        lay = W.random_layout(rng, int(rng.integers(1, 40)), 300, 2 * cpsize, allow_empty=True)
        cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
        for s in ("dcs", "nlb"):
            if lay.T % cpsize:
                continue
            for r in range(cpsize):
                got = cp.cp_partition_index(s, cup, lay.T, cpsize, r).cpu().numpy()
                ref = np.asarray(P.partition_index(s, lay.cu_seqlens_padded.tolist(), cpsize, r), dtype=np.int32)
                assert np.array_equal(got, ref)


def test_partition_device_checks():
    dev = cuda_or_skip(); cp = load_lib()
    # document 1 has padded length 6, not divisible by 2*cp_size = 4
    cup = torch.tensor([0, 8, 14, 16], dtype=torch.int32, device=dev)
    err = new_err(dev)
    cp.cp_partition_index("dcs", cup, 16, 2, 0, err=err)
    assert err.cpu().tolist() == [-2, 1]
    # last offset differs from T
    cup = torch.tensor([0, 8, 12], dtype=torch.int32, device=dev)
    err = new_err(dev)
    cp.cp_partition_index("nlb", cup, 16, 2, 1, err=err)
    assert err.cpu().tolist()[0] == -6
    # decreasing offsets
    cup = torch.tensor([0, 8, 4, 16], dtype=torch.int32, device=dev)
    err = new_err(dev)
    cp.cp_partition_index("dcs", cup, 16, 2, 0, err=err)
    assert err.cpu().tolist()[0] == -6


@pytest.mark.parametrize("cfg", W.CONFIGS, ids=lambda c: c.name)
def test_packed_mirrored_every_config(cfg):
    dev = cuda_or_skip(); cp = load_lib()
    lay = W.layout_for(cfg, "mirrored")
    if lay.T % (2 * cfg.cp):
        # the split needs T % (2 * cp_size) == 0 whatever the documents; the
        # padded buffer of the 48-document pack has it, the unpadded one not
        lay = W.layout_for(cfg, "dcs")
    assert lay.T % (2 * cfg.cp) == 0
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    err = new_err(dev)
    for r in range(cfg.cp):
        got = cp.cp_partition_index("mirrored", cup, lay.T, cfg.cp, r, err=err).cpu().numpy()
        ref = np.asarray(P.partition_index("mirrored", lay.cu_seqlens_padded.tolist(), cfg.cp, r), dtype=np.int32)
        assert np.array_equal(got, ref)
    assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("cfg", W.CONFIGS, ids=lambda c: c.name)
def test_restore_index_every_config(cfg):
    dev = cuda_or_skip(); cp = load_lib()
    for s in W.ALL_STRATEGIES:
        if s not in cfg.strategies and s != "mirrored":
            continue
        lay = W.layout_for(cfg, s)
        if s == "mirrored" and lay.T % (2 * cfg.cp):
            continue
        cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
        err = new_err(dev)
        got = cp.cp_restore_index(s, cup, lay.T, cfg.cp, err=err).cpu().numpy()
        ref = np.asarray(P.restore_index(s, lay.cu_seqlens_padded.tolist(), cfg.cp), dtype=np.int32)
        assert np.array_equal(got, ref), s
        assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("name,strategy", [("long131072_h8", "dcs"), ("padded48_gqa32x8", "dcs"),
                                           ("t32768_lognormal_gqa32x8", "mirrored"),
                                           ("t32768_lognormal_gqa32x8", "nlb")])
def test_kv_restore_round_trip_full_size(name, strategy):
    """Simulated all-gather of every rank's K slice (rank-major), then the
    restore gather: K comes back bit for bit."""
    dev = cuda_or_skip(); cp = load_lib()
    cfg = W.CONFIG_BY_NAME[name]
    lay = W.layout_for(cfg, strategy)
    cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
    k = W.make_activations(cfg.seed, lay.T, cfg.hkv * cfg.d, device="cuda:0")
    err = new_err(dev)
    idx_all = cp.cp_partition_index(strategy, cup, lay.T, cfg.cp, -1, err=err)
    gathered = cp.cp_reorder(k, idx_all, err=err)
    restore = cp.cp_restore_index(strategy, cup, lay.T, cfg.cp, err=err)
    back = cp.cp_reorder(gathered, restore, err=err)
    assert torch.equal(back.view(torch.int16), k.view(torch.int16))
    assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("n_docs", [4095, 4096, 6000])
def test_many_documents(n_docs):
    """Thousands of short documents (deep binary searches over the offset
    table), empty documents mixed in: partition and restore index bit exact."""
    dev = cuda_or_skip(); cp = load_lib()
    rng = np.random.default_rng(n_docs)
    for cpsize in (2, 3):
        lay = W.random_layout(rng, n_docs, 10, 2 * cpsize, allow_empty=True)
        cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
        err = new_err(dev)
        for s in ("dcs", "nlb"):
            if lay.T % cpsize:
                continue
            for r in range(cpsize):
                got = cp.cp_partition_index(s, cup, lay.T, cpsize, r, err=err).cpu().numpy()
                ref = np.asarray(P.partition_index(s, lay.cu_seqlens_padded.tolist(), cpsize, r), dtype=np.int32)
                assert np.array_equal(got, ref), (s, cpsize, r)
            got = cp.cp_restore_index(s, cup, lay.T, cpsize, err=err).cpu().numpy()
            ref = np.asarray(P.restore_index(s, lay.cu_seqlens_padded.tolist(), cpsize), dtype=np.int32)
            assert np.array_equal(got, ref), (s, cpsize)
        assert err.cpu().tolist() == [0, 0]


@pytest.mark.parametrize("cfg", W.CONFIGS, ids=lambda c: c.name)
def test_fused_partition_reorder_every_config(cfg):
    """cp_partition_reorder_multi: the index list equals the oracle's and the
    gathered Q / ids equal the oracle's byte gather, bit exact, for every
    strategy and rank (the packed mirrored split where T allows it)."""
    from oracle import reorder as R
    dev = cuda_or_skip(); cp = load_lib()
    strategies = list(cfg.strategies) + ([] if "mirrored" in cfg.strategies else ["mirrored"])
    for s in strategies:
        lay = W.layout_for(cfg, s)
        if s == "mirrored" and lay.T % (2 * cfg.cp):
            continue
        inp = W.make_attn_inputs(cfg, s)
        ids = torch.arange(lay.T, dtype=torch.int64) * 7 + 3
        cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
        q = inp.q.to(dev)
        idv = ids.to(dev)
        err = new_err(dev)
        for r in range(cfg.cp):
            idx, (q_loc, ids_loc) = cp.cp_partition_reorder_multi(s, cup, lay.T, cfg.cp, r, [q, idv], err=err)
            ref_idx = np.asarray(P.partition_index(s, lay.cu_seqlens_padded.tolist(), cfg.cp, r), dtype=np.int32)
            assert np.array_equal(idx.cpu().numpy(), ref_idx), (s, r)
            assert q_loc.cpu().view(torch.int16).numpy().tobytes() == \
                R.reorder(inp.q.view(torch.int16).numpy().reshape(lay.T, -1), ref_idx).tobytes(), (s, r)
            assert np.array_equal(ids_loc.cpu().numpy(), ids.numpy()[ref_idx]), (s, r)
        assert err.cpu().tolist() == [0, 0]


def test_fused_partition_reorder_random_packs_and_checks():
    """Random packs with empty documents (bit exact against the separate
    calls), and the device check of non-divisible DualChunkSwap lengths."""
    dev = cuda_or_skip(); cp = load_lib()
    rng = np.random.default_rng(11)
    for cpsize in (1, 2, 3, 5):
        for _ in range(4):
            lay = W.random_layout(rng, int(rng.integers(1, 60)), 300, 2 * cpsize, allow_empty=True)
            if lay.T == 0:
                continue
            cup = torch.from_numpy(lay.cu_seqlens_padded).to(dev)
            x = torch.from_numpy(rng.integers(0, 1 << 30, size=(lay.T, 3), dtype=np.int32)).to(dev)
            for s in ("dcs", "nlb"):
                if lay.T % cpsize:
                    continue
                for r in range(cpsize):
                    idx, (got,) = cp.cp_partition_reorder_multi(s, cup, lay.T, cpsize, r, [x])
                    ref = cp.cp_partition_index(s, cup, lay.T, cpsize, r)
                    assert torch.equal(idx, ref)
                    assert torch.equal(got, x[ref.long()])
    # document 1 has padded length 6, not divisible by 2*cp_size = 4
    cup = torch.tensor([0, 8, 14, 16], dtype=torch.int32, device=dev)
    x = torch.zeros((16, 4), dtype=torch.int32, device=dev)
    err = new_err(dev)
    cp.cp_partition_reorder_multi("dcs", cup, 16, 2, 0, [x], err=err)
    assert err.cpu().tolist()[0] == -2
