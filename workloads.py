"""Seeded synthetic inputs for packed-THD context-parallel attention.

This module only *builds inputs*: document lengths, the THD offset arrays
(`cu_seqlens`, `cu_seqlens_padded`), bf16 Q/K/V tensors and int64 id tensors.
It contains none of the method's arithmetic (no partitioning, no reordering,
no attention) and is the one module shared by the float64 oracle's tests and
by the CUDA path's tests and benchmark.

Workloads follow the five shapes of the packed-THD study (TransformerEngine
PR #3221 "Add no-load-balance THD all-gather CP", sections "Why" and "Scope
and constraints"): bf16 N(0,1) Q/K/V, document lengths not divisible by
2*cp_size, THD layout where `T` is the total number of packed tokens
(TransformerEngine issue #3564, "Problem").

Random draws use numpy's PCG64 ``default_rng`` so that the same seed gives the
same bits on x86 and Arm hosts.

Layouts
-------
* ``logical``: documents back to back, no padding (`cu_seqlens`).
* ``padded``: every document padded up to a multiple of ``pad_multiple``
  (`cu_seqlens_padded`); pad slots hold zeros (bf16) or -1 (int64 ids).
  DualChunkSwap runs on the padded layout with ``pad_multiple = 2*cp_size``;
  NO_LOAD_BALANCE and the packed mirrored partition run on the logical layout
  (``pad_between_seqs=False``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

DUAL_CHUNK_SWAP = "dcs"
NO_LOAD_BALANCE = "nlb"
PACKED_MIRRORED = "mirrored"
STRATEGIES = (DUAL_CHUNK_SWAP, NO_LOAD_BALANCE)
ALL_STRATEGIES = (DUAL_CHUNK_SWAP, NO_LOAD_BALANCE, PACKED_MIRRORED)


@dataclasses.dataclass(frozen=True)
class Config:
    """One packed-THD workload shape."""

    name: str
    seed: int
    lengths: tuple           # actual document lengths L_j
    hq: int
    hkv: int
    d: int
    cp: int
    strategies: tuple        # strategies the workload is run under
    pad_multiple_dcs: int    # padding used for the DualChunkSwap layout
    act_width: int = 0       # activation row width (elements) for the reorder workload

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))


# --------------------------------------------------------------------------
# document-length compositions
# --------------------------------------------------------------------------

def lengths_composition(seed: int, total: int, parts: int, min_len: int, forbid_mod: int) -> List[int]:
    """Rejection-sample ``parts-1`` distinct cut points in [1, total-1].

    Accept the first draw where every part is >= ``min_len`` and none is
    divisible by ``forbid_mod``.
    """
    rng = np.random.default_rng(seed)
    while True:
        cuts = np.sort(rng.choice(np.arange(1, total), size=parts - 1, replace=False))
        p = np.diff(np.concatenate([[0], cuts, [total]]))
        if (p >= min_len).all() and not (p % forbid_mod == 0).any():
            return [int(x) for x in p]


def lengths_lognormal(seed: int, total: int, median: float, sigma: float, lo: int, hi: int) -> List[int]:
    """Draw lognormal lengths (rounded, clipped to [lo, hi]) until ``total`` is
    reached; the last document is truncated so the lengths sum to ``total``."""
    rng = np.random.default_rng(seed)
    out: List[int] = []
    while sum(out) < total:
        x = rng.lognormal(math.log(median), sigma)
        out.append(int(np.clip(np.rint(x), lo, hi)))
    out[-1] -= sum(out) - total
    return out


def lengths_uniform(seed: int, n: int, lo: int, hi: int) -> List[int]:
    """``n`` lengths uniform in [lo, hi] inclusive."""
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def _build_configs():
    c1 = Config("tiny", 1, (37, 91), 2, 2, 64, 2, STRATEGIES, 4)
    c2 = Config("t8192_mha16", 2, tuple(lengths_composition(2, 8192, 16, 64, 8)), 16, 16, 128, 4,
                STRATEGIES, 8)
    c3 = Config("t32768_lognormal_gqa32x8", 3,
                tuple(lengths_lognormal(3, 32768, 2048.0, 1.0, 64, 16384)), 32, 8, 128, 8,
                STRATEGIES, 16)
    c4 = Config("padded48_gqa32x8", 4, tuple(lengths_uniform(4, 48, 256, 4096)), 32, 8, 128, 8,
                (DUAL_CHUNK_SWAP,), 16, act_width=4096)
    c5 = Config("long131072_h8", 5, (131072,), 8, 8, 128, 16, STRATEGIES, 32, act_width=8192)
    return [c1, c2, c3, c4, c5]


CONFIGS = _build_configs()
CONFIG_BY_NAME = {c.name: c for c in CONFIGS}


# --------------------------------------------------------------------------
# THD offset arrays
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Layout:
    """Physical THD layout of a pack of documents."""

    lengths: np.ndarray       # int64 [N] actual lengths
    cu_seqlens: np.ndarray    # int32 [N+1] prefix sums of actual lengths
    cu_seqlens_padded: np.ndarray  # int32 [N+1] prefix sums of padded lengths (physical offsets)

    @property
    def num_docs(self) -> int:
        return int(self.lengths.shape[0])

    @property
    def T(self) -> int:
        return int(self.cu_seqlens_padded[-1])


def make_layout(lengths: Sequence[int], pad_multiple: int = 1) -> Layout:
    """Prefix sums of the actual lengths and of the lengths rounded up to
    ``pad_multiple`` (input construction: the offset arrays every THD call takes)."""
    L = np.asarray(lengths, dtype=np.int64)
    padded = ((L + pad_multiple - 1) // pad_multiple) * pad_multiple
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    cup = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
    return Layout(L, cu, cup)


def layout_for(cfg: Config, strategy: str) -> Layout:
    if strategy == DUAL_CHUNK_SWAP:
        return make_layout(cfg.lengths, cfg.pad_multiple_dcs)
    return make_layout(cfg.lengths, 1)


def physical_slots(layout: Layout) -> np.ndarray:
    """Physical slot of every logical token, in logical order (int64 [sum L])."""
    parts = [np.arange(layout.cu_seqlens_padded[j], layout.cu_seqlens_padded[j] + layout.lengths[j])
             for j in range(layout.num_docs)]
    if not parts:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate(parts).astype(np.int64)


def to_physical(x_logical: torch.Tensor, layout: Layout, fill=0) -> torch.Tensor:
    """Scatter a logical-order tensor [sum L, ...] into the physical layout [T, ...]."""
    out = torch.full((layout.T,) + tuple(x_logical.shape[1:]), fill, dtype=x_logical.dtype)
    out[torch.from_numpy(physical_slots(layout))] = x_logical
    return out


# --------------------------------------------------------------------------
# tensors
# --------------------------------------------------------------------------

def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def randn_bf16(seed: int, stream: int, shape, scale: float = 1.0) -> torch.Tensor:
    """N(0, scale^2) float32 draws rounded to bf16 (round-to-nearest-even)."""
    a = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return torch.from_numpy(a).to(torch.bfloat16)


def make_qkv_logical(seed: int, total: int, hq: int, hkv: int, d: int):
    """Logical-order bf16 Q [total,hq,d], K/V [total,hkv,d] ~ N(0,1)."""
    q = randn_bf16(seed, 1, (total, hq, d))
    k = randn_bf16(seed, 2, (total, hkv, d))
    v = randn_bf16(seed, 3, (total, hkv, d))
    return q, k, v


def make_ids_logical(seed: int, layout: Layout, vocab: int = 32000):
    """int64 input_ids (uniform in [0, vocab)), labels (ids shifted by one within
    the document, last = -100) and position_ids (position within the document)."""
    rng = _rng(seed, 4)
    total = int(layout.lengths.sum())
    ids = rng.integers(0, vocab, size=total, dtype=np.int64)
    labels = np.full(total, -100, dtype=np.int64)
    pos = np.zeros(total, dtype=np.int64)
    off = 0
    for L in layout.lengths.tolist():
        if L > 1:
            labels[off:off + L - 1] = ids[off + 1:off + L]
        pos[off:off + L] = np.arange(L)
        off += L
    return torch.from_numpy(ids), torch.from_numpy(labels), torch.from_numpy(pos)


@dataclasses.dataclass
class AttnInputs:
    cfg: Config
    strategy: str
    layout: Layout
    q: torch.Tensor   # physical [T, hq, d] bf16 (pads zero)
    k: torch.Tensor   # physical [T, hkv, d] bf16
    v: torch.Tensor


def make_attn_inputs(cfg: Config, strategy: str) -> AttnInputs:
    """Physical-layout bf16 Q/K/V for ``cfg`` under ``strategy``. The logical
    token values are the same under both strategies (matched inputs)."""
    layout = layout_for(cfg, strategy)
    q, k, v = make_qkv_logical(cfg.seed, cfg.total_tokens, cfg.hq, cfg.hkv, cfg.d)
    if layout.T != cfg.total_tokens:
        q, k, v = (to_physical(t, layout, 0) for t in (q, k, v))
    return AttnInputs(cfg, strategy, layout, q, k, v)


def make_activations(seed: int, T: int, width: int, device: Optional[str] = None) -> torch.Tensor:
    """bf16 [T, width] ~ N(0,1) activations for the reorder workload.

    On a CUDA device the draw uses torch's seeded device generator (the values
    only need to be arbitrary bits for a bit-exact copy check)."""
    if device is not None and device.startswith("cuda"):
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000 + 5)
        return torch.randn((T, width), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return randn_bf16(seed, 5, (T, width))


def random_layout(rng: np.random.Generator, n_docs: int, max_len: int, pad_multiple: int,
                  allow_empty: bool = False) -> Layout:
    """A small random pack for property tests."""
    lo = 0 if allow_empty else 1
    L = rng.integers(lo, max_len + 1, size=n_docs)
    return make_layout(L.tolist(), pad_multiple)
