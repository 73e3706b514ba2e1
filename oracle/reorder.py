"""Reorder (gather) oracle.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The per-rank slicing of THD tensors (TransformerEngine PR #3221, "How to
use": get_batch_on_this_cp_rank over input_ids, labels, position_ids; the CPU
dataloader path selects rows by the rank's index list) is a row gather:
dst[i, :] = src[idx[i], :], byte for byte, for any row width.
"""
from __future__ import annotations

import numpy as np


def reorder(src: np.ndarray, idx) -> np.ndarray:
    """Row gather of ``src`` (any dtype, rows along axis 0) by ``idx``.

    Operates on the raw bytes of each row, so the result is bit-exact for any
    dtype (including bf16 stored as uint16 and NaN payloads)."""
    src = np.ascontiguousarray(src)
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= src.shape[0]):
        raise IndexError("reorder index out of range")
    rows = src.reshape(src.shape[0], -1).view(np.uint8) if src.size else src.reshape(src.shape[0], 0).view(np.uint8)
    out = np.take(rows, idx, axis=0)
    return out.view(src.dtype).reshape((idx.shape[0],) + src.shape[1:])


def reorder_loop(src_bytes: bytes, row_bytes: int, idx) -> bytes:
    """The same gather as a plain Python byte loop (for tiny inputs)."""
    out = bytearray()
    for i in idx:
        out += src_bytes[i * row_bytes:(i + 1) * row_bytes]
    return bytes(out)
