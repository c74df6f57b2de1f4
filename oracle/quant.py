"""Q8_0 / Q4_0 block dequantisation, fp64.

Formats, as the workload statements define them (the engine page, section 1,
names Q8_0 and Q4_0 among the GGUF types it supports; the byte layouts are the
ones the workloads give):

* Q8_0 block, 34 bytes: little-endian fp16 scale d, then 32 int8 q.
  weight_i = d * q_i.
* Q4_0 block, 18 bytes: fp16 scale d, then 16 bytes; byte j carries element j
  in its low nibble and element j + 16 in its high nibble.
  weight = d * (nibble - 8).

A matrix [rows x cols] is row-major with ceil(cols / 32) blocks per row.
"""
from __future__ import annotations

import numpy as np

BLOCK_BYTES = {8: 34, 4: 18}


def blocks_per_row(cols: int) -> int:
    return (cols + 31) // 32


def _f16(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns -> exact float64 values."""
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dequant_q8_0(blocks: np.ndarray, n_blocks: int) -> np.ndarray:
    """n_blocks Q8_0 blocks -> float64 [n_blocks, 32]."""
    b = np.asarray(blocks, dtype=np.uint8)[: n_blocks * 34].reshape(n_blocks, 34)
    d = _f16(b[:, 0].astype(np.uint16) | (b[:, 1].astype(np.uint16) << 8))
    q = b[:, 2:].view(np.int8).astype(np.float64)
    return d[:, None] * q


def dequant_q4_0(blocks: np.ndarray, n_blocks: int) -> np.ndarray:
    """n_blocks Q4_0 blocks -> float64 [n_blocks, 32]."""
    b = np.asarray(blocks, dtype=np.uint8)[: n_blocks * 18].reshape(n_blocks, 18)
    d = _f16(b[:, 0].astype(np.uint16) | (b[:, 1].astype(np.uint16) << 8))
    packed = b[:, 2:].astype(np.int64)
    q = np.empty((n_blocks, 32), dtype=np.float64)
    q[:, :16] = (packed & 0x0F) - 8      # elements 0..15: low nibbles
    q[:, 16:] = (packed >> 4) - 8        # elements 16..31: high nibbles
    return d[:, None] * q


def dequant_blocks(blocks: np.ndarray, n_blocks: int, wtype: int) -> np.ndarray:
    if wtype == 8:
        return dequant_q8_0(blocks, n_blocks)
    if wtype == 4:
        return dequant_q4_0(blocks, n_blocks)
    raise ValueError(f"unknown weight type {wtype}")


def matrix_rows(blocks: np.ndarray, cols: int, wtype: int, r0: int, r1: int) -> np.ndarray:
    """Rows [r0, r1) of a quantised [rows x cols] matrix -> float64 [r1-r0, cols]."""
    nb = blocks_per_row(cols)
    bb = BLOCK_BYTES[wtype]
    sub = np.asarray(blocks, dtype=np.uint8)[r0 * nb * bb: r1 * nb * bb]
    w = dequant_blocks(sub, (r1 - r0) * nb, wtype).reshape(r1 - r0, nb * 32)
    return w[:, :cols]


def matrix(blocks: np.ndarray, rows: int, cols: int, wtype: int) -> np.ndarray:
    """Whole quantised matrix -> float64 [rows, cols]."""
    return matrix_rows(blocks, cols, wtype, 0, rows)
