"""Q4_K, Q5_K and Q6_K block dequantisation and the dequant-GEMV, fp64.

TEST INFRASTRUCTURE (see the package docstring): only the tests, the smoke
check and the benchmark's CPU leg use it.

The engine page (section 1) lists Q4_K_M, Q5_K and Q6_K among the GGUF
weight types it runs, and quotes its 70B numbers on Q6_K and Q4_K_M files;
it prints no layout.  Reading: the K-quant super-block layouts of the GGUF
format those files use, restated here from what each field means.  Both
types cover 256 weights per super-block; a [rows x cols] matrix (cols a
multiple of 256) is row-major, cols / 256 super-blocks per row.

Q4_K, 144 bytes:
  bytes 0-1    d     fp16, scale of the sub-block scales
  bytes 2-3    dmin  fp16, scale of the sub-block minimums
  bytes 4-15   twelve bytes holding eight 6-bit scales sc_s and eight 6-bit
               minimums m_s (s = 0..7, one pair per 32 weights):
                 s < 4:  sc_s = low 6 bits of byte s, m_s = low 6 bits of byte s+4
                 s >= 4: the low 4 bits of sc_s / m_s are the low / high nibble
                         of byte s+4; their top 2 bits are the top 2 bits of
                         byte s-4 (for sc) and of byte s (for m)
  bytes 16-143 128 bytes of 4-bit codes q: byte 32g + l (g = 0..3, l = 0..31)
               holds weight 64g + l in its low nibble and weight 64g + 32 + l
               in its high nibble
  weight_i = d * sc_s * q_i - dmin * m_s       (s = i // 32)

Q5_K, 176 bytes: Q4_K's first 16 bytes (d, dmin, the twelve scale bytes),
  then 32 bytes qh of fifth code bits, then Q4_K's 128 bytes of low 4 bits.
  Weight 64g + l takes bit 2g of qh[l] as its fifth bit, weight 64g + 32 + l
  bit 2g + 1 (g = 0..3, l = 0..31); q = low | fifth << 4 (0..31) and
  weight_i = d * sc_s * q_i - dmin * m_s as for Q4_K.

Q6_K, 210 bytes:
  bytes 0-127   ql: low 4 bits of the codes
  bytes 128-191 qh: high 2 bits of the codes
  bytes 192-207 sixteen int8 scales; scale k applies to weights 16k..16k+15
  bytes 208-209 d fp16
  Weight i: half h = i // 128, o = i % 128, g = o // 32, l = o % 32.  Its
  high 2 bits are bits 2g, 2g+1 of qh[32h + l]; its low 4 bits are
      g = 0: the low nibble of ql[64h + l]    g = 1: the low nibble of ql[64h + 32 + l]
      g = 2: the high nibble of ql[64h + l]   g = 3: the high nibble of ql[64h + 32 + l]
  code = low | high << 4 (0..63); weight_i = d * scale_(i // 16) * (code - 32)
"""
from __future__ import annotations

import numpy as np

QK = 256
BLOCK_BYTES = {"q4_k": 144, "q5_k": 176, "q6_k": 210}


def _f16(lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    bits = lo.astype(np.uint16) | (hi.astype(np.uint16) << 8)
    return np.ascontiguousarray(bits).view(np.float16).astype(np.float64)


def q4_k_scales_mins(sb: np.ndarray):
    """The 12 packed bytes [n, 12] -> (sc [n, 8], m [n, 8]) as integers 0..63."""
    b = sb.astype(np.int64)
    sc = np.empty((b.shape[0], 8), dtype=np.int64)
    m = np.empty((b.shape[0], 8), dtype=np.int64)
    for s in range(4):
        sc[:, s] = b[:, s] & 63
        m[:, s] = b[:, s + 4] & 63
    for s in range(4, 8):
        sc[:, s] = (b[:, s + 4] & 0x0F) | ((b[:, s - 4] >> 6) << 4)
        m[:, s] = (b[:, s + 4] >> 4) | ((b[:, s] >> 6) << 4)
    return sc, m


def dequant_q4_k(blocks: np.ndarray, n_blocks: int) -> np.ndarray:
    """n_blocks Q4_K super-blocks -> float64 [n_blocks, 256]."""
    b = np.asarray(blocks, dtype=np.uint8)[: n_blocks * 144].reshape(n_blocks, 144)
    d = _f16(b[:, 0], b[:, 1])
    dmin = _f16(b[:, 2], b[:, 3])
    sc, m = q4_k_scales_mins(b[:, 4:16])
    qs = b[:, 16:].astype(np.int64)
    q = np.empty((n_blocks, QK), dtype=np.int64)
    for g in range(4):
        q[:, 64 * g: 64 * g + 32] = qs[:, 32 * g: 32 * g + 32] & 0x0F
        q[:, 64 * g + 32: 64 * g + 64] = qs[:, 32 * g: 32 * g + 32] >> 4
    sub = np.arange(QK) // 32
    return d[:, None] * sc[:, sub] * q - dmin[:, None] * m[:, sub]


def dequant_q5_k(blocks: np.ndarray, n_blocks: int) -> np.ndarray:
    """n_blocks Q5_K super-blocks -> float64 [n_blocks, 256]."""
    b = np.asarray(blocks, dtype=np.uint8)[: n_blocks * 176].reshape(n_blocks, 176)
    d = _f16(b[:, 0], b[:, 1])
    dmin = _f16(b[:, 2], b[:, 3])
    sc, m = q4_k_scales_mins(b[:, 4:16])
    qh = b[:, 16:48].astype(np.int64)
    qs = b[:, 48:].astype(np.int64)
    q = np.empty((n_blocks, QK), dtype=np.int64)
    for g in range(4):
        q[:, 64 * g: 64 * g + 32] = (qs[:, 32 * g: 32 * g + 32] & 0x0F) | (((qh >> (2 * g)) & 1) << 4)
        q[:, 64 * g + 32: 64 * g + 64] = (qs[:, 32 * g: 32 * g + 32] >> 4) | (((qh >> (2 * g + 1)) & 1) << 4)
    sub = np.arange(QK) // 32
    return d[:, None] * sc[:, sub] * q - dmin[:, None] * m[:, sub]


def q6_k_codes(ql: np.ndarray, qh: np.ndarray) -> np.ndarray:
    """ql [n, 128] and qh [n, 64] -> the 6-bit codes [n, 256] (0..63)."""
    ql = ql.astype(np.int64)
    qh = qh.astype(np.int64)
    code = np.empty((ql.shape[0], QK), dtype=np.int64)
    for h in range(2):
        for g in range(4):
            src = ql[:, 64 * h + 32 * (g % 2): 64 * h + 32 * (g % 2) + 32]
            low = src & 0x0F if g < 2 else src >> 4
            high = (qh[:, 32 * h: 32 * h + 32] >> (2 * g)) & 3
            code[:, 128 * h + 32 * g: 128 * h + 32 * g + 32] = low | (high << 4)
    return code


def dequant_q6_k(blocks: np.ndarray, n_blocks: int) -> np.ndarray:
    """n_blocks Q6_K super-blocks -> float64 [n_blocks, 256]."""
    b = np.asarray(blocks, dtype=np.uint8)[: n_blocks * 210].reshape(n_blocks, 210)
    code = q6_k_codes(b[:, :128], b[:, 128:192])
    scale = b[:, 192:208].view(np.int8).astype(np.int64)
    d = _f16(b[:, 208], b[:, 209])
    return d[:, None] * scale[:, np.arange(QK) // 16] * (code - 32)


def dequant_blocks(blocks: np.ndarray, n_blocks: int, fmt: str) -> np.ndarray:
    if fmt == "q4_k":
        return dequant_q4_k(blocks, n_blocks)
    if fmt == "q5_k":
        return dequant_q5_k(blocks, n_blocks)
    if fmt == "q6_k":
        return dequant_q6_k(blocks, n_blocks)
    raise ValueError(f"unknown K-quant format {fmt}")


def matrix_rows(blocks: np.ndarray, cols: int, fmt: str, r0: int, r1: int) -> np.ndarray:
    """Rows [r0, r1) of a [rows x cols] K-quant matrix -> float64 [r1-r0, cols]."""
    if cols % QK:
        raise ValueError(f"cols={cols} is not a multiple of {QK}")
    nb = cols // QK
    bb = BLOCK_BYTES[fmt]
    sub = np.asarray(blocks, dtype=np.uint8)[r0 * nb * bb: r1 * nb * bb]
    return dequant_blocks(sub, (r1 - r0) * nb, fmt).reshape(r1 - r0, cols)


def gemv(blocks: np.ndarray, rows: int, cols: int, fmt: str, x: np.ndarray, chunk_rows: int = 4096) -> np.ndarray:
    """y = W x in float64 (the dequant-GEMV's definition), dequantising rows
    in chunks so large matrices stay within memory."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(rows, dtype=np.float64)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = matrix_rows(blocks, cols, fmt, r0, r1) @ x
    return out
