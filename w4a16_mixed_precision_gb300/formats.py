"""Host-side conversion of AWQ-order 4-bit weights to the GPTQ order that
marlin_repack takes.

The pages name GPTQ and AWQ checkpoints as the inputs of the kernel ("Marlin",
dingiv.github.io, section "ExLlamaV2 (EXL2 格式)": the standard W4A16
GPTQ/AWQ weight layout; "Marlin / GPTQ-Marlin", section "Tiled layout et
repacking": GPTQ INT4 weights stored group-quantised, one scale and zero point
per group of 128) without printing either packing.  The readings taken here:

  GPTQ order (what marlin_repack takes): codes int32 [K/8][N], nibble i of word
  [r][n] is row 8r+i; zeros int32 [G][N/8], nibble j of word [g][c] is column
  8c+j.

  AWQ order: codes int32 [K][N/8] and zeros int32 [G][N/8], both packed along
  the columns, with nibble i of word [r][c] holding column 8c + order[i] for
  the interleave order = (0, 2, 4, 6, 1, 3, 5, 7).  Scales are fp16 [G][N] in
  both, and the dequantisation is (q - z) * s in both.

This runs once at load time on the host (numpy); it is not on the GEMM path.
"""
from __future__ import annotations

import numpy as np

AWQ_ORDER = (0, 2, 4, 6, 1, 3, 5, 7)


def _unpack_columns(words: np.ndarray, order) -> np.ndarray:
    """int32 [R][C/8] packed along columns -> uint8 [R][C] codes."""
    w = np.asarray(words).view(np.uint32)
    R, C8 = w.shape
    out = np.empty((R, C8 * 8), np.uint8)
    for i, col in enumerate(order):
        out[:, col::8] = (w >> np.uint32(4 * i)) & np.uint32(0xF)
    return out


def _pack_columns(codes: np.ndarray) -> np.ndarray:
    """uint codes [R][C] -> int32 [R][C/8], column 8c+j at nibble j."""
    q = np.asarray(codes, np.uint32)
    R, C = q.shape
    out = np.zeros((R, C // 8), np.uint32)
    for j in range(8):
        out |= q[:, j::8] << np.uint32(4 * j)
    return out.view(np.int32)


def _pack_rows(codes: np.ndarray) -> np.ndarray:
    """uint codes [K][N] -> int32 [K/8][N], row 8r+i at nibble i."""
    q = np.asarray(codes, np.uint32)
    K, N = q.shape
    out = np.zeros((K // 8, N), np.uint32)
    for i in range(8):
        out |= q[i::8, :] << np.uint32(4 * i)
    return out.view(np.int32)


def awq_to_gptq(qweight: np.ndarray, qzeros: np.ndarray | None = None, order=AWQ_ORDER):
    """AWQ-order codes int32 [K][N/8] (and zeros int32 [G][N/8]) -> GPTQ-order
    codes int32 [K/8][N] (and zeros int32 [G][N/8] in column order).  K must be
    a multiple of 8."""
    q = _unpack_columns(qweight, order)
    if q.shape[0] % 8:
        raise ValueError("K must be a multiple of 8")
    codes = _pack_rows(q)
    zeros = None if qzeros is None else _pack_columns(_unpack_columns(qzeros, order))
    return codes, zeros
