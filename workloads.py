"""Seeded synthetic inputs for the W4A16 matrix multiply, shared by the tests,
the benchmark and the smoke check.

This module holds no arithmetic of the method (no dequantisation, no
products, no layout permutation): it draws random inputs in the input
format and lists the workload shapes.  Both the CPU oracle and the CUDA
library consume what it returns.

Input recipe (the workloads of the pages' GEMM benchmarks, synthesised):
  X  = fp16(N(0, 1))                         [M][K]
  Qp = uniform random 32-bit words           [K/8][N]   (8 uniform 4-bit codes each,
                                                           code of row 8r+i at nibble i)
  S  = fp16(0.02 * U(0.5, 1.5))              [K/g][N]
  Zp = uniform random 32-bit words           [K/g][N/8] (explicit zeros) or None (z = 8)
2:4-sparse weights (make_sparse_weights): in every four consecutive rows of a
column two positions (uniform among the six pairs) hold uniform codes and the
other two the zero point.
Seed = CRC32 of "cfg:M:K:N:g:asym" (see seed_for).
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Problem:
    """One W4A16 matrix multiply: Y[M,N] = X[M,K] . dequant(W)[K,N]."""
    cfg: str
    M: int
    K: int
    N: int
    group: int          # 128, or K for one scale per column
    asym: bool          # explicit 4-bit zeros (True) or implicit zero 8 (False)
    sparse: bool = False  # 2:4-sparse weights, multiplied on the sparse path

    @property
    def G(self) -> int:
        return self.K // self.group

    @property
    def key(self) -> str:
        return f"{self.cfg}:{self.M}:{self.K}:{self.N}:{self.group}:{int(self.asym)}"

    def algorithmic_bytes(self) -> int:
        """Bytes the method must move: codes + scales (+ zeros) + X + Y.  2:4
        weights: the kept half of the codes plus a 4-bit index pair per four."""
        codes = self.K * self.N // 4 + self.K * self.N // 8 if self.sparse else self.K * self.N // 2
        b = codes + self.G * self.N * 2 + 2 * self.M * self.K + 2 * self.M * self.N
        if self.asym:
            b += self.G * self.N // 2
        return b

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def seed_for(key: str) -> int:
    return zlib.crc32(key.encode()) & 0xFFFFFFFF


@dataclass
class Inputs:
    X: np.ndarray          # float16 [M][K]
    Qp: np.ndarray         # int32 [K/8][N]
    S: np.ndarray          # float16 [G][N]
    Zp: np.ndarray | None  # int32 [G][N/8] or None


def make_inputs(p: Problem, seed: int | None = None) -> Inputs:
    rng = np.random.default_rng(seed_for(p.key) if seed is None else seed)
    X = rng.standard_normal((p.M, p.K), dtype=np.float32).astype(np.float16)
    if p.sparse:
        Qp, S, Zp = make_sparse_weights(p.K, p.N, p.group, p.asym, seed=int(rng.integers(2**32)))
        return Inputs(X, Qp, S, Zp)
    Qp = rng.integers(0, 2**32, size=(p.K // 8, p.N), dtype=np.uint64).astype(np.uint32).view(np.int32)
    S = (0.02 * rng.uniform(0.5, 1.5, size=(p.G, p.N))).astype(np.float16)
    Zp = None
    if p.asym:
        Zp = rng.integers(0, 2**32, size=(p.G, p.N // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    return Inputs(X, Qp, S, Zp)


def make_weights(K: int, N: int, group: int, asym: bool, seed: int):
    """Only the weight-side inputs (Qp, S, Zp) of a K x N layer."""
    rng = np.random.default_rng(seed)
    Qp = rng.integers(0, 2**32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32).view(np.int32)
    S = (0.02 * rng.uniform(0.5, 1.5, size=(K // group, N))).astype(np.float16)
    Zp = None
    if asym:
        Zp = rng.integers(0, 2**32, size=(K // group, N // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    return Qp, S, Zp


# the six ways to keep two of four positions, in ascending order
_PAIRS0 = np.array([0, 0, 0, 1, 1, 2], np.uint8)
_PAIRS1 = np.array([1, 2, 3, 2, 3, 3], np.uint8)


def make_sparse_weights(K: int, N: int, group: int, asym: bool, seed: int):
    """Weight-side inputs (Qp, S, Zp) of a 2:4-sparse K x N layer.

    In every four consecutive rows of a column, two positions (one of the six
    pairs, uniformly) get codes drawn uniformly from 0..15; the other two get
    the column's zero point (8, or the drawn zero), so at most two of every
    four weights are non-zero.  Scales as in make_weights.
    """
    rng = np.random.default_rng(seed)
    G = K // group
    z = rng.integers(0, 16, size=(G, N), dtype=np.uint8) if asym else np.full((G, N), 8, np.uint8)
    pair = rng.integers(0, 6, size=(K // 4, N), dtype=np.uint8)
    i0, i1 = _PAIRS0[pair], _PAIRS1[pair]
    v0 = rng.integers(0, 16, size=(K // 4, N), dtype=np.uint8)
    v1 = rng.integers(0, 16, size=(K // 4, N), dtype=np.uint8)
    zr = np.repeat(z, group // 4, axis=0)  # zero point of each group of four rows
    q = np.empty((K // 4, 4, N), np.uint8)
    for i in range(4):
        q[:, i, :] = np.where(i0 == i, v0, np.where(i1 == i, v1, zr))
    Qp = pack_codes(q.reshape(K, N))
    S = (0.02 * rng.uniform(0.5, 1.5, size=(G, N))).astype(np.float16)
    Zp = pack_zeros(z) if asym else None
    return Qp, S, Zp


def make_activations(M: int, K: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.standard_normal((M, K), dtype=np.float32).astype(np.float16)


# ---- input-format encoders for structured test inputs ---------------------

def pack_codes(q: np.ndarray) -> np.ndarray:
    """uint codes [K][N] in 0..15 -> GPTQ-order int32 [K/8][N] (row 8r+i at nibble i)."""
    q = np.asarray(q, np.uint32)
    K, N = q.shape
    assert K % 8 == 0 and q.max(initial=0) < 16
    out = np.zeros((K // 8, N), np.uint32)
    for i in range(8):
        out |= q[i::8, :] << np.uint32(4 * i)
    return out.view(np.int32)


def pack_zeros(z: np.ndarray) -> np.ndarray:
    """uint zeros [G][N] in 0..15 -> int32 [G][N/8] (column 8c+j at nibble j)."""
    z = np.asarray(z, np.uint32)
    G, N = z.shape
    assert N % 8 == 0 and z.max(initial=0) < 16
    out = np.zeros((G, N // 8), np.uint32)
    for j in range(8):
        out |= z[:, j::8] << np.uint32(4 * j)
    return out.view(np.int32)


# ---- the benchmark workloads (shapes of the pages' GEMM measurements) ------

SMALL = [Problem("single", 16, 4096, 4096, 128, False)]

LLAMA7B_DECODE_SHAPES = [(4096, 12288), (4096, 4096), (4096, 22016), (11008, 4096)]
LLAMA7B_DECODE_M = [1, 2, 4, 8, 16, 32]
LLAMA7B_DECODE = [Problem("7b-decode", M, K, N, 128, False)
                  for (K, N) in LLAMA7B_DECODE_SHAPES for M in LLAMA7B_DECODE_M]

LLAMA70B_SHAPES = [(8192, 10240), (8192, 8192), (8192, 57344), (28672, 8192)]
LLAMA70B_M = [1, 4, 16, 32, 64, 128]
LLAMA70B_DECODE = [Problem("70b-decode", M, K, N, 128, False)
                   for (K, N) in LLAMA70B_SHAPES for M in LLAMA70B_M]

PREFILL_SHAPES = [(8192, 8192), (8192, 28672)]
PREFILL_M = [1024, 4096, 8192]
PREFILL = [Problem("prefill", M, K, N, 128, False) for (K, N) in PREFILL_SHAPES for M in PREFILL_M]

ODD_SHAPES = [(2048, 2048), (2048, 5632), (5120, 15360), (13824, 5120)]
ODD_M = [1, 16, 48]
ASYM_ODD = [Problem("asym-odd", M, K, N, g, True)
            for (K, N) in ODD_SHAPES for M in ODD_M for g in (128, K)]

# the 7B decode linears with 2:4-sparse weights (the sparse path serves M <= 32)
SPARSE_7B_DECODE = [Problem("sparse-7b-decode", M, K, N, 128, False, True)
                    for (K, N) in LLAMA7B_DECODE_SHAPES for M in LLAMA7B_DECODE_M]
SPARSE_CONFIGS = {"sparse-7b-decode": SPARSE_7B_DECODE}

ALL_CONFIGS = {
    "single": SMALL,
    "7b-decode": LLAMA7B_DECODE,
    "70b-decode": LLAMA70B_DECODE,
    "prefill": PREFILL,
    "asym-odd": ASYM_ODD,
}
