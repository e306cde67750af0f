"""CPU oracle for the W4A16 fused matrix multiply ``Y = X . dequant(W)``.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  It shares
no code with the CUDA library in ``w4a16_mixed_precision_gb300`` and never
imports it.

The arithmetic lives in ``oracle.c`` (plain C, binary64, no FMA contraction).
This module only builds it, loads it with ctypes and marshals numpy arrays.
Definitions followed (page titles and sections):

* "Marlin / GPTQ-Marlin", section "Le problème": ``Y = X_fp16 x W_int4`` with the
  INT4 weights dequantised to FP16 before the multiply.
* "Marlin" (dingiv.github.io), section "Group size 为什么是 128": one scale and one zero point
  per 128 consecutive weights; section "反量化精度权衡": INT4 -> FP16 is
  exact, accumulation is FP32 inside the tensor core, output is FP16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_double_to_half_rne.argtypes = [ctypes.c_double]
        lib.oracle_double_to_half_rne.restype = ctypes.c_uint16
        lib.oracle_dequant_scalar.argtypes = [I, I, ctypes.c_uint16]
        lib.oracle_dequant_scalar.restype = ctypes.c_uint16
        lib.oracle_unpack_codes.argtypes = [P, I, I, P]
        lib.oracle_unpack_zeros.argtypes = [P, I, I, P]
        lib.oracle_dequant.argtypes = [P, P, P, I, I, I, P]
        lib.oracle_gemm.argtypes = [P, P, I, I, I, P, I]
        lib.oracle_w4a16.argtypes = [P, P, P, P, I, I, I, I, P, ctypes.c_int64, P, I]
        lib.oracle_repack.argtypes = [P, I, I, P]
        lib.oracle_unrepack.argtypes = [P, I, I, P]
        lib.oracle_repack_scales.argtypes = [P, I, I, P]
        lib.oracle_repack_zeros.argtypes = [P, I, I, P]
        lib.oracle_repack_scales.restype = I
        lib.oracle_repack_zeros.restype = I
        lib.oracle_round_array.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_round_array.restype = None
        lib.oracle_widen_array.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_widen_array.restype = None
        lib.oracle_sparse_compress.argtypes = [P, P, I, I, I, P, P]
        lib.oracle_sparse_expand.argtypes = [P, P, P, I, I, I, P]
        lib.oracle_w4a16_sparse.argtypes = [P, P, P, P, P, I, I, I, I, P, ctypes.c_int64, P, I]
        lib.oracle_sparse_repack.argtypes = [P, P, I, I, P, P]
        lib.oracle_sparse_unrepack.argtypes = [P, P, I, I, P, P]
        for name in ("oracle_unpack_codes", "oracle_unpack_zeros", "oracle_dequant", "oracle_gemm",
                     "oracle_w4a16", "oracle_repack", "oracle_unrepack", "oracle_sparse_compress",
                     "oracle_sparse_expand", "oracle_w4a16_sparse", "oracle_sparse_repack",
                     "oracle_sparse_unrepack"):
            getattr(lib, name).restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits16(a) -> np.ndarray:
    """fp16 array (numpy float16 or uint16 bit patterns) -> contiguous uint16 bits."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


def _i32(a) -> np.ndarray | None:
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    assert a.dtype == np.int32, a.dtype
    return np.ascontiguousarray(a)


def _threads(n: int | None) -> int:
    return n if n else (os.cpu_count() or 1)


def half_to_double(h: int) -> float:
    return _load().oracle_half_to_double(int(h) & 0xFFFF)


def double_to_half_rne(v: float) -> int:
    return int(_load().oracle_double_to_half_rne(float(v)))


def dequant_scalar(q: int, z: int, s_bits: int) -> int:
    """fp16 bits of fp16_rne((q - z) * s)."""
    return int(_load().oracle_dequant_scalar(int(q), int(z), int(s_bits) & 0xFFFF))


def unpack_codes(Qp, K: int, N: int) -> np.ndarray:
    """GPTQ-order int32 [K/8][N] -> uint8 codes [K][N]."""
    Qp = _i32(Qp)
    q = np.empty((K, N), np.uint8)
    assert _load().oracle_unpack_codes(_ptr(Qp), K, N, _ptr(q)) == 0
    return q


def unpack_zeros(Zp, G: int, N: int) -> np.ndarray:
    """Packed int32 zeros [G][N/8] (or None: z = 8) -> uint8 [G][N]."""
    Zp = _i32(Zp)
    z = np.empty((G, N), np.uint8)
    assert _load().oracle_unpack_zeros(_ptr(Zp), G, N, _ptr(z)) == 0
    return z


def dequant(Qp, S, Zp, K: int, N: int, g: int) -> np.ndarray:
    """fp16 W [K][N] = fp16_rne((q - z) * s), returned as numpy float16."""
    Qp, S, Zp = _i32(Qp), _bits16(S), _i32(Zp)
    W = np.empty((K, N), np.uint16)
    assert _load().oracle_dequant(_ptr(Qp), _ptr(S), _ptr(Zp), K, N, g, _ptr(W)) == 0
    return W.view(np.float16)


def gemm(X, W, threads: int | None = None) -> np.ndarray:
    """binary64 Y [M][N] = X [M][K] . W [K][N] (fp16 inputs), k ascending."""
    X, W = _bits16(X), _bits16(W)
    M, K = X.shape
    K2, N = W.shape
    assert K == K2
    Y = np.empty((M, N), np.float64)
    assert _load().oracle_gemm(_ptr(X), _ptr(W), M, K, N, _ptr(Y), _threads(threads)) == 0
    return Y


def w4a16(X, Qp, S, Zp, g: int, N: int, idx=None, threads: int | None = None) -> np.ndarray:
    """Y = X . dequant(W) in binary64 straight from the packed GPTQ-order inputs.

    idx: optional flat indices m*N + n; then returns y at those entries only.
    """
    X, Qp, S, Zp = _bits16(X), _i32(Qp), _bits16(S), _i32(Zp)
    M, K = X.shape
    if idx is None:
        out = np.empty((M, N), np.float64)
        count = 0
        idx_p = None
    else:
        idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
        out = np.empty(idx.shape[0], np.float64)
        count = idx.shape[0]
        idx_p = _ptr(idx)
    rc = _load().oracle_w4a16(_ptr(X), _ptr(Qp), _ptr(S), _ptr(Zp), M, K, N, g, idx_p, count,
                              _ptr(out), _threads(threads))
    assert rc == 0
    return out


def repack(Qp, K: int, N: int) -> np.ndarray:
    """GPTQ-order codes [K/8][N] -> this library's tile layout, int32 [(N/128)*(K/64)*1024]."""
    Qp = _i32(Qp)
    P = np.empty((N // 128) * (K // 64) * 1024, np.int32)
    assert _load().oracle_repack(_ptr(Qp), K, N, _ptr(P)) == 0
    return P


def repack_scales(S, N: int) -> np.ndarray:
    """fp16 scales [G][N] -> tile-major [N/128][G][128] (flattened, float16)."""
    S = _bits16(S)
    G = S.shape[0]
    out = np.empty(G * N, np.uint16)
    assert _load().oracle_repack_scales(_ptr(S), G, N, _ptr(out)) == 0
    return out.view(np.float16)


def repack_zeros(Zp, N: int) -> np.ndarray:
    """Packed zeros int32 [G][N/8] -> tile-major bytes [N/128][G][64] (flattened uint8)."""
    Zp = _i32(Zp)
    G = Zp.shape[0]
    out = np.zeros(G * N // 2, np.uint8)
    assert _load().oracle_repack_zeros(_ptr(Zp), G, N, _ptr(out)) == 0
    return out


def unrepack(P, K: int, N: int) -> np.ndarray:
    """Inverse of repack: tile layout -> GPTQ-order int32 [K/8][N]."""
    P = _i32(P)
    Qp = np.empty((K // 8, N), np.int32)
    assert _load().oracle_unrepack(_ptr(P), K, N, _ptr(Qp)) == 0
    return Qp


# ---- 2:4 structured sparsity ("Marlin", section "支持 2:4 稀疏加速"; "Marlin /
# GPTQ-Marlin", section "4. Support de la sparsité 2:4 NVIDIA") ----------------

def sparse_compress(Qp, Zp, K: int, N: int, g: int):
    """GPTQ-order codes -> (kc uint8 [K/2][N], ki uint8 [K/4][N], bad groups).

    Per group of four rows 4j..4j+3 of column n: kept positions i0 < i1 (the
    codes that differ from the zero point, completed with the lowest positions
    whose code equals it), kc[2j+t][n] = code at i_t, ki[j][n] = i0 | i1 << 2.
    bad = groups where more than two codes differ from the zero point.
    """
    Qp, Zp = _i32(Qp), _i32(Zp)
    kc = np.empty((K // 2, N), np.uint8)
    ki = np.empty((K // 4, N), np.uint8)
    bad = _load().oracle_sparse_compress(_ptr(Qp), _ptr(Zp), K, N, g, _ptr(kc), _ptr(ki))
    assert bad >= 0
    return kc, ki, int(bad)


def sparse_expand(kc, ki, Zp, K: int, N: int, g: int) -> np.ndarray:
    """Compressed form -> dense GPTQ-order int32 [K/8][N] (zero point at dropped rows)."""
    kc = np.ascontiguousarray(kc, np.uint8)
    ki = np.ascontiguousarray(ki, np.uint8)
    Zp = _i32(Zp)
    Qp = np.empty((K // 8, N), np.int32)
    assert _load().oracle_sparse_expand(_ptr(kc), _ptr(ki), _ptr(Zp), K, N, g, _ptr(Qp)) == 0
    return Qp


def w4a16_sparse(X, kc, ki, S, Zp, g: int, N: int, idx=None, threads: int | None = None) -> np.ndarray:
    """binary64 Y = X . dequant(W) for 2:4 weights, summing the kept terms only."""
    X, S, Zp = _bits16(X), _bits16(S), _i32(Zp)
    kc = np.ascontiguousarray(kc, np.uint8)
    ki = np.ascontiguousarray(ki, np.uint8)
    M, K = X.shape
    if idx is None:
        out = np.empty((M, N), np.float64)
        count, idx_p = 0, None
    else:
        idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
        out = np.empty(idx.shape[0], np.float64)
        count, idx_p = idx.shape[0], _ptr(idx)
    rc = _load().oracle_w4a16_sparse(_ptr(X), _ptr(kc), _ptr(ki), _ptr(S), _ptr(Zp), M, K, N, g,
                                     idx_p, count, _ptr(out), _threads(threads))
    assert rc == 0
    return out


def sparse_repack(kc, ki, K: int, N: int):
    """Compressed form -> this library's sparse tile layout: (codes int32
    [(N/128)*(K/64)*512], meta int32 [(N/128)*(K/64)*256])."""
    kc = np.ascontiguousarray(kc, np.uint8)
    ki = np.ascontiguousarray(ki, np.uint8)
    blocks = (N // 128) * (K // 64)
    Pc = np.empty(blocks * 512, np.int32)
    Pm = np.empty(blocks * 256, np.int32)
    assert _load().oracle_sparse_repack(_ptr(kc), _ptr(ki), K, N, _ptr(Pc), _ptr(Pm)) == 0
    return Pc, Pm


def sparse_unrepack(Pc, Pm, K: int, N: int):
    """Inverse of sparse_repack: (kc, ki)."""
    Pc, Pm = _i32(Pc), _i32(Pm)
    kc = np.empty((K // 2, N), np.uint8)
    ki = np.empty((K // 4, N), np.uint8)
    assert _load().oracle_sparse_unrepack(_ptr(Pc), _ptr(Pm), K, N, _ptr(kc), _ptr(ki)) == 0
    return kc, ki


def to_half_rne(y) -> np.ndarray:
    """Round binary64 values to fp16 with the oracle's own routine."""
    flat = np.ascontiguousarray(np.asarray(y, np.float64).ravel())
    out = np.empty(flat.size, np.uint16)
    _load().oracle_round_array(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(np.shape(y)).view(np.float16)


def widen(h) -> np.ndarray:
    """Exact binary64 values of fp16 data, with the oracle's own routine."""
    flat = _bits16(np.asarray(h).ravel())
    out = np.empty(flat.size, np.float64)
    _load().oracle_widen_array(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(np.shape(h))


def within_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, atol: float = 1e-2,
                     rtol: float = 2e-3):
    """The parity bar: |y_gpu - y_ref| <= atol + rtol*|y_ref| for every entry.

    Returns (ok, max_abs_err, worst_ratio) where worst_ratio = max of
    |err| / (atol + rtol*|y_ref|) (ok iff <= 1).
    """
    yg = np.asarray(y_gpu, np.float64)
    yr = np.asarray(y_ref, np.float64)
    err = np.abs(yg - yr)
    if err.size == 0:
        return True, 0.0, 0.0
    bound = atol + rtol * np.abs(yr)
    ratio = err / bound
    ok = bool(np.all(np.isfinite(yg)) and np.all(ratio <= 1.0))
    return ok, float(err.max()), float(ratio.max())
