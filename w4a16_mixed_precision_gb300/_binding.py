"""ctypes binding of libw4a16_gb300.so (the C ABI in include/marlin.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if the shared library is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libw4a16_gb300.so")
#: the bounds-checked build (-DMARLIN_DEBUG), built on demand by build.build(debug=True)
DEBUG_LIB_PATH = os.path.join(_PKG, "_lib", "libw4a16_gb300_debug.so")

# marlin_status_t
OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_MISALIGNED = 3
ERR_WORKSPACE_TOO_SMALL = 4
ERR_CUDA = 5
ERR_TIMEOUT = 6
ERR_BOUNDS = 7

#: every symbol include/marlin.h declares
EXPORTS = (
    "marlin_status_string",
    "marlin_packed_layout",
    "marlin_repack",
    "marlin_workspace_bytes",
    "marlin_gemm",
    "marlin_gemm_ex",
    "marlin_gemm_no_alloc",
    "marlin_gemm_host",
    "marlin_last_device_status",
    "marlin_sparse_packed_layout",
    "marlin_sparse_repack",
    "marlin_sparse_gemm",
)


class MarlinError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (build it first with __graft_entry__.build() or
    w4a16_mixed_precision_gb300.build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = open_library(path or LIB_PATH)
        return _lib


def open_library(path: str) -> ctypes.CDLL:
    """A separate handle on a build of the library (e.g. the bounds-checked
    one, libw4a16_gb300_debug.so), with the C signatures declared."""
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing")
    if True:
        lib = ctypes.CDLL(path)
        P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.marlin_status_string.argtypes = [I]
        lib.marlin_status_string.restype = ctypes.c_char_p
        lib.marlin_packed_layout.argtypes = [I, I, I, I, ctypes.POINTER(SZ), ctypes.POINTER(SZ),
                                             ctypes.POINTER(SZ)]
        lib.marlin_repack.argtypes = [P, P, P, I, I, I, P, P]
        lib.marlin_workspace_bytes.argtypes = [I, I, I, I, I, ctypes.POINTER(SZ)]
        lib.marlin_gemm.argtypes = [P, P, P, P, P, I, I, I, I, P, SZ, P]
        lib.marlin_gemm_ex.argtypes = [P, P, P, P, P, I, I, I, I, P, SZ, I, P]
        lib.marlin_gemm_ex.restype = I
        lib.marlin_last_device_status.argtypes = [P, P]
        lib.marlin_gemm_no_alloc.argtypes = [P, P, P, P, P, I, I, I, I, P]
        lib.marlin_gemm_no_alloc.restype = I
        lib.marlin_gemm_host.argtypes = [P, P, P, P, P, P, P, I, I, I, I, P, SZ, P]
        lib.marlin_gemm_host.restype = I
        lib.marlin_sparse_packed_layout.argtypes = [I, I, I, I] + [ctypes.POINTER(SZ)] * 4
        lib.marlin_sparse_repack.argtypes = [P, P, P, I, I, I, P, P, P]
        lib.marlin_sparse_gemm.argtypes = [P, P, P, P, P, P, I, I, I, I, P, SZ, P]
        for f in ("marlin_sparse_packed_layout", "marlin_sparse_repack", "marlin_sparse_gemm"):
            getattr(lib, f).restype = I
        for f in ("marlin_packed_layout", "marlin_repack", "marlin_workspace_bytes", "marlin_gemm",
                  "marlin_last_device_status"):
            getattr(lib, f).restype = I
    return lib


def status_string(status: int) -> str:
    return load().marlin_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise MarlinError(status, where)


def packed_layout(K: int, N: int, group: int, has_zeros: bool):
    """(bytes, off_scales, off_zeros) of the repacked buffer."""
    b, s, z = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().marlin_packed_layout(K, N, group, int(bool(has_zeros)), ctypes.byref(b),
                                       ctypes.byref(s), ctypes.byref(z)), "marlin_packed_layout")
    return b.value, s.value, z.value


def workspace_bytes(M: int, K: int, N: int, group: int, device: int = 0) -> int:
    b = ctypes.c_size_t()
    _check(load().marlin_workspace_bytes(M, K, N, group, device, ctypes.byref(b)),
           "marlin_workspace_bytes")
    return b.value


def repack_raw(q_ptr: int, scales_ptr: int, zeros_ptr: int | None, K: int, N: int, group: int,
               out_ptr: int, stream: int) -> int:
    """Raw call; returns the status code."""
    return load().marlin_repack(q_ptr, scales_ptr, zeros_ptr or None, K, N, group, out_ptr,
                                stream or None)


def gemm_raw(x_ptr: int, packed_ptr: int, scales_ptr: int, zeros_ptr: int | None, y_ptr: int, M: int,
             K: int, N: int, group: int, ws_ptr: int, ws_bytes: int, stream: int) -> int:
    """Raw call; returns the status code."""
    return load().marlin_gemm(x_ptr, packed_ptr, scales_ptr, zeros_ptr or None, y_ptr, M, K, N,
                              group, ws_ptr, ws_bytes, stream or None)


KERNELS = {"auto": 0, "warp": 1, "tcgen05": 2}


def gemm_ex_raw(x_ptr: int, packed_ptr: int, scales_ptr: int, zeros_ptr: int | None, y_ptr: int, M: int,
                K: int, N: int, group: int, ws_ptr: int, ws_bytes: int, kernel: int, stream: int) -> int:
    """Raw call with an explicit kernel (0 auto, 1 warp-level, 2 tcgen05); returns the status code."""
    return load().marlin_gemm_ex(x_ptr, packed_ptr, scales_ptr, zeros_ptr or None, y_ptr, M, K, N,
                                 group, ws_ptr, ws_bytes, kernel, stream or None)


def gemm_host_raw(xh_ptr: int, xd_ptr: int, packed_ptr: int, scales_ptr: int, zeros_ptr: int | None,
                  yd_ptr: int, yh_ptr: int, M: int, K: int, N: int, group: int, ws_ptr: int,
                  ws_bytes: int, stream: int) -> int:
    """Raw call of the host-buffer entry point; returns the status code."""
    return load().marlin_gemm_host(xh_ptr, xd_ptr, packed_ptr, scales_ptr, zeros_ptr or None, yd_ptr,
                                   yh_ptr, M, K, N, group, ws_ptr, ws_bytes, stream or None)


def gemm_no_alloc_raw(x_ptr: int, packed_ptr: int, scales_ptr: int, zeros_ptr: int | None, y_ptr: int,
                     M: int, K: int, N: int, group: int, stream: int) -> int:
    """Raw call of the entry point that uses the library's own scratch
    (for callers that cannot allocate a workspace); returns the status code."""
    return load().marlin_gemm_no_alloc(x_ptr, packed_ptr, scales_ptr, zeros_ptr or None, y_ptr, M, K,
                                       N, group, stream or None)


def last_device_status(ws_ptr: int, stream: int) -> int:
    return load().marlin_last_device_status(ws_ptr, stream or None)


def sparse_packed_layout(K: int, N: int, group: int, has_zeros: bool):
    """(bytes, off_meta, off_scales, off_zeros) of the repacked 2:4 buffer."""
    b, m, sc, z = (ctypes.c_size_t() for _ in range(4))
    _check(load().marlin_sparse_packed_layout(K, N, group, int(bool(has_zeros)), ctypes.byref(b),
                                              ctypes.byref(m), ctypes.byref(sc), ctypes.byref(z)),
           "marlin_sparse_packed_layout")
    return b.value, m.value, sc.value, z.value


def sparse_repack_raw(q_ptr: int, scales_ptr: int, zeros_ptr: int | None, K: int, N: int, group: int,
                      out_ptr: int, bad_ptr: int | None, stream: int) -> int:
    """Raw call of the 2:4 repack; returns the status code."""
    return load().marlin_sparse_repack(q_ptr, scales_ptr, zeros_ptr or None, K, N, group, out_ptr,
                                       bad_ptr or None, stream or None)


def sparse_gemm_raw(x_ptr: int, packed_ptr: int, meta_ptr: int | None, scales_ptr: int,
                    zeros_ptr: int | None, y_ptr: int, M: int, K: int, N: int, group: int, ws_ptr: int,
                    ws_bytes: int, stream: int) -> int:
    """Raw call of the 2:4-sparse multiply; returns the status code."""
    return load().marlin_sparse_gemm(x_ptr, packed_ptr, meta_ptr or None, scales_ptr, zeros_ptr or None,
                                     y_ptr, M, K, N, group, ws_ptr, ws_bytes, stream or None)
