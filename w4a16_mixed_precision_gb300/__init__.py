"""W4A16 fused matrix multiply ``Y = X . dequant(W)`` for GB300 (sm_103a).

The computation runs entirely in the CUDA kernels of ``libw4a16_gb300.so``
(C ABI: ``include/marlin.h``); this package marshals torch tensors into that
ABI.  PyTorch is used for device memory and streams only.  If the library is
missing, every call raises: there is no CPU or PyTorch fallback.

Typical use::

    pw = repack(q, scales, zeros, group)     # once, at load time (GPU kernel)
    ws = Workspace(max_M, K, N, group)       # once per layer shape
    y = gemm(x, pw, ws)                      # fp16 [M, N]
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _binding
from ._binding import MarlinError, status_string  # noqa: F401

__all__ = ["PackedWeights", "Workspace", "repack", "gemm", "gemm_into", "gemm_host", "device_status",
           "MarlinError", "status_string", "packed_layout", "SparsePackedWeights", "sparse_repack",
           "sparse_gemm", "sparse_gemm_into"]


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _on_current_device(*named) -> None:
    """The library launches on the current device with its current stream, so
    every tensor of a call must live there (a pointer into another GPU's memory
    would reach the kernel as a foreign address)."""
    cur = torch.cuda.current_device()
    for name, t in named:
        if t.device.index != cur:
            raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{cur}")


def _need_cuda(t: torch.Tensor, name: str, dtype=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def packed_layout(K: int, N: int, group: int, has_zeros: bool):
    return _binding.packed_layout(K, N, group, has_zeros)


@dataclass
class PackedWeights:
    """A repacked K x N weight: one uint8 buffer [codes | scales | zeros]."""
    buf: torch.Tensor
    K: int
    N: int
    group: int
    has_zeros: bool
    off_scales: int
    off_zeros: int

    @property
    def codes_ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def scales_ptr(self) -> int:
        return self.buf.data_ptr() + self.off_scales

    @property
    def zeros_ptr(self) -> int | None:
        return self.buf.data_ptr() + self.off_zeros if self.has_zeros else None


def repack(q: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor | None, group: int,
           out: torch.Tensor | None = None) -> PackedWeights:
    """GPTQ-order codes int32 [K/8, N], fp16 scales [K/group, N], optional
    packed zeros int32 [K/group, N/8] -> PackedWeights (marlin_repack)."""
    _need_cuda(q, "q", torch.int32)
    _need_cuda(scales, "scales", torch.float16)
    if zeros is not None:
        _need_cuda(zeros, "zeros", torch.int32)
    K, N = q.shape[0] * 8, q.shape[1]
    g = K if group == -1 else group
    nbytes, off_s, off_z = _binding.packed_layout(K, N, g, zeros is not None)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    elif out.numel() * out.element_size() < nbytes:
        raise ValueError("out is too small for the repacked weights")
    rc = _binding.repack_raw(q.data_ptr(), scales.data_ptr(),
                             zeros.data_ptr() if zeros is not None else None, K, N, g,
                             out.data_ptr(), _stream())
    if rc != _binding.OK:
        raise MarlinError(rc, "marlin_repack")
    return PackedWeights(out, K, N, g, zeros is not None, off_s, off_z)


class Workspace:
    """Device workspace for marlin_gemm, zeroed once; the kernel leaves it zeroed."""

    def __init__(self, max_M: int, K: int, N: int, group: int, device=None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        if dev.type != "cuda":
            raise ValueError("a workspace lives on a CUDA device")
        if dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.nbytes = _binding.workspace_bytes(max(max_M, 1), K, N, K if group == -1 else group,
                                               dev.index)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=dev)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


def gemm_into(x: torch.Tensor, w: PackedWeights, ws: Workspace, y: torch.Tensor,
              kernel: str = "auto") -> torch.Tensor:
    """y[M, N] = x[M, K] . dequant(W), fp16, on the current stream.  kernel:
    "auto" (by M), "warp" (warp-level kernel, M <= 32) or "tcgen05"."""
    _need_cuda(x, "x", torch.float16)
    _need_cuda(y, "y", torch.float16)
    M, K = x.shape
    if K != w.K or tuple(y.shape) != (M, w.N):
        raise ValueError("shape mismatch")
    _on_current_device(("x", x), ("weights", w.buf), ("workspace", ws.buf), ("y", y))
    if kernel == "auto":
        rc = _binding.gemm_raw(x.data_ptr(), w.codes_ptr, w.scales_ptr, w.zeros_ptr, y.data_ptr(), M, K,
                               w.N, w.group, ws.ptr, ws.nbytes, _stream())
    else:
        rc = _binding.gemm_ex_raw(x.data_ptr(), w.codes_ptr, w.scales_ptr, w.zeros_ptr, y.data_ptr(), M,
                                  K, w.N, w.group, ws.ptr, ws.nbytes, _binding.KERNELS[kernel], _stream())
    if rc != _binding.OK:
        raise MarlinError(rc, "marlin_gemm")
    return y


def gemm(x: torch.Tensor, w: PackedWeights, ws: Workspace) -> torch.Tensor:
    y = torch.empty((x.shape[0], w.N), dtype=torch.float16, device=x.device)
    return gemm_into(x, w, ws, y)


def gemm_host(x_host: torch.Tensor, x_dev: torch.Tensor, w: PackedWeights, ws: Workspace,
              y_dev: torch.Tensor, y_host: torch.Tensor) -> torch.Tensor:
    """y_host[M, N] = x_host[M, K] . dequant(W) through device staging buffers,
    all on the current stream (one library call: copy in, multiply, copy out).
    Host tensors should be pinned; y_host is complete once the stream is
    synchronised."""
    for t, n in ((x_host, "x_host"), (y_host, "y_host")):
        if t.device.type != "cpu" or t.dtype != torch.float16 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous fp16 host tensor")
    _need_cuda(x_dev, "x_dev", torch.float16)
    _need_cuda(y_dev, "y_dev", torch.float16)
    M, K = x_host.shape
    if (K != w.K or tuple(x_dev.shape) != (M, K) or tuple(y_dev.shape) != (M, w.N)
            or tuple(y_host.shape) != (M, w.N)):
        raise ValueError("shape mismatch")
    _on_current_device(("x_dev", x_dev), ("weights", w.buf), ("workspace", ws.buf), ("y_dev", y_dev))
    rc = _binding.gemm_host_raw(x_host.data_ptr(), x_dev.data_ptr(), w.codes_ptr, w.scales_ptr,
                                w.zeros_ptr, y_dev.data_ptr(), y_host.data_ptr(), M, K, w.N, w.group,
                                ws.ptr, ws.nbytes, _stream())
    if rc != _binding.OK:
        raise MarlinError(rc, "marlin_gemm_host")
    return y_host


def device_status(ws: Workspace) -> int:
    """Synchronise the current stream and read/clear the kernel status word."""
    return _binding.last_device_status(ws.ptr, _stream())


# ---- 2:4-sparse variant ----------------------------------------------------------

@dataclass
class SparsePackedWeights:
    """A repacked 2:4-sparse K x N weight: one uint8 buffer [codes | meta | scales | zeros]."""
    buf: torch.Tensor
    K: int
    N: int
    group: int
    has_zeros: bool
    off_meta: int
    off_scales: int
    off_zeros: int
    bad_groups: int  # groups of four rows with more than two non-zero weights (0 for 2:4 weights)

    @property
    def codes_ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def meta_ptr(self) -> int:
        return self.buf.data_ptr() + self.off_meta

    @property
    def scales_ptr(self) -> int:
        return self.buf.data_ptr() + self.off_scales

    @property
    def zeros_ptr(self) -> int | None:
        return self.buf.data_ptr() + self.off_zeros if self.has_zeros else None


def sparse_repack(q: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor | None, group: int,
                  strict: bool = True) -> SparsePackedWeights:
    """2:4-sparse GPTQ-order codes (same input formats as repack) ->
    SparsePackedWeights (marlin_sparse_repack).  Synchronises the current
    stream to read the count of groups that are not 2:4; strict: raise if any."""
    _need_cuda(q, "q", torch.int32)
    _need_cuda(scales, "scales", torch.float16)
    if zeros is not None:
        _need_cuda(zeros, "zeros", torch.int32)
    K, N = q.shape[0] * 8, q.shape[1]
    g = K if group == -1 else group
    nbytes, off_m, off_s, off_z = _binding.sparse_packed_layout(K, N, g, zeros is not None)
    out = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    bad = torch.zeros(1, dtype=torch.int32, device=q.device)
    rc = _binding.sparse_repack_raw(q.data_ptr(), scales.data_ptr(),
                                    zeros.data_ptr() if zeros is not None else None, K, N, g,
                                    out.data_ptr(), bad.data_ptr(), _stream())
    if rc != _binding.OK:
        raise MarlinError(rc, "marlin_sparse_repack")
    nbad = int(bad.item())
    if strict and nbad:
        raise ValueError(f"weights are not 2:4 sparse: {nbad} groups of four rows have more than "
                         "two codes that differ from the zero point")
    return SparsePackedWeights(out, K, N, g, zeros is not None, off_m, off_s, off_z, nbad)


def sparse_gemm_into(x: torch.Tensor, w: SparsePackedWeights, ws: Workspace, y: torch.Tensor) -> torch.Tensor:
    """y[M, N] = x[M, K] . dequant(W) for 2:4-sparse W, fp16, on the current stream."""
    _need_cuda(x, "x", torch.float16)
    _need_cuda(y, "y", torch.float16)
    M, K = x.shape
    if K != w.K or tuple(y.shape) != (M, w.N):
        raise ValueError("shape mismatch")
    _on_current_device(("x", x), ("weights", w.buf), ("workspace", ws.buf), ("y", y))
    rc = _binding.sparse_gemm_raw(x.data_ptr(), w.codes_ptr, w.meta_ptr, w.scales_ptr, w.zeros_ptr,
                                  y.data_ptr(), M, K, w.N, w.group, ws.ptr, ws.nbytes, _stream())
    if rc != _binding.OK:
        raise MarlinError(rc, "marlin_sparse_gemm")
    return y


def sparse_gemm(x: torch.Tensor, w: SparsePackedWeights, ws: Workspace) -> torch.Tensor:
    y = torch.empty((x.shape[0], w.N), dtype=torch.float16, device=x.device)
    return sparse_gemm_into(x, w, ws, y)
