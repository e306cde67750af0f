"""A linear layer over the fused W4A16 kernel: y = x . dequant(W).

The pages describe the kernel as used through a torch module that converts and
holds the compressed weights ("Marlin Project Overview", section "Requirements
and Usage": a torch module converts and holds the compressed data; users with
suitably prepared weights and scales may also call the kernel directly) and repack at load time ("Marlin /
GPTQ-Marlin", section "Tiled layout et repacking").  Here construction repacks
once on the GPU and every forward call is one marlin_gemm launch; there is no
bias and no other arithmetic outside the kernel.

With sparse=True the weights must be 2:4 ("Marlin", section "支持 2:4 稀疏加速":
two of every four weights zero at fixed positions): the layer also holds the
2:4 form.  marlin_sparse_gemm serves every M, but above 32 rows each further
32-row m-tile dequantises the weights again, and on GB300 the dense tcgen05
kernel was measured faster there (0.52-0.99x for the 2:4 path at M = 33..256
on the Llama-2-7B shapes) and, since its reducer's first poll overlaps its last
MMAs, at M = 32 too (0.97-1.00x for the 2:4 path), while the 2:4 path is
1.12-1.27x faster at M <= 16.  So the layer sends batches of up to 16 rows to
marlin_sparse_gemm and larger ones to the dense kernel.
"""
from __future__ import annotations

import numpy as np
import torch

from . import Workspace, gemm_into, repack, sparse_gemm_into, sparse_repack
from .formats import awq_to_gptq


class W4A16Linear(torch.nn.Module):
    """y[..., N] = x[..., K] . dequant(W)[K, N], fp16 in and out, fp32 accumulation."""

    # Largest batch sent to the 2:4 path.  Measured on the 7B shapes: 1.12-1.27x
    # faster than the dense call at M <= 16, 0.97-1.00x at M = 32 (where the
    # dense call runs the tcgen05 kernel).
    SPARSE_MAX_M = 16

    def __init__(self, qweight: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor | None = None,
                 group: int = 128, device=None, sparse: bool = False):
        """qweight: GPTQ-order int32 [K/8, N]; scales fp16 [K/group, N]; qzeros
        int32 [K/group, N/8] or None (z = 8); group 128, a multiple of 128
        dividing K, or -1/K for one scale per column.  sparse: the weights are
        2:4 (raises otherwise); batches of M <= SPARSE_MAX_M use the sparse path."""
        super().__init__()
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        q = qweight.to(dev, torch.int32).contiguous()
        s = scales.to(dev, torch.float16).contiguous()
        z = None if qzeros is None else qzeros.to(dev, torch.int32).contiguous()
        self.K, self.N = q.shape[0] * 8, q.shape[1]
        self.group = self.K if group == -1 else group
        self.packed = repack(q, s, z, self.group)
        self.sparse_packed = sparse_repack(q, s, z, self.group) if sparse else None
        self._ws = None
        self._ws_m = 0

    @classmethod
    def from_awq(cls, qweight: np.ndarray, scales, qzeros: np.ndarray | None = None, group: int = 128,
                 device=None) -> "W4A16Linear":
        """From AWQ-order int32 codes [K, N/8] (and zeros [K/group, N/8])."""
        codes, zeros = awq_to_gptq(np.asarray(qweight), None if qzeros is None else np.asarray(qzeros))
        return cls(torch.from_numpy(codes), torch.as_tensor(scales),
                   None if zeros is None else torch.from_numpy(zeros), group, device)

    def _workspace(self, M: int) -> Workspace:
        if self._ws is None or M > self._ws_m:
            self._ws = Workspace(M, self.K, self.N, self.group, device=self.packed.buf.device)
            self._ws_m = M
        return self._ws

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.shape[-1] != self.K:
            raise ValueError(f"expected last dimension {self.K}, got {x.shape[-1]}")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.K).contiguous()
        y = torch.empty((x2.shape[0], self.N), dtype=torch.float16, device=x2.device)
        M = x2.shape[0]
        if M > 0 and self.sparse_packed is not None and M <= self.SPARSE_MAX_M:
            sparse_gemm_into(x2, self.sparse_packed, self._workspace(M), y)
        elif M > 0:
            gemm_into(x2, self.packed, self._workspace(M), y)
        return y.reshape(*lead, self.N)
