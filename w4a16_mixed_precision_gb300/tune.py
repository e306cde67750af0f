"""Per-shape kernel choice by measurement.

marlin_gemm picks its kernel by M alone (the warp-level one up to M = 16).
This tuner times both kernels on the caller's own weights and workspace for a
given (M, K, N, group, zeros) and remembers the faster one, for callers whose
shapes sit near the crossover.  Timing: CUDA graphs of `reps` back-to-back
calls, CUDA events around a replay, after a warm-up replay.
"""
from __future__ import annotations

import torch

from . import PackedWeights, Workspace, gemm_into

_choice: dict[tuple, str] = {}


def _time(fn, reps: int) -> float:
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        fn()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
        g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def best_kernel(x: torch.Tensor, w: PackedWeights, ws: Workspace, reps: int = 20) -> str:
    """"warp" or "tcgen05", whichever is faster for this x's M and these weights
    (cached per (M, K, N, group, zeros)).  M > 32 is always "tcgen05"."""
    M = x.shape[0]
    key = (M, w.K, w.N, w.group, w.has_zeros)
    if key in _choice:
        return _choice[key]
    if M > 32:
        _choice[key] = "tcgen05"
        return "tcgen05"
    y = torch.empty((M, w.N), dtype=torch.float16, device=x.device)
    t = {k: _time(lambda k=k: gemm_into(x, w, ws, y, kernel=k), reps) for k in ("warp", "tcgen05")}
    _choice[key] = min(t, key=t.get)
    return _choice[key]


def tuned_gemm_into(x: torch.Tensor, w: PackedWeights, ws: Workspace, y: torch.Tensor) -> torch.Tensor:
    """gemm_into with the measured-best kernel for this shape."""
    return gemm_into(x, w, ws, y, kernel=best_kernel(x, w, ws))
