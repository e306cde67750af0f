"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
CUDA path through the C ABI, and bring results back as numpy."""
from __future__ import annotations

import numpy as np
import torch


def device():
    return torch.device("cuda", 0)


def run_cuda(X: np.ndarray, Qp: np.ndarray, S: np.ndarray, Zp, group: int, ws=None, reps: int = 1):
    """Y (numpy float16) of the CUDA path, plus the PackedWeights and Workspace used."""
    import w4a16_mixed_precision_gb300 as w4
    dev = device()
    q = torch.from_numpy(np.ascontiguousarray(Qp)).to(dev)
    s = torch.from_numpy(np.ascontiguousarray(S)).to(dev)
    z = torch.from_numpy(np.ascontiguousarray(Zp)).to(dev) if Zp is not None else None
    x = torch.from_numpy(np.ascontiguousarray(X)).to(dev)
    K, N = Qp.shape[0] * 8, Qp.shape[1]
    pw = w4.repack(q, s, z, group)
    if ws is None:
        ws = w4.Workspace(X.shape[0], K, N, group)
    outs = []
    for _ in range(reps):
        outs.append(w4.gemm(x, pw, ws))
    torch.cuda.synchronize()
    assert w4.device_status(ws) == 0, "kernel reported an expired wait"
    ys = [o.cpu().numpy() for o in outs]
    return (ys[0] if reps == 1 else ys), pw, ws
