"""Both fused kernels at batch sizes outside their default range.

The library sends M <= 16 to the warp-level kernel and larger M to the tcgen05
kernel; W4A16_SMALL_M_MAX (read once per process) moves that split.  Each case
runs in a child process with the split moved, so that the tcgen05 kernel is
checked at decode batches down to M = 1 and the warp-level kernel up to its
largest batch (M = 32), against the CPU oracle.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import torch
import oracle
from workloads import Problem, make_inputs
from gpu_util import run_cuda
out = []
for (M, K, N, g, asym) in {cases!r}:
    p = Problem("split", M, K, N, g, asym)
    inp = make_inputs(p)
    y, _, _ = run_cuda(inp.X, inp.Qp, inp.S, inp.Zp, g)
    ok, err, ratio = oracle.within_tolerance(y, oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, g, N))
    out.append([M, bool(ok), float(err)])
print(json.dumps(out))
"""


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _run(small_m_max, cases):
    env = dict(os.environ, W4A16_SMALL_M_MAX=str(small_m_max))
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), cases=cases)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_tcgen05_kernel_at_decode_batches():
    cases = [(1, 1024, 640, 128, False), (8, 2048, 384, 128, True), (17, 1024, 512, 1024, False),
             (24, 4096, 1280, 128, False)]
    for M, ok, err in _run(0, cases):
        assert ok, f"M={M}: max abs err {err}"


def test_warp_level_kernel_up_to_its_largest_batch():
    cases = [(25, 1024, 640, 128, True), (32, 2048, 1024, 128, False), (31, 4096, 384, 4096, True),
             (28, 384, 256, 128, True)]   # the last: 128-row units (K % 256 = 128), four token blocks
    for M, ok, err in _run(32, cases):
        assert ok, f"M={M}: max abs err {err}"


def test_forced_kernels_and_tuner_match_the_oracle():
    """marlin_gemm_ex with each kernel forced, on one workspace sized for M
    (which must serve both), and the per-shape tuner's choice."""
    import numpy as np

    import oracle
    import w4a16_mixed_precision_gb300 as w4
    from w4a16_mixed_precision_gb300 import _binding as b
    from w4a16_mixed_precision_gb300.tune import best_kernel, tuned_gemm_into
    from workloads import Problem, make_inputs
    dev = torch.device("cuda", 0)
    for M, asym in ((5, True), (24, False), (32, True)):
        p = Problem("forced", M, 1024, 640, 128, asym)
        inp = make_inputs(p)
        pw = w4.repack(torch.from_numpy(inp.Qp).to(dev), torch.from_numpy(inp.S).to(dev),
                       torch.from_numpy(inp.Zp).to(dev) if asym else None, 128)
        ws = w4.Workspace(M, p.K, p.N, 128)
        x = torch.from_numpy(inp.X).to(dev)
        ref = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, 128, p.N)
        for k in ("warp", "tcgen05"):
            y = torch.empty((M, p.N), dtype=torch.float16, device=dev)
            w4.gemm_into(x, pw, ws, y, kernel=k)
            torch.cuda.synchronize()
            assert w4.device_status(ws) == 0
            ok, err, _ = oracle.within_tolerance(y.cpu().numpy(), ref)
            assert ok, f"M={M} kernel={k}: max abs err {err}"
        assert best_kernel(x, pw, ws) in ("warp", "tcgen05")
        y = torch.empty((M, p.N), dtype=torch.float16, device=dev)
        tuned_gemm_into(x, pw, ws, y)
        torch.cuda.synchronize()
        ok, err, _ = oracle.within_tolerance(y.cpu().numpy(), ref)
        assert ok
    # the warp-level kernel has no M > 32 variant; an unknown kernel id is rejected
    ws = w4.Workspace(40, 1024, 640, 128)
    x = torch.zeros((40, 1024), dtype=torch.float16, device=dev)
    y = torch.empty((40, 640), dtype=torch.float16, device=dev)
    assert b.gemm_ex_raw(x.data_ptr(), pw.codes_ptr, pw.scales_ptr, None, y.data_ptr(), 40, 1024, 640, 128,
                         ws.ptr, ws.nbytes, 1, 0) == b.ERR_UNSUPPORTED
    assert b.gemm_ex_raw(x.data_ptr(), pw.codes_ptr, pw.scales_ptr, None, y.data_ptr(), 40, 1024, 640, 128,
                         ws.ptr, ws.nbytes, 7, 0) == b.ERR_INVALID_ARG
    assert np.isfinite(1.0)
