"""The entry point for callers that cannot allocate device memory.

marlin_gemm_no_alloc keeps its scratch in a static array of the library instead
of a caller-provided workspace, for operators whose host framework owns all
device memory or whose path cannot afford cudaMalloc's synchronisation.  Its
results must be bit-identical to marlin_gemm's (called through the C ABI with a
workspace: same kernel, same fixed reduction order), on consecutive calls that
reuse the shared array, and both must match the CPU oracle within the parity
tolerance.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import pytest

import oracle
from workloads import Problem, make_inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _prepared(p):
    import w4a16_mixed_precision_gb300 as w4
    dev = torch.device("cuda", 0)
    inp = make_inputs(p)
    pw = w4.repack(torch.from_numpy(inp.Qp).to(dev), torch.from_numpy(inp.S).to(dev),
                   torch.from_numpy(inp.Zp).to(dev) if inp.Zp is not None else None, p.group)
    x = torch.from_numpy(inp.X).to(dev)
    return pw, x


def _no_alloc(pw, x, p):
    from w4a16_mixed_precision_gb300 import _binding as b
    y = torch.empty((p.M, p.N), dtype=torch.float16, device=x.device)
    rc = b.gemm_no_alloc_raw(x.data_ptr(), pw.codes_ptr, pw.scales_ptr, pw.zeros_ptr, y.data_ptr(),
                             p.M, p.K, p.N, p.group, torch.cuda.current_stream().cuda_stream)
    assert rc == b.OK, b.status_string(rc)
    return y


def _with_workspace(pw, x, p):
    import w4a16_mixed_precision_gb300 as w4
    ws = w4.Workspace(p.M, p.K, p.N, p.group)
    y = w4.gemm(x, pw, ws)
    torch.cuda.synchronize()
    assert w4.device_status(ws) == 0
    return y


def test_no_alloc_matches_workspace_entry_point_on_consecutive_calls():
    # split column tiles (counters and partials in the shared array) on the
    # warp-level kernel, a different shape with explicit zeros, a batch of 80
    # tokens on the tcgen05 kernel (near the array's limit), then the first
    # problem again
    problems = [Problem("noalloc", 16, 4096, 4096, 128, False),
                Problem("noalloc", 5, 2048, 1024, 128, True),
                Problem("noalloc", 80, 4096, 4096, 128, False),
                Problem("noalloc", 16, 4096, 4096, 128, False)]
    for p in problems:
        pw, x = _prepared(p)
        y_ws = _with_workspace(pw, x, p).cpu()
        y_a = _no_alloc(pw, x, p)
        y_b = _no_alloc(pw, x, p)       # two calls in a row on the same scratch
        torch.cuda.synchronize()
        for y in (y_a, y_b):
            assert torch.equal(y.cpu(), y_ws), f"{p.key}: differs from marlin_gemm"
        inp = make_inputs(p)
        y_ref = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, p.group, p.N)
        ok, err, ratio = oracle.within_tolerance(y_ws.numpy(), y_ref)
        assert ok, f"{p.key}: max abs err {err}, worst ratio {ratio}"


def test_no_alloc_rejects_problems_beyond_its_scratch():
    from w4a16_mixed_precision_gb300 import _binding as b
    p = Problem("noalloc-big", 200, 1024, 1024, 128, False)
    pw, x = _prepared(p)
    y = torch.full((p.M, p.N), 7.0, dtype=torch.float16, device=x.device)
    rc = b.gemm_no_alloc_raw(x.data_ptr(), pw.codes_ptr, pw.scales_ptr, None, y.data_ptr(),
                             p.M, p.K, p.N, p.group, torch.cuda.current_stream().cuda_stream)
    assert rc == b.ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())   # nothing was launched
