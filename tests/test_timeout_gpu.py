"""Failure detection without a GPU fault: a bounded wait that runs out.

Every wait inside the kernels gives up after 2 s of global time, records
MARLIN_ERR_TIMEOUT in the workspace's status word, and lets the kernel drain
its own copies and MMAs and exit.  Here the tile arrival counters of the
workspace are preset to a value the contributors can never raise to the
expected count (a flag that nothing sets), so the reducing CTAs' waits expire.
The host must then read MARLIN_ERR_TIMEOUT, and the context must stay usable:
after re-zeroing the workspace the same call gives the oracle's result.
"""
import numpy as np
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


@pytest.mark.parametrize("M", [1, 64])   # warp-level kernel, tcgen05 kernel
def test_expired_wait_is_reported_and_context_survives(M):
    import w4a16_mixed_precision_gb300 as w4
    from w4a16_mixed_precision_gb300 import _binding as b
    p = Problem("timeout", M, 4096, 1024, 128, False)
    inp = make_inputs(p)
    dev = torch.device("cuda", 0)
    pw = w4.repack(torch.from_numpy(inp.Qp).to(dev), torch.from_numpy(inp.S).to(dev), None, 128)
    x = torch.from_numpy(inp.X).to(dev)
    ws = w4.Workspace(M, p.K, p.N, p.group)
    # counters follow the 256-byte status block: [m_tiles * n_tiles] int32
    counters = ws.buf[256:256 + 4 * (p.N // 128)].view(torch.int32)
    counters.fill_(-1000000)
    y = w4.gemm(x, pw, ws)
    torch.cuda.synchronize()
    rc = b.last_device_status(ws.ptr, torch.cuda.current_stream().cuda_stream)
    assert rc == b.ERR_TIMEOUT, b.status_string(rc)
    # the status word was cleared by the read; the context still works
    ws.buf.zero_()
    y = w4.gemm(x, pw, ws)
    torch.cuda.synchronize()
    assert w4.device_status(ws) == 0
    ok, err, ratio = oracle.within_tolerance(y.cpu().numpy(), oracle.w4a16(inp.X, inp.Qp, inp.S, None, 128, p.N))
    assert ok, f"max abs err {err}"


def test_expired_wait_on_the_sparse_path():
    """The same on the 2:4-sparse path (the sparse instantiation of the
    warp-level kernel shares its bounded waits)."""
    import w4a16_mixed_precision_gb300 as w4
    from w4a16_mixed_precision_gb300 import _binding as b
    from workloads import make_activations, make_sparse_weights
    M, K, N, g = 4, 4096, 1024, 128
    Qp, S, _ = make_sparse_weights(K, N, g, False, seed=77)
    X = make_activations(M, K, seed=78)
    dev = torch.device("cuda", 0)
    pw = w4.sparse_repack(torch.from_numpy(Qp).to(dev), torch.from_numpy(S).to(dev), None, g)
    x = torch.from_numpy(X).to(dev)
    ws = w4.Workspace(M, K, N, g)
    ws.buf[256:256 + 4 * (N // 128)].view(torch.int32).fill_(-1000000)
    w4.sparse_gemm(x, pw, ws)
    torch.cuda.synchronize()
    rc = b.last_device_status(ws.ptr, torch.cuda.current_stream().cuda_stream)
    assert rc == b.ERR_TIMEOUT, b.status_string(rc)
    ws.buf.zero_()
    y = w4.sparse_gemm(x, pw, ws)
    torch.cuda.synchronize()
    assert w4.device_status(ws) == 0
    ok, err, ratio = oracle.within_tolerance(y.cpu().numpy(), oracle.w4a16(X, Qp, S, None, g, N))
    assert ok, f"max abs err {err}"
