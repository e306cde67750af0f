"""Failure detection without a GPU fault: a bounded wait that runs out.

Every wait inside the kernels gives up after 2 s of global time, records
MARLIN_ERR_TIMEOUT in the workspace's status word, and lets the kernel drain
its own copies and MMAs and exit.  The waits are made to expire through a word
that nothing sets: the reducers of both kernels rely on the tagged partial
words alone, but in the bounds-checked (MARLIN_DEBUG) build they also wait for
their tile's word in the workspace's counter block to be non-negative; the
tests preset it negative and call through that build's C ABI.

The host must then read MARLIN_ERR_TIMEOUT, and the context must stay usable:
after re-zeroing the workspace the same call gives the oracle's result.
"""
import ctypes

import numpy as np
import pytest

import oracle
from workloads import Problem, make_inputs, make_activations, make_sparse_weights

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def dbg():
    from w4a16_mixed_precision_gb300 import _binding
    from w4a16_mixed_precision_gb300 import build as cuda_build
    return _binding.open_library(cuda_build.build(debug=True))


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _hold(ws_buf, n_tiles):
    # the counter block follows the 256-byte status block: one int32 per tile
    ws_buf[256:256 + 4 * n_tiles].view(torch.int32).fill_(-1000000)


def _workspace(lib, M, K, N, g):
    nb = ctypes.c_size_t()
    assert lib.marlin_workspace_bytes(M, K, N, g, 0, ctypes.byref(nb)) == 0
    return torch.zeros(nb.value, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("M,kernel", [(1, 1), (64, 2)])   # warp-level kernel, tcgen05 kernel
def test_expired_wait_dense(dbg, M, kernel):
    import w4a16_mixed_precision_gb300 as w4
    K, N, g = 4096, 1024, 128
    inp = make_inputs(Problem("timeout", M, K, N, g, False))
    dev = torch.device("cuda", 0)
    pw = w4.repack(torch.from_numpy(inp.Qp).to(dev), torch.from_numpy(inp.S).to(dev), None, g)
    x = torch.from_numpy(inp.X).to(dev)
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    ws = _workspace(dbg, M, K, N, g)

    def call():
        base = pw.buf.data_ptr()
        return dbg.marlin_gemm_ex(x.data_ptr(), base, base + pw.off_scales, None, y.data_ptr(), M, K, N, g,
                                  ws.data_ptr(), ws.numel(), kernel, _stream())

    _hold(ws, N // 128)
    assert call() == 0
    torch.cuda.synchronize()
    assert dbg.marlin_last_device_status(ws.data_ptr(), _stream()) == 6   # MARLIN_ERR_TIMEOUT
    ws.zero_()
    assert call() == 0
    assert dbg.marlin_last_device_status(ws.data_ptr(), _stream()) == 0
    ok, err, ratio = oracle.within_tolerance(y.cpu().numpy(), oracle.w4a16(inp.X, inp.Qp, inp.S, None, g, N))
    assert ok, f"max abs err {err}"


def test_expired_wait_on_the_sparse_path(dbg):
    """The same on the 2:4-sparse path (the sparse instantiation of the
    warp-level kernel shares its bounded waits)."""
    M, K, N, g = 4, 4096, 1024, 128
    Qp, S, _ = make_sparse_weights(K, N, g, False, seed=77)
    X = make_activations(M, K, seed=78)
    b, mo, so, zo = (ctypes.c_size_t() for _ in range(4))
    assert dbg.marlin_sparse_packed_layout(K, N, g, 0, *(ctypes.byref(v) for v in (b, mo, so, zo))) == 0
    out = torch.empty(b.value, dtype=torch.uint8, device="cuda")
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, s, x = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (Qp, S, X))
    assert dbg.marlin_sparse_repack(q.data_ptr(), s.data_ptr(), None, K, N, g, out.data_ptr(), bad.data_ptr(),
                                    _stream()) == 0
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = _workspace(dbg, M, K, N, g)
    base = out.data_ptr()

    def call():
        return dbg.marlin_sparse_gemm(x.data_ptr(), base, base + mo.value, base + so.value, None, y.data_ptr(),
                                      M, K, N, g, ws.data_ptr(), ws.numel(), _stream())

    _hold(ws, N // 128)
    assert call() == 0
    torch.cuda.synchronize()
    assert dbg.marlin_last_device_status(ws.data_ptr(), _stream()) == 6
    ws.zero_()
    assert call() == 0
    assert dbg.marlin_last_device_status(ws.data_ptr(), _stream()) == 0
    assert int(bad.item()) == 0
    ok, err, ratio = oracle.within_tolerance(y.cpu().numpy(), oracle.w4a16(X, Qp, S, None, g, N))
    assert ok, f"max abs err {err}"
