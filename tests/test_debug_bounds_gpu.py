"""The bounds-checked build (-DMARLIN_DEBUG) on the parity cases.

libw4a16_gb300_debug.so is the same sources compiled with MARLIN_DEBUG: every
global, shared-memory and tensor-memory address the kernels form (weight and
scale copies, X tiles, stage offsets, accumulator and A-slot columns, partial
words, tile counters, Y stores) is checked against the extent of its buffer;
a failed check skips the access and sets MARLIN_ERR_BOUNDS in the status word
instead of faulting.  Here the small parity cases, both kernels and the 2:4
path run through that library's C ABI: every call must report MARLIN_OK and
match the CPU oracle within the parity tolerance.
"""
import ctypes

import numpy as np
import pytest

import oracle
from workloads import Problem, make_inputs, make_sparse_weights, make_activations

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

from test_gemm_gpu import SMALL_CASES  # noqa: E402


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from w4a16_mixed_precision_gb300 import _binding
    from w4a16_mixed_precision_gb300 import build as cuda_build
    torch.cuda.set_device(0)
    return _binding.open_library(cuda_build.build(debug=True))


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.device("cuda", 0))


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _workspace(lib, M, K, N, g):
    b = ctypes.c_size_t()
    assert lib.marlin_workspace_bytes(max(M, 1), K, N, g, 0, ctypes.byref(b)) == 0
    return torch.zeros(b.value, dtype=torch.uint8, device="cuda")


def _dense(lib, X, Qp, S, Zp, g, M, K, N, kernel=0):
    b, so, zo = (ctypes.c_size_t() for _ in range(3))
    assert lib.marlin_packed_layout(K, N, g, int(Zp is not None), ctypes.byref(b), ctypes.byref(so),
                                    ctypes.byref(zo)) == 0
    out = torch.empty(b.value, dtype=torch.uint8, device="cuda")
    q, s, z, x = _t(Qp), _t(S), (_t(Zp) if Zp is not None else None), _t(X)
    assert lib.marlin_repack(q.data_ptr(), s.data_ptr(), _ptr(z), K, N, g, out.data_ptr(), _stream()) == 0
    ws = _workspace(lib, M, K, N, g)
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    rc = lib.marlin_gemm_ex(x.data_ptr(), out.data_ptr(), out.data_ptr() + so.value,
                            out.data_ptr() + zo.value if Zp is not None else None, y.data_ptr(), M, K, N, g,
                            ws.data_ptr(), ws.numel(), kernel, _stream())
    assert rc == 0, rc
    status = lib.marlin_last_device_status(ws.data_ptr(), _stream())
    assert status == 0, f"device status {status} (7 = bounds check failed)"
    return y.cpu().numpy()


@pytest.mark.parametrize("M,K,N,g,asym", SMALL_CASES)
def test_bounds_checked_parity_small(dbg, M, K, N, g, asym):
    p = Problem("parity", M, K, N, g, asym)
    inp = make_inputs(p)
    y = _dense(dbg, inp.X, inp.Qp, inp.S, inp.Zp, g, M, K, N)
    ok, err, ratio = oracle.within_tolerance(y, oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, g, N))
    assert ok, f"max abs err {err}, worst ratio {ratio}"


@pytest.mark.parametrize("M,kernel", [(1, 1), (17, 1), (32, 1), (1, 2), (24, 2)])
def test_bounds_checked_forced_kernels(dbg, M, kernel):
    """Each kernel outside its default range (1: warp-level, 2: tcgen05)."""
    K, N, g = 2048, 1024, 128
    p = Problem("forced", M, K, N, g, True)
    inp = make_inputs(p)
    y = _dense(dbg, inp.X, inp.Qp, inp.S, inp.Zp, g, M, K, N, kernel)
    ok, err, ratio = oracle.within_tolerance(y, oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, g, N))
    assert ok, f"max abs err {err}, worst ratio {ratio}"


@pytest.mark.parametrize("M,asym", [(1, False), (12, True), (32, False)])
def test_bounds_checked_sparse(dbg, M, asym):
    K, N, g = 2048, 768, 128
    Qp, S, Zp = make_sparse_weights(K, N, g, asym, seed=5 + M)
    X = make_activations(M, K, seed=6 + M)
    b, mo, so, zo = (ctypes.c_size_t() for _ in range(4))
    assert dbg.marlin_sparse_packed_layout(K, N, g, int(asym), *(ctypes.byref(v) for v in (b, mo, so, zo))) == 0
    out = torch.empty(b.value, dtype=torch.uint8, device="cuda")
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, s, z, x = _t(Qp), _t(S), (_t(Zp) if asym else None), _t(X)
    assert dbg.marlin_sparse_repack(q.data_ptr(), s.data_ptr(), _ptr(z), K, N, g, out.data_ptr(),
                                    bad.data_ptr(), _stream()) == 0
    ws = _workspace(dbg, M, K, N, g)
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    base = out.data_ptr()
    assert dbg.marlin_sparse_gemm(x.data_ptr(), base, base + mo.value, base + so.value,
                                  base + zo.value if asym else None, y.data_ptr(), M, K, N, g, ws.data_ptr(),
                                  ws.numel(), _stream()) == 0
    assert dbg.marlin_last_device_status(ws.data_ptr(), _stream()) == 0
    assert int(bad.item()) == 0
    kc, ki, _ = oracle.sparse_compress(Qp, Zp if asym else None, K, N, g)
    y_ref = oracle.w4a16_sparse(X, kc, ki, S, Zp if asym else None, g, N)
    ok, err, ratio = oracle.within_tolerance(y.cpu().numpy(), y_ref)
    assert ok, f"max abs err {err}, worst ratio {ratio}"


def test_bounds_status_is_reported_and_cleared(dbg):
    """The host side of the report: a status word with the bounds bit set (and a
    site in the next word), written from the host, comes back as
    MARLIN_ERR_BOUNDS and both words are cleared."""
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ws[:8].view(torch.int32).copy_(torch.tensor([2, 12], dtype=torch.int32))
    assert dbg.marlin_last_device_status(ws.data_ptr(), _stream()) == 7
    assert dbg.marlin_status_string(7).decode() == "MARLIN_ERR_BOUNDS"
    assert int(ws[:8].view(torch.int32).abs().sum().item()) == 0
    assert dbg.marlin_last_device_status(ws.data_ptr(), _stream()) == 0
