"""GPU parity of the fused W4A16 kernel (through the C ABI) against the CPU oracle.

Tolerance: |y_gpu - y_ref| <= 1e-2 + 2e-3*|y_ref| element by element, y_ref the
binary64 oracle; exact (bit-identical) where the arithmetic makes the fp32
accumulation exact (identity weights, one-hot activations).
"""
import numpy as np
import pytest

import oracle
from workloads import Problem, make_inputs, pack_codes, pack_zeros

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


from gpu_util import run_cuda  # noqa: E402


SMALL_CASES = [
    # M, K, N, group, asym
    (1, 128, 128, 128, False),
    (1, 4096, 384, 128, False),
    (5, 256, 384, 128, True),
    (16, 1024, 512, 128, False),       # largest batch of the warp-level kernel by default
    (17, 512, 256, 128, True),         # smallest batch of the tcgen05 kernel by default
    (24, 1024, 640, 128, False),
    (25, 1024, 640, 128, True),
    (32, 2048, 1024, 128, False),
    (33, 1024, 640, 1024, True),       # one scale per column, ragged M
    (48, 2048, 768, 128, True),
    (64, 1536, 512, 512, False),       # group 512
    (12, 2048, 640, 256, True),        # group 256, warp-level kernel
    (80, 2048, 384, 256, False),       # group 256, tcgen05 kernel
    (300, 1024, 256, 1024, True),      # one scale per column, two m-tiles
    (100, 768, 256, 128, False),
    (12, 384, 256, 128, True),         # K % 256 = 128: 128-row units, two token blocks
    (16, 640, 384, 128, False),
    (128, 1024, 384, 128, True),
    (200, 512, 1280, 128, False),
    (256, 512, 384, 128, False),
    (257, 512, 256, 128, True),        # two m-tiles, 1-row tail
    (129, 512, 384, 256, False),       # bn = 144: the second issuer's columns are N = 16
    (256, 1024, 512, 128, True),       # bn = 256 exactly, explicit zeros
    (1, 128, 128, 128, True),          # one unit, one tile, explicit zeros
    (40, 128, 256, 128, False),        # K of a single 128-row unit on the tcgen05 kernel
    (600, 1024, 512, 128, False),
    # more units than SMs, split unevenly (140 CTAs on 152 SMs: up to 15 pieces per tile):
    # the tcgen05 reducer copies its first contributors' partial tiles in bulk and
    # polls the rest
    (128, 4096, 1280, 128, False),
    (64, 4096, 1280, 128, True),
]


@pytest.mark.parametrize("M,K,N,g,asym", SMALL_CASES)
def test_parity_small(M, K, N, g, asym):
    p = Problem("parity", M, K, N, g, asym)
    inp = make_inputs(p)
    y, _, _ = run_cuda(inp.X, inp.Qp, inp.S, inp.Zp, g)
    y_ref = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, g, N)
    ok, err, ratio = oracle.within_tolerance(y, y_ref)
    assert ok, f"max abs err {err}, worst ratio {ratio}"


@pytest.mark.parametrize("K", [256, 1024])
def test_identity_weights_exact(K):
    """W = I (q = 9 on the diagonal, 8 elsewhere, s = 1): Y == X bit for bit."""
    N = K
    q = np.full((K, N), 8, np.uint32)
    q[np.arange(K), np.arange(N)] = 9
    S = np.ones((K // 128, N), np.float16)
    X = make_inputs(Problem("id", 19, K, N, 128, False)).X
    y, _, _ = run_cuda(X, pack_codes(q), S, None, 128)
    assert np.array_equal(y.view(np.uint16), X.view(np.uint16))


def test_permutation_weights_exact():
    K, N = 512, 512
    rng = np.random.default_rng(11)
    pi = rng.permutation(N)
    z = rng.integers(0, 15, size=(K // 128, N)).astype(np.uint32)
    q = np.repeat(z, 128, axis=0)
    q[np.arange(K), pi] += 1
    S = np.ones((K // 128, N), np.float16)
    X = make_inputs(Problem("perm", 7, K, N, 128, True)).X
    y, _, _ = run_cuda(X, pack_codes(q), S, pack_zeros(z), 128)
    expect = np.empty_like(X)
    expect[:, pi] = X
    assert np.array_equal(y.view(np.uint16), expect.view(np.uint16))


@pytest.mark.parametrize("asym,g", [(False, 128), (True, 128), (True, 1024)])
def test_onehot_rows_give_exact_dequant(asym, g):
    """Row m of X is one-hot at k_m: Y[m] = dequant(W)[k_m] exactly (one product,
    the rest zeros, is exact in fp32), so the GPU dequantisation must equal the
    oracle's bit for bit -- one rounding of (q - z) * s."""
    K, N = 1024, 384
    p = Problem("onehot", 1, K, N, g, asym)
    inp = make_inputs(p)
    ks = np.concatenate([np.arange(0, K, 7), [K - 1]])
    X = np.zeros((len(ks), K), np.float16)
    X[np.arange(len(ks)), ks] = 1.0
    y, _, _ = run_cuda(X, inp.Qp, inp.S, inp.Zp, g)
    W = oracle.dequant(inp.Qp, inp.S, inp.Zp, K, N, g)
    assert np.array_equal(y.view(np.uint16), W[ks].view(np.uint16))


def test_scale_doubling_bitwise():
    p = Problem("dbl", 24, 2048, 512, 128, True)
    inp = make_inputs(p)
    y1, _, _ = run_cuda(inp.X, inp.Qp, inp.S, inp.Zp, 128)
    S2 = (inp.S.astype(np.float32) * 2).astype(np.float16)
    y2, _, _ = run_cuda(inp.X, inp.Qp, S2, inp.Zp, 128)
    assert np.array_equal((y1.astype(np.float32) * 2).astype(np.float16).view(np.uint16),
                          y2.view(np.uint16))


@pytest.mark.parametrize("M,K,N", [(16, 4096, 4096), (300, 1024, 1024)])
def test_deterministic_across_runs(M, K, N):
    """Split column tiles are summed in a fixed order: repeated calls agree bit for bit."""
    p = Problem("det", M, K, N, 128, False)
    inp = make_inputs(p)
    ys, _, _ = run_cuda(inp.X, inp.Qp, inp.S, None, 128, reps=4)
    for y in ys[1:]:
        assert np.array_equal(y.view(np.uint16), ys[0].view(np.uint16))


def test_workspace_is_left_zeroed():
    p = Problem("ws", 16, 4096, 1024, 128, False)
    inp = make_inputs(p)
    _, _, ws = run_cuda(inp.X, inp.Qp, inp.S, None, 128, reps=2)
    # status word and tile counters are zero again (partials may hold data)
    head = ws.buf[:256 + 4 * 8].cpu().numpy()
    assert not head.any()


def test_m_zero_is_noop():
    import w4a16_mixed_precision_gb300 as w4
    dev = torch.device("cuda", 0)
    inp = make_inputs(Problem("m0", 1, 256, 256, 128, False))
    pw = w4.repack(torch.from_numpy(inp.Qp).to(dev), torch.from_numpy(inp.S).to(dev), None, 128)
    ws = w4.Workspace(1, 256, 256, 128)
    x = torch.empty((0, 256), dtype=torch.float16, device=dev)
    y = w4.gemm(x, pw, ws)
    assert y.shape == (0, 256)


def test_workspace_too_small_is_rejected():
    import w4a16_mixed_precision_gb300 as w4
    from w4a16_mixed_precision_gb300 import _binding as b
    dev = torch.device("cuda", 0)
    inp = make_inputs(Problem("wsz", 64, 1024, 512, 128, False))
    pw = w4.repack(torch.from_numpy(inp.Qp).to(dev), torch.from_numpy(inp.S).to(dev), None, 128)
    ws = w4.Workspace(16, 1024, 512, 128)   # sized for M = 16 only
    x = torch.from_numpy(inp.X).to(dev)
    with pytest.raises(w4.MarlinError) as e:
        w4.gemm(x, pw, ws)
    assert e.value.status == b.ERR_WORKSPACE_TOO_SMALL


def test_non_finite_propagates():
    """fp16 output overflow gives inf; a NaN activation gives NaN in its row."""
    K, N = 256, 128
    q = np.full((K, N), 15, np.uint32)     # q - 8 = 7
    S = np.full((K // 128, N), 60000.0, np.float16)   # 7 * 60000 overflows fp16 -> inf weights
    X = np.ones((2, K), np.float16)
    X[1, 3] = np.nan
    y, _, _ = run_cuda(X, pack_codes(q), S, None, 128)
    assert np.isinf(y[0]).all() and (y[0] > 0).all()
    assert np.isnan(y[1]).all()


@pytest.mark.parametrize("M,K,N,g,asym", [(4, 1024, 512, 128, False), (40, 2048, 384, 128, True)])
def test_host_buffer_entry_point_matches_device_call(M, K, N, g, asym):
    """marlin_gemm_host (copy in, multiply, copy out on one stream) returns the
    same bits as marlin_gemm on device buffers; pinned and pageable host X."""
    import w4a16_mixed_precision_gb300 as w4
    from gpu_util import device
    p = Problem("host", M, K, N, g, asym)
    inp = make_inputs(p)
    y_dev_ref, pw, ws = run_cuda(inp.X, inp.Qp, inp.S, inp.Zp, g)
    dev = device()
    for pin in (True, False):
        xh = torch.from_numpy(inp.X.copy())
        yh = torch.full((M, N), 7.0, dtype=torch.float16)
        if pin:
            xh, yh = xh.pin_memory(), yh.pin_memory()
        xd = torch.empty((M, K), dtype=torch.float16, device=dev)
        yd = torch.empty((M, N), dtype=torch.float16, device=dev)
        w4.gemm_host(xh, xd, pw, ws, yd, yh)
        torch.cuda.synchronize()
        assert w4.device_status(ws) == 0
        assert np.array_equal(yh.numpy().view(np.uint16), y_dev_ref.view(np.uint16))


def test_linear_layer_from_gptq_and_awq_weights():
    """W4A16Linear (repack at construction, one marlin_gemm per forward) on
    GPTQ-order and AWQ-order copies of the same weights, against the oracle;
    leading batch dimensions are flattened into M."""
    from w4a16_mixed_precision_gb300.formats import AWQ_ORDER
    from w4a16_mixed_precision_gb300.layer import W4A16Linear
    p = Problem("layer", 6, 1024, 384, 128, True)
    inp = make_inputs(p)
    ref = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, p.group, p.N)
    dev = torch.device("cuda", 0)
    x = torch.from_numpy(inp.X).to(dev).reshape(2, 3, p.K)
    lin = W4A16Linear(torch.from_numpy(inp.Qp), torch.from_numpy(inp.S), torch.from_numpy(inp.Zp), p.group)
    y = lin(x)
    assert tuple(y.shape) == (2, 3, p.N)
    ok, err, _ = oracle.within_tolerance(y.reshape(p.M, p.N).cpu().numpy(), ref)
    assert ok, f"GPTQ-order layer: max abs err {err}"
    # the same weights in AWQ order (columns packed, interleaved)
    q = oracle.unpack_codes(inp.Qp, p.K, p.N)
    z = oracle.unpack_zeros(inp.Zp, p.G, p.N)

    def awq_pack(codes):
        R, C = codes.shape
        out = np.zeros((R, C // 8), np.uint64)
        for c in range(C // 8):
            for i, col in enumerate(AWQ_ORDER):
                out[:, c] |= codes[:, 8 * c + col].astype(np.uint64) << np.uint64(4 * i)
        return out.astype(np.uint32).view(np.int32)

    lin2 = W4A16Linear.from_awq(awq_pack(np.asarray(q, np.uint32)), torch.from_numpy(inp.S),
                                awq_pack(np.asarray(z, np.uint32)), p.group)
    y2 = lin2(x)
    assert np.array_equal(y2.cpu().numpy().view(np.uint16), y.cpu().numpy().view(np.uint16))
