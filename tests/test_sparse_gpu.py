"""GPU parity of the 2:4-sparse path (marlin_sparse_repack + marlin_sparse_gemm,
through the C ABI) against the CPU oracle.

The sparse product equals the dense one ("Marlin", section "支持 2:4 稀疏加速";
"Marlin / GPTQ-Marlin", section "4. Support de la sparsité 2:4 NVIDIA"): the
dropped weights dequantise to exactly zero.  Tolerance as for the dense path:
|y_gpu - y_ref| <= 1e-2 + 2e-3*|y_ref| per element; the repack is bit-exact
against the oracle's layout; identity weights give Y == X bit for bit.
"""
import numpy as np
import pytest

import oracle
from workloads import SPARSE_7B_DECODE, make_activations, make_sparse_weights, pack_codes

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0") if a is not None else None


def run_sparse(X, Qp, S, Zp, g, reps=1, strict=True):
    import w4a16_mixed_precision_gb300 as w4
    K, N = Qp.shape[0] * 8, Qp.shape[1]
    pw = w4.sparse_repack(_dev(Qp), _dev(S), _dev(Zp), g, strict=strict)
    ws = w4.Workspace(X.shape[0], K, N, g)
    x = _dev(X)
    ys = [w4.sparse_gemm(x, pw, ws) for _ in range(reps)]
    torch.cuda.synchronize()
    assert w4.device_status(ws) == 0, "kernel reported an expired wait"
    out = [y.cpu().numpy() for y in ys]
    return (out[0] if reps == 1 else out), pw, ws


CASES = [
    # M, K, N, group, asym
    (1, 128, 128, 128, False),          # one unit, one tile
    (1, 4096, 384, 128, False),
    (5, 256, 384, 128, True),
    (8, 1024, 512, 128, False),
    (13, 2048, 640, 256, True),         # group 256
    (16, 1024, 512, 1024, True),        # one scale per column
    (24, 2048, 1024, 128, False),
    (32, 2048, 768, 128, True),         # four token blocks
    (17, 4096, 4096, 128, False),       # many units, tiles split across CTAs
    (9, 4096, 9728, 128, True),         # 256-row units (two chunks per consumer warp)
    (3, 11008, 512, 128, False),        # long K, few tiles
    # batches above 32 tokens: m-tiles of 32 on the same sparse kernel
    (33, 1024, 512, 128, False),        # a one-token second m-tile
    (64, 2048, 768, 128, True),
    (128, 1024, 640, 256, False),
    (256, 512, 384, 128, True),
    (600, 1024, 256, 1024, False),      # one scale per column, 19 m-tiles, ragged last
]


@pytest.mark.parametrize("M,K,N,g,asym", CASES)
def test_sparse_parity(M, K, N, g, asym):
    Qp, S, Zp = make_sparse_weights(K, N, g, asym, seed=M * 1000 + K + N)
    X = make_activations(M, K, seed=M + K)
    y, pw, _ = run_sparse(X, Qp, S, Zp, g)
    assert pw.bad_groups == 0
    kc, ki, bad = oracle.sparse_compress(Qp, Zp, K, N, g)
    assert bad == 0
    y_ref = oracle.w4a16_sparse(X, kc, ki, S, Zp, g, N)
    ok, err, ratio = oracle.within_tolerance(y, y_ref)
    assert ok, f"max abs err {err}, worst ratio {ratio}"


@pytest.mark.parametrize("asym,g", [(False, 128), (True, 128), (True, 512)])
def test_sparse_repack_bit_exact(asym, g):
    import w4a16_mixed_precision_gb300 as w4
    K, N = 1024, 640
    Qp, S, Zp = make_sparse_weights(K, N, g, asym, seed=21)
    pw = w4.sparse_repack(_dev(Qp), _dev(S), _dev(Zp), g)
    buf = pw.buf.cpu().numpy()
    kc, ki, _ = oracle.sparse_compress(Qp, Zp, K, N, g)
    Pc, Pm = oracle.sparse_repack(kc, ki, K, N)
    assert np.array_equal(buf[:Pc.nbytes].view(np.int32), Pc)
    assert np.array_equal(buf[pw.off_meta:pw.off_meta + Pm.nbytes].view(np.int32), Pm)
    sc = oracle.repack_scales(S, N)
    assert np.array_equal(buf[pw.off_scales:pw.off_scales + sc.nbytes].view(np.float16).view(np.uint16),
                          sc.view(np.uint16))
    if asym:
        zr = oracle.repack_zeros(Zp, N)
        assert np.array_equal(buf[pw.off_zeros:pw.off_zeros + zr.nbytes], zr)


def test_not_2of4_is_counted_and_rejected():
    import w4a16_mixed_precision_gb300 as w4
    K, N, g = 512, 256, 128
    q = np.full((K, N), 8, np.uint32)
    rng = np.random.default_rng(4)
    cells = rng.choice((K // 4) * N, size=29, replace=False)
    for c in cells:
        j, n = divmod(int(c), N)
        q[4 * j:4 * j + 3, n] = [1, 2, 3]            # three non-zero weights in one group
    Qp = pack_codes(q)
    S = np.ones((K // g, N), np.float16)
    with pytest.raises(ValueError):
        w4.sparse_repack(_dev(Qp), _dev(S), None, g)
    pw = w4.sparse_repack(_dev(Qp), _dev(S), None, g, strict=False)
    assert pw.bad_groups == oracle.sparse_compress(Qp, None, K, N, g)[2] == 29


@pytest.mark.parametrize("K", [256, 1024])
def test_sparse_identity_exact(K):
    """W = I is 2:4 (one non-zero per column): Y == X bit for bit."""
    N = K
    q = np.full((K, N), 8, np.uint32)
    q[np.arange(K), np.arange(N)] = 9
    S = np.ones((K // 128, N), np.float16)
    X = make_activations(19, K, seed=5)
    y, _, _ = run_sparse(X, pack_codes(q), S, None, 128)
    assert np.array_equal(y.view(np.uint16), X.view(np.uint16))


def test_sparse_onehot_rows_give_exact_dequant():
    """X = one-hot rows: row m of Y is row k_m of dequant(W), exactly (one
    product per output, no rounding in the fp32 sum)."""
    K, N, g = 512, 384, 128
    Qp, S, Zp = make_sparse_weights(K, N, g, True, seed=6)
    ks = np.array([0, 1, 2, 3, 130, 255, 256, 511])
    X = np.zeros((len(ks), K), np.float16)
    X[np.arange(len(ks)), ks] = 1.0
    y, _, _ = run_sparse(X, Qp, S, Zp, g)
    W = oracle.dequant(Qp, S, Zp, K, N, g)
    assert np.array_equal(y.view(np.uint16), W[ks].view(np.uint16))


def test_sparse_matches_dense_path_on_same_weights():
    from gpu_util import run_cuda
    K, N, g, M = 2048, 1024, 128, 12
    Qp, S, Zp = make_sparse_weights(K, N, g, True, seed=31)
    X = make_activations(M, K, seed=32)
    y_sp, _, _ = run_sparse(X, Qp, S, Zp, g)
    y_de, _, _ = run_cuda(X, Qp, S, Zp, g)
    y_ref = oracle.w4a16(X, Qp, S, Zp, g, N)
    for y in (y_sp, y_de):
        ok, err, ratio = oracle.within_tolerance(y, y_ref)
        assert ok, f"max abs err {err}, worst ratio {ratio}"


def test_sparse_deterministic_and_workspace_left_zeroed():
    K, N, g, M = 4096, 4096, 128, 16
    Qp, S, Zp = make_sparse_weights(K, N, g, False, seed=41)
    X = make_activations(M, K, seed=42)
    ys, _, ws = run_sparse(X, Qp, S, Zp, g, reps=3)
    for y in ys[1:]:
        assert np.array_equal(y.view(np.uint16), ys[0].view(np.uint16))
    assert int(ws.buf.count_nonzero().item()) == 0


def test_sparse_empty_m_and_workspace_for_large_m():
    import w4a16_mixed_precision_gb300 as w4
    K, N, g = 256, 256, 128
    Qp, S, Zp = make_sparse_weights(K, N, g, False, seed=1)
    pw = w4.sparse_repack(_dev(Qp), _dev(S), None, g)
    ws = w4.Workspace(40, K, N, g)
    y = torch.full((0, N), 7.0, dtype=torch.float16, device="cuda:0")
    w4.sparse_gemm_into(torch.zeros((0, K), dtype=torch.float16, device="cuda:0"), pw, ws, y)
    torch.cuda.synchronize()
    # a workspace sized for 40 tokens serves 40 (two m-tiles) and every smaller M
    for M in (40, 33, 1):
        y = w4.sparse_gemm(torch.ones((M, K), dtype=torch.float16, device="cuda:0"), pw, ws)
        torch.cuda.synchronize()
        assert w4.device_status(ws) == 0 and bool(torch.isfinite(y).all())
    # one that is too small is rejected before anything is launched
    tiny = w4.Workspace(1, K, N, g)
    tiny.nbytes = 256
    with pytest.raises(w4.MarlinError) as e:
        w4.sparse_gemm(torch.zeros((40, K), dtype=torch.float16, device="cuda:0"), pw, tiny)
    assert e.value.status == 4  # MARLIN_ERR_WORKSPACE_TOO_SMALL


def test_sparse_large_m_onehot_exact():
    """M = 48 (two m-tiles): one-hot X rows give the dequantised weights bit
    for bit (kept terms only; each output is one exact product)."""
    K, N, g, M = 1024, 384, 128, 48
    Qp, S, Zp = make_sparse_weights(K, N, g, True, seed=61)
    rng = np.random.default_rng(62)
    k_m = rng.integers(0, K, M)
    X = np.zeros((M, K), np.float16)
    X[np.arange(M), k_m] = 1.0
    y, _, _ = run_sparse(X, Qp, S, Zp, g)
    kc, ki, _ = oracle.sparse_compress(Qp, Zp, K, N, g)
    y_ref = oracle.w4a16_sparse(X, kc, ki, S, Zp, g, N)
    assert np.array_equal(y.view(np.uint16), y_ref.astype(np.float16).view(np.uint16))


def _sample(M, N, seed, count=384):
    rng = np.random.default_rng(seed)
    cols = np.unique(np.concatenate([[0, N - 1, 127, 128], rng.integers(0, N, 24)]))
    grid = (np.arange(M)[:, None] * N + cols[None, :]).ravel()
    return np.unique(np.concatenate([grid, rng.integers(0, M * N, count)]))


_layers = {}


def _layer(K, N, g, asym):
    """Seeded 2:4 weights of one layer shape, repacked once, with the oracle's compressed form."""
    import w4a16_mixed_precision_gb300 as w4
    key = (K, N, g, asym)
    if key not in _layers:
        _layers.clear()   # one layer resident at a time
        Qp, S, Zp = make_sparse_weights(K, N, g, asym, seed=K * 7 + N)
        kc, ki, bad = oracle.sparse_compress(Qp, Zp, K, N, g)
        assert bad == 0
        _layers[key] = (w4.sparse_repack(_dev(Qp), _dev(S), _dev(Zp), g), kc, ki, S, Zp)
    return _layers[key]


@pytest.mark.parametrize("p", SPARSE_7B_DECODE, ids=[p.key for p in SPARSE_7B_DECODE])
def test_sparse_full_size_sampled(p):
    """Every workload of the sparse benchmark at full size (same launch
    configuration), checked on sampled entries the oracle computes one by one."""
    import w4a16_mixed_precision_gb300 as w4
    pw, kc, ki, S, Zp = _layer(p.K, p.N, p.group, p.asym)
    X = make_activations(p.M, p.K, seed=p.M * 3 + p.K)
    ws = w4.Workspace(p.M, p.K, p.N, p.group)
    y = w4.sparse_gemm(_dev(X), pw, ws).cpu().numpy()
    assert w4.device_status(ws) == 0
    assert y.shape == (p.M, p.N) and np.isfinite(y).all()
    idx = _sample(p.M, p.N, seed=p.M * 7 + p.K)
    y_ref = oracle.w4a16_sparse(X, kc, ki, S, Zp, p.group, p.N, idx=idx)
    ok, err, ratio = oracle.within_tolerance(y.ravel()[idx], y_ref)
    assert ok, f"{p.key}: max abs err {err}, worst ratio {ratio}"


def test_sparse_linear_layer():
    """The layer with sparse=True serves small batches on the 2:4 path and larger
    ones on the dense kernel; its output and the dense layer's are both within
    tolerance of the oracle on either side of the switch."""
    from w4a16_mixed_precision_gb300.layer import W4A16Linear
    K, N, g = 1024, 640, 128
    Qp, S, Zp = make_sparse_weights(K, N, g, True, seed=51)
    lay_sp = W4A16Linear(torch.from_numpy(Qp), torch.from_numpy(S), torch.from_numpy(Zp), g, sparse=True)
    lay_de = W4A16Linear(torch.from_numpy(Qp), torch.from_numpy(S), torch.from_numpy(Zp), g)
    for M in (4, 16, 17, 32, 40):
        X = make_activations(M, K, seed=M)
        x = _dev(X)
        y_sp = lay_sp(x.reshape(1, M, K)).reshape(M, N).cpu().numpy()
        y_de = lay_de(x).cpu().numpy()
        y_ref = oracle.w4a16(X, Qp, S, Zp, g, N)
        for y in (y_sp, y_de):
            ok, err, ratio = oracle.within_tolerance(y, y_ref)
            assert ok, f"M={M}: max abs err {err}, worst ratio {ratio}"
    Qd, Sd, _ = make_sparse_weights(K, N, g, False, seed=52)
    Qd = Qd.copy()
    Qd[0, :] = 0x12345678                     # rows 0..7: more than two non-zero codes per group
    with pytest.raises(ValueError):
        W4A16Linear(torch.from_numpy(Qd), torch.from_numpy(Sd), None, g, sparse=True)
