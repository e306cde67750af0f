"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties the oracle to something it cannot fake: a hand-derived worked
example, IEEE-754 rounding as numpy implements it, closed forms, structural
identities (identity / permutation weights, exact scale doubling), a
pure-Python brute force on tiny inputs, and a float64 BLAS matmul.  A plausible
mistake in the oracle (a dropped term, a wrong sign, index or nibble, a
transposed operand, a double rounding) fails at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import Problem, make_inputs, pack_codes, pack_zeros

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- binary16 conversions ---------------------------------------------------

def test_half_to_double_all_patterns():
    h = np.arange(65536, dtype=np.uint16)
    ours = oracle.widen(h)
    ref = h.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_round_to_half_matches_numpy():
    rng = np.random.default_rng(1)
    # random doubles over the whole fp16 range, exact ties, subnormals, overflow edges
    v = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 6, 200000),
        # exact midpoints between neighbouring halves (ties -> even)
        (np.arange(0, 65535, dtype=np.uint16).view(np.float16).astype(np.float64)[:30000:7]
         + np.arange(1, 65536, dtype=np.uint16).view(np.float16).astype(np.float64)[:30000:7]) / 2,
        [65504.0, 65519.99, 65520.0, 65536.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14,
         -0.0, 0.0, 1e300, -1e300],
    ])
    v = v[np.isfinite(v)]
    ours = oracle.to_half_rne(v).view(np.uint16)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_dequant_rounding_exhaustive():
    """fp16_rne((q - z) * s) for every (q - z) in [-15, 15] and every fp16 s.

    Built as one dequantisation of a 32 x 65536 matrix with one group per row
    (g = 1), explicit zeros: row k has q - z = k - 15 (row 31 repeats 0).
    Reference: numpy's binary64 -> binary16 conversion of the exact product.
    """
    K, N = 32, 65536
    d = np.minimum(np.arange(K) - 15, 15)
    q = np.where(d >= 0, d, 0).astype(np.uint32)[:, None].repeat(N, 1)
    z = np.where(d < 0, -d, 0).astype(np.uint32)[:, None].repeat(N, 1)
    s = np.arange(N, dtype=np.uint16).view(np.float16)[None, :].repeat(K, 0)
    W = oracle.dequant(pack_codes(q), s, pack_zeros(z), K, N, 1)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = (d[:, None].astype(np.float64) * s.astype(np.float64)).astype(np.float16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(W), nan)
    assert np.array_equal(W.view(np.uint16)[~nan], ref.view(np.uint16)[~nan])


# ---- the worked example ---------------------------------------------------------

def _hand_case_inputs():
    K, N = 128, 8
    k = np.arange(K)[:, None]
    n = np.arange(N)[None, :]
    q = (k + 2 * n) % 16
    X = (np.arange(K) / 64.0).astype(np.float16)[None, :]
    S = (2.0 ** -np.arange(N)).astype(np.float16)[None, :]
    return X, pack_codes(q), S


def test_hand_case_literals():
    expected = {}
    with open(os.path.join(GOLDEN, "hand_case.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                n, y = line.split()
                expected[int(n)] = float(y)
    assert sorted(expected) == list(range(8))
    X, Qp, S = _hand_case_inputs()
    y = oracle.w4a16(X, Qp, S, None, 128, 8)
    assert y.shape == (1, 8)
    for n in range(8):
        assert y[0, n] == expected[n], (n, y[0, n], expected[n])
    # the same through the two-step path (dequantise, then multiply)
    W = oracle.dequant(Qp, S, None, 128, 8, 128)
    assert np.array_equal(oracle.gemm(X, W), y)


# ---- structural identities --------------------------------------------------------

@pytest.mark.parametrize("K", [128, 256, 1024])
def test_identity_weights(K):
    """q = 9 on the diagonal, 8 elsewhere, s = 1, z = 8  =>  W = I  =>  Y == X."""
    N = K
    q = np.full((K, N), 8, np.uint32)
    q[np.arange(K), np.arange(N)] = 9
    S = np.ones((K // 128, N), np.float16)
    X = make_inputs(Problem("id", 5, K, N, 128, False)).X
    y = oracle.w4a16(X, pack_codes(q), S, None, 128, N)
    assert np.array_equal(y, X.astype(np.float64))


def test_permutation_weights_with_explicit_zeros():
    """W = permutation matrix (q - z = 1 at (k, pi(k)), 0 elsewhere, s = 1)
    => Y[:, pi(k)] == X[:, k].  Zeros vary per (group, column)."""
    K = N = 256
    rng = np.random.default_rng(7)
    pi = rng.permutation(N)
    z = rng.integers(0, 15, size=(K // 128, N)).astype(np.uint32)   # 0..14 so z+1 fits in 4 bits
    zfull = np.repeat(z, 128, axis=0)
    q = zfull.copy()
    q[np.arange(K), pi] += 1
    S = np.ones((K // 128, N), np.float16)
    X = make_inputs(Problem("perm", 3, K, N, 128, True)).X
    y = oracle.w4a16(X, pack_codes(q), S, pack_zeros(z), 128, N)
    expect = np.empty_like(y)
    expect[:, pi] = X.astype(np.float64)
    assert np.array_equal(y, expect)


def test_scale_doubling_is_exact():
    p = Problem("dbl", 4, 512, 256, 128, True)
    inp = make_inputs(p)
    y1 = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, p.group, p.N)
    S2 = (inp.S.astype(np.float64) * 2).astype(np.float16)
    assert np.array_equal(S2.astype(np.float64), 2 * inp.S.astype(np.float64))
    y2 = oracle.w4a16(inp.X, inp.Qp, S2, inp.Zp, p.group, p.N)
    assert np.array_equal(y2, 2 * y1)


def test_constant_code_closed_form():
    """q = c everywhere, per-(group, column) zeros z and power-of-two scales s:
    y[m][n] = sum_j (c - z[j][n]) * s[j][n] * sum_{k in group j} x[m][k], exactly."""
    M, K, N, g, c = 3, 512, 16, 128, 11
    G = K // g
    rng = np.random.default_rng(3)
    z = rng.integers(0, 16, size=(G, N)).astype(np.uint32)
    e = rng.integers(0, 7, size=(G, N))
    S = (2.0 ** -e).astype(np.float16)
    X = make_inputs(Problem("cc", M, K, N, g, True)).X
    q = np.full((K, N), c, np.uint32)
    y = oracle.w4a16(X, pack_codes(q), S, pack_zeros(z), g, N)
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for j in range(G):
                xs = sum(Fraction(float(v)) for v in X[m, j * g:(j + 1) * g])
                tot += (c - int(z[j, n])) * Fraction(float(S[j, n])) * xs
            assert Fraction(y[m, n]) == tot, (m, n)


def test_bruteforce_python_tiny():
    """A pure-Python restatement of the definition (numpy only for the one
    fp16 rounding) on tiny inputs with several groups and explicit zeros.
    Same k order, so the binary64 sums agree bit for bit."""
    M, K, N, g = 2, 32, 16, 8
    p = Problem("bf", M, K, N, g, True)
    inp = make_inputs(p)
    y = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, g, N)
    Qp = inp.Qp.view(np.uint32)
    Zp = inp.Zp.view(np.uint32)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                qv = (int(Qp[k // 8, n]) >> (4 * (k % 8))) & 15
                zv = (int(Zp[k // g, n // 8]) >> (4 * (n % 8))) & 15
                w = float(np.float16((qv - zv) * float(inp.S[k // g, n])))
                acc += float(inp.X[m, k]) * w
            assert y[m, n] == acc, (m, n)


def test_gemm_matches_float64_blas():
    p = Problem("blas", 7, 1024, 384, 128, False)
    inp = make_inputs(p)
    W = oracle.dequant(inp.Qp, inp.S, None, p.K, p.N, p.group)
    ref = inp.X.astype(np.float64) @ W.astype(np.float64)
    import torch
    ref_t = (torch.from_numpy(inp.X.astype(np.float64)) @ torch.from_numpy(W.astype(np.float64))).numpy()
    y = oracle.gemm(inp.X, W)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y, ref_t, rtol=1e-12, atol=1e-12)
    # the fused path computes the same sums in the same order
    assert np.array_equal(oracle.w4a16(inp.X, inp.Qp, inp.S, None, p.group, p.N), y)


def test_sampled_entries_match_full():
    p = Problem("samp", 9, 768, 512, 128, True)
    inp = make_inputs(p)
    full = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, p.group, p.N)
    rng = np.random.default_rng(0)
    idx = rng.integers(0, p.M * p.N, 300)
    part = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, p.group, p.N, idx=idx)
    assert np.array_equal(part, full.ravel()[idx])


def test_per_column_group_equals_single_group():
    """g = K (one scale per column) is the one-group case of the definition."""
    p = Problem("pc", 2, 384, 128, 384, True)
    inp = make_inputs(p)
    assert inp.S.shape == (1, 128)
    y = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, p.K, p.N)
    # the same weights expressed with g = 128 and the scale row repeated per group
    S3 = np.repeat(inp.S, 3, axis=0)
    Z3 = np.repeat(inp.Zp, 3, axis=0)
    assert np.array_equal(oracle.w4a16(inp.X, inp.Qp, S3, Z3, 128, p.N), y)


def test_symmetric_is_zero_eight():
    p = Problem("sym", 2, 256, 128, 128, False)
    inp = make_inputs(p)
    z8 = pack_zeros(np.full((2, 128), 8, np.uint32))
    assert np.array_equal(oracle.w4a16(inp.X, inp.Qp, inp.S, None, 128, 128),
                          oracle.w4a16(inp.X, inp.Qp, inp.S, z8, 128, 128))


def test_unpack_nibble_order():
    """GPTQ order: nibble i of word [r][n] is row 8r + i; zeros: nibble j of
    word [g][c] is column 8c + j."""
    Qp = np.array([[0x76543210, 0x0FEDCBA9]], np.uint32).view(np.int32)
    q = oracle.unpack_codes(Qp, 8, 2)
    assert q[:, 0].tolist() == [0, 1, 2, 3, 4, 5, 6, 7]
    assert q[:, 1].tolist() == [9, 10, 11, 12, 13, 14, 15, 0]
    Zp = np.array([[0x13579BDF]], np.uint32).view(np.int32)
    assert oracle.unpack_zeros(Zp, 1, 8)[0].tolist() == [15, 13, 11, 9, 7, 5, 3, 1]


# ---- repacked layout ------------------------------------------------------------

def test_repack_layout_literals():
    """Word (nt, kb, g, l, j) of the tile layout holds, at nibble p, the code of
    row 16g + l/4 + 8(p&1) and k = 16j + 4(l%4) + 2((p>>1)&1) + (p>>2) of the
    (nt, kb) tile.  Checked against words worked out by hand."""
    K, N = 128, 256
    P = lambda q: oracle.repack(pack_codes(q), K, N).view(np.uint32).reshape(N // 128, K // 64, 8, 32, 4)
    # q = k mod 16: only l % 4 matters -> nibbles (p7..p0) = 4c + (3,3,1,1,2,2,0,0)
    Pk = P((np.arange(K) % 16)[:, None].repeat(N, 1))
    assert Pk[0, 0, 0, 0, 0] == 0x33112200
    assert Pk[1, 1, 5, 1, 3] == 0x77556644
    assert Pk[0, 1, 7, 30, 2] == 0xBB99AA88
    assert Pk[1, 0, 3, 7, 1] == 0xFFDDEECC
    # q = n mod 16: only l / 4 matters -> even nibbles r = l/4, odd nibbles r + 8
    Pn = P((np.arange(N) % 16)[None, :].repeat(K, 0))
    assert Pn[0, 0, 2, 5, 0] == 0x91919191
    assert Pn[1, 1, 6, 30, 3] == 0xF7F7F7F7


def test_repack_scales_and_zeros_tile_major():
    G, N = 3, 256
    S = (np.arange(G * N, dtype=np.float64).reshape(G, N) / 64).astype(np.float16)
    Sr = oracle.repack_scales(S, N).reshape(N // 128, G, 128)
    assert Sr[1, 2, 5] == S[2, 128 + 5] and Sr[0, 1, 127] == S[1, 127]
    z = (np.arange(G * N).reshape(G, N) * 7) % 16
    Zr = oracle.repack_zeros(pack_zeros(z), N).reshape(N // 128, G, 64)
    # byte b of tile row (nt, gi) holds columns 2b (low nibble) and 2b + 1 (high nibble)
    assert Zr[1, 2, 3] == (z[2, 128 + 6] | (z[2, 128 + 7] << 4))
    assert Zr[0, 0, 63] == (z[0, 126] | (z[0, 127] << 4))


@pytest.mark.parametrize("K,N", [(128, 128), (256, 384), (4096, 4096), (11008, 256)])
def test_repack_roundtrip(K, N):
    rng = np.random.default_rng(K * 7 + N)
    Qp = rng.integers(0, 2**32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32).view(np.int32)
    P = oracle.repack(Qp, K, N)
    assert P.size * 4 == K * N // 2
    assert np.array_equal(oracle.unrepack(P, K, N), Qp)
    # a permutation of codes: the multiset of nibbles is preserved
    def hist(a):
        a = a.view(np.uint32).ravel()
        return np.bincount(np.concatenate([(a >> (4 * i)) & 15 for i in range(8)]).astype(np.int64), minlength=16)
    assert np.array_equal(hist(P), hist(Qp))


def test_tolerance_helper():
    ok, err, r = oracle.within_tolerance(np.array([1.0, 100.0]), np.array([1.0 + 0.0119, 100.2]))
    assert ok and r <= 1.0
    ok, _, _ = oracle.within_tolerance(np.array([0.0]), np.array([0.0101]))
    assert not ok
    ok, _, _ = oracle.within_tolerance(np.array([np.nan]), np.array([0.0]))
    assert not ok
