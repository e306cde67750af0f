"""Pins of the oracle's 2:4 sparse part against values fixed outside it.

The 2:4 variant ("Marlin" (dingiv.github.io), section "支持 2:4 稀疏加速";
"Marlin / GPTQ-Marlin" (brain.gartu.xyz), section "4. Support de la sparsité
2:4 NVIDIA") computes the same product as the dense method, since every
dropped weight dequantises to exactly zero.  So the sparse oracle is pinned to
the dense oracle (itself pinned in test_oracle_pins.py), to a pure-Python
brute force on a tiny case, and to hand-derived compressed groups.
"""
import os

import numpy as np
import pytest

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sparse_24_groups.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if not line:
            continue
        z, q = int(line[0]), [int(v) for v in line[1:5]]
        rows.append((z, q, None if line[5] == "bad" else tuple(int(v) for v in line[5:9])))
    return rows


def test_golden_groups(oracle_lib):
    rows = _golden_rows()
    # one column per golden row (asymmetric zeros carry each row's z), 128 rows
    # per column: the golden group sits in rows 0..3, the rest are zero codes
    K, N, g = 128, 8 * ((len(rows) + 7) // 8), 128
    z = np.full((1, N), 8, np.uint8)
    q = np.empty((K, N), np.uint8)
    for n in range(N):
        zn = rows[n][0] if n < len(rows) else 8
        z[0, n] = zn
        q[:, n] = zn
        if n < len(rows):
            q[0:4, n] = rows[n][1]
    kc, ki, bad = oracle_lib.sparse_compress(wl.pack_codes(q), wl.pack_zeros(z), K, N, g)
    assert bad == sum(1 for r in rows if r[2] is None)
    for n, (_, _, want) in enumerate(rows):
        if want is None:
            continue
        i0, i1, c0, c1 = want
        assert (ki[0, n] & 3, ki[0, n] >> 2, kc[0, n], kc[1, n]) == (i0, i1, c0, c1), n
        # the other groups of the column are all-zero codes: rows 0, 1 kept
        assert np.all(ki[1:, n] == (0 | 1 << 2))


@pytest.mark.parametrize("asym,group", [(False, 128), (True, 128), (True, 256), (False, 512)])
def test_expand_inverts_compress(oracle_lib, asym, group):
    K, N = 512, 256
    Qp, S, Zp = wl.make_sparse_weights(K, N, group, asym, seed=11 + group)
    kc, ki, bad = oracle_lib.sparse_compress(Qp, Zp, K, N, group)
    assert bad == 0
    np.testing.assert_array_equal(oracle_lib.sparse_expand(kc, ki, Zp, K, N, group), Qp)
    # kept positions are ordered and cover every row whose code differs from z
    i0, i1 = ki & 3, ki >> 2
    assert np.all(i0 < i1)
    q = oracle_lib.unpack_codes(Qp, K, N).reshape(K // 4, 4, N)
    z = oracle_lib.unpack_zeros(Zp, K // group, N) if asym else np.full((K // group, N), 8, np.uint8)
    zr = np.repeat(z, group // 4, axis=0)
    for i in range(4):
        differs = q[:, i, :] != zr
        assert np.all(~differs | (i0 == i) | (i1 == i))


def test_violations_counted(oracle_lib):
    K, N, g = 256, 128, 128
    q = np.full((K, N), 8, np.uint8)
    rng = np.random.default_rng(5)
    cells = rng.choice((K // 4) * N, size=37, replace=False)
    for c in cells:
        j, n = divmod(int(c), N)
        nz = 3 + (c % 2)                      # three or four differing codes
        q[4 * j:4 * j + nz, n] = 1
    _, _, bad = oracle_lib.sparse_compress(wl.pack_codes(q), None, K, N, g)
    assert bad == 37


@pytest.mark.parametrize("asym,group", [(False, 128), (True, 128), (True, 384)])
def test_sparse_product_equals_dense_oracle(oracle_lib, asym, group):
    K, N, M = 768, 256, 5
    Qp, S, Zp = wl.make_sparse_weights(K, N, group, asym, seed=3 + group)
    X = wl.make_activations(M, K, seed=4)
    kc, ki, _ = oracle_lib.sparse_compress(Qp, Zp, K, N, group)
    y_sp = oracle_lib.w4a16_sparse(X, kc, ki, S, Zp, group, N)
    y_de = oracle_lib.w4a16(X, Qp, S, Zp, group, N)
    # same terms in the same (k ascending) order; the dense sum only adds exact zeros
    np.testing.assert_array_equal(y_sp, y_de)
    idx = np.array([0, 7, N + 3, 4 * N + N - 1])
    np.testing.assert_array_equal(oracle_lib.w4a16_sparse(X, kc, ki, S, Zp, group, N, idx=idx),
                                  y_de.ravel()[idx])


def test_brute_force_tiny(oracle_lib):
    # pure-Python loops over the definition: w = fp16((q - z) s), y = sum x w
    K, N, M, g = 128, 8, 2, 128
    Qp, S, Zp = wl.make_sparse_weights(K, N, g, True, seed=99)
    X = wl.make_activations(M, K, seed=98)
    q = [[(int(Qp[k // 8, n]) >> (4 * (k % 8))) & 15 for n in range(N)] for k in range(K)]
    z = [(int(Zp[0, n // 8]) >> (4 * (n % 8))) & 15 for n in range(N)]
    y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                w = float(np.float16((q[k][n] - z[n]) * float(S[0, n])))
                acc += float(X[m, k]) * w
            y[m, n] = acc
    kc, ki, bad = oracle_lib.sparse_compress(Qp, Zp, K, N, g)
    assert bad == 0
    np.testing.assert_allclose(oracle_lib.w4a16_sparse(X, kc, ki, S, Zp, g, N), y, rtol=0, atol=1e-12)


def test_tile_layout_round_trip(oracle_lib):
    K, N = 256, 384
    rng = np.random.default_rng(8)
    kc = rng.integers(0, 16, size=(K // 2, N), dtype=np.uint8)
    ki = rng.integers(0, 16, size=(K // 4, N), dtype=np.uint8)
    Pc, Pm = oracle_lib.sparse_repack(kc, ki, K, N)
    assert Pc.size * 4 == K * N // 4 and Pm.size * 4 == K * N // 8
    kc2, ki2 = oracle_lib.sparse_unrepack(Pc, Pm, K, N)
    np.testing.assert_array_equal(kc2, kc)
    np.testing.assert_array_equal(ki2, ki)
    # every code and index nibble lands in exactly one place: a single set
    # nibble travels to a single set nibble
    one = np.zeros_like(kc); one[37, 200] = 5
    Pc1, _ = oracle_lib.sparse_repack(one, np.zeros_like(ki), K, N)
    nz = np.flatnonzero(Pc1)
    assert nz.size == 1 and bin(int(Pc1[nz[0]]) & 0xFFFFFFFF).count("1") == 2


def test_non_finite_x_at_a_dropped_row(oracle_lib):
    """The 2:4 product skips the dropped terms: a NaN or inf in X at a dropped
    row does not reach Y (the dense sum would give inf * 0 = NaN there); at a
    kept row it propagates as in the dense product."""
    K, N, M, g = 128, 8, 2, 128
    q = np.full((K, N), 8, np.uint8)
    q[1, :] = 9                               # every column keeps rows 0 and 1 of group 0
    S = np.ones((1, N), np.float16)
    Qp = wl.pack_codes(q)
    kc, ki, bad = oracle_lib.sparse_compress(Qp, None, K, N, g)
    assert bad == 0 and np.all(ki[0] == (0 | 1 << 2))
    X = np.ones((M, K), np.float16)
    X[0, 2] = np.inf                          # row 2: dropped
    X[1, 1] = np.nan                          # row 1: kept
    y_sp = oracle_lib.w4a16_sparse(X, kc, ki, S, None, g, N)
    y_de = oracle_lib.w4a16(X, Qp, S, None, g, N)
    assert np.all(y_sp[0] == 1.0) and np.all(np.isnan(y_de[0]))
    assert np.all(np.isnan(y_sp[1])) and np.all(np.isnan(y_de[1]))
