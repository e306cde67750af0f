"""Full-size parity on every benchmark workload (all five configurations).

The CUDA path runs at full size in the same launch configuration the
benchmark times; the oracle computes a sample of entries one by one (every
m-tile boundary row, first/last columns of column tiles, and random entries)
and every sampled entry must meet the tolerance."""
import numpy as np
import pytest

import oracle
from workloads import ALL_CONFIGS, make_inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def sample_indices(M, N, seed, count=384):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, M - 1], np.arange(0, M, 256), np.arange(255, M, 256),
                                     rng.integers(0, M, 8)]))
    rows = rows[rows < M]
    cols = np.unique(np.concatenate([[0, N - 1, 127, 128], rng.integers(0, N, 24)]))
    grid = (rows[:, None] * N + cols[None, :]).ravel()
    rand = rng.integers(0, M * N, count)
    return np.unique(np.concatenate([grid, rand]))


CASES = [p for cfg in ALL_CONFIGS.values() for p in cfg]


@pytest.mark.parametrize("p", CASES, ids=[p.key for p in CASES])
def test_full_size_sampled(p):
    from gpu_util import run_cuda
    inp = make_inputs(p)
    y, _, _ = run_cuda(inp.X, inp.Qp, inp.S, inp.Zp, p.group)
    assert y.shape == (p.M, p.N)
    assert np.isfinite(y).all()
    idx = sample_indices(p.M, p.N, seed=p.M * 7 + p.K)
    y_ref = oracle.w4a16(inp.X, inp.Qp, inp.S, inp.Zp, p.group, p.N, idx=idx)
    ok, err, ratio = oracle.within_tolerance(y.ravel()[idx], y_ref)
    assert ok, f"{p.key}: max abs err {err}, worst ratio {ratio}"
