"""GPU repack kernel vs the oracle's layout: bit-identical bytes."""
import numpy as np
import pytest

import oracle
from workloads import make_weights

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("K,N,g,asym", [
    (128, 128, 128, False), (256, 384, 128, True), (4096, 4096, 128, False),
    (11008, 4096, 128, False), (2048, 5632, 2048, True), (13824, 5120, 128, True),
])
def test_repack_bit_exact(K, N, g, asym):
    import w4a16_mixed_precision_gb300 as w4
    dev = torch.device("cuda", 0)
    Qp, S, Zp = make_weights(K, N, g, asym, seed=K + N)
    pw = w4.repack(torch.from_numpy(Qp).to(dev), torch.from_numpy(S).to(dev),
                   torch.from_numpy(Zp).to(dev) if asym else None, g)
    buf = pw.buf.cpu().numpy()
    codes = buf[: K * N // 2].view(np.int32)
    assert np.array_equal(codes, oracle.repack(Qp, K, N))
    assert np.array_equal(buf[pw.off_scales: pw.off_scales + S.nbytes].view(np.uint16),
                          oracle.repack_scales(S, N).view(np.uint16))
    if asym:
        assert np.array_equal(buf[pw.off_zeros: pw.off_zeros + Zp.nbytes], oracle.repack_zeros(Zp, N))
    # and the round trip through the oracle's inverse recovers the GPTQ words
    assert np.array_equal(oracle.unrepack(codes, K, N), Qp)
