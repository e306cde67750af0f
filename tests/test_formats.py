"""AWQ-order -> GPTQ-order conversion (host side), checked against encoders
written here from the two packings' definitions, on random and structured
codes."""
import numpy as np

from w4a16_mixed_precision_gb300.formats import AWQ_ORDER, awq_to_gptq
from workloads import pack_codes, pack_zeros


def _awq_pack(codes: np.ndarray) -> np.ndarray:
    """uint codes [R][C] -> AWQ words [R][C/8]: nibble i holds column 8c + AWQ_ORDER[i]."""
    R, C = codes.shape
    out = np.zeros((R, C // 8), np.uint64)
    for c in range(C // 8):
        for i, col in enumerate(AWQ_ORDER):
            out[:, c] |= codes[:, 8 * c + col].astype(np.uint64) << np.uint64(4 * i)
    return out.astype(np.uint32).view(np.int32)


def test_awq_codes_and_zeros_convert_to_gptq_order():
    rng = np.random.default_rng(7)
    K, N, G = 256, 64, 2
    q = rng.integers(0, 16, size=(K, N)).astype(np.uint32)
    z = rng.integers(0, 16, size=(G, N)).astype(np.uint32)
    codes, zeros = awq_to_gptq(_awq_pack(q), _awq_pack(z))
    assert np.array_equal(codes.view(np.uint32), pack_codes(q).view(np.uint32))
    assert np.array_equal(zeros.view(np.uint32), pack_zeros(z).view(np.uint32))


def test_awq_interleave_literal_word():
    # one row of 8 columns holding codes 0..7: AWQ puts column order[i] in
    # nibble i, so the word reads 0x75316420; converted to GPTQ order (rows
    # along nibbles) each column's code sits in nibble 0 of its own word
    word = np.array([[0x75316420]], np.uint32).view(np.int32)
    q = np.zeros((8, 8), np.uint32)
    q[0, :] = np.arange(8)
    codes, _ = awq_to_gptq(np.vstack([word, np.zeros((7, 1), np.int32)]))
    assert np.array_equal(codes.view(np.uint32)[0], np.arange(8, dtype=np.uint32))
    assert np.array_equal(codes.view(np.uint32), pack_codes(q).view(np.uint32))
