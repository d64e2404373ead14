"""Pins for the oracle's fp64 matmul Y[b, n] = sum_k W[n, k] X[b, k].

The exact result of the contraction is its plain definition; integer-valued
BF16 operands make every product and partial sum exactly representable in fp64,
so the oracle must equal Python's exact integer arithmetic bit for bit.
"""
import numpy as np

import oracle
import synth


def to_bf16_bits(v):
    f = np.asarray(v, np.float32)
    b = f.view(np.uint32)
    assert ((b & 0xFFFF) == 0).all(), "values must be exact in bf16"
    return (b >> 16).astype(np.uint16)


def test_exact_integer_contraction_non_square():
    rng = np.random.default_rng(3)
    N, K, B = 7, 192, 3
    Wi = rng.integers(-8, 9, size=(N, K)) * (2 ** rng.integers(0, 4, size=(N, K)))
    Xi = rng.integers(-5, 6, size=(B, K))
    y, a = oracle.matmul(to_bf16_bits(Wi), to_bf16_bits(Xi))
    for b in range(B):
        for n in range(N):
            exact = sum(int(Wi[n, k]) * int(Xi[b, k]) for k in range(K))
            mag = sum(abs(int(Wi[n, k]) * int(Xi[b, k])) for k in range(K))
            assert y[b, n] == exact and a[b, n] == mag


def test_row_subset_matches_full():
    m = synth.tiny()
    w, x = m.weights(), m.activations(2)
    y, a = oracle.matmul(w, x)
    rows = np.array([255, 0, 17, 128])
    ys, as_ = oracle.matmul(w, x, rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(as_, a[:, rows])


def test_one_hot_selects_a_column():
    # X = e_j picks column j of W: Y[0, n] = W[n, j] exactly.
    m = synth.tiny()
    w = m.weights()
    for j in (0, 63, 64, 511):
        x = np.zeros((1, 512), np.uint16)
        x[0, j] = 0x3F80  # 1.0
        y, _ = oracle.matmul(w, x)
        assert np.array_equal(y[0], synth.bf16_to_f32(w[:, j]).astype(np.float64))
