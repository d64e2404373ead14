"""GPU parity of the tcgen05 tensor-core kernels against the oracle's fp64 contraction: variant 0 rebuilds
each 128-row tile into shared memory, variant 4 is the persistent kernel over balanced 128 x 256 units that
rebuilds each 64-weight step into shared memory; both accumulate in fp32 in tensor memory.  Every weight format
they consume (4-bit palette codes, exponent bytes, plain bf16 after full decode), ragged N (not a multiple of the
128-row tile), batch sizes from 1 to 512 (N-padding, two MMAs per K-step above 256), K-splits and both output
dtypes; the full 8B gate_proj on every row up to B = 4 and 1024+ spread rows beyond."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth
from uwtest import check_rows, oracle_ref, pick, run_matmul, tol_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mats():
    w = synth.fill((300, 1024), seed=77, scale=0.02, p1=2e-3, f1=300.0)
    return w, uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN, 256, 12), want_palette_form=True)


@pytest.mark.parametrize("variant", [0, 4])
@pytest.mark.parametrize("B", [1, 3, 16, 17, 100, 256, 300, 512])
@pytest.mark.parametrize("strategy", [uw.STRAT_DIRECT_PALETTE, uw.STRAT_EXP_ONLY, uw.STRAT_FULL_DECODE,
                                      uw.STRAT_PALETTE_TRANSCODE])
def test_tc_all_formats(mats, B, strategy, variant):
    w, m = mats
    x = synth.fill((B, w.shape[1]), seed=B * 13 + strategy)
    yref, absum = oracle.matmul(w, x)
    y = run_matmul(m, x, (strategy, uw.KERNEL_TC, 1, variant))
    ok, worst = tol_ok(y, yref, absum)
    assert ok, worst


@pytest.mark.parametrize("variant", [0, 4])
@pytest.mark.parametrize("split", [2, 3, 16])
@pytest.mark.parametrize("out_dtype", [uw.OUT_F32, uw.OUT_BF16])
def test_tc_splits_and_bf16(mats, split, out_dtype, variant):
    w, m = mats
    B = 24
    x = synth.fill((B, w.shape[1]), seed=split)
    yref, absum = oracle.matmul(w, x)
    y = run_matmul(m, x, (uw.STRAT_DIRECT_PALETTE, uw.KERNEL_TC, split, variant), out_dtype)
    ok, worst = tol_ok(y, yref, absum, out_dtype == uw.OUT_BF16)
    assert ok, worst


def test_tc_exact_integers():
    rng = np.random.default_rng(5)
    N, K, B = 200, 512, 40
    Wi = (rng.integers(-3, 4, size=(N, K)) * 2.0 ** rng.integers(0, 3, size=(N, K))).astype(np.float32)
    Xi = rng.integers(-4, 5, size=(B, K)).astype(np.float32)
    w = (Wi.view(np.uint32) >> 16).astype(np.uint16)
    x = (Xi.view(np.uint32) >> 16).astype(np.uint16)
    exact = Xi.astype(np.float64) @ Wi.astype(np.float64).T
    m = uw.Matrix(uw.encode(w, uw.CODEC_PALETTE))
    for s in (uw.STRAT_DIRECT_PALETTE, uw.STRAT_EXP_ONLY, uw.STRAT_FULL_DECODE):
        for v in (0, 4):
            assert np.array_equal(run_matmul(m, x, (s, uw.KERNEL_TC, 1, v)), exact), (s, v)


@pytest.mark.parametrize("B", [16, 64, 256, 512])
def test_tc_gate_8b(B):
    mat = synth.gate_8b()
    w = mat.weights()
    x = mat.activations(B)
    rows = check_rows(mat.N, B, seed=B)
    yref, absum = oracle_ref("gate_8b", w, x, rows)
    m = uw.Matrix(uw.encode(w, uw.CODEC_PALETTE))
    for v in (0, 4):
        y = pick(run_matmul(m, x, (uw.STRAT_DIRECT_PALETTE, uw.KERNEL_TC, 0, v)), rows)
        ok, worst = tol_ok(y, yref, absum)
        assert ok, (v, worst)
