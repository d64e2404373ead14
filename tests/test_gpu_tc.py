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


@pytest.mark.parametrize("shape", [(1000, 1024), (1024, 256), (300, 4096)])
@pytest.mark.parametrize("B", [40, 300])
@pytest.mark.parametrize("out_dtype", [uw.OUT_F32, uw.OUT_BF16])
def test_tc4_shared_row_blocks_replays_and_dirty_workspace(shape, B, out_dtype):
    # The persistent kernel combines a row block that several CTAs share through three workspace cells tagged
    # with the launch's epoch (no zeroing): 1000 x 1024 has 32 units of 128 rows x 256 weights, one per CTA, so
    # every row block is shared by four CTAs (and the last one is ragged); 1024 x 256 has one unit per row block
    # (nothing shared); 300 x 4096 shares its three blocks unevenly.  The workspace starts as garbage; the same
    # launch runs eagerly twice and then from a CUDA graph three times (a replay keeps its epoch, so the cells
    # must be back to no epoch after every launch), each against the oracle's fp64 contraction.
    t = __import__("uwtest").torch()
    from uwtest import dev_bytes, to_dev_u16
    w = synth.fill(shape, seed=shape[0] + B, scale=0.02, p1=2e-3, f1=300.0)
    m = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN, 256, 12), resident="palette")
    x_np = synth.fill((B, shape[1]), seed=B + 7)
    yref, absum = oracle.matmul(w, x_np)
    plan = uw.Plan(uw.STRAT_DIRECT_PALETTE, uw.KERNEL_TC, 0, 4)
    need = m.plan_workspace_size(B, plan)
    ws = dev_bytes(need)
    ws.fill_(0xA5)
    x = to_dev_u16(x_np)
    y = t.empty((B, shape[0]), dtype=t.float32 if out_dtype == uw.OUT_F32 else t.bfloat16, device="cuda")
    s = t.cuda.Stream()

    def check():
        t.cuda.synchronize()
        ok, worst = tol_ok(y.float().cpu().numpy().astype(np.float64), yref, absum, out_dtype == uw.OUT_BF16)
        assert ok, worst
        m.check()

    for _ in range(2):
        y.fill_(float("nan"))
        m.matmul_plan(x, B, y, plan, out_dtype, ws, need, s)
        check()
    g = t.cuda.CUDAGraph()
    with t.cuda.stream(s):
        with t.cuda.graph(g, stream=s):
            m.matmul_plan(x, B, y, plan, out_dtype, ws, need, s)
    for _ in range(3):
        y.fill_(float("nan"))
        with t.cuda.stream(s):
            g.replay()
        check()
