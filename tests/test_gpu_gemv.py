"""GPU parity of every GEMV launch shape against the oracle's fp64 contraction.

The fused reconstruct + GEMV of the Cloudflare blog "Unweight" (section on the
reconstructive matmul) runs in several launch shapes that the autotuner may pick:
consumer warps per CTA, CTAs per SM, weights per lane (32, 64 or 128), split-K,
and the tensor-pipe GEMV (mma.sync, batch up to 16).
Each is checked on matrices that exercise its corner cases: many verbatim
blocks (more than a CTA stages in shared memory), ragged row counts, a very long
K, and a palette holding exponents of 128 and above (|w| >= 2)."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth
from uwtest import check_rows, dev_bytes, oracle_ref, pick, run_matmul, strategies_for, to_dev_u16, tol_ok, torch

pytestmark = pytest.mark.gpu

VARIANTS = (0, 1, 2, 3, 4, 5, 6, 7, 8)


def _case(N, K, scale, p1, f1, seed):
    w = synth.fill((N, K), seed=seed, scale=scale, p1=p1, f1=f1)
    return w


@pytest.mark.parametrize("N,K,scale,p1,f1", [
    (300, 1024, 0.02, 0.005, 300.0),    # ~27% verbatim blocks
    (257, 2112, 8.0, 0.0, 1.0),         # palette entries >= 128 (exponents around 130)
    (96, 28672, 0.015, 1e-4, 100.0),    # long K: 128 weights per lane for 8-warp CTAs
])
@pytest.mark.parametrize("B", [1, 2, 5, 16, 32, 64])
def test_gemv_variants(N, K, scale, p1, f1, B):
    w = _case(N, K, scale, p1, f1, seed=N * 31 + K)
    x = synth.fill((B, K), seed=N + K + B)
    yref, absum = oracle.matmul(w, x)
    for codec in (uw.CODEC_PALETTE, uw.CODEC_HUFFMAN):
        m = uw.Matrix(uw.encode(w, codec), want_palette_form=True)
        for s in strategies_for(m):
            for v in VARIANTS:
                for split in (0, 2):
                    plan = (s, uw.KERNEL_GEMV, split, v)
                    try:
                        y = run_matmul(m, x, plan)
                    except uw.UwError as e:  # a launch shape that does not fit this matrix
                        assert e.status == uw.ERR_UNSUPPORTED, (plan, e)
                        continue
                    ok, worst = tol_ok(y, yref, absum)
                    assert ok, (codec, plan, worst)


def test_palette_high_exponents_present():
    # the second case above must really put exponents >= 128 in the palette
    w = _case(257, 2112, 8.0, 0.0, 1.0, seed=257 * 31 + 2112)
    _, pal = oracle.palette(w)
    assert max(pal) >= 128 and min(pal) < 128


@pytest.mark.parametrize("B", [1, 3, 8, 9, 16])
@pytest.mark.parametrize("out_dtype", [uw.OUT_F32, uw.OUT_BF16])
def test_mma_gemv_gate_8b(B, out_dtype):
    # the tensor-pipe GEMV at full size, in the launch shapes the autotuner chooses from
    mat = synth.gate_8b()
    w = mat.weights()
    x = mat.activations(B)
    rows = check_rows(mat.N, B, seed=B)
    yref, absum = oracle_ref("gate_8b", w, x, rows)
    m = uw.Matrix(uw.encode(w, uw.CODEC_PALETTE))
    for v in (6, 7):
        y = pick(run_matmul(m, x, (uw.STRAT_DIRECT_PALETTE, uw.KERNEL_GEMV, 0, v), out_dtype), rows)
        ok, worst = tol_ok(y, yref, absum, out_dtype == uw.OUT_BF16)
        assert ok, (v, worst)


@pytest.mark.parametrize("B", [1, 4, 16, 17, 32, 33, 48, 64])
@pytest.mark.parametrize("out_dtype", [uw.OUT_F32, uw.OUT_BF16])
def test_rp_gemv_gate_8b(B, out_dtype):
    # the row-parallel tensor-pipe GEMV (variant 8) at full size, from both weight forms: resident codes (direct
    # palette) and codes transcoded from the Huffman stream into the workspace
    mat = synth.gate_8b()
    w = mat.weights()
    x = mat.activations(B)
    rows = check_rows(mat.N, B, seed=100 + B)
    yref, absum = oracle_ref("gate_8b", w, x, rows)
    m = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN), want_palette_form=True)
    for s in (uw.STRAT_DIRECT_PALETTE, uw.STRAT_PALETTE_TRANSCODE):
        y = pick(run_matmul(m, x, (s, uw.KERNEL_GEMV, 0, 8), out_dtype), rows)
        ok, worst = tol_ok(y, yref, absum, out_dtype == uw.OUT_BF16)
        assert ok, (s, worst)


def test_split_target_zeroed_before_the_dependent_launch_adds():
    # The K-split GEMVs add partial sums into a zeroed fp32 target and start as dependent launches, behind a
    # preprocess kernel for the workspace pipelines.  The target is refilled with garbage before every call: a
    # zeroing that is not ordered before the adds shows up as lost or garbage partial sums.
    t = torch()
    mat = synth.gate_8b()
    w = mat.weights()
    m = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN), want_palette_form=True)
    for B, plans in ((1, [(s, uw.KERNEL_GEMV, 2, 4) for s in (1, 2, 3, 4)]),
                     (16, [(s, uw.KERNEL_GEMV, 2, 6) for s in (1, 2, 3, 4)])):
        x_np = mat.activations(B)
        rows = check_rows(mat.N, B, seed=2)
        yref, absum = oracle_ref("gate_8b", w, x_np, rows)
        x = to_dev_u16(x_np)
        y = t.empty((B, mat.N), dtype=t.float32, device="cuda")
        for p in plans:
            plan = uw.Plan(*p)
            need = m.plan_workspace_size(B, plan)
            ws = dev_bytes(need)
            for _ in range(6):
                y.fill_(3.0e30)
                m.matmul_plan(x, B, y, plan, uw.OUT_F32, ws, need)
                t.cuda.synchronize()
                got = pick(y.cpu().numpy().astype(np.float64), rows)
                ok, worst = tol_ok(got, yref, absum)
                assert ok, (p, worst)
