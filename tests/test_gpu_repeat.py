"""Repeated full-size parity of every strategy on every GEMV launch shape.

The ring-buffered GEMVs hand a shared-memory slot back to their copy engine as
soon as a warp has read it.  A missing cross-proxy fence there once let the next
bulk copy overwrite a slot before a warp's loads had read it: a few wrong rows in
a few percent of calls, visible only when every row is compared and the call is
repeated.  So each (strategy, launch shape) runs ten times on the 8B gate_proj
W[14336, 4096] (Cloudflare blog "Unweight": the four execution pipelines, the
reconstructive matmul), with the output refilled with 3e30 before each call and
every row compared with the oracle's fp64 contraction (B = 1; at B = 16, 1024+
rows spread over every CTA's range)."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import synth
from uwtest import check_rows, dev_bytes, oracle_ref, pick, to_dev_u16, tol_ok, torch

pytestmark = pytest.mark.gpu

RUNS = 10


@pytest.fixture(scope="module")
def gate():
    mat = synth.gate_8b()
    w = mat.weights()
    return mat, w, uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN), want_palette_form=True)


@pytest.mark.parametrize("B", [1, 16])
@pytest.mark.parametrize("strategy", [uw.STRAT_FULL_DECODE, uw.STRAT_EXP_ONLY, uw.STRAT_PALETTE_TRANSCODE,
                                      uw.STRAT_DIRECT_PALETTE])
def test_every_gemv_shape_all_rows_repeated(gate, strategy, B):
    t = torch()
    mat, w, m = gate
    x_np = mat.activations(B)
    rows = check_rows(mat.N, B, seed=B)
    yref, absum = oracle_ref("gate_8b", w, x_np, rows)
    x = to_dev_u16(x_np)
    y = t.empty((B, mat.N), dtype=t.float32, device="cuda")
    for variant in (0, 2, 3, 4, 5, 6, 7, 8):
        for split in (0, 2):
            plan = uw.Plan(strategy, uw.KERNEL_GEMV, split, variant)
            need = m.plan_workspace_size(B, plan)
            ws = dev_bytes(need)
            for run in range(RUNS):
                y.fill_(3.0e30)
                m.matmul_plan(x, B, y, plan, uw.OUT_F32, ws, need)
                t.cuda.synchronize()
                ok, worst = tol_ok(pick(y.cpu().numpy().astype(np.float64), rows), yref, absum)
                assert ok, (plan.as_tuple(), run, worst)
    m.check()

