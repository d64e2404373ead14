"""Non-finite activations: every strategy and kernel family gives the class (NaN, +inf, -inf, finite) that the
oracle's fp64 contraction gives for each output, and finite outputs stay within the tolerance.

The product is Y = X . W^T (Cloudflare blog "Unweight", section on the reconstructive matmul).  With an infinite
activation x_k, a row's exact result is +-inf when every non-finite term w_k x_k has one sign, and NaN when signs
mix or an activation is NaN; IEEE arithmetic reaches that class in any summation order.  The kernels must
therefore never multiply an infinite activation by a stand-in zero weight (0 * inf = NaN): the activations are
placed on positions of verbatim blocks, which some kernels handle outside their main loop."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth
from uwtest import run_matmul, strategies_for

pytestmark = pytest.mark.gpu

POS_INF, NEG_INF, NAN = 0x7F80, 0xFF80, 0x7FC0


def _classes(y):
    return np.where(np.isnan(y), 3, np.where(np.isposinf(y), 1, np.where(np.isneginf(y), 2, 0)))


def _nonfinite_case():
    # 512 x 2048 with about a fifth of the blocks verbatim; X rows: +inf at one verbatim-heavy position,
    # -inf at two, a NaN, and a finite control row
    N, K, B = 512, 2048, 4
    w = synth.fill((N, K), seed=4242, scale=0.02, p1=0.02, f1=300.0)
    x = synth.fill((B, K), seed=4243)
    _, pal = oracle.palette(w)  # the blocks holding an exponent outside the palette are the verbatim ones
    exps = (w >> 7) & 0xFF
    in_pal = np.isin(exps, np.array(pal, dtype=exps.dtype))
    block_verb = ~in_pal.reshape(N, K // 64, 64).all(axis=2)          # [N, K/64]
    cols = np.argsort(-block_verb.sum(axis=0))                        # blocks that are verbatim in most rows
    k_a, k_b, k_c = 64 * cols[0] + 5, 64 * cols[1] + 17, 64 * cols[2] + 40
    x[0, k_a] = POS_INF
    x[1, k_a] = NEG_INF
    x[1, k_b] = NEG_INF
    x[2, k_c] = NAN
    assert block_verb[:, cols[0]].mean() > 0.2 and block_verb[:, cols[2]].mean() > 0.2
    return w, x


def _check(y, yref, absum, what):
    cg, cr = _classes(y), _classes(yref)
    assert np.array_equal(cg, cr), (what, int((cg != cr).sum()))
    fin = cr == 0
    err = np.abs(y[fin] - yref[fin])
    assert (err <= 1e-4 * absum[fin] + 1e-6).all(), what


def test_nonfinite_activations_every_kernel():
    w, x = _nonfinite_case()
    with np.errstate(invalid="ignore"):
        yref, absum = oracle.matmul(w, x)
    assert (_classes(yref) == 1).any() and (_classes(yref) == 2).any() and (_classes(yref) == 3).any()
    for codec in (uw.CODEC_PALETTE, uw.CODEC_HUFFMAN):
        m = uw.Matrix(uw.encode(w, codec), want_palette_form=True)
        plans = list(strategies_for(m))
        for s in strategies_for(m):
            plans += [(s, uw.KERNEL_GEMV, sp, v) for v in (0, 1, 2, 4, 5, 6, 7, 8) for sp in (0, 2)]
            plans += [(s, uw.KERNEL_TC, 0, v) for v in (0, 4)]
        if codec == uw.CODEC_HUFFMAN:
            plans += [uw.STRAT_HUFFMAN_DIRECT, (uw.STRAT_HUFFMAN_DIRECT, uw.KERNEL_GEMV, 0, 1)]
        for p in plans:
            try:
                y = run_matmul(m, x, p)
            except uw.UwError as e:  # a launch shape that does not fit this matrix
                assert e.status == uw.ERR_UNSUPPORTED, (p, e)
                continue
            _check(y, yref, absum, (codec, p))
        m.check()
