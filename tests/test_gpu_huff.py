"""GPU parity of the Huffman-direct GEMV (the GEMV that decodes the Huffman stream itself) against the
oracle's fp64 contraction: chunk sizes and code-length limits, ragged row counts, verbatim-heavy and
single-symbol matrices, exact integer cases, fp32 and bf16 outputs, full-size 8B and 70B shapes on every row,
corrupt streams, and the cases the strategy does not take.  Cloudflare blog "Unweight": the section on the
execution pipelines (the Huffman-fed pipelines) and the section on the decode kernels (lookup table in shared
memory)."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth
from uwtest import check_rows, dev_bytes, oracle_ref, pick, run_matmul, tol_ok, to_dev_u16, torch

pytestmark = pytest.mark.gpu

HD = uw.STRAT_HUFFMAN_DIRECT


def _huffman_only(w, chunk=256, L=12):
    return uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN, chunk, L))


def _check(m, w, B, seed, out_dtype=uw.OUT_F32, variants=(0, 1)):
    # variant 0: plain loads; 1: with an L2 prefetch of each unit one unit ahead (both through an explicit plan),
    # and the strategy's default through uw_matmul
    x = synth.fill((B, w.shape[1]), seed=seed)
    yref, absum = oracle.matmul(w, x)
    for p in [HD] + [(HD, uw.KERNEL_GEMV, 0, v) for v in variants]:
        y = run_matmul(m, x, p, out_dtype)
        ok, worst = tol_ok(y, yref, absum, out_dtype == uw.OUT_BF16)
        assert ok, (p, worst)


@pytest.mark.parametrize("chunk,L", [(256, 12), (64, 12), (128, 5), (512, 9)])
@pytest.mark.parametrize("B", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("out_dtype", [uw.OUT_F32, uw.OUT_BF16])
def test_tiny_chunks_and_limits(chunk, L, B, out_dtype):
    w = synth.tiny().weights()
    m = _huffman_only(w, chunk, L)
    _check(m, w, B, seed=100 + B + chunk, out_dtype=out_dtype)


@pytest.mark.parametrize("N,K,chunk", [(1, 64, 64), (17, 192, 64), (33, 576, 192), (31, 4160, 64), (300, 1024, 256),
                                       (65, 8192, 2048), (40, 3072, 1024)])
@pytest.mark.parametrize("B", [1, 4])
def test_ragged_rows_and_chunk_columns(N, K, chunk, B):
    w = synth.fill((N, K), seed=N * 7 + K, scale=0.02, p1=0.005, f1=300.0)
    m = _huffman_only(w, chunk)
    _check(m, w, B, seed=N + K + B)


@pytest.mark.parametrize("B", [1, 3, 8])
def test_verbatim_heavy(B):
    # outliers far outside the palette in ~12% of the blocks (ten times the Gaussian configurations' share):
    # chunks mixing verbatim and coded blocks
    w = synth.fill((96, 2048), seed=21, scale=0.02, p1=0.006, f1=1e5)
    m = _huffman_only(w)
    info = m.info
    assert info["n_verbatim"] > info["n_blocks"] // 10
    _check(m, w, B, seed=22 + B)


def test_heavy_tail_rows():
    w = synth.fill((128, 8192), seed=5, kind=synth.STUDENT_T3, scale=0.02)
    for chunk, L in ((256, 12), (1024, 12), (64, 7)):
        _check(_huffman_only(w, chunk, L), w, 2, seed=chunk + L)


def test_single_symbol_palette_and_all_verbatim():
    # one exponent: every code is one bit long
    w = np.full((40, 512), 0x3C00, np.uint16) ^ (np.arange(512, dtype=np.uint16) & 0x807F)[None, :]
    _check(_huffman_only(w), w, 3, seed=31)
    # 17+ exponents in every block: every block verbatim, an empty code stream
    rng = np.random.default_rng(3)
    e = (np.arange(64) % 20 + 110).astype(np.uint16)
    w2 = np.stack([rng.permutation(np.tile(e, 8)) for _ in range(33)]).astype(np.uint16) << 7
    w2 |= rng.integers(0, 256, size=w2.shape).astype(np.uint16) & 0x807F
    m2 = _huffman_only(w2)
    assert m2.info["n_verbatim"] == m2.info["n_blocks"]
    _check(m2, w2, 2, seed=32)


def test_exact_integer_case():
    rng = np.random.default_rng(1)
    N, K, B = 70, 512, 5
    Wi = (rng.integers(-3, 4, size=(N, K)) * 2.0 ** rng.integers(0, 3, size=(N, K))).astype(np.float32)
    Xi = rng.integers(-4, 5, size=(B, K)).astype(np.float32)
    w = (Wi.view(np.uint32) >> 16).astype(np.uint16)
    x = (Xi.view(np.uint32) >> 16).astype(np.uint16)
    exact = Xi.astype(np.float64) @ Wi.astype(np.float64).T
    for chunk in (64, 256):
        for p in (HD, (HD, uw.KERNEL_GEMV, 0, 1)):
            assert np.array_equal(run_matmul(_huffman_only(w, chunk), x, p), exact)


def test_repeated_calls_and_auto_default():
    # the target is zeroed by every call; AUTO takes this strategy for a Huffman matrix without its palette form
    t = torch()
    mat = synth.tiny()
    w = mat.weights()
    m = _huffman_only(w)
    assert m.plan_for(1).strategy == HD and m.plan_for(8).strategy == HD
    assert m.plan_for(9).strategy == uw.STRAT_PALETTE_TRANSCODE
    B = 4
    x = synth.fill((B, mat.K), seed=41)
    yref, absum = oracle.matmul(w, x)
    xd = to_dev_u16(x)
    y = t.empty((B, mat.N), dtype=t.float32, device="cuda")
    need = m.workspace_size(B)
    ws = dev_bytes(need)
    for _ in range(3):
        m.matmul(xd, B, y, uw.OUT_F32, uw.STRAT_AUTO, ws, need)
    t.cuda.synchronize()
    assert tol_ok(y.cpu().numpy().astype(np.float64), yref, absum)[0]
    m.check()


def test_unsupported_cases():
    t = torch()
    w = synth.tiny().weights()
    x = to_dev_u16(synth.fill((9, 512), seed=1))
    y = t.empty((9, 256), device="cuda")
    ws = dev_bytes(1 << 20)
    m = _huffman_only(w)
    with pytest.raises(uw.UwError) as e:  # B > 8
        m.matmul(x, 9, y, uw.OUT_F32, HD, ws, 1 << 20)
    assert e.value.status == uw.ERR_UNSUPPORTED
    for plan in ((HD, uw.KERNEL_TC, 0, 0), (HD, uw.KERNEL_GEMV, 2, 0), (HD, uw.KERNEL_GEMV, 0, 4)):
        with pytest.raises(uw.UwError) as e:
            m.matmul_plan(x, 1, y, uw.Plan(*plan), uw.OUT_F32, ws, 1 << 20)
        assert e.value.status == uw.ERR_UNSUPPORTED
    for blob in (uw.encode(w, uw.CODEC_PALETTE), uw.encode(w, uw.CODEC_HUFFMAN, 256, 15)):
        with pytest.raises(uw.UwError) as e:  # palette codec; code lengths beyond the 12-bit table
            uw.Matrix(blob).matmul(x, 1, y, uw.OUT_F32, HD, ws, 1 << 20)
        assert e.value.status == uw.ERR_UNSUPPORTED


def test_corrupt_stream_latched():
    t = torch()
    w = synth.tiny().weights()
    b = bytearray(uw.encode(w, uw.CODEC_HUFFMAN))
    off, n = oracle.parse_header(bytes(b))["sections"]["bits"]
    for i in range(off + 40, off + n - 40, 97):
        b[i] ^= 0x5A
    m = uw.Matrix(bytes(b))
    x = to_dev_u16(synth.fill((1, 512), seed=2))
    y = t.empty((1, 256), device="cuda")
    need = m.workspace_size(1, HD)
    for v in (0, 1):
        m.matmul_plan(x, 1, y, uw.Plan(HD, uw.KERNEL_GEMV, 0, v), uw.OUT_F32, dev_bytes(need), need)
        with pytest.raises(uw.UwError) as e:
            m.check()
        assert e.value.status == uw.ERR_CORRUPT
        m.check()


@pytest.mark.parametrize("B", [1, 4, 8])
def test_gate_8b_full_size(B):
    mat = synth.gate_8b()
    w = mat.weights()
    x = mat.activations(B)
    rows = check_rows(mat.N, B, seed=B)
    yref, absum = oracle_ref("gate_8b", w, x, rows)
    m = _huffman_only(w)
    y = pick(run_matmul(m, x, uw.STRAT_AUTO), rows)
    ok, worst = tol_ok(y, yref, absum)
    assert ok, worst
    y = pick(run_matmul(m, x, HD, uw.OUT_BF16), rows)
    assert tol_ok(y, yref, absum, True)[0]
    y = pick(run_matmul(m, x, (HD, uw.KERNEL_GEMV, 0, 1)), rows)
    assert tol_ok(y, yref, absum)[0]
    m.check()


@pytest.mark.parametrize("which", ["down", "gate"])
def test_70b_shapes(which):
    mats = {mm.name.split(".")[-1]: mm for mm in synth.mlp_70b()}
    mat = mats[which]
    w = mat.weights()
    x = mat.activations(1)
    yref, absum = oracle_ref("70b_" + which, w, x)
    m = _huffman_only(w)
    for p in (HD, (HD, uw.KERNEL_GEMV, 0, 1)):
        y = run_matmul(m, x, p)
        ok, worst = tol_ok(y, yref, absum)
        assert ok, (p, worst)
    m.check()
