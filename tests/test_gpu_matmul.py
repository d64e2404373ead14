"""GPU parity: uw_matmul against the oracle's fp64 contraction, for every
strategy (the four pipelines of the Cloudflare blog "Unweight"), every kernel,
ragged shapes and batch sizes, fp32 and bf16 outputs; full-size configurations
are checked on every row up to B = 4 and on 1024+ rows spread over every CTA's range beyond, in the launch
configuration the bench times."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth
from uwtest import check_rows, dev_bytes, oracle_ref, pick, run_matmul, strategies_for, tol_ok, to_dev_u16, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    mat = synth.tiny()
    w = mat.weights()
    return mat, w, {c: uw.Matrix(uw.encode(w, c), want_palette_form=True) for c in (0, 1)}


@pytest.mark.parametrize("codec", [0, 1])
@pytest.mark.parametrize("B", [1, 2, 3, 5, 8, 13])
@pytest.mark.parametrize("out_dtype", [uw.OUT_F32, uw.OUT_BF16])
def test_tiny_all_strategies(tiny, codec, B, out_dtype):
    mat, w, mats = tiny
    m = mats[codec]
    x = synth.fill((B, mat.K), seed=mat.seed + 500 + B)
    yref, absum = oracle.matmul(w, x)
    for s in strategies_for(m):
        for split in (0, 1, 2):
            y = run_matmul(m, x, (s, uw.KERNEL_GEMV, split, 0), out_dtype)
            ok, worst = tol_ok(y, yref, absum, out_dtype == uw.OUT_BF16)
            assert ok, (s, split, worst)


@pytest.mark.parametrize("N,K,B", [(1, 64, 1), (17, 192, 3), (33, 576, 8), (16, 4160, 2), (300, 1024, 1)])
def test_ragged_shapes(N, K, B):
    w = synth.fill((N, K), seed=N * 7 + K, scale=0.02, p1=0.005, f1=300.0)
    x = synth.fill((B, K), seed=N + K)
    yref, absum = oracle.matmul(w, x)
    for codec in (0, 1):
        m = uw.Matrix(uw.encode(w, codec, 128, 12), want_palette_form=True)
        for s in strategies_for(m):
            y = run_matmul(m, x, s)
            ok, worst = tol_ok(y, yref, absum)
            assert ok, (codec, s, worst)


def test_exact_integer_case_all_strategies():
    # W and X small integers: every product and sum is exact in fp32 too, so Y is exact.
    rng = np.random.default_rng(1)
    N, K, B = 40, 256, 4
    Wi = (rng.integers(-3, 4, size=(N, K)) * 2.0 ** rng.integers(0, 3, size=(N, K))).astype(np.float32)
    Xi = rng.integers(-4, 5, size=(B, K)).astype(np.float32)
    w = (Wi.view(np.uint32) >> 16).astype(np.uint16)
    x = (Xi.view(np.uint32) >> 16).astype(np.uint16)
    exact = Xi.astype(np.float64) @ Wi.astype(np.float64).T
    yref, _ = oracle.matmul(w, x)
    assert np.array_equal(yref, exact)
    for codec in (0, 1):
        m = uw.Matrix(uw.encode(w, codec), want_palette_form=True)
        for s in strategies_for(m):
            assert np.array_equal(run_matmul(m, x, s), exact), (codec, s)


def test_zero_k_and_zero_b():
    t = torch()
    m = uw.Matrix(uw.encode(np.zeros((5, 0), np.uint16)))
    y = t.full((2, 5), 7.0, device="cuda")
    x = t.zeros((2, 0), dtype=t.int16, device="cuda")
    ws = dev_bytes(m.workspace_size(2))
    m.matmul(x if x.numel() else dev_bytes(16), 2, y, uw.OUT_F32, uw.STRAT_AUTO, ws, m.workspace_size(2))
    t.cuda.synchronize()
    assert (y.cpu().numpy() == 0).all()
    m2 = uw.Matrix(uw.encode(synth.tiny().weights()))
    m2.matmul(None, 0, None)  # B == 0 is a no-op


def test_error_paths():
    t = torch()
    w = synth.tiny().weights()
    mh = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN))  # no palette form
    x = to_dev_u16(synth.fill((1, 512), seed=1))
    y = t.empty((1, 256), device="cuda")
    with pytest.raises(uw.UwError) as e:
        mh.matmul(x, 1, y, uw.OUT_F32, uw.STRAT_DIRECT_PALETTE)
    assert e.value.status == uw.ERR_UNSUPPORTED
    need = mh.workspace_size(1, uw.STRAT_FULL_DECODE)
    small = dev_bytes(need)
    with pytest.raises(uw.UwError) as e:
        mh.matmul(x, 1, y, uw.OUT_F32, uw.STRAT_FULL_DECODE, small, need - 256)
    assert e.value.status == uw.ERR_WORKSPACE
    with pytest.raises(uw.UwError) as e:
        mh.matmul(x.data_ptr() + 2, 1, y, uw.OUT_F32, uw.STRAT_EXP_ONLY, small, need)
    assert e.value.status == uw.ERR_INVALID_ARG
    with pytest.raises(uw.UwError) as e:
        mh.matmul(x, -1, y)
    assert e.value.status == uw.ERR_SHAPE


@pytest.mark.parametrize("B", [1, 4, 16])
def test_gate_8b_full_size(B):
    mat = synth.gate_8b()
    w = mat.weights()
    x = mat.activations(B)
    rows = check_rows(mat.N, B, seed=B)
    yref, absum = oracle_ref("gate_8b", w, x, rows)
    m = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN), want_palette_form=True)
    for s in strategies_for(m):
        y = pick(run_matmul(m, x, s), rows)
        ok, worst = tol_ok(y, yref, absum)
        assert ok, (s, worst)
    y = pick(run_matmul(m, x, uw.STRAT_AUTO, uw.OUT_BF16), rows)
    assert tol_ok(y, yref, absum, True)[0]


@pytest.mark.parametrize("which,B", [("down", 1), ("gate", 1), ("down", 32)])
def test_70b_shapes(which, B):
    mats = {m.name.split(".")[-1]: m for m in synth.mlp_70b()}
    mat = mats[which]
    w = mat.weights()
    x = mat.activations(B)
    rows = check_rows(mat.N, B, seed=B + 1)
    yref, absum = oracle_ref("70b_" + which, w, x, rows)
    m = uw.Matrix(uw.encode(w, uw.CODEC_PALETTE))
    y = pick(run_matmul(m, x, uw.STRAT_DIRECT_PALETTE), rows)
    ok, worst = tol_ok(y, yref, absum)
    assert ok, worst


def test_autotune_and_tune_table():
    t = torch()
    mat = synth.tiny()
    w = mat.weights()
    m = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN), want_palette_form=True)
    batches = [1, 4]
    need = m.autotune_workspace_size(batches)
    ws = dev_bytes(need)
    m.autotune(batches, ws, need)
    text = m.tune_save()
    lines = [l.split() for l in text.strip().splitlines()]
    assert sorted(int(l[0]) for l in lines) == [1, 4]
    p1 = m.plan_for(1)
    assert p1.strategy in (1, 2, 3, 4, 5)
    m2 = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN), want_palette_form=True)
    m2.tune_load(text)
    assert m2.plan_for(1).as_tuple() == p1.as_tuple()
    with pytest.raises(uw.UwError):
        m2.tune_load("1 9 1 0 0 1.0\n")
    assert m2.plan_for(1).as_tuple() == p1.as_tuple()  # unchanged after a rejected load
    x = synth.fill((4, mat.K), seed=3)
    yref, absum = oracle.matmul(w, x)
    assert tol_ok(run_matmul(m, x, uw.STRAT_AUTO), yref, absum)[0]


def test_matmul_host_end_to_end():
    t = torch()
    mat = synth.tiny()
    w = mat.weights()
    m = uw.Matrix(uw.encode(w))
    B = 3
    x = synth.fill((B, mat.K), seed=8)
    yref, absum = oracle.matmul(w, x)
    xh = t.from_numpy(x.view(np.int16)).pin_memory()
    yh = t.empty((B, mat.N), dtype=t.float32).pin_memory()
    need = m.host_workspace_size(B)
    ws = dev_bytes(need)
    m.matmul_host(xh, B, yh, uw.OUT_F32, ws, need)
    assert tol_ok(yh.numpy().astype(np.float64), yref, absum)[0]
    # the asynchronous form on two streams, each call with its own buffers; results read after a synchronise
    streams = [t.cuda.Stream(), t.cuda.Stream()]
    wss = [dev_bytes(need), dev_bytes(need)]
    ys = [t.full((B, mat.N), float("nan"), dtype=t.float32).pin_memory() for _ in range(4)]
    for i in range(4):
        m.matmul_host_async(xh, B, ys[i], uw.OUT_F32, wss[i % 2], need, streams[i % 2])
    t.cuda.synchronize()
    for i in range(4):
        assert tol_ok(ys[i].numpy().astype(np.float64), yref, absum)[0], i
