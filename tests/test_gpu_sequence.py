"""The sequence runner: hard steps (matrices held as their Huffman stream alone) transcoded on a side stream into
double-buffered slots while the main stream runs the steps before them; easy steps (palette form resident) run
their AUTO plan.  Cloudflare blog "Unweight", section on scheduling hard and easy layers.  Every step's output is
compared with the oracle's fp64 contraction on every row, for several hard/easy patterns, batch sizes and output
dtypes, with and without groups of steps marked to run concurrently, eagerly and replayed from a CUDA graph
captured from the main stream."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth
from uwtest import dev_bytes, to_dev_u16, tol_ok, torch

pytestmark = pytest.mark.gpu

LAYERS = 4
SHAPES = ((384, 512), (384, 512), (512, 384))  # gate, up, down of a small MLP


@pytest.fixture(scope="module")
def stack():
    ws = [synth.fill(SHAPES[i % 3], seed=9000 + i, scale=0.02, p1=2e-3, f1=100.0) for i in range(3 * LAYERS)]
    blobs = [uw.encode(w, uw.CODEC_HUFFMAN) for w in ws]
    return ws, blobs


def _mats(blobs, hard_layers):
    return [uw.Matrix(b, resident="huffman" if (i // 3) in hard_layers else "palette") for i, b in enumerate(blobs)]


def _run(mats, ws, B, out_dtype, graph=False, decode_sms=0, tune=False, flags=None):
    t = torch()
    xs = [synth.fill((B, w.shape[1]), seed=100 * B + i) for i, w in enumerate(ws)]
    ys = [t.full((B, w.shape[0]), float("nan"), dtype=t.float32 if out_dtype == uw.OUT_F32 else t.bfloat16,
                 device="cuda") for w in ws]
    xd = [to_dev_u16(x) for x in xs]
    steps = [(m, x, y, out_dtype, flags(i) if flags else 0) for i, (m, x, y) in enumerate(zip(mats, xd, ys))]
    need = uw.sequence_workspace_size(steps, B)
    wsb = t.empty(need + 256, dtype=t.uint8, device="cuda")
    wsp = (wsb.data_ptr() + 255) // 256 * 256
    main, side = t.cuda.Stream(), t.cuda.Stream()
    if tune:
        decode_sms = uw.sequence_tune(steps, B, wsp, need, main, side)
        splits = (uw.SEQ_DIRECT, 0, 8, 16, 24, 32, 40, 48, 64, 80, 96)
        assert decode_sms in splits + (tuple(uw.SEQ_GROUPS + d for d in splits) if flags else ())
        t.cuda.synchronize()
        for y in ys:
            y.fill_(float("nan"))
    # eager (its first call also creates the thread's events)
    uw.sequence_run(steps, B, wsp, need, main, side, decode_sms)
    if graph:
        t.cuda.synchronize()
        for y in ys:
            y.fill_(float("nan"))
        g = t.cuda.CUDAGraph()
        with t.cuda.graph(g, stream=main):
            uw.sequence_run(steps, B, wsp, need, main, side, decode_sms)
        for _ in range(2):
            g.replay()
    t.cuda.synchronize()
    for i, (w, x, y) in enumerate(zip(ws, xs, ys)):
        yref, absum = oracle.matmul(w, x)
        ok, worst = tol_ok(y.float().cpu().numpy().astype(np.float64), yref, absum, out_dtype == uw.OUT_BF16)
        assert ok, (i, worst)
    for m in mats:
        m.check()


@pytest.mark.parametrize("hard_layers", [(), (1,), (0, 2), (0, 1, 2, 3)])
@pytest.mark.parametrize("B", [1, 4, 20, 100])
def test_sequence_matches_the_oracle(stack, hard_layers, B):
    ws, blobs = stack
    _run(_mats(blobs, set(hard_layers)), ws, B, uw.OUT_F32)


@pytest.mark.parametrize("hard_layers", [(1, 3), (0, 1, 2, 3)])
@pytest.mark.parametrize("decode_sms", [0, 40, uw.SEQ_DIRECT])
def test_sequence_in_a_cuda_graph_and_bf16(stack, hard_layers, decode_sms):
    ws, blobs = stack
    _run(_mats(blobs, set(hard_layers)), ws, 3, uw.OUT_BF16, graph=True, decode_sms=decode_sms)


@pytest.mark.parametrize("B", [1, 16])
def test_sequence_with_a_decode_split(stack, B):
    # the matmuls' grids sized for the SMs left beside the transcode: same results; and the tuner's choice
    ws, blobs = stack
    for d in (8, 76, 151, uw.SEQ_DIRECT):
        _run(_mats(blobs, {0, 2}), ws, B, uw.OUT_F32, decode_sms=d)
    _run(_mats(blobs, {1, 2}), ws, B, uw.OUT_F32, tune=True)


def _up_beside_gate(i):
    return uw.STEP_CONCURRENT if i % 3 == 1 else 0


def _all_after_first(i):
    return uw.STEP_CONCURRENT if i else 0


@pytest.mark.parametrize("hard_layers", [(), (1,), (0, 1, 2, 3)])
@pytest.mark.parametrize("decode_sms", [0, 40, uw.SEQ_DIRECT])
@pytest.mark.parametrize("B", [1, 20])
def test_sequence_concurrent_groups(stack, hard_layers, decode_sms, B):
    # each layer's up projection marked to overlap its gate projection: with UW_SEQ_GROUPS the groups are forked
    # onto the library's streams, eagerly and replayed from a graph captured from the main stream; without it
    # they run in order
    ws, blobs = stack
    for g in (uw.SEQ_GROUPS, 0):
        _run(_mats(blobs, set(hard_layers)), ws, B, uw.OUT_F32, graph=True, decode_sms=g + decode_sms,
             flags=_up_beside_gate)


@pytest.mark.parametrize("decode_sms", [0, uw.SEQ_DIRECT])
def test_sequence_one_group_longer_than_the_lanes(stack, decode_sms):
    # twelve independent steps in one group: four streams, the members after the fourth reuse a stream and its
    # part of the workspace after the member four places before them
    ws, blobs = stack
    _run(_mats(blobs, {1}), ws, 5, uw.OUT_BF16, graph=True, decode_sms=uw.SEQ_GROUPS + decode_sms,
         flags=_all_after_first)
    _run(_mats(blobs, {0, 3}), ws, 2, uw.OUT_F32, tune=True, flags=_all_after_first)


def test_sequence_concurrent_workspace_and_flags(stack):
    t = torch()
    ws, blobs = stack
    mats = _mats(blobs, set())
    xs = [to_dev_u16(synth.fill((2, w.shape[1]), seed=i)) for i, w in enumerate(ws[:3])]
    ys = [t.empty((2, w.shape[0]), device="cuda") for w in ws[:3]]
    plain = [(m, x, y, uw.OUT_F32, 0) for m, x, y in zip(mats, xs, ys)]
    one = uw.sequence_workspace_size(plain, 2)
    paired = uw.sequence_workspace_size(plain[:1] + [plain[1][:4] + (uw.STEP_CONCURRENT,)] + plain[2:], 2)
    three = uw.sequence_workspace_size([st[:4] + (uw.STEP_CONCURRENT if i else 0,) for i, st in enumerate(plain)], 2)
    assert paired == 2 * one and three == 3 * one  # one matmul workspace per stream the largest group uses
    with pytest.raises(uw.UwError) as e:  # an unknown flag
        uw.sequence_workspace_size(plain[:1] + [plain[1][:4] + (2,)], 2)
    assert e.value.status == uw.ERR_INVALID_ARG


def test_sequence_workspace_and_argument_errors(stack):
    t = torch()
    ws, blobs = stack
    mats = _mats(blobs, {0})
    x = to_dev_u16(synth.fill((1, 512), seed=1))
    y = t.empty((1, 384), device="cuda")
    steps = [(mats[0], x, y)]
    need = uw.sequence_workspace_size(steps, 1)
    assert need >= 2 * (384 * 512 // 2)  # two slots of 4-bit codes
    s = t.cuda.Stream()
    buf = dev_bytes(need + 256)
    p = (buf.data_ptr() + 255) // 256 * 256
    with pytest.raises(uw.UwError) as e:
        uw.sequence_run(steps, 1, p, need - 256, s, t.cuda.Stream())
    assert e.value.status == uw.ERR_WORKSPACE
    with pytest.raises(uw.UwError) as e:  # a hard step needs a separate side stream
        uw.sequence_run(steps, 1, p, need, s, s)
    assert e.value.status == uw.ERR_INVALID_ARG
    with pytest.raises(uw.UwError) as e:  # the split must leave the matmuls at least one SM
        uw.sequence_run(steps, 1, p, need, s, t.cuda.Stream(), 100000)
    assert e.value.status == uw.ERR_INVALID_ARG
    for bad in (-2, uw.SEQ_GROUPS - 2, uw.SEQ_GROUPS + 100000):  # below the direct schedule, or past the SMs
        with pytest.raises(uw.UwError) as e:
            uw.sequence_run(steps, 1, p, need, s, t.cuda.Stream(), bad)
        assert e.value.status == uw.ERR_INVALID_ARG
    uw.sequence_run(steps, 1, p, need, s, s, uw.SEQ_DIRECT)  # no transcode: one stream is enough
    uw.sequence_run([], 1, None, 0, s, s)  # nothing to run
