"""uw_matmul_noalloc: the palette-transcode matmul for callers that cannot call
cudaMalloc (an engine whose allocator owns all device memory, or a path that must
not take cudaMalloc's device synchronisation).  Its scratch is a static 36 MiB
device array inside the library.  Checked through the C ABI, on two calls in a
row, against the oracle's fp64 contraction and against the existing entry point
(uw_matmul, palette-transcode strategy), within the tolerance the other parity
tests use; sizes beyond the array are rejected, whether the 4-bit codes or the
accumulator overflow it.  This file is collected last on purpose."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth
from uwtest import dev_bytes, to_dev_u16, tol_ok, torch

pytestmark = pytest.mark.gpu

SCRATCH = 36 * 1024 * 1024


def _existing(m, x, B, out_dtype):
    t = torch()
    need = m.workspace_size(B, uw.STRAT_PALETTE_TRANSCODE)
    ws = dev_bytes(need)
    y = t.empty((B, m.N), dtype=t.float32 if out_dtype == uw.OUT_F32 else t.bfloat16, device="cuda")
    m.matmul(x, B, y, out_dtype, uw.STRAT_PALETTE_TRANSCODE, ws, need)
    t.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


def _noalloc(m, x, B, out_dtype):
    t = torch()
    y = t.full((B, m.N), float("nan"), dtype=t.float32 if out_dtype == uw.OUT_F32 else t.bfloat16, device="cuda")
    m.matmul_noalloc(x, B, y, out_dtype)
    t.cuda.synchronize()
    m.check()
    return y.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape,B", [((256, 512), 1), ((4096, 4096), 1), ((4096, 4096), 4), ((1024, 14336), 3)])
@pytest.mark.parametrize("out_dtype", [uw.OUT_F32, uw.OUT_BF16])
def test_noalloc_matches_existing_entry_point_twice(shape, B, out_dtype):
    N, K = shape
    w = synth.fill(shape, seed=N + K, scale=0.02, p1=1e-3, f1=100.0)
    x_np = synth.fill((B, K), seed=N + K + 1)
    yref, absum = oracle.matmul(w, x_np)
    m = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN))
    x = to_dev_u16(x_np)
    existing = _existing(m, x, B, out_dtype)
    assert tol_ok(existing, yref, absum, out_dtype == uw.OUT_BF16)[0]
    for _ in range(2):  # the shared array keeps the previous call's contents
        got = _noalloc(m, x, B, out_dtype)
        ok, worst = tol_ok(got, yref, absum, out_dtype == uw.OUT_BF16)
        assert ok, ("against the oracle", worst)
        ok, worst = tol_ok(got, existing, absum, out_dtype == uw.OUT_BF16)
        assert ok, ("against uw_matmul", worst)


def test_noalloc_rejects_sizes_beyond_the_array():
    # 16384 x 4800 weights -> 4-bit codes of 39.3 MB > 36 MiB
    w = np.full((16384, 4800), 0x3F80, np.uint16)
    m = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN))
    t = torch()
    x = t.zeros((1, 4800), dtype=t.int16, device="cuda")
    y = t.empty((1, 16384), device="cuda")
    with pytest.raises(uw.UwError) as e:
        m.matmul_noalloc(x, 1, y)
    assert e.value.status == uw.ERR_WORKSPACE and "static scratch" in e.value.message


def test_noalloc_rejects_an_accumulator_beyond_the_array():
    # 65536 x 64 weights: 2 MiB of codes fit, but B = 160 needs a 160 x 65536 fp32 accumulator of 40 MiB
    w = np.full((65536, 64), 0x3F80, np.uint16)
    m = uw.Matrix(uw.encode(w, uw.CODEC_HUFFMAN))
    t = torch()
    x = t.zeros((160, 64), dtype=t.int16, device="cuda")
    y = t.empty((160, 65536), device="cuda")
    with pytest.raises(uw.UwError) as e:
        m.matmul_noalloc(x, 160, y)
    assert e.value.status == uw.ERR_WORKSPACE and "accumulator" in e.value.message


def test_noalloc_rejects_palette_codec():
    m = uw.Matrix(uw.encode(synth.tiny().weights(), uw.CODEC_PALETTE))
    t = torch()
    with pytest.raises(uw.UwError) as e:
        m.matmul_noalloc(t.zeros((1, 512), dtype=t.int16, device="cuda"), 1, t.empty((1, 256), device="cuda"))
    assert e.value.status == uw.ERR_UNSUPPORTED
