"""What a loaded matrix keeps on the device, and what it then runs.

The Cloudflare blog "Unweight" (results section) measures the memory saved by keeping weights compressed.  A
Huffman blob can stay resident as its stream alone, as the 4-bit palette form alone (the post's load-time
transcode, after which the stream is dropped), or as both.  For each form: the bytes it holds on the 8B gate_proj
against 2 N K bytes of BF16, bit-exact decode, the strategies it offers against the oracle, and the ones it does not
offer rejected with UW_ERR_UNSUPPORTED."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth
from uwtest import check_rows, oracle_ref, pick, run_matmul, strategies_for, tol_ok, to_dev_u16, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gate():
    mat = synth.gate_8b()
    w = mat.weights()
    return mat, w, uw.encode(w, uw.CODEC_HUFFMAN)


def test_footprint_of_each_resident_form(gate):
    mat, w, blob = gate
    bf16 = 2 * mat.N * mat.K
    ratio = {}
    for r in ("huffman", "palette", "both"):
        m = uw.Matrix(blob, resident=r)
        ratio[r] = m.info["device_bytes"] / bf16
        assert m.info["has_huffman_stream"] == (r != "palette")
        assert m.info["has_palette_form"] == (r != "huffman")
        m.close()
    # the stream alone is the smallest form; the palette form alone drops the stream after the transcode
    assert ratio["huffman"] <= 0.70, ratio
    assert ratio["palette"] <= 0.78, ratio
    assert ratio["huffman"] < ratio["palette"] < ratio["both"], ratio


@pytest.mark.parametrize("resident", ["huffman", "palette", "both"])
def test_each_form_decodes_and_multiplies(gate, resident):
    t = torch()
    mat, w, blob = gate
    m = uw.Matrix(blob, resident=resident)
    out = t.empty(w.shape, dtype=t.int16, device="cuda")
    m.decode(out)
    m.check()
    assert np.array_equal(out.cpu().numpy().view(np.uint16), w)
    del out
    for B in (1, 16):
        x = mat.activations(B)
        rows = check_rows(mat.N, B, seed=B)
        yref, absum = oracle_ref("gate_8b", w, x, rows)
        strategies = strategies_for(m) + ([uw.STRAT_HUFFMAN_DIRECT] if resident != "palette" and B <= 8 else [])
        for s in strategies + [uw.STRAT_AUTO]:
            y = pick(run_matmul(m, x, s), rows)
            ok, worst = tol_ok(y, yref, absum)
            assert ok, (resident, B, s, worst)
    if resident == "palette":
        x = to_dev_u16(mat.activations(1))
        y = t.empty((1, mat.N), device="cuda")
        for s in (uw.STRAT_PALETTE_TRANSCODE, uw.STRAT_HUFFMAN_DIRECT):
            with pytest.raises(uw.UwError) as e:
                m.matmul(x, 1, y, uw.OUT_F32, s)
            assert e.value.status == uw.ERR_UNSUPPORTED
        with pytest.raises(uw.UwError) as e:
            m.matmul_noalloc(x, 1, y)
        assert e.value.status == uw.ERR_UNSUPPORTED
    m.check()
