"""GPU parity: uw_decode (palette and Huffman kernels) is bit-exact against the
oracle's decoder on the same blob; corrupt streams are caught on the device.
Cloudflare blog "Unweight": results paragraph (every compression is bit-exact)."""
import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth
from uwtest import dev_bytes, torch

pytestmark = pytest.mark.gpu


def _cases():
    yield "tiny", lambda: synth.tiny().weights()
    yield "enum", lambda: np.arange(65536, dtype=np.uint16).reshape(1024, 64)
    yield "bits", lambda: synth.random_bits((33, 448), seed=3)
    yield "ragged", lambda: synth.fill((17, 192), seed=4, scale=0.02, p1=0.01, f1=1e4)
    yield "heavy", lambda: synth.fill((128, 8192), seed=5, kind=synth.STUDENT_T3, scale=0.02)
    yield "one_row", lambda: synth.fill((1, 64), seed=6, scale=1.0)


@pytest.mark.parametrize("codec,chunk,L", [(0, 256, 12), (1, 256, 12), (1, 64, 5), (1, 512, 15)])
@pytest.mark.parametrize("name,make", list(_cases()), ids=[c[0] for c in _cases()])
def test_decode_bit_exact(name, make, codec, chunk, L):
    t = torch()
    w = make()
    blob = uw.encode(w, codec, chunk, L)
    ref = oracle.decode(blob)
    m = uw.Matrix(blob)
    out = t.empty(w.shape, dtype=t.int16, device="cuda")
    m.decode(out)
    m.check()
    got = out.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    assert np.array_equal(got, w)


@pytest.mark.parametrize("chunk,L", [(256, 12), (64, 5), (512, 15), (2048, 12)])
@pytest.mark.parametrize("name,make", list(_cases()), ids=[c[0] for c in _cases()])
def test_transcoded_palette_form_bit_exact(name, make, chunk, L):
    # the load-time transcode (Huffman stream -> 4-bit codes, the palette-transcode preprocess) must give codes
    # that decode to the original bits; the stream is dropped, so every later read goes through those codes
    t = torch()
    w = make()
    blob = uw.encode(w, uw.CODEC_HUFFMAN, chunk, L)
    m = uw.Matrix(blob, resident="palette")
    assert not m.info["has_huffman_stream"]
    out = t.empty(w.shape, dtype=t.int16, device="cuda")
    m.decode(out)
    m.check()
    assert np.array_equal(out.cpu().numpy().view(np.uint16), w)


@pytest.mark.parametrize("codec", [0, 1])
def test_decode_full_size_gate_8b(codec):
    t = torch()
    mat = synth.gate_8b()
    w = mat.weights()
    blob = uw.encode(w, codec)
    m = uw.Matrix(blob)
    out = t.empty(w.shape, dtype=t.int16, device="cuda")
    m.decode(out)
    m.check()
    got = out.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, w)
    # the oracle decodes the same blob to the same bits (sampled rows: the oracle is slow)
    if codec == 0:
        assert np.array_equal(oracle.decode(blob), got)


def test_empty_matrix_decode_is_noop():
    t = torch()
    m = uw.Matrix(uw.encode(np.zeros((0, 64), np.uint16)))
    m.decode(None)
    m.check()


def _corrupt_huffman_blob():
    w = synth.tiny().weights()
    b = bytearray(uw.encode(w, uw.CODEC_HUFFMAN))
    off, n = oracle.parse_header(bytes(b))["sections"]["bits"]
    for i in range(off + 40, off + n - 40, 97):  # flip bits through the stream
        b[i] ^= 0x5A
    return bytes(b)


def test_corrupt_stream_detected_at_load():
    blob = _corrupt_huffman_blob()
    uw.validate(blob)  # host checks cannot see inside the bit stream
    with pytest.raises(uw.UwError) as e:
        uw.Matrix(blob, want_palette_form=True)
    assert e.value.status == uw.ERR_CORRUPT


def test_corrupt_stream_detected_by_check():
    t = torch()
    blob = _corrupt_huffman_blob()
    m = uw.Matrix(blob)
    out = t.empty((256, 512), dtype=t.int16, device="cuda")
    m.decode(out)
    with pytest.raises(uw.UwError) as e:
        m.check()
    assert e.value.status == uw.ERR_CORRUPT
    m.check()  # the status word was cleared
