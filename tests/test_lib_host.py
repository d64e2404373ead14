"""Host-side checks of libuw.so that need no GPU: every symbol declared in
include/uw.h is exported; the library's encoder (an independent implementation)
writes exactly the oracle's bytes; blob validation rejects corrupt blobs; the
binding fails loudly when the library is missing."""
import ctypes
import struct

import numpy as np
import pytest

import lossless_bf16_weight_exponent_gb300 as uw
import oracle
import synth


@pytest.fixture(scope="module", autouse=True)
def _built():
    import lossless_bf16_weight_exponent_gb300._build as b
    b.build()


def test_exports_every_header_symbol():
    L = ctypes.CDLL(uw.LIB_PATH)
    syms = uw.header_symbols()
    assert "uw_matmul" in syms and "uw_encode" in syms and "uw_autotune" in syms
    for s in syms:
        assert hasattr(L, s), s


def _header_enums():
    """Every `UW_NAME = value` enumerator of include/uw.h."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(uw.LIB_PATH), "..", "include", "uw.h")).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(UW_[A-Z0-9_]+)\s*=\s*(\d+)", src)}


def test_binding_constants_match_the_header():
    # the ctypes binding passes plain integers across the ABI: each of its constants must be the header's value
    e = _header_enums()
    pairs = {"UW_STRAT_AUTO": uw.STRAT_AUTO, "UW_STRAT_FULL_DECODE": uw.STRAT_FULL_DECODE,
             "UW_STRAT_EXP_ONLY": uw.STRAT_EXP_ONLY, "UW_STRAT_PALETTE_TRANSCODE": uw.STRAT_PALETTE_TRANSCODE,
             "UW_STRAT_DIRECT_PALETTE": uw.STRAT_DIRECT_PALETTE, "UW_STRAT_HUFFMAN_DIRECT": uw.STRAT_HUFFMAN_DIRECT,
             "UW_CODEC_PALETTE": uw.CODEC_PALETTE, "UW_CODEC_HUFFMAN": uw.CODEC_HUFFMAN,
             "UW_OUT_F32": uw.OUT_F32, "UW_OUT_BF16": uw.OUT_BF16, "UW_KERNEL_AUTO": uw.KERNEL_AUTO,
             "UW_KERNEL_GEMV": uw.KERNEL_GEMV, "UW_KERNEL_TC": uw.KERNEL_TC, "UW_OK": uw.OK,
             "UW_ERR_INVALID_ARG": uw.ERR_INVALID_ARG, "UW_ERR_SHAPE": uw.ERR_SHAPE,
             "UW_ERR_UNSUPPORTED": uw.ERR_UNSUPPORTED, "UW_ERR_CORRUPT": uw.ERR_CORRUPT,
             "UW_ERR_NO_MEMORY": uw.ERR_NO_MEMORY, "UW_ERR_WORKSPACE": uw.ERR_WORKSPACE, "UW_ERR_CUDA": uw.ERR_CUDA,
             "UW_ERR_TIMEOUT": uw.ERR_TIMEOUT, "UW_ERR_BUFFER_TOO_SMALL": uw.ERR_BUFFER_TOO_SMALL}
    for name, value in pairs.items():
        assert e.get(name) == value, (name, e.get(name), value)
    assert sorted(uw.STRATEGIES.values()) == [v for k, v in sorted(e.items(), key=lambda t: t[1])
                                              if k.startswith("UW_STRAT_") and k != "UW_STRAT_AUTO"]


def test_binding_defines_and_step_layout_match_the_header():
    # the sequence runner's #define constants, and the uw_step struct the binding fills for it
    import os
    import re
    src = open(os.path.join(os.path.dirname(uw.LIB_PATH), "..", "include", "uw.h")).read()
    d = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(UW_[A-Z0-9_]+)\s+\(?(-?\d+)\)?", src)}
    assert d == {"UW_STEP_CONCURRENT": uw.STEP_CONCURRENT, "UW_SEQ_DIRECT": uw.SEQ_DIRECT,
                 "UW_SEQ_GROUPS": uw.SEQ_GROUPS}
    body = re.search(r"typedef struct \{([^}]*)\} uw_step;", src).group(1)
    fields = [re.sub(r"[;*]", " ", ln).split()[-1] for ln in body.strip().splitlines() if ln.strip()]
    assert fields == [f[0] for f in uw.Step._fields_] == ["m", "x", "y", "out_dtype", "flags"]
    assert ctypes.sizeof(uw.Step) == 32 and uw.Step.out_dtype.offset == 24 and uw.Step.flags.offset == 28
    # a direct schedule with groups stays distinguishable from every plain schedule
    assert uw.SEQ_GROUPS + uw.SEQ_DIRECT > 1 << 15


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(uw, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(uw, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        uw.encode(np.zeros((1, 64), np.uint16))


def _cases():
    yield "tiny", synth.tiny().weights()
    yield "enum", np.arange(65536, dtype=np.uint16).reshape(1024, 64)
    yield "bits", synth.random_bits((33, 448), seed=3)
    yield "gauss", synth.fill((96, 4096), seed=5, scale=0.02, p1=1e-4, f1=100.0)
    yield "t3", synth.fill((64, 1024), seed=6, kind=synth.STUDENT_T3, scale=0.02)
    yield "one_exp", ((np.arange(640, dtype=np.uint16) % 128) | (0x7F << 7)).reshape(5, 128)
    yield "row1", synth.fill((1, 64), seed=9, scale=0.5)
    yield "empty", np.zeros((0, 128), np.uint16)
    yield "zero_k", np.zeros((3, 0), np.uint16)
    w = synth.fill((8, 192), seed=10, scale=0.02)
    w[3, 70] = 0x7F80  # +inf -> out of palette
    yield "inf", w


@pytest.mark.parametrize("name,w", list(_cases()), ids=[c[0] for c in _cases()])
@pytest.mark.parametrize("codec,chunk,L", [(0, 256, 12), (1, 256, 12), (1, 64, 4), (1, 192, 15), (1, 1024, 7),
                                         (1, 2048, 12)])
def test_encoder_bytes_equal_oracle(name, w, codec, chunk, L):
    a = uw.encode(w, codec, chunk, L)
    b = oracle.encode(w, codec, chunk, L)
    assert a == b
    info = uw.validate(a)
    assert info["N"] == w.shape[0] and info["K"] == w.shape[1]
    if w.size:
        assert np.array_equal(oracle.decode(a), w)


def test_encoder_rejects_bad_shapes_and_options():
    with pytest.raises(uw.UwError) as e:
        uw.encode(np.zeros((2, 65), np.uint16))
    assert e.value.status == uw.ERR_SHAPE
    for chunk, L in ((100, 12), (0, 12), (256, 3), (256, 16)):
        with pytest.raises(uw.UwError) as e:
            uw.encode(np.zeros((2, 64), np.uint16), uw.CODEC_HUFFMAN, chunk, L)
        assert e.value.status == uw.ERR_INVALID_ARG


def test_buffer_too_small_reports_size():
    w = synth.tiny().weights()
    size = ctypes.c_size_t(0)
    buf = np.zeros(100, np.uint8)
    opts = uw.EncodeOpts(0, 256, 12)
    st = uw.lib().uw_encode(w.ctypes.data, 256, 512, ctypes.byref(opts), buf.ctypes.data, 100, ctypes.byref(size))
    assert st == uw.ERR_BUFFER_TOO_SMALL and size.value == len(oracle.encode(w))


# ------------------------------------------------------------------ corrupt blobs
def _blob(codec):
    return bytearray(oracle.encode(synth.tiny().weights(), codec))


def _sec(b, name):
    return oracle.parse_header(bytes(b))["sections"][name]


def _corruptions():
    def magic(b): b[0] ^= 1
    def version(b): b[4] = 2
    def trunc(b): del b[-256:]
    def shape(b): struct.pack_into("<q", b, 16, 513)
    def block(b): struct.pack_into("<I", b, 28, 32)
    def npal(b): b[40] = 17
    def dup_pal(b): b[42] = b[41]
    def verb_count(b): struct.pack_into("<Q", b, 88, struct.unpack_from("<Q", b, 88)[0] + 1)
    def sec_off(b): struct.pack_into("<Q", b, 128, 512)
    def bitmap_tail(b):
        off, n = _sec(b, "bitmap"); b[off + n - 1] |= 0x80 if (2048 % 32) else 0; b[off] ^= 1
    def prefix(b):
        off, n = _sec(b, "prefix"); struct.pack_into("<I", b, off + 4, struct.unpack_from("<I", b, off + 4)[0] + 1)
    def size_field(b): struct.pack_into("<Q", b, 112, len(b) + 256)
    return dict(magic=magic, version=version, trunc=trunc, shape=shape, block=block, npal=npal, dup_pal=dup_pal,
                verb_count=verb_count, sec_off=sec_off, bitmap=bitmap_tail, prefix=prefix, size_field=size_field)


@pytest.mark.parametrize("codec", [0, 1])
@pytest.mark.parametrize("name", list(_corruptions()))
def test_validation_rejects_corruption(codec, name):
    b = _blob(codec)
    uw.validate(bytes(b))
    _corruptions()[name](b)
    with pytest.raises(uw.UwError) as e:
        uw.validate(bytes(b))
    assert e.value.status == uw.ERR_CORRUPT


def test_validation_rejects_bad_huffman_tables():
    base = _blob(1)
    h = oracle.parse_header(bytes(base))
    # Kraft violation: lengthen one code
    b = bytearray(base); b[57] += 1
    with pytest.raises(uw.UwError):
        uw.validate(bytes(b))
    # length above the limit
    b = bytearray(base); b[57] = 13
    with pytest.raises(uw.UwError):
        uw.validate(bytes(b))
    # chunk offsets decreasing
    b = bytearray(base)
    off, n = h["sections"]["chunk_off"]
    struct.pack_into("<I", b, off + 8, 0)
    with pytest.raises(uw.UwError):
        uw.validate(bytes(b))
    # last offset != total_bits
    b = bytearray(base)
    struct.pack_into("<I", b, off + n - 4, h["total_bits"] - 1)
    with pytest.raises(uw.UwError):
        uw.validate(bytes(b))


def test_validation_rejects_bad_palette_codes():
    w = synth.fill((4, 128), seed=2, scale=0.02)
    w[:, :] = (w & 0x807F) | (np.array([0x78, 0x79, 0x7A], np.uint16)[np.arange(512) % 3].reshape(4, 128) << 7)
    b = bytearray(oracle.encode(w))
    assert oracle.parse_header(bytes(b))["n_pal"] == 3
    off, n = _sec(b, "idx")
    b[off] = 0x0F  # code 15 with a 3-entry palette
    with pytest.raises(uw.UwError) as e:
        uw.validate(bytes(b))
    assert e.value.status == uw.ERR_CORRUPT
