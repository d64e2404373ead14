"""Pins for the oracle's BF16 field split and its lossless round trip.

Cloudflare blog "Unweight": BF16 anatomy paragraphs (1 sign, 8 exponent,
7 mantissa bits; sign+mantissa stored raw) and the results paragraph
(every compression is bit-exact).
"""
import math
import warnings

import numpy as np
import pytest

import oracle
import synth

ALL = np.arange(65536, dtype=np.uint16)


def test_split_matches_ieee_fields_for_every_pattern():
    # Pin the bit positions against the value each pattern denotes (not against a
    # retyped shift): for every finite nonzero pattern, |v| = 2^(e-127) * (1 + m/128)
    # for normals and 2^-126 * m/128 for subnormals; the sign is signbit(v).
    sm, e = oracle.split(ALL)
    with np.errstate(invalid="ignore"):
        v = synth.bf16_to_f32(ALL).astype(np.float64)
    sign = (sm >> 7).astype(int)
    mant = (sm & 0x7F).astype(np.float64)
    for i in range(0, 65536):
        x = v[i]
        if math.isnan(x):
            assert e[i] == 255 and mant[i] != 0
            continue
        assert sign[i] == int(math.copysign(1.0, x) < 0)
        if math.isinf(x):
            assert e[i] == 255 and mant[i] == 0
        elif e[i] == 0:
            assert abs(x) == math.ldexp(mant[i] / 128.0, -126)
        else:
            assert abs(x) == math.ldexp(1.0 + mant[i] / 128.0, int(e[i]) - 127)


def test_split_rebuild_identity_all_65536():
    sm, e = oracle.split(ALL)
    assert np.array_equal(oracle.rebuild(sm, e), ALL)
    # the pair (sm, e) is a bijection of the 16-bit pattern
    assert len(set(zip(sm.tolist(), e.tolist()))) == 65536


@pytest.mark.parametrize("codec", [oracle.PALETTE, oracle.HUFFMAN])
def test_enumeration_matrix_round_trip(codec):
    # Every BF16 pattern once: row n holds patterns 64n..64n+63, so its exponent is
    # (n >> 1) & 0xFF and its sign n >> 9.  All 256 exponents occur 256 times, so
    # the tie rule picks exponents 0..15; rows with (n>>1)&0xFF < 16 are the 64
    # non-verbatim rows (n in [0,32) and [512,544)).
    w = ALL.reshape(1024, 64)
    blob = oracle.encode(w, codec)
    h = oracle.parse_header(blob)
    assert h["palette"] == list(range(16)) and h["n_pal"] == 16
    assert h["n_blocks"] == 1024 and h["n_verbatim"] == 960
    bitmap = np.frombuffer(oracle.section(blob, "bitmap"), np.uint32)
    expect = np.ones(1024, bool)
    expect[0:32] = False
    expect[512:544] = False
    got = ((bitmap[np.arange(1024) // 32] >> (np.arange(1024) % 32)) & 1).astype(bool)
    assert np.array_equal(got, expect)
    assert np.array_equal(oracle.decode(blob), w)


@pytest.mark.parametrize("codec", [oracle.PALETTE, oracle.HUFFMAN])
def test_random_bit_patterns_round_trip(codec):
    w = synth.random_bits((96, 320), seed=7)
    assert np.array_equal(oracle.decode(oracle.encode(w, codec, chunk=192, max_len=12)), w)
