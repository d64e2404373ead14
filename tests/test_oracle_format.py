"""Hand-worked blobs: every expected byte below was derived by hand from the
format rules in ``oracle/uw_oracle.c`` (palette by count, 64-weight verbatim
blocks, low-nibble-first codes, package-merge + canonical Huffman, MSB-first bit
string).  Cloudflare blog "Unweight": exponent statistics, verbatim-row and
direct-palette paragraphs.
"""
import struct

import numpy as np

import oracle


def bf16(sign, exp, mant):
    return (sign << 15) | (exp << 7) | mant


def u32s(b):
    return list(struct.unpack(f"<{len(b) // 4}I", b))


def test_1x64_single_exponent_palette():
    # 64 weights, all exponent 0x7F (values in [1,2)), mantissa j, sign j&1.
    w = np.array([[bf16(j & 1, 0x7F, j) for j in range(64)]], np.uint16)
    blob = oracle.encode(w, oracle.PALETTE)
    h = oracle.parse_header(blob)
    assert (h["N"], h["K"], h["codec"], h["block"], h["chunk"], h["max_len"]) == (1, 64, 0, 64, 0, 0)
    assert h["n_pal"] == 1 and h["palette"] == [0x7F] + [0] * 15 and h["code_len"] == [0] * 16
    assert (h["n_blocks"], h["n_verbatim"], h["n_chunks"], h["total_bits"]) == (1, 0, 0, 0)
    # sections: SM 64 B at 256; bitmap 4 B at 512; prefix 4 B at 768; verb 0 B at 1024;
    # idx 32 B at 1024; chunk 0 B at 1280; bits 0 B at 1280; total 1280.
    assert h["sections"] == {"sm": (256, 64), "bitmap": (512, 4), "prefix": (768, 4), "verb_exp": (1024, 0),
                             "idx": (1024, 32), "chunk_off": (1280, 0), "bits": (1280, 0)}
    assert h["blob_bytes"] == 1280 == len(blob)
    assert oracle.section(blob, "sm") == bytes(((j & 1) << 7) | j for j in range(64))
    assert oracle.section(blob, "idx") == bytes(32)
    assert blob[256 + 64:512] == bytes(512 - 320)  # zero padding


def test_1x64_single_exponent_huffman():
    w = np.array([[bf16(0, 0x7F, j) for j in range(64)]], np.uint16)
    blob = oracle.encode(w, oracle.HUFFMAN, chunk=64, max_len=12)
    h = oracle.parse_header(blob)
    # one used symbol -> length 1, code "0"; 64 bits of zeros in 2 words; 1 chunk
    assert h["code_len"] == [1] + [0] * 15 and h["total_bits"] == 64 and h["n_chunks"] == 1
    assert u32s(oracle.section(blob, "chunk_off")) == [0, 64]
    assert oracle.section(blob, "bits") == bytes(8)
    assert oracle.section(blob, "idx") == b""
    assert np.array_equal(oracle.decode(blob), w)


def test_2x128_four_exponents_codes_by_hand():
    # Exponents: 100 weights of 0x7A, 80 of 0x79, 70 of 0x78 (the palette, 3 values),
    # laid out so that block 2 (row 1, k 0..63) holds one 0x50 -> verbatim.
    # Block layout (row, k-range): b0=(0,0..63) b1=(0,64..127) b2=(1,0..63) b3=(1,64..127).
    e = np.empty((2, 128), np.uint8)
    e[0, :64] = 0x7A                       # b0: 64 x 0x7A
    e[0, 64:100] = 0x7A                    # b1: 36 x 0x7A, 28 x 0x79
    e[0, 100:] = 0x79
    e[1, :64] = 0x78                       # b2: 63 x 0x78 + one 0x50
    e[1, 10] = 0x50
    e[1, 64:116] = 0x79                    # b3: 52 x 0x79, 12 x 0x78 ... adjust counts below
    e[1, 116:] = 0x78
    sm = (np.arange(256, dtype=np.uint32) * 37 % 256).astype(np.uint8).reshape(2, 128)
    w = ((sm.astype(np.uint16) & 0x80) << 8) | (e.astype(np.uint16) << 7) | (sm & 0x7F)
    # counts over the whole matrix: 0x7A: 64+36=100, 0x79: 28+52=80, 0x78: 63+12=75, 0x50: 1
    # -> palette [0x7A, 0x79, 0x78, 0x50] (4 distinct values, all in the palette!)
    # so no block is verbatim with only 4 exponents; the palette holds every value.
    blob = oracle.encode(w.astype(np.uint16), oracle.PALETTE)
    h = oracle.parse_header(blob)
    assert h["palette"][:4] == [0x7A, 0x79, 0x78, 0x50] and h["n_pal"] == 4 and h["n_verbatim"] == 0
    idx = oracle.section(blob, "idx")
    # row 1, k=10 -> code 3 in the low nibble of byte 64+5; k=11 (0x78, code 2) high nibble
    assert idx[64 + 5] == 0x23
    # row 0, k=0,1 -> 0x7A code 0 twice; row 0 k=100,101 -> 0x79 code 1 twice
    assert idx[0] == 0x00 and idx[50] == 0x11
    assert np.array_equal(oracle.decode(blob), w)


def test_17_exponents_forces_one_verbatim_block():
    # 16 exponents 0x70..0x7F fill every block with 4 copies each (64 weights);
    # block 3 (row 1, k 64..127) additionally swaps one weight to exponent 0x20,
    # the 17th value, which has the lowest count -> outside the palette -> verbatim.
    e = np.tile(np.repeat(np.arange(0x70, 0x80, dtype=np.uint8), 4), 4).reshape(2, 128)
    e[1, 64] = 0x20
    sm = np.full((2, 128), 0x05, np.uint8)
    w = ((e.astype(np.uint16)) << 7) | 0x05
    blob = oracle.encode(w.astype(np.uint16), oracle.PALETTE)
    h = oracle.parse_header(blob)
    # counts: 0x70 -> 15 (one copy replaced), 0x71..0x7F -> 16 each, 0x20 -> 1.
    # Order: 0x71..0x7F (16 each, ascending), then 0x70 (15); 0x20 is 17th -> dropped.
    assert h["palette"] == list(range(0x71, 0x80)) + [0x70]
    assert h["n_verbatim"] == 1
    assert u32s(oracle.section(blob, "bitmap")) == [0b1000]
    assert u32s(oracle.section(blob, "prefix")) == [0]
    assert oracle.section(blob, "verb_exp") == bytes(e[1, 64:128])
    idx = np.frombuffer(oracle.section(blob, "idx"), np.uint8).reshape(2, 64)
    assert (idx[1, 32:] == 0).all()                 # verbatim block's codes are zero
    # row 0, k=0..3 exponent 0x70 -> code 15; k=4 -> 0x71 -> code 0
    assert idx[0, 0] == 0xFF and idx[0, 1] == 0xFF and idx[0, 2] == 0x00
    assert np.array_equal(oracle.decode(blob), w)
    # Huffman: symbol counts over the 3 non-verbatim blocks: code 15 (0x70) -> 12,
    # codes 0..14 -> 12 each, i.e. 16 equal counts -> every length is 4; canonical codes
    # are then the symbol numbers themselves.  Weight i (flat, non-verbatim) emits its
    # 4-bit palette index MSB-first, so each 32-bit word holds 8 consecutive codes.
    hb = oracle.encode(w.astype(np.uint16), oracle.HUFFMAN, chunk=128, max_len=12)
    hh = oracle.parse_header(hb)
    assert hh["code_len"] == [4] * 16 and hh["total_bits"] == 192 * 4 and hh["n_chunks"] == 2
    assert u32s(oracle.section(hb, "chunk_off")) == [0, 512, 768]
    words = u32s(oracle.section(hb, "bits"))
    # first 8 weights: exps 0x70 x4, 0x71 x4 -> codes 15,15,15,15,0,0,0,0
    assert words[0] == 0xFFFF0000
    assert np.array_equal(oracle.decode(hb), w)


def test_empty_and_bad_shapes():
    w = np.zeros((0, 64), np.uint16)
    for codec in (oracle.PALETTE, oracle.HUFFMAN):
        blob = oracle.encode(w, codec)
        h = oracle.parse_header(blob)
        # palette: header only; Huffman: one chunk offset word (n_chunks + 1 = 1) at 256
        assert h["n_blocks"] == 0 and h["n_pal"] == 0 and len(blob) == (256 if codec == oracle.PALETTE else 512)
        assert oracle.decode(blob).shape == (0, 64)
    try:
        oracle.encode(np.zeros((2, 65), np.uint16))
        raise AssertionError("K % 64 != 0 must be rejected")
    except oracle.OracleError:
        pass


def test_verbatim_invariants_on_tiny_config():
    import synth
    w = synth.tiny().weights()
    for codec in (oracle.PALETTE, oracle.HUFFMAN):
        blob = oracle.encode(w, codec)
        h = oracle.parse_header(blob)
        bm = np.frombuffer(oracle.section(blob, "bitmap"), np.uint32)
        pf = np.frombuffer(oracle.section(blob, "prefix"), np.uint32)
        pc = np.array([bin(int(v)).count("1") for v in bm])
        assert pf[-1] + pc[-1] == h["n_verbatim"]
        assert np.array_equal(pf[1:], np.cumsum(pc)[:-1])
        _, e = oracle.split(w)
        blk = np.arange(h["n_blocks"])
        verb = ((bm[blk // 32] >> (blk % 32)) & 1).astype(bool)
        pal = set(h["palette"][:h["n_pal"]])
        eb = e.reshape(-1, 64)
        assert all(set(row.tolist()) <= pal for row in eb[~verb])
        assert all(not set(row.tolist()) <= pal for row in eb[verb])
        if codec == oracle.HUFFMAN:
            off = np.frombuffer(oracle.section(blob, "chunk_off"), np.uint32)
            assert (np.diff(off.astype(np.int64)) >= 0).all() and off[-1] == h["total_bits"]
