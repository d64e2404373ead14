"""The benchmark's roofline accounting, on the CPU: the algorithmic bytes a pass must move are the blob sections
that the strategy's kernels read (sizes taken from the oracle's own blob header, the Huffman stream at byte
precision) plus X and Y, and the kernel names and launch counts follow the plans."""
import os
import sys

import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import lossless_bf16_weight_exponent_gb300 as uw  # noqa: E402


@pytest.mark.parametrize("B", [1, 4, 16])
def test_algorithmic_bytes_are_the_sections_each_strategy_reads(B):
    w = synth.tiny().weights()
    N, K = w.shape
    hp = oracle.parse_header(oracle.encode(w, oracle.PALETTE))
    hh = oracle.parse_header(oracle.encode(w, oracle.HUFFMAN))
    xy = 2 * B * K + 4 * B * N
    sec = lambda h, name: h["sections"][name][1]
    # direct palette: sign+mantissa bytes, 4-bit codes, verbatim exponents, verbatim bitmap and its prefix
    pal_read = sec(hp, "sm") + sec(hp, "idx") + sec(hp, "verb_exp") + sec(hp, "bitmap") + sec(hp, "prefix")
    assert bench.algorithmic_bytes(hp, 4, B) == pal_read + xy
    # Huffman-fed pipelines: the stream (to the byte) and its chunk offsets instead of the codes
    huf_read = (sec(hh, "sm") + (hh["total_bits"] + 7) // 8 + sec(hh, "chunk_off") + sec(hh, "verb_exp")
                + sec(hh, "bitmap") + sec(hh, "prefix"))
    for s in (1, 2, 3, 5):
        assert bench.algorithmic_bytes(hh, s, B) == huf_read + xy
    # the stream section is padded to whole 32-bit words only
    assert 0 <= sec(hh, "bits") - (hh["total_bits"] + 7) // 8 < 4


@pytest.mark.parametrize("plan,B,name,launches", [
    ((4, 1, 0, 4), 1, "gemv_tma_kernel", 1),
    ((4, 1, 0, 8), 4, "gemv_rp_kernel", 2),      # the zeroing kernel, then the GEMV
    ((4, 1, 0, 6), 8, "gemv_mma_kernel", 1),
    ((4, 2, 0, 4), 256, "tc4_kernel", 2),
    ((4, 2, 0, 0), 256, "tc_kernel", 1),
    ((3, 1, 0, 4), 1, "gemv_tma_kernel", 2),     # the palette transcode, then the GEMV
    ((5, 1, 0, 0), 1, "gemv_huff_kernel", 2),    # the zeroing kernel, then the Huffman-direct GEMV
    ((1, 1, 0, 1), 1, "gemv_kernel", 2),
])
def test_kernel_names_and_launches(plan, B, name, launches):
    p = uw.Plan(*plan)
    assert bench.kernel_name(p, B) == name
    assert bench.launches_per_call(p, B) == launches
