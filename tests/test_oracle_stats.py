"""Cross-checks of the oracle's codec against the statistics the Unweight post
states (Cloudflare blog "Unweight": exponent-statistics paragraph - the top-16
exponents cover >99% of a layer's weights and the exponent entropy is at most
about 2.6 bits; opening results paragraph - about 30% compression of MLP weights
with Huffman coding) on the synthetic Gaussian stand-ins for trained layers.
"""
import numpy as np

import oracle
import synth


def _sample(scale=0.02, kind=synth.NORMAL, p1=1e-4, f1=100.0):
    return synth.fill((512, 4096), seed=synth.SEED_BASE + 1, kind=kind, scale=scale, p1=p1, f1=f1)


def test_top16_coverage_and_entropy_gaussian():
    counts, pal = oracle.palette(_sample())
    c = counts.astype(np.float64)
    cover = c[pal].sum() / c.sum()
    p = c[c > 0] / c.sum()
    H = float(-(p * np.log2(p)).sum())
    assert cover > 0.99
    assert H <= 2.6


def test_compression_ratios_gaussian():
    w = _sample()
    raw = 2 * w.size
    huff = len(oracle.encode(w, oracle.HUFFMAN))
    pal = len(oracle.encode(w, oracle.PALETTE))
    # Huffman: about 30% smaller than raw BF16 (post); palette: 4 bits instead of 8
    # for the exponent -> about 25% smaller minus the verbatim overhead.
    assert 0.25 <= 1 - huff / raw <= 0.40
    assert 0.20 <= 1 - pal / raw <= 0.25
    assert huff < pal


def test_heavy_tail_has_more_verbatim_blocks():
    g = oracle.parse_header(oracle.encode(_sample(p1=0.0)))
    t = oracle.parse_header(oracle.encode(_sample(kind=synth.STUDENT_T3, p1=0.0)))
    assert t["n_verbatim"] / t["n_blocks"] > g["n_verbatim"] / g["n_blocks"]
