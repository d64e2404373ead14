"""Pins for the oracle's length-limited Huffman code (package-merge) and the
canonical code assignment.  Cloudflare blog "Unweight": the paragraph on
Huffman-coding only the exponent byte; length limit and canonical order are
the pinned readings stated in ``oracle/uw_oracle.c``.
"""
import heapq
import itertools
import math
import os
import random

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def cost(counts, lens):
    return sum(c * l for c, l in zip(counts, lens))


def kraft(lens):
    return sum(2.0 ** -l for l in lens if l)


def huffman_cost_heap(counts):
    """Textbook Huffman (repeatedly merge the two lightest): total cost = sum of merge weights."""
    h = [c for c in counts if c]
    if len(h) == 1:
        return h[0]
    heapq.heapify(h)
    total = 0
    while len(h) > 1:
        a, b = heapq.heappop(h), heapq.heappop(h)
        total += a + b
        heapq.heappush(h, a + b)
    return total


def test_rfc1951_worked_example():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "rfc1951_canonical_example.txt")) if not l.startswith("#")]
    lens = [int(r[1]) for r in rows]
    codes = oracle.canonical_codes(lens)
    for r, c, l in zip(rows, codes, lens):
        assert format(c, f"0{l}b") == r[2], r


def test_hand_worked_package_merge_tie_rule():
    for line in open(os.path.join(GOLDEN, "package_merge_ties.txt")):
        if line.startswith("#") or not line.strip():
            continue
        L, counts, lens = [p.split() for p in line.split("|")]
        assert oracle.huffman_lengths([int(c) for c in counts], int(L[0])) == [int(v) for v in lens]


def test_bruteforce_optimal_small_alphabets():
    rng = random.Random(1234)
    for trial in range(300):
        n = rng.randint(2, 6)
        L = rng.randint(max(1, math.ceil(math.log2(n))), 5)
        counts = [rng.choice([0, 1, 1, 2, 3, 5, 8, 13, 50, 400]) for _ in range(n)]
        used = [i for i, c in enumerate(counts) if c]
        lens = oracle.huffman_lengths(counts, L)
        if len(used) == 0:
            assert lens == [0] * n
            continue
        if len(used) == 1:
            assert lens == [1 if c else 0 for c in counts]
            continue
        assert all((l == 0) == (c == 0) for l, c in zip(lens, counts))
        assert max(lens) <= L and kraft(lens) == 1.0
        best = min(cost([counts[i] for i in used], v)
                   for v in itertools.product(range(1, L + 1), repeat=len(used))
                   if sum(2.0 ** -x for x in v) <= 1.0)
        assert cost(counts, lens) == best, (counts, L, lens)


def test_unlimited_equals_heap_huffman_and_entropy_bound():
    rng = random.Random(99)
    for trial in range(200):
        n = rng.randint(2, 16)
        counts = [rng.randint(0, 1000) for _ in range(n)]
        if sum(1 for c in counts if c) < 2:
            continue
        lens = oracle.huffman_lengths(counts, 15)
        if max(lens) < 15:  # limit not binding -> plain Huffman cost
            assert cost(counts, lens) == huffman_cost_heap(counts)
        tot = sum(counts)
        H = -sum(c / tot * math.log2(c / tot) for c in counts if c)
        avg = cost(counts, lens) / tot
        assert H - 1e-12 <= avg < H + 1, (counts, lens)
        assert kraft(lens) == 1.0


def test_length_limit_binds_and_stays_optimal_on_geometric_counts():
    counts = [2 ** i for i in range(16)]           # unlimited Huffman would need 15 bits
    for L in (4, 6, 8, 12):
        lens = oracle.huffman_lengths(counts, L)
        assert max(lens) <= L and kraft(lens) == 1.0
    assert max(oracle.huffman_lengths(counts, 15)) == 15


def test_canonical_codes_prefix_free_and_ordered():
    rng = random.Random(5)
    for _ in range(100):
        counts = [rng.randint(0, 50) for _ in range(16)]
        lens = oracle.huffman_lengths(counts, 12)
        codes = oracle.canonical_codes(lens)
        words = [format(c, f"0{l}b") for c, l in zip(codes, lens) if l]
        for a, b in itertools.permutations(words, 2):
            assert not b.startswith(a)
        # canonical order: sorting by (length, symbol) gives increasing code values
        # once each code is left-aligned to 15 bits
        keyed = sorted((l, s, c << (15 - l)) for s, (c, l) in enumerate(zip(codes, lens)) if l)
        vals = [v for _, _, v in keyed]
        assert vals == sorted(vals)


def test_entropy_coding_on_gaussian_exponents():
    # Coded size within 1 bit/symbol of the exponent stream's Shannon entropy.
    w = synth.fill((512, 4096), seed=11, scale=0.02)
    blob = oracle.encode(w, oracle.HUFFMAN, chunk=256, max_len=12)
    h = oracle.parse_header(blob)
    counts, pal = oracle.palette(w)
    _, e = oracle.split(w)
    bm = np.frombuffer(oracle.section(blob, "bitmap"), np.uint32)
    blk = np.arange(h["n_blocks"])
    verb = ((bm[blk // 32] >> (blk % 32)) & 1).astype(bool)
    e_nv = e.reshape(-1, 64)[~verb].ravel()
    c = np.bincount(e_nv, minlength=256).astype(np.float64)
    p = c[c > 0] / c.sum()
    H = float(-(p * np.log2(p)).sum())
    avg = h["total_bits"] / e_nv.size
    assert H <= avg < H + 1.0
