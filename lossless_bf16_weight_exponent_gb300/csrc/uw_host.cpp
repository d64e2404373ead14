// uw_host.cpp - host side of the codec: encoder, blob validation, code tables, errors.
//
// Method: Cloudflare blog "Unweight".  The BF16 anatomy paragraphs give the
// field split (sign+mantissa kept raw, exponent coded); the exponent-statistics
// paragraph gives the top-16 palette; the Huffman paragraph gives entropy
// coding of the exponent byte; the rare-exponent paragraph gives verbatim
// 64-weight runs.  The blob layout is this library's (header of 256 bytes,
// sections SM, BITMAP, PREFIX, VERB_EXP, IDX, CHUNK_OFF, BITS, each on a
// 256-byte boundary, zero gaps); it is byte-for-byte reproducible.
#include <algorithm>
#include <array>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "uw_internal.h"

namespace uw {

static thread_local char g_err[512];

uw_status fail(uw_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

void clear_error() { g_err[0] = 0; }

static inline uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

static inline void wr32(uint8_t *p, uint32_t v) { memcpy(p, &v, 4); }
static inline void wr64(uint8_t *p, uint64_t v) { memcpy(p, &v, 8); }
static inline uint32_t rd32(const uint8_t *p) { uint32_t v; memcpy(&v, p, 4); return v; }
static inline uint64_t rd64(const uint8_t *p) { uint64_t v; memcpy(&v, p, 8); return v; }

static bool little_endian()
{
    const uint16_t one = 1;
    uint8_t b;
    memcpy(&b, &one, 1);
    return b == 1;
}

// ------------------------------------------------------------------------------ code lengths
// Length-limited prefix code by package-merge (Larmore & Hirschberg 1990).  Each
// level's list holds leaves and packages; a package remembers its two children in
// the previous level's list.  A symbol's length is the number of times its leaf is
// reached from the first 2(n-1) entries of the last list.  Ordering rules: leaves
// by (count, symbol); when merging, a package goes before a leaf of equal weight.
namespace {
struct Node {
    uint64_t weight;
    int32_t sym;      // >= 0 leaf
    int32_t a, b;     // children (indices into the previous level) for packages
};
}  // namespace

static int package_merge(const uint64_t *counts, int max_len, uint8_t *lens)
{
    for (int s = 0; s < 16; s++) lens[s] = 0;
    std::vector<Node> leaves;
    for (int s = 0; s < 16; s++)
        if (counts[s]) leaves.push_back(Node{counts[s], s, -1, -1});
    const int n = (int)leaves.size();
    if (n == 0) return 0;
    if (n == 1) { lens[leaves[0].sym] = 1; return 0; }
    if ((1 << max_len) < n) return -1;
    std::stable_sort(leaves.begin(), leaves.end(),
                     [](const Node &x, const Node &y) { return x.weight < y.weight; });
    std::vector<std::vector<Node>> level;
    level.push_back(leaves);
    for (int d = 1; d < max_len; d++) {
        const std::vector<Node> &prev = level.back();
        std::vector<Node> cur;
        cur.reserve(leaves.size() + prev.size() / 2);
        size_t li = 0, pi = 0, npk = prev.size() / 2;
        while (li < leaves.size() || pi < npk) {
            bool take_pkg = false;
            if (pi < npk) {
                uint64_t pw = prev[2 * pi].weight + prev[2 * pi + 1].weight;
                take_pkg = li >= leaves.size() || pw <= leaves[li].weight;
                if (take_pkg) { cur.push_back(Node{pw, -1, (int32_t)(2 * pi), (int32_t)(2 * pi + 1)}); pi++; }
            }
            if (!take_pkg) cur.push_back(leaves[li++]);
        }
        level.push_back(std::move(cur));
    }
    // walk from the last list down: hits[d][i] = how many times entry i of level d is used
    int L = (int)level.size();
    std::vector<std::vector<uint32_t>> hits(L);
    for (int d = 0; d < L; d++) hits[d].assign(level[d].size(), 0);
    for (int i = 0; i < 2 * (n - 1); i++) hits[L - 1][i] = 1;
    for (int d = L - 1; d >= 0; d--) {
        for (size_t i = 0; i < level[d].size(); i++) {
            if (!hits[d][i]) continue;
            const Node &nd = level[d][i];
            if (nd.sym >= 0) lens[nd.sym] = (uint8_t)(lens[nd.sym] + hits[d][i]);
            else { hits[d - 1][nd.a] += hits[d][i]; hits[d - 1][nd.b] += hits[d][i]; }
        }
    }
    return 0;
}

// Canonical code values (RFC 1951 section 3.2.2 ordering: by length, then symbol).
void canonical_codes(const uint8_t *lens, uint32_t *codes)
{
    std::array<std::pair<int, int>, 16> order;
    int m = 0;
    for (int s = 0; s < 16; s++) { codes[s] = 0; if (lens[s]) order[m++] = {lens[s], s}; }
    std::sort(order.begin(), order.begin() + m);
    uint32_t code = 0;
    int prev = m ? order[0].first : 0;
    for (int i = 0; i < m; i++) {
        code <<= (order[i].first - prev);
        prev = order[i].first;
        codes[order[i].second] = code++;
    }
}

void build_decode_table(const uint8_t *lens, int max_len, std::vector<uint8_t> &table)
{
    uint32_t codes[16];
    canonical_codes(lens, codes);
    table.assign((size_t)1 << max_len, 0);
    for (int s = 0; s < 16; s++) {
        if (!lens[s]) continue;
        int fill = max_len - lens[s];
        uint32_t first = codes[s] << fill;
        for (uint32_t v = 0; v < (1u << fill); v++) table[first + v] = (uint8_t)((s << 4) | lens[s]);
    }
}

// Multi-symbol decode table for limits <= 12: entry v (the next 12 bits of the stream) packs
//   bits 0-3   total length of the whole codes it holds (<= 12)
//   bits 4-6   how many whole codes start in v (1..5)
//   bits 7-10  length of the first code
//   bits 11-30 the codes' symbols, 4 bits each, first symbol lowest
// 0 where no code matches v's prefix.
void build_multi_table(const uint8_t *lens, std::vector<uint32_t> &table)
{
    std::vector<uint8_t> single;
    build_decode_table(lens, 12, single);  // (symbol << 4) | length over 12-bit prefixes
    table.assign(4096, 0);
    for (uint32_t v = 0; v < 4096; v++) {
        uint32_t used = 0, n = 0, first = 0, syms = 0;
        while (n < 5) {
            const uint32_t peek = (v << used) & 0xFFFu;  // next 12 bits, zero-filled past v's end
            const uint8_t e = single[peek];
            const uint32_t len = e & 15u;
            if (!len || used + len > 12) break;
            if (n == 0) first = len;
            syms |= (uint32_t)(e >> 4) << (4 * n);
            used += len;
            n++;
        }
        if (n) table[v] = used | (n << 4) | (first << 7) | (syms << 11);
    }
}

// ------------------------------------------------------------------------------ layout
static void layout(const BlobHeader &h, uint64_t *off, uint64_t *len, uint64_t *total)
{
    const uint64_t n = (uint64_t)h.N * (uint64_t)h.K;
    const uint64_t words = (h.n_blocks + 31) / 32;
    len[S_SM] = n;
    len[S_BITMAP] = 4 * words;
    len[S_PREFIX] = 4 * words;
    len[S_VERB] = 64 * h.n_verbatim;
    len[S_IDX] = h.codec == UW_CODEC_PALETTE ? n / 2 : 0;
    len[S_CHUNK] = h.codec == UW_CODEC_HUFFMAN ? 4 * (h.n_chunks + 1) : 0;
    len[S_BITS] = h.codec == UW_CODEC_HUFFMAN ? 4 * ((h.total_bits + 31) / 32) : 0;
    uint64_t pos = kAlign;
    for (int s = 0; s < S_COUNT; s++) { off[s] = pos; pos = round_up(pos + len[s], kAlign); }
    *total = pos;
}

}  // namespace uw

using namespace uw;

// ------------------------------------------------------------------------------ uw_encode
extern "C" uw_status uw_encode(const uint16_t *w, int64_t N, int64_t K, const uw_encode_opts *opts, void *out,
                               size_t out_cap, size_t *out_size)
{
    clear_error();
    if (!out_size) return fail(UW_ERR_INVALID_ARG, "uw_encode: out_size is NULL");
    if (!little_endian()) return fail(UW_ERR_UNSUPPORTED, "uw_encode: big-endian host");
    if (N < 0 || K < 0 || K % kBlock) return fail(UW_ERR_SHAPE, "uw_encode: need N >= 0, K >= 0, K %% 64 == 0 (N=%lld K=%lld)",
                                                  (long long)N, (long long)K);
    if (N > ((int64_t)1 << 40) || K > ((int64_t)1 << 40) || (N && K > (((int64_t)1 << 62) / N)))
        return fail(UW_ERR_SHAPE, "uw_encode: N*K too large");
    uw_encode_opts o = opts ? *opts : uw_encode_opts{UW_CODEC_PALETTE, 256, 12};
    if (o.codec != UW_CODEC_PALETTE && o.codec != UW_CODEC_HUFFMAN) return fail(UW_ERR_INVALID_ARG, "uw_encode: bad codec");
    if (o.codec == UW_CODEC_HUFFMAN &&
        (o.chunk_weights < 64 || o.chunk_weights % 64 || o.max_code_len < 4 || o.max_code_len > 15))
        return fail(UW_ERR_INVALID_ARG, "uw_encode: chunk_weights must be a multiple of 64, max_code_len in 4..15");
    if (N * K && !w) return fail(UW_ERR_INVALID_ARG, "uw_encode: weights are NULL");

    const uint64_t n = (uint64_t)N * (uint64_t)K;
    BlobHeader h;
    h.N = N; h.K = K; h.codec = o.codec; h.block = 64;
    h.chunk = o.codec == UW_CODEC_HUFFMAN ? o.chunk_weights : 0;
    h.max_len = o.codec == UW_CODEC_HUFFMAN ? o.max_code_len : 0;
    h.n_blocks = n / 64;

    // exponent histogram (four interleaved partial counts)
    std::vector<uint64_t> part(4 * 256, 0);
    uint64_t i = 0;
    for (; i + 4 <= n; i += 4)
        for (int j = 0; j < 4; j++) part[j * 256 + ((w[i + j] >> 7) & 0xFF)]++;
    for (; i < n; i++) part[(w[i] >> 7) & 0xFF]++;
    std::array<uint64_t, 256> hist{};
    for (int e = 0; e < 256; e++) hist[e] = part[e] + part[256 + e] + part[512 + e] + part[768 + e];

    // palette: present exponents ordered by (count desc, exponent asc), first 16
    std::vector<int> present;
    for (int e = 0; e < 256; e++) if (hist[e]) present.push_back(e);
    std::stable_sort(present.begin(), present.end(), [&](int a, int b) { return hist[a] > hist[b]; });
    h.n_pal = (uint32_t)std::min<size_t>(16, present.size());
    std::array<int16_t, 256> code_of;
    code_of.fill(-1);
    for (uint32_t c = 0; c < h.n_pal; c++) { h.palette[c] = (uint8_t)present[c]; code_of[present[c]] = (int16_t)c; }

    // verbatim blocks: any exponent without a palette code
    const uint64_t words = (h.n_blocks + 31) / 32;
    std::vector<uint32_t> bitmap(words, 0);
    for (uint64_t b = 0; b < h.n_blocks; b++) {
        const uint16_t *p = w + b * 64;
        int miss = 0;
        for (int j = 0; j < 64; j++) miss |= code_of[(p[j] >> 7) & 0xFF] < 0;
        if (miss) { bitmap[b >> 5] |= 1u << (b & 31); h.n_verbatim++; }
    }
    auto is_verb = [&](uint64_t b) { return (bitmap[b >> 5] >> (b & 31)) & 1u; };

    // Huffman code over palette codes of non-verbatim blocks
    uint32_t codes[16] = {0};
    if (h.codec == UW_CODEC_HUFFMAN) {
        uint64_t sym[16] = {0};
        for (uint64_t b = 0; b < h.n_blocks; b++) {
            if (is_verb(b)) continue;
            const uint16_t *p = w + b * 64;
            for (int j = 0; j < 64; j++) sym[code_of[(p[j] >> 7) & 0xFF]]++;
        }
        if (package_merge(sym, (int)h.max_len, h.code_len)) return fail(UW_ERR_INVALID_ARG, "uw_encode: length limit too small");
        canonical_codes(h.code_len, codes);
        for (int s = 0; s < 16; s++) h.total_bits += sym[s] * h.code_len[s];
        if (h.total_bits >= ((uint64_t)1 << 32)) return fail(UW_ERR_UNSUPPORTED, "uw_encode: Huffman stream >= 2^32 bits");
        h.n_chunks = (n + h.chunk - 1) / h.chunk;
    }

    uint64_t total;
    layout(h, h.off, h.len, &total);
    h.blob_bytes = total;
    *out_size = (size_t)total;
    if (!out) return UW_OK;
    if (out_cap < total) return fail(UW_ERR_BUFFER_TOO_SMALL, "uw_encode: need %llu bytes", (unsigned long long)total);
    uint8_t *o8 = (uint8_t *)out;
    memset(o8, 0, total);

    memcpy(o8, "UWB1", 4);
    wr32(o8 + 4, 1);
    wr64(o8 + 8, (uint64_t)N);
    wr64(o8 + 16, (uint64_t)K);
    wr32(o8 + 24, h.codec);
    wr32(o8 + 28, 64);
    wr32(o8 + 32, h.chunk);
    wr32(o8 + 36, h.max_len);
    o8[40] = (uint8_t)h.n_pal;
    memcpy(o8 + 41, h.palette, 16);
    memcpy(o8 + 57, h.code_len, 16);
    wr64(o8 + 80, h.n_blocks);
    wr64(o8 + 88, h.n_verbatim);
    wr64(o8 + 96, h.n_chunks);
    wr64(o8 + 104, h.total_bits);
    wr64(o8 + 112, total);
    for (int s = 0; s < S_COUNT; s++) { wr64(o8 + 128 + 16 * s, h.off[s]); wr64(o8 + 136 + 16 * s, h.len[s]); }

    uint8_t *sm = o8 + h.off[S_SM];
    for (uint64_t k = 0; k < n; k++) sm[k] = (uint8_t)(((w[k] >> 8) & 0x80) | (w[k] & 0x7F));

    uint32_t run = 0;
    for (uint64_t k = 0; k < words; k++) {
        wr32(o8 + h.off[S_BITMAP] + 4 * k, bitmap[k]);
        wr32(o8 + h.off[S_PREFIX] + 4 * k, run);
        run += (uint32_t)__builtin_popcount(bitmap[k]);
    }
    uint8_t *ve = o8 + h.off[S_VERB];
    for (uint64_t b = 0; b < h.n_blocks; b++) {
        if (!is_verb(b)) continue;
        for (int j = 0; j < 64; j++) *ve++ = (uint8_t)((w[b * 64 + j] >> 7) & 0xFF);
    }

    if (h.codec == UW_CODEC_PALETTE) {
        uint8_t *idx = o8 + h.off[S_IDX];
        for (uint64_t b = 0; b < h.n_blocks; b++) {
            if (is_verb(b)) continue;  // codes stay 0
            const uint16_t *p = w + b * 64;
            uint8_t *q = idx + b * 32;
            for (int j = 0; j < 32; j++)
                q[j] = (uint8_t)(code_of[(p[2 * j] >> 7) & 0xFF] | (code_of[(p[2 * j + 1] >> 7) & 0xFF] << 4));
        }
    } else {
        uint8_t *co = o8 + h.off[S_CHUNK];
        uint8_t *bits = o8 + h.off[S_BITS];
        uint64_t acc = 0;        // pending bits, right-aligned
        int nacc = 0;
        uint64_t pos = 0, word = 0;
        const uint64_t blocks_per_chunk = h.chunk / 64;
        for (uint64_t c = 0; c < h.n_chunks; c++) {
            wr32(co + 4 * c, (uint32_t)pos);
            uint64_t b0 = c * blocks_per_chunk, b1 = std::min(h.n_blocks, b0 + blocks_per_chunk);
            for (uint64_t b = b0; b < b1; b++) {
                if (is_verb(b)) continue;
                const uint16_t *p = w + b * 64;
                for (int j = 0; j < 64; j++) {
                    int s = code_of[(p[j] >> 7) & 0xFF];
                    acc = (acc << h.code_len[s]) | codes[s];
                    nacc += h.code_len[s];
                    pos += h.code_len[s];
                    if (nacc >= 32) {
                        nacc -= 32;
                        wr32(bits + 4 * word++, (uint32_t)(acc >> nacc));
                        acc &= (nacc ? ((1ull << nacc) - 1) : 0);
                    }
                }
            }
        }
        if (nacc) wr32(bits + 4 * word++, (uint32_t)(acc << (32 - nacc)));
        wr32(co + 4 * h.n_chunks, (uint32_t)pos);
    }
    return UW_OK;
}

// ------------------------------------------------------------------------------ validation
namespace uw {

uw_status parse_and_validate(const uint8_t *p, size_t size, BlobHeader *out, bool deep)
{
    if (!p) return fail(UW_ERR_INVALID_ARG, "blob is NULL");
    if (size < 256) return fail(UW_ERR_CORRUPT, "blob shorter than its header");
    if (memcmp(p, "UWB1", 4) != 0) return fail(UW_ERR_CORRUPT, "bad magic");
    if (rd32(p + 4) != 1) return fail(UW_ERR_CORRUPT, "unsupported version %u", rd32(p + 4));
    BlobHeader h;
    h.N = (int64_t)rd64(p + 8);
    h.K = (int64_t)rd64(p + 16);
    h.codec = rd32(p + 24);
    h.block = rd32(p + 28);
    h.chunk = rd32(p + 32);
    h.max_len = rd32(p + 36);
    h.n_pal = p[40];
    memcpy(h.palette, p + 41, 16);
    memcpy(h.code_len, p + 57, 16);
    h.n_blocks = rd64(p + 80);
    h.n_verbatim = rd64(p + 88);
    h.n_chunks = rd64(p + 96);
    h.total_bits = rd64(p + 104);
    h.blob_bytes = rd64(p + 112);
    if (h.N < 0 || h.K < 0 || h.K % 64 || h.N > ((int64_t)1 << 40) || h.K > ((int64_t)1 << 40) ||
        (h.N && h.K > (((int64_t)1 << 62) / h.N)))
        return fail(UW_ERR_CORRUPT, "bad shape N=%lld K=%lld", (long long)h.N, (long long)h.K);
    if (h.block != 64) return fail(UW_ERR_CORRUPT, "block size %u != 64", h.block);
    const uint64_t n = (uint64_t)h.N * (uint64_t)h.K;
    if (h.n_blocks != n / 64) return fail(UW_ERR_CORRUPT, "n_blocks mismatch");
    if (h.n_pal > 16) return fail(UW_ERR_CORRUPT, "n_pal > 16");
    if (h.n_verbatim > h.n_blocks) return fail(UW_ERR_CORRUPT, "n_verbatim > n_blocks");
    if ((n > 0) != (h.n_pal > 0)) return fail(UW_ERR_CORRUPT, "palette size inconsistent with matrix size");
    for (uint32_t i = h.n_pal; i < 16; i++)
        if (h.palette[i]) return fail(UW_ERR_CORRUPT, "unused palette slot %u not zero", i);
    for (uint32_t i = 0; i < h.n_pal; i++)
        for (uint32_t j = 0; j < i; j++)
            if (h.palette[i] == h.palette[j]) return fail(UW_ERR_CORRUPT, "duplicate palette entry");
    if (h.codec == UW_CODEC_PALETTE) {
        if (h.chunk || h.max_len || h.n_chunks || h.total_bits) return fail(UW_ERR_CORRUPT, "palette blob has Huffman fields");
        for (int s = 0; s < 16; s++) if (h.code_len[s]) return fail(UW_ERR_CORRUPT, "palette blob has code lengths");
    } else if (h.codec == UW_CODEC_HUFFMAN) {
        if (h.chunk < 64 || h.chunk % 64 || h.max_len < 4 || h.max_len > 15) return fail(UW_ERR_CORRUPT, "bad chunk/length limit");
        if (h.n_chunks != (n + h.chunk - 1) / h.chunk) return fail(UW_ERR_CORRUPT, "n_chunks mismatch");
        if (h.total_bits >= ((uint64_t)1 << 32)) return fail(UW_ERR_CORRUPT, "total_bits too large");
        int used = 0;
        uint64_t kraft = 0;  // in units of 2^-15
        for (int s = 0; s < 16; s++) {
            if (!h.code_len[s]) continue;
            if (h.code_len[s] > h.max_len) return fail(UW_ERR_CORRUPT, "code length above the limit");
            if ((uint32_t)s >= h.n_pal) return fail(UW_ERR_CORRUPT, "code for a symbol outside the palette");
            used++;
            kraft += 1ull << (15 - h.code_len[s]);
        }
        if (used == 1 && kraft != (1ull << 14)) return fail(UW_ERR_CORRUPT, "single symbol must have length 1");
        if (used >= 2 && kraft != (1ull << 15)) return fail(UW_ERR_CORRUPT, "code lengths violate Kraft equality");
        if (used == 0 && h.total_bits) return fail(UW_ERR_CORRUPT, "bits without codes");
        if (used && h.total_bits == 0 && h.n_verbatim < h.n_blocks) return fail(UW_ERR_CORRUPT, "codes without bits");
    } else {
        return fail(UW_ERR_CORRUPT, "unknown codec %u", h.codec);
    }
    uint64_t off[S_COUNT], len[S_COUNT], total;
    layout(h, off, len, &total);
    for (int s = 0; s < S_COUNT; s++) {
        h.off[s] = rd64(p + 128 + 16 * s);
        h.len[s] = rd64(p + 136 + 16 * s);
        if (h.off[s] != off[s] || h.len[s] != len[s]) return fail(UW_ERR_CORRUPT, "section %d table mismatch", s);
    }
    if (h.blob_bytes != total || size < total) return fail(UW_ERR_CORRUPT, "blob size %zu, header says %llu (layout %llu)",
                                                           size, (unsigned long long)h.blob_bytes, (unsigned long long)total);
    // verbatim bitmap and its prefix
    const uint64_t words = (h.n_blocks + 31) / 32;
    uint64_t run = 0;
    for (uint64_t k = 0; k < words; k++) {
        uint32_t bm = rd32(p + h.off[S_BITMAP] + 4 * k);
        if (rd32(p + h.off[S_PREFIX] + 4 * k) != run) return fail(UW_ERR_CORRUPT, "verbatim prefix mismatch at word %llu", (unsigned long long)k);
        if (k == words - 1 && (h.n_blocks & 31)) {
            uint32_t valid = (1u << (h.n_blocks & 31)) - 1;
            if (bm & ~valid) return fail(UW_ERR_CORRUPT, "bitmap bits past the last block");
        }
        run += (uint64_t)__builtin_popcount(bm);
    }
    if (run != h.n_verbatim) return fail(UW_ERR_CORRUPT, "verbatim count mismatch");
    if (h.codec == UW_CODEC_HUFFMAN) {
        const uint8_t *co = p + h.off[S_CHUNK];
        uint32_t prev = 0;
        if (rd32(co) != 0) return fail(UW_ERR_CORRUPT, "first chunk offset not 0");
        for (uint64_t c = 1; c <= h.n_chunks; c++) {
            uint32_t v = rd32(co + 4 * c);
            if (v < prev) return fail(UW_ERR_CORRUPT, "chunk offsets decrease at %llu", (unsigned long long)c);
            prev = v;
        }
        if (prev != h.total_bits) return fail(UW_ERR_CORRUPT, "last chunk offset != total_bits");
    }
    if (deep && h.codec == UW_CODEC_PALETTE && n) {
        // every code of a non-verbatim block names a palette slot; verbatim blocks hold zero codes
        const uint8_t *idx = p + h.off[S_IDX];
        const uint8_t *bmp = p + h.off[S_BITMAP];
        for (uint64_t b = 0; b < h.n_blocks; b++) {
            bool verb = (bmp[b >> 3] >> (b & 7)) & 1;
            const uint8_t *q = idx + b * 32;
            if (verb) {
                for (int j = 0; j < 32; j++) if (q[j]) return fail(UW_ERR_CORRUPT, "verbatim block with nonzero codes");
            } else if (h.n_pal < 16) {
                for (int j = 0; j < 32; j++)
                    if ((q[j] & 15) >= h.n_pal || (q[j] >> 4) >= h.n_pal) return fail(UW_ERR_CORRUPT, "code outside the palette");
            }
        }
    }
    *out = h;
    return UW_OK;
}


void build_tile_verbatim(const BlobHeader &h, const uint8_t *blob, std::vector<uint32_t> &off,
                         std::vector<uint32_t> &mask, std::vector<uint8_t> &data)
{
    const int64_t N = h.N, K = h.K, KB = K / 64;
    const int64_t tiles = (N + 127) / 128, upk = K / 256, units = tiles * upk;
    const uint32_t *bm = (const uint32_t *)(blob + h.off[S_BITMAP]);
    const uint32_t *pf = (const uint32_t *)(blob + h.off[S_PREFIX]);
    const uint8_t *ve = blob + h.off[S_VERB];
    off.assign((size_t)units + 1, 0);
    mask.assign((size_t)units * 16, 0);
    data.clear();
    data.reserve((size_t)h.n_verbatim * 64);
    uint32_t cnt = 0;
    for (int64_t t = 0; t < tiles; t++)
        for (int64_t kq = 0; kq < upk; kq++) {
            const int64_t u = t * upk + kq;
            off[(size_t)u] = cnt;
            for (int j = 0; j < 4; j++)
                for (int r = 0; r < 128; r++) {
                    const int64_t row = t * 128 + r;
                    if (row >= N) break;
                    const uint64_t b = (uint64_t)row * (uint64_t)KB + (uint64_t)(kq * 4 + j);
                    const uint32_t w = bm[b >> 5];
                    if (!((w >> (b & 31)) & 1u)) continue;
                    mask[(size_t)u * 16 + 4 * j + (r >> 5)] |= 1u << (r & 31);
                    const uint64_t vi = pf[b >> 5] + (uint64_t)__builtin_popcount(w & ((1u << (b & 31)) - 1u));
                    data.insert(data.end(), ve + vi * 64, ve + vi * 64 + 64);
                    cnt++;
                }
        }
    off[(size_t)units] = cnt;
}

}  // namespace uw

extern "C" const char *uw_status_string(uw_status s)
{
    switch (s) {
    case UW_OK: return "UW_OK";
    case UW_ERR_INVALID_ARG: return "UW_ERR_INVALID_ARG";
    case UW_ERR_SHAPE: return "UW_ERR_SHAPE";
    case UW_ERR_UNSUPPORTED: return "UW_ERR_UNSUPPORTED";
    case UW_ERR_CORRUPT: return "UW_ERR_CORRUPT";
    case UW_ERR_NO_MEMORY: return "UW_ERR_NO_MEMORY";
    case UW_ERR_WORKSPACE: return "UW_ERR_WORKSPACE";
    case UW_ERR_CUDA: return "UW_ERR_CUDA";
    case UW_ERR_TIMEOUT: return "UW_ERR_TIMEOUT";
    case UW_ERR_BUFFER_TOO_SMALL: return "UW_ERR_BUFFER_TOO_SMALL";
    }
    return "UW_ERR_UNKNOWN";
}

extern "C" const char *uw_last_error(void) { return g_err; }

extern "C" uw_status uw_blob_validate(const void *blob, size_t size, uw_info *info)
{
    clear_error();
    BlobHeader h;
    uw_status s = parse_and_validate((const uint8_t *)blob, size, &h, true);
    if (s != UW_OK) return s;
    if (info) {
        memset(info, 0, sizeof *info);
        info->N = h.N; info->K = h.K; info->codec = h.codec; info->n_pal = h.n_pal;
        memcpy(info->palette, h.palette, 16);
        memcpy(info->code_len, h.code_len, 16);
        info->n_blocks = h.n_blocks; info->n_verbatim = h.n_verbatim; info->n_chunks = h.n_chunks;
        info->total_bits = h.total_bits; info->blob_bytes = h.blob_bytes;
        info->chunk_weights = (int32_t)h.chunk; info->max_code_len = (int32_t)h.max_len;
    }
    return UW_OK;
}
