/*
 * uw_oracle.c - plain, slow, single-threaded CPU oracle for the Unweight-style
 * lossless BF16 exponent codec and its matmul.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the bench's
 * CPU-baseline leg may load this file's library.  It shares no code, header,
 * table or helper with the CUDA library: it is written from the method's
 * description alone.
 *
 * Source: Cloudflare blog, "Unweight" (Japanese edition).  Passages used:
 *   [BF16]     the BF16 anatomy paragraphs: 1 sign bit, 8 exponent bits,
 *              7 mantissa bits; sign and mantissa look random and are kept raw.
 *   [TOP16]    the exponent-statistics paragraph: the 16 most common exponents
 *              cover >99% of a layer; entropy is at most about 2.6 bits.
 *   [HUFF]     the paragraph on Huffman-coding only the exponent byte.
 *   [VERBATIM] the paragraph on rare exponents: a run of 64 weights holding an
 *              exponent outside the top-16 palette is stored verbatim, one
 *              decision per run, no per-element branch.
 *   [PALETTE]  the four-pipelines paragraph: "direct palette" 4-bit indices
 *              from which BF16 is rebuilt on the fly.
 *   [LOSSLESS] the results paragraph: every compression is bit-exact.
 *
 * Readings where the page is silent (each one is a pinned rule of the format):
 *   - the sign+mantissa ("sm") byte is sign<<7 | mantissa; the exponent byte is
 *     bits 14..7 of the BF16 pattern; specials (zeros, subnormals, inf, NaN)
 *     are not special-cased;
 *   - palette = the 16 (or fewer) exponent values with the highest counts over
 *     the whole matrix, ties broken by the smaller exponent value; palette index
 *     i is rank i;
 *   - a block is 64 consecutive weights along K within one row (K % 64 == 0);
 *   - verbatim blocks apply to both codecs; their 64 exponent bytes are stored
 *     in block order, their 4-bit codes are 0 and they emit no Huffman symbols;
 *   - nibble order: even k in bits 3..0, odd k in bits 7..4;
 *   - Huffman lengths come from package-merge (Larmore & Hirschberg, 1990),
 *     length limit L, items sorted by (count, symbol), a package placed before
 *     an item of equal weight; one used symbol gets length 1;
 *   - codes are canonical as in RFC 1951 section 3.2.2;
 *   - the bit string is written MSB-first into 32-bit words (first bit = bit 31
 *     of word 0) and is split into chunks of C flat weights with a 32-bit
 *     absolute bit offset per chunk.
 *
 * Blob layout (little-endian; header 256 bytes; every section starts on a
 * 256-byte boundary and the gaps are zero):
 *   0 "UWB1" | 4 u32 version=1 | 8 i64 N | 16 i64 K | 24 u32 codec (0 palette,
 *   1 huffman) | 28 u32 block=64 | 32 u32 chunk C (0 for palette) | 36 u32 L
 *   (0 for palette) | 40 u8 n_pal | 41 u8 palette[16] | 57 u8 code_len[16] |
 *   80 u64 n_blocks | 88 u64 n_verbatim | 96 u64 n_chunks | 104 u64 total_bits |
 *   112 u64 blob bytes | 128 section table: 7 x (u64 offset, u64 bytes) for
 *   SM, BITMAP, PREFIX, VERB_EXP, IDX, CHUNK_OFF, BITS.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_ARG (-1)
#define OR_ERR_SHAPE (-2)
#define OR_ERR_SPACE (-3)
#define OR_ERR_CORRUPT (-4)
#define OR_ERR_RANGE (-5)

enum { SEC_SM = 0, SEC_BITMAP, SEC_PREFIX, SEC_VERB, SEC_IDX, SEC_CHUNK, SEC_BITS, N_SEC };

/* ---------------------------------------------------------------- [BF16] */
uint8_t or_sm_byte(uint16_t h) { return (uint8_t)(((h >> 8) & 0x80) | (h & 0x7F)); }
uint8_t or_exp_byte(uint16_t h) { return (uint8_t)((h >> 7) & 0xFF); }
uint16_t or_rebuild(uint8_t sm, uint8_t e)
{
    return (uint16_t)(((sm & 0x80) << 8) | ((uint16_t)e << 7) | (sm & 0x7F));
}

static double bf16_value(uint16_t h)
{
    uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/* ---------------------------------------------------------------- [TOP16] */
/* Exponent histogram over all weights and the palette: highest count first,
 * ties to the smaller exponent; at most 16 entries, only exponents present. */
int or_palette(const uint16_t *w, int64_t n, uint64_t counts[256], uint8_t pal[16])
{
    int taken[256];
    memset(counts, 0, 256 * sizeof(uint64_t));
    memset(taken, 0, sizeof(taken));
    memset(pal, 0, 16);
    for (int64_t i = 0; i < n; i++) counts[or_exp_byte(w[i])]++;
    int n_pal = 0;
    while (n_pal < 16) {
        int best = -1;
        for (int e = 0; e < 256; e++) {
            if (taken[e] || counts[e] == 0) continue;
            if (best < 0 || counts[e] > counts[best]) best = e; /* strict '>' keeps the smaller e on ties */
        }
        if (best < 0) break;
        taken[best] = 1;
        pal[n_pal++] = (uint8_t)best;
    }
    return n_pal;
}

/* ---------------------------------------------------------------- [HUFF] */
/* Package-merge for length-limited prefix codes.  Each list entry carries how
 * many times every symbol occurs inside it; the code length of a symbol is its
 * total count over the first 2(n-1) entries of the final list. */
typedef struct {
    uint64_t weight;
    int occ[16];
} pm_entry;

int or_huffman_lengths(const uint64_t *counts, int n_sym, int max_len, uint8_t *lens)
{
    if (n_sym < 0 || n_sym > 16 || max_len < 1 || max_len > 15) return OR_ERR_ARG;
    for (int s = 0; s < n_sym; s++) lens[s] = 0;
    pm_entry items[16];
    int n = 0;
    for (int s = 0; s < n_sym; s++) {
        if (counts[s] == 0) continue;
        memset(&items[n], 0, sizeof(pm_entry));
        items[n].weight = counts[s];
        items[n].occ[s] = 1;
        n++;
    }
    if (n == 0) return OR_OK;
    if (n == 1) {
        for (int s = 0; s < n_sym; s++)
            if (counts[s]) lens[s] = 1;
        return OR_OK;
    }
    if ((1 << max_len) < n) return OR_ERR_RANGE;
    /* insertion sort by (weight asc, symbol asc); items were created in symbol order */
    for (int i = 1; i < n; i++) {
        pm_entry t = items[i];
        int j = i - 1;
        while (j >= 0 && items[j].weight > t.weight) { items[j + 1] = items[j]; j--; }
        items[j + 1] = t;
    }
    pm_entry list[64], packages[32], merged[64];
    int n_list = n;
    for (int i = 0; i < n; i++) list[i] = items[i];
    for (int level = 1; level < max_len; level++) {
        int n_pk = n_list / 2;
        for (int p = 0; p < n_pk; p++) {
            packages[p].weight = list[2 * p].weight + list[2 * p + 1].weight;
            for (int s = 0; s < 16; s++) packages[p].occ[s] = list[2 * p].occ[s] + list[2 * p + 1].occ[s];
        }
        int i = 0, p = 0, m = 0;
        while (i < n || p < n_pk) {
            if (p < n_pk && (i >= n || packages[p].weight <= items[i].weight)) merged[m++] = packages[p++];
            else merged[m++] = items[i++];
        }
        n_list = m;
        for (int k = 0; k < m; k++) list[k] = merged[k];
    }
    int take = 2 * (n - 1);
    for (int k = 0; k < take; k++)
        for (int s = 0; s < n_sym; s++) lens[s] = (uint8_t)(lens[s] + list[k].occ[s]);
    return OR_OK;
}

/* Canonical codes, RFC 1951 section 3.2.2: shorter codes first, then by symbol. */
void or_canonical_codes(const uint8_t *lens, int n_sym, uint32_t *codes)
{
    int bl_count[16] = {0};
    uint32_t next_code[17] = {0};
    for (int s = 0; s < n_sym; s++) if (lens[s]) bl_count[lens[s]]++;
    uint32_t code = 0;
    for (int bits = 1; bits <= 15; bits++) {
        code = (code + (uint32_t)bl_count[bits - 1]) << 1;
        next_code[bits] = code;
    }
    for (int s = 0; s < n_sym; s++) {
        codes[s] = 0;
        if (lens[s]) codes[s] = next_code[lens[s]]++;
    }
}

/* ---------------------------------------------------------------- blob writer helpers */
static void put_u32(uint8_t *p, uint32_t v) { for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static void put_u64(uint8_t *p, uint64_t v) { for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static uint32_t get_u32(const uint8_t *p) { uint32_t v = 0; for (int i = 3; i >= 0; i--) v = (v << 8) | p[i]; return v; }
static uint64_t get_u64(const uint8_t *p) { uint64_t v = 0; for (int i = 7; i >= 0; i--) v = (v << 8) | p[i]; return v; }
static uint64_t align256(uint64_t v) { return (v + 255) / 256 * 256; }

/*
 * Encode W[N,K] (bf16 bits, row-major) into a blob.
 * codec 0 = palette (4-bit codes), 1 = Huffman (chunk C weights, length limit L).
 * If out == NULL, only *out_size is written.
 */
int or_encode(const uint16_t *w, int64_t N, int64_t K, int codec, uint32_t chunk, uint32_t max_len,
              uint8_t *out, uint64_t cap, uint64_t *out_size)
{
    if (N < 0 || K < 0 || (codec != 0 && codec != 1)) return OR_ERR_ARG;
    if (K % 64 != 0) return OR_ERR_SHAPE;
    if (codec == 1 && (chunk < 64 || chunk % 64 != 0 || max_len < 4 || max_len > 15)) return OR_ERR_ARG;
    uint64_t n = (uint64_t)N * (uint64_t)K;
    uint64_t n_blocks = n / 64;
    uint64_t n_words = (n_blocks + 31) / 32;

    /* [TOP16] palette */
    uint64_t counts[256];
    uint8_t pal[16];
    int n_pal = or_palette(w, (int64_t)n, counts, pal);
    int pal_index[256];
    for (int e = 0; e < 256; e++) pal_index[e] = -1;
    for (int i = 0; i < n_pal; i++) pal_index[pal[i]] = i;

    /* [VERBATIM] one decision per 64-weight block */
    uint8_t *verb = (uint8_t *)calloc(n_blocks ? n_blocks : 1, 1);
    uint64_t n_verb = 0;
    for (uint64_t b = 0; b < n_blocks; b++) {
        for (int j = 0; j < 64; j++)
            if (pal_index[or_exp_byte(w[b * 64 + j])] < 0) { verb[b] = 1; break; }
        n_verb += verb[b];
    }

    /* [HUFF] symbol counts over non-verbatim blocks, lengths, canonical codes */
    uint8_t lens[16] = {0};
    uint32_t codes[16] = {0};
    uint64_t n_chunks = 0, total_bits = 0;
    if (codec == 1) {
        uint64_t sym_counts[16] = {0};
        for (uint64_t b = 0; b < n_blocks; b++) {
            if (verb[b]) continue;
            for (int j = 0; j < 64; j++) sym_counts[pal_index[or_exp_byte(w[b * 64 + j])]]++;
        }
        int rc = or_huffman_lengths(sym_counts, 16, (int)max_len, lens);
        if (rc) { free(verb); return rc; }
        or_canonical_codes(lens, 16, codes);
        for (int s = 0; s < 16; s++) total_bits += sym_counts[s] * lens[s];
        if (total_bits >= ((uint64_t)1 << 32)) { free(verb); return OR_ERR_RANGE; }
        n_chunks = (n + chunk - 1) / chunk;
    }

    /* section sizes and offsets */
    uint64_t sec_bytes[N_SEC] = {0}, sec_off[N_SEC];
    sec_bytes[SEC_SM] = n;
    sec_bytes[SEC_BITMAP] = 4 * n_words;
    sec_bytes[SEC_PREFIX] = 4 * n_words;
    sec_bytes[SEC_VERB] = 64 * n_verb;
    if (codec == 0) sec_bytes[SEC_IDX] = n / 2;
    if (codec == 1) {
        sec_bytes[SEC_CHUNK] = 4 * (n_chunks + 1);
        sec_bytes[SEC_BITS] = 4 * ((total_bits + 31) / 32);
    }
    uint64_t pos = 256;
    for (int s = 0; s < N_SEC; s++) {
        sec_off[s] = pos;
        pos = align256(pos + sec_bytes[s]);
    }
    uint64_t total = pos;
    *out_size = total;
    if (!out) { free(verb); return OR_OK; }
    if (cap < total) { free(verb); return OR_ERR_SPACE; }
    memset(out, 0, total);

    /* header */
    memcpy(out, "UWB1", 4);
    put_u32(out + 4, 1);
    put_u64(out + 8, (uint64_t)N);
    put_u64(out + 16, (uint64_t)K);
    put_u32(out + 24, (uint32_t)codec);
    put_u32(out + 28, 64);
    put_u32(out + 32, codec == 1 ? chunk : 0);
    put_u32(out + 36, codec == 1 ? max_len : 0);
    out[40] = (uint8_t)n_pal;
    for (int i = 0; i < 16; i++) out[41 + i] = pal[i];
    for (int i = 0; i < 16; i++) out[57 + i] = lens[i];
    put_u64(out + 80, n_blocks);
    put_u64(out + 88, n_verb);
    put_u64(out + 96, n_chunks);
    put_u64(out + 104, total_bits);
    put_u64(out + 112, total);
    for (int s = 0; s < N_SEC; s++) {
        put_u64(out + 128 + 16 * s, sec_off[s]);
        put_u64(out + 136 + 16 * s, sec_bytes[s]);
    }

    /* [BF16] raw sign+mantissa bytes */
    uint8_t *sm = out + sec_off[SEC_SM];
    for (uint64_t i = 0; i < n; i++) sm[i] = or_sm_byte(w[i]);

    /* [VERBATIM] bitmap (LSB first), exclusive prefix per word, verbatim exponents */
    uint8_t *bm = out + sec_off[SEC_BITMAP];
    uint8_t *pf = out + sec_off[SEC_PREFIX];
    uint8_t *ve = out + sec_off[SEC_VERB];
    uint64_t seen = 0;
    for (uint64_t wd = 0; wd < n_words; wd++) {
        uint32_t bits = 0;
        put_u32(pf + 4 * wd, (uint32_t)seen);
        for (int j = 0; j < 32; j++) {
            uint64_t b = wd * 32 + j;
            if (b < n_blocks && verb[b]) { bits |= 1u << j; seen++; }
        }
        put_u32(bm + 4 * wd, bits);
    }
    uint64_t v = 0;
    for (uint64_t b = 0; b < n_blocks; b++) {
        if (!verb[b]) continue;
        for (int j = 0; j < 64; j++) ve[v * 64 + j] = or_exp_byte(w[b * 64 + j]);
        v++;
    }

    if (codec == 0) {
        /* [PALETTE] 4-bit codes, even k low nibble */
        uint8_t *idx = out + sec_off[SEC_IDX];
        for (uint64_t i = 0; i < n; i++) {
            uint64_t b = i / 64;
            uint8_t code = verb[b] ? 0 : (uint8_t)pal_index[or_exp_byte(w[i])];
            idx[i / 2] |= (uint8_t)(code << (4 * (i & 1)));
        }
    } else {
        /* [HUFF] MSB-first bit string, chunk offsets */
        uint8_t *co = out + sec_off[SEC_CHUNK];
        uint8_t *bs = out + sec_off[SEC_BITS];
        uint64_t bitpos = 0;
        for (uint64_t c = 0; c < n_chunks; c++) {
            put_u32(co + 4 * c, (uint32_t)bitpos);
            uint64_t lo = c * chunk, hi = lo + chunk;
            if (hi > n) hi = n;
            for (uint64_t i = lo; i < hi; i++) {
                if (verb[i / 64]) continue;
                int s = pal_index[or_exp_byte(w[i])];
                for (int t = lens[s] - 1; t >= 0; t--) {
                    if ((codes[s] >> t) & 1u) {
                        uint64_t word = bitpos / 32;
                        uint32_t cur = get_u32(bs + 4 * word);
                        cur |= 1u << (31 - (bitpos % 32));
                        put_u32(bs + 4 * word, cur);
                    }
                    bitpos++;
                }
            }
        }
        put_u32(co + 4 * n_chunks, (uint32_t)bitpos);
    }
    free(verb);
    return OR_OK;
}

/* ---------------------------------------------------------------- decoder ([LOSSLESS]) */
/* Rebuild W[N,K] from a blob.  w must hold N*K values. */
int or_decode(const uint8_t *blob, uint64_t size, uint16_t *w)
{
    if (size < 256 || memcmp(blob, "UWB1", 4) != 0 || get_u32(blob + 4) != 1) return OR_ERR_CORRUPT;
    uint64_t N = get_u64(blob + 8), K = get_u64(blob + 16);
    uint32_t codec = get_u32(blob + 24), chunk = get_u32(blob + 32);
    int n_pal = blob[40];
    const uint8_t *pal = blob + 41, *lens = blob + 57;
    uint64_t n = N * K, n_blocks = get_u64(blob + 80), n_chunks = get_u64(blob + 96);
    uint64_t off[N_SEC], len[N_SEC];
    for (int s = 0; s < N_SEC; s++) {
        off[s] = get_u64(blob + 128 + 16 * s);
        len[s] = get_u64(blob + 136 + 16 * s);
        if (off[s] + len[s] > size) return OR_ERR_CORRUPT;
    }
    if (n_blocks != n / 64 || len[SEC_SM] != n || n_pal > 16) return OR_ERR_CORRUPT;
    const uint8_t *sm = blob + off[SEC_SM], *bm = blob + off[SEC_BITMAP];
    const uint8_t *pf = blob + off[SEC_PREFIX], *ve = blob + off[SEC_VERB];

    /* per-block verbatim flag and the index of its exponents in VERB_EXP */
    for (uint64_t b = 0; b < n_blocks; b++) {
        uint32_t word = get_u32(bm + 4 * (b / 32));
        if (!((word >> (b % 32)) & 1u)) continue;
        uint64_t vi = get_u32(pf + 4 * (b / 32));
        for (uint64_t j = 0; j < b % 32; j++) vi += (word >> j) & 1u;
        if ((vi + 1) * 64 > len[SEC_VERB]) return OR_ERR_CORRUPT;
        for (int j = 0; j < 64; j++) w[b * 64 + j] = or_rebuild(sm[b * 64 + j], ve[vi * 64 + j]);
    }
    if (codec == 0) {
        const uint8_t *idx = blob + off[SEC_IDX];
        if (len[SEC_IDX] != n / 2) return OR_ERR_CORRUPT;
        for (uint64_t i = 0; i < n; i++) {
            uint64_t b = i / 64;
            if ((get_u32(bm + 4 * (b / 32)) >> (b % 32)) & 1u) continue;
            int code = (idx[i / 2] >> (4 * (i & 1))) & 0xF;
            if (code >= n_pal) return OR_ERR_CORRUPT;
            w[i] = or_rebuild(sm[i], pal[code]);
        }
        return OR_OK;
    }
    if (codec != 1 || chunk == 0 || n_chunks != (n + chunk - 1) / chunk) return OR_ERR_CORRUPT;
    uint32_t codes[16];
    or_canonical_codes(lens, 16, codes);
    const uint8_t *co = blob + off[SEC_CHUNK], *bs = blob + off[SEC_BITS];
    uint64_t total_bits = 8 * len[SEC_BITS];
    for (uint64_t c = 0; c < n_chunks; c++) {
        uint64_t bitpos = get_u32(co + 4 * c), end = get_u32(co + 4 * (c + 1));
        uint64_t lo = c * chunk, hi = lo + chunk;
        if (hi > n) hi = n;
        for (uint64_t i = lo; i < hi; i++) {
            uint64_t b = i / 64;
            if ((get_u32(bm + 4 * (b / 32)) >> (b % 32)) & 1u) continue;
            /* read one bit at a time until the prefix equals some symbol's code */
            uint32_t value = 0;
            int got = -1;
            for (int l = 1; l <= 15 && got < 0; l++) {
                if (bitpos >= total_bits) return OR_ERR_CORRUPT;
                uint32_t word = get_u32(bs + 4 * (bitpos / 32));
                value = (value << 1) | ((word >> (31 - bitpos % 32)) & 1u);
                bitpos++;
                for (int s = 0; s < 16; s++)
                    if (lens[s] == l && codes[s] == value) { got = s; break; }
            }
            if (got < 0 || got >= n_pal) return OR_ERR_CORRUPT;
            w[i] = or_rebuild(sm[i], pal[got]);
        }
        if (bitpos != end) return OR_ERR_CORRUPT;
    }
    return OR_OK;
}

/* ---------------------------------------------------------------- matmul */
/* Y[b, j] = sum_k W[rows[j], k] * X[b, k] in fp64 (k ascending), and the
 * magnitude sum A[b, j] = sum_k |W[rows[j], k] * X[b, k]| used by the tolerance.
 * rows == NULL means all N rows in order.  Y and A are [B, n_rows]. */
void or_matmul_rows(const uint16_t *w, int64_t N, int64_t K, const uint16_t *x, int64_t B,
                    const int64_t *rows, int64_t n_rows, double *y, double *a)
{
    if (!rows) n_rows = N;
    for (int64_t b = 0; b < B; b++) {
        for (int64_t j = 0; j < n_rows; j++) {
            int64_t r = rows ? rows[j] : j;
            double s = 0.0, m = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = bf16_value(w[r * K + k]) * bf16_value(x[b * K + k]);
                s += p;
                m += p < 0 ? -p : p;
            }
            y[b * n_rows + j] = s;
            if (a) a[b * n_rows + j] = m;
        }
    }
}

/* ---------------------------------------------------------------- array forms of the [BF16] split */
void or_split_many(const uint16_t *h, int64_t n, uint8_t *sm, uint8_t *e)
{
    for (int64_t i = 0; i < n; i++) { sm[i] = or_sm_byte(h[i]); e[i] = or_exp_byte(h[i]); }
}

void or_rebuild_many(const uint8_t *sm, const uint8_t *e, int64_t n, uint16_t *h)
{
    for (int64_t i = 0; i < n; i++) h[i] = or_rebuild(sm[i], e[i]);
}
