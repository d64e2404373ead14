// uw_internal.h - declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/uw.h"

namespace uw {

constexpr int kBlock = 64;              // weights per verbatim decision
constexpr uint64_t kAlign = 256;        // blob section alignment
constexpr int kMaxBatchBuckets = 32;

enum Section { S_SM = 0, S_BITMAP, S_PREFIX, S_VERB, S_IDX, S_CHUNK, S_BITS, S_COUNT };

struct BlobHeader {
    int64_t N = 0, K = 0;
    uint32_t codec = 0, block = 64, chunk = 0, max_len = 0;
    uint32_t n_pal = 0;
    uint8_t palette[16] = {0};
    uint8_t code_len[16] = {0};
    uint64_t n_blocks = 0, n_verbatim = 0, n_chunks = 0, total_bits = 0, blob_bytes = 0;
    uint64_t off[S_COUNT] = {0}, len[S_COUNT] = {0};
};

// error reporting (thread-local message)
uw_status fail(uw_status s, const char *fmt, ...);
void clear_error();

// host codec (uw_host.cpp)
uw_status parse_and_validate(const uint8_t *blob, size_t size, BlobHeader *h, bool deep);
void canonical_codes(const uint8_t *lens, uint32_t *codes);
// Decode table for a canonical code: entry[v] for every max_len-bit prefix v is
// (symbol << 4) | length, 0 where no code matches.
void build_decode_table(const uint8_t *lens, int max_len, std::vector<uint8_t> &table);
// Multi-symbol table over 12-bit windows (limits <= 12), see uw_host.cpp for the entry layout.
void build_multi_table(const uint8_t *lens, std::vector<uint32_t> &table);
// Tile-major verbatim stream of a blob (K % 256 == 0): per unit of 128 rows x 256 weights, a 16-word mask
// ([K-stage j][row word]) and the count prefix; the verbatim exponents reordered unit by unit, (j, row) order.
void build_tile_verbatim(const BlobHeader &h, const uint8_t *blob, std::vector<uint32_t> &off,
                         std::vector<uint32_t> &mask, std::vector<uint8_t> &data);

// --------------------------------------------------------------------------------------------
// Device view of a loaded matrix (plain pointers, passed by value to kernels).
struct DevView {
    int64_t N, K;
    uint64_t n_blocks, n_chunks;
    uint32_t chunk, max_len;
    uint32_t n_pal;
    uint8_t palette[16];
    const uint8_t *sm;        // [N*K] sign<<7 | mantissa
    const uint32_t *bitmap;   // [ceil(n_blocks/32)] verbatim flags, LSB first
    const uint32_t *prefix;   // [ceil(n_blocks/32)] verbatim blocks before each word
    const uint8_t *verb_exp;  // [n_verbatim*64] exponents of verbatim blocks
    const uint8_t *codes;     // [N*K/2] 4-bit palette codes (resident form) or nullptr
    const uint32_t *chunk_off;// [n_chunks+1] bit offsets (Huffman)
    const uint32_t *bits;     // Huffman bit string, MSB-first u32 words, + guard words
    const uint8_t *dtab;      // [1 << max_len] decode table (Huffman)
    const uint32_t *mtab;     // [4096] multi-symbol decode table (Huffman, max_len <= 12), else nullptr
    int *status;              // device status word (0 = ok)
};

// Device-side status values written by kernels.
enum DevStatus { DEV_OK = 0, DEV_CORRUPT = 1, DEV_TIMEOUT = 2 };

// Weight-stream formats consumed by the matmul kernels.
enum WFormat { FMT_PAL = 0, FMT_EXP = 1, FMT_BF16 = 2 };
// Outputs of the preprocess / decode kernels.
enum DecOut { DEC_BF16 = 0, DEC_EXP = 1, DEC_CODES = 2 };

// Operand description for a matmul launch.
struct WOperand {
    int fmt;                  // WFormat
    const uint8_t *sm;        // FMT_PAL / FMT_EXP
    const uint8_t *codes;     // FMT_PAL
    const uint8_t *exps;      // FMT_EXP: [N*K] exponent bytes
    const uint16_t *w;        // FMT_BF16: [N*K]
    const uint32_t *bitmap, *prefix;
    const uint8_t *verb_exp;  // FMT_PAL verbatim handling
    // tile-major verbatim stream (present when K % 256 == 0): for unit u = tile * (K / 256) + kq (128 rows x 256
    // weights), tmv_mask[16u + 4j + w] bit b = row 32w + b's block kq*4 + j is verbatim; its exponents follow
    // those of earlier (j, row) in the unit at tmv_data[64 * (tmv_off[u] + rank)]
    const uint32_t *tmv_off, *tmv_mask;
    const uint8_t *tmv_data;
    uint8_t palette[16];
    int64_t N, K;
    int *status;              // device status word of the matrix
    int w_from_prev;          // the weight stream was written by the preceding kernel (preprocess workspace)
};

// kernel launchers (k_decode.cu, k_gemv.cu, k_tc.cu); return cudaError_t as int
int launch_decode_palette(const DevView &v, int out_kind, void *out, void *stream);
// max_ctas > 0: at most that many CTAs (a persistent grid over the chunk groups, for a share of the SMs)
int launch_decode_huffman(const DevView &v, int out_kind, void *out, void *stream, int max_ctas = 0);
// CTAs of the Huffman decode that one SM holds at once (its shared-memory table limits them)
constexpr int kDecodeCtasPerSm = 12;
int launch_gemv(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, int split_k,
                int variant, float *acc_ws, void *stream);
// persistent bulk-copy GEMV (B <= 2); variant 0: 8 consumer warps, 2 CTAs/SM; 2: 16 warps, 1 CTA/SM with all
// shared memory; 3: 8 warps, 1 CTA/SM in half the shared memory; 1: not this kernel (the plain-load GEMV)
bool gemv_tma_supported(const WOperand &w, int64_t B, int variant);
int launch_gemv_tma(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, int split_k, int variant,
                    float *acc_ws, int *status, void *stream);
// GEMV on the tensor pipe (mma.sync m16n8k16) for B <= 16, 16 consumer warps, 1 CTA/SM; variant 6: 256
// weights of a K-slice per warp (128 when B > 8); 7: 128
bool gemv_mma_supported(const WOperand &w, int64_t B, int variant);
int launch_gemv_mma(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, int split_k, int variant,
                    float *acc_ws, int *status, void *stream);
// GEMV on the tensor pipe with row-parallel warps over balanced 128 x 256 units, one CTA per SM (GEMV variant 8):
// B <= 64, 4-bit codes, K % 256 == 0; partial sums of a row block are added into a zeroed fp32 target
bool gemv_rp_supported(const WOperand &w, int64_t B);
int launch_gemv_rp(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, float *acc_ws, void *stream);
// GEMV that decodes the Huffman stream itself (Huffman-direct strategy): B <= 8, a multi-symbol table (code
// lengths <= 12), chunks of 64..2048 weights (a multiple of 64) that divide K; partial sums of each chunk column
// are added into a zeroed fp32 target.  Variant 0: plain loads; 1: each unit's rows and stream bytes are also
// prefetched into L2 in bulk one unit ahead
bool gemv_huff_supported(const DevView &v, int64_t B, int variant = 0);
int launch_gemv_huff(const DevView &v, const uint16_t *x, int64_t B, void *y, int out_bf16, int variant, float *acc_ws,
                     void *stream);
// zeroes the fp32 target of atomic adds (count floats, 16-byte aligned) as a dependent launch: it waits for the
// preceding kernel before writing and lets the following matmul start at once
int launch_zero_target(float *p, int64_t count, void *stream);
// persistent tcgen05 GEMM with rebuilt weights in shared memory (tensor-core variant 4): B <= 512, 4-bit codes,
// K % 256 == 0.  acc_ws: the matmul workspace (the fp32 accumulator region of acc_region_bytes, then the
// row-tile cells of tile_cells_bytes); needs no zeroing
bool tc4_supported(const WOperand &w, int64_t B);
int launch_tc4(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, float *acc_ws, void *stream);
// the matmul workspace after the preprocess output: an fp32 accumulator [B][N], then three 8-byte cells per
// 128-row tile (a row tile's partial sums from several CTAs are combined through them)
inline uint64_t acc_region_bytes(int64_t B, int64_t N) { return ((uint64_t)B * (uint64_t)N * 4 + 255) / 256 * 256; }
inline uint64_t tile_cells_bytes(int64_t N) { return ((uint64_t)(N + 127) / 128 * 24 + 255) / 256 * 256; }
// a fresh tag for one launch that combines shared row blocks through those cells: a process-wide count in 40 bits,
// never 0 (a CUDA graph replays a launch with the tag it was captured with)
uint64_t next_launch_epoch();
int launch_finalize(const float *acc, void *y, int64_t count, int out_bf16, void *stream);
int launch_tc(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, int split_k, int variant,
              float *acc_ws, void *stream);
bool tc_supported(const WOperand &w, int64_t B, int variant);
int gemv_default_split(const WOperand &w, int64_t B);
int tc_default_split(const WOperand &w, int64_t B, int variant);
// SMs the calling thread's launches size their grids for: the device's, or fewer while an SmBudget is alive
int num_sms();
int device_sms();
// While alive, the calling thread's matmul launches size their persistent grids for n SMs (the decode-vs-matmul
// split: the remaining SMs are left to a concurrent decode).  Budgets nest; n <= 0 means no limit.
struct SmBudget {
    int prev;
    explicit SmBudget(int n);
    ~SmBudget();
    SmBudget(const SmBudget &) = delete;
    SmBudget &operator=(const SmBudget &) = delete;
};
// cuTensorMapEncodeTiled from the driver (nullptr when the driver lacks it)
void *tensor_map_encoder();

// One autotuned plan per batch bucket (a power of two).
struct TuneEntry {
    int64_t bucket;
    uw_plan plan;
    float us;
};

// The matmul of the palette-transcode pipeline with the 4-bit codes already transcoded into `codes` (by an earlier
// launch, on any stream, ordered before this one by the caller): no preprocess launch, and `ws` holds only the
// accumulator the kernel may need (matmul_with_codes_workspace bytes).  The matrix must hold its Huffman stream.
size_t matmul_with_codes_workspace(const uw_matrix *m, int64_t B);
uw_status matmul_with_codes(const uw_matrix *m, const uint8_t *codes, const uint16_t *x, int64_t B, void *y,
                            uw_out_dtype od, void *ws, size_t ws_bytes, void *stream);

}  // namespace uw

// A compressed matrix resident on one device.
struct uw_matrix {
    uw::BlobHeader h;
    uw::DevView v;
    void *dev = nullptr;
    size_t dev_bytes = 0;
    uint8_t *codes = nullptr;  // resident 4-bit codes (may be null for Huffman)
    const uint32_t *tmv_off = nullptr, *tmv_mask = nullptr;  // tile-major verbatim stream (K % 256 == 0)
    const uint8_t *tmv_data = nullptr;
    bool has_stream = false;  // the Huffman stream (offsets, bits, tables) is resident
    int device = 0;
    std::mutex mu;
    std::vector<uw::TuneEntry> tune;
};
