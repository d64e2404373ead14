// k_gemv_huff.cu - matrix-vector product that decodes the Huffman exponent stream inside the product
// (Huffman-direct GEMV, sm_103a), batch 1..8.
//
// Cloudflare blog "Unweight": the section on the execution pipelines has three pipelines that first decode the
// Huffman stream into an HBM workspace (full BF16, exponent bytes, or 4-bit palette codes) and a fourth that
// reads resident palette codes; the section on the decode kernels keeps the Huffman lookup table in shared
// memory.  This kernel removes the workspace from the Huffman pipelines: the stream is decoded in the GEMV,
// the exponents never leave the chip, and the matrix stays resident in its smallest form (the Huffman blob).
//
// Work is split into units of 32 weight rows x one chunk column (the C weights of chunk j of each row; K % C
// == 0, so no chunk crosses a row).  Lane l of a warp owns row 32 rb + l of its unit and decodes that row's
// chunk sequentially (the format gives a bit offset per chunk only), 16 codes at a time, through a 12-bit
// multi-symbol table in shared memory (up to five codes per lookup; the last four symbols of a chunk one at a
// time, so no lookup reads past the chunk's codes).  All lanes of a warp work on the same chunk column, so
// their activations are one broadcast load; each 16-weight group is rebuilt with the per-lane pair table
// (exponent fields of two weights per code byte) and one byte permute of the sign+mantissa bytes, and
// multiplied into fp32 accumulators.  A 64-weight block marked verbatim takes its 64 exponent bytes from the
// verbatim section and no symbols from the stream.
//
// One CTA per SM owns a balanced, contiguous range of units (row block major, chunk column minor, so a CTA walks
// contiguous memory); its warps claim units one at a time from a shared-memory counter.  A unit's partial
// sums are added with one fp32 atomic per row and batch row into a target zeroed by the preceding (dependent)
// launch.  Stream reads stop at the stream's end and guard words; an unassigned code prefix, or a chunk whose
// codes do not end exactly at the next chunk's offset, latches DEV_CORRUPT in the matrix status word.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <type_traits>

#include "dev_async.cuh"
#include "uw_internal.h"

namespace uw {

namespace {

using namespace dev;

// one CTA per SM holds the only copy of the tables, so the SM's unified cache stays mostly L1 (the lanes' row
// and stream reads are scattered 16- and 4-byte loads that reuse their 32-byte sectors); at most 24 warps, so a
// lane has up to 85 registers
template <int NB> constexpr int huff_threads() { return 768; }
// batch rows whose activations are loaded before a group's decode (their latency hides behind it)
template <int NB> __host__ __device__ constexpr int huff_early_x() { return NB < 2 ? NB : 2; }
constexpr int kMTabBytes = 4096 * 4;                      // multi-symbol table
constexpr int kHSmem = kPairTableBytes + kMTabBytes;     // 48 KB

struct HuffArgs {
    const uint8_t *sm;
    const uint32_t *bitmap, *prefix;
    const uint8_t *verb_exp;
    const uint32_t *chunk_off, *bits, *mtab;
    const uint16_t *x;
    float *acc;        // zeroed fp32 target [B][N]
    int *status;
    int64_t N, K, B;
    uint64_t n_blocks, n_chunks;
    int64_t units;     // ceil(N / 32) row blocks x cpr chunk columns
    int cpr;           // chunk columns per row: K / C
    int C;             // weights per chunk (multiple of 64, at most 2048)
    uint8_t palette[16];
};

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint4 ldg_nc16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// one bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16)
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// acc += w * x over both halves of a bf16x2 pair of weights and of activations (BF16 products are exact in
// fp32, so this equals two fp32 FMAs on the widened values)
__device__ __forceinline__ float fma2_bf16(uint32_t w2, uint32_t x2, float acc)
{
    asm("{\n .reg .b16 wl, wh, xl, xh;\n mov.b32 {wl, wh}, %1;\n mov.b32 {xl, xh}, %2;\n"
        " fma.rn.f32.bf16 %0, wl, xl, %0;\n fma.rn.f32.bf16 %0, wh, xh, %0;\n}\n"
        : "+f"(acc)
        : "r"(w2), "r"(x2));
    return acc;
}

// PF (variant 1): before a unit is decoded, each lane asks L2 for its row's C sign+mantissa bytes and its
// chunk's stream bytes in one bulk prefetch each (one unit ahead), so HBM serves contiguous runs instead of the
// 32-byte sectors the lanes' 16-byte loads fetch one at a time.  Measured on the 8B gate_proj at B = 1: 70 us
// against 64 us without it (variant 0, the default), once L1 holds the lanes' sectors.
template <int NB, bool PF>
__global__ void __launch_bounds__(huff_threads<NB>(), 1) gemv_huff_kernel(const __grid_constant__ HuffArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int next_unit;
    uint8_t *tab = smem;                                  // per-lane pair table
    uint32_t *mt = (uint32_t *)(smem + kPairTableBytes);  // multi-symbol decode table
    grid_launch_dependents();
    fill_pair_table(tab, a.palette, threadIdx.x, blockDim.x);
    // the multi-symbol table; an entry of 0 (these 12 bits start no code) becomes one 1-bit code 0 with bit 31 set,
    // so the decode loop needs no test: the flag is collected and reported after the loop
    for (int i = threadIdx.x; i < kMTabBytes / 4; i += blockDim.x) {
        const uint32_t e = __ldg(a.mtab + i);
        mt[i] = e ? e : 0x80000000u | (1u << 7) | (1u << 4) | 1u;
    }
    if (threadIdx.x == 0) next_unit = 0;
    const int64_t u0 = a.units * blockIdx.x / gridDim.x, u1 = a.units * (blockIdx.x + 1) / gridDim.x;
    grid_dependency_wait();  // X and the zeroed target belong to the stream order after the preceding kernels
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const uint8_t *tab_lane = tab + 4 * lane;
    const int64_t N = a.N, K = a.K;
    const int C = a.C, G = C / 16, nbk = C / 64;
    // stream words that may be read: the stream and all but the last few words of the 512-byte guard behind it
    const uint32_t wlim = ((__ldg(a.chunk_off + a.n_chunks) + 31) >> 5) + 120;
    const uint32_t *bits = a.bits;
    auto word_at = [&](uint32_t wn) -> uint32_t { return wn < wlim ? __ldg(bits + wn) : 0u; };
    bool bad = false;
    uint32_t bad_bits = 0;  // bit 31: a lookup met bits that start no code

    // a unit's rows and chunk column; the lane's L2 prefetches for it
    auto claim = [&]() -> int64_t {
        int t = 0;
        if (lane == 0) t = atomicAdd(&next_unit, 1);
        return u0 + __shfl_sync(0xFFFFFFFFu, t, 0);
    };
    auto prefetch_unit = [&](int64_t u) {
        const int64_t rb = u / a.cpr;
        const int j = (int)(u - rb * a.cpr);
        const int64_t r = rb * 32 + lane;
        if (r >= N) return;
        const uint64_t c = (uint64_t)r * (uint64_t)a.cpr + (uint64_t)j;
        prefetch_l2(a.sm + (uint64_t)r * (uint64_t)K + (uint64_t)j * (uint64_t)C, (uint32_t)C);
        const uint32_t b0 = (__ldg(a.chunk_off + c) >> 7) << 4, b1 = ((__ldg(a.chunk_off + c + 1) + 127) >> 7) << 4;
        if (b1 > b0) prefetch_l2((const uint8_t *)a.bits + b0, b1 - b0);
    };
    int64_t u_next = claim();
    if (PF && u_next < u1) prefetch_unit(u_next);
    for (;;) {
        const int64_t u = u_next;
        if (u >= u1) break;
        u_next = claim();
        if (PF && u_next < u1) prefetch_unit(u_next);
        const int64_t rb = u / a.cpr;
        const int j = (int)(u - rb * a.cpr);
        const int64_t r = rb * 32 + lane;
        float acc0[NB], acc1[NB];
#pragma unroll
        for (int b = 0; b < NB; b++) acc0[b] = acc1[b] = 0.f;
        if (r < N) {
            const uint64_t c = (uint64_t)r * (uint64_t)a.cpr + (uint64_t)j;
            const uint32_t pos0 = __ldg(a.chunk_off + c), pos1 = __ldg(a.chunk_off + c + 1);
            // verbatim flags of the chunk's blocks from one 64-bit window of the bitmap
            const uint64_t bb = c * (uint64_t)nbk;
            const uint64_t wb = bb >> 5;
            uint64_t win = __ldg(a.bitmap + wb);
            if ((wb + 1) * 32 < a.n_blocks) win |= (uint64_t)__ldg(a.bitmap + wb + 1) << 32;
            const uint32_t vmask = (uint32_t)(win >> (bb & 31)) & (nbk >= 32 ? 0xFFFFFFFFu : ((1u << nbk) - 1u));
            uint32_t vbase = 0;
            if (vmask) vbase = __ldg(a.prefix + wb) + __popc((uint32_t)win & ((1u << (bb & 31)) - 1u));
            int remaining = 64 * (nbk - __popc(vmask));  // codes of the chunk not yet decoded

            // 64-bit bit buffer, MSB-aligned, `avail` bits valid; the next stream word is loaded one refill ahead.
            // The absolute position of the next unread bit is always 32 (wi - 1) - avail.
            const uint32_t w0 = pos0 >> 5;
            uint64_t buf = (((uint64_t)word_at(w0) << 32) | word_at(w0 + 1)) << (pos0 & 31);
            int avail = 64 - (int)(pos0 & 31);
            uint32_t wi = w0 + 2;
            uint32_t nxt = word_at(wi++);
            uint64_t cacc = 0;  // decoded codes not yet consumed, 4 bits each, the first in the low nibble
            uint32_t sh = 0;    // 4 x the number of codes in cacc

            const uint8_t *smp = a.sm + (uint64_t)r * (uint64_t)K + (uint64_t)j * (uint64_t)C;
            const uint16_t *xp = a.x + (int64_t)j * C;
            uint4 S_next = ldg_nc16(smp);
            for (int g = 0; g < G; g++) {
                const uint4 S = S_next;
                if (g + 1 < G) S_next = ldg_nc16(smp + 16 * (g + 1));
                constexpr int XE = huff_early_x<NB>();
                uint4 Xe[XE][2];
#pragma unroll
                for (int b = 0; b < XE; b++) {
                    const uint4 *xs = (const uint4 *)(xp + b * K + 16 * g);
                    if (NB == 1 || b < a.B) {
                        Xe[b][0] = __ldg(xs);
                        Xe[b][1] = __ldg(xs + 1);
                    } else {
                        Xe[b][0] = Xe[b][1] = make_uint4(0, 0, 0, 0);
                    }
                }
                uint32_t pw[8];
                const int blk = g >> 2;
                if ((vmask >> blk) & 1u) {
                    const uint32_t vi = vbase + __popc(vmask & ((1u << blk) - 1u));
                    const uint4 E = ldg_nc16(a.verb_exp + (uint64_t)vi * 64 + (g & 3) * 16);
#pragma unroll
                    for (int q = 0; q < 4; q++) pairs_from_exps(word_of(S, q), word_of(E, q), pw[2 * q], pw[2 * q + 1]);
                } else {
                    uint32_t last_syms = 0, last_sh = 60;
                    // one multi-symbol lookup: up to five codes, `len` bits; a table entry with bit 31 set marks
                    // bits that start no code (a corrupt stream; it counts as one 1-bit code 0)
                    auto lookup = [&](bool single) {
                        const uint32_t e = mt[(uint32_t)(buf >> 52)];
                        bad_bits |= e;
                        const uint32_t len = single ? (e >> 7) & 15u : e & 15u;
                        buf <<= len;
                        avail -= (int)len;
                        last_syms = single ? (e >> 11) & 15u : e >> 11;
                        last_sh = sh;
                        cacc |= (uint64_t)last_syms << sh;
                        sh += single ? 4u : (e >> 2) & 28u;
                    };
                    if (remaining >= 21) {
                        // at least 21 codes left: more than this group can take (16, plus at most 4 carried in or
                        // out), so every lookup may decode five codes.  The refill tops the buffer up to more than
                        // 32 bits, enough for two lookups of at most 12 bits each.
                        const uint32_t sh0 = sh;
                        while (sh < 64) {
                            if (avail <= 32) {
                                buf |= (uint64_t)nxt << (32 - avail);
                                avail += 32;
                                nxt = word_at(wi++);
                            }
                            lookup(false);
                            if (sh >= 64) break;
                            lookup(false);
                        }
                        remaining -= (int)((sh - sh0) >> 2);
                    } else {
                        // the chunk's last coded group: its last four codes are decoded one lookup each, so no
                        // lookup reads past the chunk's codes
                        while (sh < 64) {
                            if (avail <= 32) {
                                buf |= (uint64_t)nxt << (32 - avail);
                                avail += 32;
                                nxt = word_at(wi++);
                            }
                            const uint32_t sh0 = sh;
                            lookup(remaining < 5);
                            remaining -= (int)((sh - sh0) >> 2);
                        }
                    }
                    const uint64_t cw = cacc;
                    // codes of the last lookup beyond the 16th stay for the next group (last_sh >= 44 here)
                    cacc = (uint64_t)(last_syms >> (64u - last_sh));
                    sh -= 64;
                    const uint32_t c0 = (uint32_t)cw, c1 = (uint32_t)(cw >> 32);
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const uint32_t Sq = word_of(S, q);
                        const uint32_t Cw = q < 2 ? c0 : c1;
                        const int jb = 2 * (q & 1);
                        pw[2 * q] = (__byte_perm(Sq, 0u, 0x1100u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb);
                        pw[2 * q + 1] = (__byte_perm(Sq, 0u, 0x3322u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb + 1);
                    }
                }
                // activations: all lanes read the same 32 bytes (one broadcast load per batch row)
#pragma unroll
                for (int b = 0; b < NB; b++) {
                    if (NB > 1 && b >= a.B) continue;
                    const uint4 *xs = (const uint4 *)(xp + b * K + 16 * g);
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const uint4 X = b < XE ? Xe[b < XE ? b : 0][h] : __ldg(xs + h);
                        acc0[b] = fma2_bf16(pw[4 * h + 0], X.x, acc0[b]);
                        acc1[b] = fma2_bf16(pw[4 * h + 1], X.y, acc1[b]);
                        acc0[b] = fma2_bf16(pw[4 * h + 2], X.z, acc0[b]);
                        acc1[b] = fma2_bf16(pw[4 * h + 3], X.w, acc1[b]);
                    }
                }
            }
            // every code of the chunk was used, and the codes ended exactly at the next chunk's offset
            if (32ull * (wi - 1) - (uint64_t)avail != (uint64_t)pos1 || sh != 0) bad = true;
#pragma unroll
            for (int b = 0; b < NB; b++)
                if (NB == 1 || b < a.B) atomicAdd(a.acc + b * N + r, acc0[b] + acc1[b]);
        }
    }
    if (bad || (bad_bits >> 31)) atomicExch(a.status, (int)DEV_CORRUPT);
}

template <int NB, bool PF>
cudaError_t launch_huff_nb(const HuffArgs &a, int64_t units, cudaStream_t st)
{
    static int per_sm[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!per_sm[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemv_huff_kernel<NB, PF>, cudaFuncAttributeMaxDynamicSharedMemorySize, kHSmem);
        if (e != cudaSuccess) return e;
        // ask for the smallest shared-memory carveout that holds the tables: the rest stays L1
        e = cudaFuncSetAttribute(gemv_huff_kernel<NB, PF>, cudaFuncAttributePreferredSharedMemoryCarveout, 25);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_huff_kernel<NB, PF>, huff_threads<NB>(), kHSmem);
        if (e != cudaSuccess) return e;
        per_sm[dev] = std::max(1, n);
    }
    const int64_t grid = std::min<int64_t>((int64_t)num_sms() * per_sm[dev], units);
    // warps per CTA: a unit is one warp's work and cannot be split, so a CTA's units should fill whole rounds of
    // its warps (47 units per SM on the 8B gate_proj: 1.97 rounds of 24 warps; 32 warps would leave the second
    // of 1.47 rounds half empty).  Of 24 and 16 warps the one with the fuller last round wins; a tie (within 2%)
    // goes to more warps.
    const int64_t per_cta = (units + grid - 1) / grid;
    int warps = huff_threads<NB>() / 32;
    double best = -1.0;
    for (int w = huff_threads<NB>() / 32; w >= 16; w -= 8) {  // 24 or 16
        const double rounds = (double)per_cta / w, fill = rounds / std::ceil(rounds);
        if (fill > best + 0.02) { best = fill; warps = w; }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)(32 * warps));
    cfg.dynamicSmemBytes = kHSmem;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_huff_kernel<NB, PF>, a);
}

template <bool PF>
cudaError_t launch_huff_pf(const HuffArgs &a, int64_t B, cudaStream_t st)
{
    if (B <= 1) return launch_huff_nb<1, PF>(a, a.units, st);
    if (B <= 2) return launch_huff_nb<2, PF>(a, a.units, st);
    if (B <= 4) return launch_huff_nb<4, PF>(a, a.units, st);
    return launch_huff_nb<8, PF>(a, a.units, st);
}

}  // namespace

bool gemv_huff_supported(const DevView &v, int64_t B, int variant)
{
    if (variant < 0 || variant > 1) return false;
    if (B < 1 || B > 8 || !v.mtab || !v.bits || !v.chunk_off || v.N <= 0 || v.K <= 0) return false;
    if (v.chunk < 64 || v.chunk > 2048 || v.chunk % 64 || v.K % v.chunk) return false;
    if (v.K > (int64_t)INT32_MAX || v.N > (int64_t)INT32_MAX) return false;
    return true;
}

int launch_gemv_huff(const DevView &v, const uint16_t *x, int64_t B, void *y, int out_bf16, int variant, float *acc_ws,
                     void *stream)
{
    if (!gemv_huff_supported(v, B, variant)) return cudaErrorInvalidValue;
    cudaStream_t st = (cudaStream_t)stream;
    HuffArgs a;
    memset(&a, 0, sizeof a);
    a.sm = v.sm;
    a.bitmap = v.bitmap;
    a.prefix = v.prefix;
    a.verb_exp = v.verb_exp;
    a.chunk_off = v.chunk_off;
    a.bits = v.bits;
    a.mtab = v.mtab;
    a.x = x;
    a.acc = out_bf16 ? acc_ws : (float *)y;
    if (!a.acc || ((uintptr_t)a.acc & 15)) return cudaErrorInvalidValue;
    a.status = v.status;
    a.N = v.N;
    a.K = v.K;
    a.B = B;
    a.n_blocks = v.n_blocks;
    a.C = (int)v.chunk;
    a.cpr = (int)(v.K / v.chunk);
    a.units = (v.N + 31) / 32 * (int64_t)a.cpr;
    a.n_chunks = v.n_chunks;
    memcpy(a.palette, v.palette, 16);
    cudaError_t e = (cudaError_t)launch_zero_target(a.acc, B * v.N, st);
    if (e != cudaSuccess) return e;
    e = variant == 1 ? launch_huff_pf<true>(a, B, st) : launch_huff_pf<false>(a, B, st);
    if (e != cudaSuccess) return e;
    if (out_bf16) return launch_finalize(acc_ws, y, B * v.N, 1, stream);
    return cudaSuccess;
}

}  // namespace uw
