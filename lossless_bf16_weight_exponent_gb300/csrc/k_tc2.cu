// k_tc2.cu - fused reconstruct + tcgen05 GEMM with the rebuilt weights in tensor memory (sm_103a), B <= 256.
//
// Cloudflare blog "Unweight", section on the reconstructive matmul: the copy engine stages the compressed
// inputs, consumer threads rebuild BF16 on chip and the tensor cores consume it at once, so rebuilt weights
// never reach HBM.  The post's H100 kernel rebuilds into shared memory for WGMMA.  On Blackwell the MMA can
// read its A operand from tensor memory, so here each rebuild thread owns one weight row: it decodes the
// row's 64 weights of a K-stage in registers and writes them with one tcgen05.st into the row's TMEM lane.
// Shared memory then carries only the compressed bytes and the activations.
//
// One CTA owns 128 rows of W (the MMA's M) and a range of 64-wide K-stages.
//   - warp 16 (one thread) TMA-loads compressed stages of 256 weights per row as boxes 128 bytes wide with the
//     128-byte swizzle: sign+mantissa as two [128 x 128] u8 boxes and the 4-bit codes as one (or exponent
//     bytes, or the bf16 tile), so a warp's 32 rows read at once land in distinct bank groups;
//   - warp 17 (one thread) TMA-loads the activation tile X [BN x 64] bf16 of each K-stage (128-byte swizzle,
//     the MMA's K-major B operand);
//   - warps 0-15 rebuild: warp w belongs to group w / 4, which rebuilds K-stages i = w / 4 (mod 4), and owns
//     TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31, i.e. rows; the 64 weights become 32 bf16x2 columns of one
//     of eight A slots (TMEM columns 256 + 32 s .. 256 + 32 s + 31);
//   - warp 18 (one thread) issues four tcgen05.mma (M = 128, N = BN, K = 16, A from TMEM, B from shared
//     memory) per K-stage; tcgen05.commit frees the A slot and the X tile once they complete.  MMAs into one
//     accumulator run one after another, and at small N their latency, not their work, sets the pace, so
//     consecutive MMAs rotate over NACC = min(8, 256 / BN) fp32 accumulators (TMEM columns q BN .. q BN +
//     BN - 1) that run concurrently.
// Epilogue: warps 0-3 read and sum the accumulators with tcgen05.ld and write Y (or fp32 atomics when K is
// split).
// Verbatim blocks: before the main loop the CTA stages, per row, which of its K-stages are verbatim and
// copies those blocks' exponents (one contiguous run of the verbatim stream per row) into shared memory.
// Every wait is bounded; on expiry the kernel latches DEV_TIMEOUT, drains its copies and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "dev_async.cuh"
#include "uw_internal.h"

namespace uw {

namespace {

using namespace dev;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kCK = 256;                      // weights per row in one compressed stage (four K-stages)
constexpr int kGroups = 4;                    // rebuild groups: group q rebuilds K-stages i = q (mod 4)
constexpr int kRebuildWarps = 4 * kGroups;    // a group has one warp per TMEM lane quarter
constexpr int kProducerWarp = kRebuildWarps;  // compressed stages
constexpr int kXWarp = kRebuildWarps + 1;     // activation tiles
constexpr int kMmaWarp = kRebuildWarps + 2;   // MMA issue, TMEM allocation
constexpr int kThreads = 32 * (kRebuildWarps + 3);
constexpr int kMaxASlots = 15;                // rebuilt K-stages in TMEM, 32 columns each, after the accumulators
constexpr int kTmemCols = 512;
constexpr int kMaskWords = 8;                 // per-row verbatim masks: up to 256 K-stages per CTA

struct Tc2Args {
    CUtensorMap tm0;   // sm [N, K] u8, box {128, 128}, swizzle 128 B | W bf16 [N, K], box {64, 128}, swizzle 128 B
    CUtensorMap tm1;   // codes [N, K/2] u8, box {128, 128}, swizzle 128 B | exps [N, K] u8, box {128, 128}, swizzle 128 B
    CUtensorMap tm_x;  // X [B, K] bf16, box {64, BN}, swizzle 128 B
    const uint32_t *bitmap, *prefix;
    const uint8_t *verb_exp;
    void *y;
    float *acc;
    int *status;
    int64_t N, K, B;
    int BN, ks_stages, cstages, xstages, cstage_bytes, nsplit, out_bf16, vcap, nacc, aslots, acol0;
    uint8_t palette[16];
};

template <int FMT> struct CStage;
template <> struct CStage<FMT_PAL> { static constexpr uint32_t bytes = 3 * 128 * 128; };   // sm x2, codes
template <> struct CStage<FMT_EXP> { static constexpr uint32_t bytes = 4 * 128 * 128; };   // sm x2, exps x2
template <> struct CStage<FMT_BF16> { static constexpr uint32_t bytes = 4 * 128 * 128; };  // bf16 x4

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) tc2_kernel(const __grid_constant__ Tc2Args a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);  // the swizzled tiles need it
    constexpr int TB = FMT == FMT_PAL ? kPairTableBytes : 0;
    const int SC = a.cstages, SX = a.xstages;
    uint8_t *tab = smem;                                      // [TB] pair table
    uint64_t *cfull = (uint64_t *)(smem + TB);               // [SC] compressed stage landed
    uint64_t *cempty = cfull + SC;                            // [SC] both of its K-stages read
    uint64_t *xfull = cempty + SC;                            // [SX] X tile landed
    uint64_t *xempty = xfull + SX;                            // [SX] MMAs reading it completed
    const int SA = a.aslots;
    uint64_t *afull = xempty + SX;                            // [SA] A slot written
    uint64_t *aempty = afull + kMaxASlots;                    // [SA] MMAs reading it completed
    uint64_t *done = aempty + kMaxASlots;                     // all MMAs completed
    uint32_t *tmem_slot = (uint32_t *)(done + 1);
    // verbatim staging, per row: mask word w bit j = K-stage 32w + j is verbatim ([w][row], conflict-free
    // reads), the row's local index before word w, the row's first local index, its first stream index
    uint32_t *vmask = (uint32_t *)(smem + TB + 1024);         // [kMaskWords][BM]
    uint32_t *vpfx = vmask + kMaskWords * BM;                 // [kMaskWords][BM]
    uint32_t *vrow = vpfx + kMaskWords * BM;                  // [BM]
    uint32_t *vglob = vrow + BM;                              // [BM]
    uint8_t *vdata = (uint8_t *)(vglob + BM);                 // [vcap][64]
    const size_t vbytes = FMT == FMT_PAL ? (size_t)(2 * kMaskWords * BM + 2 * BM) * 4 + (size_t)a.vcap * 64 : 0;
    uint8_t *xring = smem + TB + 1024 + (vbytes + 1023) / 1024 * 1024;  // [SX][BN * 128]
    uint8_t *cring = xring + (size_t)SX * a.BN * 128;                   // [SC][cstage_bytes]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t N = a.N, K = a.K;
    const int64_t row0 = (int64_t)blockIdx.x * BM;
    const int k_stage0 = blockIdx.y * a.ks_stages;
    const int nks = (int)min((int64_t)a.ks_stages, K / BK - k_stage0);
    const int ncs = (nks + 3) / 4;
    const uint32_t x_bytes = (uint32_t)a.BN * 128;

    if (FMT == FMT_PAL) fill_pair_table(tab, a.palette, threadIdx.x, blockDim.x);
    if (threadIdx.x == 0) {
        for (int s = 0; s < SC; s++) {
            mbar_init(&cfull[s], 1);
            mbar_init(&cempty[s], 16);  // the four groups of its K-stages, four warps each
        }
        for (int s = 0; s < SX; s++) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], 1);
        }
        for (int s = 0; s < SA; s++) {
            mbar_init(&afull[s], 4);
            mbar_init(&aempty[s], 1);
        }
        mbar_init(done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == kProducerWarp) {
        // -------------------------------------------------------------------------------- compressed stages
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < ncs; c++) {
                const int s = c % SC;
                if (c >= SC && !mbar_wait(&cempty[s], ((c / SC) - 1) & 1)) { ok = false; break; }
                uint8_t *st = cring + (size_t)s * a.cstage_bytes;
                const int kw = k_stage0 * BK + c * kCK;  // first weight of the stage
                mbar_expect_tx(&cfull[s], CStage<FMT>::bytes);
                if (FMT == FMT_BF16) {
#pragma unroll
                    for (int j = 0; j < 4; j++) tma2d(st + j * 16384, &a.tm0, kw + j * BK, (int)row0, &cfull[s]);
                } else {
                    tma2d(st, &a.tm0, kw, (int)row0, &cfull[s]);
                    tma2d(st + 16384, &a.tm0, kw + 128, (int)row0, &cfull[s]);
                    if (FMT == FMT_PAL) tma2d(st + 32768, &a.tm1, kw / 2, (int)row0, &cfull[s]);
                    else {
                        tma2d(st + 32768, &a.tm1, kw, (int)row0, &cfull[s]);
                        tma2d(st + 49152, &a.tm1, kw + 128, (int)row0, &cfull[s]);
                    }
                }
                issued = c + 1;
            }
            if (!ok) {
                atomicExch(a.status, (int)DEV_TIMEOUT);
                for (int c = max(0, issued - SC); c < issued; c++) mbar_wait(&cfull[c % SC], (c / SC) & 1);
            }
        }
    } else if (warp == kXWarp) {
        // -------------------------------------------------------------------------------- activation tiles
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nks; i++) {
                const int s = i % SX;
                if (i >= SX && !mbar_wait(&xempty[s], ((i / SX) - 1) & 1)) { ok = false; break; }
                mbar_expect_tx(&xfull[s], x_bytes);
                tma2d(xring + (size_t)s * a.BN * 128, &a.tm_x, (k_stage0 + i) * BK, 0, &xfull[s]);
                issued = i + 1;
            }
            if (!ok) {
                atomicExch(a.status, (int)DEV_TIMEOUT);
                for (int i = max(0, issued - SX); i < issued; i++) mbar_wait(&xfull[i % SX], (i / SX) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t id = idesc_bf16(BM, a.BN);
            const int nacc = a.nacc;
            int q = 0;  // accumulator of the next MMA
            for (int i = 0; i < nks; i++) {
                const int sa = i % SA, sx = i % SX;
                if (!mbar_wait(&afull[sa], (i / SA) & 1) || !mbar_wait(&xfull[sx], (i / SX) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_tmem = tmem + a.acol0 + 32 * sa;
                const uint32_t x_base = saddr(xring + (size_t)sx * a.BN * 128);
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++) {
                    const int n = 4 * i + kk;  // MMAs issued so far: the first nacc initialise their accumulators
                    mma_ts(tmem + (uint32_t)(q * a.BN), a_tmem + 8 * kk, smem_desc_sw128(x_base + 32 * kk), id,
                           n >= nacc ? 1u : 0u);
                    q = q + 1 == nacc ? 0 : q + 1;
                }
                mma_commit(&aempty[sa]);
                mma_commit(&xempty[sx]);
            }
            if (!ok) atomicExch(a.status, (int)DEV_TIMEOUT);
            mma_commit(done);  // arrives once every MMA issued above has completed
        }
    } else {
        // -------------------------------------------------------------------------------- rebuild (warps 0-15)
        const int group = warp >> 2, quarter = warp & 3;
        const int r = 32 * quarter + lane;  // the row (TMEM lane) this thread rebuilds
        const uint8_t *tab_lane = tab + 4 * lane;
        if (FMT == FMT_PAL) {
            // --- stage the tile's verbatim information (overlaps the producers' first loads)
            const int tid = threadIdx.x;  // 0..511
            uint32_t cnt = 0;
            if (tid < BM) {
                const int64_t row = row0 + tid;
                if (row < N) {
                    const uint64_t fb = (uint64_t)row * (uint64_t)(K / BK) + (uint64_t)k_stage0;
                    uint32_t lo[kMaskWords + 1];
#pragma unroll
                    for (int w = 0; w <= kMaskWords; w++)  // all loads first: one round trip
                        lo[w] = 32 * w < nks + 32 ? __ldg(a.bitmap + (fb >> 5) + w) : 0u;
                    const uint32_t pf0 = __ldg(a.prefix + (fb >> 5));
#pragma unroll
                    for (int w = 0; w < kMaskWords; w++) {
                        uint32_t m = 0;
                        const int first = 32 * w;
                        if (first < nks) {
                            m = (uint32_t)((((uint64_t)lo[w + 1] << 32) | lo[w]) >> (fb & 31));
                            const int valid = nks - first;
                            if (valid < 32) m &= (1u << valid) - 1u;
                        }
                        vmask[w * BM + tid] = m;
                        vpfx[w * BM + tid] = cnt;  // local count before this word (row-relative)
                        cnt += __popc(m);
                    }
                    vglob[tid] = pf0 + __popc(lo[0] & ((1u << (fb & 31)) - 1u));
                } else {
#pragma unroll
                    for (int w = 0; w < kMaskWords; w++) vmask[w * BM + tid] = vpfx[w * BM + tid] = 0;
                    vglob[tid] = 0;
                }
                vrow[tid] = cnt;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kRebuildWarps) : "memory");
            if (warp == 0) {  // exclusive scan of the per-row counts
                uint32_t c4[4], sum = 0;
#pragma unroll
                for (int q = 0; q < 4; q++) { c4[q] = vrow[4 * lane + q]; sum += c4[q]; }
                uint32_t incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += t;
                }
                uint32_t run = incl - sum;
#pragma unroll
                for (int q = 0; q < 4; q++) { vrow[4 * lane + q] = run; run += c4[q]; }
            }
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kRebuildWarps) : "memory");
            // copy each row's run of verbatim exponents (contiguous in the stream) into shared memory
            for (int rr = warp; rr < BM; rr += kRebuildWarps) {
                const uint32_t base = vrow[rr];
                const uint32_t n = (rr + 1 < BM ? vrow[rr + 1]
                                                : base + vpfx[(kMaskWords - 1) * BM + rr] +
                                                      __popc(vmask[(kMaskWords - 1) * BM + rr])) - base;
                const uint4 *src = (const uint4 *)(a.verb_exp + (uint64_t)vglob[rr] * 64);
                for (uint32_t q = lane; q < n * 4; q += 32)
                    if (base + q / 4 < (uint32_t)a.vcap) ((uint4 *)(vdata + (uint64_t)base * 64))[q] = __ldg(src + q);
            }
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kRebuildWarps) : "memory");
        }
        const uint32_t t_lane = (uint32_t)(32 * quarter) << 16;
        for (int i = group; i < nks; i += kGroups) {
            const int c = i >> 2, sub = i & 3, cs = c % SC, sa = i % SA;
            if (!mbar_wait(&cfull[cs], (c / SC) & 1)) { ok = false; break; }
            const uint8_t *cst = cring + (size_t)cs * a.cstage_bytes;
            uint4 d0[4], d1[4];  // PAL: sm pieces, codes (d1[0..1]); EXP: sm, exps; BF16: the 8 pieces
            if (FMT == FMT_BF16) {
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    d0[p] = *(const uint4 *)(cst + sub * 16384 + r * 128 + ((p ^ (r & 7)) << 4));
                    d1[p] = *(const uint4 *)(cst + sub * 16384 + r * 128 + (((p + 4) ^ (r & 7)) << 4));
                }
            } else {
                // sm box h = sub / 2 holds K-stages 2h, 2h + 1: this one is its half q = sub % 2
                const int h = sub >> 1, q = sub & 1;
#pragma unroll
                for (int p = 0; p < 4; p++)
                    d0[p] = *(const uint4 *)(cst + h * 16384 + r * 128 + (((4 * q + p) ^ (r & 7)) << 4));
                if (FMT == FMT_PAL) {
                    // the codes box holds all four K-stages: 32 code bytes each
#pragma unroll
                    for (int p = 0; p < 2; p++)
                        d1[p] = *(const uint4 *)(cst + 32768 + r * 128 + (((2 * sub + p) ^ (r & 7)) << 4));
                } else {
#pragma unroll
                    for (int p = 0; p < 4; p++)
                        d1[p] = *(const uint4 *)(cst + 32768 + h * 16384 + r * 128 + (((4 * q + p) ^ (r & 7)) << 4));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&cempty[cs]);  // the stage's bytes are in registers
            if (i >= SA && !mbar_wait(&aempty[sa], ((i / SA) - 1) & 1)) { ok = false; break; }
            uint32_t v[32];  // the row's 64 weights of K-stage i as bf16x2 pairs
            if (FMT == FMT_PAL) {
                const uint32_t m = vmask[(i >> 5) * BM + r];
                if (__builtin_expect((m >> (i & 31)) & 1u, 0)) {
                    const uint32_t li = vrow[r] + vpfx[(i >> 5) * BM + r] + __popc(m & ((1u << (i & 31)) - 1u));
                    const uint64_t gi = (uint64_t)vglob[r] + (li - vrow[r]);
#pragma unroll
                    for (int p = 0; p < 4; p++) {
                        const uint4 ev = li < (uint32_t)a.vcap ? *(const uint4 *)(vdata + (uint64_t)li * 64 + 16 * p)
                                                                : __ldg((const uint4 *)(a.verb_exp + gi * 64 + 16 * p));
#pragma unroll
                        for (int q = 0; q < 4; q++)
                            pairs_from_exps(word_of(d0[p], q), word_of(ev, q), v[8 * p + 2 * q], v[8 * p + 2 * q + 1]);
                    }
                } else {
#pragma unroll
                    for (int p = 0; p < 4; p++)
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            // weights 4wq .. 4wq + 3: their codes are bytes 2wq, 2wq + 1 of the row's 32 code bytes
                            const int wq = 4 * p + q;
                            const uint32_t Cw = word_of(d1[wq >> 3], (wq >> 1) & 3);
                            const int jb = 2 * (wq & 1);
                            const uint32_t S = word_of(d0[p], q);
                            v[2 * wq] = (__byte_perm(S, 0u, 0x1100u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb);
                            v[2 * wq + 1] = (__byte_perm(S, 0u, 0x3322u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb + 1);
                        }
                }
            } else if (FMT == FMT_EXP) {
#pragma unroll
                for (int p = 0; p < 4; p++)
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        pairs_from_exps(word_of(d0[p], q), word_of(d1[p], q), v[8 * p + 2 * q], v[8 * p + 2 * q + 1]);
            } else {
#pragma unroll
                for (int p = 0; p < 4; p++)
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        v[4 * p + q] = word_of(d0[p], q);
                        v[16 + 4 * p + q] = word_of(d1[p], q);
                    }
            }
            tmem_st32(tmem + t_lane + a.acol0 + 32 * sa, v);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[sa]);
        }
        if (!ok) atomicExch(a.status, (int)DEV_TIMEOUT);
    }

    // ------------------------------------------------------------------------------------ epilogue (warps 0-3)
    if (warp < 4) {
        const bool got = mbar_wait(done, 0);
        if (!got) atomicExch(a.status, (int)DEV_TIMEOUT);
        tc_fence_after();
        const int64_t row = row0 + 32 * warp + lane;
        // accumulators that received no MMA (fewer MMAs than accumulators) hold no data: skip them
        const int nused = min(a.nacc, 4 * nks);
        for (int c0 = 0; c0 < a.BN && c0 < a.B; c0 += 16) {
            float f16[16];
#pragma unroll
            for (int t = 0; t < 16; t++) f16[t] = 0.f;
            for (int q = 0; q < nused; q++) {
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(q * a.BN + c0), v);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; t++) f16[t] += __uint_as_float(v[t]);
            }
            if (got && row < N) {
#pragma unroll
                for (int t = 0; t < 16; t++) {
                    const int64_t b = c0 + t;
                    if (b < a.B) {
                        const int64_t o = b * N + row;
                        const float f = f16[t];
                        if (a.nsplit > 1) atomicAdd(a.acc + o, f);
                        else if (a.out_bf16) ((__nv_bfloat16 *)a.y)[o] = __float2bfloat16_rn(f);
                        else ((float *)a.y)[o] = f;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------------------------- host side
bool make_map2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
                uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw)
{
    auto fn = (PFN_cuTensorMapEncodeTiled_v12000)tensor_map_encoder();
    if (!fn || !base || ((uintptr_t)base & 15)) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Tc2Shape {
    int BN, cstages, xstages, cstage_bytes, ks_stages, nsplit, vcap, nacc, aslots, acol0;
    size_t smem;
};

bool tc2_shape(const WOperand &w, int64_t B, int split_k, Tc2Shape &s)
{
    if (B < 1 || B > 256 || w.N <= 0 || w.K < BK || w.K % BK) return false;
    if (w.N > (int64_t)INT32_MAX || w.K > (int64_t)INT32_MAX) return false;
    s.BN = (int)((B + 15) / 16 * 16);
    // one accumulator at columns [0, BN) (rotating over several did not help); eight A slots after it
    s.nacc = 1;
    s.acol0 = (s.BN + 31) / 32 * 32;
    s.aslots = std::min(8, (kTmemCols - s.acol0) / 32);
    s.cstage_bytes = w.fmt == FMT_PAL ? (int)CStage<FMT_PAL>::bytes : (int)CStage<FMT_EXP>::bytes;
    // activation tiles are small but each carries a full memory latency: keep ~16 KB of them in flight
    s.xstages = std::max(2, std::min(8, (16 * 1024) / (s.BN * 128)));
    const size_t cap = 227 * 1024;
    const bool pal = w.fmt == FMT_PAL;
    s.vcap = pal ? 128 : 0;
    const size_t vbytes = pal ? (size_t)(2 * kMaskWords * BM + 2 * BM) * 4 + (size_t)s.vcap * 64 : 0;
    const size_t fixed = 1024 /* alignment slack */ + (pal ? kPairTableBytes : 0) + 1024 + (vbytes + 1023) / 1024 * 1024 +
                         (size_t)s.xstages * s.BN * 128;
    if (fixed + 2 * (size_t)s.cstage_bytes > cap) return false;
    s.cstages = (int)std::min<size_t>(8, (cap - fixed) / s.cstage_bytes);
    s.smem = fixed + (size_t)s.cstages * s.cstage_bytes;
    const int64_t tiles = (w.N + BM - 1) / BM;
    const int kst = (int)(w.K / BK);
    int split = std::max(split_k, (kst + 32 * kMaskWords - 1) / (32 * kMaskWords));  // <= 256 K-stages per CTA
    if (split_k <= 0) {
        // the split with the best wave efficiency (one CTA per SM), at least 8 K-stages per CTA
        const int64_t slots = num_sms();
        double best = -1;
        const int min_split = split;
        for (int sp = min_split; sp <= std::max(16, min_split); sp++) {
            if (kst / sp < 8 && sp > min_split) break;
            const int64_t ctas = tiles * sp;
            const int64_t waves = (ctas + slots - 1) / slots;
            const double eff = (double)ctas / (double)(waves * slots) - 0.02 * (sp - 1);
            if (eff > best + 1e-9) { best = eff; split = sp; }
        }
    }
    s.ks_stages = (kst + split - 1) / split;
    s.nsplit = (kst + s.ks_stages - 1) / s.ks_stages;
    return true;
}

template <int FMT>
cudaError_t launch2_fmt(const Tc2Args &a, dim3 grid, size_t smem, cudaStream_t st)
{
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tc2_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    tc2_kernel<FMT><<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool tc2_supported(const WOperand &w, int64_t B)
{
    Tc2Shape s;
    return tensor_map_encoder() != nullptr && tc2_shape(w, B, 0, s);
}

int tc2_default_split(const WOperand &w, int64_t B)
{
    Tc2Shape s;
    return tc2_shape(w, B, 0, s) ? s.nsplit : 1;
}

int launch_tc2(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, int split_k, float *acc_ws,
               void *stream)
{
    Tc2Shape s;
    if (!tc2_shape(w, B, split_k, s)) return cudaErrorInvalidValue;
    cudaStream_t st = (cudaStream_t)stream;
    Tc2Args a;
    memset(&a, 0, sizeof a);
    const uint64_t N = (uint64_t)w.N, K = (uint64_t)w.K;
    bool ok = true;
    if (w.fmt == FMT_BF16) {
        ok &= make_map2d(&a.tm0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w.w, K, N, K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
        ok &= make_map2d(&a.tm0, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.sm, K, N, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
        if (w.fmt == FMT_PAL)
            ok &= make_map2d(&a.tm1, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, K / 2, N, K / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
        else
            ok &= make_map2d(&a.tm1, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.exps, K, N, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    ok &= make_map2d(&a.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, (uint64_t)B, K * 2, 64, (uint32_t)s.BN,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;
    a.bitmap = w.bitmap;
    a.prefix = w.prefix;
    a.verb_exp = w.verb_exp;
    a.y = y;
    a.status = w.status;
    a.N = w.N;
    a.K = w.K;
    a.B = B;
    a.BN = s.BN;
    a.ks_stages = s.ks_stages;
    a.cstages = s.cstages;
    a.xstages = s.xstages;
    a.cstage_bytes = s.cstage_bytes;
    a.nsplit = s.nsplit;
    a.out_bf16 = out_bf16;
    a.vcap = s.vcap;
    a.nacc = s.nacc;
    a.aslots = s.aslots;
    a.acol0 = s.acol0;
    memcpy(a.palette, w.palette, 16);
    if (s.nsplit > 1) {
        a.acc = out_bf16 ? acc_ws : (float *)y;
        if (!a.acc) return cudaErrorInvalidValue;
        cudaError_t e = cudaMemsetAsync(a.acc, 0, (size_t)B * N * 4, st);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)((N + BM - 1) / BM), (unsigned)s.nsplit);
    cudaError_t e;
    if (w.fmt == FMT_PAL) e = launch2_fmt<FMT_PAL>(a, grid, s.smem, st);
    else if (w.fmt == FMT_EXP) e = launch2_fmt<FMT_EXP>(a, grid, s.smem, st);
    else e = launch2_fmt<FMT_BF16>(a, grid, s.smem, st);
    if (e != cudaSuccess) return e;
    if (s.nsplit > 1 && out_bf16) return launch_finalize(acc_ws, y, B * w.N, 1, stream);
    return cudaSuccess;
}

}  // namespace uw
