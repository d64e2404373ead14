// k_tc3.cu - persistent fused reconstruct + tcgen05 GEMM, rebuilt weights in tensor memory (sm_103a), B <= 256.
//
// Cloudflare blog "Unweight", section on the reconstructive matmul: compressed inputs are staged by the copy
// engine, rebuilt on chip and consumed by the tensor cores at once.  This kernel keeps the copy engine busy
// for the whole launch: one CTA per SM walks a balanced, contiguous range of work units (a unit is 128 rows of
// W x 256 weights of K, four 64-wide K-stages), crossing tile boundaries, so there are no waves, no per-tile
// prologue and no pipeline drain between tiles.  The verbatim side information of a unit (which of its blocks
// are verbatim, and their exponents) comes from the tile-major verbatim stream built at load time and travels
// with the unit's compressed bytes, so no staging pass precedes the main loop.
//
//   - warp 16 (one thread, the warp's lanes prefetch offsets) TMA-loads per unit: two sign+mantissa boxes
//     [128 rows x 128 B] and one code box [128 x 128 B], all with the 128-byte swizzle (or exponent / bf16
//     boxes), plus the unit's 64-byte verbatim mask and up to VC verbatim blocks by bulk copy;
//   - warp 17 (one thread) TMA-loads the activation tile X [BN x 64] of each K-stage;
//   - warps 0-15: group g = warp / 4 rebuilds K-stage g of every unit; warp w owns TMEM lanes (rows)
//     32 (w % 4) .. 32 (w % 4) + 31; each thread decodes its row's 64 weights and stores them with one
//     tcgen05.st into one of eight A slots;
//   - warp 18 (one thread) issues the MMAs (M = 128, N = BN, K = 16, A from TMEM, B = X from shared memory)
//     into the accumulator of the current segment (a segment is a run of units of one tile); two accumulator
//     buffers when they fit, so a segment's results are read while the next one accumulates;
//   - the four warps of group 0 write a finished segment: tcgen05.ld, fp32 atomics into the zeroed output.
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
constexpr int kUnitK = 256;                   // weights of K per unit (four K-stages)
constexpr int kRebuildWarps = 16;             // four groups, one warp per TMEM lane quarter
constexpr int kProducerWarp = kRebuildWarps;
constexpr int kXWarp = kRebuildWarps + 1;
constexpr int kMmaWarp = kRebuildWarps + 2;
constexpr int kThreads = 32 * (kRebuildWarps + 3);
constexpr int kASlots = 8;
constexpr int kTmemCols = 512;
constexpr int kVC = 32;                       // verbatim blocks of a unit staged with it (beyond: global loads)
constexpr int kVSlot = 64 + kVC * 64;         // mask + staged blocks

struct Tc3Args {
    CUtensorMap tm0;   // sm [N, K] u8 box {128, 128} | W bf16 [N, K] box {64, 128}; swizzle 128 B
    CUtensorMap tm1;   // codes [N, K/2] u8 box {128, 128} | exps [N, K] u8 box {128, 128}; swizzle 128 B
    CUtensorMap tm_x;  // X [B, K] bf16 box {64, BN}, swizzle 128 B
    const uint32_t *tmv_off, *tmv_mask;
    const uint8_t *tmv_data;
    float *acc;        // [B, N] fp32, zeroed before the launch; segments add into it
    int *status;
    int64_t N, K, B;
    int BN, cstages, xstages, cstage_bytes, upk, nbuf, acol0;
    int64_t units;
    uint8_t palette[16];
};

template <int FMT> struct CStage3;
template <> struct CStage3<FMT_PAL> { static constexpr uint32_t bytes = 3 * 128 * 128; };   // sm x2, codes
template <> struct CStage3<FMT_EXP> { static constexpr uint32_t bytes = 4 * 128 * 128; };   // sm x2, exps x2
template <> struct CStage3<FMT_BF16> { static constexpr uint32_t bytes = 4 * 128 * 128; };  // bf16 x4

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) tc3_kernel(const __grid_constant__ Tc3Args a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    constexpr int TB = FMT == FMT_PAL ? kPairTableBytes : 0;
    const int SC = a.cstages, SX = a.xstages;
    uint8_t *tab = smem;
    uint64_t *cfull = (uint64_t *)(smem + TB);   // [SC]
    uint64_t *cempty = cfull + SC;                // [SC] the four groups have read the unit
    uint64_t *xfull = cempty + SC;                // [SX]
    uint64_t *xempty = xfull + SX;                // [SX]
    uint64_t *afull = xempty + SX;                // [kASlots]
    uint64_t *aempty = afull + kASlots;           // [kASlots]
    uint64_t *accfull = aempty + kASlots;         // [2] a segment's MMAs completed
    uint64_t *accempty = accfull + 2;             // [2] its accumulator was read
    uint32_t *tmem_slot = (uint32_t *)(accempty + 2);
    uint8_t *vring = smem + TB + 1024;                                          // [SC][kVSlot] (FMT_PAL)
    const size_t vbytes = FMT == FMT_PAL ? (size_t)SC * kVSlot : 0;
    uint8_t *xring = smem + TB + 1024 + (vbytes + 1023) / 1024 * 1024;          // [SX][BN * 128]
    uint8_t *cring = xring + (size_t)SX * a.BN * 128;                           // [SC][cstage_bytes]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t N = a.N;
    const int64_t U = a.units, G = gridDim.x;
    const int64_t u0 = U * blockIdx.x / G, u1 = U * (blockIdx.x + 1) / G;
    const int nu = (int)(u1 - u0);
    const int nks = 4 * nu;
    const int upk = a.upk;
    const uint32_t x_bytes = (uint32_t)a.BN * 128;

    if (FMT == FMT_PAL) fill_pair_table(tab, a.palette, threadIdx.x, blockDim.x);
    if (threadIdx.x == 0) {
        for (int s = 0; s < SC; s++) {
            mbar_init(&cfull[s], 1);
            mbar_init(&cempty[s], 16);
        }
        for (int s = 0; s < SX; s++) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], 1);
        }
        for (int s = 0; s < kASlots; s++) {
            mbar_init(&afull[s], 4);
            mbar_init(&aempty[s], 1);
        }
        for (int s = 0; s < 2; s++) {
            mbar_init(&accfull[s], 1);
            mbar_init(&accempty[s], 4);
        }
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
        // -------------------------------------------------------------------------------- units
        uint32_t o0 = 0, o1 = 0;  // lane l: verbatim offsets of unit u0 + 32 * window + l and the next one
        int issued = 0;
        for (int c = 0; c < nu; c++) {
            const int s = c % SC;
            const int64_t u = u0 + c;
            if (FMT == FMT_PAL && (c & 31) == 0) {
                const int64_t ul = u + lane;
                o0 = ul <= U ? __ldg(a.tmv_off + ul) : 0u;
                o1 = ul + 1 <= U ? __ldg(a.tmv_off + ul + 1) : 0u;
            }
            const uint32_t start = __shfl_sync(0xFFFFFFFFu, o0, c & 31);
            const uint32_t nv = min(__shfl_sync(0xFFFFFFFFu, o1, c & 31) - start, (uint32_t)kVC);
            int go = 1;
            if (lane == 0) {
                if (c >= SC && !mbar_wait(&cempty[s], ((c / SC) - 1) & 1)) go = 0;
                else {
                    const int t = (int)(u / upk), kq = (int)(u % upk);
                    const int kw = kq * kUnitK, row0 = t * BM;
                    uint8_t *st = cring + (size_t)s * a.cstage_bytes;
                    mbar_expect_tx(&cfull[s], CStage3<FMT>::bytes + (FMT == FMT_PAL ? 64u + 64u * nv : 0u));
                    if (FMT == FMT_BF16) {
#pragma unroll
                        for (int j = 0; j < 4; j++) tma2d(st + j * 16384, &a.tm0, kw + j * BK, row0, &cfull[s]);
                    } else {
                        tma2d(st, &a.tm0, kw, row0, &cfull[s]);
                        tma2d(st + 16384, &a.tm0, kw + 128, row0, &cfull[s]);
                        if (FMT == FMT_PAL) {
                            tma2d(st + 32768, &a.tm1, kw / 2, row0, &cfull[s]);
                            uint8_t *vs = vring + (size_t)s * kVSlot;
                            asm volatile(
                                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 64, [%2];" ::"r"(
                                    saddr(vs)),
                                "l"(a.tmv_mask + 16 * u), "r"(saddr(&cfull[s]))
                                : "memory");
                            if (nv)
                                asm volatile(
                                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                        saddr(vs + 64)),
                                    "l"(a.tmv_data + (uint64_t)start * 64), "r"(nv * 64u), "r"(saddr(&cfull[s]))
                                    : "memory");
                        } else {
                            tma2d(st + 32768, &a.tm1, kw, row0, &cfull[s]);
                            tma2d(st + 49152, &a.tm1, kw + 128, row0, &cfull[s]);
                        }
                    }
                }
            }
            if (!__shfl_sync(0xFFFFFFFFu, go, 0)) { ok = false; break; }
            issued = c + 1;
        }
        if (lane == 0 && !ok) {
            atomicExch(a.status, (int)DEV_TIMEOUT);
            for (int c = max(0, issued - SC); c < issued; c++) mbar_wait(&cfull[c % SC], (c / SC) & 1);
        }
    } else if (warp == kXWarp) {
        // -------------------------------------------------------------------------------- activation tiles
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nks; i++) {
                const int s = i % SX;
                if (i >= SX && !mbar_wait(&xempty[s], ((i / SX) - 1) & 1)) { ok = false; break; }
                const int64_t u = u0 + (i >> 2);
                const int kstage = (int)(u % upk) * 4 + (i & 3);
                mbar_expect_tx(&xfull[s], x_bytes);
                tma2d(xring + (size_t)s * a.BN * 128, &a.tm_x, kstage * BK, 0, &xfull[s]);
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
            int seg = -1, ab = 0;
            int64_t prev_t = -1;
            for (int c = 0; c < nu && ok; c++) {
                const int64_t t = (u0 + c) / upk;
                bool first = false;
                if (t != prev_t) {  // a new segment: its accumulator buffer must have been read out
                    seg++;
                    ab = seg % a.nbuf;
                    if (seg >= a.nbuf && !mbar_wait(&accempty[ab], ((seg / a.nbuf) - 1) & 1)) { ok = false; break; }
                    first = true;
                    prev_t = t;
                }
                for (int j = 0; j < 4; j++) {
                    const int i = 4 * c + j, sa = i % kASlots, sx = i % SX;
                    if (!mbar_wait(&afull[sa], (i / kASlots) & 1) || !mbar_wait(&xfull[sx], (i / SX) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tmem = tmem + a.acol0 + 32 * sa;
                    const uint32_t x_base = saddr(xring + (size_t)sx * a.BN * 128);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; kk++)
                        mma_ts(tmem + (uint32_t)(ab * a.BN), a_tmem + 8 * kk, smem_desc_sw128(x_base + 32 * kk), id,
                               (first && j == 0 && kk == 0) ? 0u : 1u);
                    mma_commit(&aempty[sa]);
                    mma_commit(&xempty[sx]);
                }
                const bool last = c + 1 == nu || (u0 + c + 1) / upk != t;
                if (ok && last) mma_commit(&accfull[ab]);
            }
            if (!ok) {
                atomicExch(a.status, (int)DEV_TIMEOUT);
                // let the epilogue finish: every segment's completion barrier must still arrive once
                mma_commit(&accfull[0]);
                mma_commit(&accfull[1]);
            }
        }
    } else {
        // -------------------------------------------------------------------------------- rebuild (warps 0-15)
        const int group = warp >> 2, quarter = warp & 3;
        const int r = 32 * quarter + lane;
        const uint8_t *tab_lane = tab + 4 * lane;
        const uint32_t t_lane = (uint32_t)(32 * quarter) << 16;
        int seg = -1;
        int64_t prev_t = -1, seg_t = -1;
        // group 0 writes out a finished segment: wait for its MMAs, read the accumulator, add into the output
        auto write_segment = [&](int sg, int64_t tile) {
            const int buf = sg % a.nbuf;
            const bool got = mbar_wait(&accfull[buf], (sg / a.nbuf) & 1);
            if (!got) atomicExch(a.status, (int)DEV_TIMEOUT);
            tc_fence_after();
            const int64_t row = tile * BM + r;
            for (int c0 = 0; c0 < a.BN && c0 < a.B; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + t_lane + (uint32_t)(buf * a.BN + c0), v);
                tmem_wait_ld();
                if (got && row < N) {
#pragma unroll
                    for (int q = 0; q < 16; q++)
                        if (c0 + q < a.B) atomicAdd(a.acc + (int64_t)(c0 + q) * N + row, __uint_as_float(v[q]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accempty[buf]);
        };
        for (int c = 0; c < nu; c++) {
            const int64_t u = u0 + c;
            const int64_t t = u / upk;
            if (t != prev_t) {
                if (group == 0 && seg >= 0) write_segment(seg, seg_t);
                seg++;
                seg_t = t;
                prev_t = t;
            }
            const int i = 4 * c + group, cs = c % SC, sa = i % kASlots;
            if (!mbar_wait(&cfull[cs], (c / SC) & 1)) { ok = false; break; }
            const uint8_t *cst = cring + (size_t)cs * a.cstage_bytes;
            uint4 d0[4], d1[4];
            uint4 ev[4];
            bool verb = false;
            if (FMT == FMT_BF16) {
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    d0[p] = *(const uint4 *)(cst + group * 16384 + r * 128 + ((p ^ (r & 7)) << 4));
                    d1[p] = *(const uint4 *)(cst + group * 16384 + r * 128 + (((p + 4) ^ (r & 7)) << 4));
                }
            } else {
                const int h = group >> 1, q = group & 1;
#pragma unroll
                for (int p = 0; p < 4; p++)
                    d0[p] = *(const uint4 *)(cst + h * 16384 + r * 128 + (((4 * q + p) ^ (r & 7)) << 4));
                if (FMT == FMT_PAL) {
#pragma unroll
                    for (int p = 0; p < 2; p++)
                        d1[p] = *(const uint4 *)(cst + 32768 + r * 128 + (((2 * group + p) ^ (r & 7)) << 4));
                    // verbatim: mask words [K-stage][row word]; rank = blocks before (group, r) in the unit
                    const uint32_t *mk = (const uint32_t *)(vring + (size_t)cs * kVSlot);
                    const uint32_t m = mk[4 * group + quarter];
                    if (__builtin_expect((m >> lane) & 1u, 0)) {
                        verb = true;
                        uint32_t rank = __popc(m & ((1u << lane) - 1u));
                        for (int w = 0; w < 4 * group + quarter; w++) rank += __popc(mk[w]);
                        if (rank < (uint32_t)kVC) {
#pragma unroll
                            for (int p = 0; p < 4; p++)
                                ev[p] = *(const uint4 *)(vring + (size_t)cs * kVSlot + 64 + rank * 64 + 16 * p);
                        } else {
                            const uint64_t gi = (uint64_t)__ldg(a.tmv_off + u) + rank;
#pragma unroll
                            for (int p = 0; p < 4; p++) ev[p] = __ldg((const uint4 *)(a.tmv_data + gi * 64 + 16 * p));
                        }
                    }
                } else {
#pragma unroll
                    for (int p = 0; p < 4; p++)
                        d1[p] = *(const uint4 *)(cst + 32768 + h * 16384 + r * 128 + (((4 * q + p) ^ (r & 7)) << 4));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&cempty[cs]);  // the unit's bytes this warp needs are in registers
            if (i >= kASlots && !mbar_wait(&aempty[sa], ((i / kASlots) - 1) & 1)) { ok = false; break; }
            uint32_t v[32];
            if (FMT == FMT_PAL) {
                if (verb) {
#pragma unroll
                    for (int p = 0; p < 4; p++)
#pragma unroll
                        for (int q = 0; q < 4; q++)
                            pairs_from_exps(word_of(d0[p], q), word_of(ev[p], q), v[8 * p + 2 * q], v[8 * p + 2 * q + 1]);
                } else {
#pragma unroll
                    for (int p = 0; p < 4; p++)
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const int wq = 4 * p + q;  // weights 4wq .. 4wq + 3: code bytes 2wq, 2wq + 1
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
        if (group == 0 && seg >= 0) write_segment(seg, seg_t);
        if (!ok) atomicExch(a.status, (int)DEV_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

bool make_map3(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer)
{
    auto fn = (PFN_cuTensorMapEncodeTiled_v12000)tensor_map_encoder();
    if (!fn || !base || ((uintptr_t)base & 15)) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Tc3Shape {
    int BN, cstages, xstages, cstage_bytes, nbuf, acol0;
    int64_t units;
    size_t smem;
};

bool tc3_shape(const WOperand &w, int64_t B, Tc3Shape &s)
{
    if (B < 1 || B > 256 || w.N <= 0 || w.K <= 0 || w.K % kUnitK) return false;
    if (w.N > (int64_t)INT32_MAX || w.K > (int64_t)INT32_MAX) return false;
    if (w.fmt == FMT_PAL && (!w.tmv_off || !w.tmv_mask || !w.tmv_data)) return false;
    s.BN = (int)((B + 15) / 16 * 16);
    s.nbuf = 2 * s.BN <= 256 ? 2 : 1;
    s.acol0 = (s.nbuf * s.BN + 31) / 32 * 32;
    if (s.acol0 + 32 * kASlots > kTmemCols) return false;
    s.cstage_bytes = w.fmt == FMT_PAL ? (int)CStage3<FMT_PAL>::bytes : (int)CStage3<FMT_EXP>::bytes;
    s.xstages = std::max(2, std::min(8, (16 * 1024) / (s.BN * 128)));
    const size_t cap = 227 * 1024;
    const bool pal = w.fmt == FMT_PAL;
    // stages: as many as fit (at most 6), counting the staged verbatim slot of each
    for (s.cstages = 6; s.cstages >= 2; s.cstages--) {
        const size_t v = pal ? ((size_t)s.cstages * kVSlot + 1023) / 1024 * 1024 : 0;
        const size_t need = 1024 + (pal ? kPairTableBytes : 0) + 1024 + v + (size_t)s.xstages * s.BN * 128 +
                            (size_t)s.cstages * s.cstage_bytes;
        if (need <= cap) { s.smem = need; break; }
    }
    if (s.cstages < 2) return false;
    s.units = (w.N + BM - 1) / BM * (w.K / kUnitK);
    return true;
}

template <int FMT>
cudaError_t launch3_fmt(const Tc3Args &a, int grid, size_t smem, cudaStream_t st)
{
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tc3_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    tc3_kernel<FMT><<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool tc3_supported(const WOperand &w, int64_t B)
{
    Tc3Shape s;
    return tensor_map_encoder() != nullptr && tc3_shape(w, B, s);
}

int launch_tc3(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, float *acc_ws, void *stream)
{
    Tc3Shape s;
    if (!tc3_shape(w, B, s)) return cudaErrorInvalidValue;
    cudaStream_t st = (cudaStream_t)stream;
    Tc3Args a;
    memset(&a, 0, sizeof a);
    const uint64_t N = (uint64_t)w.N, K = (uint64_t)w.K;
    bool ok = true;
    if (w.fmt == FMT_BF16) {
        ok &= make_map3(&a.tm0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w.w, K, N, K * 2, 64, 128);
    } else {
        ok &= make_map3(&a.tm0, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.sm, K, N, K, 128, 128);
        if (w.fmt == FMT_PAL) ok &= make_map3(&a.tm1, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, K / 2, N, K / 2, 128, 128);
        else ok &= make_map3(&a.tm1, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.exps, K, N, K, 128, 128);
    }
    ok &= make_map3(&a.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, (uint64_t)B, K * 2, 64, (uint32_t)s.BN);
    if (!ok) return cudaErrorInvalidValue;
    a.tmv_off = w.tmv_off;
    a.tmv_mask = w.tmv_mask;
    a.tmv_data = w.tmv_data;
    a.status = w.status;
    a.N = w.N;
    a.K = w.K;
    a.B = B;
    a.BN = s.BN;
    a.cstages = s.cstages;
    a.xstages = s.xstages;
    a.cstage_bytes = s.cstage_bytes;
    a.upk = (int)(w.K / kUnitK);
    a.nbuf = s.nbuf;
    a.acol0 = s.acol0;
    a.units = s.units;
    memcpy(a.palette, w.palette, 16);
    // segments of a tile may come from several CTAs: they all add into a zeroed fp32 target
    a.acc = out_bf16 ? acc_ws : (float *)y;
    if (!a.acc) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(a.acc, 0, (size_t)B * N * 4, st);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(num_sms(), s.units);
    if (w.fmt == FMT_PAL) e = launch3_fmt<FMT_PAL>(a, grid, s.smem, st);
    else if (w.fmt == FMT_EXP) e = launch3_fmt<FMT_EXP>(a, grid, s.smem, st);
    else e = launch3_fmt<FMT_BF16>(a, grid, s.smem, st);
    if (e != cudaSuccess) return e;
    if (out_bf16) return launch_finalize(acc_ws, y, B * w.N, 1, stream);
    return cudaSuccess;
}

}  // namespace uw
