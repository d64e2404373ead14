// k_tc.cu - fused reconstruct + tcgen05 tensor-core GEMM (sm_103a), batch sizes where the product is a dense
// contraction.
//
// Cloudflare blog "Unweight", section on the reconstructive matmul: producer threads stage compressed inputs
// with the copy engine; consumer threads rebuild BF16 in shared memory and feed it straight to the tensor
// cores, so reconstructed weights never leave the SM.  The post's H100 kernel uses WGMMA; this is the
// Blackwell form: tcgen05.mma with the fp32 accumulator in tensor memory.
//
// One CTA owns a tile of 128 rows of W (the MMA's M) and a range of K.  Per 64-wide K-stage:
//   - warp 16 (one thread) TMA-loads the sign+mantissa tile [128 x 64] u8, the 4-bit code tile [128 x 32] u8
//     (or the exponent tile, or - full-decode pipeline - the bf16 tile straight into the MMA layout) and the
//     X tile [BN x 64] bf16 with 128-byte swizzle; one mbarrier counts the bytes;
//   - warps 0-15 (two groups of eight taking alternate K-stages) rebuild BF16 from the staged bytes into the
//     K-major SWIZZLE_128B layout tcgen05 reads (row r, 16-byte chunk c at (r/8)*1024 + (r%8)*128 +
//     ((c ^ (r%8)) * 16)), fence the generic-proxy writes for the async proxy and arrive on a second mbarrier;
//   - one thread of warp 17 issues four tcgen05.mma (M=128, N=BN <= 256, K=16; a second MMA for columns
//     256..511) accumulating in TMEM, and tcgen05.commit releases the stage when they complete.
// Epilogue: warps 0-3 read their 32 TMEM lanes (rows) with tcgen05.ld and write Y[b, row] coalesced (fp32,
// bf16, or fp32 atomics when K is split).  All waits are bounded; TMEM is always freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "uw_internal.h"

namespace uw {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kGroupWarps = 8;                       // warps rebuilding one stage (256 threads, 2 chunks each)
constexpr int kRebuildGroups = 2;                    // groups rebuild alternate stages concurrently
constexpr int kRebuildWarps = kGroupWarps * kRebuildGroups;
constexpr int kProducerWarp = kRebuildWarps;
constexpr int kMmaWarp = kRebuildWarps + 1;
constexpr int kThreads = 32 * (kRebuildWarps + 2);
constexpr int kTabBytes = 256 * 64;   // pair table, 16 replicas (offset 64*b + 4*(lane & 15))
constexpr int kMaskWords = 8;         // per-row verbatim stage masks: up to 256 K-stages per CTA
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct TcArgs {
    CUtensorMap tm_sm;   // sm [N, K] u8, box {64, 128}
    CUtensorMap tm_aux;  // codes [N, K/2] u8 box {32,128} | exps [N, K] u8 box {64,128} | W bf16 [N,K] box {64,128} sw128
    CUtensorMap tm_x;    // X [B, K] bf16, box {64, min(BN, 256)}, 128-byte swizzle
    const uint32_t *bitmap, *prefix;
    const uint8_t *verb_exp;
    void *y;
    float *acc;
    int *status;
    int64_t N, K, B;
    int BN, ks_stages, stages, stage_bytes, tmem_cols, nsplit, out_bf16, fmt;
    int vcap;            // verbatim blocks staged in shared memory per CTA (beyond: global loads)
    uint8_t palette[16];
};

__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtime()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(n) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(saddr(b)), "r"(parity)
                 : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity)
{
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = gtime();
    for (;;) {
        for (int i = 0; i < 64; i++)
            if (mbar_test(b, parity)) return true;
        if (gtime() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            saddr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(saddr(bar))
        : "memory");
}

// K-major, 128-byte-swizzled shared-memory matrix descriptor (8-row core groups 1024 bytes apart)
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr)
{
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major), 16 bytes
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 1024 bytes between 8-row groups
    d |= (uint64_t)1 << 46;            // descriptor version for this architecture family
    d |= (uint64_t)2 << 61;            // layout: 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, both K-major, M x N
__host__ __device__ constexpr uint32_t instr_desc(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
                     d_tmem),
                 "l"(a), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar)) : "memory");
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ void pairs_from_exps(uint32_t S, uint32_t E, uint32_t &p01, uint32_t &p23)
{
    const uint32_t hi = (S & 0x80808080u) | ((E >> 1) & 0x7F7F7F7Fu);
    const uint32_t lo = (S & 0x7F7F7F7Fu) | ((E << 7) & 0x80808080u);
    p01 = __byte_perm(lo, hi, 0x5140u);
    p23 = __byte_perm(lo, hi, 0x7362u);
}

__device__ __forceinline__ uint32_t pair_exp(const uint8_t *tab_lane, uint32_t C, int j)
{
    const uint32_t off = (j == 0 ? (C << 6) : (C >> (8 * j - 6))) & 0x3FC0u;  // byte j of C, times 64
    return *(const uint32_t *)(tab_lane + off);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ TcArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-align the dynamic window (the swizzled tiles need it)
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = a.stages;
    uint8_t *tab = smem;                                                  // [kTabBytes] (FMT_PAL)
    uint64_t *full = (uint64_t *)(smem + kTabBytes);                     // [S]
    uint64_t *afull = full + S;                                           // [S]
    uint64_t *empty = afull + S;                                          // [S]
    uint64_t *done = empty + S;                                           // [1]
    uint32_t *tmem_slot = (uint32_t *)(done + 1);
    // verbatim staging: per row, stage masks (bit i = K-stage i is a verbatim block), running local indices,
    // the row's first index in the verbatim stream, and the staged exponents themselves
    uint32_t *vmask = (uint32_t *)(smem + kTabBytes + 1024);          // [128][kMaskWords]
    uint32_t *vpfx = vmask + BM * kMaskWords;                          // [128][kMaskWords]
    uint32_t *vrow = vpfx + BM * kMaskWords;                           // [128] local index of the row's first block
    uint32_t *vglob = vrow + BM;                                       // [128] stream index of the row's first block
    uint8_t *vdata = (uint8_t *)(vglob + BM);                          // [vcap][64]
    uint8_t *ring = smem + kTabBytes + 1024 + 2 * BM * kMaskWords * 4 + 2 * BM * 4 + (size_t)a.vcap * 64;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t N = a.N, K = a.K;
    const int64_t row0 = (int64_t)blockIdx.x * BM;
    const int k_stage0 = blockIdx.y * a.ks_stages;
    const int nks = (int)min((int64_t)a.ks_stages, K / BK - k_stage0);
    const int xrows = a.BN < 256 ? a.BN : 256;
    const uint32_t x_bytes = (uint32_t)a.BN * 128;
    const uint32_t stage_tx = (FMT == FMT_BF16 ? 16384u : (8192u + (FMT == FMT_PAL ? 4096u : 8192u))) + x_bytes;

    if (FMT == FMT_PAL)
        for (int i = threadIdx.x; i < 256 * 4; i += blockDim.x) {
            const int b = i >> 2, q = i & 3;
            const uint32_t v = ((uint32_t)a.palette[b >> 4] << 23) | ((uint32_t)a.palette[b & 15] << 7);
            *(uint4 *)(tab + 64 * b + 16 * q) = make_uint4(v, v, v, v);
        }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&afull[s], kGroupWarps);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                     "r"(a.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == kProducerWarp) {
        // -------------------------------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nks; i++) {
                const int s = i % S;
                if (i >= S && !mbar_wait(&empty[s], ((i / S) - 1) & 1)) { ok = false; break; }
                uint8_t *st = ring + (size_t)s * a.stage_bytes;
                const int kx = (k_stage0 + i) * BK;
                mbar_expect_tx(&full[s], stage_tx);
                if (FMT == FMT_BF16) {
                    tma2d(st, &a.tm_aux, kx, (int)row0, &full[s]);
                } else {
                    uint8_t *smt = st + 16384 + x_bytes;
                    tma2d(smt, &a.tm_sm, kx, (int)row0, &full[s]);
                    if (FMT == FMT_PAL) tma2d(smt + 8192, &a.tm_aux, kx / 2, (int)row0, &full[s]);
                    else tma2d(smt + 8192, &a.tm_aux, kx, (int)row0, &full[s]);
                }
                for (int h = 0; h * 256 < a.BN; h++) tma2d(st + 16384 + h * 256 * 128, &a.tm_x, kx, h * 256, &full[s]);
                issued = i + 1;
            }
            if (!ok) {
                atomicExch(a.status, (int)DEV_TIMEOUT);
                for (int i = max(0, issued - S); i < issued; i++) mbar_wait(&full[i % S], (i / S) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t id0 = instr_desc(BM, xrows);
            const uint32_t id1 = instr_desc(BM, a.BN > 256 ? a.BN - 256 : 16);
            int i = 0;
            for (; i < nks; i++) {
                const int s = i % S;
                const bool got = FMT == FMT_BF16 ? mbar_wait(&full[s], (i / S) & 1) : mbar_wait(&afull[s], (i / S) & 1);
                if (!got) { ok = false; break; }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                uint8_t *st = ring + (size_t)s * a.stage_bytes;
                const uint32_t a_base = saddr(st), x_base = saddr(st + 16384);
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++) {
                    const uint64_t ad = smem_desc(a_base + 32 * kk);
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    mma_bf16(tmem, ad, smem_desc(x_base + 32 * kk), id0, acc);
                    if (a.BN > 256) mma_bf16(tmem + 256, ad, smem_desc(x_base + 256 * 128 + 32 * kk), id1, acc);
                }
                mma_commit(&empty[s]);
            }
            if (!ok) atomicExch(a.status, (int)DEV_TIMEOUT);
            mma_commit(done);  // arrives once every MMA issued above has completed
        }
    } else {
        // -------------------------------------------------------------------------------- rebuild (warps 0-15)
        if (FMT != FMT_BF16) {
            const int tid = threadIdx.x;            // 0..511
            const int group = warp / kGroupWarps;   // stages i with i % kRebuildGroups == group
            const int gtid = tid % (32 * kGroupWarps);
            const uint8_t *tab_lane = tab + 4 * (lane & 15);
            if (FMT == FMT_PAL) {
                // --- stage the tile's verbatim information (overlaps the producer's first loads)
                uint32_t cnt = 0;
                if (tid < BM) {
                    const int64_t row = row0 + tid;
                    uint64_t fb = 0;
                    if (row < N) {
                        fb = (uint64_t)row * (uint64_t)(K / BK) + (uint64_t)k_stage0;
                        for (int w = 0; w < kMaskWords; w++) {
                            uint32_t m = 0;
                            const int first = 32 * w;
                            if (first < nks) {
                                const uint64_t bb = fb + (uint64_t)first;
                                const uint64_t lo = __ldg(a.bitmap + (bb >> 5)), hi = __ldg(a.bitmap + (bb >> 5) + 1);
                                m = (uint32_t)(((hi << 32) | lo) >> (bb & 31));
                                const int valid = nks - first;
                                if (valid < 32) m &= (1u << valid) - 1u;
                            }
                            vmask[tid * kMaskWords + w] = m;
                            vpfx[tid * kMaskWords + w] = cnt;  // local count before this word (row-relative)
                            cnt += __popc(m);
                        }
                        vglob[tid] = __ldg(a.prefix + (fb >> 5)) + __popc(__ldg(a.bitmap + (fb >> 5)) & ((1u << (fb & 31)) - 1u));
                    } else {
                        for (int w = 0; w < kMaskWords; w++) { vmask[tid * kMaskWords + w] = 0; vpfx[tid * kMaskWords + w] = 0; }
                        vglob[tid] = 0;
                    }
                    vrow[tid] = cnt;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(32 * kRebuildWarps) : "memory");
                // exclusive scan of the per-row counts (one warp)
                if (warp == 0) {
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
                for (int r = warp; r < BM; r += kRebuildWarps) {
                    const uint32_t base = vrow[r];
                    const uint32_t n = (r + 1 < BM ? vrow[r + 1] : base + vpfx[r * kMaskWords + kMaskWords - 1] +
                                                                     __popc(vmask[r * kMaskWords + kMaskWords - 1])) - base;
                    const uint4 *src = (const uint4 *)(a.verb_exp + (uint64_t)vglob[r] * 64);
                    for (uint32_t q = lane; q < n * 4; q += 32)
                        if (base + q / 4 < (uint32_t)a.vcap) ((uint4 *)(vdata + (uint64_t)base * 64))[q] = __ldg(src + q);
                }
                asm volatile("bar.sync 1, %0;" ::"n"(32 * kRebuildWarps) : "memory");
            }
            for (int i = group; i < nks; i += kRebuildGroups) {
                const int s = i % S;
                if (!mbar_wait(&full[s], (i / S) & 1)) { ok = false; break; }
                uint8_t *st = ring + (size_t)s * a.stage_bytes;
                const uint8_t *smt = st + 16384 + x_bytes;
#pragma unroll
                for (int j = 0; j < 2; j++) {
                    const int item = gtid + 256 * j;
                    const int r = item >> 2, c = item & 3;
                    const uint4 sv = *(const uint4 *)(smt + r * 64 + c * 16);
                    uint32_t pw[8];
                    bool verb = false;
                    uint32_t vlocal = 0;
                    if (FMT == FMT_PAL) {
                        const uint32_t m = vmask[r * kMaskWords + (i >> 5)];
                        verb = (m >> (i & 31)) & 1u;
                        vlocal = vpfx[r * kMaskWords + (i >> 5)] + __popc(m & ((1u << (i & 31)) - 1u));
                    }
                    if (FMT == FMT_EXP || verb) {
                        uint4 ev;
                        if (FMT == FMT_EXP) ev = *(const uint4 *)(smt + 8192 + r * 64 + c * 16);
                        else {
                            const uint32_t li = vrow[r] + vlocal;
                            ev = li < (uint32_t)a.vcap ? *(const uint4 *)(vdata + (uint64_t)li * 64 + c * 16)
                                                       : __ldg((const uint4 *)(a.verb_exp + ((uint64_t)vglob[r] + vlocal) * 64 + c * 16));
                        }
#pragma unroll
                        for (int q = 0; q < 4; q++) pairs_from_exps(word_of(sv, q), word_of(ev, q), pw[2 * q], pw[2 * q + 1]);
                    } else {
                        const uint2 cc = *(const uint2 *)(smt + 8192 + r * 32 + c * 8);
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const uint32_t Sw = word_of(sv, q);
                            const uint32_t Cw = q < 2 ? cc.x : cc.y;
                            const int jb = 2 * (q & 1);
                            pw[2 * q] = (__byte_perm(Sw, 0u, 0x1100u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb);
                            pw[2 * q + 1] = (__byte_perm(Sw, 0u, 0x3322u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb + 1);
                        }
                    }
                    uint8_t *arow = st + (r >> 3) * 1024 + (r & 7) * 128;
                    *(uint4 *)(arow + (((2 * c) ^ (r & 7)) << 4)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    *(uint4 *)(arow + (((2 * c + 1) ^ (r & 7)) << 4)) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[s]);
            }
            if (!ok) atomicExch(a.status, (int)DEV_TIMEOUT);
        }
    }

    // ------------------------------------------------------------------------------------ epilogue (warps 0-3)
    if (warp < 4) {
        const bool got = mbar_wait(done, 0);
        if (!got) atomicExch(a.status, (int)DEV_TIMEOUT);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int64_t row = row0 + 32 * warp + lane;
        for (int c0 = 0; c0 < a.BN && c0 < a.B; c0 += 16) {
            uint32_t v[16];
            const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0;
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (got && row < N) {
#pragma unroll
                for (int t = 0; t < 16; t++) {
                    const int64_t b = c0 + t;
                    if (b < a.B) {
                        const int64_t o = b * N + row;
                        const float f = __uint_as_float(v[t]);
                        if (a.nsplit > 1) atomicAdd(a.acc + o, f);
                        else if (a.out_bf16) ((__nv_bfloat16 *)a.y)[o] = __float2bfloat16_rn(f);
                        else ((float *)a.y)[o] = f;
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
    }
}

// ---------------------------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return (PFN_cuTensorMapEncodeTiled_v12000)tensor_map_encoder(); }

bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct TcShape {
    int BN, tmem_cols, stage_bytes, stages, ks_stages, nsplit, vcap;
    size_t smem;
};

int pad_batch(int64_t B) { return B <= 256 ? (int)((B + 15) / 16 * 16) : 512; }

bool tc_shape(const WOperand &w, int64_t B, int split_k, TcShape &s)
{
    if (B < 1 || B > 512 || w.N <= 0 || w.K < BK || w.K % BK) return false;
    if (w.N > (int64_t)INT32_MAX || w.K > (int64_t)INT32_MAX) return false;
    s.BN = pad_batch(B);
    s.tmem_cols = 32;
    while (s.tmem_cols < s.BN) s.tmem_cols *= 2;
    const int aux = w.fmt == FMT_BF16 ? 0 : 8192 + (w.fmt == FMT_PAL ? 4096 : 8192);
    s.stage_bytes = (16384 + s.BN * 128 + aux + 1023) / 1024 * 1024;
    const size_t fixed = 1024 /* alignment slack */ + kTabBytes + 1024 + 2 * BM * kMaskWords * 4 + 2 * BM * 4;
    const size_t cap = 227 * 1024;
    const int min_v = w.fmt == FMT_PAL ? 64 : 0;  // always room for at least 64 staged verbatim blocks
    if (fixed + (size_t)min_v * 64 + 2 * (size_t)s.stage_bytes > cap) return false;
    s.stages = (int)std::min<size_t>(5, (cap - fixed - (size_t)min_v * 64) / s.stage_bytes);
    s.vcap = w.fmt == FMT_PAL ? (int)std::min<size_t>(512, (cap - fixed - (size_t)s.stages * s.stage_bytes) / 64) : 0;
    s.vcap &= ~15;  // the ring after the staged blocks stays 1024-aligned
    s.smem = fixed + (size_t)s.vcap * 64 + (size_t)s.stages * s.stage_bytes;
    // at most 512 TMEM columns per SM: raise the shared-memory request so fewer CTAs co-reside if needed
    const size_t per_sm = 233472;
    const int max_by_tmem = 512 / s.tmem_cols;
    if ((int)(per_sm / (s.smem + 1024)) > max_by_tmem) s.smem = std::min(cap, per_sm / max_by_tmem - 1024 + 1);
    const int ctas_per_sm = std::max(1, (int)(per_sm / (s.smem + 1024)));
    const int64_t tiles = (w.N + BM - 1) / BM;
    const int kst = (int)(w.K / BK);
    int split = std::max(split_k, (kst + 32 * kMaskWords - 1) / (32 * kMaskWords));  // <= 256 stages per CTA
    if (split_k <= 0) {
        // choose the split with the best wave efficiency, at least 4 K-stages per CTA
        const int64_t slots = (int64_t)num_sms() * ctas_per_sm;
        double best = -1;
        const int min_split = split;
        for (int sp = min_split; sp <= std::max(16, min_split); sp++) {
            if (kst / sp < 4 && sp > min_split) break;
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
cudaError_t launch_fmt(const TcArgs &a, dim3 grid, size_t smem, cudaStream_t st)
{
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tc_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    tc_kernel<FMT><<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

// Variant 4: the persistent kernel with the rebuilt weights in shared memory (k_tc4.cu, B <= 512, 4-bit codes,
// K % 256 == 0); any other variant or shape: this one.
bool tc_supported(const WOperand &w, int64_t B, int variant)
{
    TcShape s;
    if (variant == 4 && tc4_supported(w, B)) return true;
    return encode_fn() != nullptr && tc_shape(w, B, 0, s);
}

int tc_default_split(const WOperand &w, int64_t B, int variant)
{
    TcShape s;
    if (variant == 4 && tc4_supported(w, B)) return 1;
    return tc_shape(w, B, 0, s) ? s.nsplit : 1;
}

int launch_tc(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, int split_k, int variant,
              float *acc_ws, void *stream)
{
    if (variant == 4 && tc4_supported(w, B)) {
        const int e = launch_tc4(w, x, B, y, out_bf16, acc_ws, stream);
        if (e != cudaErrorInvalidValue) return e;  // else: no tensor map for these operands, use this kernel
    }
    TcShape s;
    if (!tc_shape(w, B, split_k, s)) return cudaErrorInvalidValue;
    cudaStream_t st = (cudaStream_t)stream;
    TcArgs a;
    memset(&a, 0, sizeof a);
    const uint64_t N = (uint64_t)w.N, K = (uint64_t)w.K;
    bool ok = true;
    if (w.fmt == FMT_BF16) {
        ok &= make_map(&a.tm_aux, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w.w, K, N, K * 2, 64, 128, true);
    } else {
        ok &= make_map(&a.tm_sm, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.sm, K, N, K, 64, 128, false);
        if (w.fmt == FMT_PAL) ok &= make_map(&a.tm_aux, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, K / 2, N, K / 2, 32, 128, false);
        else ok &= make_map(&a.tm_aux, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.exps, K, N, K, 64, 128, false);
    }
    ok &= make_map(&a.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, (uint64_t)B, K * 2, 64, (uint32_t)std::min(s.BN, 256), true);
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
    a.stages = s.stages;
    a.stage_bytes = s.stage_bytes;
    a.tmem_cols = s.tmem_cols;
    a.nsplit = s.nsplit;
    a.out_bf16 = out_bf16;
    a.fmt = w.fmt;
    a.vcap = s.vcap;
    memcpy(a.palette, w.palette, 16);
    if (s.nsplit > 1) {
        a.acc = out_bf16 ? acc_ws : (float *)y;
        if (!a.acc) return cudaErrorInvalidValue;
        cudaError_t e = cudaMemsetAsync(a.acc, 0, (size_t)B * N * 4, st);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)((N + BM - 1) / BM), (unsigned)s.nsplit);
    cudaError_t e;
    if (w.fmt == FMT_PAL) e = launch_fmt<FMT_PAL>(a, grid, s.smem, st);
    else if (w.fmt == FMT_EXP) e = launch_fmt<FMT_EXP>(a, grid, s.smem, st);
    else e = launch_fmt<FMT_BF16>(a, grid, s.smem, st);
    if (e != cudaSuccess) return e;
    if (s.nsplit > 1 && out_bf16) return launch_finalize(acc_ws, y, B * w.N, 1, stream);
    return cudaSuccess;
}

void *tensor_map_encoder()
{
    static void *fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = p;
    });
    return fn;
}

}  // namespace uw
