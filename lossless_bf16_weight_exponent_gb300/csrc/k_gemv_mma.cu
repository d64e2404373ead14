// k_gemv_mma.cu - fused reconstruct + matrix-vector product for batch 1..16 on the tensor pipe (sm_103a).
//
// Cloudflare blog "Unweight", section on the reconstructive matmul: the weights
// are rebuilt from the exponent data and the sign+mantissa bytes on chip and fed
// straight into the product.  For batch 1-16 the product has too few columns for
// the tcgen05 tiles, but a warp-level mma.sync m16n8k16 (bf16 in, fp32
// accumulate) still takes the multiply-adds and the reduction over K off the
// CUDA cores: the activations are the 16 x 16 A operand (M = batch, zero rows
// beyond B) and eight rebuilt weight rows are the 16 x 8 B operand.
//
// Layout.  A stage is 8 weight rows by one K-slice.  Warp 0 (one elected thread)
// moves a stage with one 3-D tensor copy per stream, the stream seen as
// [chunks of 128 bytes][rows][16 x 8-byte elements] with the 128-byte swizzle,
// so shared memory holds [chunk][row][128 B] and the 16-byte piece s of row r
// sits at piece s ^ (r % 8): the eight rows a warp reads at once fall in eight
// different bank groups.  Consumer warp w owns K range [KW w, KW (w + 1)) of
// the slice (KW = 256 or 128 weights); in each 64-weight step lane (g, t) = (lane / 4, lane % 4) reads
// the 16 consecutive weights 16t..16t+15 of row g (one 16-byte sm piece and
// 8 bytes of codes), rebuilds them as eight bf16x2 pairs and issues four MMAs.
// The MMA's logical k is permuted so each lane's pairs are physically
// consecutive weights: in MMA s of the step, logical (2t, 2t+1) is weight
// 16t + 4s + {0, 1} and logical (2t + 8, 2t + 9) is weight 16t + 4s + {2, 3};
// the activations use the same order, so lane (g, t) keeps X[g][16t..16t+15]
// (and X[g + 8][...] when B > 8) of every step of its range in registers.  The
// accumulator lane (g, t) ends a stage with rows 2t, 2t + 1 of batch rows g and
// g + 8; the warps' partial sums meet in shared memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "uw_internal.h"

namespace uw {

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait: far above any legitimate stall
constexpr int kTableBytes = 256 * 128;            // palette pair table (see pair_exp)
constexpr int kRowsPerStage = 8;

struct MmaArgs {  // 64-byte aligned through its tensor maps
    CUtensorMap tm0;  // sm bytes | bf16 weights: [K / 128 or K / 64 chunks][N rows][16 x u64], box {16, 8, chunks}
    CUtensorMap tm1;  // codes [K / 256][N][16 x u64] | exponent bytes [K / 128][N][16 x u64]
    WOperand w;
    const uint16_t *x;
    int64_t B;
    void *y;
    float *acc;
    int out_bf16;
    int nsplit;
    int klen;        // K-slice length (C * weights per warp)
    int stages;      // ring depth
    int stage_bytes;
    int blocks_cta;  // max 8-row blocks of one CTA
    int bm_words;
    int vcap;
    int w_from_prev;
    int *status;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Hand a ring slot back to the producer once the warp has read it: the slot was read with generic-proxy loads
// and the next tensor copy writes it through the async proxy, so each lane fences its reads across the proxies
// (as the PTX memory model requires), the warp converges and one lane arrives on the slot's "empty" barrier.
__device__ __forceinline__ void release_slot(uint64_t *empty_bar, int lane)
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar);
}

// Wait until the barrier's phase with this parity completes; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 64; i++)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// L2 policies: the weight streams are read once per launch (evict first); X is read by every CTA (evict last)
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 ldg_hint(const void *src, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(src), "l"(pol));
    return v;
}

__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, "
        "%4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Palette pair table: for a code byte b (codes c0 = b & 15, c1 = b >> 4) the exponent fields of the bf16x2
// pair, (pal[c1] << 23) | (pal[c0] << 7), stored for each lane at byte offset 128*b + 4*lane (no two lanes
// share a bank).
__device__ __forceinline__ uint32_t pair_exp(const uint8_t *tab_lane, uint32_t C, int j)
{
    const uint32_t b = prmt(C, 0u, 0x4440u | (uint32_t)j);  // byte j of C
    return *(const uint32_t *)(tab_lane + b * 128u);
}

// bf16x2 pairs (weights 0,1 and 2,3) from four sign+mantissa bytes and four exponent bytes
__device__ __forceinline__ void pairs_from_exps(uint32_t S, uint32_t E, uint32_t &p01, uint32_t &p23)
{
    const uint32_t hi = (S & 0x80808080u) | ((E >> 1) & 0x7F7F7F7Fu);
    const uint32_t lo = (S & 0x7F7F7F7Fu) | ((E << 7) & 0x80808080u);
    p01 = __byte_perm(lo, hi, 0x5140u);
    p23 = __byte_perm(lo, hi, 0x7362u);
}

// D += A * B, m16n8k16, bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// stage bytes per slice weight: sm 8 + codes 4 (per 8 rows: 12 per weight column) | sm + exps 16 | bf16 16
template <int FMT> struct StageFmt;
template <> struct StageFmt<FMT_PAL> { static constexpr int bytes_per_col = 12, off1_per_col = 8; };
template <> struct StageFmt<FMT_EXP> { static constexpr int bytes_per_col = 16, off1_per_col = 8; };
template <> struct StageFmt<FMT_BF16> { static constexpr int bytes_per_col = 16, off1_per_col = 0; };

// MB = 1: B <= 8 (A rows g only); MB = 2: B <= 16 (A rows g and g + 8).  KW: weights of the slice per
// consumer warp (256 keeps K = 4096 in one slice; 128 halves the activation registers)
// A verbatim step's lanes rebuild its weights from the staged exponents inside the loop.  (Counting verbatim blocks
// as zero weights and adding their products after the loop would be cheaper at small B, but X is the MMA's operand
// for all eight rows, so a zero weight would meet an infinite activation as 0 * inf = NaN.)
template <int MB, int KW, int FMT>
__global__ void __launch_bounds__(544, 1) gemv_mma_kernel(const __grid_constant__ MmaArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int NJ = KW / 64;    // 64-weight steps per warp
    const int64_t N = a.w.N, K = a.w.K;
    const int64_t KB = K / 64;     // blocks per row
    const int64_t k0 = (int64_t)blockIdx.y * a.klen;
    const int64_t nblk = (N + kRowsPerStage - 1) / kRowsPerStage;
    // the CTA's 8-row blocks: balanced partition over gridDim.x; rows [r0, r1)
    const int64_t bk0 = nblk * blockIdx.x / gridDim.x, bk1 = nblk * (blockIdx.x + 1) / gridDim.x;
    const int64_t r0 = bk0 * kRowsPerStage, r1 = min(bk1 * kRowsPerStage, N);
    const int nrows = r1 > r0 ? (int)(r1 - r0) : 0;
    const int n_stages = (int)(bk1 - bk0);
    const uint64_t wb0 = ((uint64_t)r0 * KB) >> 5;
    const int n_bw = nrows ? (int)((((uint64_t)r1 * KB - 1) >> 5) - wb0 + 1) : 0;

    constexpr int TB = FMT == FMT_PAL ? kTableBytes : 0;
    uint8_t *tab = smem;                                               // [TB] pair table
    uint64_t *full = (uint64_t *)(smem + TB);                          // [stages]
    uint64_t *empty = full + a.stages;                                 // [stages]
    uint64_t *vfull = empty + a.stages;                                // staged verbatim exponents landed
    float *part = (float *)(smem + TB + 1024);                         // [blocks_cta * 8][B]
    const int part_bytes = (a.blocks_cta * kRowsPerStage * (int)a.B * 4 + 1023) / 1024 * 1024;
    const int bm_bytes = (a.bm_words * 4 + 1023) / 1024 * 1024;
    uint32_t *bm = (uint32_t *)(smem + TB + 1024 + part_bytes);        // [bm_words] bitmap
    uint32_t *pf = (uint32_t *)(smem + TB + 1024 + part_bytes + bm_bytes);
    uint8_t *vx = smem + TB + 1024 + part_bytes + 2 * bm_bytes;         // [vcap][64] verbatim exps
    uint8_t *ring = vx + ((size_t)a.vcap * 64 + 1023) / 1024 * 1024;   // 1024-aligned (128-byte swizzle)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = (int)(blockDim.x >> 5) - 1;  // consumer warps
    const uint32_t stage_tx = (uint32_t)(StageFmt<FMT>::bytes_per_col * a.klen);
    if (threadIdx.x == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&a.tm0) : "memory");
        if (FMT != FMT_BF16) asm volatile("prefetch.tensormap [%0];" ::"l"(&a.tm1) : "memory");
        for (int s = 0; s < a.stages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C);
        }
        mbar_init(vfull, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer: two tensor copies per stage
        if (lane == 0) {
            if (a.w_from_prev) grid_dependency_wait();  // the workspace is written by the preceding kernel
            const uint64_t pol_w = l2_evict_first();
            const uint64_t fb = (uint64_t)r0 * KB, lb = (uint64_t)r1 * KB;  // first block, one past last
            int issued = 0;
            bool ok = true, verb_issued = FMT != FMT_PAL;
            for (int i = 0; i < n_stages; i++) {
                const int slot = i % a.stages;
                if (!verb_issued && (i == a.stages || i + 1 == n_stages)) {
                    // the ring is primed: stage the CTA's verbatim run [v_begin, v_end) of the verbatim stream
                    uint32_t v_staged = 0;
                    uint64_t v_begin = 0;
                    if (nrows) {
                        const uint64_t lwd = (lb & 31) ? lb >> 5 : (lb - 1) >> 5;
                        const uint32_t bw0 = __ldg(a.w.bitmap + (fb >> 5)), pw0 = __ldg(a.w.prefix + (fb >> 5));
                        const uint32_t bw1 = __ldg(a.w.bitmap + lwd), pw1 = __ldg(a.w.prefix + lwd);
                        v_begin = pw0 + __popc(bw0 & ((1u << (fb & 31)) - 1u));
                        const uint64_t v_end = (lb & 31) ? pw1 + __popc(bw1 & ((1u << (lb & 31)) - 1u)) : pw1 + __popc(bw1);
                        v_staged = (uint32_t)min(v_end - v_begin, (uint64_t)a.vcap);
                    }
                    mbar_arrive_expect_tx(vfull, v_staged * 64);
                    if (v_staged) bulk_g2s(vx, a.w.verb_exp + v_begin * 64, v_staged * 64, vfull);
                    verb_issued = true;
                }
                if (i >= a.stages && !mbar_wait(&empty[slot], ((i / a.stages) - 1) & 1)) { ok = false; break; }
                uint8_t *st = ring + (size_t)slot * a.stage_bytes;
                const int row = (int)(r0 + (int64_t)i * kRowsPerStage);
                mbar_arrive_expect_tx(&full[slot], stage_tx);
                if (FMT == FMT_BF16) tma3d(st, &a.tm0, 0, row, (int)(k0 >> 6), &full[slot], pol_w);
                else {
                    tma3d(st, &a.tm0, 0, row, (int)(k0 >> 7), &full[slot], pol_w);
                    tma3d(st + StageFmt<FMT>::off1_per_col * a.klen, &a.tm1, 0, row,
                          (int)(FMT == FMT_PAL ? k0 >> 8 : k0 >> 7), &full[slot], pol_w);
                }
                issued = i + 1;
            }
            if (!verb_issued) mbar_arrive_expect_tx(vfull, 0);  // no stages (or a timeout before priming)
            // consumers wait for the verbatim run only when they meet a verbatim block: it must land before exit
            if (FMT == FMT_PAL && !mbar_wait(vfull, 0)) ok = false;
            if (!ok) {
                atomicExch(a.status, (int)DEV_TIMEOUT);
                for (int i = max(0, issued - a.stages); i < issued; i++) mbar_wait(&full[i % a.stages], (i / a.stages) & 1);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int ctid = threadIdx.x - 32;
    if (FMT == FMT_PAL) {
        for (int i = ctid; i < 256 * 8; i += C * 32) {
            const int b = i >> 3, q = i & 7;
            const uint32_t v = ((uint32_t)a.w.palette[b >> 4] << 23) | ((uint32_t)a.w.palette[b & 15] << 7);
            *(uint4 *)(tab + 128 * b + 16 * q) = make_uint4(v, v, v, v);
        }
        for (int i = ctid; i < a.bm_words; i += C * 32) {  // words past the CTA's blocks read as "not verbatim"
            bm[i] = i < n_bw ? __ldg(a.w.bitmap + wb0 + i) : 0u;
            pf[i] = i < n_bw ? __ldg(a.w.prefix + wb0 + i) : 0u;
        }
    }
    for (int i = ctid; i < a.blocks_cta * kRowsPerStage * (int)a.B; i += C * 32) part[i] = 0.f;
    const uint8_t *tab_lane = tab + 4 * lane;
    const int cw = warp - 1;
    const int g = lane >> 2, t = lane & 3;
    const int kw0 = cw * KW;  // the warp's K range within the slice
    grid_dependency_wait();   // X (and Y, written below) belong to the stream order after the preceding kernel
    // activations: X[g][k0 + kw0 + 64j + 16t ...] as A rows g (and g + 8)
    uint32_t xa[NJ][8], xb[MB == 2 ? NJ : 1][8];
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        const int64_t kk = k0 + kw0 + 64 * j + 16 * t;
#pragma unroll
        for (int m = 0; m < MB; m++) {
            const int64_t b = g + 8 * m;
            uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
            if (b < a.B && kk < K) {
                const uint4 *src = (const uint4 *)(a.x + b * K + kk);
                lo = ldg_hint(src, l2_evict_last());
                hi = ldg_hint(src + 1, l2_evict_last());
            }
            uint32_t *dst = m == 0 ? xa[j] : xb[MB == 2 ? j : 0];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                dst[q] = word_of(lo, q);
                dst[4 + q] = word_of(hi, q);
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(C * 32) : "memory");  // table, bitmap words, zeroed sums in place
    bool ok = true, vx_ready = false;
    uint64_t v_begin = 0;
    uint32_t v_staged = 0;
    for (int i = 0; i < n_stages && ok; i++) {
        const int slot = i % a.stages;
        if (!mbar_wait(&full[slot], (i / a.stages) & 1)) { ok = false; break; }
        const uint8_t *st = ring + (size_t)slot * a.stage_bytes;
        const int64_t row_base = r0 + (int64_t)i * kRowsPerStage;
        const int64_t row = row_base + g;  // the weight row this lane rebuilds
        const bool live = row < r1;
        // the lane's 16 weights of step j: sm bytes (x0) and codes (x1.x/.y) | exponent bytes (x1) | bf16 (x0, x1)
        auto load_step = [&](int j, uint4 &x0, uint4 &x1) {
            const int kl = kw0 + 64 * j;  // first weight of the step within the slice
            if (FMT == FMT_BF16) {
                const uint8_t *line = st + (kl >> 6) * 1024 + g * 128;
                x0 = *(const uint4 *)(line + (((2 * t) ^ g) << 4));
                x1 = *(const uint4 *)(line + (((2 * t + 1) ^ g) << 4));
            } else {
                const int s0 = ((kl & 127) >> 4) + t;
                x0 = *(const uint4 *)(st + (kl >> 7) * 1024 + g * 128 + ((s0 ^ g) << 4));
                if (FMT == FMT_PAL) {
                    const int cb = ((kl & 255) >> 1) + 8 * t;  // code byte within the 128-byte line
                    const uint2 cc = *(const uint2 *)(st + 8 * a.klen + (kl >> 8) * 1024 + g * 128 +
                                                      (((cb >> 4) ^ g) << 4) + (cb & 8));
                    x1 = make_uint4(cc.x, cc.y, 0u, 0u);
                } else {
                    x1 = *(const uint4 *)(st + 8 * a.klen + (kl >> 7) * 1024 + g * 128 + ((s0 ^ g) << 4));
                }
            }
        };
        // two steps (B > 8) go to registers at once and the slot is handed back before
        // the compute; otherwise each step is read when it is used and the slot is released afterwards
        constexpr bool kEarly = NJ <= 2;
        uint4 d0[NJ], d1[NJ];
        if (kEarly) {
#pragma unroll
            for (int j = 0; j < NJ; j++) load_step(j, d0[j], d1[j]);
        }
        // verbatim flags of the lane's steps: bit j of `vwin` (the steps' blocks are consecutive)
        uint32_t vwin = 0;
        uint32_t bl0 = 0;
        if (FMT == FMT_PAL && live) {
            bl0 = (uint32_t)((uint64_t)(row - r0) * KB + (uint64_t)((k0 + kw0) >> 6) + ((uint64_t)r0 * KB & 31));
            const uint64_t w2 = ((uint64_t)bm[(bl0 >> 5) + 1] << 32) | bm[bl0 >> 5];
            vwin = (uint32_t)(w2 >> (bl0 & 31)) & ((1u << NJ) - 1u);
        }
        if (kEarly) release_slot(&empty[slot], lane);

        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        // The lane's steps.  VB: some lane of the warp has a verbatim step; its lanes rebuild that step's weights
        // from the block's exponents.  The warp is converged again for the MMAs.
        auto run_steps = [&](auto VB) {
            constexpr bool vb = decltype(VB)::value;
#pragma unroll
            for (int j = 0; j < NJ; j++) {
                if (k0 + kw0 + 64 * j >= K) continue;  // past the end of K (last slice; warp-uniform)
                if (!kEarly) load_step(j, d0[j], d1[j]);
                uint32_t pw[8];  // pairs of weights 16t + 2q, 16t + 2q + 1 of the step
                if (FMT == FMT_PAL && vb && ((vwin >> j) & 1u)) {
                    if (!vx_ready) {  // first verbatim block met by this lane: the staged run must have landed
                        if (!mbar_wait(vfull, 0)) ok = false;
                        const uint64_t fb = (uint64_t)r0 * KB;
                        v_begin = pf[0] + __popc(bm[0] & ((1u << (fb & 31)) - 1u));
                        const uint64_t lb = (uint64_t)r1 * KB, lw = lb >> 5;
                        const uint64_t v_end = lw - wb0 < (uint64_t)n_bw
                                                   ? pf[lw - wb0] + __popc(bm[lw - wb0] & ((1u << (lb & 31)) - 1u))
                                                   : pf[n_bw - 1] + __popc(bm[n_bw - 1]);
                        v_staged = (uint32_t)min(v_end - v_begin, (uint64_t)a.vcap);
                        vx_ready = true;
                    }
                    const uint32_t bl = bl0 + j;
                    const uint64_t vi = pf[bl >> 5] + __popc(bm[bl >> 5] & ((1u << (bl & 31)) - 1u));
                    const uint64_t vl = vi - v_begin;
                    const uint4 ev = vl < (uint64_t)v_staged ? *(const uint4 *)(vx + vl * 64 + 16 * t)
                                                              : __ldg((const uint4 *)(a.w.verb_exp + vi * 64 + 16 * t));
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        pairs_from_exps(word_of(d0[j], q), word_of(ev, q), pw[2 * q], pw[2 * q + 1]);
                } else if (FMT == FMT_PAL) {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const uint32_t S = word_of(d0[j], q);
                        const uint32_t Cw = q < 2 ? d1[j].x : d1[j].y;
                        const int jb = 2 * (q & 1);
                        pw[2 * q] = (__byte_perm(S, 0u, 0x1100u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb);
                        pw[2 * q + 1] = (__byte_perm(S, 0u, 0x3322u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb + 1);
                    }
                } else if (FMT == FMT_EXP) {
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        pairs_from_exps(word_of(d0[j], q), word_of(d1[j], q), pw[2 * q], pw[2 * q + 1]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; q++) { pw[q] = word_of(d0[j], q); pw[4 + q] = word_of(d1[j], q); }
                }
                if (FMT == FMT_PAL && vb) __syncwarp();  // after the per-lane verbatim branch
#pragma unroll
                for (int s = 0; s < 4; s++)
                    mma16816(acc, xa[j][2 * s], MB == 2 ? xb[MB == 2 ? j : 0][2 * s] : 0u, xa[j][2 * s + 1],
                             MB == 2 ? xb[MB == 2 ? j : 0][2 * s + 1] : 0u, pw[2 * s], pw[2 * s + 1]);
            }
        };
        if (FMT == FMT_PAL && __any_sync(__activemask(), vwin != 0)) run_steps(std::true_type{});
        else run_steps(std::false_type{});
        if (!kEarly) release_slot(&empty[slot], lane);
        // acc: rows row_base + 2t, 2t + 1 of batch rows g (acc[0..1]) and g + 8 (acc[2..3])
#pragma unroll
        for (int m = 0; m < MB; m++) {
            const int64_t b = g + 8 * m;
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int64_t rw = row_base + 2 * t + e;
                if (b < a.B && rw < r1) atomicAdd(&part[(rw - r0) * a.B + b], acc[2 * m + e]);
            }
        }
    }
    if (!ok) atomicExch(a.status, (int)DEV_TIMEOUT);
    asm volatile("bar.sync 1, %0;" ::"r"(C * 32) : "memory");
    for (int i = ctid; i < nrows * (int)a.B; i += C * 32) {
        const int64_t b = i % a.B, rl = i / a.B;
        const int64_t o = b * N + r0 + rl;
        const float v = part[i];
        if (a.nsplit > 1) atomicAdd(a.acc + o, v);
        else if (a.out_bf16) ((__nv_bfloat16 *)a.y)[o] = __float2bfloat16_rn(v);
        else ((float *)a.y)[o] = v;
    }
}

struct MmaShape {
    int consumers, per_sm, klen, nsplit, stages, stage_bytes, blocks_cta, bm_words, vcap, ctas;
    size_t smem;
};

// 16 consumer warps, one CTA per SM; each warp owns 256 / MB (variant 6) or 128 (variant 7) weights of a slice
int mma_kw(int64_t B, int variant) { return variant == 7 || B > 8 ? 128 : 256; }

bool plan_mma(const WOperand &w, int64_t B, int split_k, int variant, MmaShape &s)
{
    if (B < 1 || B > 16 || w.K <= 0 || w.K % 256 || w.N <= 0) return false;
    if (!tensor_map_encoder()) return false;
    s.consumers = 16;
    s.per_sm = 1;
    const size_t cap = 227 * 1024;
    s.klen = s.consumers * mma_kw(B, variant);
    s.nsplit = (int)((w.K + s.klen - 1) / s.klen);  // the slice is fixed by the warps' K ranges
    (void)split_k;
    const int bpc = w.fmt == FMT_PAL ? 12 : 16;
    s.stage_bytes = bpc * s.klen;
    const int64_t nblk = (w.N + kRowsPerStage - 1) / kRowsPerStage;
    s.ctas = (int)std::max<int64_t>(1, std::min<int64_t>(nblk, (int64_t)num_sms() * s.per_sm / s.nsplit));
    s.blocks_cta = (int)((nblk + s.ctas - 1) / s.ctas);
    const int64_t rows_cta = (int64_t)s.blocks_cta * kRowsPerStage;
    s.bm_words = (int)(rows_cta * (w.K / 64) / 32 + 2);
    const int64_t cta_blocks = rows_cta * (w.K / 64);
    s.vcap = w.fmt == FMT_PAL ? (int)std::min<int64_t>(64, std::max<int64_t>(16, cta_blocks * 3 / 100)) : 0;
    const size_t fixed = (w.fmt == FMT_PAL ? kTableBytes : 0) + 1024 + ((size_t)rows_cta * B * 4 + 1023) / 1024 * 1024 +
                         2 * (((size_t)s.bm_words * 4 + 1023) / 1024 * 1024) + ((size_t)s.vcap * 64 + 1023) / 1024 * 1024;
    if (fixed + 2 * (size_t)s.stage_bytes > cap) return false;
    s.stages = (int)std::min<size_t>(8, (cap - fixed) / s.stage_bytes);
    s.smem = fixed + (size_t)s.stages * s.stage_bytes;
    return true;
}

// tensor maps of the stage copies: dims (innermost first) {16 x u64, N rows, chunks}, box {16, 8, chunks per slice}
bool make_mma_maps(const WOperand &w, const MmaShape &s, CUtensorMap &m0, CUtensorMap &m1)
{
    auto enc = (PFN_cuTensorMapEncodeTiled_v12000)tensor_map_encoder();
    if (!enc) return false;
    auto make = [&](CUtensorMap &m, const void *base, uint64_t row_bytes, uint64_t line_weights) {
        if (!base || ((uintptr_t)base & 15)) return false;
        cuuint64_t dims[3] = {16, (cuuint64_t)w.N, (cuuint64_t)(w.K / line_weights)};
        cuuint64_t strides[2] = {row_bytes, 128};
        cuuint32_t box[3] = {16, (cuuint32_t)kRowsPerStage, (cuuint32_t)(s.klen / line_weights)};
        cuuint32_t estr[3] = {1, 1, 1};
        if (box[2] > 256) return false;
        return enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    const uint64_t K = (uint64_t)w.K;
    if (w.fmt == FMT_PAL) return make(m0, w.sm, K, 128) && make(m1, w.codes, K / 2, 256);
    if (w.fmt == FMT_EXP) return make(m0, w.sm, K, 128) && make(m1, w.exps, K, 128);
    return make(m0, w.w, 2 * K, 64);
}

template <int MB, int KW, int FMT>
cudaError_t launch_mma_one(const MmaArgs &a, dim3 grid, int threads, size_t smem, cudaStream_t st)
{
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<MB, KW, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<MB, KW, FMT>, a);
}

template <int MB, int KW>
cudaError_t launch_mma_fmt(int fmt, const MmaArgs &a, dim3 grid, int threads, size_t smem, cudaStream_t st)
{
    if (fmt == FMT_PAL) return launch_mma_one<MB, KW, FMT_PAL>(a, grid, threads, smem, st);
    if (fmt == FMT_EXP) return launch_mma_one<MB, KW, FMT_EXP>(a, grid, threads, smem, st);
    return launch_mma_one<MB, KW, FMT_BF16>(a, grid, threads, smem, st);
}

}  // namespace

bool gemv_mma_supported(const WOperand &w, int64_t B, int variant)
{
    MmaShape s;
    return (variant == 6 || variant == 7) && plan_mma(w, B, 0, variant, s);
}

int launch_gemv_mma(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, int split_k, int variant,
                    float *acc_ws, int *status, void *stream)
{
    MmaShape s;
    if (!plan_mma(w, B, split_k, variant, s)) return cudaErrorInvalidValue;
    cudaStream_t st = (cudaStream_t)stream;
    MmaArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!make_mma_maps(w, s, a.tm0, a.tm1)) return cudaErrorInvalidValue;
    a.w = w;
    a.x = x;
    a.B = B;
    a.y = y;
    a.out_bf16 = out_bf16;
    a.nsplit = s.nsplit;
    a.klen = s.klen;
    a.stages = s.stages;
    a.stage_bytes = s.stage_bytes;
    a.blocks_cta = s.blocks_cta;
    a.bm_words = s.bm_words;
    a.vcap = s.vcap;
    a.w_from_prev = w.w_from_prev;
    a.status = status;
    if (s.nsplit > 1) {
        a.acc = out_bf16 ? acc_ws : (float *)y;
        if (!a.acc) return cudaErrorInvalidValue;
        // zeroed by a kernel, not a memset: this kernel is a dependent launch, and its wait orders it only after
        // a preceding kernel (a memset before it could still be running when its atomics start)
        if ((uintptr_t)a.acc & 15) return cudaErrorInvalidValue;
        cudaError_t e = (cudaError_t)launch_zero_target(a.acc, B * w.N, st);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)s.ctas, (unsigned)s.nsplit, 1);
    const int threads = 32 * (1 + s.consumers);
    cudaError_t e = B > 8                          ? launch_mma_fmt<2, 128>(w.fmt, a, grid, threads, s.smem, st)
                    : mma_kw(B, variant) == 256 ? launch_mma_fmt<1, 256>(w.fmt, a, grid, threads, s.smem, st)
                                                : launch_mma_fmt<1, 128>(w.fmt, a, grid, threads, s.smem, st);
    if (e != cudaSuccess) return e;
    if (s.nsplit > 1 && out_bf16) return launch_finalize(acc_ws, y, B * w.N, 1, stream);
    return cudaSuccess;
}

}  // namespace uw
