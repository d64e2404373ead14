// k_gemv_tma.cu - persistent fused reconstruct + GEMV fed by bulk-async copies (sm_103a), B <= 2.
//
// Cloudflare blog "Unweight", section on the reconstructive matmul: a producer
// moves compressed inputs from HBM into a circular shared-memory buffer with the
// copy engine and runs ahead of the consumers; consumers rebuild BF16 from the
// exponent data and the sign+mantissa bytes and feed the product at once.  The
// H100 kernel in the post feeds WGMMA; at batch 1-2 this contraction is a
// matrix-vector product bound by HBM, so the consumers here use fp32 FMAs.
//
// One CTA per SM owns a contiguous range of rows.  Warp 0 (one elected thread)
// issues cp.async.bulk copies of whole row slices - sign+mantissa bytes and the
// 4-bit codes (or exponent bytes, or plain bf16) - into a ring of S stages, each
// stage RS rows, with an mbarrier per stage for "full" (transaction bytes) and
// one for "empty" (one arrive per consumer warp).  Consumer warp c handles row
// slot c / WK of a stage and the c % WK-th piece of the K-slice: lane l owns the
// weights k = piece*32*LW + 16*l + 512*g (g < LW/16), so its X values stay in
// registers for the whole kernel and its 16-byte shared loads are bank-conflict
// free.  A consumer copies its part of a stage into registers and releases the
// slot before computing on it.  Two 4-bit codes (one code byte) select the
// exponent fields of a bf16x2 pair from a 32 KB per-lane table in shared memory,
// so a warp's lookups never share a bank.  A stage without verbatim blocks in the
// warp runs a straight-line body; otherwise a lane whose 16 weights lie in a
// verbatim block rebuilds them from that block's exponents, which the producer
// stages (the CTA's contiguous run of them) with one bulk copy before the ring
// fills.  Lane sums of four consecutive stages
// are reduced together (a transposed butterfly), and row sums meet in shared
// memory and are written once at the end.  A warp hands a slot back only after a
// cross-proxy fence on its reads (the next bulk copy writes it through the async
// proxy).  Every
// mbarrier wait is bounded by a global-timer limit; on expiry the kernel latches
// DEV_TIMEOUT, drains the copies it issued and returns.
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

struct TmaArgs {  // 64-byte aligned through its tensor maps
    // whole-stage tensor copies (tmap != 0): the weight streams seen as [rows][2048-weight chunks][chunk bytes]
    // in 8-byte elements, one box = one stage (rs rows x the K-slice)
    CUtensorMap tm0;  // sm bytes, or bf16 weights
    CUtensorMap tm1;  // codes or exponent bytes
    int tmap;
    WOperand w;
    const uint16_t *x;
    int64_t B;
    void *y;
    float *acc;
    int out_bf16;
    int nsplit;
    int ks;          // K-slice length (multiple of 64)
    int rs;          // rows per stage
    int stages;      // ring depth
    int wk;          // consumer warps per row
    int stage_bytes; // bytes of one stage
    int rows_cta;    // max rows owned by one CTA
    int bm_words;    // max verbatim-bitmap words of one CTA's rows
    int w_from_prev; // the weight stream is written by the preceding kernel (a preprocess workspace)
    int vcap;        // verbatim blocks of the CTA whose exponents are staged in shared memory (beyond: global loads)
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

// Hand a ring slot back to the producer once the warp has read it.  The slot was read with generic-proxy loads
// and is refilled by the bulk-copy engine, which writes through the async proxy; the PTX memory model orders a
// thread's generic accesses before a later async-proxy access to the same bytes only through a proxy fence.  So
// every lane fences its own reads, the warp converges, and one lane arrives on the slot's "empty" barrier.
// Without the fence the next copy into the slot intermittently landed before a warp's loads had read it (wrong
// rows in about 3% of full-decode runs on the 8B gate_proj, always in a warp that released its slot early).
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

__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, "
        "%4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// acc += w * x for both halves of a bf16x2 pair of weights and of activations: BF16 products are exact in
// fp32, so this equals two fp32 FMAs on the widened values, without widening them first.
__device__ __forceinline__ float fma2_bf16(uint32_t w2, uint32_t x2, float acc)
{
    asm("{\n .reg .b16 wl, wh, xl, xh;\n mov.b32 {wl, wh}, %1;\n mov.b32 {xl, xh}, %2;\n"
        " fma.rn.f32.bf16 %0, wl, xl, %0;\n fma.rn.f32.bf16 %0, wh, xh, %0;\n}\n"
        : "+f"(acc)
        : "r"(w2), "r"(x2));
    return acc;
}

__device__ __forceinline__ void pairs_from_exps(uint32_t S, uint32_t E, uint32_t &p01, uint32_t &p23)
{
    const uint32_t hi = (S & 0x80808080u) | ((E >> 1) & 0x7F7F7F7Fu);
    const uint32_t lo = (S & 0x7F7F7F7Fu) | ((E << 7) & 0x80808080u);
    p01 = __byte_perm(lo, hi, 0x5140u);
    p23 = __byte_perm(lo, hi, 0x7362u);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Palette pair table: for a code byte b (codes c0 = b & 15, c1 = b >> 4) the exponent fields of the bf16x2
// pair, (pal[c1] << 23) | (pal[c0] << 7), stored for each lane at byte offset 128*b + 4*lane, so a warp's 32
// lookups always hit 32 different banks.  The offset of byte j of a code word C is one byte extract and one
// integer multiply-add (which the scheduler may issue on the FMA pipe, leaving the ALU pipe to the rebuild).
constexpr int kTableBytes = 256 * 128;

__device__ __forceinline__ uint32_t pair_exp(const uint8_t *tab_lane, uint32_t C, int j)
{
    const uint32_t b = prmt(C, 0u, 0x4440u | (uint32_t)j);  // byte j of C
    return *(const uint32_t *)(tab_lane + b * 128u);
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// bytes per weight in a stage, per format
template <int FMT> struct Fmt;
template <> struct Fmt<FMT_PAL> { static constexpr int num = 3, den = 2; };   // sm + 4-bit code
template <> struct Fmt<FMT_EXP> { static constexpr int num = 2, den = 1; };   // sm + exponent byte
template <> struct Fmt<FMT_BF16> { static constexpr int num = 2, den = 1; };  // bf16

// Sum each of v0..v3 over the warp's 32 lanes (a transposed butterfly: 6 shuffles for the four sums).
// Lane L ends with the sum of v[((L >> 3) & 2) | ((L >> 3) & 1)], i.e. lanes 0, 8, 16, 24 hold sums 0..3.
__device__ __forceinline__ float reduce4(float v0, float v1, float v2, float v3, int lane)
{
    const bool u16 = lane & 16, u8 = lane & 8;
    const float s0 = u16 ? v0 : v2, s1 = u16 ? v1 : v3;  // what the partner keeps
    const float k0 = u16 ? v2 : v0, k1 = u16 ? v3 : v1;
    const float b0 = k0 + __shfl_xor_sync(0xFFFFFFFFu, s0, 16);
    const float b1 = k1 + __shfl_xor_sync(0xFFFFFFFFu, s1, 16);
    float c = (u8 ? b1 : b0) + __shfl_xor_sync(0xFFFFFFFFu, u8 ? b0 : b1, 8);
    c += __shfl_xor_sync(0xFFFFFFFFu, c, 4);
    c += __shfl_xor_sync(0xFFFFFFFFu, c, 2);
    c += __shfl_xor_sync(0xFFFFFFFFu, c, 1);
    return c;
}

template <int NB, int LW, int FMT>
__global__ void __launch_bounds__(544, 1) gemv_tma_kernel(const __grid_constant__ TmaArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int G = LW / 16;
    const int64_t N = a.w.N, K = a.w.K;
    const int64_t k0 = (int64_t)blockIdx.y * a.ks;
    const int klen = (int)min((int64_t)a.ks, K - k0);
    const int64_t b0 = (int64_t)blockIdx.z * NB;
    // rows of this CTA: balanced partition of N over gridDim.x
    const int64_t r0 = N * blockIdx.x / gridDim.x, r1 = N * (blockIdx.x + 1) / gridDim.x;
    const int nrows = (int)(r1 - r0);
    const int n_stages = (nrows + a.rs - 1) / a.rs;
    // verbatim bitmap words covering the CTA's rows
    const uint64_t wb0 = ((uint64_t)r0 * K / 64) >> 5;
    const int n_bw = nrows ? (int)((((uint64_t)r1 * K / 64 - 1) >> 5) - wb0 + 1) : 0;

    constexpr int TB = FMT == FMT_PAL ? kTableBytes : 0;
    uint8_t *tab = smem;                                                      // [TB] pair table
    uint64_t *full = (uint64_t *)(smem + TB);                                 // [stages]
    uint64_t *empty = full + a.stages;                                        // [stages]
    uint64_t *vfull = empty + a.stages;                                       // staged verbatim records landed
    float *part = (float *)(smem + TB + 1024);                                // [rows_cta][NB]
    const int part_bytes = (a.rows_cta * NB * 4 + 1023) / 1024 * 1024;
    const int bm_bytes = (a.bm_words * 4 + 1023) / 1024 * 1024;
    uint32_t *bm = (uint32_t *)(smem + TB + 1024 + part_bytes);              // [bm_words] bitmap
    uint32_t *pf = (uint32_t *)(smem + TB + 1024 + part_bytes + bm_bytes);   // [bm_words] prefix
    uint8_t *ring = smem + TB + 1024 + part_bytes + 2 * bm_bytes;            // 1024-aligned: tensor copies want 128
    uint8_t *vx = ring + (size_t)a.stages * a.stage_bytes;                    // [vcap][64] verbatim exponents

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = a.rs * a.wk;  // consumer warps
    const int CT = C * 32;

    if (threadIdx.x == 0) {
        if (a.tmap) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&a.tm0) : "memory");
            if (FMT != FMT_BF16) asm volatile("prefetch.tensormap [%0];" ::"l"(&a.tm1) : "memory");
        }
        for (int s = 0; s < a.stages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C);
        }
        mbar_init(vfull, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // a dependent launch may start its prologue and stream its own weights from here on
    grid_launch_dependents();

    const uint32_t wbytes = (uint32_t)((int64_t)klen * Fmt<FMT>::num / Fmt<FMT>::den);  // per row
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // lane 0 runs the ring's barriers; lane r issues the copies of row r of each stage, so a stage's copies
        // leave in one warp instruction rather than one after another
        if (a.w_from_prev) grid_dependency_wait();  // the workspace is written by the preceding kernel
        const uint64_t pol_w = l2_evict_first();
        int issued = 0;
        bool ok = true;
        if (FMT == FMT_PAL && lane == 0) {
            // first of all, the exponents of the CTA's verbatim blocks: ranks [v_begin, v_end) of the verbatim
            // stream are one contiguous run (the CTA's rows are), of which the first vcap blocks are staged
            uint32_t v_staged = 0;
            uint64_t v_begin = 0;
            if (nrows) {
                const uint64_t fb = (uint64_t)r0 * K / 64, lb = (uint64_t)r1 * K / 64;
                const uint64_t lwd = (lb & 31) ? lb >> 5 : (lb - 1) >> 5;
                const uint32_t bw0 = __ldg(a.w.bitmap + (fb >> 5)), pw0 = __ldg(a.w.prefix + (fb >> 5));
                const uint32_t bw1 = __ldg(a.w.bitmap + lwd), pw1 = __ldg(a.w.prefix + lwd);
                v_begin = pw0 + __popc(bw0 & ((1u << (fb & 31)) - 1u));
                const uint64_t v_end = (lb & 31) ? pw1 + __popc(bw1 & ((1u << (lb & 31)) - 1u)) : pw1 + __popc(bw1);
                v_staged = (uint32_t)min(v_end - v_begin, (uint64_t)a.vcap);
            }
            mbar_arrive_expect_tx(vfull, v_staged * 64);
            if (v_staged) bulk_g2s_hint(vx, a.w.verb_exp + v_begin * 64, v_staged * 64, vfull, pol_w);
        }
        for (int i = 0; i < n_stages; i++) {
            const int slot = i % a.stages;
            const int64_t g0 = r0 + (int64_t)i * a.rs;
            const int nr = (int)min((int64_t)a.rs, r1 - g0);
            const bool whole = a.tmap && nr == a.rs && klen == a.ks;  // one tensor copy per stream: the whole stage
            uint8_t *st = ring + (size_t)slot * a.stage_bytes;
            int go = 1;
            if (lane == 0) {
                if (i >= a.stages && !mbar_wait(&empty[slot], ((i / a.stages) - 1) & 1)) go = 0;
                else {
                    mbar_arrive_expect_tx(&full[slot], wbytes * nr);
                    if (whole) {
                        if (FMT == FMT_BF16) tma3d(st, &a.tm0, 0, (int)(k0 >> 10), (int)g0, &full[slot], pol_w);
                        else {
                            tma3d(st, &a.tm0, 0, (int)(k0 >> 11), (int)g0, &full[slot], pol_w);
                            tma3d(st + a.rs * klen, &a.tm1, 0, (int)(k0 >> 11), (int)g0, &full[slot], pol_w);
                        }
                    }
                }
            }
            if (!__shfl_sync(0xFFFFFFFFu, go, 0)) { ok = false; break; }
            for (int r = whole ? 32 : lane; r < nr; r += 32) {
                const uint64_t off = (uint64_t)(g0 + r) * K + k0;
                if (FMT == FMT_PAL) {
                    bulk_g2s_hint(st + r * klen, a.w.sm + off, klen, &full[slot], pol_w);
                    bulk_g2s_hint(st + a.rs * klen + r * (klen / 2), a.w.codes + off / 2, klen / 2, &full[slot], pol_w);
                } else if (FMT == FMT_EXP) {
                    bulk_g2s_hint(st + r * klen, a.w.sm + off, klen, &full[slot], pol_w);
                    bulk_g2s_hint(st + a.rs * klen + r * klen, a.w.exps + off, klen, &full[slot], pol_w);
                } else {
                    bulk_g2s_hint(st + r * 2 * klen, a.w.w + off, 2 * klen, &full[slot], pol_w);
                }
            }
            issued = i + 1;
        }
        if (lane == 0) {
            // the staged verbatim exponents must land before the CTA may exit
            if (FMT == FMT_PAL && !mbar_wait(vfull, 0)) ok = false;
            if (!ok) {
                atomicExch(a.status, (int)DEV_TIMEOUT);
                // drain: every issued stage's copies must land before the CTA may exit
                for (int i = max(0, issued - a.stages); i < issued; i++) mbar_wait(&full[i % a.stages], (i / a.stages) & 1);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int ctid = threadIdx.x - 32;
    if (FMT == FMT_PAL)
        for (int i = ctid; i < a.bm_words; i += CT) {  // words past the CTA's blocks read as "not verbatim"
            bm[i] = i < n_bw ? __ldg(a.w.bitmap + wb0 + i) : 0u;
            pf[i] = i < n_bw ? __ldg(a.w.prefix + wb0 + i) : 0u;
        }
    for (int i = ctid; i < a.rows_cta * NB; i += CT) part[i] = 0.f;
    const int c = warp - 1;
    const int slot_row = c / a.wk, piece = c % a.wk;
    const int kbase = piece * 32 * LW + 16 * lane;
    if (FMT == FMT_PAL) {
        // entry row b holds the pair for code byte b once per lane: consecutive threads store consecutive
        // 16-byte chunks (bank-conflict free)
        for (int i = ctid; i < 256 * 8; i += CT) {
            const int b = i >> 3, q = i & 7;
            const uint32_t v = ((uint32_t)a.w.palette[b >> 4] << 23) | ((uint32_t)a.w.palette[b & 15] << 7);
            *(uint4 *)(tab + 128 * b + 16 * q) = make_uint4(v, v, v, v);
        }
    }
    grid_dependency_wait();   // X (and Y, written below) belong to the stream order after the preceding kernel
    const uint8_t *tab_lane = tab + 4 * lane;
    asm volatile("bar.sync 1, %0;" ::"r"(CT) : "memory");  // bitmap words and zeroed row sums are in place
    // the CTA's run of verbatim blocks: ranks [v_begin, v_end) of the verbatim stream, the first v_staged of them
    // staged in shared memory by the producer
    uint64_t v_begin = 0;
    uint32_t v_staged = 0;
    bool v_ready = false;
    if (FMT == FMT_PAL && nrows) {
        const uint64_t fb = (uint64_t)r0 * K / 64, lb = (uint64_t)r1 * K / 64;
        v_begin = pf[0] + __popc(bm[0] & ((1u << (fb & 31)) - 1u));
        const uint64_t lw = (lb >> 5) - wb0;
        const uint64_t v_end = lw < (uint64_t)n_bw ? pf[lw] + __popc(bm[lw] & ((1u << (lb & 31)) - 1u))
                                                    : pf[n_bw - 1] + __popc(bm[n_bw - 1]);
        v_staged = (uint32_t)min(v_end - v_begin, (uint64_t)a.vcap);
    }
    uint32_t xr[NB][LW / 2];  // bf16x2 activations of the lane's weights
#pragma unroll
    for (int j = 0; j < NB; j++)
#pragma unroll
        for (int g = 0; g < G; g++) {
            const int kk = kbase + 512 * g;
            uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
            if (kk < klen && b0 + j < a.B) {
                const uint4 *src = (const uint4 *)(a.x + (b0 + j) * K + k0 + kk);
                lo = ldg_hint(src, l2_evict_last());
                hi = ldg_hint(src + 1, l2_evict_last());
            }
#pragma unroll
            for (int q = 0; q < 4; q++) {
                xr[j][8 * g + q] = word_of(lo, q);
                xr[j][8 * g + 4 + q] = word_of(hi, q);
            }
        }
    // block index of the lane's first group in the first stage, relative to the CTA's first bitmap word
    // (32-bit: a CTA's blocks number far fewer than 2^32), advanced by one stage of rows per stage
    uint32_t bl_lane = (uint32_t)((((uint64_t)(r0 + slot_row) * K + k0 + kbase) >> 6) - wb0 * 32);
    const uint32_t bl_step = (uint32_t)((uint64_t)a.rs * K / 64);
    const bool all_groups = kbase + 512 * (G - 1) < klen;  // every group of the lane lies inside the K-slice
    bool ok = true;
    float vs[4][NB];  // lane sums of the last four stages, oldest first, awaiting one joint reduction
#pragma unroll
    for (int q = 0; q < 4; q++)
#pragma unroll
        for (int j = 0; j < NB; j++) vs[q][j] = 0.f;
    for (int i = 0; i < n_stages && ok; i++) {
        const int slot = i % a.stages;
        if (!mbar_wait(&full[slot], (i / a.stages) & 1)) { ok = false; break; }
        const int64_t row = r0 + (int64_t)i * a.rs + slot_row;
        const bool live = row < r1;
        const uint8_t *st = ring + (size_t)slot * a.stage_bytes;
        // the lane's 16 weights of group g: FMT_PAL sm bytes and codes (x1.x/.y); FMT_EXP sm and exponents;
        // bf16 the two halves
        auto load_group = [&](int g, uint4 &x0, uint4 &x1) {
            const int kk = kbase + 512 * g;
            x0 = x1 = make_uint4(0, 0, 0, 0);
            if (live && kk < klen) {
                if (FMT == FMT_PAL) {
                    x0 = *(const uint4 *)(st + slot_row * klen + kk);
                    const uint2 cc = *(const uint2 *)(st + a.rs * klen + slot_row * (klen / 2) + kk / 2);
                    x1.x = cc.x;
                    x1.y = cc.y;
                } else if (FMT == FMT_EXP) {
                    x0 = *(const uint4 *)(st + slot_row * klen + kk);
                    x1 = *(const uint4 *)(st + a.rs * klen + slot_row * klen + kk);
                } else {
                    x0 = *(const uint4 *)(st + slot_row * 2 * klen + 2 * kk);
                    x1 = *(const uint4 *)(st + slot_row * 2 * klen + 2 * kk + 16);
                }
            }
        };
        // small parts are copied into registers at once and the slot goes back to the producer before the
        // compute; larger ones are read group by group and the slot is released after the compute
        constexpr bool kEarly = G * NB <= 4;
        uint4 d0[G], d1[G];
        if (kEarly) {
#pragma unroll
            for (int g = 0; g < G; g++) load_group(g, d0[g], d1[g]);
        }
        // verbatim flags of the lane's groups this stage: bit 8g of `vwin` (groups are 8 blocks apart)
        uint64_t vwin = 0;
        const uint32_t bl0 = bl_lane;
        bl_lane += bl_step;
        if (FMT == FMT_PAL && live) {
            if (G <= 4) {
                const uint64_t w2 = ((uint64_t)bm[(bl0 >> 5) + 1] << 32) | bm[bl0 >> 5];
                vwin = (w2 >> (bl0 & 31)) & (G == 1 ? 0x1ull : G == 2 ? 0x101ull : 0x01010101ull);
            } else {
#pragma unroll
                for (int g = 0; g < G; g++) {
                    const uint32_t bl = bl0 + 8 * g;
                    vwin |= (uint64_t)((bm[bl >> 5] >> (bl & 31)) & 1u) << (8 * g);
                }
            }
        }
        if (kEarly) release_slot(&empty[slot], lane);

        float acc0[NB], acc1[NB];
#pragma unroll
        for (int j = 0; j < NB; j++) acc0[j] = acc1[j] = 0.f;
        // The 16 exponents of the verbatim group of the lane whose block is bl (relative to the CTA's first
        // bitmap word) at K-slice position kk: from the staged run, or from global memory beyond it.
        auto verbatim_exps = [&](uint32_t bl, int kk) -> uint4 {
            const uint32_t wd = bl >> 5;
            const uint64_t rank = (uint64_t)pf[wd] + __popc(bm[wd] & ((1u << (bl & 31)) - 1u));
            const uint64_t vl = rank - v_begin;
            const int q = (kk >> 4) & 3;  // the group's quarter of its 64-weight block
            if (vl < v_staged) {
                if (!v_ready) {  // the first verbatim group this lane meets: the staged run must have landed
                    if (!mbar_wait(vfull, 0)) ok = false;
                    v_ready = true;
                }
                return *(const uint4 *)(vx + vl * 64 + 16 * q);
            }
            return __ldg((const uint4 *)(a.w.verb_exp + rank * 64 + 16 * q));
        };
        // The lane's groups of this stage.  BD: some group of the warp lies past the CTA's rows or the K-slice
        // (those are skipped).  VB: some lane of the warp has a verbatim group; that lane rebuilds the group from
        // the block's own exponents instead of the palette (its codes are all zero).  Without BD the groups are
        // straight-line code.
        auto run_groups = [&](auto BD, auto VB) {
            constexpr bool bd = decltype(BD)::value, vb = decltype(VB)::value;
#pragma unroll
            for (int g = 0; g < G; g++) {
                if (bd && (!live || kbase + 512 * g >= klen)) continue;  // past the CTA's rows or the K-slice
                if (!kEarly) load_group(g, d0[g], d1[g]);
                uint32_t pw[8];  // 8 bf16x2 pairs of weights
                if (FMT == FMT_PAL) {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const uint32_t S = word_of(d0[g], q);
                        const uint32_t Cw = q < 2 ? d1[g].x : d1[g].y;
                        const int jb = 2 * (q & 1);
                        pw[2 * q] = (__byte_perm(S, 0u, 0x1100u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb);
                        pw[2 * q + 1] = (__byte_perm(S, 0u, 0x3322u) & 0x807F807Fu) | pair_exp(tab_lane, Cw, jb + 1);
                    }
                    if (vb && ((vwin >> (8 * g)) & 1u)) {
                        const uint4 E = verbatim_exps(bl0 + 8 * g, kbase + 512 * g);
#pragma unroll
                        for (int q = 0; q < 4; q++) pairs_from_exps(word_of(d0[g], q), word_of(E, q), pw[2 * q], pw[2 * q + 1]);
                    }
                } else if (FMT == FMT_EXP) {
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        pairs_from_exps(word_of(d0[g], q), word_of(d1[g], q), pw[2 * q], pw[2 * q + 1]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; q++) { pw[q] = word_of(d0[g], q); pw[4 + q] = word_of(d1[g], q); }
                }
#pragma unroll
                for (int j = 0; j < NB; j++)
#pragma unroll
                    for (int t = 0; t < 8; t += 2) {
                        acc0[j] = fma2_bf16(pw[t], xr[j][8 * g + t], acc0[j]);
                        acc1[j] = fma2_bf16(pw[t + 1], xr[j][8 * g + t + 1], acc1[j]);
                    }
            }
        };
        // the votes are warp-uniform: every lane of the warp takes the same body
        const unsigned am = __activemask();
        const bool bd = !__all_sync(am, live && all_groups), vb = FMT == FMT_PAL && __any_sync(am, vwin != 0);
        if (!bd) {
            if (!vb) run_groups(std::false_type{}, std::false_type{});
            else run_groups(std::false_type{}, std::true_type{});
        } else {
            run_groups(std::true_type{}, std::true_type{});
        }
        if (!kEarly) release_slot(&empty[slot], lane);
        // shift the lane sum in; every fourth stage (and after the last) reduce four stages at once
#pragma unroll
        for (int j = 0; j < NB; j++) {
            vs[0][j] = vs[1][j];
            vs[1][j] = vs[2][j];
            vs[2][j] = vs[3][j];
            vs[3][j] = acc0[j] + acc1[j];
        }
        if ((i & 3) == 3 || i + 1 == n_stages) {
#pragma unroll
            for (int j = 0; j < NB; j++) {
                const float v = reduce4(vs[0][j], vs[1][j], vs[2][j], vs[3][j], lane);
                const int q = ((lane >> 3) & 2) | ((lane >> 3) & 1);
                const int si = i - 3 + q;  // stage whose row sum this lane holds
                const int64_t rw = r0 + (int64_t)si * a.rs + slot_row;
                // stages before i & ~3 were reduced earlier (their slots hold zeros)
                if ((lane & 7) == 0 && si >= (i & ~3) && rw < r1) atomicAdd(&part[(rw - r0) * NB + j], v);
#pragma unroll
                for (int t = 0; t < 4; t++) vs[t][j] = 0.f;
            }
        }
    }
    if (!ok) atomicExch(a.status, (int)DEV_TIMEOUT);
    asm volatile("bar.sync 1, %0;" ::"r"(CT) : "memory");  // row sums complete
    // write the CTA's rows
    for (int i = ctid; i < nrows * NB; i += C * 32) {
        const int rl = i / NB, j = i - rl * NB;
        if (b0 + j >= a.B) continue;
        const int64_t o = (b0 + j) * N + r0 + rl;
        const float v = part[i];
        if (a.nsplit > 1) atomicAdd(a.acc + o, v);
        else if (a.out_bf16) ((__nv_bfloat16 *)a.y)[o] = __float2bfloat16_rn(v);
        else ((float *)a.y)[o] = v;
    }
}

template <int NB, int LW, int FMT>
cudaError_t launch_one(const TmaArgs &a, dim3 grid, int threads, size_t smem, cudaStream_t st)
{
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemv_tma_kernel<NB, LW, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    return cudaLaunchKernelEx(&cfg, gemv_tma_kernel<NB, LW, FMT>, a);
}

template <int NB, int LW>
cudaError_t launch_lw(int fmt, const TmaArgs &a, dim3 grid, int threads, size_t smem, cudaStream_t st)
{
    if (fmt == FMT_PAL) return launch_one<NB, LW, FMT_PAL>(a, grid, threads, smem, st);
    if (fmt == FMT_EXP) return launch_one<NB, LW, FMT_EXP>(a, grid, threads, smem, st);
    return launch_one<NB, LW, FMT_BF16>(a, grid, threads, smem, st);
}

struct TmaShape {
    int nsplit, ks, lw, wk, rs, stages, stage_bytes, rows_cta, bm_words, vcap, ctas;
    size_t smem;
};

// Pick K-slice, lane width, rows per stage and ring depth for (N, K, B, fmt).
//   max_warps : consumer warps per CTA (8 keeps a CTA at <= 288 threads, so two fit on an SM)
//   per_sm    : CTAs per SM of this launch (1 leaves room for the next launch's CTA)
// X lives in <= 64 bf16x2 registers per lane; shared memory per CTA stays under the per_sm share
// (half of 227 KB when a second CTA - of this launch or of the next one - should fit beside it).
bool plan_shape(const WOperand &w, int64_t B, int split_k, int max_warps, int per_sm, size_t smem_cap, int lw_pref,
                TmaShape &s)
{
    const int nb = B <= 1 ? 1 : 2;
    const int max_x_regs = 64;  // bf16x2 registers: LW/2 per batch row
    int split = std::max(1, split_k);
    for (;; split++) {
        if (split > 64) return false;
        // K-slices of whole 2048-weight chunks when K allows, so stages can move as single tensor copies
        const int gran = w.K % 2048 == 0 ? 2048 : 64;
        const int ks = (int)(((w.K + split - 1) / split + gran - 1) / gran * gran);
        int lw = lw_pref;
        while (lw < 128 && (ks + 32 * lw - 1) / (32 * lw) > max_warps) lw *= 2;
        const int wk = (ks + 32 * lw - 1) / (32 * lw);
        if (wk > max_warps || lw / 2 * nb > max_x_regs) continue;
        s.nsplit = (int)((w.K + ks - 1) / ks);
        s.ks = ks;
        s.lw = lw;
        s.wk = wk;
        break;
    }
    s.rs = std::max(1, std::min(8, max_warps / s.wk));
    const int num = w.fmt == FMT_PAL ? 3 : 4, den = 2;
    s.stage_bytes = (int)(((int64_t)s.rs * s.ks * num / den + 127) / 128 * 128);
    const int groups = (int)((B + nb - 1) / nb);
    s.ctas = std::max(1, num_sms() * per_sm / std::max(1, s.nsplit * groups));
    s.ctas = (int)std::min<int64_t>(s.ctas, (w.N + s.rs - 1) / s.rs);
    s.rows_cta = (int)((w.N + s.ctas - 1) / s.ctas) + 1;
    s.bm_words = (int)((int64_t)s.rows_cta * (w.K / 64) / 32 + 2);
    const size_t fixed = (w.fmt == FMT_PAL ? kTableBytes : 0) + 1024 + ((size_t)s.rows_cta * nb * 4 + 1023) / 1024 * 1024 +
                         2 * (((size_t)s.bm_words * 4 + 1023) / 1024 * 1024);
    if (fixed + 2 * (size_t)s.stage_bytes > smem_cap) return false;
    s.stages = (int)std::min<size_t>(8, (smem_cap - fixed) / s.stage_bytes);
    s.smem = fixed + (size_t)s.stages * s.stage_bytes;
    // exponents of verbatim blocks in the shared memory left over (at most 1024 blocks)
    s.vcap = w.fmt == FMT_PAL ? (int)std::min<size_t>(1024, (smem_cap - s.smem) / 64) : 0;
    s.smem += (size_t)s.vcap * 64;
    return true;
}

// Tensor maps that move one whole stage (rs rows x one K-slice) per stream in a single copy.  A row of a
// stream is split into chunks of 2048 weights (sm and exponent bytes: 2048 B; codes: 1024 B; bf16 weights:
// 1024 weights = 2048 B per chunk), each chunk a run of 8-byte elements, so the box is {chunk, chunks per
// slice, rs} and lands in shared memory row after row exactly like the per-row copies.  Needs K and the
// slice to be whole chunks; otherwise the kernel falls back to per-row bulk copies.
bool make_stage_maps(const WOperand &w, const TmaShape &s, CUtensorMap &m0, CUtensorMap &m1)
{
    auto enc = (PFN_cuTensorMapEncodeTiled_v12000)tensor_map_encoder();
    if (!enc || w.K % 2048 || s.ks % 2048 || w.N <= 0) return false;
    auto make = [&](CUtensorMap &m, const void *base, uint64_t chunk_bytes, uint64_t chunks, uint64_t row_bytes,
                    uint32_t box_chunks) {
        if (!base || ((uintptr_t)base & 15) || box_chunks > 256 || s.rs > 256) return false;
        cuuint64_t dims[3] = {chunk_bytes / 8, chunks, (cuuint64_t)w.N};
        cuuint64_t strides[2] = {chunk_bytes, row_bytes};
        cuuint32_t box[3] = {(cuuint32_t)(chunk_bytes / 8), box_chunks, (cuuint32_t)s.rs};
        cuuint32_t estr[3] = {1, 1, 1};
        return enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    const uint64_t K = (uint64_t)w.K, ks = (uint64_t)s.ks;
    if (w.fmt == FMT_PAL)
        return make(m0, w.sm, 2048, K / 2048, K, (uint32_t)(ks / 2048)) &&
               make(m1, w.codes, 1024, K / 2048, K / 2, (uint32_t)(ks / 2048));
    if (w.fmt == FMT_EXP)
        return make(m0, w.sm, 2048, K / 2048, K, (uint32_t)(ks / 2048)) &&
               make(m1, w.exps, 2048, K / 2048, K, (uint32_t)(ks / 2048));
    return make(m0, w.w, 2048, K / 1024, 2 * K, (uint32_t)(ks / 1024));
}

struct Knobs {
    int max_warps, per_sm;
    size_t cap;
    int lw;
};

// Variants (1 is the plain-load GEMV, not this kernel):
//   0: 8 consumer warps, 2 CTAs/SM, 32 weights per lane and row     4: as 0 with 64 weights per lane
//   2: 16 consumer warps, 1 CTA/SM with all shared memory            5: as 2 with 64 weights per lane
//   3: 8 consumer warps, 1 CTA/SM in half the shared memory (room for the next launch's CTA)
Knobs knobs_of(int variant)
{
    switch (variant) {
    case 2: return Knobs{16, 1, 227 * 1024, 32};
    case 3: return Knobs{8, 1, 113 * 1024, 32};
    case 4: return Knobs{8, 2, 113 * 1024, 64};
    case 5: return Knobs{16, 1, 227 * 1024, 64};
    default: return Knobs{8, 2, 113 * 1024, 32};
    }
}

bool plan_variant(const WOperand &w, int64_t B, int split_k, int variant, TmaShape &s)
{
    const Knobs k = knobs_of(variant);
    return plan_shape(w, B, split_k, k.max_warps, k.per_sm, k.cap, k.lw, s);
}

}  // namespace

bool gemv_tma_supported(const WOperand &w, int64_t B, int variant)
{
    TmaShape s;
    return variant != 1 && B >= 1 && B <= 2 && w.N > 0 && w.K > 0 &&
           plan_variant(w, B, 0, variant, s);
}

int launch_gemv_tma(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, int split_k, int variant,
                    float *acc_ws, int *status, void *stream)
{
    TmaShape s;
    if (!plan_variant(w, B, split_k, variant, s)) return cudaErrorInvalidValue;
    const int nb = B <= 1 ? 1 : 2;
    cudaStream_t st = (cudaStream_t)stream;
    TmaArgs a;
    std::memset(&a, 0, sizeof(a));
    a.w = w;
    a.x = x;
    a.B = B;
    a.y = y;
    a.acc = nullptr;
    a.out_bf16 = out_bf16;
    a.nsplit = s.nsplit;
    a.ks = s.ks;
    a.rs = s.rs;
    a.stages = s.stages;
    a.wk = s.wk;
    a.stage_bytes = s.stage_bytes;
    a.rows_cta = s.rows_cta;
    a.bm_words = s.bm_words;
    a.w_from_prev = w.w_from_prev;
    a.vcap = s.vcap;
    a.status = status;
    a.tmap = make_stage_maps(w, s, a.tm0, a.tm1) ? 1 : 0;
    if (s.nsplit > 1) {
        a.acc = out_bf16 ? acc_ws : (float *)y;
        if (!a.acc) return cudaErrorInvalidValue;
        // zeroed by a kernel, not a memset: this kernel is a dependent launch, and its wait orders it only after
        // a preceding kernel (a memset before it could still be running when its atomics start)
        if ((uintptr_t)a.acc & 15) return cudaErrorInvalidValue;
        cudaError_t e = (cudaError_t)launch_zero_target(a.acc, B * w.N, st);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)s.ctas, (unsigned)s.nsplit, (unsigned)((B + nb - 1) / nb));
    const int threads = 32 * (1 + s.rs * s.wk);
    cudaError_t e;
    if (nb == 1) {
        e = s.lw == 32 ? launch_lw<1, 32>(w.fmt, a, grid, threads, s.smem, st)
          : s.lw == 64 ? launch_lw<1, 64>(w.fmt, a, grid, threads, s.smem, st)
                       : launch_lw<1, 128>(w.fmt, a, grid, threads, s.smem, st);
    } else {
        e = s.lw == 32 ? launch_lw<2, 32>(w.fmt, a, grid, threads, s.smem, st)
                       : launch_lw<2, 64>(w.fmt, a, grid, threads, s.smem, st);
    }
    if (e != cudaSuccess) return e;
    if (s.nsplit > 1 && out_bf16) return launch_finalize(acc_ws, y, B * w.N, 1, stream);
    return cudaSuccess;
}

}  // namespace uw
