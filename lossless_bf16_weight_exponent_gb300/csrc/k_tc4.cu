// k_tc4.cu - persistent fused reconstruct + tcgen05 GEMM with the rebuilt weights in shared memory (sm_103a),
// B <= 512, direct-palette operands.
//
// Cloudflare blog "Unweight", section on the reconstructive matmul: compressed inputs are staged by the copy
// engine, rebuilt on chip and consumed by the tensor cores at once, so the bf16 matrix never reaches HBM.
// One CTA per SM walks a balanced, contiguous range of units (128 rows of W x 256 weights of K, the units of the
// tile-major verbatim stream), row block by row block with K innermost; a unit is four 64-weight steps.
//   - warp 16 (one thread; lanes prefetch the units' verbatim offsets and mask words) TMA-loads per step the
//     sign+mantissa box [128 rows x 64 B] and the code box [128 x 32 B] (dense rows), the unit's 64-byte verbatim
//     mask and up to kVCs of the step's verbatim blocks into a deep ring of weight stages, each freed as soon as
//     it is rebuilt;
//   - warp 17 (one thread) TMA-loads the activation tile X [BN x 64] bf16 of each step (128-byte swizzle) into
//     its own ring, each stage freed when the step's MMAs complete;
//   - warps 0-15 rebuild each step: thread (row, chunk) turns 8 sign+mantissa bytes and 4 code bytes into 8
//     bf16 (one pair-table lookup per two weights) and stores them as one 16-byte chunk of the K-major
//     128-byte-swizzled A tile; a warp's reads cover whole 128-byte lines and its stores one chunk of every
//     bank group, so neither conflicts;
//   - warp 18 (one thread) issues per step four tcgen05.mma (M = 128, N = BN <= 256, K = 16; two per K-slice
//     above 256) from the A tile and the X tile into the tensor-memory accumulator of the current segment (a run
//     of units of one row block); two accumulator buffers when they fit;
//   - warps 19-26 write a finished segment.  A segment that covers its whole row block (every unit of K) is
//     stored at once (fp32, or rounded to bf16).  A row block shared by several CTAs is combined through two
//     cells of the workspace tagged with the launch's epoch, so they need no zeroing.  The CTA whose range
//     starts inside the block has the block's last units as its first segment and finishes its share early:
//     it stores the share and raises the block's flag.  The others (the block's first units end their
//     ranges) wait for the flag and add theirs with fp32 atomics.  With two sharers and fp32 output the adder
//     then clears the flag; otherwise the adders count themselves, and the last rounds the block to bf16 when
//     that is the output and clears the cells.  No kernel zeroes the target first, so nothing waits on a
//     zeroing pass between launches.
// Every wait is bounded; on expiry the kernel latches DEV_TIMEOUT, drains its copies and MMAs and frees TMEM.
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

constexpr int kRows = 128;            // rows per unit (the MMA's M)
constexpr int kUnitK = 256;           // weights of K per unit
constexpr int kStepK = 64;            // weights of K per step (one 128-byte swizzle row of bf16)
constexpr int kRebuildWarps = 16;
constexpr int kProdWarp = 16;
constexpr int kXWarp = 17;
constexpr int kMmaWarp = 18;
constexpr int kEpiWarp0 = 19;
constexpr int kEpiWarps = 8;          // two per tensor-memory lane quarter
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr uint32_t kSmBytes = kRows * 64;      // sign+mantissa box of a step
constexpr uint32_t kCodeBytes = kRows * 32;    // code box of a step
constexpr uint32_t kVOff = kSmBytes + kCodeBytes;
constexpr int kVCs = 8;                        // verbatim blocks of a step staged with it (beyond: global loads)
constexpr uint32_t kWStage = 13312;            // sm box, code box, verbatim slot (64 + 8 x 64 bytes); 1024-aligned
constexpr uint32_t kASlot = kRows * 128;       // a rebuilt A tile [128 x 64] bf16
constexpr int kTab = 256 * 64;                 // pair table, 16 replicas: entry b for lane l at 64 b + 4 (l % 16)
constexpr int kMaxSW = 8, kMaxSX = 6, kMaxSA = 4;
constexpr uint32_t kBarBytes = 512;
constexpr size_t kSmemCap = 227 * 1024;
static_assert(kVOff + 64 + kVCs * 64 <= kWStage, "weight stage layout");
static_assert((2 * kMaxSW + 2 * kMaxSX + 2 * kMaxSA + 5) * 8 + 4 <= kBarBytes, "barrier region");

struct Tc4Args {
    CUtensorMap tm_sm;     // sm [N, K] u8, box {64, 128}, dense
    CUtensorMap tm_codes;  // codes [N, K/2] u8, box {32, 128}, dense
    CUtensorMap tm_x;      // X [B, K] bf16, box {64, min(BN, 256)}, 128-byte swizzle
    const uint32_t *tmv_off, *tmv_mask;
    const uint8_t *tmv_data;
    void *y;               // [B, N] fp32 or bf16
    float *acc;            // [B, N] fp32 workspace rows of the shared row blocks (bf16 output only)
    TileCells *cells;      // one per 128-row tile
    unsigned long long epoch;  // this launch's tag (40 bits, never 0)
    int out_bf16;
    int *status;
    int64_t N, B, units;
    int upk, BN, SW, SX, SA, nbuf, buf_stride, tmem_cols, w_from_prev;
    uint8_t palette[16];
};

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// generic-proxy writes to shared memory made visible to the tensor cores (async proxy)
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// four bf16x2 pairs of 8 weights from 8 sign+mantissa bytes (S0, S1) and 4 code bytes C
__device__ __forceinline__ uint4 rebuild8(const uint8_t *tab, uint32_t S0, uint32_t S1, uint32_t C)
{
    uint32_t p[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const uint32_t Sw = q < 2 ? S0 : S1;
        const uint32_t b = prmt(C, 0u, 0x4440u | (uint32_t)q);
        const uint32_t e = *(const uint32_t *)(tab + b * 64u);
        p[q] = (__byte_perm(Sw, 0u, (q & 1) ? 0x3322u : 0x1100u) & 0x807F807Fu) | e;
    }
    return make_uint4(p[0], p[1], p[2], p[3]);
}

__device__ __forceinline__ uint4 rebuild8_exps(uint32_t S0, uint32_t S1, uint32_t E0, uint32_t E1)
{
    uint4 r;
    pairs_from_exps(S0, E0, r.x, r.y);
    pairs_from_exps(S1, E1, r.z, r.w);
    return r;
}

// pair table with 16 replicas: for a code byte b the exponent fields of the bf16x2 pair, (pal[b >> 4] << 23) |
// (pal[b & 15] << 7), at byte offset 64 b + 4 r for replica r
__device__ __forceinline__ void fill_pair_table16(uint8_t *tab, const uint8_t *palette, int tid, int nthreads)
{
    for (int i = tid; i < 256 * 4; i += nthreads) {
        const int b = i >> 2, q = i & 3;
        const uint32_t v = ((uint32_t)palette[b >> 4] << 23) | ((uint32_t)palette[b & 15] << 7);
        *(uint4 *)(tab + 64 * b + 16 * q) = make_uint4(v, v, v, v);
    }
}

__global__ void __launch_bounds__(kThreads, 1) tc4_kernel(const __grid_constant__ Tc4Args a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t pad = (1024u - (saddr(smem_raw) & 1023u)) & 1023u;
    const int SW = a.SW, SX = a.SX, SA = a.SA;
    const uint32_t XB = (uint32_t)a.BN * 128;        // one X tile
    uint8_t *wring = smem_raw + pad;                 // [SW][kWStage]: sm box, code box, verbatim slot
    uint8_t *xring = wring + SW * kWStage;           // [SX][XB]: X tiles, 128-byte swizzle
    uint8_t *aslots = xring + SX * XB;               // [SA][kASlot]: rebuilt A tiles, 128-byte swizzle
    uint8_t *tab = aslots + SA * kASlot;             // [kTab]
    uint64_t *wfull = (uint64_t *)(tab + kTab);      // [SW] a step's weight copies landed
    uint64_t *wempty = wfull + kMaxSW;               // [SW] the step was rebuilt
    uint64_t *xfull = wempty + kMaxSW;               // [SX] a step's X tile landed
    uint64_t *xempty = xfull + kMaxSX;               // [SX] the step's MMAs completed
    uint64_t *afull = xempty + kMaxSX;               // [SA] an A tile is rebuilt
    uint64_t *aempty = afull + kMaxSA;               // [SA] an A tile's MMAs completed
    uint64_t *accfull = aempty + kMaxSA;             // [2] a segment's MMAs completed
    uint64_t *accempty = accfull + 2;                // [2] a segment's accumulator was read out
    uint64_t *done = accempty + 2;                   // [1] every MMA of the CTA completed
    uint32_t *tmem_slot = (uint32_t *)(done + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t U = a.units, G = gridDim.x;
    const int64_t u0 = U * blockIdx.x / G, u1 = U * (blockIdx.x + 1) / G;
    const int nu = (int)(u1 - u0);
    const int nsteps = 4 * nu;
    const int upk = a.upk;
    const int XR = a.BN <= 256 ? a.BN : a.BN / 2;  // X rows per MMA (the MMA's N)

    if (threadIdx.x == 32 * kProdWarp) {
        for (int s = 0; s < SW; s++) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wempty[s], kRebuildWarps);
        }
        for (int s = 0; s < SX; s++) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], 1);
        }
        for (int s = 0; s < SA; s++) {
            mbar_init(&afull[s], kRebuildWarps);
            mbar_init(&aempty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&accfull[b], 1);
            mbar_init(&accempty[b], kEpiWarps);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // a dependent launch may start its prologue from here on
    grid_launch_dependents();

    if (warp == kProdWarp) {
        // ---------------------------------------------------------------------------------------- weight copies
        // the weights are not the preceding kernel's unless a preprocess kernel just wrote them
        if (a.w_from_prev) grid_dependency_wait();
        bool ok = true;
        int64_t tile = u0 / upk;
        int kq = (int)(u0 % upk), s = 0, issued = 0;
        uint32_t ph = 0, o0 = 0;
        // lane l < 16: word l of the unit's verbatim mask ([step l / 4][row word l % 4]); the next unit's in flight
        uint32_t mw_cur = lane < 16 ? __ldg(a.tmv_mask + 16 * u0 + lane) : 0u;
        uint32_t mw_nxt = (lane < 16 && nu > 1) ? __ldg(a.tmv_mask + 16 * (u0 + 1) + lane) : 0u;
        for (int i = 0; i < nsteps; i++) {
            const int j = i & 3, c = i >> 2;
            const int64_t u = u0 + c;
            if (j == 0) {
                if ((c & 31) == 0) o0 = u + lane < U ? __ldg(a.tmv_off + u + lane) : 0u;  // 32 units' offsets
                if (c > 0) {
                    mw_cur = mw_nxt;
                    mw_nxt = (lane < 16 && c + 1 < nu) ? __ldg(a.tmv_mask + 16 * (u + 1) + lane) : 0u;
                }
            }
            const uint32_t voff = __shfl_sync(0xFFFFFFFFu, o0, c & 31);
            const uint32_t pc = __popc(mw_cur);
            const uint32_t cnt = __reduce_add_sync(0xFFFFFFFFu, (lane >> 2) == j ? pc : 0u);
            const uint32_t pre = __reduce_add_sync(0xFFFFFFFFu, (lane >> 2) < j ? pc : 0u);
            int go = 1;
            if (lane == 0) {
                if (i >= SW && !mbar_wait(&wempty[s], ph ^ 1u)) go = 0;
                else {
                    const uint32_t nv = min(cnt, (uint32_t)kVCs);
                    uint8_t *st = wring + s * kWStage;
                    const int kx = kq * kUnitK + j * kStepK, row0 = (int)(tile * kRows);
                    const uint32_t fb = saddr(&wfull[s]);
                    mbar_expect_tx(&wfull[s], kSmBytes + kCodeBytes + 64u + 64u * nv);
                    tma2d(st, &a.tm_sm, kx, row0, &wfull[s]);
                    tma2d(st + kSmBytes, &a.tm_codes, kx / 2, row0, &wfull[s]);
                    bulk_copy(saddr(st + kVOff), a.tmv_mask + 16 * u, 64u, fb);
                    if (nv) bulk_copy(saddr(st + kVOff + 64), a.tmv_data + (uint64_t)(voff + pre) * 64, nv * 64u, fb);
                }
            }
            if (!__shfl_sync(0xFFFFFFFFu, go, 0)) { ok = false; break; }
            issued = i + 1;
            if (j == 3 && ++kq == upk) { kq = 0; tile++; }
            if (++s == SW) { s = 0; ph ^= 1u; }
        }
        if (lane == 0 && !ok) {
            atomicExch(a.status, (int)DEV_TIMEOUT);
            for (int i = max(0, issued - SW); i < issued; i++) mbar_wait(&wfull[i % SW], (i / SW) & 1);
        }
    } else if (warp == kXWarp) {
        // ---------------------------------------------------------------------------------------- X copies
        if (lane == 0) {
            grid_dependency_wait();  // X may be the preceding kernel's output
            bool ok = true;
            int kq = (int)(u0 % upk), s = 0, issued = 0;
            uint32_t ph = 0;
            for (int i = 0; i < nsteps; i++) {
                const int j = i & 3;
                if (i >= SX && !mbar_wait(&xempty[s], ph ^ 1u)) { ok = false; break; }
                uint8_t *xt = xring + s * XB;
                const int kx = kq * kUnitK + j * kStepK;
                mbar_expect_tx(&xfull[s], XB);
                tma2d(xt, &a.tm_x, kx, 0, &xfull[s]);
                if (a.BN > 256) tma2d(xt + (uint32_t)XR * 128, &a.tm_x, kx, XR, &xfull[s]);
                issued = i + 1;
                if (j == 3 && ++kq == upk) kq = 0;
                if (++s == SX) { s = 0; ph ^= 1u; }
            }
            if (!ok) {
                atomicExch(a.status, (int)DEV_TIMEOUT);
                for (int i = max(0, issued - SX); i < issued; i++) mbar_wait(&xfull[i % SX], (i / SX) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t id = idesc_bf16(kRows, XR);
            bool ok = true, first = false;
            int sx = 0, sa = 0, seg = -1, buf = 0;
            uint32_t phx = 0, pha = 0;
            int64_t tile = u0 / upk, seg_t = -1;
            int kq = (int)(u0 % upk);
            for (int i = 0; i < nsteps; i++) {
                const int j = i & 3;
                if (j == 0 && tile != seg_t) {
                    // a new segment: its accumulator buffer must have been read out
                    seg++;
                    buf = seg % a.nbuf;
                    if (seg >= a.nbuf && !mbar_wait(&accempty[buf], ((seg / a.nbuf) - 1) & 1)) { ok = false; break; }
                    first = true;
                    seg_t = tile;
                }
                if (!mbar_wait(&afull[sa], pha) || !mbar_wait(&xfull[sx], phx)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a_base = saddr(aslots + sa * kASlot);
                const uint32_t x_base = saddr(xring + sx * XB);
                const uint32_t d = tmem + (uint32_t)(buf * a.buf_stride);
#pragma unroll
                for (int kk = 0; kk < kStepK / 16; kk++) {
                    const uint32_t acc_flag = (first && kk == 0) ? 0u : 1u;
                    const uint64_t ad = smem_desc_sw128(a_base + 32 * kk);
                    mma_ss(d, ad, smem_desc_sw128(x_base + 32 * kk), id, acc_flag);
                    if (a.BN > 256)
                        mma_ss(d + (uint32_t)XR, ad, smem_desc_sw128(x_base + (uint32_t)XR * 128 + 32 * kk), id, acc_flag);
                }
                first = false;
                mma_commit(&aempty[sa]);
                mma_commit(&xempty[sx]);
                if (j == 3) {
                    const bool last_unit = (i >> 2) + 1 == nu;
                    if (++kq == upk) { kq = 0; tile++; }
                    if (last_unit || tile != seg_t) mma_commit(&accfull[buf]);
                }
                if (++sx == SX) { sx = 0; phx ^= 1u; }
                if (++sa == SA) { sa = 0; pha ^= 1u; }
            }
            if (!ok) {
                atomicExch(a.status, (int)DEV_TIMEOUT);
                // the epilogue still waits for its segments: let it through (the status marks the result)
                mma_commit(&accfull[0]);
                mma_commit(&accfull[1]);
            }
            // every MMA issued has completed before the accumulators are freed
            mma_commit(done);
            if (!mbar_wait(done, 0)) atomicExch(a.status, (int)DEV_TIMEOUT);
        }
    } else if (warp < kRebuildWarps) {
        // ---------------------------------------------------------------------------------------- rebuild
        fill_pair_table16(tab, a.palette, threadIdx.x, 32 * kRebuildWarps);
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kRebuildWarps) : "memory");
        const uint8_t *tab_l = tab + 4 * (lane & 15);
        const int c = lane & 7;  // 16-byte chunk (8 weights) of the row
        bool ok = true;
        int s = 0, sa = 0;
        uint32_t ph = 0, pha = 0;
        for (int i = 0; i < nsteps; i++) {
            const int j = i & 3;
            if (!mbar_wait(&wfull[s], ph)) { ok = false; break; }
            if (i >= SA && !mbar_wait(&aempty[sa], pha ^ 1u)) { ok = false; break; }
            const uint8_t *st = wring + s * kWStage;
            uint8_t *at = aslots + sa * kASlot;
            const uint32_t *mk = (const uint32_t *)(st + kVOff);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int r = 4 * warp + (lane >> 3) + 64 * h;
                const uint2 Sv = *(const uint2 *)(st + r * 64 + 8 * c);
                const uint32_t Cv = *(const uint32_t *)(st + kSmBytes + r * 32 + 4 * c);
                uint4 v = rebuild8(tab_l, Sv.x, Sv.y, Cv);
                const int wi = 4 * j + (r >> 5);
                const uint32_t mw = mk[wi];
                if ((mw >> ((4 * warp + 64 * h) & 31)) & 0xFu) {
                    // a verbatim block among the warp's four rows (the same word and bits for every lane)
                    if ((mw >> (r & 31)) & 1u) {
                        uint32_t rs = __popc(mw & ((1u << (r & 31)) - 1u));
                        for (int w2 = 4 * j; w2 < wi; w2++) rs += __popc(mk[w2]);
                        uint2 E;
                        if (rs < (uint32_t)kVCs) E = *(const uint2 *)(st + kVOff + 64 + rs * 64 + 8 * c);
                        else {
                            uint32_t pre = 0;
                            for (int w2 = 0; w2 < 4 * j; w2++) pre += __popc(mk[w2]);
                            const int64_t u = u0 + (i >> 2);
                            E = __ldg((const uint2 *)(a.tmv_data + ((uint64_t)__ldg(a.tmv_off + u) + pre + rs) * 64 + 8 * c));
                        }
                        v = rebuild8_exps(Sv.x, Sv.y, E.x, E.y);
                    }
                    __syncwarp();
                }
                *(uint4 *)(at + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4)) = v;
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&wempty[s]);
                mbar_arrive(&afull[sa]);
            }
            if (++s == SW) { s = 0; ph ^= 1u; }
            if (++sa == SA) { sa = 0; pha ^= 1u; }
        }
        if (!ok) atomicExch(a.status, (int)DEV_TIMEOUT);
    } else {
        // ---------------------------------------------------------------------------------------- epilogue
        grid_dependency_wait();  // Y and the workspace may belong to the preceding kernel
        const int q = warp & 3, half = (warp - kEpiWarp0) >> 2;
        const int et = threadIdx.x - 32 * kEpiWarp0;  // 0 .. 255 over the epilogue warps
        const bool lead = et == 0;
        const uint32_t t_lane = (uint32_t)(32 * q) << 16;
        volatile uint32_t *bcast = tmem_slot + 1;  // the lead thread's word to the other epilogue threads
        auto epi_sync = [] { asm volatile("bar.sync 2, %0;" ::"r"(32 * kEpiWarps) : "memory"); };
        int64_t tile = u0 / upk;
        int kq = (int)(u0 % upk), seg = 0;
        for (int cu = 0; cu < nu; cu++) {
            const int64_t t_cur = tile;
            if (++kq == upk) { kq = 0; tile++; }
            if (cu + 1 < nu && tile == t_cur) continue;
            // segment seg (row block t_cur) is complete once its accumulator is
            const int buf = seg % a.nbuf;
            const bool got = mbar_wait(&accfull[buf], (seg / a.nbuf) & 1);
            if (!got) atomicExch(a.status, (int)DEV_TIMEOUT);
            tc_fence_after();
            // the CTAs that share the row block: one of them (whole) or several (combined through its cells); the
            // one holding the block's last unit starts its range inside the block and stores its share
            const int64_t b_lo = cta_of_unit(t_cur * upk, U, G), b_hi = cta_of_unit(t_cur * upk + upk - 1, U, G);
            const bool whole = b_lo == b_hi;
            const bool storer = !whole && (int64_t)blockIdx.x == b_hi;
            const bool counted = !whole && (a.out_bf16 || b_hi - b_lo >= 2);  // adders count themselves
            TileCells *cell = a.cells + t_cur;
            if (!whole && !storer) {
                if (lead) {
                    // the stored share must be visible before this one is added (bounded wait)
                    const uint64_t t0 = gtime();
                    while (ld_acquire(&cell->flag) != a.epoch)
                        if (gtime() - t0 > kWaitLimitNs) {
                            atomicExch(a.status, (int)DEV_TIMEOUT);
                            break;
                        }
                }
                epi_sync();
            }
            const int64_t row = t_cur * kRows + 32 * q + lane;
            float *tf = a.out_bf16 ? a.acc : (float *)a.y;  // where a shared block's sums meet
            for (int c0 = 16 * half; c0 < a.B; c0 += 32) {
                uint32_t v[16];
                tmem_ld16(tmem + t_lane + (uint32_t)(buf * a.buf_stride + c0), v);
                tmem_wait_ld();
                if (row < a.N) {
#pragma unroll
                    for (int e = 0; e < 16; e++) {
                        if (c0 + e >= a.B) break;
                        const int64_t o = (int64_t)(c0 + e) * a.N + row;
                        const float f = __uint_as_float(v[e]);
                        if (whole) {
                            if (a.out_bf16) ((__nv_bfloat16 *)a.y)[o] = __float2bfloat16_rn(f);
                            else ((float *)a.y)[o] = f;
                        } else if (storer) {
                            tf[o] = f;
                        } else {
                            atomicAdd(tf + o, f);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accempty[buf]);
            if (storer) {
                // the share is visible at gpu scope before the flag
                __threadfence();
                epi_sync();
                if (lead) st_release(&cell->flag, a.epoch);
            } else if (!whole && !counted) {
                // the only adder: the flag goes back to no epoch (a CUDA graph replays this launch with the same one)
                if (lead) cell->flag = 0ull;
            } else if (counted) {
                __threadfence();
                epi_sync();
                if (lead) {
                    const uint32_t d = tagged_count(&cell->done, a.epoch);
                    __threadfence();
                    *bcast = d + 1 == (uint32_t)(b_hi - b_lo) ? 1u : 0u;
                }
                epi_sync();
                if (*bcast) {
                    // the block's last adder: every share is in
                    __threadfence();
                    if (a.out_bf16) {
                        for (int i = et; i < kRows * (int)a.B; i += 32 * kEpiWarps) {
                            const int64_t rr = t_cur * kRows + (i % kRows);
                            const int64_t o = (int64_t)(i / kRows) * a.N + rr;
                            if (rr < a.N) ((__nv_bfloat16 *)a.y)[o] = __float2bfloat16_rn(__ldcg(a.acc + o));
                        }
                    }
                    if (lead) {
                        cell->done = 0ull;
                        cell->flag = 0ull;
                    }
                }
                epi_sync();  // the broadcast word is free again
            }
            seg++;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
    }
}

bool make_map4(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
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

struct Tc4Shape {
    int BN, SW, SX, SA, nbuf, buf_stride, tmem_cols;
    int64_t units;
    size_t smem;
};

size_t tc4_smem(const Tc4Shape &s)
{
    return 1024 + (size_t)s.SW * kWStage + (size_t)s.SX * s.BN * 128 + (size_t)s.SA * kASlot + kTab + kBarBytes;
}

bool tc4_shape(const WOperand &w, int64_t B, Tc4Shape &s)
{
    if (B < 1 || B > 512 || w.fmt != FMT_PAL || w.N <= 0 || w.K <= 0 || w.K % kUnitK) return false;
    if (w.N > (int64_t)INT32_MAX - kRows || w.K > (int64_t)INT32_MAX) return false;
    if (!w.tmv_off || !w.tmv_mask || !w.tmv_data || !w.codes || !tensor_map_encoder()) return false;
    s.BN = B <= 256 ? (int)((B + 15) / 16 * 16) : (int)((B + 31) / 32 * 32);
    // A tiles, then X tiles (about 96 KB of them; two above 128 batch rows), then as many weight stages as fit.
    // Above 128 batch rows a third A tile in place of the third X tile was 3% faster at 256 rows (8B and 70B
    // gate); at 512 rows the two X tiles of 64 KB leave room for two A tiles only.
    s.SA = s.BN <= 256 ? 3 : 2;
    s.SX = s.BN <= 128 ? std::max(2, std::min(kMaxSX, 98304 / (s.BN * 128))) : 2;
    s.SW = 0;
    const size_t base = tc4_smem(s);
    if (base + 3 * (size_t)kWStage > kSmemCap) return false;
    s.SW = (int)std::min<size_t>(kMaxSW, (kSmemCap - base) / kWStage);
    s.nbuf = s.BN <= 256 ? 2 : 1;
    s.buf_stride = s.BN <= 128 ? 128 : 256;
    s.tmem_cols = s.BN <= 128 ? 256 : 512;
    s.units = (w.N + kRows - 1) / kRows * (w.K / kUnitK);
    s.smem = tc4_smem(s);
    return s.smem <= kSmemCap;
}

}  // namespace

bool tc4_supported(const WOperand &w, int64_t B)
{
    Tc4Shape s;
    return tc4_shape(w, B, s);
}

int launch_tc4(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, float *acc_ws, void *stream)
{
    Tc4Shape s;
    if (!tc4_shape(w, B, s)) return cudaErrorInvalidValue;
    cudaStream_t st = (cudaStream_t)stream;
    Tc4Args a;
    memset(&a, 0, sizeof a);
    const uint64_t N = (uint64_t)w.N, K = (uint64_t)w.K;
    const int XR = s.BN <= 256 ? s.BN : s.BN / 2;
    bool ok = make_map4(&a.tm_sm, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.sm, K, N, K, 64, kRows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map4(&a.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, K / 2, N, K / 2, 32, kRows,
                        CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map4(&a.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, (uint64_t)B, K * 2, 64, (uint32_t)XR,
                        CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;
    a.tmv_off = w.tmv_off;
    a.tmv_mask = w.tmv_mask;
    a.tmv_data = w.tmv_data;
    a.status = w.status;
    a.N = w.N;
    a.B = B;
    a.units = s.units;
    a.upk = (int)(w.K / kUnitK);
    a.BN = s.BN;
    a.SW = s.SW;
    a.SX = s.SX;
    a.SA = s.SA;
    a.nbuf = s.nbuf;
    a.buf_stride = s.buf_stride;
    a.tmem_cols = s.tmem_cols;
    a.w_from_prev = w.w_from_prev;
    memcpy(a.palette, w.palette, 16);
    // a row block shared by several CTAs meets in Y (fp32) or in the workspace's accumulator (bf16), through its
    // cells after the accumulator region; nothing needs zeroing
    if (!acc_ws || ((uintptr_t)acc_ws & 15) || !y || ((uintptr_t)y & 15)) return cudaErrorInvalidValue;
    a.y = y;
    a.acc = acc_ws;
    a.cells = (TileCells *)((uint8_t *)acc_ws + acc_region_bytes(B, w.N));
    a.out_bf16 = out_bf16;
    a.epoch = next_launch_epoch();
    cudaError_t e = cudaSuccess;
    static bool attr = false;
    if (!attr) {
        e = cudaFuncSetAttribute(tc4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemCap);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(num_sms(), s.units));
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = s.smem;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc4_kernel, a);
}

}  // namespace uw
