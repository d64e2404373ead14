// k_gemv_rp.cu - fused reconstruct + matrix-vector product on the tensor pipe, row-parallel warps (sm_103a),
// batch 1..64, direct-palette operands.
//
// Cloudflare blog "Unweight", section on the reconstructive matmul: the weights are rebuilt from the
// exponent data and the sign+mantissa bytes on chip and fed straight into the product.  This is the
// warp-level tensor-pipe form for small batches: mma.sync m16n8k16 (bf16 in, fp32 accumulate) with sixteen
// rebuilt weight rows as the A operand and the activations as B (N = 8 batch rows per MMA, NB such tiles).
//
// Work is split into units of 128 weight rows x 256 weights of K (the layout of the tile-major verbatim
// stream).  One CTA per SM walks a balanced, contiguous range of units, row block by row block and K
// innermost, so each consumer warp accumulates its rows over the whole range in registers; a run of one row
// block's units (a segment) ends with one fp32 atomic add per output and warp into a zeroed target.
//   - warp 16 (one thread; the warp's lanes prefetch the units' verbatim offsets) TMA-loads per unit two
//     sign+mantissa boxes and one code box of [128 rows x 128 B] with the 128-byte swizzle, the four X tiles
//     [8 NB x 64] bf16 of the unit's K range, the unit's 64-byte verbatim mask and up to kVC of its verbatim
//     blocks; one mbarrier counts the bytes;
//   - warps 0-15: warp w owns the 16 rows 16 (w % 8) .. + 15 of the block for the unit's 64-weight steps
//     2 (w / 8) and 2 (w / 8) + 1 (one sign+mantissa box).  Lane (g, t) = (lane / 4, lane % 4) rebuilds weights
//     16t .. 16t + 15 of rows r0 = 16 (w % 8) + rev3(g) and r0 + 8 (rev3 = 3-bit reversal: with it the
//     swizzled row reads of a warp touch every bank once) from one 16-byte sm piece and 8 code bytes per row,
//     one pair-table lookup per two weights, and issues four MMAs per step and batch tile.  The MMA's logical
//     k is permuted so that each lane's pairs are physically consecutive weights; the X fragments are read
//     from the staged X tile in the same order.  A step holding a verbatim block of the warp's rows rebuilds
//     that block's weights from the staged exponents instead (a warp-uniform test, then a per-lane fix-up).
// Every wait is bounded; on expiry the kernel latches DEV_TIMEOUT, drains its copies and returns.
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

constexpr int kRows = 128;                 // rows per unit
constexpr int kUnitK = 256;                // weights of K per unit (four 64-weight steps)
constexpr int kWarps = 16;                 // consumer warps: 8 groups of 16 rows x 2 halves of the unit's steps
constexpr int kThreads = 32 * (kWarps + 1);
constexpr int kTab = 256 * 128;            // pair table: entry b for lane l at 128 b + 4 l (no bank conflicts)
constexpr uint32_t kBoxBytes = kRows * 128;
constexpr int kSmemCap = 227 * 1024;

// verbatim blocks of a unit staged with it (beyond: global loads); at NB = 4 four, so that the kernel leaves
// 1 KB of the SM's shared memory to the one-warp CTA of the zeroing kernel that runs beside it
__host__ __device__ constexpr int vc_of(int NB) { return NB == 4 ? 4 : 16; }
constexpr int kBarArea = 64;  // the ring's full and empty barriers (at most 3 stages x 2 x 8 bytes)
// ring stages: three up to 32 batch rows, two beyond (the X tiles grow with the batch)
__host__ __device__ constexpr int stages_of(int NB) { return NB <= 4 ? 3 : 2; }
__host__ __device__ constexpr int vslot_of(int NB) { return 64 + vc_of(NB) * 64; }
// one stage: two sm boxes, one code box, four X tiles of 8 NB rows (all 1024-byte multiples)
__host__ __device__ constexpr uint32_t stage_of(int NB) { return 3 * kBoxBytes + 4 * (uint32_t)NB * 1024; }
// dynamic shared memory: alignment slack, table, barriers, verbatim slots, ring
constexpr size_t smem_of(int NB)
{
    return 1024 + kTab + kBarArea + (size_t)stages_of(NB) * (vslot_of(NB) + stage_of(NB));
}
static_assert(smem_of(4) <= (size_t)kSmemCap && smem_of(8) <= (size_t)kSmemCap, "shared memory of the batch shapes");
static_assert(2 * 3 * 8 <= kBarArea, "barrier area");
// each shape leaves room for a one-warp CTA beside it: 228 KB per SM, 1 KB reserved per CTA
static_assert(smem_of(1) + 2048 <= 228 * 1024 && smem_of(2) + 2048 <= 228 * 1024 && smem_of(3) + 2048 <= 228 * 1024 &&
                  smem_of(4) + 2048 <= 228 * 1024 && smem_of(6) + 2048 <= 228 * 1024 && smem_of(8) + 2048 <= 228 * 1024,
              "room for the zeroing kernel's CTA");

struct RpArgs {
    CUtensorMap tm_sm;     // sm [N, K] u8, box {128, 128}, 128-byte swizzle
    CUtensorMap tm_codes;  // codes [N, K/2] u8, box {128, 128}, 128-byte swizzle
    CUtensorMap tm_x;      // X [B, K] bf16, box {64, 8 NB}, 128-byte swizzle
    const uint32_t *tmv_off, *tmv_mask;
    const uint8_t *tmv_data;
    float *acc;            // [B, N] fp32, zeroed before the launch
    int *status;
    int64_t N, B;
    int upk;               // units per row block (K / 256)
    int w_from_prev;       // the codes were written by the preceding kernel (a preprocess workspace)
    int64_t units;
    uint8_t palette[16];
};

// D += A * B, m16n8k16, bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
    return bytes;
}

// eight bf16x2 pairs (weights 16t + 2i, 16t + 2i + 1 in pw[i]) of one row's step from its 16 sign+mantissa
// bytes S and its 8 code bytes C; tab: shared-memory pair table at this lane's column
__device__ __forceinline__ void rebuild16(const uint8_t *tab, const uint4 &S, const uint2 &C, uint32_t (&pw)[8])
{
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const uint32_t Sw = word_of(S, q);
        const uint32_t Cw = q < 2 ? C.x : C.y;
        const uint32_t b0 = prmt(Cw, 0u, 0x4440u | (uint32_t)(2 * (q & 1)));
        const uint32_t b1 = prmt(Cw, 0u, 0x4440u | (uint32_t)(2 * (q & 1) + 1));
        const uint32_t e0 = *(const uint32_t *)(tab + b0 * 128u);
        const uint32_t e1 = *(const uint32_t *)(tab + b1 * 128u);
        pw[2 * q] = (__byte_perm(Sw, 0u, 0x1100u) & 0x807F807Fu) | e0;
        pw[2 * q + 1] = (__byte_perm(Sw, 0u, 0x3322u) & 0x807F807Fu) | e1;
    }
}

__device__ __forceinline__ void rebuild16_exps(const uint4 &S, const uint4 &E, uint32_t (&pw)[8])
{
#pragma unroll
    for (int q = 0; q < 4; q++) pairs_from_exps(word_of(S, q), word_of(E, q), pw[2 * q], pw[2 * q + 1]);
}

// exponents 16t .. 16t + 15 of the verbatim block of (step j, bit bi of mask word wi) of unit u: staged with the
// unit when it is among the first kVC of the unit's verbatim blocks in (step, row) order, else from global memory
template <int kVC>
__device__ __forceinline__ uint4 verbatim_exps(const RpArgs &a, const uint8_t *vs, int wi, uint32_t mw, int bi, int t,
                                               int64_t u)
{
    uint32_t rank = __popc(mw & ((1u << bi) - 1u));
    for (int i = 0; i < wi; i++) rank += __popc(((const uint32_t *)vs)[i]);
    if (rank < (uint32_t)kVC) return *(const uint4 *)(vs + 64 + rank * 64 + 16 * t);
    return __ldg((const uint4 *)(a.tmv_data + ((uint64_t)__ldg(a.tmv_off + u) + rank) * 64 + 16 * t));
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Zeroes the fp32 target of the atomic adds.  Launched as a dependent of the preceding kernel, it lets the
// matmul that follows it start at once (streaming its weights) and zeroes only once the preceding kernel is done.
// One warp per CTA: a CTA this small fits beside a resident matmul CTA (the matmul kernels leave it 1 KB of
// shared memory and the registers of one warp), so every CTA of this grid starts, and lets the next matmul
// launch, while the preceding matmul still runs.  A grid of 256-thread CTAs did not fit beside them and held
// the next launch back until the preceding one had drained.
constexpr int kZeroThreads = 32;
__global__ void __launch_bounds__(kZeroThreads) zero_target_kernel(float4 *p, int64_t n4, float *tail, int n_tail)
{
    grid_launch_dependents();
    grid_dependency_wait();
    const int64_t stride = (int64_t)gridDim.x * kZeroThreads;
    int64_t i = blockIdx.x * (int64_t)kZeroThreads + threadIdx.x;
    for (; i + 3 * stride < n4; i += 4 * stride) {
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        p[i + stride] = make_float4(0.f, 0.f, 0.f, 0.f);
        p[i + 2 * stride] = make_float4(0.f, 0.f, 0.f, 0.f);
        p[i + 3 * stride] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (; i < n4; i += stride) p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (blockIdx.x == 0 && (int)threadIdx.x < n_tail) tail[threadIdx.x] = 0.f;
}

// NB: batch tiles of 8 rows (B <= 8 NB)
template <int NB>
__global__ void __launch_bounds__(kThreads, 1) gemv_rp_kernel(const __grid_constant__ RpArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    constexpr uint32_t kStage = stage_of(NB);
    constexpr int kStages = stages_of(NB);
    constexpr int kVC = vc_of(NB), kVSlot = vslot_of(NB);
    constexpr uint32_t kXTile = (uint32_t)NB * 1024;  // one X tile: 8 NB rows x 128 B
    const uint32_t pad = (1024u - (saddr(smem_raw) & 1023u)) & 1023u;
    uint8_t *ring = smem_raw + pad;                   // [kStages][kStage], 1024-aligned
    uint8_t *tab = ring + kStages * kStage;           // [kTab]
    uint64_t *full = (uint64_t *)(tab + kTab);        // [kStages]
    uint64_t *empty = full + kStages;                 // [kStages]
    uint8_t *vslots = tab + kTab + kBarArea;          // [kStages][kVSlot]: 64-byte mask, then staged blocks

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t U = a.units, G = gridDim.x;
    const int64_t u0 = U * blockIdx.x / G, u1 = U * (blockIdx.x + 1) / G;
    const int nu = (int)(u1 - u0);
    const int upk = a.upk;

    if (threadIdx.x == 32 * kWarps) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // a dependent launch may start its prologue and stream its own weights from here on
    grid_launch_dependents();

    if (warp == kWarps) {
        // -------------------------------------------------------------------------------- producer
        uint32_t o0 = 0, o1 = 0;  // lane l: verbatim offsets of unit u0 + 32 * window + l and the next one
        int64_t tile = u0 / upk;
        int kq = (int)(u0 % upk), s = 0, issued = 0;
        uint32_t ph = 0;
        bool ok = true;
        // the weights (unless a preprocess kernel just wrote them) are not the preceding kernel's: the first
        // stages' weight copies leave before the wait for it, their X tiles after it
        if (a.w_from_prev) grid_dependency_wait();
        const int primed = a.w_from_prev ? 0 : min(nu, kStages);
        for (int c = 0; c < nu; c++) {
            const int64_t u = u0 + c;
            if (c == primed && primed > 0 && lane == 0) {
                grid_dependency_wait();
                int k2 = (int)(u0 % upk);
                for (int i = 0; i < primed; i++) {
                    uint8_t *st = ring + i * kStage;
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        tma2d(st + 3 * kBoxBytes + j * kXTile, &a.tm_x, k2 * kUnitK + 64 * j, 0, &full[i]);
                    if (++k2 == upk) k2 = 0;
                }
            }
            if ((c & 31) == 0) {
                const int64_t ul = u + lane;
                o0 = ul <= U ? __ldg(a.tmv_off + ul) : 0u;
                o1 = ul + 1 <= U ? __ldg(a.tmv_off + ul + 1) : 0u;
            }
            const uint32_t start = __shfl_sync(0xFFFFFFFFu, o0, c & 31);
            const uint32_t nv = min(__shfl_sync(0xFFFFFFFFu, o1, c & 31) - start, (uint32_t)kVC);
            int go = 1;
            if (lane == 0) {
                if (c >= kStages && !mbar_wait(&empty[s], ph ^ 1u)) go = 0;
                else {
                    const int kw = kq * kUnitK, row0 = (int)(tile * kRows);
                    uint8_t *st = ring + s * kStage;
                    uint8_t *vs = vslots + s * kVSlot;
                    const uint32_t fb = saddr(&full[s]);
                    mbar_expect_tx(&full[s], 3 * kBoxBytes + 4 * kXTile + 64u + 64u * nv);
                    tma2d(st, &a.tm_sm, kw, row0, &full[s]);
                    tma2d(st + kBoxBytes, &a.tm_sm, kw + 128, row0, &full[s]);
                    tma2d(st + 2 * kBoxBytes, &a.tm_codes, kw / 2, row0, &full[s]);
                    if (c >= primed) {
#pragma unroll
                        for (int j = 0; j < 4; j++)
                            tma2d(st + 3 * kBoxBytes + j * kXTile, &a.tm_x, kw + 64 * j, 0, &full[s]);
                    }
                    bulk_copy(saddr(vs), a.tmv_mask + 16 * u, 64u, fb);
                    if (nv) bulk_copy(saddr(vs + 64), a.tmv_data + (uint64_t)start * 64, nv * 64u, fb);
                }
            }
            if (!__shfl_sync(0xFFFFFFFFu, go, 0)) { ok = false; break; }
            issued = c + 1;
            if (++kq == upk) { kq = 0; tile++; }
            if (++s == kStages) { s = 0; ph ^= 1u; }
        }
        if (lane == 0 && primed > 0 && nu == primed) {
            // every unit fit in the first stages: their X tiles still have to leave
            grid_dependency_wait();
            int k2 = (int)(u0 % upk);
            for (int i = 0; i < primed; i++) {
#pragma unroll
                for (int j = 0; j < 4; j++)
                    tma2d(ring + i * kStage + 3 * kBoxBytes + j * kXTile, &a.tm_x, k2 * kUnitK + 64 * j, 0, &full[i]);
                if (++k2 == upk) k2 = 0;
            }
        }
        if (lane == 0 && !ok) {
            atomicExch(a.status, (int)DEV_TIMEOUT);
            for (int c = max(0, issued - kStages); c < issued; c++) mbar_wait(&full[c % kStages], (c / kStages) & 1);
        }
        return;
    }

    // ------------------------------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    const int rg = warp & 7, hh = warp >> 3;
    const int pg = ((g & 1) << 2) | (g & 2) | (g >> 2);  // 3-bit reversal of g
    const int r0 = 16 * rg + pg;                          // this lane rebuilds rows r0 and r0 + 8 of the block
    const uint8_t *tab_l = tab + 4 * lane;
    // byte offsets within a stage for row r0 (row r0 + 8 is 1024 bytes further, with the same swizzle phase)
    uint32_t o_sm[2], o_c[2];
#pragma unroll
    for (int jj = 0; jj < 2; jj++) {
        o_sm[jj] = hh * kBoxBytes + r0 * 128 + (((4 * jj + t) ^ pg) << 4);
        o_c[jj] = 2 * kBoxBytes + r0 * 128 + (((4 * hh + 2 * jj + (t >> 1)) ^ pg) << 4) + 8 * (t & 1);
    }
    const uint32_t o_x0 = 3 * kBoxBytes + 2 * hh * kXTile + g * 128 + (((2 * t) ^ g) << 4);
    const uint32_t o_x1 = 3 * kBoxBytes + 2 * hh * kXTile + g * 128 + (((2 * t + 1) ^ g) << 4);
    const int wi_base = rg >> 1, bsh = 16 * (rg & 1);
    fill_pair_table(tab, a.palette, threadIdx.x, 32 * kWarps);
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kWarps) : "memory");  // the table, among the consumer warps
    grid_dependency_wait();  // the target is zeroed by the preceding kernel

    float acc[NB][4];
#pragma unroll
    for (int n = 0; n < NB; n++)
#pragma unroll
        for (int e = 0; e < 4; e++) acc[n][e] = 0.f;
    // a finished segment: acc[n][e] is row r0 + 8 (e / 2), batch row 8n + 2t + e % 2; added into the target
    auto flush = [&](int64_t tl) {
#pragma unroll
        for (int n = 0; n < NB; n++)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int64_t b = 8 * n + 2 * t + (e & 1);
                const int64_t row = tl * kRows + r0 + 8 * (e >> 1);
                if (b < a.B && row < a.N) atomicAdd(a.acc + b * a.N + row, acc[n][e]);
                acc[n][e] = 0.f;
            }
    };
    bool ok = true;
    int64_t tile = u0 / upk, seg_t = tile;
    int kq = (int)(u0 % upk), s = 0;
    uint32_t ph = 0;
    for (int c = 0; c < nu; c++) {
        if (tile != seg_t) {
            flush(seg_t);
            seg_t = tile;
        }
        if (!mbar_wait(&full[s], ph)) { ok = false; break; }
        const uint8_t *st = ring + s * kStage;
        const uint8_t *vs = vslots + s * kVSlot;
#pragma unroll
        for (int jj = 0; jj < 2; jj++) {
            const int j = 2 * hh + jj;
            const uint4 S0 = *(const uint4 *)(st + o_sm[jj]);
            const uint4 S1 = *(const uint4 *)(st + o_sm[jj] + 1024);
            const uint2 C0 = *(const uint2 *)(st + o_c[jj]);
            const uint2 C1 = *(const uint2 *)(st + o_c[jj] + 1024);
            uint32_t p0[8], p1[8];
            rebuild16(tab_l, S0, C0, p0);
            rebuild16(tab_l, S1, C1, p1);
            const int wi = 4 * j + wi_base;
            const uint32_t mw = *(const uint32_t *)(vs + 4 * wi);
            if ((mw >> bsh) & 0xFFFFu) {
                // a verbatim block among the warp's 16 rows at this step (the same word for every lane)
                const int64_t u = u0 + c;
                if ((mw >> (bsh + pg)) & 1u) rebuild16_exps(S0, verbatim_exps<kVC>(a, vs, wi, mw, bsh + pg, t, u), p0);
                if ((mw >> (bsh + pg + 8)) & 1u)
                    rebuild16_exps(S1, verbatim_exps<kVC>(a, vs, wi, mw, bsh + pg + 8, t, u), p1);
                __syncwarp();  // the MMAs need the warp converged after the per-lane branches
            }
#pragma unroll
            for (int n = 0; n < NB; n++) {
                // X row 8n + g: the lane's 16 values 16t .. 16t + 15 of the step (two 16-byte pieces)
                const uint4 xa = *(const uint4 *)(st + o_x0 + jj * kXTile + n * 1024);
                const uint4 xb = *(const uint4 *)(st + o_x1 + jj * kXTile + n * 1024);
                const uint32_t xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                for (int q = 0; q < 4; q++) mma16816(acc[n], p0[2 * q], p1[2 * q], p0[2 * q + 1], p1[2 * q + 1], xv[2 * q], xv[2 * q + 1]);
            }
        }
        // the stage was read with generic-proxy loads and the next tensor copy into it writes through the async
        // proxy: each lane fences its reads across the proxies before the warp hands the stage back
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++kq == upk) { kq = 0; tile++; }
        if (++s == kStages) { s = 0; ph ^= 1u; }
    }
    if (ok) flush(seg_t);
    else atomicExch(a.status, (int)DEV_TIMEOUT);
}

bool make_map_rp(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer)
{
    auto fn = (PFN_cuTensorMapEncodeTiled_v12000)tensor_map_encoder();
    if (!fn || !base || ((uintptr_t)base & 15)) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool rp_shape(const WOperand &w, int64_t B, int *nb, int64_t *units)
{
    if (B < 1 || B > 64 || w.fmt != FMT_PAL || w.N <= 0 || w.K <= 0 || w.K % kUnitK) return false;
    if (w.N > (int64_t)INT32_MAX - kRows || w.K > (int64_t)INT32_MAX) return false;
    if (!w.tmv_off || !w.tmv_mask || !w.tmv_data || !w.codes || !tensor_map_encoder()) return false;
    *nb = (int)((B + 7) / 8);
    if (*nb > 4) *nb = *nb <= 6 ? 6 : 8;
    *units = (w.N + kRows - 1) / kRows * (w.K / kUnitK);
    return true;
}

template <int NB>
cudaError_t launch_rp_nb(const RpArgs &a, int grid, cudaStream_t st)
{
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemv_rp_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_of(NB));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = smem_of(NB);
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_rp_kernel<NB>, a);
}


}  // namespace

int launch_zero_target(float *p, int64_t n, void *stream)
{
    const int64_t n4 = n / 4;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((n4 + kZeroThreads - 1) / kZeroThreads, (int64_t)num_sms()));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3((unsigned)kZeroThreads);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, zero_target_kernel, (float4 *)p, n4, p + 4 * n4, (int)(n - 4 * n4));
}

bool gemv_rp_supported(const WOperand &w, int64_t B)
{
    int nb;
    int64_t units;
    return rp_shape(w, B, &nb, &units);
}

int launch_gemv_rp(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, float *acc_ws, void *stream)
{
    int nb;
    int64_t units;
    if (!rp_shape(w, B, &nb, &units)) return cudaErrorInvalidValue;
    cudaStream_t st = (cudaStream_t)stream;
    RpArgs a;
    memset(&a, 0, sizeof a);
    const uint64_t N = (uint64_t)w.N, K = (uint64_t)w.K;
    bool ok = make_map_rp(&a.tm_sm, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.sm, K, N, K, 128, kRows) &&
              make_map_rp(&a.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, K / 2, N, K / 2, 128, kRows) &&
              make_map_rp(&a.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, (uint64_t)B, K * 2, 64, (uint32_t)(8 * nb));
    if (!ok) return cudaErrorInvalidValue;
    a.tmv_off = w.tmv_off;
    a.tmv_mask = w.tmv_mask;
    a.tmv_data = w.tmv_data;
    a.status = w.status;
    a.N = w.N;
    a.B = B;
    a.upk = (int)(w.K / kUnitK);
    a.units = units;
    memcpy(a.palette, w.palette, 16);
    // a row block's partial sums come from both halves of the warps and possibly from two CTAs: all add into a
    // zeroed fp32 target
    a.acc = out_bf16 ? acc_ws : (float *)y;
    if (!a.acc) return cudaErrorInvalidValue;
    a.w_from_prev = w.w_from_prev;
    if ((uintptr_t)a.acc & 15) return cudaErrorInvalidValue;
    cudaError_t e = (cudaError_t)launch_zero_target(a.acc, B * w.N, st);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(num_sms(), units);
    switch (nb) {
    case 1: e = launch_rp_nb<1>(a, grid, st); break;
    case 2: e = launch_rp_nb<2>(a, grid, st); break;
    case 3: e = launch_rp_nb<3>(a, grid, st); break;
    case 4: e = launch_rp_nb<4>(a, grid, st); break;
    case 6: e = launch_rp_nb<6>(a, grid, st); break;
    default: e = launch_rp_nb<8>(a, grid, st); break;
    }
    if (e != cudaSuccess) return e;
    if (out_bf16) return launch_finalize(acc_ws, y, B * w.N, 1, stream);
    return cudaSuccess;
}

}  // namespace uw
