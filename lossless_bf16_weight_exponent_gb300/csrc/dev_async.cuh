// dev_async.cuh - device helpers shared by the matmul kernels: mbarriers with bounded waits, bulk and tensor
// copies into shared memory, and the tcgen05 tensor-memory operations.  Inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace uw {
namespace dev {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait: far above any legitimate stall

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

// Wait until the barrier's phase with this parity completes; false after kWaitLimitNs.
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
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr)
{
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major), 16 bytes
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 1024 bytes between 8-row groups
    d |= (uint64_t)1 << 46;            // descriptor version for this architecture family
    d |= (uint64_t)2 << 61;            // layout: 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, both K-major, M x N
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem descriptor] * B[smem descriptor]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
                     d_tmem),
                 "l"(a), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
}

// D[tmem] (+)= A[tmem: row m in lane m, k pairs in consecutive 32-bit columns] * B[smem descriptor]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
                     d_tmem),
                 "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
}

// arrive on the barrier once every MMA issued so far by this thread has completed
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar)) : "memory");
}

// 32 consecutive 32-bit TMEM columns of this warp's 32 lanes <- 32 registers of each thread
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes -> 16 registers of each thread
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
        "[%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// bf16x2 pairs (weights 0,1 and 2,3) from four sign+mantissa bytes and four exponent bytes
__device__ __forceinline__ void pairs_from_exps(uint32_t S, uint32_t E, uint32_t &p01, uint32_t &p23)
{
    const uint32_t hi = (S & 0x80808080u) | ((E >> 1) & 0x7F7F7F7Fu);
    const uint32_t lo = (S & 0x7F7F7F7Fu) | ((E << 7) & 0x80808080u);
    p01 = __byte_perm(lo, hi, 0x5140u);
    p23 = __byte_perm(lo, hi, 0x7362u);
}

// Per-lane palette pair table (32 KB): for a code byte b (codes c0 = b & 15, c1 = b >> 4) the exponent fields
// of the bf16x2 pair, (pal[c1] << 23) | (pal[c0] << 7), at byte offset 128*b + 4*lane: a warp's lookups never
// share a bank.
constexpr int kPairTableBytes = 256 * 128;

__device__ __forceinline__ void fill_pair_table(uint8_t *tab, const uint8_t *palette, int tid, int nthreads)
{
    for (int i = tid; i < 256 * 8; i += nthreads) {
        const int b = i >> 3, q = i & 7;
        const uint32_t v = ((uint32_t)palette[b >> 4] << 23) | ((uint32_t)palette[b & 15] << 7);
        *(uint4 *)(tab + 128 * b + 16 * q) = make_uint4(v, v, v, v);
    }
}

__device__ __forceinline__ uint32_t pair_exp(const uint8_t *tab_lane, uint32_t C, int j)
{
    const uint32_t b = prmt(C, 0u, 0x4440u | (uint32_t)j);  // byte j of C
    return *(const uint32_t *)(tab_lane + b * 128u);
}

// ---------------------------------------------------------------------------- row blocks shared by CTAs
// A persistent kernel over a balanced partition of row-block units stores a row block that one CTA covers and
// combines a block that several CTAs share through three 8-byte cells of the caller's workspace, tagged with the
// launch's epoch so that they need no zeroing: the adders' count ((epoch << 24) | count), the flag (the epoch,
// once the storing CTA's sums are visible) and a spare.

struct TileCells {
    unsigned long long done, flag, spare;
};

// count one more in a tagged cell of this epoch (a cell of another epoch counts as 0); returns the count before
__device__ __forceinline__ uint32_t tagged_count(unsigned long long *cell, unsigned long long epoch)
{
    unsigned long long cur = *(volatile unsigned long long *)cell;
    for (;;) {
        const unsigned long long nxt = (cur >> 24) == epoch ? cur + 1 : (epoch << 24) | 1ull;
        const unsigned long long prev = atomicCAS(cell, cur, nxt);
        if (prev == cur) return (uint32_t)(nxt & 0xFFFFFFu) - 1u;
        cur = prev;
    }
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// the CTA holding unit u of a balanced partition of U units over G CTAs (u0(b) = U b / G)
__device__ __forceinline__ int64_t cta_of_unit(int64_t u, int64_t U, int64_t G) { return ((u + 1) * G - 1) / U; }

}  // namespace dev
}  // namespace uw
