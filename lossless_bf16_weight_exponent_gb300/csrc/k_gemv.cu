// k_gemv.cu - fused reconstruct + GEMV on CUDA cores (sm_103a), batch groups of <= 8.
//
// Cloudflare blog "Unweight", section on the reconstructive matmul: compressed
// weights are read from HBM, BF16 is rebuilt on-chip (here in registers, as fp32
// bit patterns: fp32 bits = bf16 bits << 16) and consumed at once, so the
// uncompressed matrix never travels through HBM.  The same kernel also serves
// the exponent-only pipeline (sign+mantissa bytes + exponent bytes) and the
// full-decode pipeline (plain BF16 weights).
//
// Shape of the work: a CTA of 8 warps owns 16 rows of W (2 per warp) and one
// K-slice; its slice of X (up to 8 batch rows) sits in shared memory as fp32 in
// a bank-conflict-free swizzle.  Lane l of a warp reads 16 consecutive weights of
// each of its two rows per step (a 16-byte sign+mantissa load, an 8-byte code
// load), so a warp step covers 512 weights with fully coalesced loads.  Weight
// reconstruction per element: one byte permute (sm byte to bits 31..16), one
// palette lookup of (exponent << 23) from a 16-entry shared table, one LOP3.
// Verbatim blocks (one bitmap test per 16 weights; a block never straddles a
// lane's 16) take their exponents from the verbatim stream instead.
// K-splits accumulate with fp32 atomics into Y (fp32 output) or into a
// workspace that a finalize kernel converts to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "uw_internal.h"

namespace uw {

namespace {

struct GemvArgs {
    WOperand w;
    const uint16_t *x;
    int64_t B;
    void *y;        // final output (nsplit == 1)
    float *acc;     // fp32 accumulation target (nsplit > 1)
    int out_bf16;
    int nsplit;
    int64_t ks;     // K-slice length (multiple of 64)
};

__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_stream8(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// raw compressed data of 16 weights of one row
template <int FMT> struct Raw;
template <> struct Raw<FMT_PAL> { uint4 s; uint2 c; uint32_t bw; };
template <> struct Raw<FMT_EXP> { uint4 s; uint4 e; };
template <> struct Raw<FMT_BF16> { uint4 lo, hi; };

template <int FMT>
__device__ __forceinline__ void load_raw(const WOperand &w, uint64_t off, Raw<FMT> &r)
{
    if constexpr (FMT == FMT_PAL) {
        r.s = ld_stream16(w.sm + off);
        r.c = ld_stream8(w.codes + off / 2);
        r.bw = __ldg(w.bitmap + (off >> 11));
    } else if constexpr (FMT == FMT_EXP) {
        r.s = ld_stream16(w.sm + off);
        r.e = ld_stream16(w.exps + off);
    } else {
        r.lo = ld_stream16(w.w + off);
        r.hi = ld_stream16(w.w + off + 8);
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// bf16x2 from 4 sign+mantissa bytes S and 4 exponent bytes E: returns the pairs (w1:w0) and (w3:w2).
__device__ __forceinline__ void pairs_from_exps(uint32_t S, uint32_t E, uint32_t &p01, uint32_t &p23)
{
    const uint32_t hi = (S & 0x80808080u) | ((E >> 1) & 0x7F7F7F7Fu);   // sign | exponent bits 7..1
    const uint32_t lo = (S & 0x7F7F7F7Fu) | ((E << 7) & 0x80808080u);   // exponent bit 0 | mantissa
    p01 = __byte_perm(lo, hi, 0x5140u);
    p23 = __byte_perm(lo, hi, 0x7362u);
}

// fp32 values of a bf16x2 pair: low half then high half
__device__ __forceinline__ void unpack2(uint32_t p, float &f0, float &f1)
{
    f0 = __uint_as_float(p * 65536u);  // a multiply keeps this shift off the integer ALU pipe
    f1 = __uint_as_float(p & 0xFFFF0000u);
}

// Palette pair table: for a code byte b (codes c0 = b & 15, c1 = b >> 4) the exponent fields of a bf16x2
// pair, (pal[c1] << 23) | (pal[c0] << 7).  Replicated for each of the 32 lanes at byte offset b*128 + 4*lane,
// so a warp's 32 lookups always touch 32 different banks.
constexpr int kPairTableBytes = 256 * 32 * 4;

__device__ __forceinline__ uint32_t pair_exp(const uint8_t *tab_lane, uint32_t C, int j)
{
    // byte j of C, times 128
    const uint32_t off = (j == 0 ? (C << 7) : (C >> (8 * j - 7))) & 0x7F80u;
    return *(const uint32_t *)(tab_lane + off);
}

template <int FMT>
__device__ __forceinline__ void rebuild16(const WOperand &w, uint64_t off, const Raw<FMT> &r, const uint8_t *tab_lane,
                                          float *f)
{
    if constexpr (FMT == FMT_PAL) {
        const uint64_t b = off >> 6;
        if (__builtin_expect((r.bw >> (b & 31)) & 1u, 0)) {
            const uint64_t vi = __ldg(w.prefix + (b >> 5)) + __popc(r.bw & ((1u << (b & 31)) - 1u));
            const uint4 ev = __ldg((const uint4 *)(w.verb_exp + vi * 64 + (off & 63)));
#pragma unroll
            for (int q = 0; q < 4; q++) {
                uint32_t p01, p23;
                pairs_from_exps(word_of(r.s, q), word_of(ev, q), p01, p23);
                unpack2(p01, f[4 * q], f[4 * q + 1]);
                unpack2(p23, f[4 * q + 2], f[4 * q + 3]);
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const uint32_t S = word_of(r.s, q);
                const uint32_t C = q < 2 ? r.c.x : r.c.y;
                const int j = 2 * (q & 1);
                const uint32_t p01 = (__byte_perm(S, 0u, 0x1100u) & 0x807F807Fu) | pair_exp(tab_lane, C, j);
                const uint32_t p23 = (__byte_perm(S, 0u, 0x3322u) & 0x807F807Fu) | pair_exp(tab_lane, C, j + 1);
                unpack2(p01, f[4 * q], f[4 * q + 1]);
                unpack2(p23, f[4 * q + 2], f[4 * q + 3]);
            }
        }
    } else if constexpr (FMT == FMT_EXP) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t p01, p23;
            pairs_from_exps(word_of(r.s, q), word_of(r.e, q), p01, p23);
            unpack2(p01, f[4 * q], f[4 * q + 1]);
            unpack2(p23, f[4 * q + 2], f[4 * q + 3]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; i++) unpack2(word_of(i < 4 ? r.lo : r.hi, i & 3), f[2 * i], f[2 * i + 1]);
    }
}

// logical 4-float chunk c of the X slice lives at chunk (c & ~3) | ((c & 3) ^ ((c >> 3) & 3))
__device__ __forceinline__ int swz_chunk(int c) { return (c & ~3) | ((c & 3) ^ ((c >> 3) & 3)); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

template <int NB, int FMT>
__global__ void __launch_bounds__(256) gemv_kernel(GemvArgs a)
{
    extern __shared__ float4 xs4[];
    const int64_t N = a.w.N, K = a.w.K;
    const int64_t k0 = (int64_t)blockIdx.y * a.ks;
    const int klen = (int)(a.ks < K - k0 ? a.ks : K - k0);
    const int ksp = (int)a.ks;  // row pitch of the X slice (floats)
    const int64_t b0 = (int64_t)blockIdx.z * NB;
    uint8_t *tab = (uint8_t *)(xs4 + NB * (ksp / 4));
    if constexpr (FMT == FMT_PAL) {
        for (int i = threadIdx.x; i < 256 * 32; i += blockDim.x) {
            const int b = i >> 5;
            ((uint32_t *)tab)[i] = ((uint32_t)a.w.palette[b >> 4] << 23) | ((uint32_t)a.w.palette[b & 15] << 7);
        }
    }

    // X slice -> fp32, swizzled
    const int chunks = klen / 4;
    for (int i = threadIdx.x; i < NB * chunks; i += blockDim.x) {
        const int j = i / chunks, c = i - j * chunks;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b0 + j < a.B) {
            const uint2 raw = *(const uint2 *)(a.x + (b0 + j) * K + k0 + 4 * c);
            v = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                            __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
        }
        xs4[j * (ksp / 4) + swz_chunk(c)] = v;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint8_t *tab_lane = tab + 4 * lane;
    const int64_t row0 = (int64_t)blockIdx.x * 16 + warp * 2;
    const bool ok0 = row0 < N, ok1 = row0 + 1 < N;
    const uint64_t base0 = (uint64_t)row0 * K + k0, base1 = base0 + K;
    float acc[2][NB];
#pragma unroll
    for (int r = 0; r < 2; r++)
#pragma unroll
        for (int j = 0; j < NB; j++) acc[r][j] = 0.f;

    int kk = lane * 16;
    Raw<FMT> cur0, cur1, nxt0, nxt1;
    if (kk < klen) {
        if (ok0) load_raw<FMT>(a.w, base0 + kk, cur0);
        if (ok1) load_raw<FMT>(a.w, base1 + kk, cur1);
    }
    for (; kk < klen; kk += 512) {
        const int kn = kk + 512;
        if (kn < klen) {
            if (ok0) load_raw<FMT>(a.w, base0 + kn, nxt0);
            if (ok1) load_raw<FMT>(a.w, base1 + kn, nxt1);
        }
        float w0[16], w1[16];
        if (ok0) rebuild16<FMT>(a.w, base0 + kk, cur0, tab_lane, w0);
        else {
#pragma unroll
            for (int i = 0; i < 16; i++) w0[i] = 0.f;
        }
        if (ok1) rebuild16<FMT>(a.w, base1 + kk, cur1, tab_lane, w1);
        else {
#pragma unroll
            for (int i = 0; i < 16; i++) w1[i] = 0.f;
        }
        const int c0 = kk >> 2;
        const int sw = (c0 >> 3) & 3;
#pragma unroll
        for (int j = 0; j < NB; j++) {
            const float4 *xr = xs4 + j * (ksp / 4) + c0;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float4 xv = xr[q ^ sw];
                acc[0][j] = fmaf(w0[4 * q + 0], xv.x, acc[0][j]);
                acc[1][j] = fmaf(w1[4 * q + 0], xv.x, acc[1][j]);
                acc[0][j] = fmaf(w0[4 * q + 1], xv.y, acc[0][j]);
                acc[1][j] = fmaf(w1[4 * q + 1], xv.y, acc[1][j]);
                acc[0][j] = fmaf(w0[4 * q + 2], xv.z, acc[0][j]);
                acc[1][j] = fmaf(w1[4 * q + 2], xv.z, acc[1][j]);
                acc[0][j] = fmaf(w0[4 * q + 3], xv.w, acc[0][j]);
                acc[1][j] = fmaf(w1[4 * q + 3], xv.w, acc[1][j]);
            }
        }
        cur0 = nxt0;
        cur1 = nxt1;
    }

#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int64_t row = row0 + r;
#pragma unroll
        for (int j = 0; j < NB; j++) {
            const float v = warp_sum(acc[r][j]);
            if (lane == 0 && row < N && b0 + j < a.B) {
                const int64_t o = (b0 + j) * N + row;
                if (a.nsplit > 1) atomicAdd(a.acc + o, v);
                else if (a.out_bf16) ((__nv_bfloat16 *)a.y)[o] = __float2bfloat16_rn(v);
                else ((float *)a.y)[o] = v;
            }
        }
    }
}

__global__ void finalize_kernel(const float *acc, void *y, int64_t count, int out_bf16)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count; i += (int64_t)gridDim.x * blockDim.x) {
        if (out_bf16) ((__nv_bfloat16 *)y)[i] = __float2bfloat16_rn(acc[i]);
        else ((float *)y)[i] = acc[i];
    }
}

constexpr int64_t kMaxSlice = 160 * 1024;  // bytes of X slice per CTA
constexpr int kMaxSmem = (int)kMaxSlice + kPairTableBytes;

template <int NB, int FMT>
cudaError_t launch_nb(const GemvArgs &a, dim3 grid, size_t smem, cudaStream_t st)
{
    static bool attr_set = false;  // set once, outside any stream capture (first call is never captured)
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NB, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kMaxSmem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    gemv_kernel<NB, FMT><<<grid, 256, smem, st>>>(a);
    return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_fmt(int nb, const GemvArgs &a, dim3 grid, size_t smem, cudaStream_t st)
{
    switch (nb) {
    case 1: return launch_nb<1, FMT>(a, grid, smem, st);
    case 2: return launch_nb<2, FMT>(a, grid, smem, st);
    case 4: return launch_nb<4, FMT>(a, grid, smem, st);
    default: return launch_nb<8, FMT>(a, grid, smem, st);
    }
}

int batch_group(int64_t B) { return B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8; }

}  // namespace

int gemv_default_split(const WOperand &w, int64_t B)
{
    const int nb = batch_group(B);
    const int64_t tiles = (w.N + 15) / 16 * ((B + nb - 1) / nb);
    const int64_t target = 4LL * num_sms();
    int64_t split = tiles >= target ? 1 : (target + tiles - 1) / tiles;
    split = std::min<int64_t>(split, std::max<int64_t>(1, w.K / 512));
    while ((int64_t)nb * ((w.K + split - 1) / split) * 4 > 96 * 1024) split++;
    return (int)split;
}

int launch_gemv(const WOperand &w, const uint16_t *x, int64_t B, void *y, int out_bf16, int split_k, int variant,
                float *acc_ws, void *stream)
{
    if (B <= 0 || w.N == 0) return cudaSuccess;
    cudaStream_t st = (cudaStream_t)stream;
    if ((variant == 6 || variant == 7) && w.K > 0 && gemv_mma_supported(w, B, variant)) {
        const int e = launch_gemv_mma(w, x, B, y, out_bf16, split_k, variant, acc_ws, w.status, stream);
        if (e != cudaErrorInvalidValue) return e;  // else: no tensor map for these operands, use the CUDA-core GEMV
    }
    if (variant == 8 && gemv_rp_supported(w, B)) {
        const int e = launch_gemv_rp(w, x, B, y, out_bf16, acc_ws, stream);
        if (e != cudaErrorInvalidValue) return e;  // else: no tensor map for these operands
    }
    if (variant != 1 && w.K > 0) {
        // the default (variant 0) falls back to the one-CTA-per-SM shape when two CTAs do not fit
        const int v = (variant == 0 || variant > 5) && !gemv_tma_supported(w, B, 0) ? 2 : variant > 5 ? 0 : variant;
        if (gemv_tma_supported(w, B, v)) return launch_gemv_tma(w, x, B, y, out_bf16, split_k, v, acc_ws, w.status, stream);
    }
    const int nb = batch_group(B);
    if (w.K == 0) {
        size_t bytes = (size_t)B * w.N * (out_bf16 ? 2 : 4);
        return cudaMemsetAsync(y, 0, bytes, st);
    }
    int split = split_k > 0 ? split_k : gemv_default_split(w, B);
    int64_t ks = (w.K + split - 1) / split;
    ks = (ks + 63) / 64 * 64;
    while ((int64_t)nb * ks * 4 > kMaxSlice) { split++; ks = ((w.K + split - 1) / split + 63) / 64 * 64; }
    const int nsplit = (int)((w.K + ks - 1) / ks);
    GemvArgs a{w, x, B, y, nullptr, out_bf16, nsplit, ks};
    const size_t count = (size_t)B * w.N;
    if (nsplit > 1) {
        a.acc = out_bf16 ? acc_ws : (float *)y;
        if (!a.acc) return cudaErrorInvalidValue;
        cudaError_t e = cudaMemsetAsync(a.acc, 0, count * 4, st);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)((w.N + 15) / 16), (unsigned)nsplit, (unsigned)((B + nb - 1) / nb));
    const size_t smem = (size_t)nb * ks * 4 + (w.fmt == FMT_PAL ? kPairTableBytes : 0);
    cudaError_t e;
    if (w.fmt == FMT_PAL) e = launch_fmt<FMT_PAL>(nb, a, grid, smem, st);
    else if (w.fmt == FMT_EXP) e = launch_fmt<FMT_EXP>(nb, a, grid, smem, st);
    else e = launch_fmt<FMT_BF16>(nb, a, grid, smem, st);
    if (e != cudaSuccess) return e;
    if (nsplit > 1 && out_bf16) return launch_finalize(acc_ws, y, (int64_t)count, 1, stream);
    return cudaSuccess;
}

int launch_finalize(const float *acc, void *y, int64_t count, int out_bf16, void *stream)
{
    if (!count) return cudaSuccess;
    int blocks = (int)std::min<int64_t>((count + 255) / 256, (int64_t)num_sms() * 8);
    finalize_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(acc, y, count, out_bf16);
    return cudaGetLastError();
}

}  // namespace uw
