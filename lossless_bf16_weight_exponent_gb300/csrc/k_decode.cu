// k_decode.cu - decode / preprocess kernels (sm_103a).
//
// Cloudflare blog "Unweight", section on the four execution pipelines: the
// full-decode pipeline rebuilds BF16 into HBM; the exponent-only pipeline writes
// only exponent bytes; the palette-transcode pipeline turns the Huffman stream
// into 4-bit palette codes; the section on the decode kernels puts the Huffman
// lookup table in shared memory.
//
// Palette decode: one thread per 16 weights (16-byte sign+mantissa load, 8-byte
// code load), one verbatim test per 16 weights (a 64-weight block never splits).
// Huffman decode: one thread per chunk of C weights, 64-bit bit buffer, a
// 2^L-entry decode table in shared memory; a stream that does not end exactly at
// its chunk's end offset, or hits an unassigned prefix, latches DEV_CORRUPT.
#include <cuda_runtime.h>

#include "uw_internal.h"

namespace uw {

__device__ __forceinline__ uint4 ldg_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ldg_stream8(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t byte_of(const uint4 &v, int i)
{
    uint32_t w = i < 4 ? v.x : i < 8 ? v.y : i < 12 ? v.z : v.w;
    return (w >> (8 * (i & 3))) & 0xFF;
}

// bf16 pair (lo, hi) from sm and exponent bytes
__device__ __forceinline__ uint32_t bf16_of(uint32_t sm, uint32_t e)
{
    return ((sm & 0x80u) << 8) | (e << 7) | (sm & 0x7Fu);
}

// ------------------------------------------------------------------------------ palette decode
template <int OUT>
__global__ void __launch_bounds__(256) decode_palette_kernel(DevView v, void *out)
{
    __shared__ uint32_t pal[16];
    if (threadIdx.x < 16) pal[threadIdx.x] = v.palette[threadIdx.x];
    __syncthreads();
    const uint64_t n = (uint64_t)v.N * (uint64_t)v.K;
    const uint64_t groups = n / 16;
    for (uint64_t g = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; g < groups; g += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t off = g * 16;
        const uint64_t b = g >> 2;
        uint4 s = ldg_stream16(v.sm + off);
        uint32_t bw = __ldg(v.bitmap + (b >> 5));
        uint32_t e[16];
        if ((bw >> (b & 31)) & 1u) {
            uint64_t vi = __ldg(v.prefix + (b >> 5)) + __popc(bw & ((1u << (b & 31)) - 1u));
            uint4 ev = ldg_stream16(v.verb_exp + vi * 64 + (g & 3) * 16);
#pragma unroll
            for (int i = 0; i < 16; i++) e[i] = byte_of(ev, i);
        } else {
            uint2 c = ldg_stream8(v.codes + off / 2);
#pragma unroll
            for (int i = 0; i < 16; i++) e[i] = pal[((i < 8 ? c.x : c.y) >> (4 * (i & 7))) & 15u];
        }
        if (OUT == DEC_BF16) {
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 8; i++)
                h[i] = bf16_of(byte_of(s, 2 * i), e[2 * i]) | (bf16_of(byte_of(s, 2 * i + 1), e[2 * i + 1]) << 16);
            uint4 *o = (uint4 *)((uint16_t *)out + off);
            o[0] = make_uint4(h[0], h[1], h[2], h[3]);
            o[1] = make_uint4(h[4], h[5], h[6], h[7]);
        } else {
            uint32_t q[4];
#pragma unroll
            for (int i = 0; i < 4; i++) q[i] = e[4 * i] | (e[4 * i + 1] << 8) | (e[4 * i + 2] << 16) | (e[4 * i + 3] << 24);
            *(uint4 *)((uint8_t *)out + off) = make_uint4(q[0], q[1], q[2], q[3]);
        }
    }
}

int launch_decode_palette(const DevView &v, int out_kind, void *out, void *stream)
{
    const uint64_t groups = (uint64_t)v.N * (uint64_t)v.K / 16;
    if (!groups) return cudaSuccess;
    uint64_t want = (groups + 255) / 256, cap = (uint64_t)num_sms() * 8;
    int blocks = (int)(want < cap ? want : cap);
    cudaStream_t st = (cudaStream_t)stream;
    if (out_kind == DEC_BF16) decode_palette_kernel<DEC_BF16><<<blocks, 256, 0, st>>>(v, out);
    else if (out_kind == DEC_EXP) decode_palette_kernel<DEC_EXP><<<blocks, 256, 0, st>>>(v, out);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------ Huffman decode
template <int OUT>
__global__ void __launch_bounds__(128) decode_huffman_kernel(DevView v, void *out)
{
    extern __shared__ uint8_t dtab[];
    __shared__ uint8_t pal[16];
    const int L = (int)v.max_len;
    {
        const uint4 *src = (const uint4 *)v.dtab;
        uint4 *dst = (uint4 *)dtab;
        for (int i = threadIdx.x; i < (1 << L) / 16; i += blockDim.x) dst[i] = src[i];
        if (threadIdx.x < 16) pal[threadIdx.x] = v.palette[threadIdx.x];
    }
    __syncthreads();
    const uint64_t c = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    if (c >= v.n_chunks) return;
    const uint64_t n = (uint64_t)v.N * (uint64_t)v.K;
    const uint32_t pos0 = v.chunk_off[c], pos1 = v.chunk_off[c + 1];
    const uint64_t b0 = c * (v.chunk / 64);
    const uint64_t b1 = (n / 64 < b0 + v.chunk / 64) ? n / 64 : b0 + v.chunk / 64;

    uint32_t wi = pos0 >> 5;
    const int sh = pos0 & 31;
    uint64_t buf = (((uint64_t)v.bits[wi] << 32) | v.bits[wi + 1]) << sh;
    int avail = 64 - sh;
    wi += 2;
    uint32_t used = 0;
    const uint32_t budget = pos1 - pos0;
    bool bad = false;

    for (uint64_t b = b0; b < b1 && !bad; b++) {
        const uint32_t bw = __ldg(v.bitmap + (b >> 5));
        const bool verb = (bw >> (b & 31)) & 1u;
        const uint8_t *ve = nullptr;
        if (verb) ve = v.verb_exp + (uint64_t)(__ldg(v.prefix + (b >> 5)) + __popc(bw & ((1u << (b & 31)) - 1u))) * 64;
#pragma unroll 1
        for (int q = 0; q < 4; q++) {  // 16 weights per step
            uint32_t sym[16];
            if (verb) {
                if (OUT != DEC_CODES) {
                    uint4 ev = *(const uint4 *)(ve + q * 16);
#pragma unroll
                    for (int i = 0; i < 16; i++) sym[i] = byte_of(ev, i);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; i++) sym[i] = 0;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    if (avail < 32) {
                        buf |= (uint64_t)v.bits[wi++] << (32 - avail);
                        avail += 32;
                    }
                    uint32_t ent = dtab[(uint32_t)(buf >> (64 - L))];
                    uint32_t len = ent & 15u;
                    bad |= (len == 0);
                    len = len ? len : 1;
                    buf <<= len;
                    avail -= (int)len;
                    used += len;
                    sym[i] = OUT == DEC_CODES ? (ent >> 4) : pal[ent >> 4];
                }
            }
            const uint64_t off = b * 64 + q * 16;
            if (OUT == DEC_BF16) {
                uint4 s = *(const uint4 *)(v.sm + off);
                uint32_t h[8];
#pragma unroll
                for (int i = 0; i < 8; i++)
                    h[i] = bf16_of(byte_of(s, 2 * i), sym[2 * i]) | (bf16_of(byte_of(s, 2 * i + 1), sym[2 * i + 1]) << 16);
                uint4 *o = (uint4 *)((uint16_t *)out + off);
                o[0] = make_uint4(h[0], h[1], h[2], h[3]);
                o[1] = make_uint4(h[4], h[5], h[6], h[7]);
            } else if (OUT == DEC_EXP) {
                uint32_t w4[4];
#pragma unroll
                for (int i = 0; i < 4; i++)
                    w4[i] = sym[4 * i] | (sym[4 * i + 1] << 8) | (sym[4 * i + 2] << 16) | (sym[4 * i + 3] << 24);
                *(uint4 *)((uint8_t *)out + off) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            } else {
                uint32_t w2[2] = {0, 0};
#pragma unroll
                for (int i = 0; i < 16; i++) w2[i >> 3] |= sym[i] << (4 * (i & 7));
                *(uint2 *)((uint8_t *)out + off / 2) = make_uint2(w2[0], w2[1]);
            }
        }
        if (used > budget) bad = true;  // overran the chunk: stop before reading further
    }
    if (bad || used != budget) atomicExch(v.status, (int)DEV_CORRUPT);
}

int launch_decode_huffman(const DevView &v, int out_kind, void *out, void *stream)
{
    if (!v.n_chunks) return cudaSuccess;
    const int threads = 128;
    const int blocks = (int)((v.n_chunks + threads - 1) / threads);
    const size_t smem = (size_t)1 << v.max_len;
    cudaStream_t st = (cudaStream_t)stream;
    static bool attr_set = false;  // set once, outside any stream capture (uw_load runs these kernels first)
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_huffman_kernel<DEC_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 32768);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_huffman_kernel<DEC_EXP>, cudaFuncAttributeMaxDynamicSharedMemorySize, 32768);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_huffman_kernel<DEC_CODES>, cudaFuncAttributeMaxDynamicSharedMemorySize, 32768);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    switch (out_kind) {
    case DEC_BF16: decode_huffman_kernel<DEC_BF16><<<blocks, threads, smem, st>>>(v, out); break;
    case DEC_EXP: decode_huffman_kernel<DEC_EXP><<<blocks, threads, smem, st>>>(v, out); break;
    case DEC_CODES: decode_huffman_kernel<DEC_CODES><<<blocks, threads, smem, st>>>(v, out); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace uw
