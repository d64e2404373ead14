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
// Huffman decode: one thread per chunk of C weights, 64-bit bit buffer, a decode
// table in shared memory.  With a length limit of at most 12 a 12-bit
// multi-symbol table gives up to five codes per lookup and each block's four
// groups of 16 codes are decoded one group at a time (a group's lookups run in a
// tight loop, its output leaves in one store); longer limits take one symbol
// per lookup.  A stream that does not end exactly at its chunk's end offset, or
// hits an unassigned prefix, latches DEV_CORRUPT.
#include <cuda_runtime.h>

#include <algorithm>

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
constexpr int kDecThreads = 128;        // chunks per CTA

// 16 codes (a u64 of nibbles) -> 16 exponent bytes through the palette
__device__ __forceinline__ uint4 exps_of_codes(uint64_t codes, const uint8_t *pal)
{
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const uint32_t c = (uint32_t)(codes >> (16 * q));
        w[q] = (uint32_t)pal[c & 15] | ((uint32_t)pal[(c >> 4) & 15] << 8) | ((uint32_t)pal[(c >> 8) & 15] << 16) |
               ((uint32_t)pal[(c >> 12) & 15] << 24);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// 16 weights of bf16 from 16 sign+mantissa bytes and 16 exponent bytes, stored at o[0..1]
__device__ __forceinline__ void store_bf16x16(uint4 *o, const uint4 &s, const uint4 &e)
{
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 8; i++) h[i] = bf16_of(byte_of(s, 2 * i), byte_of(e, 2 * i)) | (bf16_of(byte_of(s, 2 * i + 1), byte_of(e, 2 * i + 1)) << 16);
    o[0] = make_uint4(h[0], h[1], h[2], h[3]);
    o[1] = make_uint4(h[4], h[5], h[6], h[7]);
}

// The non-verbatim blocks of a chunk are decoded as one stream of 64*m symbols (their codes are
// concatenated in the bit string); each full word of 16 codes is routed to its block.  Chunks hold at most
// kMaxChunkBlocks blocks on this path; larger chunks fall back to one stream per block of the same loop.
constexpr int kMaxChunkBlocks = 8;

template <int OUT>
__global__ void __launch_bounds__(kDecThreads) decode_huffman_kernel(DevView v, void *out)
{
    extern __shared__ uint32_t dsm[];
    __shared__ uint16_t pal2[256];  // exponent pair of a code byte: pal[b & 15] | pal[b >> 4] << 8
    const bool multi = v.mtab != nullptr;
    const int L = multi ? 12 : (int)v.max_len;
    uint32_t *mt = dsm;                               // multi-symbol table, or the single-symbol byte table
    if (multi) {
        const uint4 *src = (const uint4 *)v.mtab;
        for (int i = threadIdx.x; i < 1024; i += blockDim.x) ((uint4 *)mt)[i] = src[i];
    } else {
        const uint4 *src = (const uint4 *)v.dtab;
        for (int i = threadIdx.x; i < (1 << L) / 16; i += blockDim.x) ((uint4 *)mt)[i] = src[i];
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        pal2[i] = (uint16_t)(v.palette[i & 15] | (v.palette[i >> 4] << 8));
    __syncthreads();
    // an entry of 0 (these 12 bits start no code) is read as one 1-bit code 0 with bit 31 set: the decode loop
    // needs no test, and the flag is collected and reported after it
    if (multi)
        for (int i = threadIdx.x; i < 4096; i += blockDim.x)
            if (mt[i] == 0u) mt[i] = 0x80000000u | (1u << 7) | (1u << 4) | 1u;
    __syncthreads();
    // a persistent grid (fewer CTAs than groups of kDecThreads chunks, when it is given a share of the SMs) walks
    // the groups with a stride
    for (uint64_t c_first = (uint64_t)blockIdx.x * kDecThreads; c_first < v.n_chunks;
         c_first += (uint64_t)gridDim.x * kDecThreads) {
    const uint64_t c_last = min((uint64_t)v.n_chunks, c_first + kDecThreads);
    if (threadIdx.x == 0) {
        // the CTA's chunks are one contiguous run of the stream: one bulk prefetch into L2, so each thread's
        // first read of a 32-byte sector finds it there instead of in DRAM
        const uint32_t b0 = (__ldg(v.chunk_off + c_first) >> 3) & ~15u;
        const uint32_t b1 = (uint32_t)((((uint64_t)__ldg(v.chunk_off + c_last) + 127u) >> 7) << 4);
        if (b1 > b0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"((const uint8_t *)v.bits + b0), "r"(b1 - b0)
                         : "memory");
    }
    const uint8_t *dt = (const uint8_t *)mt;
    const uint64_t c = c_first + threadIdx.x;
    if (c >= c_last) continue;
    // next 32-bit word of the stream (absolute word number); a corrupt stream that runs past the stream's end and
    // its 512-byte guard reads zeros there, and the chunk's length check reports it
    const uint32_t w_lim = ((v.chunk_off[v.n_chunks] + 31) >> 5) + 120;
    auto word_at = [&](uint32_t wn) -> uint32_t { return wn < w_lim ? v.bits[wn] : 0u; };
    const uint64_t n = (uint64_t)v.N * (uint64_t)v.K;
    const uint32_t pos0 = v.chunk_off[c], pos1 = v.chunk_off[c + 1];
    const uint64_t b0 = c * (v.chunk / 64);
    const uint64_t b1 = (n / 64 < b0 + v.chunk / 64) ? n / 64 : b0 + v.chunk / 64;

    // 64-bit bit buffer, MSB-aligned; `nxt` is the next stream word, loaded one refill ahead so the load's
    // latency hides behind the symbols decoded meanwhile
    uint32_t wi = pos0 >> 5;
    const int sh = pos0 & 31;
    uint64_t buf = (((uint64_t)word_at(wi) << 32) | word_at(wi + 1)) << sh;
    int avail = 64 - sh;
    wi += 2;
    uint32_t nxt = word_at(wi++);
    uint32_t used = 0;
    const uint32_t budget = pos1 - pos0;
    bool bad = false;

    // write verbatim block b (its exponents from the verbatim section; 4-bit codes: zeros)
    auto write_verbatim = [&](uint64_t b, uint32_t bw) {
        const uint4 *ve = (const uint4 *)(v.verb_exp + (uint64_t)(__ldg(v.prefix + (b >> 5)) + __popc(bw & ((1u << (b & 31)) - 1u))) * 64);
        if (OUT == DEC_CODES) {
            uint4 *o = (uint4 *)((uint8_t *)out + b * 32);
            o[0] = make_uint4(0, 0, 0, 0);
            o[1] = make_uint4(0, 0, 0, 0);
        } else if (OUT == DEC_EXP) {
            uint4 *o = (uint4 *)((uint8_t *)out + b * 64);
#pragma unroll
            for (int q = 0; q < 4; q++) o[q] = ve[q];
        } else {
            uint4 *o = (uint4 *)((uint16_t *)out + b * 64);
            const uint4 *sp = (const uint4 *)(v.sm + b * 64);
#pragma unroll
            for (int q = 0; q < 4; q++) store_bf16x16(o + 2 * q, sp[q], ve[q]);
        }
    };

    if (multi) {
        // the chunk's coded blocks take its symbols in order; count them first
        uint32_t nverb = 0;
        for (uint64_t wb = b0 >> 5; wb <= (b1 - 1) >> 5 && b1 > b0; wb++) {
            uint32_t w = __ldg(v.bitmap + wb);
            const uint64_t lo = wb * 32;
            if (b0 > lo) w &= ~0u << (uint32_t)(b0 - lo);
            if (b1 < lo + 32) w &= (1u << (uint32_t)(b1 - lo)) - 1u;
            nverb += __popc(w);
        }
        int remaining = 64 * ((int)(b1 - b0) - (int)nverb);  // codes of the chunk not yet decoded
        uint32_t bad_bits = 0;  // bit 31: a lookup met bits that start no code
        uint64_t cacc = 0;      // decoded codes not yet used, 4 bits each, the first in the low nibble
        uint32_t sh = 0;        // 4 x the number of codes in cacc
        uint32_t bw = 0;
        uint64_t bw_at = ~0ull;
        for (uint64_t b = b0; b < b1; b++) {
            if ((b >> 5) != bw_at) {
                bw_at = b >> 5;
                bw = __ldg(v.bitmap + bw_at);
            }
            if ((bw >> (b & 31)) & 1u) {
                write_verbatim(b, bw);
                continue;
            }
            uint64_t cw[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                uint32_t last_syms = 0, last_sh = 60;
                // one lookup: up to five codes (one when `single`), `len` bits
                auto lookup = [&](bool single) {
                    const uint32_t e = mt[(uint32_t)(buf >> 52)];
                    bad_bits |= e;
                    const uint32_t len = single ? (e >> 7) & 15u : e & 15u;
                    buf <<= len;
                    avail -= (int)len;
                    last_syms = single ? (e >> 11) & 15u : e >> 11;
                    last_sh = sh;
                    cacc |= (uint64_t)last_syms << sh;
                    sh += single ? 4u : (e >> 2) & 28u;
                };
                if (remaining >= 21) {
                    // more codes left than this group can take (16, plus at most 4 carried in or out): every
                    // lookup may decode five; a refill leaves more than 32 bits, enough for two lookups
                    const uint32_t sh0 = sh;
                    while (sh < 64) {
                        if (avail <= 32) {
                            buf |= (uint64_t)nxt << (32 - avail);
                            avail += 32;
                            nxt = word_at(wi++);
                        }
                        lookup(false);
                        if (sh >= 64) break;
                        lookup(false);
                    }
                    remaining -= (int)((sh - sh0) >> 2);
                } else {
                    // the chunk's last coded group: its last four codes one lookup each, so no lookup takes a code
                    // past the chunk's end
                    while (sh < 64) {
                        if (avail <= 32) {
                            buf |= (uint64_t)nxt << (32 - avail);
                            avail += 32;
                            nxt = word_at(wi++);
                        }
                        const uint32_t sh0 = sh;
                        lookup(remaining < 5);
                        remaining -= (int)((sh - sh0) >> 2);
                    }
                }
                cw[q] = cacc;
                // codes of the last lookup beyond the 16th stay for the next group (last_sh >= 44 here)
                cacc = (uint64_t)(last_syms >> (64u - last_sh));
                sh -= 64;
                if (remaining < 0) break;  // a corrupt stream: the end check below reports it
            }
            if (remaining < 0) {
                bad = true;
                break;
            }
            if (OUT == DEC_CODES) {
                uint4 *o = (uint4 *)((uint8_t *)out + b * 32);
                o[0] = make_uint4((uint32_t)cw[0], (uint32_t)(cw[0] >> 32), (uint32_t)cw[1], (uint32_t)(cw[1] >> 32));
                o[1] = make_uint4((uint32_t)cw[2], (uint32_t)(cw[2] >> 32), (uint32_t)cw[3], (uint32_t)(cw[3] >> 32));
            } else {
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    uint32_t e[4];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const uint32_t cb = (uint32_t)(cw[q] >> (16 * i));
                        e[i] = (uint32_t)pal2[cb & 0xFF] | ((uint32_t)pal2[cb >> 8 & 0xFF] << 16);
                    }
                    const uint4 ev = make_uint4(e[0], e[1], e[2], e[3]);
                    if (OUT == DEC_EXP) *(uint4 *)((uint8_t *)out + b * 64 + q * 16) = ev;
                    else {
                        const uint4 sv = *(const uint4 *)(v.sm + b * 64 + q * 16);
                        store_bf16x16((uint4 *)((uint16_t *)out + b * 64 + q * 16), sv, ev);
                    }
                }
            }
        }
        // every code of the chunk was used, no code started on unassigned bits, and the codes ended exactly at the
        // next chunk's offset
        const uint64_t at = 32ull * (wi - 1) - (uint64_t)avail;
        if (bad || (bad_bits >> 31) || sh != 0 || at != (uint64_t)pos1) atomicExch(v.status, (int)DEV_CORRUPT);
        continue;
    }

    // emit 16 codes (one u64 word) of non-verbatim block b, quarter q
    auto emit = [&](uint64_t b, int q, uint64_t cw) {
        if (OUT == DEC_CODES) {
            *(uint64_t *)((uint8_t *)out + b * 32 + q * 8) = cw;
        } else {
            uint32_t e[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const uint32_t cb = (uint32_t)(cw >> (16 * i));
                e[i] = (uint32_t)pal2[cb & 0xFF] | ((uint32_t)pal2[cb >> 8 & 0xFF] << 16);
            }
            const uint4 ev = make_uint4(e[0], e[1], e[2], e[3]);
            if (OUT == DEC_EXP) {
                *(uint4 *)((uint8_t *)out + b * 64 + q * 16) = ev;
            } else {
                const uint4 sv = *(const uint4 *)(v.sm + b * 64 + q * 16);
                store_bf16x16((uint4 *)((uint16_t *)out + b * 64 + q * 16), sv, ev);
            }
        }
    };

    for (uint64_t bs = b0; bs < b1 && !bad; bs += kMaxChunkBlocks) {
        const uint64_t be = min(b1, bs + kMaxChunkBlocks);
        const int nb = (int)(be - bs);
        // verbatim flags of blocks bs .. be - 1 from one 64-bit window of the bitmap
        const uint64_t wlo = __ldg(v.bitmap + (bs >> 5));
        const uint64_t whi = ((bs >> 5) + 1) * 32 < v.n_blocks ? __ldg(v.bitmap + (bs >> 5) + 1) : 0ull;
        const uint32_t vmask = (uint32_t)(((whi << 32) | wlo) >> (bs & 31)) & ((1u << nb) - 1u);
        // verbatim blocks are written here directly
        for (uint32_t m = vmask; m; m &= m - 1) {
            const uint64_t b = bs + (uint64_t)(__ffs(m) - 1);
            write_verbatim(b, __ldg(v.bitmap + (b >> 5)));
        }
        // the non-verbatim blocks of the group take the group's symbols in order, 16 codes per output word
        uint32_t rem = ~vmask & ((1u << nb) - 1u);
        const int total = 64 * __popc(rem);
        int cur = rem ? __ffs(rem) - 1 : 0, q = 0;
        int produced = 0, fill = 0;
        uint64_t acc = 0;
        auto put = [&](uint64_t bits4, int cnt) {  // bits4 holds exactly cnt codes
            acc |= bits4 << (4 * fill);
            fill += cnt;
            if (fill >= 16) {
                emit(bs + (uint64_t)cur, q, acc);
                if (++q == 4) {
                    q = 0;
                    rem &= rem - 1;
                    cur = rem ? __ffs(rem) - 1 : 0;
                }
                fill -= 16;
                acc = fill ? bits4 >> (4 * (cnt - fill)) : 0;
            }
        };
        auto advance = [&](uint32_t len) {
            buf <<= len;
            avail -= (int)len;
            used += len;
            if (avail < 32) {
                buf |= (uint64_t)nxt << (32 - avail);
                avail += 32;
                nxt = word_at(wi++);
            }
        };
        // (limits above 12 bits: one symbol per lookup of the 2^L-entry table)
        while (produced < total) {
            const uint32_t e = dt[(uint32_t)(buf >> (64 - L))];
            uint32_t len = e & 15u;
            const uint32_t sym = e >> 4;
            if (len == 0) { bad = true; len = 1; }
            advance(len);
            put(sym, 1);
            produced++;
        }
        if (used > budget) bad = true;  // overran the chunk: stop before reading further
    }
    if (bad || used != budget) atomicExch(v.status, (int)DEV_CORRUPT);
    }
}

int launch_decode_huffman(const DevView &v, int out_kind, void *out, void *stream, int max_ctas)
{
    if (!v.n_chunks) return cudaSuccess;
    const int threads = kDecThreads;
    int blocks = (int)((v.n_chunks + threads - 1) / threads);
    if (max_ctas > 0) blocks = std::min(blocks, max_ctas);
    const size_t tab_bytes = v.mtab ? 16384 : std::max<size_t>(16384, (size_t)1 << v.max_len);
    const size_t smem = tab_bytes;  // decode table
    cudaStream_t st = (cudaStream_t)stream;
    static bool attr_set = false;  // set once, outside any stream capture (uw_load runs these kernels first)
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_huffman_kernel<DEC_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_huffman_kernel<DEC_EXP>, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_huffman_kernel<DEC_CODES>, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536);
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
