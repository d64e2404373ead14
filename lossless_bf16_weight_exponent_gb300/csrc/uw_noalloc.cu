// uw_noalloc.cu - the palette-transcode matmul with its scratch in a static device array.
//
// Some callers cannot call cudaMalloc: an inference engine whose allocator has
// reserved all of the device's memory at start-up (every later cudaMalloc fails
// or fragments its pool), or code on a latency-critical path that must not take
// the device-wide synchronisation cudaMalloc / cudaFree may imply.  For them,
// uw_matmul_noalloc runs the same kernels as uw_matmul with the palette-transcode
// pipeline, but its scratch (the transcoded 4-bit codes and, when the K-split
// needs one, the fp32 accumulator) lives in the array below, which the driver
// places on every device that loads this library and keeps there until the
// process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "uw_internal.h"

// Library-owned scratch: UW_NOALLOC_SCRATCH_BYTES (36 MiB) per device.
#define UW_NOALLOC_SCRATCH_BYTES (36u * 1024u * 1024u)
static __device__ __align__(256) uint8_t g_noalloc_scratch[UW_NOALLOC_SCRATCH_BYTES];

namespace {

// The array's device address belongs to the CUDA context that loaded this module: the device's primary context,
// or a context a driver-API caller created.  After cudaDeviceReset the primary context is a new one, and the
// module (with the array) is loaded again, possibly elsewhere.  So the address is looked up once per context and
// cached under the context's unique id (cuCtxGetId: never reused within the process).
struct ScratchEntry {
    unsigned long long ctx_id;
    void *ptr;
};
std::mutex g_mu;
std::vector<ScratchEntry> g_cache;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// The current context's unique id; false if there is no current context or the driver lacks cuCtxGetId.
bool current_context_id(unsigned long long *id)
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = (CtxGetCurrentFn)p;
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = (CtxGetIdFn)p;
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context.  In host code the array's name is only a host-side
// stand-in, so the address comes from cudaGetSymbolAddress, with the context current; it is cached per context.
// Without cuCtxGetId (a driver older than CUDA 12) every call looks it up again.
uw_status scratch_address(void **out)
{
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> g(g_mu);
    if (have_id)
        for (const ScratchEntry &e : g_cache)
            if (e.ctx_id == id) { *out = e.ptr; return UW_OK; }
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
        return uw::fail(UW_ERR_CUDA, "uw_matmul_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    // the lookup above made the device's primary context current if no context was: take its id now
    if (!have_id) have_id = current_context_id(&id);
    if (have_id) g_cache.push_back(ScratchEntry{id, p});
    *out = p;
    return UW_OK;
}

uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

}  // namespace

extern "C" uw_status uw_matmul_noalloc(const uw_matrix *m, const uint16_t *x_dev, int64_t B, void *y_dev,
                                       uw_out_dtype out_dtype, uw_stream stream)
{
    uw::clear_error();
    if (!m) return uw::fail(UW_ERR_INVALID_ARG, "uw_matmul_noalloc: NULL matrix");
    uw_info info;
    uw_status s = uw_get_info(m, &info);
    if (s != UW_OK) return s;
    if (info.codec != UW_CODEC_HUFFMAN || !info.has_huffman_stream)
        return uw::fail(UW_ERR_UNSUPPORTED,
                        "uw_matmul_noalloc: needs a Huffman-coded matrix with its stream resident (palette transcode)");
    if (B < 0) return uw::fail(UW_ERR_SHAPE, "uw_matmul_noalloc: B < 0");
    if (B == 0 || info.N == 0) return UW_OK;
    if (!x_dev || !y_dev || ((uintptr_t)x_dev & 15) || ((uintptr_t)y_dev & 15))
        return uw::fail(UW_ERR_INVALID_ARG, "uw_matmul_noalloc: X/Y NULL or not 16-byte aligned");
    if (out_dtype != UW_OUT_F32 && out_dtype != UW_OUT_BF16)
        return uw::fail(UW_ERR_INVALID_ARG, "uw_matmul_noalloc: bad output dtype");
    const uint64_t n = (uint64_t)info.N * (uint64_t)info.K;
    const uint64_t codes_bytes = round_up(n / 2 + 64, 256);
    const uint64_t acc_bytes = uw::acc_region_bytes(B, info.N) + uw::tile_cells_bytes(info.N);
    if (codes_bytes + acc_bytes > UW_NOALLOC_SCRATCH_BYTES)
        return uw::fail(UW_ERR_WORKSPACE,
                        "uw_matmul_noalloc: needs %llu scratch bytes (4-bit codes %llu + accumulator %llu), "
                        "the static scratch holds %u",
                        (unsigned long long)(codes_bytes + acc_bytes), (unsigned long long)codes_bytes,
                        (unsigned long long)acc_bytes, UW_NOALLOC_SCRATCH_BYTES);
    void *scratch = nullptr;
    s = scratch_address(&scratch);
    if (s != UW_OK) return s;
    // Same plan as uw_matmul with UW_STRAT_PALETTE_TRANSCODE on the GEMV kernel, workspace = the static array.
    uw_plan plan{};
    plan.strategy = UW_STRAT_PALETTE_TRANSCODE;
    plan.kernel = UW_KERNEL_GEMV;
    return uw_matmul_plan(m, x_dev, B, y_dev, out_dtype, &plan, scratch, UW_NOALLOC_SCRATCH_BYTES, stream);
}
