// uw_runtime.cu - device residency, strategy dispatch and autotuning behind the C ABI.
//
// Cloudflare blog "Unweight": section on the four execution pipelines (full
// decode, exponent-only, palette transcode, direct palette) and the autotuning
// section (measure real throughput on the target GPU, vary one choice at a time
// until nothing improves, keep a per-matrix, per-batch-size table of pipeline,
// matmul variant and split).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <sstream>
#include <string>
#include <vector>

#include "uw_internal.h"

using namespace uw;

namespace {

uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

int64_t bucket_of(int64_t B)
{
    int64_t b = 1;
    while (b < B) b <<= 1;
    return b;
}

}  // namespace

namespace uw {

int device_sms()
{
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

static thread_local int t_sm_budget = 0;

int num_sms()
{
    const int n = device_sms();
    return t_sm_budget > 0 ? std::min(t_sm_budget, n) : n;
}

SmBudget::SmBudget(int n) : prev(t_sm_budget) { t_sm_budget = n; }
SmBudget::~SmBudget() { t_sm_budget = prev; }

}  // namespace uw

static uw_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(UW_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define UW_CUDA(call, what)                                        \
    do {                                                           \
        cudaError_t e_ = (cudaError_t)(call);                      \
        if (e_ != cudaSuccess) return cuda_fail(e_, what);         \
    } while (0)

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// ------------------------------------------------------------------------------ load / free
extern "C" uw_status uw_load(const void *blob, size_t size, int resident, uw_stream stream, uw_matrix **out)
{
    clear_error();
    if (!out) return fail(UW_ERR_INVALID_ARG, "uw_load: out is NULL");
    *out = nullptr;
    if (resident < UW_RESIDENT_HUFFMAN || resident > UW_RESIDENT_PALETTE)
        return fail(UW_ERR_INVALID_ARG, "uw_load: resident %d out of range", resident);
    BlobHeader h;
    uw_status s = parse_and_validate((const uint8_t *)blob, size, &h, true);
    if (s != UW_OK) return s;
    const uint8_t *p = (const uint8_t *)blob;
    const uint64_t n = (uint64_t)h.N * (uint64_t)h.K;
    const bool huff = h.codec == UW_CODEC_HUFFMAN;
    // what stays resident: the 4-bit codes (a palette blob always; a Huffman blob unless only its stream is
    // wanted) and the Huffman stream with its offsets and tables (a Huffman blob unless only the codes are)
    const bool resident_codes = !huff || resident != UW_RESIDENT_HUFFMAN;
    const bool resident_stream = huff && resident != UW_RESIDENT_PALETTE;
    const bool multi = huff && h.max_len <= 12;
    const uint64_t tab_bytes = huff ? ((uint64_t)1 << h.max_len) : 16;

    // device layout: every piece 256-aligned, streams padded so vector loads may run past the end
    uint64_t off = 0;
    auto take = [&](uint64_t bytes) { uint64_t o = off; off = round_up(off + bytes, 256); return o; };
    const uint64_t o_sm = take(n + 64);
    const uint64_t o_bm = take(h.len[S_BITMAP] + 16);
    const uint64_t o_pf = take(h.len[S_PREFIX] + 16);
    const uint64_t o_ve = take(h.len[S_VERB] + 16);
    const uint64_t o_codes = resident_codes ? take(n / 2 + 64) : 0;
    // the Huffman stream: in the matrix's own memory when it stays resident, else in a load-time buffer that
    // only feeds the transcode into the codes
    uint64_t hoff = 0;
    auto take_h = [&](uint64_t bytes) {
        if (resident_stream) return take(bytes);
        uint64_t o = hoff; hoff = round_up(hoff + bytes, 256); return o;
    };
    const uint64_t o_co = huff ? take_h(h.len[S_CHUNK] + 16) : 0;
    const uint64_t o_bits = huff ? take_h(h.len[S_BITS] + 512) : 0;
    const uint64_t o_tab = huff ? take_h(tab_bytes) : 0;
    const uint64_t o_mtab = multi ? take_h(4096 * 4) : 0;
    const uint64_t o_st = take(256);
    // tile-major verbatim stream for the unit-walking kernels (units of 128 rows x 256 weights)
    std::vector<uint32_t> tmv_off, tmv_mask;
    std::vector<uint8_t> tmv_data;
    const bool tmv = h.K % 256 == 0 && h.N > 0;
    if (tmv) build_tile_verbatim(h, p, tmv_off, tmv_mask, tmv_data);
    const uint64_t o_tmo = tmv ? take(tmv_off.size() * 4 + 16) : 0;
    const uint64_t o_tmm = tmv ? take(tmv_mask.size() * 4 + 16) : 0;
    const uint64_t o_tmd = tmv ? take(tmv_data.size() + 64) : 0;

    uw_matrix *m = new (std::nothrow) uw_matrix();
    if (!m) return fail(UW_ERR_NO_MEMORY, "uw_load: host allocation");
    m->h = h;
    cudaGetDevice(&m->device);
    cudaError_t e = cudaMalloc(&m->dev, off);
    if (e != cudaSuccess) { delete m; return fail(UW_ERR_NO_MEMORY, "uw_load: cudaMalloc(%llu): %s", (unsigned long long)off, cudaGetErrorString(e)); }
    m->dev_bytes = off;
    uint8_t *d = (uint8_t *)m->dev;
    uint8_t *hd = d;  // base of the Huffman pieces
    if (huff && !resident_stream) {
        if ((e = cudaMalloc(&hd, hoff)) != cudaSuccess) {
            cudaFree(m->dev); delete m;
            return fail(UW_ERR_NO_MEMORY, "uw_load: cudaMalloc(%llu): %s", (unsigned long long)hoff, cudaGetErrorString(e));
        }
    }
    cudaStream_t st = (cudaStream_t)stream;
    auto fail_free = [&](uw_status code) {
        if (hd != d) cudaFree(hd);
        cudaFree(m->dev); delete m; return code;
    };
    if ((e = cudaMemsetAsync(d, 0, off, st)) != cudaSuccess) return fail_free(cuda_fail(e, "uw_load: memset"));
    if (hd != d && (e = cudaMemsetAsync(hd, 0, hoff, st)) != cudaSuccess) return fail_free(cuda_fail(e, "uw_load: memset"));
    auto up = [&](uint8_t *base, uint64_t dst, int sec) -> cudaError_t {
        if (!h.len[sec]) return cudaSuccess;
        return cudaMemcpyAsync(base + dst, p + h.off[sec], h.len[sec], cudaMemcpyHostToDevice, st);
    };
    if ((e = up(d, o_sm, S_SM)) || (e = up(d, o_bm, S_BITMAP)) || (e = up(d, o_pf, S_PREFIX)) || (e = up(d, o_ve, S_VERB)) ||
        (!huff && (e = up(d, o_codes, S_IDX))) || (huff && ((e = up(hd, o_co, S_CHUNK)) || (e = up(hd, o_bits, S_BITS)))))
        return fail_free(cuda_fail(e, "uw_load: upload"));
    if (tmv && ((e = cudaMemcpyAsync(d + o_tmo, tmv_off.data(), tmv_off.size() * 4, cudaMemcpyHostToDevice, st)) ||
                (e = cudaMemcpyAsync(d + o_tmm, tmv_mask.data(), tmv_mask.size() * 4, cudaMemcpyHostToDevice, st)) ||
                (!tmv_data.empty() &&
                 (e = cudaMemcpyAsync(d + o_tmd, tmv_data.data(), tmv_data.size(), cudaMemcpyHostToDevice, st)))))
        return fail_free(cuda_fail(e, "uw_load: verbatim stream upload"));
    std::vector<uint8_t> table;
    std::vector<uint32_t> mtable;
    if (huff) {
        build_decode_table(h.code_len, (int)h.max_len, table);
        if ((e = cudaMemcpyAsync(hd + o_tab, table.data(), table.size(), cudaMemcpyHostToDevice, st)))
            return fail_free(cuda_fail(e, "uw_load: table upload"));
        if (multi) {
            build_multi_table(h.code_len, mtable);
            if ((e = cudaMemcpyAsync(hd + o_mtab, mtable.data(), mtable.size() * 4, cudaMemcpyHostToDevice, st)))
                return fail_free(cuda_fail(e, "uw_load: table upload"));
        }
    }
    DevView &v = m->v;
    memset(&v, 0, sizeof v);
    v.N = h.N; v.K = h.K; v.n_blocks = h.n_blocks; v.n_chunks = h.n_chunks;
    v.chunk = h.chunk; v.max_len = h.max_len; v.n_pal = h.n_pal;
    memcpy(v.palette, h.palette, 16);
    v.sm = d + o_sm;
    v.bitmap = (const uint32_t *)(d + o_bm);
    v.prefix = (const uint32_t *)(d + o_pf);
    v.verb_exp = d + o_ve;
    m->codes = resident_codes ? d + o_codes : nullptr;
    v.codes = m->codes;
    if (huff) {
        v.chunk_off = (const uint32_t *)(hd + o_co);
        v.bits = (const uint32_t *)(hd + o_bits);
        v.dtab = hd + o_tab;
        v.mtab = multi ? (const uint32_t *)(hd + o_mtab) : nullptr;
    }
    v.status = (int *)(d + o_st);
    m->tmv_off = tmv ? (const uint32_t *)(d + o_tmo) : nullptr;
    m->tmv_mask = tmv ? (const uint32_t *)(d + o_tmm) : nullptr;
    m->tmv_data = tmv ? d + o_tmd : nullptr;
    m->has_stream = resident_stream;
    if (huff && resident_codes) {
        // the post's load-time transcode of the Huffman stream into the direct-palette form
        if ((e = (cudaError_t)launch_decode_huffman(v, DEC_CODES, m->codes, st)))
            return fail_free(cuda_fail(e, "uw_load: palette transcode"));
    }
    if ((e = cudaStreamSynchronize(st))) return fail_free(cuda_fail(e, "uw_load: synchronize"));
    int dev_status = 0;
    if ((e = cudaMemcpy(&dev_status, v.status, sizeof(int), cudaMemcpyDeviceToHost)))
        return fail_free(cuda_fail(e, "uw_load: status read"));
    if (dev_status) return fail_free(fail(UW_ERR_CORRUPT, "uw_load: Huffman stream failed to decode"));
    if (hd != d) {
        // only the codes stay: the stream, its offsets and tables are gone
        cudaFree(hd);
        v.chunk_off = nullptr;
        v.bits = nullptr;
        v.dtab = nullptr;
        v.mtab = nullptr;
    }
    *out = m;
    return UW_OK;
}

extern "C" void uw_free(uw_matrix *m)
{
    if (!m) return;
    // no device-wide synchronisation of its own: cudaFree already waits for work still using the allocation
    cudaFree(m->dev);
    delete m;
}

extern "C" uw_status uw_get_info(const uw_matrix *m, uw_info *out)
{
    clear_error();
    if (!m || !out) return fail(UW_ERR_INVALID_ARG, "uw_get_info: NULL argument");
    const BlobHeader &h = m->h;
    memset(out, 0, sizeof *out);
    out->N = h.N; out->K = h.K; out->codec = h.codec; out->n_pal = h.n_pal;
    memcpy(out->palette, h.palette, 16);
    memcpy(out->code_len, h.code_len, 16);
    out->n_blocks = h.n_blocks; out->n_verbatim = h.n_verbatim; out->n_chunks = h.n_chunks;
    out->total_bits = h.total_bits; out->blob_bytes = h.blob_bytes;
    out->device_bytes = m->dev_bytes;
    out->has_palette_form = m->codes != nullptr;
    out->has_huffman_stream = m->has_stream;
    out->chunk_weights = (int32_t)h.chunk; out->max_code_len = (int32_t)h.max_len;
    return UW_OK;
}

extern "C" uw_status uw_check(const uw_matrix *m, uw_stream stream)
{
    clear_error();
    if (!m) return fail(UW_ERR_INVALID_ARG, "uw_check: NULL matrix");
    UW_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "uw_check: synchronize");
    int s = 0;
    UW_CUDA(cudaMemcpy(&s, m->v.status, sizeof s, cudaMemcpyDeviceToHost), "uw_check: status read");
    if (s) {
        UW_CUDA(cudaMemset(m->v.status, 0, sizeof s), "uw_check: status clear");
        if (s == DEV_TIMEOUT) return fail(UW_ERR_TIMEOUT, "a bounded device wait expired");
        return fail(UW_ERR_CORRUPT, "a device decoder found a corrupt stream");
    }
    return UW_OK;
}

// ------------------------------------------------------------------------------ decode
extern "C" uw_status uw_decode(const uw_matrix *m, uint16_t *w_dev, uw_stream stream)
{
    clear_error();
    if (!m) return fail(UW_ERR_INVALID_ARG, "uw_decode: NULL matrix");
    const uint64_t n = (uint64_t)m->h.N * (uint64_t)m->h.K;
    if (!n) return UW_OK;
    if (!w_dev || !aligned16(w_dev)) return fail(UW_ERR_INVALID_ARG, "uw_decode: output NULL or not 16-byte aligned");
    int e;
    // from the resident codes when there are any (a streaming decode), else from the Huffman stream
    if (m->codes) e = launch_decode_palette(m->v, DEC_BF16, w_dev, stream);
    else e = launch_decode_huffman(m->v, DEC_BF16, w_dev, stream);
    if (e) return cuda_fail((cudaError_t)e, "uw_decode: launch");
    return UW_OK;
}

// ------------------------------------------------------------------------------ plans
static bool strategy_ok(const uw_matrix *m, int s)
{
    switch (s) {
    case UW_STRAT_FULL_DECODE:
    case UW_STRAT_EXP_ONLY: return true;
    case UW_STRAT_PALETTE_TRANSCODE: return m->has_stream;
    case UW_STRAT_DIRECT_PALETTE: return m->codes != nullptr;
    case UW_STRAT_HUFFMAN_DIRECT: return m->has_stream && gemv_huff_supported(m->v, 1);
    default: return false;
    }
}

static int fmt_of(int strategy)
{
    return strategy == UW_STRAT_FULL_DECODE ? FMT_BF16 : strategy == UW_STRAT_EXP_ONLY ? FMT_EXP : FMT_PAL;
}

static uint64_t preprocess_bytes(const uw_matrix *m, int strategy)
{
    const uint64_t n = (uint64_t)m->h.N * (uint64_t)m->h.K;
    switch (strategy) {
    case UW_STRAT_FULL_DECODE: return round_up(2 * n + 64, 256);
    case UW_STRAT_EXP_ONLY: return round_up(n + 64, 256);
    case UW_STRAT_PALETTE_TRANSCODE: return round_up(n / 2 + 64, 256);
    default: return 0;
    }
}

static WOperand operand_shape(const uw_matrix *m, int strategy)
{
    WOperand w;
    memset(&w, 0, sizeof w);
    w.fmt = fmt_of(strategy);
    w.N = m->h.N;
    w.K = m->h.K;
    memcpy(w.palette, m->h.palette, 16);
    w.sm = m->v.sm;
    w.bitmap = m->v.bitmap;
    w.prefix = m->v.prefix;
    w.verb_exp = m->v.verb_exp;
    w.tmv_off = m->tmv_off;
    w.tmv_mask = m->tmv_mask;
    w.tmv_data = m->tmv_data;
    w.codes = m->codes;
    w.status = m->v.status;
    return w;
}

static int resolve_kernel(const uw_matrix *m, const uw_plan &p, int64_t B)
{
    if (p.kernel != UW_KERNEL_AUTO) return p.kernel;
    WOperand w = operand_shape(m, p.strategy);
    if (B > 2 && tc_supported(w, B, p.variant)) return UW_KERNEL_TC;
    return UW_KERNEL_GEMV;
}

static uint64_t split_bytes(const uw_matrix *m, int64_t B, const uw_plan &p, int kernel)
{
    WOperand w = operand_shape(m, p.strategy);
    int split = p.split_k > 0 ? p.split_k
                              : (kernel == UW_KERNEL_TC ? tc_default_split(w, B, p.variant) : gemv_default_split(w, B));
    // the GEMV may raise the split to fit its X slice; reserve the accumulator whenever a split is possible, and
    // the row-tile cells of the tensor-core kernel
    (void)split;
    return acc_region_bytes(B, m->h.N) + tile_cells_bytes(m->h.N);
}

// the kernel and launch shape for a strategy and batch when no tuned plan exists
static uw_plan default_plan_for_strategy(const uw_matrix *m, int64_t B, int strategy)
{
    uw_plan p{};
    p.strategy = strategy;
    p.kernel = UW_KERNEL_AUTO;
    if (strategy == UW_STRAT_HUFFMAN_DIRECT) {
        // one kernel: the GEMV that decodes the Huffman stream itself
        p.kernel = UW_KERNEL_GEMV;
        return p;
    }
    const WOperand w = operand_shape(m, p.strategy);
    if (B >= 2 && B <= 64 && gemv_rp_supported(w, B)) {
        // a few batch rows: the row-parallel tensor-pipe GEMV streams the weights once for all of them
        p.kernel = UW_KERNEL_GEMV;
        p.variant = 8;
        return p;
    }
    if (B > 64 && tc4_supported(w, B)) {
        // a dense contraction: the persistent tcgen05 kernel
        p.kernel = UW_KERNEL_TC;
        p.variant = 4;
        return p;
    }
    if (B > 2 && B <= 16 && gemv_mma_supported(w, B, 6)) {
        // a few batch rows: the tensor-pipe GEMV streams the weights once for all of them
        p.kernel = UW_KERNEL_GEMV;
        p.variant = 6;
        return p;
    }
    p.kernel = resolve_kernel(m, p, B);
    if (p.kernel == UW_KERNEL_GEMV && gemv_tma_supported(w, B, 4)) p.variant = 4;
    return p;
}

static uw_plan default_plan(const uw_matrix *m, int64_t B)
{
    if (m->codes) return default_plan_for_strategy(m, B, UW_STRAT_DIRECT_PALETTE);
    // a Huffman matrix without its palette form: decode in the GEMV where it applies, else transcode first
    if (m->has_stream && gemv_huff_supported(m->v, B))
        return default_plan_for_strategy(m, B, UW_STRAT_HUFFMAN_DIRECT);
    return default_plan_for_strategy(m, B, UW_STRAT_PALETTE_TRANSCODE);
}

extern "C" uw_status uw_plan_for(const uw_matrix *m, int64_t B, uw_plan *out)
{
    clear_error();
    if (!m || !out) return fail(UW_ERR_INVALID_ARG, "uw_plan_for: NULL argument");
    const int64_t bk = bucket_of(std::max<int64_t>(B, 1));
    {
        std::lock_guard<std::mutex> g(const_cast<uw_matrix *>(m)->mu);
        for (const TuneEntry &t : m->tune)
            if (t.bucket == bk) { *out = t.plan; return UW_OK; }
    }
    *out = default_plan(m, B);
    return UW_OK;
}

static uw_status check_plan(const uw_matrix *m, int64_t B, const uw_plan &p, int *kernel)
{
    if (p.strategy < UW_STRAT_FULL_DECODE || p.strategy > UW_STRAT_HUFFMAN_DIRECT)
        return fail(UW_ERR_INVALID_ARG, "plan strategy %d out of range", p.strategy);
    if (!strategy_ok(m, p.strategy))
        return fail(UW_ERR_UNSUPPORTED, "strategy %d not available for this matrix (codec %u, palette form %d)", p.strategy,
                    m->h.codec, m->codes != nullptr);
    if (p.split_k < 0 || p.variant < 0) return fail(UW_ERR_INVALID_ARG, "negative split or variant");
    if (p.strategy == UW_STRAT_HUFFMAN_DIRECT) {
        if (p.kernel != UW_KERNEL_AUTO && p.kernel != UW_KERNEL_GEMV)
            return fail(UW_ERR_UNSUPPORTED, "the Huffman-direct strategy runs on the GEMV kernel only");
        if (p.split_k > 1 || p.variant > 1)
            return fail(UW_ERR_UNSUPPORTED, "the Huffman-direct GEMV has no K-split and launch variants 0 and 1 only");
        if (!gemv_huff_supported(m->v, B, p.variant))
            return fail(UW_ERR_UNSUPPORTED, "the Huffman-direct GEMV takes 1 <= B <= 8 (B=%lld)", (long long)B);
        *kernel = UW_KERNEL_GEMV;
        return UW_OK;
    }
    int k = resolve_kernel(m, p, B);
    if (k == UW_KERNEL_TC && !tc_supported(operand_shape(m, p.strategy), B, p.variant))
        return fail(UW_ERR_UNSUPPORTED, "tensor-core kernel not available for B=%lld variant %d", (long long)B, p.variant);
    if (k != UW_KERNEL_GEMV && k != UW_KERNEL_TC) return fail(UW_ERR_INVALID_ARG, "kernel %d out of range", p.kernel);
    *kernel = k;
    return UW_OK;
}

extern "C" uw_status uw_plan_workspace_size(const uw_matrix *m, int64_t B, const uw_plan *plan, size_t *bytes)
{
    clear_error();
    if (!m || !plan || !bytes) return fail(UW_ERR_INVALID_ARG, "uw_plan_workspace_size: NULL argument");
    int kernel;
    uw_status s = check_plan(m, std::max<int64_t>(B, 1), *plan, &kernel);
    if (s != UW_OK) return s;
    *bytes = preprocess_bytes(m, plan->strategy) + split_bytes(m, std::max<int64_t>(B, 1), *plan, kernel);
    return UW_OK;
}

extern "C" uw_status uw_workspace_size(const uw_matrix *m, int64_t B, uw_strategy strategy, size_t *bytes)
{
    clear_error();
    if (!m || !bytes) return fail(UW_ERR_INVALID_ARG, "uw_workspace_size: NULL argument");
    if (strategy != UW_STRAT_AUTO && (strategy < UW_STRAT_FULL_DECODE || strategy > UW_STRAT_HUFFMAN_DIRECT))
        return fail(UW_ERR_INVALID_ARG, "uw_workspace_size: strategy %d out of range", (int)strategy);
    if (strategy != UW_STRAT_AUTO && !strategy_ok(m, strategy))
        return fail(UW_ERR_UNSUPPORTED, "strategy %d not available for this matrix", (int)strategy);
    uw_plan p;
    if (strategy == UW_STRAT_AUTO) uw_plan_for(m, B, &p);
    else p = default_plan_for_strategy(m, std::max<int64_t>(B, 1), strategy);
    return uw_plan_workspace_size(m, B, &p, bytes);
}

extern "C" uw_status uw_matmul_plan(const uw_matrix *m, const uint16_t *x, int64_t B, void *y, uw_out_dtype od,
                                    const uw_plan *plan, void *ws, size_t ws_bytes, uw_stream stream)
{
    clear_error();
    if (!m || !plan) return fail(UW_ERR_INVALID_ARG, "uw_matmul: NULL matrix or plan");
    if (B < 0) return fail(UW_ERR_SHAPE, "uw_matmul: B < 0");
    if (B == 0 || m->h.N == 0) return UW_OK;
    if (!x || !y || !aligned16(x) || !aligned16(y) || (ws && !aligned16(ws)))
        return fail(UW_ERR_INVALID_ARG, "uw_matmul: X/Y/workspace NULL or not 16-byte aligned");
    if (od != UW_OUT_F32 && od != UW_OUT_BF16) return fail(UW_ERR_INVALID_ARG, "uw_matmul: bad output dtype");
    int kernel;
    uw_status s = check_plan(m, B, *plan, &kernel);
    if (s != UW_OK) return s;
    const uint64_t pre = preprocess_bytes(m, plan->strategy);
    const uint64_t need = pre + split_bytes(m, B, *plan, kernel);
    if (ws_bytes < need || (need && !ws))
        return fail(UW_ERR_WORKSPACE, "uw_matmul: workspace %zu bytes, need %llu", ws_bytes, (unsigned long long)need);
    uint8_t *wsp = (uint8_t *)ws;
    WOperand w = operand_shape(m, plan->strategy);
    int e = 0;
    switch (plan->strategy) {
    case UW_STRAT_FULL_DECODE:
        e = m->codes ? launch_decode_palette(m->v, DEC_BF16, wsp, stream) : launch_decode_huffman(m->v, DEC_BF16, wsp, stream);
        w.w = (const uint16_t *)wsp;
        w.w_from_prev = 1;
        break;
    case UW_STRAT_EXP_ONLY:
        e = m->codes ? launch_decode_palette(m->v, DEC_EXP, wsp, stream) : launch_decode_huffman(m->v, DEC_EXP, wsp, stream);
        w.exps = wsp;
        w.w_from_prev = 1;
        break;
    case UW_STRAT_PALETTE_TRANSCODE:
        e = launch_decode_huffman(m->v, DEC_CODES, wsp, stream);
        w.codes = wsp;
        w.w_from_prev = 1;
        break;
    default: break;
    }
    if (e) return cuda_fail((cudaError_t)e, "uw_matmul: preprocess launch");
    float *acc = (float *)(wsp + pre);
    if (plan->strategy == UW_STRAT_HUFFMAN_DIRECT) {
        e = launch_gemv_huff(m->v, x, B, y, od == UW_OUT_BF16, plan->variant, acc, stream);
        if (e) return cuda_fail((cudaError_t)e, "uw_matmul: Huffman-direct GEMV launch");
        return UW_OK;
    }
    if (kernel == UW_KERNEL_TC) e = launch_tc(w, x, B, y, od == UW_OUT_BF16, plan->split_k, plan->variant, acc, stream);
    else e = launch_gemv(w, x, B, y, od == UW_OUT_BF16, plan->split_k, plan->variant, acc, stream);
    if (e) return cuda_fail((cudaError_t)e, "uw_matmul: matmul launch");
    return UW_OK;
}

namespace uw {

uint64_t next_launch_epoch()
{
    static std::atomic<uint64_t> launches{0};
    uint64_t e;
    do e = (launches.fetch_add(1) + 1) & ((1ull << 40) - 1);
    while (!e);
    return e;
}

size_t matmul_with_codes_workspace(const uw_matrix *m, int64_t B)
{
    const uw_plan p = default_plan_for_strategy(m, std::max<int64_t>(B, 1), UW_STRAT_PALETTE_TRANSCODE);
    int kernel;
    if (check_plan(m, std::max<int64_t>(B, 1), p, &kernel) != UW_OK) return 0;
    return split_bytes(m, std::max<int64_t>(B, 1), p, kernel);
}

uw_status matmul_with_codes(const uw_matrix *m, const uint8_t *codes, const uint16_t *x, int64_t B, void *y,
                            uw_out_dtype od, void *ws, size_t ws_bytes, void *stream)
{
    if (B == 0 || m->h.N == 0) return UW_OK;
    const uw_plan p = default_plan_for_strategy(m, B, UW_STRAT_PALETTE_TRANSCODE);
    int kernel;
    uw_status s = check_plan(m, B, p, &kernel);
    if (s != UW_OK) return s;
    const uint64_t need = split_bytes(m, B, p, kernel);
    if (ws_bytes < need || (need && !ws))
        return fail(UW_ERR_WORKSPACE, "matmul workspace %zu bytes, need %llu", ws_bytes, (unsigned long long)need);
    WOperand w = operand_shape(m, UW_STRAT_PALETTE_TRANSCODE);
    w.codes = codes;
    w.w_from_prev = 0;  // written by a launch the caller ordered before this one (another stream's kernel)
    float *acc = (float *)ws;
    const int e = kernel == UW_KERNEL_TC ? launch_tc(w, x, B, y, od == UW_OUT_BF16, p.split_k, p.variant, acc, stream)
                                         : launch_gemv(w, x, B, y, od == UW_OUT_BF16, p.split_k, p.variant, acc, stream);
    if (e) return cuda_fail((cudaError_t)e, "matmul launch");
    return UW_OK;
}

}  // namespace uw

extern "C" uw_status uw_matmul(const uw_matrix *m, const uint16_t *x, int64_t B, void *y, uw_out_dtype od,
                               uw_strategy strategy, void *ws, size_t ws_bytes, uw_stream stream)
{
    clear_error();
    if (!m) return fail(UW_ERR_INVALID_ARG, "uw_matmul: NULL matrix");
    if (strategy != UW_STRAT_AUTO && (strategy < UW_STRAT_FULL_DECODE || strategy > UW_STRAT_HUFFMAN_DIRECT))
        return fail(UW_ERR_INVALID_ARG, "uw_matmul: strategy %d out of range", (int)strategy);
    if (strategy != UW_STRAT_AUTO && !strategy_ok(m, strategy))
        return fail(UW_ERR_UNSUPPORTED, "strategy %d not available for this matrix (codec %u, palette form %d)",
                    (int)strategy, m->h.codec, m->codes != nullptr);
    uw_plan p;
    if (strategy == UW_STRAT_AUTO) uw_plan_for(m, B, &p);
    else p = default_plan_for_strategy(m, std::max<int64_t>(B, 1), strategy);
    return uw_matmul_plan(m, x, B, y, od, &p, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------------------ host end-to-end
extern "C" uw_status uw_host_workspace_size(const uw_matrix *m, int64_t B, uw_out_dtype od, size_t *bytes)
{
    clear_error();
    if (!m || !bytes) return fail(UW_ERR_INVALID_ARG, "uw_host_workspace_size: NULL argument");
    size_t w = 0;
    uw_status s = uw_workspace_size(m, B, UW_STRAT_AUTO, &w);
    if (s != UW_OK) return s;
    *bytes = round_up(w, 256) + round_up((uint64_t)B * m->h.K * 2, 256) +
             round_up((uint64_t)B * m->h.N * (od == UW_OUT_BF16 ? 2 : 4), 256);
    return UW_OK;
}

extern "C" uw_status uw_matmul_host_async(const uw_matrix *m, const uint16_t *x_host, int64_t B, void *y_host,
                                          uw_out_dtype od, void *ws, size_t ws_bytes, uw_stream stream)
{
    clear_error();
    if (!m) return fail(UW_ERR_INVALID_ARG, "uw_matmul_host: NULL matrix");
    if (B == 0 || m->h.N == 0) return UW_OK;
    if (!x_host || !y_host) return fail(UW_ERR_INVALID_ARG, "uw_matmul_host: NULL host buffer");
    size_t need = 0, inner = 0;
    uw_status s = uw_host_workspace_size(m, B, od, &need);
    if (s != UW_OK) return s;
    if (ws_bytes < need || !ws) return fail(UW_ERR_WORKSPACE, "uw_matmul_host: workspace %zu bytes, need %zu", ws_bytes, need);
    uw_workspace_size(m, B, UW_STRAT_AUTO, &inner);
    uint8_t *p = (uint8_t *)ws;
    uint8_t *xd = p + round_up(inner, 256);
    uint8_t *yd = xd + round_up((uint64_t)B * m->h.K * 2, 256);
    const size_t xb = (size_t)B * m->h.K * 2, yb = (size_t)B * m->h.N * (od == UW_OUT_BF16 ? 2 : 4);
    cudaStream_t st = (cudaStream_t)stream;
    UW_CUDA(cudaMemcpyAsync(xd, x_host, xb, cudaMemcpyHostToDevice, st), "uw_matmul_host: H2D");
    s = uw_matmul(m, (const uint16_t *)xd, B, yd, od, UW_STRAT_AUTO, p, round_up(inner, 256), stream);
    if (s != UW_OK) return s;
    UW_CUDA(cudaMemcpyAsync(y_host, yd, yb, cudaMemcpyDeviceToHost, st), "uw_matmul_host: D2H");
    return UW_OK;
}

extern "C" uw_status uw_matmul_host(const uw_matrix *m, const uint16_t *x_host, int64_t B, void *y_host,
                                    uw_out_dtype od, void *ws, size_t ws_bytes, uw_stream stream)
{
    uw_status s = uw_matmul_host_async(m, x_host, B, y_host, od, ws, ws_bytes, stream);
    if (s != UW_OK) return s;
    UW_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "uw_matmul_host: synchronize");
    return UW_OK;
}

// ------------------------------------------------------------------------------ autotune
namespace {

std::vector<int> split_candidates(const uw_matrix *m)
{
    std::vector<int> v = {0, 1, 2, 4, 8};
    v.erase(std::remove_if(v.begin(), v.end(), [&](int s) { return s > 1 && (int64_t)s * 512 > m->h.K; }), v.end());
    return v;
}

}  // namespace

extern "C" uw_status uw_autotune_workspace_size(const uw_matrix *m, const int64_t *batches, int n, size_t *bytes)
{
    clear_error();
    if (!m || !bytes || (n && !batches) || n < 0) return fail(UW_ERR_INVALID_ARG, "uw_autotune_workspace_size: bad arguments");
    uint64_t best = 0;
    for (int i = 0; i < n; i++) {
        const int64_t B = std::max<int64_t>(batches[i], 1);
        uint64_t pre = 0;
        for (int s = UW_STRAT_FULL_DECODE; s <= UW_STRAT_HUFFMAN_DIRECT; s++)
            if (strategy_ok(m, s)) pre = std::max(pre, preprocess_bytes(m, s));
        const uint64_t acc = round_up((uint64_t)B * m->h.N * 4, 256);
        const uint64_t xy = round_up((uint64_t)B * m->h.K * 2, 256) + round_up((uint64_t)B * m->h.N * 4, 256);
        best = std::max(best, pre + acc + xy);
    }
    *bytes = best;
    return UW_OK;
}

extern "C" uw_status uw_autotune(uw_matrix *m, const int64_t *batches, int n, void *ws, size_t ws_bytes, uw_stream stream)
{
    clear_error();
    size_t need = 0;
    uw_status s = uw_autotune_workspace_size(m, batches, n, &need);
    if (s != UW_OK) return s;
    if (ws_bytes < need || (need && !ws)) return fail(UW_ERR_WORKSPACE, "uw_autotune: workspace %zu bytes, need %zu", ws_bytes, need);
    cudaStream_t st = (cudaStream_t)stream;
    cudaEvent_t e0, e1;
    UW_CUDA(cudaEventCreate(&e0), "uw_autotune: event");
    UW_CUDA(cudaEventCreate(&e1), "uw_autotune: event");
    // a buffer of twice the L2 size, rewritten before each timed launch, so every candidate streams its weights
    // from HBM as it will in use (without it a matrix that fits in L2 is timed warm); skipped if it cannot be had
    void *flush = nullptr;
    size_t flush_bytes = 0;
    {
        int dev = 0, l2 = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
        flush_bytes = 2 * (size_t)l2;
        if (flush_bytes == 0 || cudaMalloc(&flush, flush_bytes) != cudaSuccess) {
            cudaGetLastError();
            flush = nullptr;
        }
    }
    uw_status result = UW_OK;
    for (int bi = 0; bi < n && result == UW_OK; bi++) {
        const int64_t B = std::max<int64_t>(batches[bi], 1);
        uint8_t *base = (uint8_t *)ws;
        // X and Y live at the end of the workspace; X is filled with a fixed bf16 pattern (1.0)
        const uint64_t xb = round_up((uint64_t)B * m->h.K * 2, 256), yb = round_up((uint64_t)B * m->h.N * 4, 256);
        uint8_t *xd = base + need - xb - yb, *yd = base + need - yb;
        const size_t inner_cap = need - xb - yb;
        if (cudaMemsetAsync(xd, 0x3F, (size_t)B * m->h.K * 2, st) != cudaSuccess) { result = fail(UW_ERR_CUDA, "uw_autotune: memset"); break; }

        auto time_plan = [&](const uw_plan &p, float *us) -> bool {
            size_t wsz = 0;
            if (uw_plan_workspace_size(m, B, &p, &wsz) != UW_OK || wsz > inner_cap) return false;
            float samples[7];
            for (int r = 0; r < 2; r++)
                if (uw_matmul_plan(m, (const uint16_t *)xd, B, yd, UW_OUT_F32, &p, base, inner_cap, stream) != UW_OK) return false;
            // a sample: three back-to-back launches (as in a model, where matmuls follow one another and the next
            // one's start overlaps the last one's end), after the L2 flush
            for (int r = 0; r < 7; r++) {
                if (flush) cudaMemsetAsync(flush, r, flush_bytes, st);
                cudaEventRecord(e0, st);
                for (int q = 0; q < 3; q++)
                    if (uw_matmul_plan(m, (const uint16_t *)xd, B, yd, UW_OUT_F32, &p, base, inner_cap, stream) != UW_OK)
                        return false;
                cudaEventRecord(e1, st);
                if (cudaEventSynchronize(e1) != cudaSuccess) return false;
                cudaEventElapsedTime(&samples[r], e0, e1);
                samples[r] /= 3.f;
            }
            std::sort(samples, samples + 7);
            *us = samples[3] * 1000.f;
            return true;
        };

        uw_plan best = default_plan(m, B);
        if (best.kernel == UW_KERNEL_AUTO) best.kernel = resolve_kernel(m, best, B);
        float best_us = 0;
        if (!time_plan(best, &best_us)) best_us = 3.0e38f;
        // seeds the coordinate descent could not reach one coordinate at a time: each GEMV launch shape and the
        // tensor-core kernel, on the default strategy
        {
            std::vector<uw_plan> seeds;
            for (int v = 0; v <= 8; v++) seeds.push_back(uw_plan{best.strategy, UW_KERNEL_GEMV, 0, v});
            seeds.push_back(uw_plan{best.strategy, UW_KERNEL_TC, 0, 0});
            seeds.push_back(uw_plan{best.strategy, UW_KERNEL_TC, 0, 4});
            for (const uw_plan &p : seeds) {
                if (memcmp(&p, &best, sizeof p) == 0) continue;
                float us;
                if (time_plan(p, &us) && us < best_us * 0.98f) { best = p; best_us = us; }
            }
        }
        // coordinate descent over (strategy, kernel, split, variant)
        for (int round = 0; round < 3; round++) {
            bool improved = false;
            for (int coord = 0; coord < 4; coord++) {
                std::vector<int> values;
                if (coord == 0) { for (int v = UW_STRAT_FULL_DECODE; v <= UW_STRAT_HUFFMAN_DIRECT; v++) if (strategy_ok(m, v)) values.push_back(v); }
                else if (coord == 1) values = {UW_KERNEL_GEMV, UW_KERNEL_TC};
                else if (coord == 2) values = split_candidates(m);
                else if (best.kernel == UW_KERNEL_TC) values = {0, 4};
                else values = {0, 1, 2, 3, 4, 5, 6, 7, 8};
                for (int v : values) {
                    uw_plan p = best;
                    if (coord == 0) {
                        p.strategy = v;
                        if (v == UW_STRAT_HUFFMAN_DIRECT) p = default_plan_for_strategy(m, B, v);  // its only shape
                    } else if (coord == 1) p.kernel = v;
                    else if (coord == 2) p.split_k = v;
                    else p.variant = v;
                    if (memcmp(&p, &best, sizeof p) == 0) continue;
                    float us;
                    if (time_plan(p, &us) && us < best_us * 0.98f) { best = p; best_us = us; improved = true; }
                }
            }
            if (!improved) break;
        }
        cudaGetLastError();  // candidates that failed to launch leave no sticky error
        if (best_us >= 3.0e38f) { result = fail(UW_ERR_UNSUPPORTED, "uw_autotune: no plan ran for B=%lld", (long long)B); break; }
        std::lock_guard<std::mutex> g(m->mu);
        const int64_t bk = bucket_of(B);
        bool found = false;
        for (TuneEntry &t : m->tune)
            if (t.bucket == bk) { t.plan = best; t.us = best_us; found = true; }
        if (!found) m->tune.push_back(TuneEntry{bk, best, best_us});
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (flush) cudaFree(flush);
    return result;
}

extern "C" uw_status uw_tune_save(const uw_matrix *m, char *buf, size_t cap, size_t *len)
{
    clear_error();
    if (!m || !len) return fail(UW_ERR_INVALID_ARG, "uw_tune_save: NULL argument");
    std::ostringstream os;
    {
        std::lock_guard<std::mutex> g(const_cast<uw_matrix *>(m)->mu);
        for (const TuneEntry &t : m->tune) {
            char line[160];
            snprintf(line, sizeof line, "%lld %d %d %d %d %.3f\n", (long long)t.bucket, t.plan.strategy, t.plan.kernel,
                     t.plan.split_k, t.plan.variant, t.us);
            os << line;
        }
    }
    const std::string s = os.str();
    *len = s.size();
    if (!buf) return UW_OK;
    if (cap < s.size() + 1) return fail(UW_ERR_BUFFER_TOO_SMALL, "uw_tune_save: need %zu bytes", s.size() + 1);
    memcpy(buf, s.c_str(), s.size() + 1);
    return UW_OK;
}

extern "C" uw_status uw_tune_load(uw_matrix *m, const char *text)
{
    clear_error();
    if (!m || !text) return fail(UW_ERR_INVALID_ARG, "uw_tune_load: NULL argument");
    std::vector<TuneEntry> table;
    std::istringstream is(text);
    std::string line;
    while (std::getline(is, line)) {
        if (line.find_first_not_of(" \t\r") == std::string::npos) continue;
        long long b;
        int st, k, sp, va;
        float us;
        char extra;
        if (sscanf(line.c_str(), "%lld %d %d %d %d %f %c", &b, &st, &k, &sp, &va, &us, &extra) != 6)
            return fail(UW_ERR_INVALID_ARG, "uw_tune_load: malformed line '%s'", line.c_str());
        if (b < 1 || (b & (b - 1)) || st < UW_STRAT_FULL_DECODE || st > UW_STRAT_HUFFMAN_DIRECT || k < UW_KERNEL_GEMV ||
            k > UW_KERNEL_TC || sp < 0 || va < 0)
            return fail(UW_ERR_INVALID_ARG, "uw_tune_load: out-of-range value in '%s'", line.c_str());
        table.push_back(TuneEntry{b, uw_plan{st, k, sp, va}, us});
    }
    std::lock_guard<std::mutex> g(m->mu);
    m->tune = table;
    return UW_OK;
}

extern "C" const char *uw_version(void) { return "uw 0.1 (sm_103a)"; }
