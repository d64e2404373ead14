// uw_sequence.cu - a sequence of matmuls with the Huffman decode of "hard" matrices on a side stream.
//
// Cloudflare blog "Unweight", section on scheduling the pipelines: MLP layers alternate between "hard" ones, held
// Huffman-coded and needing a preprocess, and "easy" ones, held in the pre-transcoded palette form.  While the
// main stream runs attention and the easy layers, the next hard layer's weights are decoded on other CUDA streams
// into preprocess slots that are double-buffered; the down projection, consumed last in a layer, has the longest
// runway.  Here a step is hard when its matrix holds only its Huffman stream: its 4-bit codes are transcoded on
// the side stream into one of two slots of the workspace as soon as the slot is free (the matmul that read it two
// hard steps earlier is done), and the main stream's matmul waits only for that transcode.  Easy steps run their
// AUTO plan.  Everything is enqueued at once and ordered by events; the main stream ends joined with the side
// stream, so the whole sequence can be captured in one CUDA graph from the main stream.
//
// The section on the decode kernels adds that the decoder and the matmul cannot share an SM on H100 (the matmul's
// shared memory leaves no room for the decoder's table), so the SMs are split between them and the split is tuned.
// Here `decode_sms` d > 0 sizes the main stream's persistent matmul grids for the device's SMs minus d and gives the
// transcode a persistent grid of d SMs' worth of CTAs, so the two run side by side; d = UW_SEQ_DIRECT (-1) runs
// no transcode at all: every step, hard or easy, takes its own AUTO plan on the main stream (for a hard step at
// batch 8 or less, the GEMV that decodes the Huffman stream inside the product).  uw_sequence_tune times these
// schedules and returns the fastest: when a matmul already holds HBM at its peak, a transcode beside it cannot
// hide, and decoding inside the product costs less than transcoding first.
//
// Steps the caller marks UW_STEP_CONCURRENT may overlap the step before them (an MLP's gate and up projections
// read the same input).  On one stream each matmul waits for the whole preceding grid (its output may be the next
// one's input), its prologue overlapped with that grid's end by programmatic dependent launch; a UW_SEQ_GROUPS
// schedule instead runs a group of independent steps on the main stream and up to three streams of the library's
// own, forked and joined with events, so that the members overlap each other, at the cost of full dependencies
// at the fork and the join.  Which wins depends on the shapes and B, so the tuner times both.
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <utility>
#include <vector>

#include "uw_internal.h"

using namespace uw;

namespace {

uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

bool is_hard(const uw_matrix *m) { return m->codes == nullptr && m->has_stream; }

uint64_t slot_bytes_of(const uw_matrix *m) { return round_up((uint64_t)m->h.N * (uint64_t)m->h.K / 2 + 64, 256); }

constexpr int kLanes = 4;  // streams a group of concurrent steps runs on: the caller's and three of the library's

struct Layout {
    uint64_t slot;  // bytes of one preprocess slot (the largest hard matrix's codes)
    uint64_t mm;    // bytes of one lane's matmul workspace (the largest any step needs)
    int hard;       // hard steps
    int lanes;      // lanes the largest group of concurrent steps needs (each has its own matmul workspace)
};

uw_status layout_of(const uw_step *steps, int n, int64_t B, Layout *L)
{
    L->slot = L->mm = 0;
    L->hard = 0;
    L->lanes = 1;
    for (int i = 0, g = 0; i < n; i++) {
        g = (i > 0 && (steps[i].flags & UW_STEP_CONCURRENT)) ? g + 1 : 1;
        L->lanes = std::max(L->lanes, std::min(g, kLanes));
        if (steps[i].flags & ~UW_STEP_CONCURRENT) return fail(UW_ERR_INVALID_ARG, "uw_sequence: step %d has unknown flags", i);
        const uw_matrix *m = steps[i].m;
        if (!m) return fail(UW_ERR_INVALID_ARG, "uw_sequence: step %d has no matrix", i);
        if (is_hard(m)) {
            L->hard++;
            L->slot = std::max(L->slot, slot_bytes_of(m));
            L->mm = std::max<uint64_t>(L->mm, round_up(matmul_with_codes_workspace(m, B), 256));
            // the direct schedule runs the step's own AUTO plan instead
            size_t b = 0;
            uw_status s = uw_workspace_size(m, B, UW_STRAT_AUTO, &b);
            if (s != UW_OK) return s;
            L->mm = std::max<uint64_t>(L->mm, round_up(b, 256));
        } else {
            size_t b = 0;
            uw_status s = uw_workspace_size(m, B, UW_STRAT_AUTO, &b);
            if (s != UW_OK) return s;
            L->mm = std::max<uint64_t>(L->mm, round_up(b, 256));
        }
    }
    return UW_OK;
}

// The events a sequence uses, one set per thread and device, created by the thread's first call on that device
// and kept (a call captured into a CUDA graph then creates nothing).  Reusing them across calls is safe: a
// stream wait binds to the event's latest record when the wait is enqueued, and every wait of a call follows its
// own records.
using EventSet = std::array<cudaEvent_t, 6 + kLanes>;  // start, ready[2], freed[2], done, fork, join[kLanes - 1]
uw_status thread_events(EventSet **out)
{
    thread_local std::vector<std::pair<int, EventSet>> sets;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(UW_ERR_CUDA, "uw_sequence_run: cudaGetDevice: %s", cudaGetErrorString(e));
    for (auto &p : sets)
        if (p.first == dev) { *out = &p.second; return UW_OK; }
    EventSet es{};
    for (auto &ev : es)
        if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) {
            for (auto &d : es)
                if (d) cudaEventDestroy(d);
            return fail(UW_ERR_CUDA, "uw_sequence_run: event creation: %s", cudaGetErrorString(e));
        }
    sets.emplace_back(dev, es);
    *out = &sets.back().second;
    return UW_OK;
}

// The library's streams for groups of concurrent steps, kLanes - 1 per thread and device, created with the events.
using LaneStreams = std::array<cudaStream_t, kLanes - 1>;
uw_status thread_lanes(LaneStreams **out)
{
    thread_local std::vector<std::pair<int, LaneStreams>> sets;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(UW_ERR_CUDA, "uw_sequence_run: cudaGetDevice: %s", cudaGetErrorString(e));
    for (auto &p : sets)
        if (p.first == dev) { *out = &p.second; return UW_OK; }
    LaneStreams ls{};
    for (auto &st : ls)
        if ((e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking)) != cudaSuccess) {
            for (auto &d : ls)
                if (d) cudaStreamDestroy(d);
            return fail(UW_ERR_CUDA, "uw_sequence_run: stream creation: %s", cudaGetErrorString(e));
        }
    sets.emplace_back(dev, ls);
    *out = &sets.back().second;
    return UW_OK;
}

}  // namespace

extern "C" uw_status uw_sequence_workspace_size(const uw_step *steps, int n, int64_t B, size_t *bytes)
{
    clear_error();
    if (!bytes || n < 0 || (n && !steps) || B < 0) return fail(UW_ERR_INVALID_ARG, "uw_sequence_workspace_size: bad arguments");
    Layout L;
    uw_status s = layout_of(steps, n, B, &L);
    if (s != UW_OK) return s;
    *bytes = (L.hard ? 2 * L.slot : 0) + L.mm * (uint64_t)L.lanes;
    return UW_OK;
}

extern "C" uw_status uw_sequence_run(const uw_step *steps, int n, int64_t B, void *ws, size_t ws_bytes, uw_stream stream,
                                     uw_stream side_stream, int decode_sms)
{
    clear_error();
    if (n < 0 || (n && !steps) || B < 0) return fail(UW_ERR_INVALID_ARG, "uw_sequence_run: bad arguments");
    const bool groups = decode_sms >= UW_SEQ_GROUPS + UW_SEQ_DIRECT;
    if (groups) decode_sms -= UW_SEQ_GROUPS;
    if (decode_sms < UW_SEQ_DIRECT || decode_sms >= device_sms())
        return fail(UW_ERR_INVALID_ARG, "uw_sequence_run: decode_sms %d outside [-1, %d)", decode_sms, device_sms());
    if (n == 0 || B == 0) return UW_OK;
    Layout L;
    uw_status s = layout_of(steps, n, B, &L);
    if (s != UW_OK) return s;
    const uint64_t need = (L.hard ? 2 * L.slot : 0) + L.mm * (uint64_t)L.lanes;
    if (ws_bytes < need || (need && !ws)) return fail(UW_ERR_WORKSPACE, "uw_sequence_run: workspace %zu bytes, need %llu", ws_bytes, (unsigned long long)need);
    if (ws && ((uintptr_t)ws & 255)) return fail(UW_ERR_INVALID_ARG, "uw_sequence_run: workspace not 256-byte aligned");
    if (L.hard && decode_sms != UW_SEQ_DIRECT && stream == side_stream)
        return fail(UW_ERR_INVALID_ARG, "uw_sequence_run: the side stream must differ from the main stream");
    for (int i = 0; i < n; i++)
        if (steps[i].out_dtype != UW_OUT_F32 && steps[i].out_dtype != UW_OUT_BF16)
            return fail(UW_ERR_INVALID_ARG, "uw_sequence_run: step %d has a bad output dtype", i);
    uint8_t *slot[2] = {(uint8_t *)ws, (uint8_t *)ws + L.slot};
    uint8_t *mm = (uint8_t *)ws + (L.hard ? 2 * L.slot : 0);
    cudaStream_t main = (cudaStream_t)stream, side = (cudaStream_t)side_stream;
    const bool transcode = L.hard && decode_sms != UW_SEQ_DIRECT;

    EventSet *ev = nullptr;
    s = thread_events(&ev);
    if (s != UW_OK) return s;
    LaneStreams *lanes = nullptr;
    if (groups && L.lanes > 1 && (s = thread_lanes(&lanes)) != UW_OK) return s;
    cudaEvent_t start = (*ev)[0], ready[2] = {(*ev)[1], (*ev)[2]}, freed[2] = {(*ev)[3], (*ev)[4]}, done = (*ev)[5];
    cudaEvent_t fork = (*ev)[6];
    // the split: the matmuls' grids for the SMs left, the transcode's for d SMs
    SmBudget budget(decode_sms > 0 ? device_sms() - decode_sms : 0);
    const int decode_ctas = decode_sms > 0 ? decode_sms * kDecodeCtasPerSm : 0;
    cudaError_t e = cudaSuccess;

    // steps [i0, i1), which the caller marked concurrent after i0: the main stream and the lanes, each member
    // with its own matmul workspace; a single step runs on the main stream
    auto run_group = [&](int i0, int i1) -> uw_status {
        const int n_g = i1 - i0;
        const int used = std::min(n_g, kLanes);
        if (used > 1) {
            if ((e = cudaEventRecord(fork, main)) != cudaSuccess) return fail(UW_ERR_CUDA, "uw_sequence_run: %s", cudaGetErrorString(e));
            for (int l = 1; l < used; l++)
                if ((e = cudaStreamWaitEvent((*lanes)[l - 1], fork, 0)) != cudaSuccess)
                    return fail(UW_ERR_CUDA, "uw_sequence_run: %s", cudaGetErrorString(e));
        }
        uw_status r = UW_OK;
        for (int j = 0; j < n_g && r == UW_OK; j++) {
            const int l = j % kLanes;
            const uw_step &st = steps[i0 + j];
            cudaStream_t sl = l ? (*lanes)[l - 1] : main;
            r = uw_matmul(st.m, st.x, B, st.y, (uw_out_dtype)st.out_dtype, UW_STRAT_AUTO, mm + (uint64_t)l * L.mm, L.mm,
                          (uw_stream)sl);
        }
        // join every forked lane, also after a failed step, so that a capture from the main stream stays joined
        for (int l = 1; l < used; l++) {
            cudaEvent_t join = (*ev)[6 + l];
            if ((e = cudaEventRecord(join, (*lanes)[l - 1])) != cudaSuccess || (e = cudaStreamWaitEvent(main, join, 0)) != cudaSuccess)
                return r != UW_OK ? r : fail(UW_ERR_CUDA, "uw_sequence_run: %s", cudaGetErrorString(e));
        }
        return r;
    };
    // where the group starting at step i ends: the run of steps marked concurrent after it (without UW_SEQ_GROUPS,
    // and for a hard step of the transcode schedule, the step alone)
    auto group_end = [&](int i) {
        if (!groups || (transcode && is_hard(steps[i].m))) return i + 1;
        int j = i + 1;
        while (j < n && (steps[j].flags & UW_STEP_CONCURRENT) && !(transcode && is_hard(steps[j].m))) j++;
        return j;
    };

    if (!transcode) {
        for (int i = 0; i < n && s == UW_OK;) {
            const int j = group_end(i);
            s = run_group(i, j);
            i = j;
        }
        return s;
    }

    // events: the side stream starts after the work already on the main stream; ready[k] - slot k holds the codes of
    // the hard step that uses it next; freed[k] - the matmul that read slot k is done; done - the side stream's end
    std::vector<int> hard;
    for (int i = 0; i < n; i++)
        if (is_hard(steps[i].m)) hard.push_back(i);
    e = cudaEventRecord(start, main);
    if (!e) e = cudaStreamWaitEvent(side, start, 0);
    // the transcode of hard step j into slot j % 2, on the side stream, once the matmul of hard step j - 2 is done
    auto enqueue_transcode = [&](int j) -> cudaError_t {
        const int k = j & 1;
        cudaError_t r = cudaSuccess;
        if (j >= 2) r = cudaStreamWaitEvent(side, freed[k], 0);
        if (!r) r = (cudaError_t)launch_decode_huffman(steps[hard[j]].m->v, DEC_CODES, slot[k], side, decode_ctas);
        if (!r) r = cudaEventRecord(ready[k], side);
        return r;
    };
    for (int j = 0; j < std::min<int>(2, (int)hard.size()) && !e; j++) e = enqueue_transcode(j);
    int hj = 0;
    for (int i = 0; i < n && !e && s == UW_OK;) {
        const uw_step &st = steps[i];
        if (hj < (int)hard.size() && hard[hj] == i) {
            const int k = hj & 1;
            e = cudaStreamWaitEvent(main, ready[k], 0);
            if (!e) s = matmul_with_codes(st.m, slot[k], st.x, B, st.y, (uw_out_dtype)st.out_dtype, mm, L.mm, main);
            if (!e && s == UW_OK) e = cudaEventRecord(freed[k], main);
            if (!e && s == UW_OK && hj + 2 < (int)hard.size()) e = enqueue_transcode(hj + 2);
            hj++;
            i++;
        } else {
            const int j = group_end(i);
            s = run_group(i, j);
            i = j;
        }
    }
    // join: the main stream ends after the side stream's last transcode
    if (!e) e = cudaEventRecord(done, side);
    if (!e) e = cudaStreamWaitEvent(main, done, 0);
    if (e) return fail(UW_ERR_CUDA, "uw_sequence_run: %s", cudaGetErrorString(e));
    return s;
}

extern "C" uw_status uw_sequence_tune(const uw_step *steps, int n, int64_t B, void *ws, size_t ws_bytes, uw_stream stream,
                                      uw_stream side_stream, int *decode_sms)
{
    clear_error();
    if (!decode_sms) return fail(UW_ERR_INVALID_ARG, "uw_sequence_tune: decode_sms is NULL");
    *decode_sms = 0;
    if (n == 0 || B == 0) return UW_OK;
    cudaStream_t main = (cudaStream_t)stream;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        return fail(UW_ERR_CUDA, "uw_sequence_tune: event creation failed");
    }
    const int sms = device_sms();
    bool flagged = false;
    for (int i = 1; i < n; i++) flagged |= (steps[i].flags & UW_STEP_CONCURRENT) != 0;
    std::vector<int> cand;
    for (int g : {0, UW_SEQ_GROUPS})
        if (g == 0 || flagged)
            for (int d : {UW_SEQ_DIRECT, 0, 8, 16, 24, 32, 40, 48, 64, 80, 96})
                if (d < sms) cand.push_back(g + d);
    // one candidate: an eager run (checks it and creates the thread's events and streams), then the sequence
    // captured into a graph, two replays, and three bursts of three replays timed; where `stream` cannot be
    // captured (the legacy default stream), five eager runs, the last three timed
    auto timed = [&](int d, float *ms) -> uw_status {
        uw_status s = uw_sequence_run(steps, n, B, ws, ws_bytes, stream, side_stream, d);
        if (s != UW_OK) return s;
        cudaGraph_t g = nullptr;
        cudaGraphExec_t ge = nullptr;
        if (cudaStreamBeginCapture(main, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
            s = uw_sequence_run(steps, n, B, ws, ws_bytes, stream, side_stream, d);
            cudaError_t e = cudaStreamEndCapture(main, &g);
            if (s != UW_OK) {
                if (g) cudaGraphDestroy(g);
                return s;
            }
            if (e != cudaSuccess || cudaGraphInstantiate(&ge, g, 0) != cudaSuccess) ge = nullptr;
        }
        cudaGetLastError();  // a refused capture leaves its error behind; the eager timing below stands in
        float t[3];
        for (int r = 0; r < 5; r++) {
            if (r >= 2) cudaEventRecord(e0, main);
            for (int k = 0; k < (ge && r >= 2 ? 3 : 1); k++) {
                if (ge) {
                    if (cudaGraphLaunch(ge, main) != cudaSuccess) s = fail(UW_ERR_CUDA, "uw_sequence_tune: graph launch failed");
                } else {
                    s = uw_sequence_run(steps, n, B, ws, ws_bytes, stream, side_stream, d);
                }
                if (s != UW_OK) break;
            }
            if (s != UW_OK) break;
            if (r >= 2) {
                cudaEventRecord(e1, main);
                if (cudaEventSynchronize(e1) != cudaSuccess) {
                    s = fail(UW_ERR_CUDA, "uw_sequence_tune: %s", cudaGetErrorString(cudaGetLastError()));
                    break;
                }
                cudaEventElapsedTime(&t[r - 2], e0, e1);
            }
        }
        if (ge) cudaGraphExecDestroy(ge);
        if (g) cudaGraphDestroy(g);
        if (s != UW_OK) return s;
        std::sort(t, t + 3);
        *ms = t[1];
        return UW_OK;
    };
    float best = 3.0e38f;
    uw_status result = UW_OK;
    for (int d : cand) {
        float ms = 0.0f;
        uw_status s = timed(d, &ms);
        if (s != UW_OK) {
            if (d == 0 || s == UW_ERR_CUDA) {  // the plain schedule must run; a CUDA error ends the search
                result = s;
                break;
            }
            continue;  // a split this sequence cannot take (a budget too small for a kernel)
        }
        if (ms < best * 0.99f) { best = ms; *decode_sms = d; }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return result;
}
