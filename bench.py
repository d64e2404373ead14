"""Benchmark: fused decompress + matmul on the Llama-3.1-8B-shaped gate_proj W[14336,4096].

One step = one uw_matmul of the autotuned plan (AUTO) at B=1 on a Huffman-coded
matrix held on the device as its 4-bit palette form (the stream is transcoded at
load time and dropped), i.e. one pass of the whole hot path: strategy lookup,
(preprocess if the plan has one), on-chip BF16 reconstruction and the
contraction.  Inputs are larger than L2: the step rotates over several device
copies of the compressed matrix (each copy its own uw_matrix), so every step
streams its weights from HBM.  Steps are replayed through CUDA graphs captured
from the same C-ABI calls.

Timing: nvidia-smi samples the clocks from before an untimed load ramp; then,
after a barrier and a synchronize, the stream starts with a short spin kernel
(a fixed number of clock cycles, about 2 ms) while the warm-up steps and the
timed steps (between two CUDA events) are queued behind it.  So the GPU runs
warm-up and timed steps back to back with no idle gap and no host launch
latency inside the timed region; a synchronize and a barrier close it.  (The
spin ends by itself: under a profiler that launches synchronously it only
delays the queue.)

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle (the
plain C decoder + fp64 matmul) on the host cores instead.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 2 ** 20
E2E_STREAMS = 3  # independent calls in flight in the end-to-end and concurrent measurements
WORKLOAD = "gate_8b"
REF_BUDGET_S = 90.0  # CPU seconds of the reference arm's whole run (warm-up and timed steps)
CSRC = os.path.join(ROOT, "lossless_bf16_weight_exponent_gb300", "csrc")

# DRAM bytes (read + write) per launch of a kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by (workload, batch, kernel name), with the source file of the kernel and the first
# 16 hex digits of its SHA-256 at capture time.  When the source has changed since, the figure no longer describes
# the kernel and the line reports null.
MEASURED_TRAFFIC = {
    ("gate_8b", 1, "gemv_tma_kernel"): (89030656 + 2406144, "k_gemv_tma.cu", "695ab47d5dc64a39"),
}


def source_sha16(fname):
    try:
        with open(os.path.join(CSRC, fname), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None


KERNEL_SOURCE = {"gemv_tma_kernel": "k_gemv_tma.cu", "gemv_rp_kernel": "k_gemv_rp.cu", "gemv_mma_kernel": "k_gemv_mma.cu",
                 "gemv_huff_kernel": "k_gemv_huff.cu", "gemv_kernel": "k_gemv.cu", "tc4_kernel": "k_tc4.cu",
                 "tc_kernel": "k_tc.cu"}


def measured_traffic(workload, B, kname):
    """(bytes per launch, capture note) when a capture of this kernel as it stands exists, else (None, why)."""
    e = MEASURED_TRAFFIC.get((workload, B, kname))
    if e is None:
        return None, "no ncu capture of this kernel and workload"
    nbytes, fname, sha = e
    if source_sha16(fname) != sha:
        return None, f"{fname} changed since its ncu capture"
    return nbytes, f"ncu capture of {kname} ({fname} sha256 {sha})"


def kernel_name(plan, B):
    """The kernel a plan launches (the dominant kernel of a step), as named in ncu launch lists."""
    import lossless_bf16_weight_exponent_gb300 as uw
    if plan.strategy == uw.STRAT_HUFFMAN_DIRECT:
        return "gemv_huff_kernel"
    if plan.kernel == uw.KERNEL_TC or (plan.kernel == uw.KERNEL_AUTO and B > 2):
        return "tc4_kernel" if plan.variant == 4 else "tc_kernel"
    if plan.variant == 8:
        return "gemv_rp_kernel"
    if plan.variant in (6, 7) and B <= 16:
        return "gemv_mma_kernel"
    if plan.variant == 1 or B > 2:
        return "gemv_kernel"
    return "gemv_tma_kernel"


def launches_per_call(plan, B):
    """Kernels of this library that one uw_matmul of the plan launches (fp32 output): a preprocess kernel for the
    Huffman-fed pipelines, the zeroing kernel of the kernels that add into a zeroed target, the matmul kernel.
    (Memset nodes of the K-split kernels are not kernels of this library.)"""
    import lossless_bf16_weight_exponent_gb300 as uw
    pre = 1 if plan.strategy in (uw.STRAT_FULL_DECODE, uw.STRAT_EXP_ONLY, uw.STRAT_PALETTE_TRANSCODE) else 0
    zero = 1 if kernel_name(plan, B) in ("gemv_rp_kernel", "tc4_kernel", "gemv_huff_kernel") else 0
    return pre + zero + 1


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--batch", type=int, default=1)
    p.add_argument("--no-breakdown", action="store_true", help="skip the per-strategy and per-workload points")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-autotune", action="store_true")
    p.add_argument("--points-budget", type=float, default=150.0,
                   help="seconds the per-workload points may take (points past it are listed as skipped)")
    p.add_argument("--json-out", default=None)
    p.add_argument("--workload", default="gate_8b",
                   choices=["gate_8b", "down_8b", "gate_70b", "down_70b", "heavy_tail", "tiny"],
                   help="matrix recipe (the JSON line's headline workload is gate_8b)")
    p.add_argument("--plan", default=None, help="force a plan 'strategy,kernel,split,variant' (skips autotuning)")
    p.add_argument("--sweep", action="store_true",
                   help="time every configuration (tiny, 8B gate, 8B MLP stack, heavy tail, 70B gate/down) at each of "
                        "its batch sizes under the autotuned plan; one JSON line per (configuration, B)")
    p.add_argument("--stack-layers", type=int, default=32, help="layers of the 8B MLP stack")
    p.add_argument("--resident", default="palette", choices=["palette", "huffman", "both"],
                   help="what stays resident of the Huffman blob: the palette form alone (default), the Huffman "
                        "stream alone (AUTO then decodes the stream inside the GEMV for B <= 8), or both")
    return p.parse_args(argv)


def workload_matrix(name):
    import synth
    if name == "gate_8b":
        return synth.gate_8b()
    if name == "down_8b":
        return synth.stack_8b(1)[2]
    if name == "gate_70b":
        return synth.mlp_70b()[0]
    if name == "down_70b":
        return synth.mlp_70b()[2]
    if name == "heavy_tail":
        return synth.heavy_tail()
    return synth.tiny()


def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, which)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def algorithmic_bytes(info, strategy, B, out_bytes=4):
    """Bytes a pass must move at minimum: the compressed stream the strategy reads, X and Y."""
    N, K = info["N"], info["K"]
    n = N * K
    words = (info["n_blocks"] + 31) // 32
    common = n + 64 * info["n_verbatim"] + 8 * words  # sm bytes, verbatim exponents, bitmap + prefix
    if strategy == 4:   # direct palette: resident 4-bit codes
        w = common + n // 2
    else:               # Huffman-fed pipelines read the bit stream and its chunk offsets
        w = common + (info["total_bits"] + 7) // 8 + 4 * (info["n_chunks"] + 1)
    return w + 2 * B * K + out_bytes * B * N


class Clocks:
    """nvidia-smi sampling of SM and memory clocks and throttle reasons while the GPU works."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,clocks.mem,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.gpu = gpu_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-i", str(self.gpu), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
            return
        # until the first sample is written (or a second has passed)
        t0 = time.time()
        while time.time() - t0 < 1.0:
            self.f.flush()
            if os.path.getsize(self.f.name) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mem, mx, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                mx = float(r[3])
                mem.append(float(r[4]))
                for nm, v in zip(names, r[7:11]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except Exception:
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "mem_mhz": statistics.median(mem) if mem else None, "reasons": sorted(reasons), "samples": len(sm),
                "window": "from before the untimed load ramp to the end of the timed region"}


def hold_stream(stream, seconds=2e-3, mhz=2070.0):
    """Queue a spin kernel of about `seconds` at the maximum SM clock on `stream` (torch's cycle-count sleep), so
    that the launches that follow are all queued before the first of them runs."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(seconds * mhz * 1e6))


def gpu_id(dev):
    """nvidia-smi selector of the CUDA device in use (UUID; CUDA_VISIBLE_DEVICES may remap indices)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else str(dev)


def dist_setup():
    """Rank, world size and local rank from the launcher's environment.  One process per GPU: NCCL when CUDA is
    present, else gloo (the host-side path the CPU tests run)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The largest of every rank's v (the slowest rank's time bounds the whole job)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step, steps, world, ms_total):
    """Whole-job GB/s: every rank runs `steps` steps of `bytes_per_step` (weak scaling: the work per rank is fixed),
    over the slowest rank's time."""
    return bytes_per_step * world * steps / (ms_total * 1e-3) / 1e9


# ------------------------------------------------------------------ CPU oracle (reference arm / baseline)
def oracle_step_seconds(blob, w_shape, x_np, steps):
    """The oracle as it stands: decode the blob (plain C) and the fp64 matmul, `steps` times."""
    import oracle
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        w = oracle.decode(blob)
        oracle.matmul(w, x_np)
        times.append(time.perf_counter() - t0)
    return times


def run_reference(args):
    """The oracle as it stands, on the host cores: exactly `--warmup` (at least 3) untimed and `--steps` timed
    steps, each a bounded sample of the workload: the first rows of the recipe's W, encoded by the oracle as their
    own Huffman blob, decoded in plain C and multiplied in fp64.  The sample's rows are sized from a short probe so
    that the whole run takes about REF_BUDGET_S seconds of CPU work; throughput counts the sample's bytes."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import synth
    oracle.build()
    synth.build()
    mat = synth.gate_8b()
    w = mat.weights()
    x = mat.activations(args.batch)
    steps, warm = max(1, args.steps), max(3, args.warmup)
    probe_rows = min(mat.N, 256)
    probe = oracle.encode(np.ascontiguousarray(w[:probe_rows]), oracle.HUFFMAN)
    per_row = min(oracle_step_seconds(probe, (probe_rows, mat.K), x, 2)) / probe_rows
    rows = int(min(mat.N, max(64, REF_BUDGET_S / ((steps + warm) * per_row))))
    blob = oracle.encode(np.ascontiguousarray(w[:rows]), oracle.HUFFMAN)
    oracle_step_seconds(blob, (rows, mat.K), x, warm)
    times = oracle_step_seconds(blob, (rows, mat.K), x, steps)
    sec = sum(times) / len(times)
    eff = (2 * rows * mat.K + 2 * args.batch * mat.K + 4 * args.batch * rows) / sec / 1e9
    sample = (f"each step: the first {rows} of the {mat.N} rows of W (as their own Huffman blob), plain-C decode + "
              f"fp64 GEMV at B={args.batch}")
    line = {
        "impl": "reference", "metric": "effective BF16 weight GB/s, fused decompress+matmul (B=%d)" % args.batch,
        "value": eff, "unit": "GB/s", "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{WORKLOAD} W[14336,4096] bf16 N(0,0.02)+1e-4x100, Huffman blob",
                                         "batch": args.batch},
        "cpu_baseline": {"value": eff, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": eff, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ helpers of the GPU arm
def load_copies(blob, resident, min_copies=2):
    """Enough device copies of one matrix that a rotation over them streams from HBM (3x L2 at least)."""
    import lossless_bf16_weight_exponent_gb300 as uw
    base = uw.Matrix(blob, resident=resident)
    copies = min(64, max(min_copies, int(np.ceil(3 * L2_BYTES / max(1, base.info["device_bytes"])))))
    return [base] + [uw.Matrix(blob, resident=resident) for _ in range(copies - 1)]


def autotune_shared(mats, batches):
    """Autotune the first copy for `batches` and share its table with the others."""
    import torch
    need = mats[0].autotune_workspace_size(batches)
    tws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    mats[0].autotune(batches, tws, need)
    del tws
    table = mats[0].tune_save()
    for m in mats[1:]:
        m.tune_load(table)


def time_graph(fn, n, reps, stream):
    """Median µs of one replay of a CUDA graph holding n calls of fn(i, stream), after warm-up replays."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(n):
            fn(i, stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(i, stream)
        for _ in range(3):
            g.replay()
        stream.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts)


def concurrent_device(mats, mat, B, K, W, stream, nstreams=E2E_STREAMS):
    """The same K matmuls as independent calls on `nstreams` streams (call i on stream i % nstreams, each stream with
    its own Y and workspace), forked from and joined back to `stream` inside one CUDA graph; CUDA events on `stream`
    around a replay, after W warm-up calls and behind the 2 ms spin kernel.  On one stream each matmul's consumers
    wait for the preceding grid to finish (its output may be their input); independent calls on several streams
    overlap instead.  Returns milliseconds for the K calls."""
    import torch

    import lossless_bf16_weight_exponent_gb300 as uw
    copies = len(mats)
    side = [torch.cuda.Stream() for _ in range(nstreams)]
    ws_bytes = max(m.workspace_size(B) for m in mats)
    wss = [torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") for _ in side]
    ys = [torch.empty((B, mat.N), dtype=torch.float32, device="cuda") for _ in side]
    x = torch.from_numpy(mat.activations(B).view(np.int16)).cuda()

    def calls(first, n):
        for i in range(first, first + n):
            j = i % nstreams
            mats[i % copies].matmul(x, B, ys[j], uw.OUT_F32, uw.STRAT_AUTO, wss[j], ws_bytes, side[j])

    def fork_join(first, n):
        for sd in side:
            sd.wait_stream(stream)
        calls(first, n)
        for sd in side:
            stream.wait_stream(sd)

    with torch.cuda.stream(stream):
        fork_join(0, W + K)  # every plan warmed outside capture
        stream.synchronize()
        gw, gt = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gw, stream=stream):
            fork_join(0, W)
        with torch.cuda.graph(gt, stream=stream):
            fork_join(W, K)
        gw.replay()
        gt.replay()
        stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream)
    with torch.cuda.stream(stream):
        gw.replay()
        e0.record(stream)
        gt.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def encode_many(recipes, threads=None):
    """Blobs of many matrices, generated and encoded on a thread pool (both run in C with the GIL released)."""
    import lossless_bf16_weight_exponent_gb300 as uw
    threads = threads or max(1, min(16, (os.cpu_count() or 4)))

    def one(r):
        return uw.encode(r.weights(), uw.CODEC_HUFFMAN)
    with cf.ThreadPoolExecutor(threads) as ex:
        return list(ex.map(one, recipes))


def point_line(cfg, mat_desc, B, us, comp_bytes, eff_bytes, flops, plan, hbm, tf_peak, extra=None):
    d = {"config": cfg, "matrix": mat_desc, "B": B, "us": round(us, 2),
         "compressed_GBps": round(comp_bytes / us / 1e3, 1), "compressed_frac": round(comp_bytes / us / 1e3 / hbm, 3),
         "effective_GBps": round(eff_bytes / us / 1e3, 1), "effective_frac": round(eff_bytes / us / 1e3 / hbm, 3),
         "tflops": round(flops / us / 1e6, 1), "tensor_frac": round(flops / us / 1e6 / tf_peak, 3), "plan": plan}
    if extra:
        d.update(extra)
    return d


def measure_workload(cfg, mat, batches, resident, stream, hbm, tf_peak, blob=None):
    """Graph-timed, autotuned points of one matrix recipe: one line per batch size."""
    import torch

    import lossless_bf16_weight_exponent_gb300 as uw
    blob = blob if blob is not None else uw.encode(mat.weights(), uw.CODEC_HUFFMAN)
    single = mat.N * mat.K * 2 < L2_BYTES // 2
    mats = [uw.Matrix(blob, resident=resident)] if single else load_copies(blob, resident)
    copies = len(mats)
    autotune_shared(mats, batches)
    info = mats[0].info
    out = []
    for B in batches:
        ws_bytes = max(m.workspace_size(B) for m in mats)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        x = torch.from_numpy(mat.activations(B).view(np.int16)).cuda()
        y = torch.empty((B, mat.N), dtype=torch.float32, device="cuda")
        n = 32 if copies > 1 else 64
        us = time_graph(lambda i, s: mats[i % copies].matmul(x, B, y, uw.OUT_F32, uw.STRAT_AUTO, ws, ws_bytes, s),
                        n, 7, stream) / n
        plan = mats[0].plan_for(B)
        strat = 4 if info["has_palette_form"] else 5
        eff = 2 * mat.N * mat.K + 2 * B * mat.K + 4 * B * mat.N
        out.append(point_line(cfg, f"W[{mat.N},{mat.K}]", B, us, algorithmic_bytes(info, strat, B), eff,
                              2.0 * B * mat.N * mat.K, plan.as_tuple(), hbm, tf_peak,
                              {"kernel": kernel_name(plan, B), "resident": resident,
                               "resident_ratio": round(info["device_bytes"] / (2 * mat.N * mat.K), 4),
                               "l2": "matrix smaller than L2" if copies == 1 else
                               f"{copies} copies rotated, inputs larger than L2",
                               "verbatim_block_fraction": round(info["n_verbatim"] / info["n_blocks"], 4)}))
        del ws, x, y
    del mats
    torch.cuda.empty_cache()
    return out


def measure_stack(layers, batches, stream, hbm, tf_peak, hard_every=(8, 4, 2, 1)):
    """The 8B MLP stack: gate, up, down per layer (per-layer seeds), one graph per pass over all 3 x layers
    matmuls.  All layers easy (palette form resident, AUTO: direct palette); then hard layers (the Huffman stream
    alone) every k-th layer, run by uw_sequence_run under the schedule uw_sequence_tune picks: a side-stream
    transcode into double-buffered slots (with a decode SM split) or the direct schedule (each hard step's own AUTO
    plan, the Huffman-direct GEMV up to B = 8); then every matrix as the Huffman stream alone under AUTO.  Each
    pattern runs twice: every step after the one before it, and with each layer's up projection marked
    UW_STEP_CONCURRENT beside its gate projection (both read the layer's input; up writes its own buffer).  The
    gate/up shape and the down shape are autotuned once each per form and the tables shared by shape."""
    import torch

    import lossless_bf16_weight_exponent_gb300 as uw
    import synth
    recipes = synth.stack_8b(layers)
    blobs = encode_many(recipes)
    pal = [uw.Matrix(b, resident="palette") for b in blobs]
    huf = [uw.Matrix(b, resident="huffman") for b in blobs]
    del blobs
    for mats in (pal, huf):
        for first in (0, 2):
            need = mats[first].autotune_workspace_size(batches)
            tws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
            mats[first].autotune(batches, tws, need)
            del tws
            table = mats[first].tune_save()
            for i in range(first, len(mats), 3) if first == 2 else [i for i in range(len(mats)) if i % 3 != 2]:
                mats[i].tune_load(table)
    bf16_bytes = sum(2 * m.info["N"] * m.info["K"] for m in pal)
    side = torch.cuda.Stream()
    out = []
    for B in batches:
        x_in = torch.from_numpy(recipes[0].activations(B).view(np.int16)).cuda()            # [B, 4096]
        x_mid = torch.from_numpy(recipes[2].activations(B).view(np.int16)).cuda()           # [B, 14336]
        y_mid = torch.empty((B, 14336), dtype=torch.float32, device="cuda")
        y_up = torch.empty((B, 14336), dtype=torch.float32, device="cuda")
        y_out = torch.empty((B, 4096), dtype=torch.float32, device="cuda")

        def steps_of(mats, grouped):
            return [(m, x_mid if i % 3 == 2 else x_in, (y_mid, y_up, y_out)[i % 3], uw.OUT_F32,
                     uw.STEP_CONCURRENT if grouped and i % 3 == 1 else 0) for i, m in enumerate(mats)]
        flops = sum(2.0 * B * m.info["N"] * m.info["K"] for m in pal)
        eff = sum(2 * m.info["N"] * m.info["K"] + 2 * B * m.info["K"] + 4 * B * m.info["N"] for m in pal)
        patterns = [(name + suffix, k, grouped) for name, k in [("all easy", 0)] + [(f"hard every {k}", k)
                                                                                  for k in hard_every]
                    for suffix, grouped in (("", False), (", gate+up concurrent", True))]
        base_us = None
        for name, k, grouped in patterns:
            mats = [huf[i] if k and (i // 3) % k == k - 1 else pal[i] for i in range(len(pal))]
            steps = steps_of(mats, grouped)
            need = uw.sequence_workspace_size(steps, B)
            wsb = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
            wsp = (wsb.data_ptr() + 255) // 256 * 256
            hard = sum(1 for m in mats if not m.info["has_palette_form"])
            # the schedule: the decode-vs-matmul SM split, and whether the gate/up groups overlap
            d = uw.sequence_tune(steps, B, wsp, need, stream, side) if hard or grouped else 0
            overlap = d >= uw.SEQ_GROUPS + uw.SEQ_DIRECT
            d = d - uw.SEQ_GROUPS if overlap else d
            us = time_graph(lambda i, s: uw.sequence_run(steps, B, wsp, need, s, side,
                                                         d + (uw.SEQ_GROUPS if overlap else 0)), 1, 5, stream)
            # the transcode slots are resident while the sequence runs; the direct schedule uses none
            resident = sum(m.info["device_bytes"] for m in mats) + (need if hard and d != uw.SEQ_DIRECT else 0)
            base_us = base_us or us
            comp = sum(algorithmic_bytes(m.info, 4 if m.info["has_palette_form"] else 3, B) for m in mats)
            out.append(point_line("stack_8b", f"{layers} layers x (gate, up W[14336,4096]; down W[4096,14336])", B,
                                  us, comp, eff, flops,
                                  {"gate_up": pal[0].plan_for(B).as_tuple(), "down": pal[2].plan_for(B).as_tuple()},
                                  hbm, tf_peak,
                                  {"schedule": name, "matmuls": len(mats), "hard_matmuls": hard, "decode_sms": d,
                                   "groups_overlapped": overlap,
                                   "hard_steps": ("none" if not hard else "own AUTO plan (direct schedule)"
                                                  if d == uw.SEQ_DIRECT else "side-stream transcode"),
                                   "us_per_matmul": round(us / len(mats), 2), "time_vs_all_easy": round(us / base_us, 3),
                                   "resident_ratio": round(resident / bf16_bytes, 4),
                                   "api": "uw_sequence_run, schedule from uw_sequence_tune"}))
            del wsb
        # every matrix as the Huffman stream alone, AUTO plan per call
        if B <= 8:
            ws_bytes = max(m.workspace_size(B) for m in huf[:3])
            ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")

            def call(i, s):
                huf[i].matmul(x_mid if i % 3 == 2 else x_in, B, y_out if i % 3 == 2 else y_mid, uw.OUT_F32,
                              uw.STRAT_AUTO, ws, ws_bytes, s)
            us = time_graph(call, len(huf), 5, stream)
            comp = sum(algorithmic_bytes(m.info, 5, B) for m in huf)
            out.append(point_line("stack_8b", f"{layers} layers x (gate, up W[14336,4096]; down W[4096,14336])", B,
                                  us, comp, eff, flops, {"all": huf[0].plan_for(B).as_tuple()}, hbm, tf_peak,
                                  {"schedule": "all Huffman stream alone (AUTO)", "matmuls": len(huf),
                                   "us_per_matmul": round(us / len(huf), 2), "time_vs_all_easy": round(us / base_us, 3),
                                   "resident_ratio": round(sum(m.info["device_bytes"] for m in huf) / bf16_bytes, 4)}))
            del ws
    del pal, huf
    torch.cuda.empty_cache()
    return out


def strategy_breakdown(blob, mat, info_both, hbm_peak):
    """Per (B, strategy) timing of single eager calls rotating device copies that hold both the stream and the
    palette form (every strategy available), L2 not warm."""
    import torch

    import lossless_bf16_weight_exponent_gb300 as uw
    mats = load_copies(blob, "both")
    copies = len(mats)
    out = {}
    names = {1: "full_decode", 2: "exp_only", 3: "palette_transcode", 4: "direct_palette", 5: "huffman_direct"}
    for B in (1, 4, 16):
        x = torch.from_numpy(mat.activations(B).view(np.int16)).cuda()
        y = torch.empty((B, mat.N), dtype=torch.float32, device="cuda")
        eff = 2 * mat.N * mat.K + 2 * B * mat.K + 4 * B * mat.N
        row = {}
        for s, nm in names.items():
            if s == 5 and B > 8:
                continue  # the Huffman-direct GEMV takes B <= 8
            need = mats[0].workspace_size(B, s)
            ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
            for i in range(6):
                mats[i % copies].matmul(x, B, y, uw.OUT_F32, s, ws, need)
            st = torch.cuda.current_stream()
            reps = 40
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
            for i in range(reps):
                ev[2 * i].record(st)
                mats[i % copies].matmul(x, B, y, uw.OUT_F32, s, ws, need)
                ev[2 * i + 1].record(st)
            torch.cuda.synchronize()
            us = statistics.median(ev[2 * i].elapsed_time(ev[2 * i + 1]) * 1e3 for i in range(reps))
            alg = algorithmic_bytes(info_both, s, B)
            row[nm] = {"us": round(us, 2), "eff_GBps": round(eff / us / 1e3, 1),
                       "compressed_GBps": round(alg / us / 1e3, 1), "compressed_frac": round(alg / us / 1e3 / hbm_peak, 3)}
        out[f"B={B}"] = row
    del mats
    torch.cuda.empty_cache()
    return out


def footprint(blob, N, K):
    """Device bytes each resident form of the Huffman blob holds, against 2 N K bytes of BF16."""
    import lossless_bf16_weight_exponent_gb300 as uw
    out = {}
    for r in ("huffman", "palette", "both"):
        m = uw.Matrix(blob, resident=r)
        out[r] = round(m.info["device_bytes"] / (2 * N * K), 4)
        m.close()
    return out


def e2e_async(mats, mat, B, steps):
    """End-to-end throughput through uw_matmul_host_async: every step copies its X from pinned host memory, runs the
    matmul of the autotuned plan and copies Y back into pinned host memory; independent calls go round-robin to
    three streams, each with its own workspace and host buffers, so one call's copies and start overlap other calls'
    matmuls (with two streams a call's kernel still waited on its own copies; three keep the GPU busy).  Timed on
    the host clock from the first call to every stream's completion."""
    import torch
    copies = len(mats)
    streams = [torch.cuda.Stream() for _ in range(E2E_STREAMS)]
    need = max(m.host_workspace_size(B) for m in mats)
    wss = [torch.empty(need, dtype=torch.uint8, device="cuda") for _ in streams]
    xh = [torch.from_numpy(mat.activations(B).view(np.int16)).pin_memory() for _ in streams]
    yh = [torch.empty((B, mat.N), dtype=torch.float32).pin_memory() for _ in streams]

    def run(n):
        for i in range(n):
            j = i % len(streams)
            mats[i % copies].matmul_host_async(xh[j], B, yh[j], 0, wss[j], need, streams[j])
        for s in streams:
            s.synchronize()
    run(20)
    t0 = time.perf_counter()
    run(steps)
    return time.perf_counter() - t0


def cpu_baseline(blob, w, mat, B):
    x = mat.activations(B)
    times = oracle_step_seconds(blob, w.shape, x, 2)
    sec = sum(times) / len(times)
    eff = (2 * mat.N * mat.K + 2 * B * mat.K + 4 * B * mat.N) / sec / 1e9
    return {"value": eff, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"2 full steps: plain-C decode of the Huffman blob + fp64 GEMV at B={B}"}


# ------------------------------------------------------------------ GPU arm
def run_ours(args):
    import torch

    import lossless_bf16_weight_exponent_gb300 as uw
    import synth

    rank, world, local = dist_setup()
    dev = torch.cuda.current_device()
    hbm_peak, tf_peak, tf_sust, peak_kind = peaks()
    B = args.batch
    mat = workload_matrix(args.workload)
    w = mat.weights()
    blob = uw.encode(w, uw.CODEC_HUFFMAN)
    mats = load_copies(blob, args.resident)
    base = mats[0]
    info = base.info
    resident_bytes = info["device_bytes"]
    copies = len(mats)

    # autotune on one copy (batches of the workload), share the table with the others
    tune_batches = [1, 4, 16] if B in (1, 4, 16) else [B]
    if args.plan:
        vals = [int(v) for v in args.plan.split(",")]
        text = "%d %d %d %d %d 0\n" % (1 << max(0, (B - 1).bit_length()), *vals)
        for m in mats:
            m.tune_load(text)
    elif not args.no_autotune:
        autotune_shared(mats, tune_batches)
    plan = base.plan_for(B)
    ws_bytes = max(m.workspace_size(B) for m in mats)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    x = torch.from_numpy(mat.activations(B).view(np.int16)).cuda()
    y = torch.empty((B, mat.N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def step(i, s):
        mats[i % copies].matmul(x, B, y, uw.OUT_F32, uw.STRAT_AUTO, ws, ws_bytes, s)

    # CUDA graphs of G steps each, replayed to reach exactly n steps
    K, W = args.steps, max(3, args.warmup)
    G = min(64, K)
    graphs = {}

    def graph_for(n):
        if n not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                for i in range(n):  # warm the plan outside capture once
                    step(i, stream)
                stream.synchronize()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(n):
                        step(i, stream)
            graphs[n] = g
        return graphs[n]

    def run_steps(n):
        full, rem = divmod(n, G)
        gf = graph_for(G) if full else None
        gr = graph_for(rem) if rem else None
        with torch.cuda.stream(stream):
            for _ in range(full):
                gf.replay()
            if gr is not None:
                gr.replay()

    # every graph the warm-up and the timed region replay exists before timing starts
    for n in {G, K % G, W % G, min(W, G)} - {0}:
        graph_for(n)
    # a first estimate of the step time, for the length of the clock ramp
    t0 = time.perf_counter()
    run_steps(G)
    stream.synchronize()
    est = max((time.perf_counter() - t0) / G, 1e-6)

    clocks = Clocks(gpu_id(dev))
    clocks.start()
    run_steps(G * max(1, int(min(2e5, 0.5 / est) // G)))   # untimed load ramp: the sampled clocks see the GPU working
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream)
    run_steps(W)
    with torch.cuda.stream(stream):
        e0.record(stream)
    run_steps(K)
    with torch.cuda.stream(stream):
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world)
    ms_step = ms_total / K

    alg = algorithmic_bytes(info, plan.strategy, B)
    eff_bytes = 2 * mat.N * mat.K + 2 * B * mat.K + 4 * B * mat.N
    value = job_throughput(eff_bytes, K, world, ms_total)
    launches_per_step = launches_per_call(plan, B)

    # e2e through the public API with host buffers: H2D of X and D2H of Y inside the timed region, every step
    # the same steps as independent calls on several streams (device-timed), rank 0's extra line
    conc_ms = concurrent_device(mats, mat, B, K, W, stream) if rank == 0 else None
    e2e_steps = min(max(K, 200), 4000)
    e2e_s = max_over_ranks(e2e_async(mats, mat, B, e2e_steps), world)
    e2e_value = job_throughput(eff_bytes, e2e_steps, world, e2e_s * 1e3)

    forms = footprint(blob, mat.N, mat.K) if rank == 0 else None
    breakdown, points = {}, []
    if not args.no_breakdown and rank == 0 and args.workload == "gate_8b":
        breakdown = strategy_breakdown(blob, mat, uw.Matrix(blob, resident="both").info, hbm_peak)
        points = measure_points(args, stream, hbm_peak, tf_peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(blob, w, mat, B)

    if rank == 0:
        achieved = alg / (ms_step * 1e-3) / 1e9
        kname = kernel_name(plan, B)
        traffic, traffic_note = measured_traffic(args.workload, B, kname)
        form = {"palette": "Huffman blob transcoded at load time into its palette form, the stream dropped",
                "huffman": "Huffman blob alone", "both": "Huffman blob + its palette form"}[args.resident]
        line = {
            "metric": "effective BF16 weight GB/s, fused decompress+matmul (B=%d)" % B,
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms_step, "us_per_matmul": ms_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate", "data": "synthetic",
            "config": {"workload": f"{args.workload}: W[{mat.N},{mat.K}] bf16 ({mat.name} recipe), {form}; "
                                   f"X[{B},{mat.K}] N(0,1)",
                       "batch": B, "plan": plan.as_tuple(), "copies_rotated": copies,
                       "l2": f"inputs larger than L2: {copies} copies x {resident_bytes / 1e6:.1f} MB resident",
                       "timing": "warm-up and timed steps queued behind a 2 ms spin kernel, then CUDA events on the "
                                 "launching stream around the timed steps",
                       "compression": {"huffman_bits_per_weight": 8 * info["blob_bytes"] / (mat.N * mat.K),
                                       "verbatim_block_fraction": info["n_verbatim"] / info["n_blocks"]},
                       "footprint": {"resident_bytes": resident_bytes, "bf16_bytes": 2 * mat.N * mat.K,
                                     "resident_ratio": resident_bytes / (2 * mat.N * mat.K),
                                     "ratio_by_form": forms}},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic, "traffic_source": traffic_note,
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": alg, "kernel": kname},
            "effective_frac_of_peak": value / world / hbm_peak,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": 2 * B * mat.K,
                    "d2h_bytes_per_step": 4 * B * mat.N, "us_per_call": e2e_s / e2e_steps * 1e6, "steps": e2e_steps,
                    "api": f"uw_matmul_host_async, independent calls round-robin on {E2E_STREAMS} streams, pinned host "
                           "X and Y"},
            "concurrent": {"streams": E2E_STREAMS, "steps": K, "us_per_matmul": conc_ms / K * 1e3,
                           "value": eff_bytes * K / (conc_ms * 1e-3) / 1e9, "unit": "GB/s",
                           "compressed_frac": alg / (conc_ms / K * 1e-3) / 1e9 / hbm_peak,
                           "effective_frac": eff_bytes / (conc_ms / K * 1e-3) / 1e9 / hbm_peak,
                           "note": "the same matmuls as independent calls round-robin on several streams in one "
                                   "CUDA graph (fork/join), CUDA events on the launching stream; `value` above is "
                                   "the dependent chain on one stream"},
            "gpu_launches": launches_per_step * K,
            "clocks": clk,
            "cpu_baseline": cpu,
            "breakdown": breakdown,
            "points": points,
        }
        s = json.dumps(line)
        print(s, flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                f.write(s + "\n")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_points(args, stream, hbm, tf_peak):
    """Graph-timed, autotuned points of the other workloads (each within the points budget): the 8B gate as the
    Huffman stream alone, the heavy-tailed matrix, the 70B gate and down projections, the 96-matmul 8B stack."""
    import synth
    t_start = time.time()
    m70 = synth.mlp_70b()
    todo = [("gate_8b/huffman", synth.gate_8b(), [1, 4], "huffman"),
            ("heavy_tail", synth.heavy_tail(), [1, 64], "palette"),
            ("gate_70b", m70[0], [1, 32, 256, 512], "palette"),
            ("down_70b", m70[2], [1, 32, 256, 512], "palette"),
            ("stack_8b", None, [1], "palette")]
    out = []
    for cfg, mat, bs, resident in todo:
        if time.time() - t_start > args.points_budget:
            out.append({"config": cfg, "skipped": f"points budget of {args.points_budget:.0f} s spent"})
            continue
        if cfg == "stack_8b":
            out += measure_stack(args.stack_layers, bs, stream, hbm, tf_peak)
        else:
            out += measure_workload(cfg, mat, bs, resident, stream, hbm, tf_peak)
    return out


def run_sweep(args):
    """Every configuration of the workload list at each of its batch sizes, autotuned plan, graph replays over
    enough resident copies that a pass streams from HBM (except the tiny matrix, smaller than L2)."""
    import torch

    import synth
    hbm, tf_peak, _, _ = peaks()
    stream = torch.cuda.Stream()
    m70 = synth.mlp_70b()
    single = [("tiny", synth.tiny(), [1], "palette"), ("gate_8b", synth.gate_8b(), [1, 4, 16], "palette"),
              ("heavy_tail", synth.heavy_tail(), [1, 16, 64], "palette"),
              ("gate_70b", m70[0], [1, 32, 256, 512], "palette"), ("down_70b", m70[2], [1, 32, 256, 512], "palette"),
              ("gate_8b/huffman", synth.gate_8b(), [1, 4, 8], "huffman"),
              ("gate_70b/huffman", m70[0], [1, 8], "huffman"), ("down_70b/huffman", m70[2], [1], "huffman")]
    for cfg, mat, bs, resident in single:
        for d in measure_workload(cfg, mat, bs, resident, stream, hbm, tf_peak):
            print(json.dumps(d), flush=True)
    for d in measure_stack(args.stack_layers, [1, 8, 32, 128], stream, hbm, tf_peak, hard_every=(8, 4, 2)):
        print(json.dumps(d), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
