"""Benchmark: fused decompress + matmul on the Llama-3.1-8B-shaped gate_proj W[14336,4096].

One step = one uw_matmul of the autotuned plan (AUTO) at B=1 on a Huffman-coded
matrix loaded with its resident palette form, i.e. one pass of the whole hot
path: strategy lookup, (preprocess if the plan has one), on-chip BF16
reconstruction and the contraction.  Inputs are larger than L2: the step rotates
over several device copies of the compressed matrix (each copy its own uw_matrix),
so every step streams its weights from HBM.  Steps are replayed through CUDA
graphs captured from the same C-ABI calls.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle (the
plain C decoder + fp64 matmul) on the host cores instead.
"""
from __future__ import annotations

import argparse
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
WORKLOAD = "gate_8b"

# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu capture of that kernel as it stands
# (profiles/launches_bench_gate8b_b1.md, profiles/gemv_mma_kernel_gate8b_b4.md). Keyed by (workload, batch,
# kernel name); a kernel change invalidates it.
MEASURED_TRAFFIC = {("gate_8b", 1, "gemv_tma_kernel"): 91.928320e6,
                    ("gate_8b", 4, "gemv_mma_kernel"): 93.158400e6}


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


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--batch", type=int, default=1)
    p.add_argument("--no-breakdown", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-autotune", action="store_true")
    p.add_argument("--json-out", default=None)
    p.add_argument("--workload", default="gate_8b",
                   choices=["gate_8b", "down_8b", "gate_70b", "down_70b", "heavy_tail", "tiny"],
                   help="matrix recipe (the JSON line's headline workload is gate_8b)")
    p.add_argument("--plan", default=None, help="force a plan 'strategy,kernel,split,variant' (skips autotuning)")
    p.add_argument("--sweep", action="store_true",
                   help="time every configuration (tiny, 8B gate, 8B MLP stack, heavy tail, 70B gate/down) at each of "
                        "its batch sizes under the autotuned plan; one JSON line per (configuration, B)")
    p.add_argument("--stack-layers", type=int, default=32, help="layers of the 8B MLP stack in --sweep")
    p.add_argument("--resident", default="palette", choices=["palette", "huffman"],
                   help="what stays resident: the Huffman blob with its palette form (default), or the Huffman blob "
                        "alone (AUTO then decodes the stream inside the GEMV for B <= 8)")
    return p.parse_args()


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
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


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
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

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
        time.sleep(0.3)

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
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for nm, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except Exception:
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


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
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import lossless_bf16_weight_exponent_gb300 as uw
    import oracle
    import synth
    oracle.build()
    mat = synth.gate_8b()
    w = mat.weights()
    blob = oracle.encode(w, oracle.HUFFMAN)
    x = mat.activations(args.batch)
    steps = max(1, min(args.steps, 3))
    warm = min(args.warmup, 1)
    if warm:
        oracle_step_seconds(blob, w.shape, x, warm)
    times = oracle_step_seconds(blob, w.shape, x, steps)
    sec = sum(times) / len(times)
    eff = (2 * mat.N * mat.K + 2 * args.batch * mat.K + 4 * args.batch * mat.N) / sec / 1e9
    line = {
        "impl": "reference", "metric": "effective BF16 weight GB/s, fused decompress+matmul (B=%d)" % args.batch,
        "value": eff, "unit": "GB/s", "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{WORKLOAD} W[14336,4096] bf16 N(0,0.02)+1e-4x100, Huffman blob",
                                         "batch": args.batch},
        "cpu_baseline": {"value": eff, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{steps} full steps: decode of the Huffman blob + fp64 GEMV (B={args.batch})"},
        "e2e": {"value": eff, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def run_ours(args):
    import torch

    import lossless_bf16_weight_exponent_gb300 as uw
    import synth

    rank, world, local = dist_setup()
    dev = torch.cuda.current_device()
    B = args.batch
    mat = workload_matrix(args.workload)
    w = mat.weights()
    blob = uw.encode(w, uw.CODEC_HUFFMAN)
    pal_form = args.resident == "palette"
    base = uw.Matrix(blob, want_palette_form=pal_form)
    info = base.info
    resident = info["device_bytes"]
    copies = max(2, int(np.ceil(3 * L2_BYTES / max(1, resident))))
    mats = [base] + [uw.Matrix(blob, want_palette_form=pal_form) for _ in range(copies - 1)]

    # autotune on one copy (batches of the workload), share the table with the others
    tune_batches = [1, 4, 16] if B in (1, 4, 16) else [B]
    if args.plan:
        vals = [int(v) for v in args.plan.split(",")]
        text = "%d %d %d %d %d 0\n" % (1 << max(0, (B - 1).bit_length()), *vals)
        for m in mats:
            m.tune_load(text)
    elif not args.no_autotune:
        need = base.autotune_workspace_size(tune_batches)
        tws = torch.empty(need, dtype=torch.uint8, device="cuda")
        base.autotune(tune_batches, tws, need)
        del tws
        table = base.tune_save()
        for m in mats[1:]:
            m.tune_load(table)
    plan = base.plan_for(B)
    ws_bytes = max(m.workspace_size(B) for m in mats)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    x = torch.from_numpy(mat.activations(B).view(np.int16)).cuda()
    y = torch.empty((B, mat.N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def step(i, s):
        mats[i % copies].matmul(x, B, y, uw.OUT_F32, uw.STRAT_AUTO, ws, ws_bytes, s)

    # CUDA graphs of G steps each, replayed to reach exactly K steps
    K, W = args.steps, args.warmup
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

    run_steps(max(W, 3))
    if K >= G:
        graph_for(G)          # build every graph the timed region replays before timing starts
    if K % G:
        graph_for(K % G)
    run_steps(min(K, G))
    stream.synchronize()
    clocks = Clocks(gpu_id(dev))
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_steps(K)
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world)
    ms_step = ms_total / K

    hbm_peak, tf_peak, peak_kind = peaks()
    alg = algorithmic_bytes(info, plan.strategy, B)
    eff_bytes = 2 * mat.N * mat.K + 2 * B * mat.K + 4 * B * mat.N
    value = job_throughput(eff_bytes, K, world, ms_total)

    launches_per_step = launches_per_call(plan, B)

    # e2e through the public API with host buffers: H2D of X and D2H of Y inside the timed region
    xh = torch.from_numpy(mat.activations(B).view(np.int16)).pin_memory()
    yh = torch.empty((B, mat.N), dtype=torch.float32).pin_memory()
    hneed = max(m.host_workspace_size(B) for m in mats)
    hws = torch.empty(hneed, dtype=torch.uint8, device="cuda")
    e2e_steps = min(max(K, 10), 2000)
    for i in range(20):
        mats[i % copies].matmul_host(xh, B, yh, uw.OUT_F32, hws, hneed, stream)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        mats[i % copies].matmul_host(xh, B, yh, uw.OUT_F32, hws, hneed, stream)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = job_throughput(eff_bytes, e2e_steps, world, e2e_s * 1e3)

    breakdown = {}
    if not args.no_breakdown and rank == 0 and args.workload == "gate_8b" and pal_form:
        breakdown = strategy_breakdown(mats, mat, info, copies, hbm_peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(blob, w, mat, B)

    if rank == 0:
        achieved = alg / (ms_step * 1e-3) / 1e9
        kname = kernel_name(plan, B)
        traffic = MEASURED_TRAFFIC.get((args.workload, B, kname))
        line = {
            "metric": "effective BF16 weight GB/s, fused decompress+matmul (B=%d)" % B,
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": max(W, 3),
            "ms_per_step": ms_step, "us_per_matmul": ms_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate", "data": "synthetic",
            "config": {"workload": f"{args.workload}: W[{mat.N},{mat.K}] bf16 ({mat.name} recipe), "
                                   + ("Huffman blob + resident palette form" if pal_form else "Huffman blob alone")
                                   + f"; X[{B},{mat.K}] N(0,1)",
                       "batch": B, "plan": plan.as_tuple(), "copies_rotated": copies,
                       "l2": f"inputs larger than L2: {copies} copies x {resident / 1e6:.1f} MB resident",
                       "compression": {"huffman_bits_per_weight": 8 * info["blob_bytes"] / (mat.N * mat.K),
                                       "verbatim_block_fraction": info["n_verbatim"] / info["n_blocks"]}},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic, "peak_kind": peak_kind,
                         "algorithmic_bytes_per_launch": alg, "kernel": kname},
            "effective_frac_of_peak": value / world / hbm_peak,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": 2 * B * mat.K,
                    "d2h_bytes_per_step": 4 * B * mat.N, "us_per_call": e2e_s / e2e_steps * 1e6},
            "gpu_launches": launches_per_step * K,
            "clocks": clk,
            "cpu_baseline": cpu,
            "breakdown": breakdown,
        }
        s = json.dumps(line)
        print(s, flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                f.write(s + "\n")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def strategy_breakdown(mats, mat, info, copies, hbm_peak):
    """Per (B, strategy) timing of single calls rotating the copies (eager launches, L2 not warm)."""
    import torch

    import lossless_bf16_weight_exponent_gb300 as uw
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
            if s == 4 and not mats[0].info["has_palette_form"]:
                continue
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
            alg = algorithmic_bytes(info, s, B)
            row[nm] = {"us": round(us, 2), "eff_GBps": round(eff / us / 1e3, 1),
                       "compressed_GBps": round(alg / us / 1e3, 1), "compressed_frac": round(alg / us / 1e3 / hbm_peak, 3)}
        auto = mats[0].plan_for(B)
        row["auto_plan"] = auto.as_tuple()
        out[f"B={B}"] = row
    return out


def cpu_baseline(blob, w, mat, B):
    x = mat.activations(B)
    times = oracle_step_seconds(blob, w.shape, x, 2)
    sec = sum(times) / len(times)
    eff = (2 * mat.N * mat.K + 2 * B * mat.K + 4 * B * mat.N) / sec / 1e9
    return {"value": eff, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"2 full steps: plain-C decode of the Huffman blob + fp64 GEMV at B={B}"}


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


def run_sweep(args):
    """Every configuration of the workload list at each of its batch sizes, autotuned plan, graph replays over
    enough resident copies that a pass streams from HBM (except the tiny matrix, smaller than L2)."""
    import torch

    import lossless_bf16_weight_exponent_gb300 as uw
    import synth
    hbm, tf_peak, peak_kind = peaks()
    stream = torch.cuda.Stream()
    single = [("tiny", synth.tiny(), [1]), ("gate_8b", synth.gate_8b(), [1, 4, 16]),
              ("heavy_tail", synth.heavy_tail(), [1, 16, 64]),
              ("gate_70b", synth.mlp_70b()[0], [1, 32, 256, 512]), ("down_70b", synth.mlp_70b()[2], [1, 32, 256, 512])]

    def line(cfg, mat_desc, B, us, comp_bytes, eff_bytes, flops, plan, extra=None):
        d = {"config": cfg, "matrix": mat_desc, "B": B, "us": round(us, 2),
             "compressed_GBps": round(comp_bytes / us / 1e3, 1), "compressed_frac": round(comp_bytes / us / 1e3 / hbm, 3),
             "effective_GBps": round(eff_bytes / us / 1e3, 1), "effective_frac": round(eff_bytes / us / 1e3 / hbm, 3),
             "tflops": round(flops / us / 1e6, 1), "tensor_frac": round(flops / us / 1e6 / tf_peak, 3),
             "plan": plan, "peak_kind": peak_kind}
        if extra:
            d.update(extra)
        print(json.dumps(d), flush=True)

    # the same matrices held as the Huffman blob alone (no palette form): the Huffman-fed pipelines
    single += [("gate_8b/huffman", synth.gate_8b(), [1, 4, 8]), ("gate_70b/huffman", synth.mlp_70b()[0], [1, 8]),
               ("down_70b/huffman", synth.mlp_70b()[2], [1])]
    for cfg, mat, bs in single:
        pal_form = not cfg.endswith("/huffman")
        blob = uw.encode(mat.weights(), uw.CODEC_HUFFMAN)
        base = uw.Matrix(blob, want_palette_form=pal_form)
        info = base.info
        copies = 1 if cfg == "tiny" else max(2, int(np.ceil(3 * L2_BYTES / info["device_bytes"])))
        mats = [base] + [uw.Matrix(blob, want_palette_form=pal_form) for _ in range(copies - 1)]
        need = base.autotune_workspace_size(bs)
        tws = torch.empty(need, dtype=torch.uint8, device="cuda")
        base.autotune(bs, tws, need)
        del tws
        table = base.tune_save()
        for m in mats[1:]:
            m.tune_load(table)
        for B in bs:
            ws_bytes = base.workspace_size(B)
            ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
            x = torch.from_numpy(mat.activations(B).view(np.int16)).cuda()
            y = torch.empty((B, mat.N), dtype=torch.float32, device="cuda")
            n = 32 if copies > 1 else 64
            us = time_graph(lambda i, s: mats[i % copies].matmul(x, B, y, uw.OUT_F32, uw.STRAT_AUTO, ws, ws_bytes, s),
                            n, 7, stream) / n
            eff = 2 * mat.N * mat.K + 2 * B * mat.K + 4 * B * mat.N
            line(cfg, f"W[{mat.N},{mat.K}]", B, us, algorithmic_bytes(info, 4 if pal_form else 5, B), eff,
                 2.0 * B * mat.N * mat.K,
                 base.plan_for(B).as_tuple(),
                 {"l2": "matrix smaller than L2" if copies == 1 else f"{copies} copies rotated, inputs larger than L2",
                  "verbatim_block_fraction": round(info["n_verbatim"] / info["n_blocks"], 4)})
        del mats, base
        torch.cuda.empty_cache()

    # 8B MLP stack: gate, up, down per layer, one graph per pass over the whole stack
    L = args.stack_layers
    recipes = synth.stack_8b(L)
    mats, infos, tables = [], [], {}
    for r in recipes:
        blob = uw.encode(r.weights(), uw.CODEC_HUFFMAN)
        m = uw.Matrix(blob, want_palette_form=True)
        mats.append(m)
        infos.append(m.info)
    bs = [1, 8, 32, 128]
    for shape_first in (0, 2):  # autotune the gate shape and the down shape once, share by shape
        m0 = mats[shape_first]
        need = m0.autotune_workspace_size(bs)
        tws = torch.empty(need, dtype=torch.uint8, device="cuda")
        m0.autotune(bs, tws, need)
        del tws
        tables[shape_first] = m0.tune_save()
    for i, m in enumerate(mats):
        m.tune_load(tables[0 if i % 3 != 2 else 2])
    for B in bs:
        ws_bytes = max(m.workspace_size(B) for m in mats[:3])
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        x_in = torch.from_numpy(recipes[0].activations(B).view(np.int16)).cuda()            # [B, 4096]
        x_mid = torch.from_numpy(recipes[2].activations(B).view(np.int16)).cuda()           # [B, 14336]
        y_mid = torch.empty((B, 14336), dtype=torch.float32, device="cuda")
        y_out = torch.empty((B, 4096), dtype=torch.float32, device="cuda")

        def call(i, s):
            m = mats[i]
            if i % 3 == 2:
                m.matmul(x_mid, B, y_out, uw.OUT_F32, uw.STRAT_AUTO, ws, ws_bytes, s)
            else:
                m.matmul(x_in, B, y_mid, uw.OUT_F32, uw.STRAT_AUTO, ws, ws_bytes, s)
        us = time_graph(call, len(mats), 5, stream)
        comp = sum(algorithmic_bytes(inf, 4, B) for inf in infos)
        eff = sum(2 * inf["N"] * inf["K"] + 2 * B * inf["K"] + 4 * B * inf["N"] for inf in infos)
        flops = sum(2.0 * B * inf["N"] * inf["K"] for inf in infos)
        line("stack_8b", f"{L} layers x (gate, up W[14336,4096]; down W[4096,14336])", B, us, comp, eff, flops,
             {"gate_up": mats[0].plan_for(B).as_tuple(), "down": mats[2].plan_for(B).as_tuple()},
             {"matmuls": len(mats), "us_per_matmul": round(us / len(mats), 2)})


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
