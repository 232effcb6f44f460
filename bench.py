"""Benchmark of the W4A16 weight-only linear layer on one B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload: the 70B-shaped FFN gate (8192 -> 28672) and down (28672 -> 8192)
projections, G = 128, weights ~ N(0, 0.015) quantised by the library's
packer, activations ~ N(0, 1) in BF16.  One step = one pass of the whole hot
path over one batch: decode (M = 1, the GEMV) on gate and down, then prefill
(M = 2048, the tensor-core GEMM) on gate and down.

`value` is the decode metric: effective weight GB/s of the GEMV at M = 1,
counting packed codes + FP16 scales + 4-bit zeros + x + y bytes.  The
prefill metric (TFLOP/s at M = 2048) is reported beside it under "gemm".
Both are whole-job figures with inputs resident in HBM; "e2e" repeats the
measurement through the same C entry points with pinned host buffers and the
host<->device copies inside the timed region.

Cold L2: each matrix has 3 device copies used in turn, so between two reads
of the same copy at least 244 MB of other weights (L2 = 126 MB) stream by.

`--impl reference` times the CPU oracle (the plain C implementation the tests
compare against) on the host cores: the decode GEMVs in full, the prefill
GEMMs on a sampled set of output rows.  That arm exists for comparison only.
"""
import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

WORKLOAD = "ffn70b"
M_DECODE, M_PREFILL = 1, 2048
G = 128
METRIC = "W4A16 GEMV weight GB/s (% of HBM peak) at M=1; GEMM TFLOP/s at M=2048"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def gemv_bytes(M, N, K, G):
    """Algorithmic bytes of one decode launch: packed codes (K/2 per row),
    one FP16 scale and one 4-bit zero per (row, group), x and y in BF16."""
    return N * K // 2 + N * (K // G) * 2 + N * (K // G) // 2 + M * K * 2 + M * N * 2


def q4k_bytes(M, N, K):
    """Algorithmic bytes of one decode launch on the super-block layout: codes
    (K/2 per row), one 16-byte record per 256 channels, x and y in BF16."""
    return N * K // 2 + N * (K // 256) * 16 + M * K * 2 + M * N * 2


def _ordinal(n):
    """1st, 2nd, 3rd, 4th, ..., 11th, 12th, 13th, 21st, 32nd ..."""
    suffix = "th" if 10 <= n % 100 <= 20 else {1: "st", 2: "nd", 3: "rd"}.get(n % 10, "th")
    return f"{n}{suffix}"


def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def _code_only(text):
    """C++ source without comments and whitespace, so that edits to comments do
    not mark stored counters as stale (string literals hold no comment markers here)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", "", text)


def kernel_hashes():
    """Hashes of the code (comments and whitespace removed) of the kernels whose
    ncu counters are stored in profiles/."""
    out = {}
    for name in ("gemv.cu", "gemm_tc.cu"):
        p = os.path.join(ROOT, "w4a16_weight_only_linear_b300", "csrc", name)
        if os.path.exists(p):
            out[name] = hashlib.sha256(_code_only(open(p).read()).encode()).hexdigest()[:16]
    return out


def stored_traffic(kernel, key):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(key)
    if not d or d.get("source_hash") != kernel_hashes().get(kernel):
        return None
    return d.get("dram_bytes_per_launch")


def max_over_ranks(values, device):
    """Elementwise maximum of a list of floats over all ranks of the process
    group (the list itself when there is no group or a single rank): every
    per-phase time of the job is the slowest rank's."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_gbs(bytes_per_rank_step, steps, ms, world):
    """Whole-job GB/s: the bytes all `world` ranks moved in `steps` steps over
    the slowest rank's time `ms` (milliseconds)."""
    return world * bytes_per_rank_step * steps / (ms * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def retain_pool_memory(dev_index, nbytes=8 << 30):
    """Application policy for stream-ordered scratch: the tensor-core path takes
    its FP16 copy of x from the device's current memory pool, and a pool with
    the default release threshold (0) returns that memory to the driver at every
    synchronisation, so the next call maps it again.  A serving process keeps it:
    here the threshold of the current pool is raised to `nbytes`.  Returns the
    threshold set, or None when the runtime bindings are missing."""
    try:
        from cuda.bindings import driver as cdrv
        from cuda.bindings import runtime as crt
    except ImportError:
        return None
    err, pool = crt.cudaDeviceGetMemPool(dev_index)
    if err != crt.cudaError_t.cudaSuccess:
        return None
    err, = crt.cudaMemPoolSetAttribute(pool, crt.cudaMemPoolAttr.cudaMemPoolAttrReleaseThreshold,
                                       cdrv.cuuint64_t(nbytes))
    return nbytes if err == crt.cudaError_t.cudaSuccess else None


def run_ours(args):
    import w4a16_weight_only_linear_b300 as w4

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    wk = wl.WORKLOADS[WORKLOAD]
    pk = peaks()
    copies = 3
    pool_keep = retain_pool_memory(local)

    # weights: generated once per matrix (seeded), packed on the device; each rank
    # is an independent replica (the layer has no exchange step on one GPU)
    mats = []
    for j, lin in enumerate(wk.linears):
        w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac).to(dev)
        packed = [w4.w4a16_pack(w, G) for _ in range(copies)]
        del w
        mats.append((lin, packed))
    torch.cuda.synchronize()
    gemm_ok = all(w4.w4a16_linear_path(M_PREFILL, lin.N, lin.K, G) == 2 for lin, _ in mats)
    try:
        xt = torch.zeros(M_PREFILL, mats[0][0].K, dtype=torch.bfloat16, device=dev)
        w4.w4a16_linear(xt, *mats[0][1][0], G)
        torch.cuda.synchronize()
        del xt
    except w4.W4A16Error:
        gemm_ok = False

    xs_dec = [wl.activations_bf16(M_DECODE, lin.K, wl.act_seed(wk, j)).to(dev) for j, (lin, _) in enumerate(mats)]
    xs_pre = [wl.activations_bf16(M_PREFILL, lin.K, wl.act_seed(wk, j) + 7).to(dev) for j, (lin, _) in enumerate(mats)]
    ys_dec = [torch.empty(M_DECODE, lin.N, dtype=torch.bfloat16, device=dev) for lin, _ in mats]
    ys_pre = [torch.empty(M_PREFILL, lin.N, dtype=torch.bfloat16, device=dev) for lin, _ in mats]

    # Decode: one CUDA graph per matrix holding `steps` back-to-back GEMV
    # launches cycling the device copies (a launch is ~20-50 us, so host launch
    # gaps would otherwise show).  Prefill: eager launches (each ~1 ms; the call
    # also converts x to FP16 in stream-ordered scratch).  A step is one launch
    # per (phase, matrix), so the per-(phase, matrix) times add up to the step
    # time, and each time / steps is that call's mean duration on the GPU.
    phases = [("dec", xs_dec, ys_dec)] + ([("pre", xs_pre, ys_pre)] if gemm_ok else [])

    def launch(phase, j, i, stream):
        _, xs, ys = next(ph for ph in phases if ph[0] == phase)
        lin, packed = mats[j]
        w4.w4a16_linear(xs[j], *packed[i % copies], G, out=ys[j], stream=stream)

    for i in range(args.warmup):                       # eager warm-up steps
        for ph, _, _ in phases:
            for j in range(len(mats)):
                launch(ph, j, i, torch.cuda.current_stream())
    torch.cuda.synchronize()
    graphs = {}
    cap_stream = torch.cuda.Stream()
    for j in range(len(mats)):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap_stream):
            for i in range(args.steps):
                launch("dec", j, i, torch.cuda.current_stream())
        graphs[("dec", j)] = gr
    for gr in graphs.values():                          # one untimed replay each
        gr.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    stream = torch.cuda.current_stream()
    keys = [("dec", j) for j in range(len(mats))] + ([("pre", j) for j in range(len(mats))] if gemm_ok else [])
    evs = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for k in keys}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        # The sampler's start leaves the GPU idle for a few hundred ms.  One untimed replay of
        # the first decode graph, enqueued right before the start event, puts the first timed
        # launch behind running work, as every later one is (in a decode step the layer
        # always follows another kernel); the timed region itself holds exactly `steps` steps.
        graphs[keys[0]].replay()
        t0.record(stream)
        for k in keys:
            evs[k][0].record(stream)
            if k[0] == "dec":
                graphs[k].replay()
            else:
                for i in range(args.steps):
                    launch("pre", k[1], i, stream)
            evs[k][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    # every time below is the slowest rank's
    dec_ms = [evs[("dec", j)][0].elapsed_time(evs[("dec", j)][1]) for j in range(len(mats))]
    pre_ms = [evs[("pre", j)][0].elapsed_time(evs[("pre", j)][1]) for j in range(len(mats))] if gemm_ok else []
    times = max_over_ranks([t0.elapsed_time(t1)] + dec_ms + pre_ms, dev)
    total_ms, dec_ms, pre_ms = times[0], times[1:1 + len(mats)], (times[1 + len(mats):] if gemm_ok else None)
    if world > 1:
        torch.distributed.barrier()
    dec_bytes = [gemv_bytes(M_DECODE, lin.N, lin.K, G) for lin, _ in mats]
    dec_gbs = job_gbs(sum(dec_bytes), args.steps, sum(dec_ms), world)
    out = {
        "metric": METRIC, "value": round(dec_gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "ffn70b: 70B-shaped FFN gate 8192->28672 and down 28672->8192, G=128, "
                               "decode M=1 (GEMV) + prefill M=2048 (tcgen05 GEMM), weights N(0,0.015), x N(0,1)",
                   "M_decode": M_DECODE, "M_prefill": M_PREFILL if gemm_ok else None, "G": G,
                   "l2": f"inputs larger than L2: {copies} rotating device copies of each 122 MB packed matrix",
                   "timing": "decode: CUDA-graph replay of `steps` launches per matrix; prefill: `steps` eager calls per matrix; CUDA events on the launch stream",
                   "scratch_pool": ("device's current memory pool, release threshold "
                                    f"{pool_keep >> 30} GiB set by the application" if pool_keep else
                                    "device's current memory pool, default release threshold"),
                   "parallelism": f"replicas x{world}"},
    }
    # roofline, per kernel, from the CUDA-event durations inside the timed region
    gemv_launch_ms = sum(dec_ms) / (len(mats) * args.steps)
    gemv_bytes_per_launch = sum(dec_bytes) / len(mats)
    gemv_ach = gemv_bytes_per_launch / (gemv_launch_ms * 1e-3) / 1e9
    roof_gemv = {"kernel": "gemv (M=1, mean of gate and down launches)", "bound": "hbm",
                 "achieved": round(gemv_ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                 "frac": round(gemv_ach / pk["hbm_gbs"], 4), "peak_source": pk["source"],
                 "traffic": stored_traffic("gemv.cu", "gemv_ffn70b_M1"),
                 "algorithmic_bytes_per_launch": gemv_bytes_per_launch,
                 "launch_us": round(gemv_launch_ms * 1e3, 3),
                 "per_matrix_gbs": {lin.name: round(b / (ms / args.steps * 1e-3) / 1e9, 1)
                                    for (lin, _), b, ms in zip(mats, dec_bytes, dec_ms)}}
    out["roofline"] = roof_gemv
    launches = len(mats) * args.steps
    if gemm_ok:
        flops = [gemm_flops(M_PREFILL, lin.N, lin.K) for lin, _ in mats]
        tflops = world * sum(flops) * args.steps / (sum(pre_ms) * 1e-3) / 1e12
        gemm_launch_ms = sum(pre_ms) / (len(mats) * args.steps)
        ach = (sum(flops) / len(mats)) / (gemm_launch_ms * 1e-3) / 1e12
        roof_gemm = {"kernel": "prefill call = x->FP16 conversion + tcgen05 GEMM (M=2048, mean of gate and down)",
                     "bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(ach / pk["bf16_tflops"], 4),
                     "frac_of_sustained_peak": round(ach / pk["bf16_tflops_sustained"], 4),
                     "peak_source": pk["source"],
                     "peak_kind": "burst (dense BF16 GEMM timed alone); FP16 kind::f16 runs at the same rate",
                     "traffic": stored_traffic("gemm_tc.cu", "gemm_ffn70b_M2048"),
                     "algorithmic_flops_per_launch": sum(flops) / len(mats),
                     "launch_us": round(gemm_launch_ms * 1e3, 3),
                     "per_matrix_tflops": {lin.name: round(f / (ms / args.steps * 1e-3) / 1e12, 1)
                                           for (lin, _), f, ms in zip(mats, flops, pre_ms)}}
        out["gemm"] = {"value": round(tflops, 1), "unit": "TFLOP/s", "roofline": roof_gemm}
        launches += 2 * len(mats) * args.steps          # x -> FP16 conversion + GEMM per call
        # the dominant kernel by time is the prefill GEMM
        out["roofline_gemv"] = roof_gemv
        out["roofline"] = roof_gemm
    else:
        out["gemm"] = {"value": None, "unit": "TFLOP/s", "note": "tensor-core GEMM not available for this shape"}
    out["gpu_launches"] = launches
    out["clocks"] = clk.summary()
    out["e2e"] = e2e_ours(w4, mats, dev, args, gemm_ok)
    if rank == 0:
        out["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def e2e_ours(w4, mats, dev, args, gemm_ok):
    """Same metric through the C entry points, host buffers: every step copies
    x from pinned host memory, runs the layer and reads y back to the host."""
    wk = wl.WORKLOADS[WORKLOAD]
    # the step's inputs (x of every matrix) travel in one host->device copy and its
    # outputs in one device->host copy; the layer calls take views of those buffers
    xs = [wl.activations_bf16(M_DECODE, lin.K, wl.act_seed(wk, j)) for j, (lin, _) in enumerate(mats)]
    hx_all = torch.cat([x.reshape(-1) for x in xs]).pin_memory()
    hy_all = torch.empty(sum(M_DECODE * lin.N for lin, _ in mats), dtype=torch.bfloat16).pin_memory()
    dx_all = torch.empty_like(hx_all, device=dev)
    dy_all = torch.empty_like(hy_all, device=dev)
    dx, dy, ox, oy = [], [], 0, 0
    for lin, _ in mats:             # every view starts on a 16-byte boundary (K, N multiples of 8)
        dx.append(dx_all[ox:ox + M_DECODE * lin.K].view(M_DECODE, lin.K))
        dy.append(dy_all[oy:oy + M_DECODE * lin.N].view(M_DECODE, lin.N))
        ox += M_DECODE * lin.K
        oy += M_DECODE * lin.N
    stream = torch.cuda.current_stream()
    steps = max(args.steps, 200)            # ~15 ms of steps: a few host hiccups do not dominate
    ncopy = len(mats[0][1])

    def run(n):
        for i in range(n):
            dx_all.copy_(hx_all, non_blocking=True)
            for j, (lin, packed) in enumerate(mats):
                w4.w4a16_linear(dx[j], *packed[i % ncopy], G, out=dy[j], stream=stream)
            hy_all.copy_(dy_all, non_blocking=True)
        torch.cuda.synchronize()

    run(50)                                 # the host path (binding, caches, launch) warmed up
    # garbage left by the set-up and the device-timed region would otherwise be scanned by
    # the collector's runs during the loop (the collector stays on while it runs)
    gc.collect()
    t = time.perf_counter()
    run(steps)
    dt_ms = max_over_ranks([(time.perf_counter() - t) * 1e3], dev)[0]      # the slowest rank's
    world = int(os.environ.get("WORLD_SIZE", "1"))
    byts = sum(gemv_bytes(M_DECODE, lin.N, lin.K, G) for lin, _ in mats)
    return {"value": round(job_gbs(byts, steps, dt_ms, world), 1), "unit": "GB/s",
            "h2d_bytes_per_step": hx_all.numel() * 2,
            "d2h_bytes_per_step": hy_all.numel() * 2,
            "scope": "decode GEMVs (M=1) of the step, host wall clock, pinned buffers: one copy of the step's "
                     "inputs in, eager layer calls, one copy of its outputs back"}


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline and the reference arm)
# ---------------------------------------------------------------------------

def _oracle_setup():
    import oracle
    wk = wl.WORKLOADS[WORKLOAD]
    mats = []
    for j, lin in enumerate(wk.linears):
        w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac)
        mats.append((lin, oracle.pack(wl.bits_u16(w), G)))
    xs = [wl.bits_u16(wl.activations_bf16(M_DECODE, lin.K, wl.act_seed(wk, j))) for j, (lin, _) in enumerate(mats)]
    return oracle, mats, xs


def _oracle_decode_pass(oracle, mats, xs):
    for (lin, (q, s, z)), x in zip(mats, xs):
        oracle.linear(x, q, s, z, lin.N, lin.K, G)


def cpu_baseline(args, budget_s=10.0):
    oracle, mats, xs = _oracle_setup()
    threads = oracle.max_threads()
    byts = sum(gemv_bytes(M_DECODE, lin.N, lin.K, G) for lin, _ in mats)
    n, t0 = 0, time.perf_counter()
    while True:
        _oracle_decode_pass(oracle, mats, xs)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(byts * n / dt / 1e9, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full decode passes (M=1 gate and down GEMVs, FP64 oracle) in {dt:.1f} s"}


REF_ROW_FRACTION = 32   # the reference arm's step: every 32nd output row of each matrix


def _oracle_sampled_pass(oracle, mats, xs):
    for (lin, (q, s, z)), x in zip(mats, xs):
        ns = np.arange(0, lin.N, REF_ROW_FRACTION, dtype=np.int64)
        oracle.linear_sampled(x, q, s, z, lin.K, G, np.zeros_like(ns), ns)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle, mats, xs = _oracle_setup()
    threads = oracle.max_threads()
    byts = sum(gemv_bytes(M_DECODE, lin.N // REF_ROW_FRACTION, lin.K, G) for lin, _ in mats)
    for _ in range(args.warmup):
        _oracle_sampled_pass(oracle, mats, xs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_sampled_pass(oracle, mats, xs)
    dt = time.perf_counter() - t0
    v = byts * args.steps / dt / 1e9
    out = {"metric": METRIC, "value": round(v, 3), "unit": "GB/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference",
           "config": {"workload": "ffn70b decode: gate 8192->28672 and down 28672->8192, G=128, M=1",
                      "M_decode": M_DECODE, "G": G, "parallelism": "host cores"},
           "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
                            "sample": f"{args.steps} steps, each the M=1 gate and down GEMVs on every "
                                      f"{_ordinal(REF_ROW_FRACTION)} output row (FP64 oracle)"},
           "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_profile(args):
    """Small case for ncu captures: by default one packed 70B gate matrix
    (8192 -> 28672, ~122 MB of packed weights, above L2), `warmup` + 2 calls of
    one phase, no timing and no CPU leg.  `--workload W` profiles matrix
    `--matrix` of another workload at `--m` activation rows (default: 1 for
    decode, the workload's largest M for prefill) and group size `--g` (default:
    the workload's first); the dual workload runs its paired call.  Weights are
    packed into enough rotating copies that more than 2x L2 streams between two
    uses of a copy, so the captured call reads cold weights."""
    import w4a16_weight_only_linear_b300 as w4
    q4k = args.format == "q4k"
    if q4k and args.profile != "decode":
        raise SystemExit("--format q4k profiles the decode kernel only")
    name = "ffn70b_q4k" if q4k else (args.workload or WORKLOAD)
    wk = wl.WORKLOADS[name]
    j = int(args.matrix)
    lin = wk.linears[j]
    Gv = 32 if q4k else (args.g or (G if name == WORKLOAD else wk.Gs[0]))
    if args.m:
        M = args.m
    elif name == WORKLOAD or q4k:
        M = M_DECODE if args.profile == "decode" else M_PREFILL
    else:
        M = 1 if args.profile == "decode" else max(wk.Ms)
    mats = [j, 1 - j] if wk.dual else [j]
    one = sum(q4k_bytes(1, wk.linears[i].N, wk.linears[i].K) if q4k else
              gemv_bytes(1, wk.linears[i].N, wk.linears[i].K, Gv) for i in mats)
    copies = max(1, -(-2 * 126 * 2 ** 20 // one) + 1)
    packs = []
    for i in mats:
        li = wk.linears[i]
        w = wl.weight_f16(li.N, li.K, wk.sigma, wl.matrix_seed(wk, i), wk.outlier_frac).cuda()
        packs.append([w4.q4k_pack(w) if q4k else w4.w4a16_pack(w, Gv) for _ in range(copies)])
        del w
    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j)).cuda()
    ys = [torch.empty(M, wk.linears[i].N, dtype=torch.bfloat16, device="cuda") for i in mats]
    calls = args.warmup + 2
    for c in range(calls):
        pk = [p[c % copies] for p in packs]
        if q4k:
            w4.q4k_linear(x, *pk[0], out=ys[0])
        elif wk.dual:
            w4.w4a16_linear_dual(x, pk[0], pk[1], Gv, out=(ys[0], ys[1]))
        else:
            w4.w4a16_linear(x, *pk[0], Gv, out=ys[0])
    torch.cuda.synchronize()
    assert w4.w4a16_device_status() == 0
    print(json.dumps({"profile": args.profile, "workload": name, "format": args.format,
                      "matrix": "+".join(wk.linears[i].name for i in mats), "M": M, "N": lin.N, "K": lin.K,
                      "G": Gv, "calls": calls, "weight_copies": copies}))


# ---------------------------------------------------------------------------
# per-config sweep (the other workloads; not the bench line)
# ---------------------------------------------------------------------------

def _graph_us(launch, n, replays=5):
    """Median over `replays` of the per-launch time of a CUDA graph holding `n`
    launches (launch(i, stream) issues launch i); one untimed replay first."""
    torch.cuda.synchronize()
    for i in range(3):                                  # eager warm-up
        launch(i, torch.cuda.current_stream())
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.graph(gr, stream=cap):
        for i in range(n):
            launch(i, torch.cuda.current_stream())
    gr.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gr.replay()                                     # untimed: the timed launches follow running work
        e0.record(stream)
        gr.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / n)
    del gr
    return statistics.median(ts)


def _eager_us(launch, n, replays=5):
    """Median over `replays` of the per-launch time of `n` back-to-back eager launches."""
    stream = torch.cuda.current_stream()
    for i in range(3):
        launch(i, stream)
    torch.cuda.synchronize()
    ts = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            launch(i, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / n)
    return statistics.median(ts)


def run_sweep(args):
    """Decode and small-batch timings of every workload in workloads.py other
    than the bench's own: one JSON line per (workload, matrix, M, G, path) and
    a crossover summary per G for the batch sweep.  Each figure is the median
    of 5 replays of a CUDA graph of `steps` back-to-back launches over enough
    rotating weight copies that more than 2x L2 streams between two reads of a
    copy.  The tensor-core path is timed as back-to-back eager calls (it takes
    its scratch from the stream-ordered pool on every call, whose release
    threshold is raised as in the bench line)."""
    import w4a16_weight_only_linear_b300 as w4
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    retain_pool_memory(0)
    pk = peaks()
    n = args.steps
    l2_bytes = 126 * 2 ** 20

    def packed_copies(wk, j, lin, Gv):
        w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac).to(dev)
        one = gemv_bytes(1, lin.N, lin.K, Gv)
        copies = max(2, -(-2 * l2_bytes // one) + 1)
        out = [w4.w4a16_pack(w, Gv) for _ in range(copies)]
        del w
        return out

    def emit(rec):
        print(json.dumps(rec), flush=True)
        return rec

    def record(wk, lin, M, Gv, path, us, nmat=1, extra_bytes=0):
        byts = nmat * gemv_bytes(M, lin.N, lin.K, Gv) - (nmat - 1) * M * lin.K * 2 + extra_bytes   # x read once
        fl = nmat * gemm_flops(M, lin.N, lin.K)
        return emit({"sweep": wk.name, "matrix": lin.name if nmat == 1 else ("gate+up" if nmat == 2 else "q+k+v"),
                     "M": M, "N": lin.N,
                     "K": lin.K, "G": Gv, "path": path, "us": round(us, 2),
                     "gbs": round(byts / (us * 1e-6) / 1e9, 1), "frac_hbm": round(byts / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                     "tflops": round(fl / (us * 1e-6) / 1e12, 2),
                     "frac_tensor": round(fl / (us * 1e-6) / 1e12 / pk["bf16_tflops"], 4)})

    results = []
    names = ("single_4096", "layer13b_decode", "up13b_sweep", "gateup13b_dual", "ffn13b_awq", "up13b_w8",
             "ffn70b_q4k")
    if args.only:
        names = tuple(nm for nm in names if nm in args.only.split(","))
    for name in names:
        wk = wl.WORKLOADS[name]
        if wk.q4k:
            # the super-block layout (decode kernel only), beside the 4-bit G = 32 layer of the
            # same weights, and the gate projection paired with a second matrix of its shape
            def q4k_rec(lin, M, path, us, nmat=1):
                byts = nmat * q4k_bytes(M, lin.N, lin.K) - (nmat - 1) * M * lin.K * 2
                return emit({"sweep": wk.name, "matrix": lin.name if nmat == 1 else ("gate+up" if nmat == 2 else "q+k+v"),
                     "M": M, "N": lin.N,
                             "K": lin.K, "G": 32, "path": path, "us": round(us, 2),
                             "gbs": round(byts / (us * 1e-6) / 1e9, 1),
                             "frac_hbm": round(byts / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4)})
            dual = []
            for j, lin in enumerate(wk.linears):
                w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac).to(dev)
                copies = max(2, -(-2 * l2_bytes // q4k_bytes(1, lin.N, lin.K)) + 1)
                cps = [w4.q4k_pack(w) for _ in range(copies)]
                g32 = [w4.w4a16_pack(w, 32) for _ in range(copies)]
                del w
                for M in wk.Ms:
                    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j)).to(dev)
                    y = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
                    us = _graph_us(lambda i, s: w4.q4k_linear(x, *cps[i % copies], out=y, stream=s), n)
                    results.append(q4k_rec(lin, M, "q4k gemv", us))
                    if w4.w4a16_linear_path(M, lin.N, lin.K, 32) == 1:      # where the 4-bit GEMV takes it
                        us = _graph_us(lambda i, s: w4.w4a16_linear_gemv(x, *g32[i % copies], 32, out=y, stream=s), n)
                        results.append(record(wk, lin, M, 32, "w4 g32 gemv", us))
                del g32
                if j == 0:
                    dual.append(cps)
                    w2 = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, 2), wk.outlier_frac).to(dev)
                    dual.append([w4.q4k_pack(w2) for _ in range(copies)])
                    del w2
                    for M in wk.Ms:
                        x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j)).to(dev)
                        yg = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
                        yu = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
                        us = _graph_us(lambda i, s: w4.q4k_linear_dual(x, dual[0][i % copies], dual[1][i % copies],
                                                                       out=(yg, yu), stream=s), n)
                        results.append(q4k_rec(lin, M, "q4k dual", us, nmat=2))
                    dual = []
                del cps
            continue
        if wk.bits == 8:
            # the 8-bit variant in both storages: the word layout (four codes per word, one scale
            # and one 8-bit zero per group; bytes = codes + scales + 8-bit zeros + x + y) and the
            # two planes of a 2K-channel 4-bit layer (bytes = what the kernels read: both planes'
            # scales and 4-bit zeros, x once, y)
            for j, lin in enumerate(wk.linears):
                for Gv in wk.Gs:
                    w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac).to(dev)
                    word_bytes = (lin.N * lin.K + lin.N * (lin.K // Gv) * 3)          # codes, scales, zeros
                    ncp = max(2, -(-2 * l2_bytes // word_bytes) + 1)
                    cps_w = [w4.w8a16_pack(w, Gv) for _ in range(ncp)]
                    cps_p = [w4.w8a16_planes_pack(w, Gv) for _ in range(ncp)]
                    del w
                    for M in wk.Ms:
                        x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j)).to(dev)
                        y = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
                        for store, cps, fn, byts, graph in (
                                ("word", cps_w, w4.w8a16_linear, word_bytes + M * lin.K * 2 + M * lin.N * 2,
                                 M <= 8 and Gv <= 128),
                                ("planes", cps_p, w4.w8a16_planes_linear,
                                 gemv_bytes(M, lin.N, 2 * lin.K, Gv) - M * lin.K * 2,
                                 w4.w4a16_linear_path(M, lin.N, 2 * lin.K, Gv) == 1)):
                            f = (lambda cps, fn: lambda i, s: fn(x, *cps[i % len(cps)], Gv, out=y, stream=s))(cps, fn)
                            us = _graph_us(f, n) if graph else _eager_us(f, n)
                            results.append(emit({"sweep": wk.name, "matrix": lin.name, "M": M, "N": lin.N,
                                                 "K": lin.K, "G": Gv,
                                                 "path": f"w8 {store} " + ("gemv" if graph else "gemm (eager)"),
                                                 "us": round(us, 2), "gbs": round(byts / (us * 1e-6) / 1e9, 1),
                                                 "frac_hbm": round(byts / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                                                 "tflops": round(gemm_flops(M, lin.N, lin.K) / (us * 1e-6) / 1e12, 2),
                                                 "frac_tensor": round(gemm_flops(M, lin.N, lin.K) / (us * 1e-6) / 1e12
                                                                      / pk["bf16_tflops"], 4)}))
                    del cps_w, cps_p
            continue
        if wk.act_scaled:
            # activation scale fused into x staging (the x_scale vector counts as bytes read);
            # the tensor-core path allocates stream-ordered scratch, so M > 8 is timed eagerly
            for j, lin in enumerate(wk.linears):
                for Gv in wk.Gs:
                    xsc = wl.act_scale_f32(lin.K, wl.matrix_seed(wk, j) + 70).to(dev)
                    w = wl.awq_weight_f16(wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j),
                                                        wk.outlier_frac), xsc.cpu()).to(dev)
                    one = gemv_bytes(1, lin.N, lin.K, Gv)
                    cps = [w4.w4a16_pack(w, Gv) for _ in range(max(2, -(-2 * l2_bytes // one) + 1))]
                    del w
                    for M in wk.Ms:
                        x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j)).to(dev)
                        y = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
                        fn = lambda i, s: w4.w4a16_linear_act_scaled(x, xsc, *cps[i % len(cps)], Gv, out=y,
                                                                     stream=s)
                        graph = w4.w4a16_linear_path(M, lin.N, lin.K, Gv) == 1
                        us = _graph_us(fn, n) if graph else _eager_us(fn, n)
                        results.append(record(wk, lin, M, Gv, "gemv+scale" if graph else "gemm+scale (eager)", us,
                                              extra_bytes=lin.K * 4))
                    del cps
            continue
        if wk.dual:
            for Gv in wk.Gs:
                gate = packed_copies(wk, 0, wk.linears[0], Gv)
                up = packed_copies(wk, 1, wk.linears[1], Gv)
                nc = min(len(gate), len(up))
                for M in wk.Ms:
                    lin = wk.linears[0]
                    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, 0)).to(dev)
                    yg = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
                    yu = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
                    us = _graph_us(lambda i, s: w4.w4a16_linear_dual(x, gate[i % nc], up[i % nc], Gv, out=(yg, yu),
                                                                      stream=s), n)
                    results.append(record(wk, lin, M, Gv, "dual", us, nmat=2))
                del gate, up
            continue
        for j, lin in enumerate(wk.linears):
            for Gv in wk.Gs:
                cps = packed_copies(wk, j, lin, Gv)
                for M in wk.Ms:
                    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j)).to(dev)
                    y = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
                    paths = []
                    if w4.w4a16_linear_path(M, lin.N, lin.K, Gv) == 1 or M <= 16:
                        paths.append(("gemv", w4.w4a16_linear_gemv))
                    if name == "up13b_sweep":
                        paths.append(("gemm", w4.w4a16_linear_gemm))
                    for pname, fn in paths:
                        # the tensor-core call allocates its x copy and split workspace stream-ordered,
                        # so it is timed as back-to-back eager calls
                        timer = _eager_us if pname == "gemm" else _graph_us
                        try:
                            us = timer(lambda i, s: fn(x, *cps[i % len(cps)], Gv, out=y, stream=s), n)
                        except w4.W4A16Error:
                            continue
                        results.append(record(wk, lin, M, Gv, pname, us))
                del cps
        if name == "layer13b_decode":
            # the attention projections q, k and v share x: one launch over the three matrices
            lins = wk.linears[:3]
            Gv = wk.Gs[0]
            cps3 = [packed_copies(wk, j, lin, Gv) for j, lin in enumerate(lins)]
            nc = min(len(c) for c in cps3)
            for M in wk.Ms:
                x = wl.activations_bf16(M, lins[0].K, wl.act_seed(wk, 0)).to(dev)
                ys = [torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev) for lin in lins]
                us = _graph_us(lambda i, s: w4.w4a16_linear_multi(x, [c[i % nc] for c in cps3], Gv, out=ys,
                                                                  stream=s), n)
                rec = record(wk, lins[0], M, Gv, "multi (q,k,v)", us, nmat=3)
                results.append(rec)
            del cps3
    assert w4.w4a16_device_status() == 0

    # crossover on the batch sweep, per G: the smallest M at which the tensor-core path is
    # faster than the GEMV, and M* = the smallest M whose best achieved FLOP/s reaches 50 % of
    # the tensor peak, or where the GEMV's weight GB/s drops below 90 % of its M = 1 value,
    # whichever comes first
    cross = {}
    sw = [r for r in results if r["sweep"] == "up13b_sweep"]
    for Gv in sorted({r["G"] for r in sw}):
        rs = [r for r in sw if r["G"] == Gv]
        Ms = sorted({r["M"] for r in rs})
        t = {(r["M"], r["path"]): r for r in rs}
        faster = next((M for M in Ms if (M, "gemm") in t and ((M, "gemv") not in t or
                                                               t[(M, "gemm")]["us"] < t[(M, "gemv")]["us"])), None)
        gv1 = t.get((1, "gemv"), {}).get("gbs")
        drop = next((M for M in Ms if (M, "gemv") in t and gv1 and t[(M, "gemv")]["gbs"] < 0.9 * gv1), None)
        # "50 % of the tensor roofline" read as half the dense tensor peak (the HBM-bound roofline
        # of a small M is met by the GEMV at M = 1 already)
        reach = None
        for M in Ms:
            best = min((t[(M, pth)] for pth in ("gemv", "gemm") if (M, pth) in t), key=lambda r: r["us"])
            if best["tflops"] >= 0.5 * pk["bf16_tflops"]:
                reach = M
                break
        rule = min([m for m in (reach, drop) if m is not None], default=None)
        cross[str(Gv)] = {"gemm_faster_from_M": faster, "gemv_below_90pct_from_M": drop, "M_star": rule,
                          "dispatch_gemv_up_to_M": max([M for M in Ms if w4.w4a16_linear_path(M, 13824, 5120, Gv) == 1],
                                                       default=None)}
    emit({"crossover": cross, "note": "pages: 16 to 32"})


def run_oracle_table(args):
    """The CPU oracle timed on this machine's host cores for every configuration
    (a reported baseline, never a target): for each (workload, matrix, M) one
    seeded problem, timed at 1 thread and at all threads on a bounded sample of
    output rows (and, for M = 2048, a 64-row activation subset), each figure
    extrapolated to the full launch by the work it covers.  One JSON line per
    point: GB/s for decode rows (the GEMV's algorithmic bytes), GFLOP/s for the
    prefill rows."""
    import oracle
    threads_all = oracle.max_threads()
    points = [("single_4096", 0, 1, 128), ("layer13b_decode", 0, 1, 128), ("layer13b_decode", 4, 1, 128),
              ("layer13b_decode", 6, 1, 128)]
    points += [("up13b_sweep", 0, M, 128) for M in (1, 2, 4, 8, 16, 32)]
    points += [("gateup13b_dual", 0, M, 128) for M in (1, 4)]
    points += [("ffn70b", j, M, 128) for j in (0, 1) for M in (1, 2048)]
    for name, j, M, Gv in points:
        wk = wl.WORKLOADS[name]
        lin = wk.linears[j]
        w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac)
        q, s_, z = oracle.pack(wl.bits_u16(w), Gv)
        del w
        Ms = min(M, 64)                                   # activation rows actually computed
        x = wl.bits_u16(wl.activations_bf16(Ms, lin.K, wl.act_seed(wk, j)))
        nmat = 2 if wk.dual else 1
        rec = {"oracle_table": name, "matrix": lin.name if nmat == 1 else "gate+up (2 GEMVs)", "M": M,
               "N": lin.N, "K": lin.K, "G": Gv}
        for label, nthreads, target in (("1_thread", 1, 1.0e8), ("all_threads", threads_all, 4.0e8)):
            stride = max(1, int(Ms * lin.N * lin.K / target))
            ns = np.arange(0, lin.N, stride, dtype=np.int64)
            ms = np.repeat(np.arange(Ms, dtype=np.int64), ns.size)
            nn = np.tile(ns, Ms)
            oracle.linear_sampled(x, q, s_, z, lin.K, Gv, ms[:64], nn[:64], nthreads)      # warm
            t0 = time.perf_counter()
            oracle.linear_sampled(x, q, s_, z, lin.K, Gv, ms, nn, nthreads)
            dt = time.perf_counter() - t0
            frac = (ms.size / (M * lin.N))                # share of the launch's outputs computed
            full_s = nmat * dt / frac
            if M > 16:
                rec[label] = {"gflops": round(nmat * gemm_flops(M, lin.N, lin.K) / full_s / 1e9, 3),
                              "s_per_launch": round(full_s, 3), "threads": nthreads,
                              "sample": f"{ms.size} outputs ({Ms} rows x every {_ordinal(stride)} column)"}
            else:
                byts = nmat * gemv_bytes(M, lin.N, lin.K, Gv) - (nmat - 1) * M * lin.K * 2
                rec[label] = {"gbs": round(byts / full_s / 1e9, 4), "s_per_launch": round(full_s, 4),
                              "threads": nthreads, "sample": f"{ms.size} outputs (every {_ordinal(stride)} column)"}
        oracle.linear_sampled(x, q, s_, z, lin.K, Gv, ms[:1], nn[:1], threads_all)       # back to all threads
        rec["extrapolated"] = True
        print(json.dumps(rec), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", choices=["decode", "prefill"], default=None,
                    help="small case for ncu: one matrix, warmup + 2 calls of one phase")
    ap.add_argument("--matrix", default="0", help="with --profile: the workload's matrix index (70B: 0 = gate, 1 = down)")
    ap.add_argument("--workload", default="", help="with --profile: a workloads.py workload other than the bench's")
    ap.add_argument("--m", type=int, default=0, help="with --profile: activation rows")
    ap.add_argument("--g", type=int, default=0, help="with --profile: group size")
    ap.add_argument("--format", choices=["w4", "q4k"], default="w4",
                    help="with --profile decode: the 4-bit group layout or the super-block layout")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep", action="store_true",
                    help="time the other workloads (decode layers, batch x group sweep, dual) instead")
    ap.add_argument("--only", default="", help="with --sweep: comma-separated workload names to time")
    ap.add_argument("--oracle-table", action="store_true",
                    help="time the CPU oracle at 1 thread and all threads for every configuration")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.oracle_table:
        run_oracle_table(args)
    elif args.profile:
        run_profile(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
