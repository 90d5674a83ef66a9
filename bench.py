"""Benchmark of the fused dequantise-and-multiply on GB300.

Headline workload (one "step"): the 40 decoder Linears of a whisper-large-v3-turbo-shaped
model (4 layers x {self q,k,v,o; cross q,k,v,o; fc1 1280->5120; fc2 5120->1280}), NF4 with
double-quantised absmax, bf16 activations, one pass at each of M = 1, 4 and 16 rows:
120 fused dequant-matmuls, run as one grouped launch per M (the 40 Linears of the sweep
have independent inputs, so one persistent kernel streams all their weights).  Weights are packed once (load time) and stay resident;
every step reads a different weight copy (9 copies, 487 MB > 3x the 129 MB L2), so each
step streams its weights from HBM.  Metric: algorithmic GB/s (packed weights + scales + x +
y + bias bytes per step / device time).

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

N > 1 runs one process per GPU (torchrun), each an independent replica of the workload
(weak scaling); the time is the max over ranks.  --impl reference times the CPU oracle
(the plain numpy implementation the tests check against) on a bounded sample of the same
workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------- helpers
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), \
        int(os.environ.get("WORLD_SIZE", "1"))


def max_over_ranks(x, world, device=None):
    """The largest value of x over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step, steps, world, t_seconds_max):
    """Whole-job GB/s: every rank processed its own copy of the workload (weak scaling)."""
    return world * bytes_per_rank_step * steps / t_seconds_max / 1e9


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            return json.load(f)
    except Exception:
        return None


def peak_hbm(peaks):
    if peaks:
        for k in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
            if k in peaks and peaks[k]:
                return float(peaks[k]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def peak_tflops(peaks, sustained):
    if peaks:
        keys = ("bf16_tflops_sustained",) if sustained else ("bf16_tflops",)
        for k in keys + ("bf16_tflops",):
            if k in peaks and peaks[k]:
                return float(peaks[k]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload
def nf4_linear_bytes(N, K, M, has_bias):
    w = N * K // 2 + N * K // 64 + 4 * ((N * K // 64 + 255) // 256) + 4
    return w + M * K * 2 + M * N * 2 + (N * 2 if has_bias else 0)


def decoder_workload():
    from bit_weight_quantized_matmul_gb300 import workloads as wl
    return wl.turbo_decoder_sweep(), (1, 4, 16)


def step_bytes(linears, Ms):
    return sum(nf4_linear_bytes(l["N"], l["K"], M, l["bias"]) for M in Ms for l in linears)


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, local_rank, world):
    import torch
    import torch.distributed as dist
    from bit_weight_quantized_matmul_gb300 import build as B
    B.build()
    from bit_weight_quantized_matmul_gb300 import wq
    from bit_weight_quantized_matmul_gb300 import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    linears, Ms = decoder_workload()
    R = 9  # weight copies: 9 x 54 MB > 3 x L2
    # pack once from the seeded generator, then clone to R resident copies
    packed0 = []
    for l in linears:
        W = torch.from_numpy(wl.weight(l["seed"], l["N"], l["K"])).to(dev)
        packed0.append(wq.pack("nf4", W))
        del W
    copies = [packed0] + [[(p.clone(), s.clone()) for p, s in packed0] for _ in range(R - 1)]
    biases = [wl.bias(l["seed"], l["N"]).to(dev) if l["bias"] else None for l in linears]
    # every activation / output of a step lives in one contiguous buffer (views per Linear, each
    # 16-byte aligned), so the end-to-end run moves a step's inputs and results in one copy each way
    def carve(shapes, fill=None):
        sizes = [(m * n + 7) // 8 * 8 for m, n in shapes]
        flat = torch.empty(sum(sizes), dtype=torch.bfloat16, device=dev)
        views, off = [], 0
        for (m, n), sz in zip(shapes, sizes):
            views.append(flat[off:off + m * n].view(m, n))
            off += sz
        return flat, views
    x_flat, x_views = carve([(M, l["K"]) for M in Ms for l in linears])
    y_flat, y_views = carve([(M, l["N"]) for M in Ms for l in linears])
    xs = {M: x_views[j * len(linears):(j + 1) * len(linears)] for j, M in enumerate(Ms)}
    ys = {M: y_views[j * len(linears):(j + 1) * len(linears)] for j, M in enumerate(Ms)}
    for M in Ms:
        for i, l in enumerate(linears):
            xs[M][i].copy_(wl.activations(l["seed"] * 7 + M, M, l["K"]).to(dev))
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)

    def grouped_pass(copy, M):
        probs = [(ys[M][i], xs[M][i], copies[copy][i][0], copies[copy][i][1], l["N"], l["K"], biases[i])
                 for i, l in enumerate(linears)]
        wq.linear_grouped(probs, "nf4", weights_static=True)

    def chained_pass(copy, M):
        for i, l in enumerate(linears):
            p, s = copies[copy][i]
            wq.linear_into(ys[M][i], xs[M][i], p, s, "nf4", l["N"], l["K"], biases[i], weights_static=True)

    # eager warm-up of every path once (sets kernel attributes before capture)
    with torch.cuda.stream(stream):
        for M in Ms:
            grouped_pass(0, M)
            chained_pass(0, M)
    torch.cuda.synchronize()

    def capture(pass_fn):
        gs = []
        for j in range(3):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for mi, M in enumerate(Ms):
                    pass_fn((3 * j + mi) % R, M)
            gs.append(g)
        return gs

    graphs = capture(grouped_pass)
    chained_graphs = capture(chained_pass)
    launches_per_step = len(Ms)
    bytes_per_step = step_bytes(linears, Ms)

    def barrier():
        if world > 1:
            dist.barrier()

    def timed(gs, steps):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for k in range(steps):
                gs[k % 3].replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(ev0.elapsed_time(ev1), world, dev)

    with torch.cuda.stream(stream):
        for w in range(args.warmup):
            graphs[w % 3].replay()
            chained_graphs[w % 3].replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank)
    clocks.start()
    t_ms = timed(graphs, args.steps)
    clk = clocks.stop()
    ms_per_step = t_ms / args.steps
    value = job_throughput(bytes_per_step, args.steps, world, t_ms * 1e-3)  # GB/s, all ranks
    ch_steps = max(3, min(args.steps, 2000))
    t_ch = timed(chained_graphs, ch_steps)
    chained = {"value": round(bytes_per_step * ch_steps / (t_ch * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(t_ch / ch_steps, 5), "steps": ch_steps,
               "what": "same step as 120 dependent single-Linear launches (split-K cluster kernel), "
                       "CUDA graph with programmatic dependent launch"}

    # ---- end to end through the public API: pinned host x in, y out, every step
    xh = x_flat.cpu().pin_memory()
    yh = torch.empty(y_flat.shape, dtype=y_flat.dtype).pin_memory()
    h2d = x_flat.numel() * 2
    d2h = y_flat.numel() * 2
    e2e_steps = max(3, min(args.steps, 200))

    def e2e_step(k):
        with torch.cuda.stream(stream):
            x_flat.copy_(xh, non_blocking=True)
            graphs[k % 3].replay()
            yh.copy_(y_flat, non_blocking=True)
        stream.synchronize()

    for k in range(2):
        e2e_step(k)
    barrier()
    t0 = time.perf_counter()
    for k in range(e2e_steps):
        e2e_step(k)
    t_e2e = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e_value = job_throughput(bytes_per_step, e2e_steps, world, t_e2e)

    peaks = read_peaks()
    pk, pk_src = peak_hbm(peaks)
    achieved = bytes_per_step / (ms_per_step * 1e-3) / 1e9  # per GPU; same kernel throughout the region
    traffic = load_traffic("wq_tcp_kernel", "decoder_nf4")
    out = {
        "metric": "4-bit dequant-linear effective HBM bandwidth, decode (M<=16)",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nf4 weights, bf16 activations, fp32 accumulate",
        "data": "synthetic (seeded counter-based generator; random-init weights of the model's shapes)",
        "config": {"workload": "whisper-large-v3-turbo decoder sweep: 4 layers x 10 NF4 Linears "
                               "(1280x1280 x8, 5120x1280, 1280x5120), M in {1,4,16} -> 120 launches/step",
                   "fmt": "nf4 block 64, double-quant absmax (int8 per 256, fp32 scale)",
                   "l2": "inputs larger than L2: 9 rotated weight copies (487 MB)",
                   "bytes_per_step": bytes_per_step,
                   "launch": "one grouped launch per M (40 independent Linears each), CUDA graph, PDL",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": pk, "unit": "GB/s",
                     "frac": round(achieved / pk, 4), "peak_source": pk_src, "traffic": traffic,
                     "kernel": "wq_tcp_kernel (persistent grouped decode: BN=16, 256-element chunks, "
                               "block scales folded after the MMA)",
                     "algorithmic_bytes_per_launch": round(bytes_per_step / launches_per_step, 1)},
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "note": "per step: one pinned-host -> device copy of all 120 activations, the 3 grouped "
                        "launches, one device -> pinned-host copy of all 120 outputs, synchronised"},
        "chained": chained,
        "gpu_launches": launches_per_step * args.steps,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0 and not args.no_extra:
        out["extra"] = extra_gemm(wq, wl, dev, peaks)
    return out


def load_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, when it matches the current kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d.get(workload, {}).get("dram_bytes_per_launch")
    except Exception:
        return None


def extra_gemm(wq, wl, dev, peaks):
    """Encoder-side context (configs 2 and 3 shapes): the fc1 Linear (N=5120, K=1280) at
    M = 1500 x 4 in NVFP4 W4A16, and in W4A4 (GEMM alone, and with the runtime activation
    quantiser); each measured call is one CUDA graph (the quantiser's kernels and the GEMM
    replay back to back); L2 flushed before every replay; median of 10."""
    import torch
    M, N, K = 6000, 5120, 1280
    W = torch.from_numpy(wl.weight(101, N, K)).to(dev)
    p, s = wq.pack("nvfp4", W)
    x = wl.activations(101, M, K, outlier_frac=0.001).to(dev)
    b = wl.bias(101, N).to(dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    act = (torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
           torch.empty((M, K // 16), dtype=torch.uint8, device=dev),
           torch.empty(1, dtype=torch.float32, device=dev))
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        ts = []
        for _ in range(10):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    t16 = timed(lambda: wq.linear_into(y, x, p, s, "nvfp4", N, K, b))
    wq.quant_act_nvfp4(x, out=act)
    t44 = timed(lambda: wq.linear_into(y, act, p, s, "nvfp4_w4a4", N, K, b))
    t44q = timed(lambda: (wq.quant_act_nvfp4(x, out=act), wq.linear_into(y, act, p, s, "nvfp4_w4a4", N, K, b)))
    fl = 2.0 * M * N * K
    pk, src = peak_tflops(peaks, sustained=False)
    tf = lambda t: round(fl / (t * 1e-3) / 1e12, 1)
    return {"workload": "encoder fc1 (N=5120, K=1280) at M=6000 (4 x 1500 frames), L2 flushed",
            "w4a16_nvfp4": {"value": tf(t16), "unit": "TFLOP/s", "ms": round(t16, 4),
                            "frac_of_bf16_peak": round(tf(t16) / pk, 4)},
            "w4a4_nvfp4_gemm": {"value": tf(t44), "unit": "TFLOP/s", "ms": round(t44, 4),
                                "frac_of_fp4_nominal": round(tf(t44) / (4 * pk), 4)},
            "w4a4_nvfp4_with_act_quant": {"value": tf(t44q), "unit": "TFLOP/s", "ms": round(t44q, 4)},
            "peak": {"bf16": pk, "source": src, "fp4": "4 x bf16 (nominal ratio)"}}


# ---------------------------------------------------------------- encoder workloads
def run_encoder(args, rank, local_rank, world):
    """Configs 2 / 3: the encoder Linear shapes (q/k/v/o 1280x1280, fc1 5120x1280, fc2
    1280x5120) at M = 1500 x B for B in {1, 4, 16}, NVFP4 weights, bf16 activations with 0.1 %
    outliers x20; W4A16, or W4A4 with the runtime activation quantiser inside the step.  One step
    = the 9 GEMMs; each GEMM (with its quantiser, for W4A4) is one CUDA graph replay, timed with
    CUDA events after an L2 flush (excluded)."""
    import torch
    from bit_weight_quantized_matmul_gb300 import build as B
    B.build()
    from bit_weight_quantized_matmul_gb300 import wq
    from bit_weight_quantized_matmul_gb300 import workloads as wl
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w4a4 = args.workload == "encoder_w4a4"
    cases = []
    for si, (name, N, K) in enumerate(wl.encoder_shapes()):
        W = torch.from_numpy(wl.weight(100 + si, N, K)).to(dev)
        p, s = wq.pack("nvfp4", W)
        b = wl.bias(100 + si, N).to(dev)
        for Bw in (1, 4, 16):
            M = 1500 * Bw
            x = wl.activations(100 + si, M, K, outlier_frac=0.001).to(dev)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            act = (torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
                   torch.empty((M, K // 16), dtype=torch.uint8, device=dev),
                   torch.empty(1, dtype=torch.float32, device=dev))
            cases.append(dict(name=name, B=Bw, M=M, N=N, K=K, p=p, s=s, b=b, x=x, y=y, act=act))
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def launch(c):
        if w4a4:
            wq.quant_act_nvfp4(c["x"], out=c["act"])
            wq.linear_into(c["y"], c["act"], c["p"], c["s"], "nvfp4_w4a4", c["N"], c["K"], c["b"])
        else:
            wq.linear_into(c["y"], c["x"], c["p"], c["s"], "nvfp4", c["N"], c["K"], c["b"])

    for _ in range(args.warmup):
        for c in cases:
            launch(c)
    torch.cuda.synchronize()
    for c in cases:
        c["graph"] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(c["graph"]):
            launch(c)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(len(cases) * args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    k = 0
    for _ in range(args.steps):
        for c in cases:
            flush.zero_()
            ev[k][0].record()
            c["graph"].replay()
            ev[k][1].record()
            k += 1
    torch.cuda.synchronize()
    clk = clocks.stop()
    per = [e0.elapsed_time(e1) for e0, e1 in ev]
    t_ms = max_over_ranks(sum(per), world, dev)
    flops_step = sum(2.0 * c["M"] * c["N"] * c["K"] for c in cases)
    value = world * flops_step * args.steps / (t_ms * 1e-3) / 1e12
    peaks = read_peaks()
    pk, src = peak_tflops(peaks, sustained=False)
    by = {}
    for i, c in enumerate(cases):
        ts = sorted(per[j] for j in range(i, len(per), len(cases)))
        by[f"{c['name']}_B{c['B']}"] = round(2.0 * c["M"] * c["N"] * c["K"] / (ts[len(ts) // 2] * 1e-3) / 1e12, 1)
    return {"metric": "4-bit dequant-linear TFLOP/s, encoder (M = 1500 x B)", "value": round(value, 2),
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "nvfp4 weights, " + ("nvfp4 activations" if w4a4 else "bf16 activations"),
            "data": "synthetic (seeded counter-based generator)",
            "config": {"workload": ("W4A4 (activation quantiser in the step)" if w4a4 else "W4A16") +
                                   ": encoder Linears qkvo/fc1/fc2 at M=1500*B, B in {1,4,16} (9 GEMMs/step)",
                       "l2": "flushed (256 MB write) before every launch, outside the timed events",
                       "launch": "one CUDA graph replay per GEMM (W4A4: the quantiser's kernels and the GEMM)"},
            "roofline": {"bound": "tensor", "achieved": round(value / world, 2), "peak": pk * (4 if w4a4 else 1),
                         "unit": "TFLOP/s", "frac": round(value / world / (pk * (4 if w4a4 else 1)), 4),
                         "peak_source": src + (" bf16 x 4 (nominal fp4 ratio)" if w4a4 else ""), "traffic": None},
            "per_gemm_tflops_median": by, "clocks": clk, "gpu_launches": len(per) * (3 if w4a4 else 1)}


# ---------------------------------------------------------------- CPU oracle
_ORACLE_CACHE = {}


def _oracle_inputs():
    """Oracle-packed weights and fp32 inputs of the decoder sweep (built once, not timed)."""
    if "items" not in _ORACLE_CACHE:
        from bit_weight_quantized_matmul_gb300 import workloads as wl
        from oracle import quant as Q
        linears, Ms = decoder_workload()
        items = []
        for l in linears:
            p = Q.nf4_pack(wl.weight(l["seed"], l["N"], l["K"]))
            b = wl.bf16_as_f32(wl.bias(l["seed"], l["N"])) if l["bias"] else None
            for M in Ms:
                x = wl.bf16_as_f32(wl.activations(l["seed"] * 7 + M, M, l["K"]))
                items.append((l, M, p, x, b))
        _ORACLE_CACHE["items"] = items
    return _ORACLE_CACHE["items"]


def cpu_baseline(seconds=15.0):
    """The oracle (numpy NF4 decode + fp64 matmul, as it stands) on a bounded sample of the
    same workload: whole passes over the step's 120 Linear-calls, repeated until ``seconds``
    of CPU work (a partial pass at the end counts the Linears it finished)."""
    from oracle import linear as L
    items = _oracle_inputs()
    done_bytes, t_total, n = 0, 0.0, 0
    while t_total < seconds:
        for l, M, p, x, b in items:
            t0 = time.perf_counter()
            L.linear_w4a16(x, p, b)
            t_total += time.perf_counter() - t0
            done_bytes += nf4_linear_bytes(l["N"], l["K"], M, l["bias"])
            n += 1
            if t_total >= seconds:
                break
    return {"value": round(done_bytes / t_total / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} Linear-calls of the step's 120 (whole passes in order), numpy NF4 decode + "
                      f"fp64 matmul, {t_total:.1f} s of CPU time",
            "threads_note": "numpy elementwise single-threaded; fp64 matmul on the BLAS thread pool"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, on the same config and metric; each step a bounded
    time-sliced sample so that warm-up + steps take about two minutes."""
    if rank != 0:
        return None
    _oracle_inputs()
    per = max(0.2, min(args.ref_step_seconds, 120.0 / (args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(seconds=per)
    t0 = time.perf_counter()
    vals = [cpu_baseline(seconds=per)["value"] for _ in range(args.steps)]
    elapsed = time.perf_counter() - t0
    v = statistics.median(vals)
    return {"impl": "reference", "metric": "4-bit dequant-linear effective HBM bandwidth, decode (M<=16)",
            "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1000 * elapsed / max(1, args.steps), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32 decode, fp64 matmul",
            "data": "synthetic (seeded counter-based generator)",
            "config": {"workload": "whisper-large-v3-turbo decoder sweep: 4 layers x 10 NF4 Linears, "
                                   "M in {1,4,16}; each step a bounded sample of it"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{per:.2f} s of oracle work per step over the step's Linear-calls"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=5.0)
    ap.add_argument("--workload", default="decoder_nf4", choices=["decoder_nf4", "encoder_w4a16", "encoder_w4a4"])
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    out = run_ours(args, rank, local_rank, world) if args.workload == "decoder_nf4" else \
        run_encoder(args, rank, local_rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
