"""Benchmark of the fused pre-norm linear layer on GB300.

One step = one fused RMSNorm + linear call over one batch: x [512, 14336]
fp16 with 1 % outlier rows against W [49152, 14336], FP32 statistics and
accumulation (the largest norm + GEMM workload that fits one GPU).  The same
JSON line carries, under "other_configs", the LayerNorm + linear + bias
workload x [8, 128, 8192] against W [8192, 8192] in TFLOP/s and the
decode-sized LayerNorm + linear + bias bf16 workload (K = 8192, N = 28672)
at M = 1, 4 and 16 in HBM GB/s, each timed the same way with its own
roofline and CPU-oracle baseline.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--m M] [--no-cpu-baseline]
                  [--no-other-configs] [--no-alternatives]

--impl reference times the fp64 CPU oracle (the reference arm of this
build) on the host cores, each step a bounded sample of rows of the same
workload.  Under torchrun with N > 1 every rank runs an independent replica
on its own GPU (the layer's rows are independent; no collective on the data
path) and the job value is N x work / max-over-ranks time.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and torch.cuda.synchronize(), timed with CUDA events on the launching
stream.  Inputs rotate over enough independent sets (x, W, bias, y) that the
bytes touched between two uses of one set exceed twice the L2 size, so no
step finds its weights in L2.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

L2_BYTES = 129 * 2 ** 20
DEFAULT_WORKLOAD = "rms_linear_f16_m512_k14336_n49152_outliers"
# Measured in the same run as the default workload, reported under
# "other_configs": (workload, M override).
OTHER_CONFIGS = (("ln_linear_bias_f16_m1024_k8192_n8192", None),
                 ("decode_ln_linear_bias_bf16_k8192_n28672", 1),
                 ("decode_ln_linear_bias_bf16_k8192_n28672", 4),
                 ("decode_ln_linear_bias_bf16_k8192_n28672", 16))
METRIC = "fused LN/RMSNorm+GEMM TFLOP/s (% dense FP16 peak); HBM GB/s at M\u226416"
PROFILES = os.path.join(ROOT, "profiles")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------
# distributed plumbing (replicas)
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier():
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value: float) -> float:
    """Largest `value` over all ranks (the job's time is its slowest rank)."""
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time."""
    return units_per_rank * world / max_seconds


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
class ClockSampler:
    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self) -> dict:
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    p = [c.strip() for c in line.split(",")]
                    if len(p) < 10:
                        continue
                    try:
                        ts = time.mktime(time.strptime(p[1].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                        ts += float("0." + p[1].split(".")[1]) if "." in p[1] else 0.0
                        rows.append(dict(ts=ts, sm=float(p[2]), sm_max=float(p[3]),
                                         power=float(p[4]) if p[4] not in ("[N/A]", "N/A") else None,
                                         hw=p[6], hw_thermal=p[7], sw_thermal=p[8], sw_power=p[9]))
                    except (ValueError, IndexError):
                        continue
        finally:
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if self.t0 - 0.05 <= r["ts"] <= self.t1 + 0.05]
        extended = False
        if len(inside) < 3:
            # The timed region was shorter than a few sampling periods: use
            # the samples nearest to it (the same load ran around it).
            mid = 0.5 * (self.t0 + self.t1)
            inside = sorted(rows, key=lambda r: abs(r["ts"] - mid))[:3]
            extended = True
        reasons = set()
        for r in inside:
            for k, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                            ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[k].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["sm_max"] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside),
                "window_extended": extended}


# ----------------------------------------------------------------------------
LEAD_IN_MS = 3.0


def lead_in(stream):
    """Keep the GPU busy for a few milliseconds before a timed region starts,
    so that the host has queued the first steps by the time the start event
    is reached (otherwise the first step's launch latency on the host is
    timed as GPU time).  The sleep precedes the start event: it is not
    timed."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(LEAD_IN_MS * 1e-3 * 2.1e9))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash() -> str:
    """Hash of the sources of the tile kernel, to tell whether a stored ncu
    traffic figure still describes the kernel that runs."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "normalization_gemm_row_gb300", "csrc")
    for name in ("ngr_gemm_kernel.cuh", "ngr_gemm2_kernel.cuh", "ngr_gemm4_kernel.cuh", "ngr_gemm.cu",
                 "ngr_ptx.cuh", "ngr_internal.h", "ngr_decode.cu", "ngr_rowstats.cu"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    path = os.path.join(PROFILES, f"traffic_{workload}.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_hash") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------
# ----------------------------------------------------------- per-op details
_NORM_IDS = {"none": 0, "layer": 1, "rms": 2}
_ACT_IDS = {"none": 0, "silu": 1, "relu": 2, "gelu": 3}
_TWO_GEMM = ("ffn", "mlp", "mlp_swiglu")


def op_keys(w):
    """Input tensors of workload ``w``'s op, in the generator's key names."""
    return {"ffn": ["x", "W1", "W2"],
            "mlp": ["x", "gamma", "beta", "W1", "b1", "W2", "b2"],
            "swiglu": ["x", "gamma", "beta", "Wg", "Wu"],
            "mlp_swiglu": ["x", "gamma", "beta", "Wg", "Wu", "Wd"],
            "linear_residual_norm": ["x", "W", "bias", "residual", "gamma", "beta"]}.get(
        w.op, ["x", "gamma", "beta", "W", "bias"])


def op_out_cols(w):
    return w.K if w.op in _TWO_GEMM else w.N


def op_kernel_flops(w, decode):
    """FLOPs of each kernel one call launches, in launch order (the
    statistics kernel counts 0): statistics for norm ops and for decode
    calls (which also clear split-K counters), then one GEMM per product
    (SwiGLU's gate and up share one)."""
    g = 2.0 * w.M * w.N * w.K
    has_norm = w.op in ("layernorm_linear", "rmsnorm_linear") or w.norm != "none"
    if w.op == "swiglu":
        return ([0.0] if has_norm else []) + [2 * g]
    if w.op == "linear_residual_norm":
        return ([0.0] if decode else []) + [g, 0.0]
    if w.op == "mlp_swiglu":
        return ([0.0] if has_norm or decode else []) + [2 * g, g]
    if w.op in ("ffn", "mlp"):
        return ([0.0] if has_norm or decode else []) + [g, g]
    return ([0.0] if has_norm or decode else []) + [g]


def oracle_run(w, host, rows, lib):
    """The oracle for the listed rows of workload ``w`` (fp64)."""
    import oracle
    if w.op == "layernorm_linear":
        return oracle.layernorm_linear(host["x"], host["gamma"], host["beta"], host["W"],
                                       host["bias"], w.eps, rows, lib)
    if w.op == "rmsnorm_linear":
        return oracle.rmsnorm_linear(host["x"], host["gamma"], host["W"], host["bias"], w.eps,
                                     rows, lib)
    if w.op == "linear_silu":
        return oracle.linear_silu(host["x"], host["W"], host["bias"], rows, lib)
    if w.op == "ffn":
        return oracle.ffn(host["x"], host["W1"], host["W2"], rows, lib)
    nid = _NORM_IDS[w.norm]
    if w.op == "norm_linear":
        return oracle.norm_linear(nid, _ACT_IDS[w.act], host["x"], host["gamma"], host["beta"],
                                  host["W"], host["bias"], w.eps, rows, lib)
    if w.op == "mlp":
        return oracle.mlp(nid, _ACT_IDS[w.act], host["x"], host["gamma"], host["beta"],
                          host["W1"], host["b1"], host["W2"], host["b2"], w.eps, rows, lib)
    if w.op == "swiglu":
        return oracle.swiglu(nid, host["x"], host["gamma"], host["beta"], host["Wg"],
                             host["Wu"], w.eps, rows, lib)
    if w.op == "linear_residual_norm":
        return oracle.linear_residual_norm(nid, host["x"], host["W"], host["bias"],
                                           host["residual"], host["gamma"], host["beta"], w.eps,
                                           rows, lib)[1]
    return oracle.mlp_swiglu(nid, host["x"], host["gamma"], host["beta"], host["Wg"],
                             host["Wu"], host["Wd"], w.eps, rows, lib)


def our_arm(args, rank, world, local, workload, m_override):
    import normalization_gemm_row_gb300 as ngr
    from normalization_gemm_row_gb300 import binding as B
    from normalization_gemm_row_gb300 import inputs

    ngr.build()
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    w = inputs.BY_NAME[workload]
    if m_override is not None:
        w = w.with_m(m_override)
    M, K, N = w.M, w.K, w.N
    decode = M <= 32
    two_gemm = w.op in _TWO_GEMM

    # Input sets: one seeded draw on the host, copied to every set (identical
    # values, distinct buffers), enough sets that the bytes between two uses
    # of a set exceed 2 x L2.
    host = inputs.make(w)
    keys = [k for k in op_keys(w) if host.get(k) is not None]
    out_cols = op_out_cols(w)
    set_bytes = sum(host[k].numel() * host[k].element_size() for k in keys) + M * out_cols * 2
    n_sets = max(2, min(16, math.ceil(2 * L2_BYTES / set_bytes) + 1))
    op_code = {"layernorm_linear": B.OP_LAYERNORM_LINEAR, "rmsnorm_linear": B.OP_RMSNORM_LINEAR,
               "linear_silu": B.OP_LINEAR_SILU, "ffn": B.OP_FFN, "norm_linear": B.OP_NORM_LINEAR,
               "mlp": B.OP_MLP, "swiglu": B.OP_SWIGLU, "mlp_swiglu": B.OP_MLP_SWIGLU,
               "linear_residual_norm": B.OP_LINEAR_RESIDUAL_NORM}[w.op]
    sets = []
    for _ in range(n_sets):
        s = {k: host[k].to(dev) for k in keys}
        s["y"] = torch.empty((M, out_cols), dtype=w.dtype, device=dev)
        if two_gemm or w.op == "linear_residual_norm":
            s["h"] = torch.empty((M, N), dtype=w.dtype, device=dev)
        nb = B.ngr_workspace_bytes(op_code, M, K, N, 0)
        s["ws"] = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
        sets.append(s)
    nid, aid = _NORM_IDS[w.norm], _ACT_IDS[w.act]

    def step(s, stream=None):
        g = s.get
        if w.op == "layernorm_linear":
            ngr.fused_layernorm_linear(s["x"], s["gamma"], s["beta"], s["W"], g("bias"), w.eps,
                                       out=s["y"], workspace=s["ws"], stream=stream)
        elif w.op == "rmsnorm_linear":
            ngr.fused_rmsnorm_linear(s["x"], s["gamma"], s["W"], g("bias"), w.eps,
                                     out=s["y"], workspace=s["ws"], stream=stream)
        elif w.op == "linear_silu":
            ngr.fused_linear_silu(s["x"], s["W"], g("bias"), out=s["y"], workspace=s["ws"],
                                  stream=stream)
        elif w.op == "ffn":
            ngr.ffn_linear_silu_linear(s["x"], s["W1"], s["W2"], out=s["y"], h=s["h"],
                                       workspace=s["ws"], stream=stream)
        elif w.op == "norm_linear":
            ngr.fused_norm_linear_act(s["x"], s["W"], norm=nid, act=aid, gamma=g("gamma"),
                                      beta=g("beta"), bias=g("bias"), eps=w.eps, out=s["y"],
                                      workspace=s["ws"], stream=stream)
        elif w.op == "mlp":
            ngr.fused_mlp(s["x"], s["W1"], s["W2"], norm=nid, act=aid, gamma=g("gamma"),
                          beta=g("beta"), b1=g("b1"), b2=g("b2"), eps=w.eps, out=s["y"],
                          h=s["h"], workspace=s["ws"], stream=stream)
        elif w.op == "linear_residual_norm":
            ngr.fused_linear_residual_norm(s["x"], s["W"], s["gamma"], norm=nid, beta=g("beta"),
                                           bias=g("bias"), residual=s["residual"], eps=w.eps,
                                           out=s["y"], h=s["h"], workspace=s["ws"],
                                           stream=stream)
        elif w.op == "swiglu":
            ngr.fused_norm_swiglu(s["x"], s["Wg"], s["Wu"], norm=nid, gamma=g("gamma"),
                                  beta=g("beta"), eps=w.eps, out=s["y"], workspace=s["ws"],
                                  stream=stream)
        else:
            ngr.fused_mlp_swiglu(s["x"], s["Wg"], s["Wu"], s["Wd"], norm=nid, gamma=g("gamma"),
                                 beta=g("beta"), eps=w.eps, out=s["y"], h=s["h"],
                                 workspace=s["ws"], stream=stream)

    kernel_flops = op_kernel_flops(w, decode)
    kernels_per_step = len(kernel_flops)
    stream = torch.cuda.current_stream(dev)
    for i in range(args.warmup):
        step(sets[i % n_sets])
    torch.cuda.synchronize(dev)

    # -------------------------------------------------- timed region (value)
    clocks = ClockSampler(local if world > 1 else dev.index)
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    lead_in(stream)
    ev0.record(stream)
    for i in range(args.steps):
        step(sets[i % n_sets])
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark_end()
    barrier()
    clock_info = clocks.stop()
    ms_total = ev0.elapsed_time(ev1)
    ms_total_max = max_over_ranks(ms_total)
    flops = w.flops
    algo_bytes = sum(host[k].numel() * host[k].element_size() for k in keys) + M * out_cols * 2
    if two_gemm:
        algo_bytes += 2 * M * N * 2  # H written once and read once
    if w.op == "linear_residual_norm":
        algo_bytes += 2 * M * N * 2  # h written once and read once
    ms_step = ms_total_max / args.steps
    if decode:
        unit = "GB/s"
        value = job_value(algo_bytes * args.steps / 1e9, world, ms_total_max / 1e3)
    else:
        unit = "TFLOP/s"
        value = job_value(flops * args.steps / 1e12, world, ms_total_max / 1e3)
    metric = METRIC

    # ------------------------- dominant-kernel time (CUDA events per kernel)
    torch.cuda.synchronize(dev)
    B.kernel_timing_start(args.steps)
    for i in range(args.steps):
        step(sets[i % n_sets])
    times = B.kernel_timing_stop()
    assert len(times) == args.steps and all(len(t) == kernels_per_step for t in times), times[:2]
    per_kernel = [statistics.mean(t[j] for t in times) for j in range(kernels_per_step)]
    dom = max(range(kernels_per_step), key=lambda j: per_kernel[j])
    peaks = measured_peaks()
    if decode:
        achieved = algo_bytes / (per_kernel[dom] / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        achieved = kernel_flops[dom] / (per_kernel[dom] / 1e3) / 1e12
        # fp16 and bf16 run at the same dense tensor rate (ratio 1).
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = stored_traffic(w.name if m_override is None else f"{w.name}_m{M}")
    roof["peak_source"] = peaks["source"] + " (burst)"
    roof["kernel_ms"] = per_kernel[dom]
    roof["kernel_ms_all"] = per_kernel

    # ----------------------------------------- end to end from host buffers
    # per-step activations copied in: x, and the residual stream when the op has one
    in_keys = [k for k in ("x", "residual") if k in keys]
    in_host = {k: host[k].pin_memory() for k in in_keys}
    y_host = torch.empty((M, out_cols), dtype=w.dtype).pin_memory()
    for i in range(min(3, args.warmup + 1)):
        s = sets[i % n_sets]
        for k in in_keys:
            s[k].copy_(in_host[k], non_blocking=True)
        step(s)
        y_host.copy_(s["y"], non_blocking=True)
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    lead_in(stream)
    e0.record(stream)
    for i in range(args.steps):
        s = sets[i % n_sets]
        for k in in_keys:
            s[k].copy_(in_host[k], non_blocking=True)
        step(s)
        y_host.copy_(s["y"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_serial_ms = max_over_ranks(e0.elapsed_time(e1))

    # The same steps with the copies of neighbouring steps overlapped, as a
    # serving loop would issue them: host-to-device copies on one stream,
    # the library calls on a second and device-to-host copies on a third,
    # ordered by events (a set's inputs are not overwritten before the call
    # that reads them has run, nor its output before it has been copied).
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    in_done = [torch.cuda.Event() for _ in range(n_sets)]
    comp_done = [torch.cuda.Event() for _ in range(n_sets)]
    out_done = [torch.cuda.Event() for _ in range(n_sets)]
    for ev in comp_done + out_done:
        ev.record(stream)
    torch.cuda.synchronize(dev)

    def pipelined(n):
        for i in range(n):
            j = i % n_sets
            s = sets[j]
            s_in.wait_event(comp_done[j])
            with torch.cuda.stream(s_in):
                for k in in_keys:
                    s[k].copy_(in_host[k], non_blocking=True)
            in_done[j].record(s_in)
            s_comp.wait_event(in_done[j])
            s_comp.wait_event(out_done[j])
            step(s, stream=s_comp)
            comp_done[j].record(s_comp)
            s_out.wait_event(comp_done[j])
            with torch.cuda.stream(s_out):
                y_host.copy_(s["y"], non_blocking=True)
            out_done[j].record(s_out)

    pipelined(min(3, args.warmup + 1))
    torch.cuda.synchronize(dev)
    barrier()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    lead_in(s_in)
    p0.record(s_in)
    pipelined(args.steps)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_comp)
    p1.record(s_in)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = max_over_ranks(p0.elapsed_time(p1))

    def e2e_val(ms):
        if decode:
            return job_value(algo_bytes * args.steps / 1e9, world, ms / 1e3)
        return job_value(flops * args.steps / 1e12, world, ms / 1e3)

    e2e = {"value": e2e_val(e2e_ms), "unit": unit,
           "h2d_bytes_per_step": sum(host[k].numel() * host[k].element_size() for k in in_keys),
           "d2h_bytes_per_step": M * out_cols * 2,
           "overlap": "copies of neighbouring steps overlap the calls (3 streams)",
           "serial_value": e2e_val(e2e_serial_ms),
           "serial_note": "copy in, call, copy out one after the other on one stream"}

    # ---------------- same workload through the inference-mode fold (a7)
    alternatives = {}
    if w.op in ("layernorm_linear", "rmsnorm_linear") and not args.no_alternatives:
        nrm = 1 if w.op == "layernorm_linear" else 2
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        folded = [B.fold_prepare(nrm, s["gamma"], s.get("beta"), s["W"], s.get("bias")) for s in sets]
        p1.record(stream)
        torch.cuda.synchronize(dev)
        prep_ms = p0.elapsed_time(p1) / n_sets

        def fstep(i):
            s = sets[i % n_sets]
            Wf, cb = folded[i % n_sets]
            B.fused_norm_linear_folded(nrm, s["x"], Wf, cb, w.eps, out=s["y"], workspace=s["ws"])

        for i in range(args.warmup):
            fstep(i)
        torch.cuda.synchronize(dev)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        lead_in(stream)
        f0.record(stream)
        for i in range(args.steps):
            fstep(i)
        f1.record(stream)
        torch.cuda.synchronize(dev)
        fms = f0.elapsed_time(f1) / args.steps
        B.kernel_timing_start(args.steps)
        for i in range(args.steps):
            fstep(i)
        ftimes = B.kernel_timing_stop()
        fk = [statistics.mean(t[j] for t in ftimes) for j in range(len(ftimes[0]))]
        fval = (algo_bytes / (fms / 1e3) / 1e9) if decode else (flops / (fms / 1e3) / 1e12)
        alternatives["inference_fold"] = {
            "what": "gamma folded into W once (W' = gamma o W, c = colsum W', b' = beta.W + bias); "
                    "per step: row statistics + one GEMM on raw x, y = rstd acc - rstd mu c + b'",
            "value": fval, "unit": unit, "ms_per_step": fms, "kernel_ms": fk,
            "prepare_ms_once_per_weight": prep_ms,
            "frac": (fval / (peaks["hbm_gbs"] if decode else peaks["bf16_tflops"])),
        }
        del folded
    # ------------- the same steps on one input set (whatever of it L2 holds)
    if not args.no_alternatives:
        for i in range(args.warmup):
            step(sets[0])
        torch.cuda.synchronize(dev)
        w0 = torch.cuda.Event(enable_timing=True)
        w1 = torch.cuda.Event(enable_timing=True)
        lead_in(stream)
        w0.record(stream)
        for i in range(args.steps):
            step(sets[0])
        w1.record(stream)
        torch.cuda.synchronize(dev)
        wms = w0.elapsed_time(w1) / args.steps
        alternatives["same_inputs_every_step"] = {
            "what": "every step on input set 0, so x and W stay in L2 as far as it holds them "
                    "(the headline value rotates sets larger than L2)",
            "value": (algo_bytes / (wms / 1e3) / 1e9) if decode else (flops / (wms / 1e3) / 1e12),
            "unit": unit, "ms_per_step": wms}
    # ---------------- unfused torch pipeline on the same GPU (cuBLAS GEMM)
    if not args.no_alternatives:
        import torch.nn.functional as F

        tacts = {"none": lambda t: t, "silu": F.silu, "relu": F.relu,
                 "gelu": lambda t: F.gelu(t, approximate="none")}

        def tnorm(s):
            if w.norm == "layer":
                return F.layer_norm(s["x"], (K,), s["gamma"], s["beta"], w.eps)
            if w.norm == "rms":
                return F.rms_norm(s["x"], (K,), s["gamma"], w.eps)
            return s["x"]

        def tstep(i):
            s = sets[i % n_sets]
            if w.op == "layernorm_linear":
                return F.linear(F.layer_norm(s["x"], (K,), s["gamma"], s["beta"], w.eps), s["W"], s.get("bias"))
            if w.op == "rmsnorm_linear":
                return F.linear(F.rms_norm(s["x"], (K,), s["gamma"], w.eps), s["W"], s.get("bias"))
            if w.op == "linear_silu":
                return F.silu(F.linear(s["x"], s["W"], s.get("bias")))
            if w.op == "ffn":
                return F.linear(F.silu(F.linear(s["x"], s["W1"])), s["W2"])
            if w.op == "norm_linear":
                return tacts[w.act](F.linear(tnorm(s), s["W"], s.get("bias")))
            if w.op == "mlp":
                return F.linear(tacts[w.act](F.linear(tnorm(s), s["W1"], s.get("b1"))), s["W2"],
                                s.get("b2"))
            if w.op == "linear_residual_norm":
                hh = F.linear(s["x"], s["W"], s.get("bias")) + s["residual"]
                return (F.rms_norm(hh, (N,), s["gamma"], w.eps) if w.norm == "rms"
                        else F.layer_norm(hh, (N,), s["gamma"], s["beta"], w.eps))
            a = tnorm(s)
            h = F.silu(F.linear(a, s["Wg"])) * F.linear(a, s["Wu"])
            return h if w.op == "swiglu" else F.linear(h, s["Wd"])

        for i in range(args.warmup):
            tstep(i)
        torch.cuda.synchronize(dev)

        def twindow():
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            lead_in(stream)
            t0.record(stream)
            for i in range(args.steps):
                tstep(i)
            t1.record(stream)
            torch.cuda.synchronize(dev)
            return t0.elapsed_time(t1) / args.steps

        def owindow():
            o0 = torch.cuda.Event(enable_timing=True)
            o1 = torch.cuda.Event(enable_timing=True)
            lead_in(stream)
            o0.record(stream)
            for i in range(args.steps):
                step(sets[i % n_sets])
            o1.record(stream)
            torch.cuda.synchronize(dev)
            return o0.elapsed_time(o1) / args.steps

        # Three windows of K steps of each, alternating (the side that goes
        # first alternates too), each after a short idle gap, so that both
        # sides see the same clocks and power state; medians.
        tw, ow = [], []
        for i in range(3):
            for side in ((twindow, tw), (owindow, ow))[::1 if i % 2 == 0 else -1]:
                time.sleep(0.2)
                side[1].append(side[0]())
        tms = statistics.median(tw)
        oms = statistics.median(ow)
        alternatives["torch_unfused_same_gpu"] = {
            "what": "the same computation as separate torch ops (layer_norm/rms_norm, linear on "
                    "cuBLAS, activations, the SwiGLU product), intermediates written to HBM",
            "value": (algo_bytes / (tms / 1e3) / 1e9) if decode else (flops / (tms / 1e3) / 1e12),
            "unit": unit, "ms_per_step": tms,
            "ours_in_alternating_windows_ms_per_step": oms}

    out = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if w.dtype == torch.float16 else "bf16",
        "data": "synthetic (seeded; shapes and distributions of the pages' workload)",
        "config": {"workload": w.name, "op": w.op, "M": M, "K": K, "N": N,
                   "bias": w.bias, "eps": w.eps, "global_batch": M * world,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"{n_sets} rotating input sets of {set_bytes / 2**20:.0f} MiB "
                         f"(> 2 x L2 between reuses)",
                   "accumulate": "fp32", "statistics": "fp32"},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": kernels_per_step * args.steps,
        "clocks": clock_info,
        "pct_of_dense_fp16_peak": None if decode else 100.0 * value / world / peaks["bf16_tflops"],
        "alternatives": alternatives,
    }
    return out, w, host


def cpu_baseline(w, host, target_s: float):
    """The fp64 oracle as it stands on the host cores, on a bounded sample
    of rows of the same workload.  Returns the cpu_baseline object."""
    import oracle
    oracle.build()
    lib = oracle.load()
    M = w.M

    def run(rows):
        oracle_run(w, host, rows, lib)

    threads = oracle.num_threads(lib)
    if w.M <= 32:
        # decode: the whole batch (its cost is streaming W once in fp64)
        t = time.perf_counter()
        run(list(range(M)))
        dt = time.perf_counter() - t
        nbytes = (w.N * w.K + M * w.K + M * w.N) * 2
        return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                "sample": f"all {M} rows of {w.name} (fp64), {dt:.1f} s"}
    probe_rows = list(range(min(M, max(4, threads))))
    t = time.perf_counter()
    run(probe_rows)
    per_row = (time.perf_counter() - t) / len(probe_rows)
    n = int(max(len(probe_rows), min(M, target_s / max(per_row, 1e-9))))
    n = max(threads, (n // threads) * threads) if n >= threads else n
    n = min(n, M)
    rows = list(range(n))
    # When the whole batch takes well under the target, time several passes.
    reps = max(1, int(target_s / max(per_row * n, 1e-9))) if n == M else 1
    t = time.perf_counter()
    for _ in range(reps):
        run(rows)
    dt = time.perf_counter() - t
    flops_per_row = w.flops / w.M
    value = flops_per_row * n * reps / dt / 1e12
    what = f"{reps} passes over all {M} rows" if reps > 1 else f"{n} of {M} rows"
    return {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{what} of {w.name} (fp64, all columns), {dt:.1f} s"}


def reference_arm(args, rank):
    """The fp64 CPU oracle timed as the reference arm, on rank 0 only."""
    if rank != 0:
        return None
    import oracle
    from normalization_gemm_row_gb300 import inputs
    oracle.build()
    lib = oracle.load()
    w = inputs.BY_NAME[args.workload]
    if args.m is not None:
        w = w.with_m(args.m)
    host = inputs.make(w)
    threads = oracle.num_threads(lib)
    decode = w.M <= 32
    rows_per_step = max(1, min(w.M, args.ref_rows or threads))

    def step(i):
        r0 = (i * rows_per_step) % w.M
        rows = [(r0 + j) % w.M for j in range(rows_per_step)]
        oracle_run(w, host, rows, lib)

    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t
    if decode:
        # rows_per_step rows of the batch stream all of W once per step
        nbytes = (w.N * w.K + w.M * w.K + w.M * w.N) * 2 * rows_per_step / w.M
        value, unit = nbytes * args.steps / dt / 1e9, "GB/s"
    else:
        flops = w.flops / w.M * rows_per_step * args.steps
        value, unit = flops / dt / 1e12, "TFLOP/s"
    return {
        "impl": "reference",
        "metric": METRIC, "value": value,
        "unit": unit, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": w.name, "op": w.op, "M": w.M, "K": w.K, "N": w.N,
                   "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": f"{rows_per_step} of {w.M} rows per step, fp64"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--m", type=int, default=None, help="override M (decode workload: 1, 4 or 16)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-alternatives", action="store_true",
                    help="skip the inference-fold and unfused-torch comparison runs")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="measure only --workload (default: the default workload plus "
                         "the LayerNorm and decode workloads under other_configs)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-rows", type=int, default=0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_setup(args.gpus)

    if args.impl == "reference":
        out = reference_arm(args, rank)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return 0

    out, w, host = our_arm(args, rank, world, local, args.workload, args.m)
    if rank == 0:
        out["cpu_baseline"] = None if args.no_cpu_baseline else cpu_baseline(w, host, args.cpu_seconds)
    del host
    if args.workload == DEFAULT_WORKLOAD and args.m is None and not args.no_other_configs:
        others = {}
        for name, m in OTHER_CONFIGS:
            gc.collect()
            torch.cuda.empty_cache()
            o, w2, h2 = our_arm(args, rank, world, local, name, m)
            if rank == 0:
                o["cpu_baseline"] = (None if args.no_cpu_baseline
                                     else cpu_baseline(w2, h2, args.cpu_seconds / 3))
            del h2
            for k in ("metric", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                      "vs_baseline", "data"):
                o.pop(k, None)
            others[name if m is None else f"{name}_m{m}"] = o
        out["other_configs"] = others
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
