"""Benchmark of the attention forward on GB300: prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one attention forward (every step of the method: tiling, online
softmax, both contractions, epilogue) over the workload's whole batch.  The
default workload is the pages' benchmark shape (B=1, H=8, Nq=4096, Nkv=8192,
D=128, non-causal, bf16).  The metric is TFLOPS = 4*B*Hq*Nq*Nkv*D (halved
when causal) / time.

Timing: inputs resident in HBM; L2 is flushed (a 512 MiB write) before every
timed step, outside the step's CUDA-event pair, since the inputs are smaller
than L2; events are recorded on the stream the kernel is launched on; the
timed loop is bracketed by a barrier and a device synchronisation; the slowest
rank's time counts.  With N>1 (torchrun) every rank runs its own replica of
the workload (the method partitions by batch and head, with no exchange), so
``value`` is the work of all ranks over the slowest rank's time (weak
scaling).

``--impl reference`` times the CPU oracle (float64, host cores) on bounded
samples of the same workload: one 128-row query tile per step.

The line's ``sdpa`` object times torch's scaled_dot_product_attention
(cuDNN, flash and memory-efficient backends, each alone) on the same inputs
and in the same way, for comparison (``--no-sdpa`` skips it).  Its
``configs`` object times each of the five workloads the metric is specified
on (tiny, the pages' shape, causal D64, causal GQA, long causal with large
logits) in this process with the same steps, warm-up and L2 flush
(``--no-configs`` skips it); ``value`` stays the chosen workload's.  With
the configs, a head-dim-128 workload also gets ``low_precision``: the same
shape with Q and K in e4m3 (per-tensor descales) and in MXFP8 (a ue8m0
scale per 32 elements), timed the same way.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_io_aware_fa2_gb300.workloads import (HEADLINE, WORKLOADS,  # noqa
                                                make_inputs, quantize_e4m3,
                                                quantize_mxfp8)

METRIC = ("attention fwd TFLOPS (4·B·H·Nq·Nkv·D, "
          "causal ½) and % of GB300 BF16 peak")
UNIT = "TFLOPS"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-sdpa", action="store_true",
                    help="skip the torch SDPA comparison column")
    ap.add_argument("--sdpa-steps", type=int, default=None,
                    help="steps of each SDPA backend (default: --steps)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the five specification workloads")
    ap.add_argument("--schedule", default="auto",
                    choices=["auto", "plain", "stream"],
                    help="force the library's schedule (fa_set_schedule) for "
                         "every call of the run; auto: the planner's choice")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, device="cpu"):
    """Largest value of ``x`` over all ranks of the default process group
    (``x`` itself without one).  NCCL needs ``device`` to be the rank's GPU;
    gloo works on the CPU."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or \
            dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank, ms_slowest, world_size):
    """Whole-job throughput: every rank's work over the slowest rank's time
    (each rank runs its own replica of the workload: weak scaling)."""
    return world_size * flops_per_rank / (ms_slowest * 1e-3) / 1e12


def hbm_peak():
    """Measured copy bandwidth (GB/s) from MEASURED_PEAKS.json, or None."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f).get("hbm_gbs", 0.0)) or None
    return None


# The pages' own figures, on other hardware: context, not targets.
PAGES_CONTEXT = {
    "rtx5090_tflops_b1_h8_q4096_kv8192_bf16": [186.7, 203.6],
    "rtx5090_sol_tflops": 209.5,
    "thunderkittens_h100_tensor_util_claimed": 0.95,
    "note": "figures the pages print for other GPUs (RTX 5090, H100)",
}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "MEASURED_PEAKS.json bf16_tflops (burst)"
    return FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s bf16"


# Device-code headers of each attention kernel (host-side changes in the API
# file leave recorded counters valid).
KERNEL_SOURCES = {
    "fa_fwd_kernel": ("fa_fwd_kernel.cuh", "sm103_ptx.cuh"),
    "fa_fwd_persist_kernel": ("fa_fwd_persist.cuh", "fa_fwd_kernel.cuh",
                              "sm103_ptx.cuh"),
    "fa_fwd_stream_kernel": ("fa_fwd_stream.cuh", "fa_fwd_kernel.cuh",
                             "sm103_ptx.cuh"),
    "fa_fwd_wide_kernel": ("fa_fwd_wide.cuh", "fa_fwd_kernel.cuh",
                           "sm103_ptx.cuh"),
    "fa_fwd_mx_kernel": ("fa_fwd_mx.cuh", "fa_fwd_wide.cuh",
                         "fa_fwd_kernel.cuh", "sm103_ptx.cuh"),
}


def kernel_for(w):
    """The attention kernel that runs a workload on this device: head dims
    192 and 256 (and split causal shapes at 64) take the one-tile kernel,
    the stream and persistent schedules and MXFP8 inputs have kernels of
    their own, the rest run the two-tile kernel."""
    from exact_io_aware_fa2_gb300 import fa
    if w.mx:
        return "fa_fwd_mx_kernel"
    sch = fa.schedule(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D, w.causal)
    if sch["kind"] == "stream":
        return "fa_fwd_stream_kernel"
    if sch["kind"] == "persist":
        return "fa_fwd_persist_kernel"
    if w.D in (192, 256) or (w.D == 64 and w.causal):
        return "fa_fwd_wide_kernel"
    return "fa_fwd_kernel"


def kernel_source_hash(kernel="fa_fwd_kernel"):
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[kernel]):
        p = os.path.join(ROOT, "exact_io_aware_fa2_gb300", "csrc", name)
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(w):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources of the workload's kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(w.name)
    if not e or e.get("kernel_src_sha") != kernel_source_hash(kernel_for(w)):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True,
                             timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def cpu_baseline(w, q, k, v, seconds):
    """The oracle as it stands, on this host's cores, over (batch, head)
    slices of the workload (repeating the workload if it is short) until
    about ``seconds`` of CPU work (at least one slice)."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    group = w.Hq // w.Hkv
    slices = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    t0 = time.perf_counter()
    done = 0
    while True:
        b, h = slices[done % len(slices)]
        hk = h // group
        oracle.attention_fp64(q[b:b + 1, h:h + 1], k[b:b + 1, hk:hk + 1],
                              v[b:b + 1, hk:hk + 1], w.scale, w.causal)
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    flops = w.flops / len(slices) * done
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cores,
            "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"{done} (batch, head) slices of {w.name} "
                      f"({len(slices)} per workload), float64, {dt:.1f} s"}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    q, k, v = make_inputs(w)
    group = w.Hq // w.Hkv
    n_tiles = (w.Nq + 127) // 128
    units = [(b, h, t) for b in range(w.B) for h in range(w.Hq)
             for t in range(n_tiles)]

    def step(i):
        b, h, t = units[i % len(units)]
        rows = list(range(t * 128, min(w.Nq, t * 128 + 128)))
        oracle.attention_rows_fp64(q, k, v, w.scale, w.causal, b, h, rows)
        kv = min(w.Nkv, rows[-1] + 1) if w.causal else w.Nkv
        # flops of this tile, counted like the metric (causal: visible half)
        vis = sum(min(r + 1, w.Nkv) for r in rows) if w.causal else \
            len(rows) * kv
        return 4.0 * vis * w.D

    for i in range(args.warmup):
        step(i)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += step(args.warmup + i)
    dt = time.perf_counter() - t0
    val = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **w.as_dict(),
                   "sample": "one 128-row query tile per step"},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores,
                         "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": "one 128-row query tile of the workload "
                                   "per step, float64"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


SDPA_BACKENDS = ("CUDNN_ATTENTION", "FLASH_ATTENTION", "EFFICIENT_ATTENTION")


def sdpa_column(w, q, k, v, o_ours, flush, stream, steps, warmup=5):
    """torch's scaled_dot_product_attention on the same resident inputs, one
    backend at a time, timed exactly like our kernel (time_steps: the same
    step and warm-up counts, L2 flushed before each step, CUDA events on the
    launching stream).  A comparison, not part of the
    path.  Grouped-query shapes use SDPA's own GQA support; a backend that
    lacks it gets K/V expanded to every query head beforehand (untimed),
    which the entry notes.  Returns {backend: {...}} with TFLOPS and the
    largest |O_sdpa - O_ours|, or the reason a backend did not run."""
    from torch.nn.attention import SDPBackend, sdpa_kernel
    import torch.nn.functional as F
    out = {}
    for name in SDPA_BACKENDS:
        backend = getattr(SDPBackend, name)
        entry = {}
        try:
            kk, vv, gqa = k, v, w.Hq != w.Hkv
            with sdpa_kernel([backend]):
                def step():
                    return F.scaled_dot_product_attention(
                        q, kk, vv, is_causal=w.causal, scale=w.scale,
                        enable_gqa=gqa)
                try:
                    res = step()
                except RuntimeError:
                    if not gqa:
                        raise
                    g = w.Hq // w.Hkv
                    kk = k.repeat_interleave(g, dim=1)
                    vv = v.repeat_interleave(g, dim=1)
                    gqa = False
                    entry["note"] = "K/V expanded to Hq heads (untimed)"
                    res = step()
                starts, ends = time_steps(step, flush, stream, steps,
                                          warmup, torch.cuda.synchronize)
                torch.cuda.synchronize()
            per = [a.elapsed_time(b) for a, b in zip(starts, ends)]
            ms = sum(per) / steps
            entry.update({
                "value": w.flops / (ms * 1e-3) / 1e12, "unit": UNIT,
                "ms_per_step": ms, "ms_per_step_median":
                    statistics.median(per), "steps": steps,
                "max_abs_diff_vs_ours":
                    float((res.float() - o_ours.float()).abs().max())})
        except Exception as exc:  # a backend this GPU/torch cannot run
            entry = {"unavailable": f"{type(exc).__name__}: "
                                    f"{str(exc).splitlines()[0][:160]}"}
        if (w.qk8 or w.mx) and "unavailable" not in entry:
            entry["note"] = (entry.get("note", "") +
                             " bf16 Q/K/V: torch SDPA takes no e4m3 inputs"
                             ).strip()
        out[name.lower()] = entry
    return out


# The five workloads the metric is specified on (tiny, the pages' shape,
# causal D64, causal GQA, long causal with large logits), each timed in the
# bench process the same way as the headline and reported in ``configs``.
SPEC_WORKLOADS = ("tiny_128_d64", "pages_b1_h8_q4096_kv8192_d128",
                  "causal_b4_h16_n2048_d64",
                  "causal_gqa_b2_hq32_hkv8_n8192_d128",
                  "causal_b1_h16_n32768_d128_large_logits")


def time_steps(launch, flush, stream, steps, warmup, barrier):
    """CUDA-event pairs around each of ``steps`` calls of ``launch``, after
    ``warmup`` (at least 3) untimed ones and a barrier.  L2 is flushed (a
    512 MiB write) before every call, outside its event pair; events are
    recorded on the launching stream.  Before the first timed call a few
    flushes are queued, so the host runs ahead of the GPU and no step's
    events include host launch time.  Returns (starts, ends); the caller
    synchronises (barrier) after."""
    for i in range(max(3, warmup)):
        flush.fill_(float(i))
        launch()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier()
    for i in range(4):
        flush.fill_(float(-i))
    for i in range(steps):
        flush.fill_(float(i))                        # evict L2 (untimed)
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    return starts, ends


def spec_configs(args, fa, flush, stream, dev, headline):
    """Every workload of SPEC_WORKLOADS timed like the headline (same steps,
    warm-up, L2 flush and events) in this process: TFLOPS from the mean
    step, the median step, and the fraction of the bf16 peak."""
    peak, _ = peaks()
    out = {}
    for name in SPEC_WORKLOADS:
        w = WORKLOADS[name]
        q, k, v = (t.to(dev) for t in make_inputs(w))
        o = torch.empty_like(q)
        lse = torch.empty(w.B, w.Hq, w.Nq, dtype=torch.float32, device=dev)

        def launch():
            fa.fwd(q, k, v, scale=w.scale, causal=w.causal, out=o, lse=lse)

        def sync():
            torch.cuda.synchronize(dev)
        starts, ends = time_steps(launch, flush, stream, args.steps,
                                  args.warmup, sync)
        sync()
        if fa.last_device_error() != 0:
            raise RuntimeError(f"bounded-wait timeout timing {name}")
        per = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        mean, med = sum(per) / len(per), statistics.median(per)
        tf = w.flops / (mean * 1e-3) / 1e12
        out[name] = {
            "value": tf, "unit": UNIT, "ms_per_step": mean,
            "ms_per_step_median": med,
            "value_at_median": w.flops / (med * 1e-3) / 1e12,
            "frac": tf / peak, "steps": args.steps,
            "kernel": kernel_for(w),
            "schedule": fa.schedule(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D,
                                    w.causal),
            "headline": name == headline.name}
        del q, k, v, o, lse
    return out


def low_precision_column(args, fa, w, q_h, k_h, v, o_bf16, lse_bf16, flush,
                         stream, dev):
    """The same workload with Q and K in 8 bits, timed like the headline:
    e4m3 with one descale per tensor (fa_fwd_qk8) and MXFP8, e4m3 with a
    ue8m0 scale per 32 elements (fa_fwd_mxfp8).  TFLOPS from the mean step,
    the fraction of the peak for half the flops at the e4m3 rate (4/3 of the
    bf16 peak) and of the bf16 peak, and the largest difference from the
    bf16 path's O and LSE on these inputs (the inputs' quantisation, not a
    parity measure: parity of both paths is against the oracle on the
    dequantised inputs)."""
    peak, _ = peaks()
    o = torch.empty_like(o_bf16)
    lse = torch.empty_like(lse_bf16)
    (q8e, qd), (k8e, kd) = quantize_e4m3(q_h), quantize_e4m3(k_h)
    q8e, k8e = q8e.to(dev), k8e.to(dev)
    (q8m, qs), (k8m, ks) = quantize_mxfp8(q_h), quantize_mxfp8(k_h)
    q8m, k8m, qs, ks = (t.to(dev) for t in (q8m, k8m, qs, ks))
    # the e4m3 path runs the schedule the planner gives the shape (two-tile
    # or stream kernel in their QK8 form)
    k_qk8 = kernel_for(w) if kernel_for(w) in ("fa_fwd_kernel",
                                               "fa_fwd_stream_kernel") \
        else "fa_fwd_kernel"
    runs = {
        "qk8": (f"{k_qk8} (QK8)", lambda: fa.fwd_qk8(
            q8e, k8e, v, scale=w.scale, q_descale=qd, k_descale=kd,
            causal=w.causal, out=o, lse=lse)),
        "mxfp8": ("fa_fwd_mx_kernel", lambda: fa.fwd_mxfp8(
            q8m, k8m, v, qs, ks, scale=w.scale, causal=w.causal, out=o,
            lse=lse)),
    }
    out = {}
    for name, (kernel, launch) in runs.items():
        def sync():
            torch.cuda.synchronize(dev)
        starts, ends = time_steps(launch, flush, stream, args.steps,
                                  args.warmup, sync)
        sync()
        if fa.last_device_error() != 0:
            raise RuntimeError(f"bounded-wait timeout timing {name}")
        per = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        mean = sum(per) / len(per)
        tf = w.flops / (mean * 1e-3) / 1e12
        out[name] = {
            "workload": w.name, "value": tf, "unit": UNIT,
            "ms_per_step": mean, "ms_per_step_median": statistics.median(per),
            "frac_of_e4m3_qk_peak": tf / (peak * 4.0 / 3.0),
            "frac_of_bf16_peak": tf / peak, "steps": args.steps,
            "kernel": kernel,
            "max_abs_diff_o_vs_bf16_path":
                float((o.float() - o_bf16.float()).abs().max()),
            "max_abs_diff_lse_vs_bf16_path":
                float((lse - lse_bf16).abs().max())}
    return out


def run_ours(args, w):
    from exact_io_aware_fa2_gb300 import fa
    fa.set_schedule(args.schedule)
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    q_h, k_h, v_h = make_inputs(w)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.Nq, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if w.qk8:
        # e4m3 Q and K with per-tensor descales (the fa_fwd_qk8 path)
        (q8_h, qd), (k8_h, kd) = quantize_e4m3(q_h), quantize_e4m3(k_h)
        q8, k8 = q8_h.to(dev), k8_h.to(dev)
    if w.mx:
        # MXFP8 Q and K: e4m3 with a ue8m0 scale per 32 elements
        (q8_h, qs_h), (k8_h, ks_h) = quantize_mxfp8(q_h), quantize_mxfp8(k_h)
        q8, k8, qs, ks = (t.to(dev) for t in (q8_h, k8_h, qs_h, ks_h))

    def launch():
        if w.qk8:
            fa.fwd_qk8(q8, k8, v, scale=w.scale, q_descale=qd, k_descale=kd,
                       causal=w.causal, out=o, lse=lse)
        elif w.mx:
            fa.fwd_mxfp8(q8, k8, v, qs, ks, scale=w.scale, causal=w.causal,
                         out=o, lse=lse)
        else:
            fa.fwd(q, k, v, scale=w.scale, causal=w.causal, out=o, lse=lse)

    launch()
    torch.cuda.synchronize(dev)
    if fa.last_device_error() != 0:
        raise RuntimeError("bounded-wait timeout in the first call")

    smi_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(dev.index))
                    .split(",")[dev.index]) if os.environ.get(
        "CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else dev.index
    with ClockSampler(smi_index) as clk:
        # the sampler starts first; the warm-up steps run after its start-up
        time.sleep(0.3)
        barrier()
        wall0 = time.perf_counter()
        starts, ends = time_steps(launch, flush, stream, args.steps,
                                  args.warmup, barrier)
        barrier()
        wall = time.perf_counter() - wall0
        if fa.last_device_error() != 0:
            raise RuntimeError("bounded-wait timeout during the timed loop")
        per = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
        configs = None
        lowp = None
        if ws == 1 and not args.no_configs:
            configs = spec_configs(args, fa, flush, stream, dev, w)
            if not (w.qk8 or w.mx) and w.D == 128:
                launch()
                lowp = low_precision_column(args, fa, w, q_h, k_h, v, o,
                                            lse, flush, stream, dev)
    ms = sum(per) / len(per)
    ms_max = max_over_ranks(ms, dev)
    value = job_tflops(w.flops, ms_max, ws)
    per_launch_tflops = w.flops / (ms * 1e-3) / 1e12
    peak, peak_src = peaks()
    # DRAM bytes of one launch (ncu, committed) over its measured time
    traffic = recorded_traffic(w)
    hbm_gbs = traffic / (ms * 1e-3) / 1e9 if traffic else None
    hbm_frac = (hbm_gbs / hbm_peak()) if hbm_gbs and hbm_peak() else None
    peak_src += ", of measured" if "MEASURED" in peak_src else ", of fallback"
    if w.qk8 or w.mx:
        # Half the flops (Q K^T) run as e4m3 products at twice the bf16 rate
        # (the nominal 4.5 vs 2.25 PFLOP/s), half (P V) at the bf16 rate:
        # the step's peak is 2 / (1/(2P) + 1/P) = 4P/3.
        peak *= 4.0 / 3.0
        peak_src += "; x4/3: QK^T at the e4m3 rate (2x bf16), PV at bf16"
    # A split-KV step is the forward kernel plus the merge; the step time
    # (both kernels) then stands for the forward kernel's, a lower bound.
    if w.mx:
        # fa_fwd_mxfp8 runs one 128-row query tile per CTA, never split
        sched = {"kind": "one_tile", "ctas": w.B * w.Hq * -(-w.Nq // 128),
                 "pieces": 1, "blocks_per_cta": 0}
    else:
        sched = fa.schedule(w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.D, w.causal)
    split = sched["kind"] == "split_kv"
    launches_per_step = 2 if split else 1

    # ---- end to end through the public API with host buffers ----
    if w.qk8 or w.mx:
        host_in = (q8_h, k8_h, v_h) + ((qs_h, ks_h) if w.mx else ())
        pinned = [t.pin_memory() for t in host_in]
        dev_in = [torch.empty_like(t, device=dev) for t in host_in]
        o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

        def e2e_step():
            for d_, h_ in zip(dev_in, pinned):
                d_.copy_(h_, non_blocking=True)
            if w.mx:
                fa.fwd_mxfp8(*dev_in, scale=w.scale, causal=w.causal, out=o,
                             lse=lse)
            else:
                fa.fwd_qk8(dev_in[0], dev_in[1], dev_in[2], scale=w.scale,
                           q_descale=qd, k_descale=kd, causal=w.causal,
                           out=o, lse=lse)
            o_h.copy_(o, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()
    else:
        host_in = (q_h, k_h, v_h)
        qp, kp, vp = (t.pin_memory() for t in host_in)
        bufs = fa.host_buffers(qp, kp, vp, device=dev)

        def e2e_step():
            fa.fwd_host(qp, kp, vp, scale=w.scale, causal=w.causal,
                        bufs=bufs)
    for _ in range(3):
        e2e_step()
    e2e_steps = max(5, min(args.steps, 50))
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    barrier()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()

    sdpa = None
    if ws == 1 and not args.no_sdpa:
        sdpa = sdpa_column(w, q, k, v, o, flush, stream,
                           args.sdpa_steps or args.steps, args.warmup)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, q_h, k_h, v_h, args.cpu_seconds)

    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    dev_name = torch.cuda.get_device_name(dev)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 QK^T, bf16 PV" if w.qk8 else
                 "mxfp8 QK^T (e4m3, ue8m0 per 32), bf16 PV" if w.mx else "bf16",
        "data": "synthetic",
        "pct_of_peak": 100.0 * per_launch_tflops / peak,
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                   "Nq": w.Nq, "Nkv": w.Nkv, "D": w.D, "causal": w.causal,
                   "scale": w.scale, "seed": 0, "global_batch": w.B * ws,
                   "parallelism": f"replicas{ws}" if ws > 1 else "single",
                   "l2": "flushed (512 MiB write) before every timed step",
                   "device": dev_name},
        "roofline": {"bound": "tensor", "achieved": per_launch_tflops,
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": per_launch_tflops / peak,
                     "peak_source": peak_src,
                     "traffic": traffic,
                     "hbm_gbs_achieved": hbm_gbs,
                     "hbm_frac_of_measured_copy": hbm_frac,
                     "kernel": f"{kernel_for(w)}<SPLIT> + fa_merge_kernel"
                     if split else kernel_for(w),
                     "schedule": sched,
                     "algorithmic_flops_per_launch": w.flops},
        "cpu_baseline": cpu,
        "pages_context": PAGES_CONTEXT if w.name == HEADLINE else None,
        "e2e": {"value": job_tflops(w.flops, e2e_s * 1e3, ws), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3},
        "gpu_launches": args.steps * launches_per_step,
        "sdpa": sdpa,
        "clocks": clk.summary(),
        "wall_s_timed_loop": wall,
        "ms_per_step_min": min(per), "ms_per_step_median":
            statistics.median(per),
        "ms_per_step_all": per,
        "configs": configs,
        "low_precision": lowp,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
