"""Benchmark of the ExpCast-FP8 + V-Smooth attention hot path on GB300.

A step is one pass of the whole hot path over one batch: vc_attn_prepare (Q/K block quantisation,
k-means grouping, stable argsort, K/V gather, bf16 block means, residual codes) followed by
vc_attn_forward. `value` = 4*B*H*S^2*D per step / step time (TFLOP/s, inputs resident in HBM).
Prepare and forward are each captured once in a CUDA graph; a step replays both.
The forward alone (the pages' kernel metric, preprocessing outside the timer) is reported as
`forward_tflops` and in `roofline`: the median of 12 graph replays after 3 warm-ups. The ablation
arms of the pages (ExpCast off, V-Smooth off, linear key order) are timed the same way, in a random
order. The FP8 dense tensor rate of this GPU is measured in the same run (probe/fp8_mma_peak.cu) and
the forward's fraction of it is `pct_fp8_peak`. The prepare time is split into grouping and
quantisation and amortised over the grouping schedule of the pages (a 40-step run regroups at
steps 0, 4, 8).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config wan] [--impl reference]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import re
import math
import os
import random
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "attention TFLOP/s (4BHS^2D/t) at S=75600,H=40,D=128; % of FP8 dense peak"
FP8_OVER_BF16 = 4.5 / 2.25  # nominal dense FP8 / BF16 tensor ratio on GB300


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="wan")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ablations", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's time: every replica does the same work, so the job ends with the last one."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_replica: float, world: int, ms_per_step: float) -> float:
    """Replicas only (weak scaling): all ranks' work over the slowest rank's step time."""
    return world * flops_per_replica / (ms_per_step * 1e-3) / 1e12


def workload_name(cfg):
    return (f"{cfg['name']}: B={cfg['B']} H={cfg['H']} S={cfg['S']} D={cfg['D']} "
            f"grid={'x'.join(map(str, cfg['grid']))} k={cfg['k']} iters={cfg['iters']}")


FWD_SOURCES = ("vc_fwd.cu", "vc_fwd_common.cuh", "vc_device.cuh", "vc_internal.h")  # the D = 128 kernel
FWD2_SOURCES = ("vc_fwd2.cu", "vc_fwd_common.cuh", "vc_device.cuh", "vc_internal.h")  # the D = 64 kernel


def forward_kernel_name(D: int) -> str:
    return "vc_fwd_kernel<128>" if D == 128 else "vc_fwd2_kernel<64>"


def code_only(text: str) -> str:
    """C/CUDA source without its comments and blank lines, each line stripped of surrounding whitespace (the
    sources contain no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).strip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def forward_source_hash(D: int = 128) -> str:
    """First 16 hex digits of the sha256 of the forward kernel's code (the sources without comments), which the
    committed ncu counters are valid for: a change of comments alone keeps the hash."""
    h = hashlib.sha256()
    for name in (FWD_SOURCES if D == 128 else FWD2_SOURCES):
        with open(os.path.join(ROOT, "bit_fp8_attention_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(cfg):
    """DRAM bytes (read + write) per forward launch from the committed ncu summary of this workload, or None
    when there is none or it was taken on other forward sources than the ones built now."""
    path = os.path.join(ROOT, "profiles", f"vc_fwd_kernel_{cfg['name']}_d{cfg['D']}_s{cfg['S']}_dram.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    m_hash = re.search(r"forward source sha256/16: `?([0-9a-f]{16})", text)
    m_bytes = re.search(r"traffic per launch: (\d+) bytes", text)
    if not (m_hash and m_bytes) or m_hash.group(1) != forward_source_hash(cfg["D"]):
        return None
    return int(m_bytes.group(1))


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [r[0] for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2][1:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def parse_cpulist(text: str) -> set[int]:
    """'0-3,8,10-11' -> {0, 1, 2, 3, 8, 10, 11} (the sysfs cpulist format)."""
    cpus: set[int] = set()
    for part in text.strip().split(","):
        if part:
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def bind_near_gpu(dev) -> str:
    """Run this process on the host cores next to the GPU (its PCI device's local_cpulist), so that the
    pinned host buffers of the end-to-end loop are allocated in that node's memory. Returns what was done;
    the caller restores the previous core set afterwards."""
    props = torch.cuda.get_device_properties(dev)
    try:
        bdf = f"{props.pci_domain_id:04x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bdf}/local_cpulist") as f:
            local = parse_cpulist(f.read())
    except (AttributeError, OSError, ValueError):
        return "unknown"
    allowed = os.sched_getaffinity(0)
    near = local & allowed
    if not near:
        return "no local core in this process's set"
    if near != allowed:
        os.sched_setaffinity(0, near)
    return f"{len(near)} local cores"


def launches_per_step(cfg) -> int:
    # prepare: Q quant, k-means init, (assign, label histogram, scan, scatter, update) x iters,
    # K' quant, block means, residual pack; then the fused forward
    return 5 + 5 * cfg["iters"] + 1


# ---------------------------------------------------------------------------------------------
# Measurement support: CUDA-graph timing, kernel counts, the FP8 tensor-rate probe
# ---------------------------------------------------------------------------------------------
_probe = None


def probe_lib():
    """libvc_probe.so (built beside the attention library): FP8 tensor-rate probe and kernel counting."""
    global _probe
    if _probe is None:
        path = os.path.join(ROOT, "bit_fp8_attention_gb300", "_build", "libvc_probe.so")
        L = ctypes.CDLL(path)
        L.vc_probe_fp8_peak.restype = ctypes.c_int
        L.vc_probe_fp8_peak.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_float),
                                        ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]
        L.vc_probe_capture_begin.restype = ctypes.c_int
        L.vc_probe_capture_begin.argtypes = [ctypes.c_void_p]
        L.vc_probe_capture_end.restype = ctypes.c_int
        L.vc_probe_capture_end.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_int)]
        _probe = L
    return _probe


def count_kernels(fn) -> int:
    """Kernels that one call of fn() enqueues, counted from a captured graph (the graph is discarded)."""
    L = probe_lib()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        if L.vc_probe_capture_begin(cs.cuda_stream) != 0:
            raise RuntimeError("stream capture failed to start")
        try:
            fn()
        finally:
            nk, nn = ctypes.c_int(), ctypes.c_int()
            rc = L.vc_probe_capture_end(cs.cuda_stream, ctypes.byref(nk), ctypes.byref(nn))
    if rc != 0:
        raise RuntimeError("stream capture failed")
    return nk.value


def capture(fn) -> torch.cuda.CUDAGraph:
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def graph_times(g: torch.cuda.CUDAGraph, reps: int = 12, warm: int = 3) -> list[float]:
    """Per-replay device times (ms, CUDA events on the replaying stream) after `warm` untimed replays."""
    for _ in range(warm):
        g.replay()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def median_ms(fn, reps: int = 12, warm: int = 3) -> float:
    """Median device time of fn() over `reps` CUDA-graph replays (fn is captured once)."""
    return statistics.median(graph_times(capture(fn), reps, warm))


def fp8_tensor_peak(target_ms: float = 150.0) -> dict:
    """Dense FP8 (E4M3) tcgen05 rate of this GPU, all SMs, measured now: M=128 N=256 K=32 MMAs."""
    L = probe_lib()
    ms, fl, st = ctypes.c_float(), ctypes.c_double(), ctypes.c_int()
    iters = 4000
    for _ in range(4):
        rc = L.vc_probe_fp8_peak(iters, ctypes.byref(ms), ctypes.byref(fl), ctypes.byref(st))
        if rc != 0 or st.value != 0:
            raise RuntimeError(f"FP8 tensor-rate probe failed (rc {rc}, status {st.value})")
        if ms.value >= 0.5 * target_ms:
            break
        iters = int(iters * target_ms / max(ms.value, 1e-3))
    return {"tflops": fl.value / (ms.value * 1e-3) / 1e12, "ms": ms.value,
            "how": "one CTA per SM, chained tcgen05.mma.cta_group::1.kind::f8f6f4 M=128 N=256 K=32 "
                   "(E4M3 operands in shared memory, fp32 accumulators in TMEM), CUDA events"}


# ---------------------------------------------------------------------------------------------
# CPU oracle legs (the only places this file runs the oracle)
# ---------------------------------------------------------------------------------------------
def score_std_per_head(Q, K, n: int = 4096, seed: int = 0) -> list[float]:
    """std of q.k/sqrt(D) over random pairs, per head of batch 0 (finds the near-uniform heads)."""
    B, H, S, D = Q.shape
    g = torch.Generator(device=Q.device).manual_seed(seed)
    ia = torch.randint(0, S, (n,), device=Q.device, generator=g)
    ib = torch.randint(0, S, (n,), device=Q.device, generator=g)
    out = []
    for h in range(H):
        s = (Q[0, h, ia].float() * K[0, h, ib].float()).sum(dim=1) / math.sqrt(D)
        out.append(float(s.std()))
    return out


def exact_error_report(cfg, Q, K, V, O, perm, heads, rows_per_head: int = 64, seed: int = 0):
    """Relative L2 error against exact fp64 attention ("VC-Attention" Sec. 3.1, Prop. 3.1, Sec. 4.2) on
    sampled rows: the GPU's output, the oracle's quantised algorithm (i) fed the GPU's pi, and the GPU
    against (i)."""
    import oracle

    S = cfg["S"]
    rng = np.random.default_rng(seed)
    acc = {"gpu_vs_exact": [], "oracle_vs_exact": [], "gpu_vs_oracle": []}
    per_head = {}
    for h in heads:
        rows = np.sort(rng.choice(S, min(S, rows_per_head), replace=False))
        q, k, v = (oracle._u16(t[0, h]) for t in (Q, K, V))
        exact = oracle.attention_exact(q, k, v, rows)
        prep = oracle.prepare_head(q, k, v, cfg["k"], cfg["iters"], perm=perm[0, h].cpu().numpy())
        quant, _, _ = oracle.forward_head(prep, rows)
        gpu = O[0, h, torch.from_numpy(rows).to(O.device)].float().cpu().numpy().astype(np.float64)
        d = {"gpu_vs_exact": (gpu, exact), "oracle_vs_exact": (quant, exact), "gpu_vs_oracle": (gpu, quant)}
        per_head[h] = {}
        for key, (a, b) in d.items():
            acc[key].append((float(np.sum((a - b) ** 2)), float(np.sum(b ** 2))))
            per_head[h][key] = float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
    agg = {key: math.sqrt(sum(x for x, _ in v) / max(sum(y for _, y in v), 1e-300)) for key, v in acc.items()}
    agg["heads"] = list(heads)
    agg["rows_per_head"] = rows_per_head
    agg["max_per_head"] = {key: max(per_head[h][key] for h in heads) for key in acc}
    return agg


def spread_heads(H: int, n: int) -> list[int]:
    """Up to n head indices spread evenly over 0..H-1 (always including 0)."""
    n = max(1, min(n, H))
    return sorted({(i * H) // n for i in range(n)})


def cpu_baseline(cfg, Q, K, V, rows_per_head: int = 64, max_heads: int = 8, kmeans_heads: int = 2):
    """The oracle, as it stands, timed on the workload. Small workloads (B*H*S^2 <= 2^24: the tiny config)
    run whole: every k-means round, the quantise/gather/demean and the forward on
    every row of every head. Larger ones run a bounded sample, extrapolated to one step: one Lloyd round on
    `kmeans_heads` heads, quantise/gather/demean and the forward on `rows_per_head` random query rows of up
    to `max_heads` heads spread over batch 0 (about 15-20 s on 16 cores for the Wan-like workload); per-head
    means of the sampled times scale to all B*H heads, rounds and rows."""
    import oracle

    oracle.build()
    S, D, k = cfg["S"], cfg["D"], cfg["k"]
    n_heads_total = cfg["B"] * cfg["H"]
    full = n_heads_total * S * S <= (1 << 24) and Q.shape[1] == cfg["H"]  # small workloads: every head, every row
    if full:
        rows_per_head, max_heads, kmeans_heads = S, cfg["H"], cfg["H"]
    rounds = cfg["iters"] if full else 1
    heads = spread_heads(Q.shape[1], max_heads)
    rng = np.random.default_rng(0)
    km, prep_t, fwd_t = [], [], []
    labels = np.arange(S, dtype=np.int32) * k // S
    perm = oracle.stable_argsort(labels, k)
    for i, h in enumerate(heads):
        q, kk, v = (oracle._u16(t[0, h].cpu()) for t in (Q, K, V))
        if i < kmeans_heads:
            t0 = time.perf_counter()
            oracle.kmeans(v, k, rounds)
            km.append(time.perf_counter() - t0)
        t0 = time.perf_counter()
        prep = oracle.prepare_head(q, kk, v, k, cfg["iters"], perm=perm)
        prep_t.append(time.perf_counter() - t0)
        rows = rng.choice(S, min(S, rows_per_head), replace=False)
        t0 = time.perf_counter()
        oracle.forward_head(prep, rows)
        fwd_t.append((time.perf_counter() - t0) / len(rows))
    t_km = statistics.mean(km) * (cfg["iters"] // rounds) * n_heads_total
    t_prep = statistics.mean(prep_t) * n_heads_total
    t_fwd = statistics.mean(fwd_t) * S * n_heads_total
    t_step = t_km + t_prep + t_fwd
    return {
        "value": synth.flops(cfg) / t_step / 1e12,
        "unit": "TFLOP/s",
        "cores": oracle.num_threads(),
        "kind": "oracle",
        "sample": ((f"whole workload: {cfg['iters']} k-means rounds, quantise/gather/demean and the forward on all "
                    f"{S} rows, every head of batch 0" + (f" (x{cfg['B']} batches)" if cfg["B"] > 1 else "") +
                    f"; step {t_step:.1f} s")
                   if full else
                   (f"heads {heads} of batch 0: 1 k-means round on {len(km)} of them (x{cfg['iters']} rounds "
                    f"x {n_heads_total} heads), quantise/gather/demean on each (x{n_heads_total} heads), forward on "
                    f"{min(S, rows_per_head)} random query rows of each (x{S} rows x {n_heads_total} heads); "
                    f"extrapolated step {t_step:.1f} s")),
        "extrapolated_step_s": t_step,
    }


def run_reference(args, cfg, rank):
    """Reference arm: the CPU oracle, timed as it stands on the host cores, same metric/config.

    One reference step is a bounded sample of the workload (one head: one k-means round, the
    quantisation/gather/demeaning, the forward on 16 query rows); `ms_per_step` is its measured wall
    time and `value` the full step's FLOPs over the step time extrapolated from that sample."""
    if rank != 0:
        return
    import oracle

    oracle.build()
    Q, K, V = synth.make_inputs(dict(cfg, H=1), seed=0, device="cpu")
    times, walls = [], []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        base = cpu_baseline(dict(cfg), Q, K, V, rows_per_head=16, max_heads=1, kmeans_heads=1)
        if i >= args.warmup:
            walls.append(time.perf_counter() - t0)
            times.append(base["extrapolated_step_s"])
    t = statistics.mean(times)
    value = synth.flops(cfg) / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(walls) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(cfg),
                   "sample": ("one step = the oracle on head 0 of the same generator: one k-means round, "
                              "quantise/gather/demean, forward on 16 query rows; value extrapolates it to "
                              f"the whole step ({t:.0f} s per full step)")},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": base["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
def main():
    args = parse()
    rank, world, local = dist_env()
    cfg = synth.config(args.config)
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    from bit_fp8_attention_gb300 import build as _b

    _b.build()
    import bit_fp8_attention_gb300 as vc

    Q, K, V = synth.make_inputs(cfg, seed=rank, device=dev)
    stream = torch.cuda.current_stream()
    flops = synth.flops(cfg)
    B, H, S, D = cfg["B"], cfg["H"], cfg["S"], cfg["D"]
    plan = vc.vc_attn_prepare(Q, K, V, cfg["k"], cfg["iters"])
    O = torch.empty_like(Q)

    def prep():
        vc.vc_attn_prepare(Q, K, V, cfg["k"], cfg["iters"], plan=plan)

    def fwd():
        vc.vc_attn_forward(plan, O)

    prep()
    fwd()  # eager first calls: per-device launch attributes are set outside any capture
    torch.cuda.synchronize()
    kernels_per_step = count_kernels(prep) + count_kernels(fwd)
    g_prep, g_fwd = capture(prep), capture(fwd)

    for _ in range(args.warmup):
        g_prep.replay()
        g_fwd.replay()
    torch.cuda.synchronize()
    rc, bits = vc.vc_plan_status(plan)
    if rc != 0:
        raise RuntimeError(f"kernel status {rc} bits {bits}")

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        t_start.record(stream)
        for e0, e1, e2 in step_events:
            e0.record(stream)
            g_prep.replay()
            e1.record(stream)
            g_fwd.replay()
            e2.record(stream)
        t_end.record(stream)
        barrier()
        # the forward alone, the pages' protocol: median of 12 graph replays after 3 warm-ups
        fwd_reps = graph_times(g_fwd, reps=12, warm=3)
    ms_total = t_start.elapsed_time(t_end)
    step_fwd_ms = [e1.elapsed_time(e2) for _, e1, e2 in step_events]
    step_prep_ms = [e0.elapsed_time(e1) for e0, e1, _ in step_events]
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps
    value = whole_job_tflops(flops, world, ms_step)
    clocks = clk.summary()
    rc, bits = vc.vc_plan_status(plan)
    if rc != 0:
        raise RuntimeError(f"kernel status {rc} bits {bits}")
    fwd_med = statistics.median(fwd_reps)
    fwd_tflops = flops / (fwd_med * 1e-3) / 1e12

    # Ablations of the pages ("VC-Attention" Sec. 4, "Open-VC Attention" results): ExpCast off (fp32
    # exp2 + E4M3 cast per score), V-Smooth off (identity pi, no means, V itself quantised per head),
    # linear instead of mid-window key order; each a graph of the forward, 12 replays, arms shuffled.
    ablations = None
    if not args.no_ablations:
        p_plain = vc.vc_attn_prepare_ex(Q, K, V, cfg["k"], cfg["iters"], flags=0)
        O_ab = torch.empty_like(O)
        F = vc.VC_FLAGS_DEFAULT
        arms = {"default": (plan, F), "expcast_off": (plan, F & ~vc.VC_EXPCAST),
                "vsmooth_off": (p_plain, F & ~vc.VC_VSMOOTH), "linear_order": (plan, F & ~vc.VC_MIDWINDOW)}
        order = list(arms)
        random.Random(1234).shuffle(order)
        ablations = {"order": order}
        for name in order:
            pl, fl = arms[name]
            vc.vc_attn_forward(pl, O_ab, flags=fl)  # eager first call of this instantiation
            torch.cuda.synchronize()
            ms = median_ms(lambda: vc.vc_attn_forward(pl, O_ab, flags=fl))
            ablations[name] = {"forward_ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "flags": fl}
        rc, bits = vc.vc_plan_status(p_plain)
        if rc != 0:
            raise RuntimeError(f"kernel status {rc} bits {bits} (V-Smooth-off plan)")
        p_plain.destroy()
        del O_ab

    # Prepare split: quantisation/gather/means with the permutation given, versus the full prepare with
    # k-means and argsort; medians of graph replays.
    perm = vc.vc_plan_get(plan, vc.VC_PLAN_PERM)
    t_prep_full = statistics.median(step_prep_ms + graph_times(g_prep, reps=6))
    t_prep_quant = median_ms(lambda: vc.vc_attn_prepare_ex(Q, K, V, cfg["k"], cfg["iters"], perm=perm, plan=plan),
                             reps=7)
    # the QK Hadamard rotation fused into the Q and K quantisers ("VC-Attention" Sec. 3.4): its prepare cost
    t_prep_quant_rot = median_ms(lambda: vc.vc_attn_prepare_ex(Q, K, V, cfg["k"], cfg["iters"], perm=perm, plan=plan,
                                                               flags=vc.VC_VSMOOTH | vc.VC_QK_HADAMARD), reps=7)
    t_group = max(t_prep_full - t_prep_quant, 0.0)
    # The grouping schedule's actions ("VC-Attention" Sec. 3.4, App. A): a warm-started regroup with half
    # the rounds, pi kept with new means, pi kept without means; amortised over the pages' 40-step run.
    prep()
    warm_iters = max(1, cfg["iters"] // 2)
    t_step = {
        vc.VC_STEP_GROUP: t_prep_full,
        vc.VC_STEP_GROUP_WARM: median_ms(lambda: vc.vc_attn_prepare_ex(
            Q, K, V, cfg["k"], warm_iters, flags=vc.STEP_PREPARE_FLAGS[vc.VC_STEP_GROUP_WARM], plan=plan), reps=7),
        vc.VC_STEP_REUSE: median_ms(lambda: vc.vc_attn_prepare_ex(
            Q, K, V, cfg["k"], cfg["iters"], flags=vc.STEP_PREPARE_FLAGS[vc.VC_STEP_REUSE], plan=plan), reps=7),
        vc.VC_STEP_PLAIN: median_ms(lambda: vc.vc_attn_prepare_ex(
            Q, K, V, cfg["k"], cfg["iters"], flags=vc.STEP_PREPARE_FLAGS[vc.VC_STEP_PLAIN], plan=plan), reps=7),
    }
    n_sched = 40
    sched_prepare_ms = sum(t_step[vc.vc_schedule_action(s_, n_sched, 4)] for s_ in range(n_sched)) / n_sched
    prep()
    fwd()
    torch.cuda.synchronize()

    # V residual repair ("Open-VC Attention", "Why V residual repair"): no V-Smooth, one V scale per
    # head, the 0.5% of tokens with the largest residual energy repaired; against the same path without.
    n_rep = vc.repair_rows_for(cfg["S"], 0.005)
    O_rep = torch.empty_like(O)
    p_rep = vc.vc_attn_prepare_repair(Q, K, V, n_rep)
    p_plain = vc.vc_attn_prepare_repair(Q, K, V, 0)
    rep_flags = vc.VC_EXPCAST | vc.VC_MIDWINDOW
    vc.vc_attn_forward(p_rep, O_rep, flags=rep_flags)
    vc.vc_attn_forward(p_plain, O_rep, flags=rep_flags)
    torch.cuda.synchronize()
    repair = {"rho": 0.005, "rows_per_head": n_rep,
              "prepare_ms": median_ms(lambda: vc.vc_attn_prepare_repair(Q, K, V, n_rep, plan=p_rep), reps=7),
              "prepare_ms_no_repair": median_ms(lambda: vc.vc_attn_prepare_repair(Q, K, V, 0, plan=p_plain), reps=7),
              "forward_ms": median_ms(lambda: vc.vc_attn_forward(p_rep, O_rep, flags=rep_flags)),
              "forward_ms_no_repair": median_ms(lambda: vc.vc_attn_forward(p_plain, O_rep, flags=rep_flags))}
    repair["forward_overhead_pct"] = 100.0 * (repair["forward_ms"] / repair["forward_ms_no_repair"] - 1.0)
    p_rep.destroy()
    p_plain.destroy()
    del O_rep
    torch.cuda.synchronize()

    # End to end through the public API from pinned host memory, every step's copies inside the timed
    # region. As a serving loop would run it: the host-to-device copies of step i+1's inputs and the
    # device-to-host copy of step i-1's output run on their own streams while step i computes
    # (device inputs and outputs double-buffered); the compute stream only waits for its own inputs.
    e2e = None
    if not args.no_e2e:
        all_cores = os.sched_getaffinity(0)
        placement = bind_near_gpu(dev)
        Qh, Kh, Vh = (t.cpu().pin_memory() for t in (Q, K, V))
        Oh = [torch.empty(O.shape, dtype=O.dtype, device="cpu").pin_memory() for _ in range(2)]
        Qd = [torch.empty_like(Q) for _ in range(2)]
        Kd = [torch.empty_like(K) for _ in range(2)]
        Vd = [torch.empty_like(V) for _ in range(2)]
        Od = [torch.empty_like(O) for _ in range(2)]
        # one stream per input tensor, so that the three host-to-device copies can use several copy engines
        s_ins, s_out = [torch.cuda.Stream() for _ in range(3)], torch.cuda.Stream()
        s_in = s_ins[0]
        ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("free", "done", "out")}
        ev_in = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]

        def e2e_run(n, start=None):
            for i in range(n):
                b = i % 2
                for si, e, (dst, src) in zip(s_ins, ev_in[b], ((Qd[b], Qh), (Kd[b], Kh), (Vd[b], Vh))):
                    with torch.cuda.stream(si):
                        if i == 0 and start is not None:
                            si.wait_event(start)  # the timed region starts before the first copy
                        if i >= 2:
                            si.wait_event(ev["free"][b])  # prepare(i-2) has read these input buffers
                        dst.copy_(src, non_blocking=True)
                        e.record(si)
                for e in ev_in[b]:
                    stream.wait_event(e)
                vc.vc_attn_prepare(Qd[b], Kd[b], Vd[b], cfg["k"], cfg["iters"], stream=stream, plan=plan)
                ev["free"][b].record(stream)
                if i >= 2:
                    stream.wait_event(ev["out"][b])  # the output of step i-2 has left this buffer
                vc.vc_attn_forward(plan, Od[b], stream=stream)
                ev["done"][b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev["done"][b])
                    Oh[b].copy_(Od[b], non_blocking=True)
                    ev["out"][b].record(s_out)

        e2e_run(2)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        with torch.cuda.stream(s_in):
            Qd[0].copy_(Qh, non_blocking=True)
        b.record(s_in)
        torch.cuda.synchronize()
        h2d_gbs = Q.numel() * Q.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9
        a.record(s_out)
        with torch.cuda.stream(s_out):
            Oh[0].copy_(Od[0], non_blocking=True)
        b.record(s_out)
        torch.cuda.synchronize()
        d2h_gbs = O.numel() * O.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9
        # enough steps that the pipeline's fill (step 0's inputs) and drain (the last output) are small
        n_e2e = max(2, min(max(args.steps, 10), 20))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        a.record(stream)
        e2e_run(n_e2e, start=a)
        s_out.wait_stream(stream)
        b.record(s_out)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / n_e2e, world, dev)
        nbytes = Q.numel() * Q.element_size()
        e2e = {"value": whole_job_tflops(flops, world, e2e_ms), "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": 3 * nbytes, "d2h_bytes_per_step": nbytes,
               "copies": "own streams (one per input tensor), double-buffered: step i+1's inputs and step i-1's "
                         "output move while step i computes",
               "steps": n_e2e, "h2d_gbs_alone": h2d_gbs, "d2h_gbs_alone": d2h_gbs, "host_cores": placement}
        del Qh, Kh, Vh, Oh, Qd, Kd, Vd, Od
        os.sched_setaffinity(0, all_cores)

    # The dense FP8 tensor rate of this GPU, measured now (the forward's own peak) with clocks sampled.
    with ClockSampler(local) as clk_peak:
        peak = fp8_tensor_peak()
    peak["clocks"] = clk_peak.summary()
    bf16_burst, bf16_sus, src = measured_peaks()
    fp8_from_bf16 = bf16_burst * FP8_OVER_BF16
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": workload_name(cfg), "parallelism": "replicas" if world > 1 else "single GPU",
                   "step": "vc_attn_prepare (k-means grouping + quantisation) + vc_attn_forward, "
                           "each replayed from a CUDA graph",
                   "l2": f"inputs larger than L2 (Q, K, V {3 * Q.numel() * 2 / 1e9:.2f} GB), no flush"},
        "forward_ms": fwd_med, "forward_tflops": fwd_tflops,
        "forward_timing": "median of 12 CUDA-graph replays after 3 warm-ups",
        "forward_ms_in_steps": statistics.median(step_fwd_ms),
        "fp8_peak_measured": peak,
        "pct_fp8_peak": 100.0 * fwd_tflops / peak["tflops"],
        "pct_fp8_peak_of_bf16x2": 100.0 * fwd_tflops / fp8_from_bf16,
        "prepare_ms": t_prep_full, "prepare_quant_ms": t_prep_quant, "grouping_ms": t_group,
        "amortised_prepare_ms": t_prep_quant + 3.0 / 40.0 * t_group,
        "schedule": {"steps": 40, "reuse": 4, "warm_iters": warm_iters,
                     "prepare_ms_per_action": {"group": t_step[vc.VC_STEP_GROUP],
                                               "group_warm": t_step[vc.VC_STEP_GROUP_WARM],
                                               "reuse": t_step[vc.VC_STEP_REUSE], "plain": t_step[vc.VC_STEP_PLAIN]},
                     "prepare_ms_per_step": sched_prepare_ms},
        "ablations": ablations,
        "repair": repair,
        "qk_hadamard": {"prepare_quant_ms": t_prep_quant_rot, "prepare_quant_ms_without": t_prep_quant},
        "roofline": {"bound": "tensor", "kernel": forward_kernel_name(cfg["D"]), "achieved": fwd_tflops,
                     "peak": fp8_from_bf16,
                     "unit": "TFLOP/s", "frac": fwd_tflops / fp8_from_bf16, "traffic": profiled_traffic(cfg),
                     "peak_source": f"{src} bf16 burst {bf16_burst:.0f} TFLOP/s x {FP8_OVER_BF16:.0f} "
                                    "(FP8/BF16 nominal), as the roofline rule prescribes; against the FP8 "
                                    "tensor rate measured in this run see frac_of_fp8_measured",
                     "frac_of_fp8_measured": fwd_tflops / peak["tflops"]},
        "clocks": clocks,
        "gpu_launches": kernels_per_step * args.steps,
        "gpu_launches_how": (f"counted: {kernels_per_step} kernel nodes in the captured prepare and forward "
                             f"graphs, replayed once per step"),
    }
    if e2e:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, Q, K, V)
        line["cpu_baseline"].pop("extrapolated_step_s", None)
        # error against exact fp64 attention on sampled rows (the oracle's leg)
        stds = score_std_per_head(Q, K)
        near_uniform = [h for h in range(H) if stds[h] < 1.5]
        regular = [h for h in range(H) if stds[h] >= 1.5]
        pick = regular[:: max(1, len(regular) // 3)][:3]
        perm_all = vc.vc_plan_get(plan, vc.VC_PLAN_PERM)
        torch.cuda.synchronize()
        line["exact_err"] = {"heads": exact_error_report(cfg, Q, K, V, O, perm_all, pick)}
        if near_uniform:
            line["exact_err"]["near_uniform_heads"] = exact_error_report(cfg, Q, K, V, O, perm_all,
                                                                         near_uniform[:2])
        line["exact_err"]["what"] = ("rel-L2 over sampled rows: GPU vs exact fp64 attention, the oracle's "
                                     "quantised algorithm (fed the GPU's pi) vs exact, and GPU vs that oracle")
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.destroy()
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
