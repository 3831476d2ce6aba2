#!/usr/bin/env python
"""Benchmark: causal prefill attention TFLOP/s at 32K tokens on GB300.

Workload (default): batch 1, 32 query heads / 8 KV heads, 32768 tokens, head
dim 128, Gaussian N(0,1) Q/K/V drawn in bf16 from seed 0 (``workloads``).
One step is one pass of the whole hot path over that input:
  * FP8 path (the headline ``value``): quantise Q, K, V per 128-token block
    (one quantiser launch for the three) and run FP8 causal attention (1
    launch);
  * BF16 path (reported under ``bf16``): BF16 causal attention (1 launch).
TFLOP/s counts causal FLOPs B*Hq*S^2*(Dqk+Dv) per step.

Timing: W untimed warm-up steps, then exactly K steps; each step bracketed by
CUDA events on the launching stream, with a 256 MiB L2 flush between steps
(outside the events; the inputs are larger than L2 as well). Barrier and
device synchronisation on both sides; the time is the max over ranks. Under
torchrun every rank runs its own replica of the workload on its own GPU
(replicas only: the path has no exchange step), and ``value`` counts the
work of all ranks.

``--impl reference`` times the CPU oracle (float64 attention and the fp32
quantiser emulation) on a bounded sample of the same workload; only rank 0
runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal prefill attn TFLOP/s (FP8, BF16) at 32K tokens; % of GB300 dense peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0          # nominal dense fp8 / bf16 tensor-core rate ratio on GB300
# Per-SM rates of the softmax's two special-function steps, measured on a
# GB300 with register-only microbenchmarks: ex2.approx.ftz.f32 results per
# clock (30.5 measured with 8 to 32 warps per SM, 32 the unit's rate), and
# cvt.rn.satfinite.e4m3x2.f32 converted elements per clock (94.5 to 98.5
# with 16 warps per SM, inputs perturbed each iteration, the folding of the
# results subtracted).
EX2_PER_CLK_SM = 32.0
E4M3_CVT_PER_CLK_SM = 98.5
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["zyfa", "reference"], default="zyfa")
    p.add_argument("--workload", default=None, help="workload name (default: the 32K GQA shape)")
    p.add_argument("--hadamard", action="store_true", help="rotate Q and K before quantisation")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-split", action="store_true",
                   help="small problems: keep one CTA per query-tile pair (no split key ranges)")
    p.add_argument("--graph", action="store_true",
                   help="also time the FP8 step and the BF16 call replayed from CUDA graphs (no host work "
                        "between launches: the device time of small workloads)")
    p.add_argument("--chunks", type=int, default=0,
                   help="pieces of the host pipeline along the sequence (0: the library's default)")
    p.add_argument("--paged", action="store_true",
                   help="also time the attention kernels over a shuffled paged K/V cache")
    p.add_argument("--ctx", type=int, default=0,
                   help="with --paged: cached tokens before the queries (multiple of 128); the last S - ctx "
                        "tokens are the new chunk")
    p.add_argument("--decode", type=int, default=0,
                   help="also time a decode step: this many sequences of S - 1 cached tokens and one new token, "
                        "through the paged calls")
    p.add_argument("--cpu-worker", default=None, help=argparse.SUPPRESS)
    return p.parse_args()


# --------------------------------------------------------------------- peaks --
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# The attention kernel and the host code that picks its work order (the
# order decides how much K/V is re-read from HBM).
ATTN_SOURCES = ("attention.cu", "api.cu")


def source_hash(*kernel_files: str) -> str:
    """First 16 hex digits of the SHA-256 of the named csrc files, concatenated."""
    hs = hashlib.sha256()
    for kernel_file in kernel_files:
        with open(os.path.join(ROOT, "bf16_causal_prefill_gb300", "csrc", kernel_file), "rb") as f:
            hs.update(f.read())
    return hs.hexdigest()[:16]


def traffic_from_profiles(kernel_files, tag: str):
    """Per-launch DRAM bytes recorded in profiles/ for `tag`, if the sources
    still have the hash the counters were taken with; else None."""
    h = source_hash(*kernel_files)
    pat = re.compile(rf"^traffic\[{re.escape(tag)}\]:\s*([0-9.eE+]+)\s+bytes/launch\s+src=([0-9a-f]+)")
    pdir = os.path.join(ROOT, "profiles")
    for name in sorted(os.listdir(pdir)) if os.path.isdir(pdir) else []:
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name)) as f:
            for line in f:
                m = pat.match(line.strip())
                if m and m.group(2) == h:
                    return float(m.group(1))
    return None


# -------------------------------------------------------------------- clocks --
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                     util=float(parts[4]), hw=parts[6], hwt=parts[7], swt=parts[8],
                                     swpc=parts[9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        loaded = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swpc", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["max"] for r in loaded),
                "power_w_max": max(r["power"] for r in loaded), "samples": len(loaded),
                "reasons": sorted(reasons)}


def clocks_rejected(c) -> bool:
    if not c:
        return False
    if set(c["reasons"]) & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}:
        return True
    return c["sm_mhz"] < 0.5 * c["sm_max_mhz"] and not c["reasons"]


# ---------------------------------------------------------- CPU oracle timing --
class OracleSampler:
    """Times the oracle's FP8 path on a sample of the workload: the first
    min(S, 4096) tokens are quantised once (fp32 quantiser emulation), then
    each call computes random (batch, head, row) outputs in float64 for a
    time budget. Per-element and per-FLOP times extrapolate to the full
    workload."""

    def __init__(self, workload_name: str, hadamard: bool):
        import numpy as np
        import workloads
        from oracle import fp8 as ofp8

        self.w = w = workloads.get(workload_name)
        self.s_lim = min(w.S, 4096)
        q, k, v = workloads.make_qkv(w.with_seq(self.s_lim, name=w.name))
        q32, k32, v32 = q.float().numpy(), k.float().numpy(), v.float().numpy()
        had = hadamard and w.Dqk == 128
        t0 = time.perf_counter()
        cq, sq = ofp8.quantize_fp8(q32, had)
        ck, sk = ofp8.quantize_fp8(k32, had)
        cv, sv = ofp8.quantize_fp8(v32, False)
        self.qd, self.kd, self.vd = (ofp8.dequantize_fp8(cq, sq), ofp8.dequantize_fp8(ck, sk),
                                     ofp8.dequantize_fp8(cv, sv))
        self.t_quant = time.perf_counter() - t0
        self.elems = q32.size + k32.size + v32.size
        self.rng = np.random.default_rng(0)

    def step(self, budget_s: float):
        from oracle import attention as oattn
        w = self.w
        flops, rows = 0.0, 0
        t1 = time.perf_counter()
        while time.perf_counter() - t1 < budget_s or rows == 0:
            b = int(self.rng.integers(0, w.B))
            h = int(self.rng.integers(0, w.Hq))
            i = int(self.rng.integers(0, self.s_lim))
            oattn.causal_attention_rows(self.qd, self.kd, self.vd, w.softmax_scale, b, h, [i])
            flops += 2.0 * (i + 1) * (w.Dqk + w.Dv)
            rows += 1
        t_attn = time.perf_counter() - t1
        full_elems = w.B * w.S * (w.Hq * w.Dqk + w.Hkv * (w.Dqk + w.Dv))
        t_full = self.t_quant / self.elems * full_elems + t_attn / flops * w.causal_flops
        return {"value": w.causal_flops / t_full / 1e12, "t_full_s": t_full, "rows": rows,
                "sample": (f"oracle FP8 path (fp32 quantiser emulation, dequantise, float64 attention) on the "
                           f"first {self.s_lim} tokens: Q/K/V quantised once ({self.t_quant:.1f} s), then "
                           f"{rows} random (batch, head, row) outputs ({t_attn:.1f} s); per-element and "
                           f"per-FLOP times extrapolated to the full workload ({t_full:.0f} s)")}


def _pin_cpu_threads():
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"


def run_cpu_worker(spec: str):
    d = json.loads(spec)
    res = OracleSampler(d["workload"], d["hadamard"]).step(d["budget_s"])
    print("CPU_WORKER_RESULT " + json.dumps(res))


def cpu_baseline(workload_name: str, budget_s: float, hadamard: bool):
    """Run the oracle sample in a fresh single-threaded process."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    env.pop("CUDA_VISIBLE_DEVICES", None)
    spec = json.dumps({"workload": workload_name, "budget_s": budget_s, "hadamard": hadamard})
    p = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", spec], env=env,
                       capture_output=True, text=True, timeout=900)
    for line in p.stdout.splitlines():
        if line.startswith("CPU_WORKER_RESULT "):
            res = json.loads(line[len("CPU_WORKER_RESULT "):])
            res.update({"unit": UNIT, "cores": 1, "kind": "oracle"})
            return res
    raise RuntimeError(f"cpu baseline worker failed:\n{p.stdout[-2000:]}\n{p.stderr[-2000:]}")


# ---------------------------------------------------------------- distributed --
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------- main --
def measure_fp8_gemm(dev, n: int = 8192, reps: int = 10):
    """Burst rate of the library's dense e4m3 GEMM on this GPU: cuBLASLt
    through torch._scaled_mm, n^3, tensor-wise scales, bf16 out, best of
    `reps` after 3 warm-ups (the method of the measured bf16 figure). The
    attention kernel is also compared with it; the roofline's peak stays the
    measured bf16 burst x the nominal fp8/bf16 ratio. None if the library
    call is not available."""
    import torch
    try:
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
        bt = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev, dtype=torch.float32)

        def gemm():
            return torch._scaled_mm(a, bt.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

        for _ in range(3):
            gemm()
        torch.cuda.synchronize(dev)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            gemm()
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except (RuntimeError, AttributeError, TypeError):
        return None


def main_reference(args):
    _pin_cpu_threads()
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import workloads
    name = args.workload or workloads.BENCH
    w = workloads.get(name)
    K, W = args.steps, max(args.warmup, 3)
    per_step = max(0.3, min(6.0, 150.0 / (K + W)))
    sampler = OracleSampler(name, args.hadamard)
    for _ in range(W):
        sampler.step(per_step * 0.2)
    t_full = []
    last = None
    for _ in range(K):
        last = sampler.step(per_step)
        t_full.append(last["t_full_s"])
    t_mean = statistics.mean(t_full)
    value = w.causal_flops / t_mean / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": W, "ms_per_step": t_mean * 1e3, "extrapolated": True,
        "ms_per_step_note": ("extrapolated: each step times the oracle on a sample of the workload and scales "
                             "its per-element and per-FLOP times to the full workload; the run itself takes "
                             "about steps x the sample time"),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3 path emulated (fp32 quantiser, float64 attention)",
        "data": "synthetic (seeded Gaussian, bf16)",
        "config": {"workload": name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "Dqk": w.Dqk, "Dv": w.Dv,
                   "path": "oracle: quantise Q/K/V + attention", "hadamard": bool(args.hadamard)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "each step: " + last["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_paged(args, w, qd, kd, vd, timed, dev):
    """Kernel-only throughput of the paged calls on the same workload: each
    batch row's K/V in 128-token pages at shuffled cache positions, the last
    S - ctx tokens as the new chunk (its queries) after ctx cached ones."""
    import torch
    import bf16_causal_prefill_gb300 as zyfa
    ctx = args.ctx
    if ctx % 128 or not 0 <= ctx < w.S or w.S % 128:
        raise SystemExit("--ctx must be a multiple of 128 below S (and S a multiple of 128)")
    B, S, n = w.B, w.S, w.S // 128
    Lq = S - ctx
    perm = torch.randperm(B * n, generator=torch.Generator().manual_seed(0)).to(dev)
    kc = torch.empty((B * n, 128, w.Hkv, w.Dqk), dtype=torch.bfloat16, device=dev)
    vc = torch.empty((B * n, 128, w.Hkv, w.Dv), dtype=torch.bfloat16, device=dev)
    kc[perm] = kd.reshape(B * n, 128, w.Hkv, w.Dqk)
    vc[perm] = vd.reshape(B * n, 128, w.Hkv, w.Dv)
    bt = perm.view(B, n).to(torch.int32).contiguous()
    qn = qd[:, ctx:].reshape(B * Lq, w.Hq, w.Dqk).contiguous()
    cu = [i * Lq for i in range(B + 1)]
    ctxs = [ctx] * B
    had = bool(args.hadamard) and w.Dqk == 128
    q8, qs = zyfa.quantize_fp8_varlen(qn, cu, had)
    kc8, ks = zyfa.quantize_fp8_cache(kc, had)
    vc8, vs = zyfa.quantize_fp8_cache(vc, False)
    o = torch.empty((B * Lq, w.Hq, w.Dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(fp8, ev=None):
        if ev is not None:
            ev[0].record(stream)
        if fp8:
            zyfa.attn_fwd_fp8_paged(q8, qs, kc8, ks, vc8, vs, cu, ctxs, bt, w.softmax_scale, out=o)
        else:
            zyfa.attn_fwd_bf16_paged(qn, kc, vc, cu, ctxs, bt, w.softmax_scale, out=o)
        if ev is not None:
            ev[1].record(stream)

    steps = max(3, min(args.steps, 50))
    _, t8 = timed(lambda ev=None: step(True, ev), steps, 3)
    _, t16 = timed(lambda ev=None: step(False, ev), steps, 3)
    # causal FLOPs of the chunk: query i (position ctx + i) sees ctx + i + 1 keys
    flops = 2.0 * B * w.Hq * (w.Dqk + w.Dv) * (Lq * ctx + Lq * (Lq + 1) / 2)
    return {"ctx": ctx, "new_tokens": Lq, "page_tokens": 128, "pages": B * n, "steps": steps,
            "fp8_kernel": flops / (t8 * 1e-3) / 1e12, "bf16_kernel": flops / (t16 * 1e-3) / 1e12, "unit": UNIT,
            "ms_per_launch": {"fp8": t8, "bf16": t16},
            "layout": "K/V pages at shuffled cache positions (seeded permutation), block table on the device"}


def run_decode(args, w, timed, dev):
    """A decode step through the paged calls: N sequences, each S - 1 cached
    tokens plus one new token (its query), K/V pages at shuffled positions.
    Inputs drawn on the device from a seeded generator. Reports the K/V
    bytes each call must read over its time (the memory roofline of decode)."""
    import torch
    import bf16_causal_prefill_gb300 as zyfa
    N, L = args.decode, w.S
    n = (L + 127) // 128
    g = torch.Generator(device=dev).manual_seed(0)
    kc = torch.randn((N * n, 128, w.Hkv, w.Dqk), generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn((N * n, 128, w.Hkv, w.Dv), generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn((N, w.Hq, w.Dqk), generator=g, device=dev).to(torch.bfloat16)
    perm = torch.randperm(N * n, generator=torch.Generator().manual_seed(1)).to(dev)
    bt = perm.view(N, n).to(torch.int32).contiguous()
    cu = list(range(N + 1))
    ctxs = [L - 1] * N
    q8, qs = zyfa.quantize_fp8_decode(q)
    kc8, ks = zyfa.quantize_fp8_cache(kc)
    vc8, vs = zyfa.quantize_fp8_cache(vc)
    o = torch.empty((N, w.Hq, w.Dv), dtype=torch.bfloat16, device=dev)
    lens = [L] * N
    stream = torch.cuda.current_stream(dev)

    def step(fp8, ev=None):
        if ev is not None:
            ev[0].record(stream)
        if fp8:
            zyfa.attn_decode_fp8_paged(q8, qs, kc8, ks, vc8, vs, lens, bt, w.softmax_scale, out=o)
        else:
            zyfa.attn_decode_bf16_paged(q, kc, vc, lens, bt, w.softmax_scale, out=o)
        if ev is not None:
            ev[1].record(stream)

    steps = max(3, min(args.steps, 50))
    _, t8 = timed(lambda ev=None: step(True, ev), steps, 3)
    _, t16 = timed(lambda ev=None: step(False, ev), steps, 3)
    kv8 = N * L * w.Hkv * (w.Dqk + w.Dv)          # bytes of e4m3 K and V the step must read
    flops = 2.0 * N * w.Hq * (w.Dqk + w.Dv) * L
    peaks, src = load_peaks()
    bw = {"fp8": kv8 / (t8 * 1e-3) / 1e9, "bf16": 2 * kv8 / (t16 * 1e-3) / 1e9}
    return {"seqs": N, "ctx": L - 1, "new_tokens_per_seq": 1, "steps": steps,
            "ms_per_launch": {"fp8": t8, "bf16": t16}, "kv_read_GBps": bw,
            "frac_of_hbm": {k: v / peaks["hbm_gbs"] for k, v in bw.items()}, "hbm_peak_source": src,
            "tflops": {"fp8": flops / (t8 * 1e-3) / 1e12, "bf16": flops / (t16 * 1e-3) / 1e12},
            "path": "decode calls: one unit per (sequence, KV head), the group's query heads as tile rows"}


def run_graph(fp8_step, bf16_step, flush, K, w, world):
    """The FP8 step and the BF16 call captured once into CUDA graphs and
    replayed K times each (L2 flushed between replays, CUDA events around
    each replay): the device time without the host's per-call work."""
    import torch
    import bf16_causal_prefill_gb300 as zyfa
    res = {}
    for name, step in (("fp8_step", fp8_step), ("bf16", bf16_step)):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(K):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = max_over_ranks(sum(ts) / len(ts), world)
        res[name] = {"ms": ms, "value": world * w.causal_flops / (ms * 1e-3) / 1e12, "unit": UNIT}
        zyfa.device_status()
    res["note"] = "one graph per path, replayed; the gap to the eager timing is host work per call"
    return res


def main():
    args = parse_args()
    if args.cpu_worker:
        run_cpu_worker(args.cpu_worker)
        return
    if args.impl == "reference":
        main_reference(args)
        return

    import torch
    import __graft_entry__
    import bf16_causal_prefill_gb300 as zyfa
    import workloads

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    zyfa.lib()
    dev = torch.device("cuda", local)
    name = args.workload or workloads.BENCH
    w = workloads.get(name)
    K, W = args.steps, max(args.warmup, 3)
    had = bool(args.hadamard) and w.Dqk == 128

    q, k, v = workloads.make_qkv(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    nb = zyfa.scale_blocks(w.S)
    q8 = torch.empty(qd.shape, dtype=torch.uint8, device=dev)
    k8 = torch.empty(kd.shape, dtype=torch.uint8, device=dev)
    v8 = torch.empty(vd.shape, dtype=torch.uint8, device=dev)
    qs = torch.empty((w.B, w.Hq, nb), dtype=torch.float32, device=dev)
    ks = torch.empty((w.B, w.Hkv, nb), dtype=torch.float32, device=dev)
    vs = torch.empty((w.B, w.Hkv, nb), dtype=torch.float32, device=dev)
    o8 = torch.empty((w.B, w.S, w.Hq, w.Dv), dtype=torch.bfloat16, device=dev)
    o16 = torch.empty_like(o8)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # Small problems split each query-tile pair's keys across CTAs (the
    # library decides; this workspace lets it): allocated once, outside the
    # timed steps. Large problems need none and run the unsplit kernels.
    split_c = 0 if args.no_split else zyfa.lib().zyfa_attn_split_tiles(w.B, w.S, w.Hq)
    ws_bytes = zyfa.lib().zyfa_attn_workspace_bytes(w.B, w.S, w.Hq) if split_c > 0 else 0
    split_ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else False

    def fp8_step(ev_attn=None):
        zyfa.quantize_fp8_qkv(qd, kd, vd, had, out=((q8, qs), (k8, ks), (v8, vs)))
        if ev_attn is not None:
            ev_attn[0].record(stream)
        zyfa.attn_fwd_fp8(q8, qs, k8, ks, v8, vs, w.softmax_scale, out=o8, split=split_ws)
        if ev_attn is not None:
            ev_attn[1].record(stream)

    def bf16_step(ev_attn=None):
        if ev_attn is not None:
            ev_attn[0].record(stream)
        zyfa.attn_fwd_bf16(qd, kd, vd, w.softmax_scale, out=o16, split=split_ws)
        if ev_attn is not None:
            ev_attn[1].record(stream)

    def timed(step, n_steps, n_warm):
        for _ in range(n_warm):
            step()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_steps)]
        ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_steps)]
        barrier(world)
        torch.cuda.synchronize()
        for i in range(n_steps):
            flush.zero_()
            ev[i][0].record(stream)
            step(ev_k[i])
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        t_step = sum(a.elapsed_time(b) for a, b in ev) / n_steps          # ms
        t_kern = sum(a.elapsed_time(b) for a, b in ev_k) / n_steps        # ms
        zyfa.device_status()
        return t_step, t_kern

    sampler = ClockSampler(local)
    for attempt in range(2):
        sampler.start()
        t8, t8k = timed(fp8_step, K, W)
        t16, t16k = timed(bf16_step, K, W)
        clocks = sampler.stop()
        if not clocks_rejected(clocks):
            break
    t8 = max_over_ranks(t8, world)
    t16 = max_over_ranks(t16, world)

    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.pin_memory() for t in (q, k, v))
        ho = torch.empty(o8.shape, dtype=torch.bfloat16).pin_memory()
        ws = zyfa.prefill_fp8_host_workspace(w.B, w.S, w.Hq, w.Hkv, w.Dqk, w.Dv, device=dev)

        def e2e_step(ev_attn=None):
            if ev_attn is not None:
                ev_attn[0].record(stream)
            zyfa.prefill_fp8_host(hq, hk, hv, had, w.softmax_scale, out=ho, n_chunks=args.chunks, workspace=ws)
            if ev_attn is not None:
                ev_attn[1].record(stream)

        te, _ = timed(e2e_step, max(3, min(K, 20)), 3)
        te = max_over_ranks(te, world)

        # The pieces alone: inputs host -> device, output device -> host
        # (whole tensors on one stream), next to the device step timed above.
        def h2d_step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            qd.copy_(hq, non_blocking=True)
            kd.copy_(hk, non_blocking=True)
            vd.copy_(hv, non_blocking=True)
            if ev is not None:
                ev[1].record(stream)

        def d2h_step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            ho.copy_(o8, non_blocking=True)
            if ev is not None:
                ev[1].record(stream)

        n_copy = max(3, min(K, 10))
        t_h2d, _ = timed(h2d_step, n_copy, 2)
        t_d2h, _ = timed(d2h_step, n_copy, 2)
        h2d_b = sum(t.numel() * t.element_size() for t in (q, k, v))
        d2h_b = o8.numel() * o8.element_size()
        serial = t_h2d + t8 + t_d2h
        e2e = {"value": world * w.causal_flops / (te * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in (q, k, v))),
               "d2h_bytes_per_step": int(o8.numel() * o8.element_size()), "ms_per_step": te,
               "path": "prefill_fp8_host: pinned host bf16 Q/K/V -> device, quantise + FP8 attention, "
                       "bf16 O -> pinned host, pipelined along the sequence",
               "chunks": args.chunks,
               "breakdown": {"h2d_ms": t_h2d, "h2d_GBps": h2d_b / (t_h2d * 1e-3) / 1e9,
                             "device_ms": t8, "d2h_ms": t_d2h, "d2h_GBps": d2h_b / (t_d2h * 1e-3) / 1e9,
                             "serial_ms": serial, "e2e_ms": te, "hidden_ms": serial - te,
                             "note": "pieces timed alone (whole-tensor copies on one stream, the device FP8 step); "
                                     "hidden_ms = the part of their sum the pipeline overlaps"}}

    graph = None
    if args.graph:
        graph = run_graph(fp8_step, bf16_step, flush, K, w, world)

    paged = None
    if args.paged:
        paged = run_paged(args, w, qd, kd, vd, timed, dev)
    decode = None
    if args.decode > 0:
        decode = run_decode(args, w, timed, dev)

    peaks, src = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    fp8_peak_sus = peaks["bf16_tflops_sustained"] * FP8_PER_BF16
    v8 = world * w.causal_flops / (t8 * 1e-3) / 1e12
    v16 = world * w.causal_flops / (t16 * 1e-3) / 1e12
    a8 = w.causal_flops / (t8k * 1e-3) / 1e12
    a16 = w.causal_flops / (t16k * 1e-3) / 1e12
    tr8 = traffic_from_profiles(ATTN_SOURCES, f"attn_fwd_fp8:{name}")
    tr16 = traffic_from_profiles(ATTN_SOURCES, f"attn_fwd_bf16:{name}")
    # Secondary bounds of the FP8 kernel: one exponential and one e4m3
    # conversion per causal score, B*Hq*S^2/2 of each per launch, against the
    # per-SM rates above at the median SM clock sampled during the timed region.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks["sm_mhz"] if clocks else peaks.get("sm_max_mhz", 2070.0)
    n_scores = 0.5 * w.B * w.Hq * w.S * w.S
    secondary = {
        "scores_per_launch": n_scores, "sm_count": sms, "sm_mhz": mhz,
        "exp2": {"achieved_per_s": n_scores / (t8k * 1e-3), "peak_per_s": EX2_PER_CLK_SM * sms * mhz * 1e6,
                 "frac": n_scores / (t8k * 1e-3) / (EX2_PER_CLK_SM * sms * mhz * 1e6),
                 "peak_note": f"{EX2_PER_CLK_SM:g} ex2/clk/SM (measured) x SMs x sampled clock"},
        "e4m3_cvt": {"achieved_per_s": n_scores / (t8k * 1e-3),
                     "peak_per_s": E4M3_CVT_PER_CLK_SM * sms * mhz * 1e6,
                     "frac": n_scores / (t8k * 1e-3) / (E4M3_CVT_PER_CLK_SM * sms * mhz * 1e6),
                     "peak_note": f"{E4M3_CVT_PER_CLK_SM:g} converted elements/clk/SM (measured) x SMs x sampled clock"},
    }

    if rank != 0:
        return
    fp8_gemm = measure_fp8_gemm(dev)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(name, 12.0, had)
    line = {
        "metric": METRIC, "value": v8, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": t8, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3", "data": "synthetic (seeded Gaussian N(0,1), drawn in bf16, quantised per 128-token block)",
        "config": {"workload": name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "Dqk": w.Dqk, "Dv": w.Dv,
                   "path": ("fp8: quantise Q,K,V (1 launch) + fp8 causal attention with key ranges split "
                            "across CTAs (2 launches: chunks, combine)" if ws_bytes else
                            "fp8: quantise Q,K,V (1 launch) + fp8 causal attention (1 launch)"),
                   "split_key_ranges": bool(ws_bytes), "split_chunk_blocks": max(split_c, 0),
                   "hadamard": had, "parallelism": f"replicas x{world}",
                   "l2": "256 MiB flush between timed steps; inputs larger than L2"},
        "pct_of_peak": {"fp8_attention_kernel": a8 / fp8_peak, "fp8_step": v8 / world / fp8_peak,
                        "bf16_attention_kernel": a16 / peaks["bf16_tflops"],
                        "peak_source": f"{src} (fp8 = bf16 x {FP8_PER_BF16:g}, nominal ratio)"},
        "roofline": {"bound": "tensor", "achieved": a8, "peak": fp8_peak, "unit": UNIT, "frac": a8 / fp8_peak,
                     "traffic": tr8, "kernel": "attn_fwd_fp8",
                     "peak_note": (f"the fp8 peak is nominal: {src} bf16 burst {peaks['bf16_tflops']:g} TFLOP/s x "
                                   f"{FP8_PER_BF16:g}, the nominal fp8/bf16 tensor-core ratio; sustained-peak frac "
                                   f"{a8 / fp8_peak_sus:.3f}; measured_fp8_gemm: the library's e4m3 GEMM "
                                   f"timed in this run"),
                     "measured_fp8_gemm": None if fp8_gemm is None else {
                         "tflops": fp8_gemm, "frac": a8 / fp8_gemm,
                         "how": "cuBLASLt e4m3 8192^3 GEMM (torch._scaled_mm, bf16 out), best of 10 after the "
                                "timed steps"},
                     "ms_per_launch": t8k, "secondary": secondary},
        "bf16": {"value": v16, "unit": UNIT, "ms_per_step": t16, "dtype": "bf16", "gpu_launches": (2 if ws_bytes else 1) * K,
                 "roofline": {"bound": "tensor", "achieved": a16, "peak": peaks["bf16_tflops"], "unit": UNIT,
                              "frac": a16 / peaks["bf16_tflops"], "traffic": tr16, "kernel": "attn_fwd_bf16",
                              "peak_note": f"bf16 burst (of {src}); sustained-peak frac "
                                           f"{a16 / peaks['bf16_tflops_sustained']:.3f}"}},
        "gpu_launches": (3 if ws_bytes else 2) * K,
        **({"paged": paged} if paged is not None else {}),
        **({"graph": graph} if graph is not None else {}),
        **({"decode": decode} if decode is not None else {}),
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": None if cpu is None else {
            "value": cpu["value"], "unit": UNIT, "cores": cpu["cores"], "kind": "oracle", "sample": cpu["sample"]},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
