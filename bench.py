"""Benchmark of the sequence-parallel attention hot path on GB300.

One step is one training pass of the whole path over one batch of synthetic
input in natural sequence order, through the library's C ABI: usp_attn_fwd
then usp_attn_bwd with the natural-order flag. For windows, packed batches
and sequences up to 16K tokens (contiguous or zigzag) the tensor-core kernels
read and write the caller's tensors in place; otherwise the layout's extract
(fused with the Ulysses seq->head exchange when ud > 1) and restore run inside
the calls, and the backward reuses the forward's rank-major copies. Both
passes run the ring attention with the fused LSE merge; the backward adds
Delta and the ring return of dK/dV.
The metric is useful attention TFLOP/s (masked pairs not counted; backward
= 2.5x forward). The standalone tree/linear LSE merge, the layout permute and
the Ulysses exchange are timed on their own in the same run ("merge",
"permute").

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torchrun; every rank runs its own replica of the
workload (the virtual ranks already live in one GPU), scaling is weak.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("causal attn TFLOP/s (useful FLOPs) & % of GB300 BF16 dense peak, "
          "S=8K–128K")
DEFAULT_WORKLOAD = "usp_ud2_ring4_s8k"
DEFAULT_DECODE = "decode_gqa_b8_s128k_cp8"
# the e4m3 forward is reported on the shapes of the S = 32K zigzag workload
DEFAULT_FP8 = "sweep_zigzag_cp8_s32k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
KERNEL_SOURCES = {
    "attn_fwd_tc": "attn_fwd_tc.cu", "attn_bwd_tc": "attn_bwd_tc.cu",
    "attn_fwd_simt": "attn_simt.cu", "attn_bwd_dq_simt": "attn_simt.cu",
    "attn_bwd_dkdv_simt": "attn_simt.cu", "attn_bwd_preprocess": "attn_simt.cu",
    "permute_layout": "permute.cu", "permute_ulysses": "permute.cu",
    "merge_linear": "merge.cu", "merge_tree": "merge.cu",
    "attn_decode_split": "decode.cu", "attn_fwd_fp8": "attn_fwd_fp8.cu",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-gate", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(kernel: str):
    src = KERNEL_SOURCES.get(kernel)
    if not src:
        return None
    # the kernel's translation unit and every shared header it may include
    csrc = os.path.join(ROOT, "sequence_long_context_gb300", "csrc")
    headers = sorted(f for f in os.listdir(csrc) if f.endswith((".cuh", ".h")))
    h = hashlib.sha256()
    for name in [src] + headers:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since the capture; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    want = source_hash(kernel)
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if not line.startswith("#") and len(parts) == 4 and parts[0] == kernel and parts[1] == workload \
                    and parts[2] == want:
                return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = f"/tmp/usp_clocks_{os.getpid()}.csv"

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def oracle_sample(w, seed: int, budget_s: float):
    """Time the CPU oracle (as it stands) on a bounded sample of workload w:
    forward + backward of one (batch 0, head 0) pair, on the longest causal
    prefix of the sequence that fits the time budget. Returns
    (useful TFLOP/s, seconds, sample description, threads)."""
    import numpy as np
    import torch

    from oracle import attention
    from sequence_long_context_gb300 import flops
    from sequence_long_context_gb300.workloads import make_inputs

    one = w.replace(B=1, Hq=1, Hkv=1, ud=1, varlen=False)
    x = make_inputs(one.replace(S=w.S), seed=seed, with_grad=w.backward)
    S = w.S
    while True:
        # estimate from a quarter-length run, scale by the pair count ratio
        t0 = time.perf_counter()
        s_small = max(64, S // 4)
        sl = {k: v[:, :s_small] for k, v in x.items() if k != "cu_seqlens"}
        attention.attn_fwd(sl["q"], sl["k"], sl["v"], w.scale, w.causal, w.window, w.sink_tokens)
        t_small = time.perf_counter() - t0
        est = t_small * (S / s_small) ** 2 * (3.5 if w.backward else 1.0)
        if est <= budget_s or S <= 256:
            break
        S //= 2
    sl = {k: v[:, :S] for k, v in x.items() if k != "cu_seqlens"}
    t0 = time.perf_counter()
    attention.attn_fwd(sl["q"], sl["k"], sl["v"], w.scale, w.causal, w.window, w.sink_tokens)
    if w.backward:
        attention.attn_bwd(sl["q"], sl["k"], sl["v"], sl["dout"], w.scale, w.causal,
                           w.window, w.sink_tokens)
    dt = time.perf_counter() - t0
    f = flops.attention_flops(one.replace(S=S))["total"]
    threads = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info
        blas = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        threads = min(threads, blas) if blas else threads
    except Exception:
        pass
    desc = (f"fp64 NumPy oracle, batch 0 head 0 of {w.name}, causal prefix "
            f"S={S} of {w.S}, {'fwd+bwd' if w.backward else 'fwd'} "
            f"(1 of {w.B * w.Hq if not w.varlen else w.Hq} (batch, head) pairs)")
    return f / dt / 1e12, dt, desc, threads


def workload_config(w, total_flop: float, world: int) -> dict:
    """The `config` object both arms print for workload w."""
    return {"workload": w.name, "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv,
            "D": w.D, "layout": w.layout, "cp": w.cp, "ulysses": w.ud,
            "causal": w.causal, "window": w.window, "sink_tokens": w.sink_tokens,
            "backward": w.backward,
            "useful_tflop_per_step": total_flop / 1e12,
            "parallelism": f"virtual ring cp={w.cp} x ulysses {w.ud} on one GPU; "
                           f"{world} replica(s)",
            "l2": "no flush: step inputs larger than L2"}


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time (the job ends when its last rank does)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_rank_step: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return flop_per_rank_step * world / (ms * 1e-3) / 1e12


def run_reference(args):
    """The oracle timed on the host cores, as the reference arm."""
    import numpy as np  # noqa: F401

    from sequence_long_context_gb300 import flops
    from sequence_long_context_gb300.workloads import WORKLOADS, draw_cu_seqlens

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    cu = draw_cu_seqlens(w.S, w.seg_lo, w.seg_hi, args.seed) if w.varlen else None
    total = flops.attention_flops(w, cu.tolist() if cu is not None else None)["total"]
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    vals, times = [], []
    desc, thr = "", 0
    for i in range(args.warmup + args.steps):
        v, dt, desc, thr = oracle_sample(w, args.seed, budget)
        if i >= args.warmup:
            vals.append(v)
            times.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, total, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def make_step(usp, w, x, cu_dev, keep=None):
    """One training pass of workload w over the natural-order inputs `inp`:
    forward and backward on natural-order tensors (the layout's extract and
    restore inside the calls, fused with the Ulysses exchange), the backward
    reusing the forward's rank-major copies of q, k, v, out from the shared
    workspace. Returns the natural-order results [O(, dQ, dK, dV)]; `keep`
    (a dict), if given, receives each step's LSE under "lse"."""
    kw = dict(causal=w.causal, window=w.window, sink_tokens=w.sink_tokens,
              cu_seqlens=cu_dev, cp=w.cp, ud=w.ud, layout=w.layout, natural=True)
    # one workspace for the forward and the backward of every step
    ws = usp.attn_workspace(x["q"], x["k"], cu_seqlens=cu_dev, cp=w.cp, ud=w.ud,
                            natural=True)

    def fwd(inp):
        out, lse = usp.attn_forward(inp["q"], inp["k"], inp["v"], workspace=ws, **kw)
        if keep is not None:
            keep["lse"] = lse
        return out, lse

    def bwd(inp, out, lse):
        return list(usp.attn_backward(inp["q"], inp["k"], inp["v"], out, lse, inp["dout"],
                                      workspace=ws, saved_exchange=True, **kw))

    def step(inp):
        out, lse = fwd(inp)
        res = [out]
        if w.backward:
            res += bwd(inp, out, lse)
        return res

    # the two halves, for callers that interleave copies with them
    step.fwd, step.bwd = fwd, bwd
    return step


def rank_major_kernels(usp, torch, w, x, cu_dev, F, steps, peak):
    """The step's attention kernels on rank-major copies of the inputs (the
    layout's extract done once, outside the timed loop; the Ulysses exchange
    inside the calls as usual): each kernel's average CUDA-event time and
    useful TFLOP/s against `peak`. The natural-order step above has the same
    kernels read the caller's tensors in place."""
    kw = dict(causal=w.causal, window=w.window, sink_tokens=w.sink_tokens,
              cu_seqlens=cu_dev, cp=w.cp, ud=w.ud, layout=w.layout)
    names = ["q", "k", "v"] + (["dout"] if w.backward else [])
    xp = {n: usp.permute(x[n], "extract", w.layout, w.cp) for n in names}
    ws = usp.attn_workspace(xp["q"], xp["k"], cu_seqlens=cu_dev, cp=w.cp, ud=w.ud)

    def run():
        o, l = usp.attn_forward(xp["q"], xp["k"], xp["v"], workspace=ws, **kw)
        if w.backward:
            usp.attn_backward(xp["q"], xp["k"], xp["v"], o, l, xp["dout"], workspace=ws,
                              saved_exchange=True, **kw)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    usp.usp_profile_enable(True)
    for _ in range(steps):
        run()
    torch.cuda.synchronize()
    usp.usp_profile_enable(False)
    ks = usp.usp_profile_read()
    res = {"inputs": "rank-major copies (extract outside the timed loop)", "steps": steps}
    for part, kname, work in (("fwd", "attn_fwd_tc", F["fwd"]), ("bwd", "attn_bwd_tc", F["bwd"])):
        n, tot = ks.get(kname, (0, 0.0))
        if n:
            avg = tot / n
            ach = work / (avg * 1e-3) / 1e12
            res[part] = {"kernel": kname, "avg_ms": avg, "achieved": ach, "frac": ach / peak}
    del xp, ws
    return res


def gate_point(usp, flops, torch, name, dev, seed, steps, warmup, pk, timed):
    """Forward and backward tensor-core kernels of one zigzag sweep point,
    each kernel's average CUDA-event time over `steps` training steps and its
    useful TFLOP/s against the bf16 peak (burst when the timed region is
    short, sustained beyond 2 s; both fractions are reported)."""
    from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    x = make_inputs(w, seed=seed, device=str(dev))
    F = flops.attention_flops(w)
    step = make_step(usp, w, x, None)
    for _ in range(warmup):
        step(x)
    torch.cuda.synchronize()
    usp.usp_profile_enable(True)
    ms = timed(lambda: step(x), steps)
    usp.usp_profile_enable(False)
    ks = usp.usp_profile_read()
    region_s = ms * steps / 1e3
    peak = pk["bf16_tflops_sustained"] if region_s > 2.0 else pk["bf16_tflops"]
    res = {"workload": name, "S": w.S, "step_ms": ms, "steps": steps,
           "step_tflops": F["total"] / (ms * 1e-3) / 1e12,
           "peak_used": "bf16_tflops_sustained" if region_s > 2.0 else "bf16_tflops"}
    for part, kname, work in (("fwd", "attn_fwd_tc", F["fwd"]), ("bwd", "attn_bwd_tc", F["bwd"])):
        n, tot = ks.get(kname, (0, 0.0))
        if not n:
            res[part] = {"error": f"{kname} did not run"}
            continue
        avg = tot / n
        ach = work / (avg * 1e-3) / 1e12
        res[part] = {"kernel": kname, "avg_ms": avg, "useful_tflop": work / 1e12,
                     "achieved": ach, "frac": ach / peak,
                     "frac_of_burst": ach / pk["bf16_tflops"],
                     "frac_of_sustained": ach / pk["bf16_tflops_sustained"]}
    del x, step
    torch.cuda.empty_cache()
    return res


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    import __graft_entry__
    import sequence_long_context_gb300 as usp
    from sequence_long_context_gb300 import flops
    from sequence_long_context_gb300.workloads import WORKLOADS, make_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build() if rank == 0 else None
    if world > 1:
        dist.barrier()
        __graft_entry__.build()

    w = WORKLOADS[args.workload]
    x = make_inputs(w, seed=args.seed + rank, device=str(dev))
    cu = x.get("cu_seqlens")
    cu_dev = cu.to(dev) if cu is not None else None
    F = flops.attention_flops(w, cu.tolist() if cu is not None else None)
    names = ["q", "k", "v"] + (["dout"] if w.backward else [])

    step = make_step(usp, w, x, cu_dev)

    def timed(fn, n):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(n):
            fn()
        b.record(st)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return max_over_ranks(a.elapsed_time(b) / n, world, dev)

    for _ in range(args.warmup):
        step(x)
    torch.cuda.synchronize()

    # device-resident timed region (inputs 4 x 128 MiB > L2: no flush needed)
    usp.usp_profile_enable(True)
    l0 = usp.usp_launch_count()
    with ClockSampler(local) as clk:
        ms = timed(lambda: step(x), args.steps)
    launches = (usp.usp_launch_count() - l0) // args.steps
    usp.usp_profile_enable(False)
    kstats = usp.usp_profile_read()
    clocks = clk.summary()

    pk, pk_src = peaks()
    timed_s = ms * args.steps / 1e3
    tensor_peak = pk["bf16_tflops_sustained"] if timed_s > 2.0 else pk["bf16_tflops"]
    tensor_peak_name = "bf16_tflops_sustained" if timed_s > 2.0 else "bf16_tflops"
    kernels = {}
    for name, (n, tot) in sorted(kstats.items()):
        avg = tot / max(n, 1)
        kernels[name] = {"launches_per_step": n / args.steps, "avg_ms": avg,
                         "share": tot / max(1e-9, sum(t for _, t in kstats.values()))}
    # dominant kernel and its algorithmic work per launch
    fwd_k = [k for k in kernels if k.startswith("attn_fwd")]
    # the backward's contraction kernels (not its HBM-bound preprocess/convert)
    bwd_k = [k for k in kernels if k.startswith("attn_bwd")
             and "preprocess" not in k and "convert" not in k]
    cand = []
    for k in fwd_k:
        cand.append((kstats[k][1], k, F["fwd"]))
    if bwd_k:
        tot_bwd = sum(kstats[k][1] for k in bwd_k)
        nb = kstats[bwd_k[0]][0]
        cand.append((tot_bwd, "+".join(bwd_k), F["bwd"]))
    dom = max(cand) if cand else None
    roofline = None
    if dom:
        tot_ms, name, work = dom
        n_launch = kstats[name.split("+")[0]][0]
        avg_ms = tot_ms / max(n_launch, 1)
        achieved = work / (avg_ms * 1e-3) / 1e12
        roofline = {"kernel": name, "bound": "tensor", "achieved": achieved,
                    "peak": tensor_peak, "unit": "TFLOP/s",
                    "frac": achieved / tensor_peak,
                    "traffic": traffic_for(name.split("+")[0], w.name),
                    "peak_source": f"{pk_src} {tensor_peak_name}",
                    "work_per_launch": work, "avg_ms": avg_ms}
    # HBM kernels: algorithmic bytes per launch
    elem = 2 if w.dtype == "bf16" else 4
    q_bytes = (1 if w.varlen else w.B) * w.S * w.Hq * w.D * elem
    kv_bytes = (1 if w.varlen else w.B) * w.S * w.Hkv * w.D * elem
    # tensor bytes moved per step (each byte is read once and written once):
    # q, k, v in and O out in the forward; the backward reuses the forward's
    # copies (saved_exchange) and moves dO in and dQ, dK, dV out. With
    # Ulysses the layout's extract / restore ride along with the exchange
    # (permute_ulysses); without, they are the layout permutes.
    fam = "permute_ulysses" if w.ud > 1 else "permute_layout"
    moved = {fam: (4 if w.backward else 2) * (q_bytes + kv_bytes)}
    for k, mv in moved.items():
        if k in kernels:
            per_launch = 2 * mv / kernels[k]["launches_per_step"]
            gbs = per_launch / (kernels[k]["avg_ms"] * 1e-3) / 1e9
            kernels[k].update({"bytes_per_launch": per_launch, "GB_s": gbs,
                               "frac_hbm": gbs / pk["hbm_gbs"]})

    # the same attention kernels on rank-major copies of the step's inputs
    try:
        rank_major = rank_major_kernels(usp, torch, w, x, cu_dev, F, args.steps, tensor_peak)
    except Exception as e:  # report, do not hide
        rank_major = {"error": repr(e)}
    torch.cuda.empty_cache()

    # standalone merge on its own workload (4 partials of B*S*Hq rows)
    merge_res = None
    try:
        rows = (1 if w.varlen else w.B) * w.S * w.Hq
        n = max(2, min(w.cp, 8))
        g = torch.Generator(device=dev).manual_seed(7)
        op = torch.randn(n, rows, w.D, device=dev, generator=g)
        lp = torch.randn(n, rows, device=dev, generator=g)
        oo = torch.empty(rows, w.D, dtype=torch.bfloat16, device=dev)
        lo = torch.empty(rows, device=dev)
        for tree in (0, 1):
            fn = lambda: usp.usp_merge_partials(op, lp, n, rows, w.D, tree, oo, torch.bfloat16, lo)  # noqa: E731
            for _ in range(3):
                fn()
            mms = timed(fn, 10)
            by = n * rows * (4 * w.D + 4) + rows * (2 * w.D + 4)
            gbs = by / (mms * 1e-3) / 1e9
            merge_res = merge_res or {}
            merge_res["tree" if tree else "linear"] = {
                "n": n, "rows": rows, "D": w.D, "ms": mms, "bytes": by, "GB_s": gbs,
                "frac_hbm": gbs / pk["hbm_gbs"]}
        del op, lp
    except Exception as e:  # report, do not hide
        merge_res = {"error": repr(e)}

    # standalone layout permute and Ulysses exchange on the step's q tensor
    # (the natural-order step above runs neither: its kernels read the
    # caller's tensors in place); both are HBM-bound copies, 2 bytes moved
    # per byte of the tensor, and the tensor exceeds L2
    permute_res = None
    try:
        src = x["q"]
        dst = torch.empty_like(src)
        Bp = 1 if w.varlen else w.B
        Hp, Sp = w.Hq, w.S
        by = 2 * src.numel() * src.element_size()
        kinds = [("extract", 1)] + ([("seq2head", w.ud)] if w.ud > 1 else [])
        for kind, udp in kinds:
            fn = lambda: usp.usp_permute(src, dst, kind, w.layout, Bp, Sp, Hp, w.D, w.cp, udp,  # noqa: E731
                                         src.element_size())
            for _ in range(3):
                fn()
            pms = timed(fn, 10)
            gbs = by / (pms * 1e-3) / 1e9
            permute_res = permute_res or {}
            permute_res[kind] = {"layout": w.layout, "cp": w.cp, "ud": udp,
                                 "tensor_bytes": src.numel() * src.element_size(),
                                 "ms": pms, "bytes": by, "GB_s": gbs,
                                 "frac_hbm": gbs / pk["hbm_gbs"]}
        del dst
    except Exception as e:  # report, do not hide
        permute_res = {"error": repr(e)}

    # decode step (split-KV partials over the sharded cache + tree merge) on
    # its own workload: HBM-bound, reported against the copy bandwidth
    decode_res = None
    if not args.no_decode:
        try:
            from sequence_long_context_gb300.workloads import (DECODE_WORKLOADS,
                                                               make_decode_inputs)
            dw = DECODE_WORKLOADS[DEFAULT_DECODE]
            dx = make_decode_inputs(dw, seed=args.seed, device=str(dev))
            dfn = lambda: usp.attn_decode(dx["q"], dx["k"], dx["v"], causal=dw.causal,  # noqa: E731
                                          cp=dw.cp, splits=dw.splits, tree_order=True)
            for _ in range(3):
                dfn()
            usp.usp_profile_enable(True)
            dms = timed(dfn, 10)
            usp.usp_profile_enable(False)
            dk = usp.usp_profile_read()
            rows = dw.B * dw.Tq * dw.Hq
            n_part = dw.cp * dw.splits
            q_bytes = rows * dw.D * 2
            part_bytes = n_part * rows * (dw.D + 1) * 4
            split_bytes = dw.kv_bytes + q_bytes + part_bytes
            step_bytes = split_bytes + part_bytes + rows * (dw.D * 2 + 4)
            sp = dk.get("attn_decode_split")
            split_ms = sp[1] / sp[0] if sp else None
            decode_res = {
                "workload": dw.name, "B": dw.B, "Tq": dw.Tq, "S": dw.S, "Hq": dw.Hq,
                "Hkv": dw.Hkv, "D": dw.D, "cp": dw.cp, "splits": dw.splits,
                "step_ms": dms, "step_GB_s": step_bytes / (dms * 1e-3) / 1e9,
                "step_frac_hbm": step_bytes / (dms * 1e-3) / 1e9 / pk["hbm_gbs"],
                "split_kernel_ms": split_ms,
                "split_GB_s": split_bytes / (split_ms * 1e-3) / 1e9 if split_ms else None,
                "split_frac_hbm": (split_bytes / (split_ms * 1e-3) / 1e9 / pk["hbm_gbs"]
                                   if split_ms else None),
                "algorithmic_bytes": step_bytes,
                "traffic": traffic_for("attn_decode_split", dw.name)}
            del dx
        except Exception as e:  # report, do not hide
            decode_res = {"error": repr(e)}

    # end to end: every step uploads its inputs from pinned host memory and
    # reads its results back into pinned host memory. The copies run on their
    # own streams, double-buffered: step i+1's upload and step i-1's readback
    # overlap step i's kernels, as a training loop with a prefetching loader
    # runs. The forward starts once q, k, v are in (dout may still be on its
    # way) and out goes back once the forward is done. The first upload and
    # the last readback are inside the timed region.
    e2e = None
    if not args.no_e2e:
        host = {n: x[n].cpu().pin_memory() for n in names}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        # two copy streams each way: every tensor's copy is one cudaMemcpyAsync
        # and they alternate between the streams (more than one copy engine)
        ups = [torch.cuda.Stream(device=dev) for _ in range(2)]
        downs = [torch.cuda.Stream(device=dev) for _ in range(2)]
        slots = [{n: torch.empty_like(x[n]) for n in names} for _ in range(2)]
        outs_host = [None, None]

        def e2e_run(n):
            cs = torch.cuda.current_stream()
            ready = [[], []]
            freed = [None, None]
            # the host runs at most two steps ahead of the readbacks, so the
            # allocator recycles the same blocks (no allocation, which may
            # synchronize the device, inside the timed region)
            read_back = []

            def upload(i):
                # one event per tensor: the forward waits for q, k, v only,
                # the backward for dout too
                s = i % 2
                ready[s] = {}
                for j, nm in enumerate(names):
                    u = ups[j % len(ups)]
                    if freed[s] is not None:
                        u.wait_event(freed[s])
                    with torch.cuda.stream(u):
                        slots[s][nm].copy_(host[nm], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(u)
                    ready[s][nm] = ev

            for u in ups:
                u.wait_stream(cs)
            upload(0)
            for i in range(n):
                s = i % 2
                if i >= 2:
                    for ev in read_back[i - 2]:
                        ev.synchronize()
                if i + 1 < n:
                    upload(i + 1)
                for nm in ("q", "k", "v"):
                    cs.wait_event(ready[s][nm])
                out, lse = step.fwd(slots[s])
                fdone = torch.cuda.Event()
                fdone.record(cs)
                outs = [out]
                if w.backward:
                    cs.wait_event(ready[s]["dout"])
                    outs += step.bwd(slots[s], out, lse)
                done = torch.cuda.Event()
                done.record(cs)
                freed[s] = done
                if outs_host[s] is None:
                    outs_host[s] = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
                                    for o in outs]
                # the output's readback starts once the forward is done, the
                # gradients' once the backward is
                for j, (hb, o) in enumerate(zip(outs_host[s], outs)):
                    d = downs[j % len(downs)]
                    d.wait_event(fdone if j == 0 else done)
                    with torch.cuda.stream(d):
                        o.record_stream(d)
                        hb.copy_(o, non_blocking=True)
                rbs = []
                for d in downs:
                    ev = torch.cuda.Event()
                    ev.record(d)
                    rbs.append(ev)
                read_back.append(rbs)
                del outs
            for d in downs:
                cs.wait_stream(d)

        e2e_run(4)
        n_e2e = max(3, min(2 * args.steps, 20))
        ems = timed(lambda: e2e_run(n_e2e), 1) / n_e2e
        d2h = sum(t.numel() * t.element_size() for t in outs_host[0])
        e2e = {"value": job_tflops(F["total"], world, ems), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems,
               "steps": n_e2e,
               "copies": "double-buffered, two H2D and two D2H streams; the forward waits "
                         "for q, k, v only, out is read back once the forward is done"}

    # fp8 (E4M3) forward: the inputs are quantized once, outside the timed
    # region; the forward (V transpose + attention) runs on resident codes.
    # Tensor-bound: reported against the measured bf16 peak times the
    # nominal e4m3 / bf16 rate ratio (4.5 / 2.25 PFLOP/s dense).
    fp8_res = None
    if not args.no_fp8:
        try:
            fw = WORKLOADS[DEFAULT_FP8]
            fx = make_inputs(fw, seed=args.seed, device=str(dev))
            codes = []
            for n in "qkv":
                t = usp.permute(fx[n], "extract", fw.layout, fw.cp)
                inv = 256.0 / float(t.float().abs().max())
                codes.append((usp.quantize_e4m3(t, inv), 1.0 / inv))
            del fx
            (q8, qd), (k8, kd), (v8, vd) = codes
            fws = torch.empty(usp.usp_attn_fwd_fp8_workspace_size(
                fw.B, fw.S, fw.Hq, fw.Hkv, fw.D, fw.cp, fw.ud), dtype=torch.uint8, device=dev)
            ffn = lambda: usp.attn_forward_fp8(  # noqa: E731
                q8, k8, v8, qd, kd, vd, causal=fw.causal, window=fw.window,
                sink_tokens=fw.sink_tokens, cp=fw.cp, ud=fw.ud, layout=fw.layout,
                workspace=fws)
            for _ in range(3):
                ffn()
            usp.usp_profile_enable(True)
            fms = timed(ffn, 10)
            usp.usp_profile_enable(False)
            fk = usp.usp_profile_read()
            ff = flops.attention_flops(fw)["fwd"]
            fp8_peak = 2.0 * pk["bf16_tflops"]
            att = fk.get("attn_fwd_fp8")
            att_ms = att[1] / att[0] if att else None
            fp8_res = {
                "workload": fw.name, "B": fw.B, "S": fw.S, "Hq": fw.Hq, "Hkv": fw.Hkv,
                "D": fw.D, "cp": fw.cp, "layout": fw.layout, "causal": fw.causal,
                "dtype": "e4m3", "forward_ms": fms,
                "forward_tflops": ff / (fms * 1e-3) / 1e12,
                "kernel_ms": att_ms,
                "roofline": {"kernel": "attn_fwd_fp8", "bound": "tensor",
                             "achieved": ff / (att_ms * 1e-3) / 1e12 if att_ms else None,
                             "peak": fp8_peak, "unit": "TFLOP/s",
                             "frac": ff / (att_ms * 1e-3) / 1e12 / fp8_peak if att_ms else None,
                             "peak_source": "measured bf16_tflops x 2 (nominal e4m3/bf16 ratio)",
                             "traffic": traffic_for("attn_fwd_fp8", fw.name)},
                "kernels": {k: {"launches_per_step": v[0] / 10, "avg_ms": v[1] / v[0]}
                            for k, v in fk.items()}}
            del codes, q8, k8, v8, fws
        except Exception as e:  # report, do not hide
            fp8_res = {"error": repr(e)}

    # the throughput gate: the zigzag causal sweep (B=1, 32/8 heads, D=128,
    # cp=8) at S = 32K, and the end of the metric's range at S = 128K. It runs
    # after every other measurement: its S = 128K steps keep the GPU at full
    # power for seconds, and the short measurements timed after them ran
    # about 1 % slower.
    gate = None
    if not args.no_gate:
        gate = {"targets": {"fwd_frac": 0.60, "bwd_frac": 0.45, "at": "sweep_zigzag_cp8_s32k"}}
        for gname, gsteps in (("sweep_zigzag_cp8_s32k", 10), ("sweep_zigzag_cp8_s128k", 2)):
            try:
                gate[gname] = gate_point(usp, flops, torch, gname, dev, args.seed, gsteps, 3,
                                         peaks()[0], timed)
            except Exception as e:  # report, do not hide
                gate[gname] = {"error": repr(e)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, desc, thr = oracle_sample(w, args.seed, 20.0)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": desc, "seconds": dt}

    value = job_tflops(F["total"], world, ms)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": workload_config(w, F["total"], world),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(launches * args.steps), "clocks": clocks,
        "gate": gate, "kernels": kernels, "kernels_rank_major": rank_major,
        "merge": merge_res, "permute": permute_res, "decode": decode_res,
        "fp8": fp8_res,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
