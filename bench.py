"""Benchmark: one training step of the SwiGLU MLP block (forward + backward) at the
pages' target shape M=11136, D=3584, H=14336, Dout=3584, bf16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  `value` is whole-step TFLOP/s (fwd 6MDH + bwd
12MDH flops per step, summed over ranks) from CUDA events around K steps whose
inputs are resident in HBM (468 MB of inputs per step, larger than the 129 MB
L2, so no flush is needed).  Per-kernel durations come from the library's launch
trace (events around every kernel, on its stream) over the same timed region.
`e2e` repeats the step through the public API with the inputs copied in from
pinned host memory and the outputs copied back every step (wall clock around
the whole run; the copies of neighbouring steps overlap a step's compute, see
bwd_gemm_epilogue_gb300/pipeline.py).  `cpu_baseline` times
the fp64 CPU oracle on a bounded sample of the same workload.

Multi-GPU: the block does not shard here; each rank runs an independent replica
(weak scaling), ranks meet only at the barriers around the timed region.

--impl reference times the CPU oracle (the only reference this method has)
on the host cores, on a bounded per-step sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "target"
# The pages' own number for this workload: drop-h path, full fwd+bwd 7.3664 ms on a B200
# (Drop-H report, single-MLP target-shape table) -> 10299.0 GF / 7.3664 ms.
PAGES_FULL_MS_B200 = 7.3664


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["target", "prefill", "decode", "stack4", "moe8", "moe64",
                                           "fp8_target", "fp8_prefill", "fp8_decode", "tp2"],
                    default="target",
                    help="target: the block at the pages' target shape (the headline line); "
                         "prefill / decode: the 4096- and 16-token LLaMA-7B-shaped blocks; "
                         "stack4: four target blocks trained end to end (with memory); "
                         "moe8 / moe64: mixture-of-experts layers, grouped launches over the experts; "
                         "fp8_*: the FP8 forward (E4M3, quantising epilogue) at the target / prefill / "
                         "decode shapes, with the bf16 forward timed beside it; "
                         "tp2: one rank's shard of the target block split over two tensor-parallel "
                         "ranks (its chunked forward and evented backward against the same shard in "
                         "one piece; the reductions need a second GPU)")
    ap.add_argument("--residual", action="store_true",
                    help="time the residual block y = x + MLP(x) (residual-add epilogues; D == Dout)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=25.0, help="CPU time the oracle sample is sized for (it tends to finish in about 60 %% of it)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """The slowest rank's value (timings are reported as the max over ranks)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every rank runs its own replica (weak scaling)."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


# ----------------------------------------------------------------------------- clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(gpu_index)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = sorted({n for _, _, flags in rows for n, f in zip(names, flags) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": seen, "samples": len(rows)}


# ----------------------------------------------------------------------------- oracle sample

def oracle_sample(s, x, W1, W2, dy, preact, n_rows: int, n_cols: int, seed: int = 0):
    """Run the CPU oracle on a sample of the workload: forward and row-wise backward
    for n_rows token rows, weight gradients for n_cols hidden columns.
    Returns (seconds, flops, threads)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    rows = rng.choice(s.M, size=n_rows, replace=False)
    cols = rng.choice(s.H, size=n_cols, replace=False)
    t0 = time.perf_counter()
    if n_rows:
        oracle.fwd(x, W1, W2, rows=rows)
        oracle.bwd_rows(W1, W2, preact, dy, rows=rows)
    if n_cols:
        oracle.bwd_cols(x, W2, preact, dy, cols=cols)
    dt = time.perf_counter() - t0
    per_row = 2 * (s.D * 2 * s.H + s.H * s.Dout) + 2 * (s.Dout * s.H + 2 * s.H * s.D)
    per_col = 2 * s.M * s.Dout * 2 + 2 * 2 * s.M * s.D
    return dt, n_rows * per_row + n_cols * per_col, oracle.num_threads()


def cpu_baseline(s, x, W1, W2, dy, preact, seconds: float):
    """Size a sample to about `seconds` of CPU time (three quarters token rows, one quarter
    hidden columns) from a calibration on as many rows and columns as the oracle has
    threads (it runs rows, or columns, in parallel), then time it."""
    import oracle
    nt = max(1, oracle.num_threads())
    dt_r, f_r, _ = oracle_sample(s, x, W1, W2, dy, preact, nt, 0, seed=99)
    dt_c, f_c, _ = oracle_sample(s, x, W1, W2, dy, preact, 0, nt, seed=98)
    n_rows = max(1, int(0.75 * seconds / max(dt_r / nt, 1e-6)))
    n_cols = max(1, int(0.25 * seconds / max(dt_c / nt, 1e-6)))
    dt, flops, threads = oracle_sample(s, x, W1, W2, dy, preact, min(n_rows, s.M), min(n_cols, s.H))
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"fwd + row-wise bwd for {min(n_rows, s.M)} of {s.M} token rows and weight grads for "
                      f"{min(n_cols, s.H)} of {s.H} hidden columns of the target block ({flops / 1e9:.1f} GFLOP in "
                      f"{dt:.1f} s, fp64)"}


# ----------------------------------------------------------------------------- profile summary

def kernel_source_hash() -> str:
    """Hash of the kernel sources with runs of white space collapsed: a change of
    formatting keeps the counters taken before it, any other edit voids them."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bwd_gemm_epilogue_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            text = open(os.path.join(csrc, name), "rb").read()
            h.update(name.encode() + b"\0" + re.sub(rb"\s+", b" ", text).strip() + b"\0")
    return h.hexdigest()[:16]


def measured_traffic(kind: str, workload: str = "target"):
    """DRAM bytes per launch of `kind` from the committed ncu summary of the target
    step, or None for another workload or when the kernel sources changed since."""
    if workload != "target":
        return None
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        data = json.load(open(path))
    except (OSError, ValueError):
        return None
    if data.get("source_hash") != kernel_source_hash():
        return None
    k = data.get("kernels", {}).get(kind)
    return None if k is None else k.get("dram_bytes_per_launch")


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# The sustained bf16 figure is cuBLAS back to back for seconds under the power cap; a
# timed region shorter than this runs at burst clocks, so its kernels are held to the
# burst figure.
SUSTAINED_AFTER_S = 2.0


def tensor_peak(pk: dict, pk_src: str, region_s: float):
    """(peak TFLOP/s, description) for kernels timed inside a region of `region_s` seconds."""
    if region_s >= SUSTAINED_AFTER_S:
        return pk["bf16_tflops_sustained"], (f"{pk_src} bf16_tflops_sustained (timed region {region_s:.2f} s, "
                                             f">= {SUSTAINED_AFTER_S:.0f} s)")
    return pk["bf16_tflops"], f"{pk_src} bf16_tflops burst (timed region {region_s:.2f} s, < {SUSTAINED_AFTER_S:.0f} s)"


# ----------------------------------------------------------------------------- our arm

def write_ceiling_gbs(nbytes: int, dev) -> float:
    """HBM bandwidth of a write-only stream of `nbytes` (torch fill_ of a bf16 buffer),
    best of 5 repetitions of 10 fills, CUDA events."""
    import torch

    t = torch.empty(max(1, nbytes // 2), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        t.fill_(1.0)
    best = float("inf")
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            t.fill_(1.0)
        e1.record()
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1) / 10)
    return t.numel() * 2 / (best * 1e-3) / 1e9


def block_memory_mib(M: int, D: int, H: int, Dout: int, bwd_workspace_bytes: int) -> dict:
    """Device memory of one block beyond its inputs (x, W1, W2, dy), as the pages' memory
    table counts it: after the forward the saved preact and the output y; at the
    backward's peak also the backward workspace (h, grad_preact) and dx, dW1, dW2."""
    mib = 2 ** 20
    after_fwd = (M * 2 * H + M * Dout) * 2
    peak = after_fwd + bwd_workspace_bytes + (M * D + 2 * H * D + Dout * H) * 2
    return {"after_fwd": round(after_fwd / mib, 1), "bwd_peak": round(peak / mib, 1),
            "pages_drop_h_b200": {"after_fwd": 686.1, "peak": 1905.1}}


def graph_replay_timing(step, dev, K: int, step_flops: float):
    """The same step captured once into a CUDA graph and replayed K times: the launch
    gaps between the step's short kernels go away (the decode step is launch-bound)."""
    import torch

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for _ in range(3):
            step()
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        g.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / K
    return {"ms_per_step": round(ms, 4), "tflops": round(step_flops / (ms * 1e-3) / 1e12, 1),
            "what": "one fwd+bwd step captured into a CUDA graph, replayed back to back"}


def eager_comparison(step, x, W1, W2, dy, step_flops, dev, blocks: int = 4, n: int = 10):
    """The pages' unfused drop-h step on the same GPU: torch.matmul (cuBLAS) for the five
    GEMMs and eager element-wise kernels for the SwiGLU forward/backward, grad_h written to
    and read back from HBM.  Timed in alternating blocks with this library's step (context
    for the fused path, not a product path)."""
    import torch
    import torch.nn.functional as F

    H = W2.shape[1]

    def eager_step():
        pre = x @ W1.t()
        left, gate = pre[:, :H], pre[:, H:]
        h = left * F.silu(gate)
        _ = h @ W2.t()
        gh = dy @ W2
        sig = torch.sigmoid(gate)
        silu = gate * sig
        gp = torch.cat([gh * silu, gh * left * (sig + silu * (1 - sig))], dim=1)
        h2 = left * silu
        _ = gp @ W1
        _ = gp.t() @ x
        _ = dy.t() @ h2

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    for _ in range(3):
        eager_step()
        step()
    torch.cuda.synchronize(dev)
    ours, base = [], []
    for b in range(blocks):
        for name in (("ours", "eager") if b % 2 == 0 else ("eager", "ours")):
            (ours if name == "ours" else base).append(timed(step if name == "ours" else eager_step))
    o, e = statistics.median(ours), statistics.median(base)
    return {"ms_per_step": round(e, 4), "tflops": round(step_flops / (e * 1e-3) / 1e12, 1),
            "ours_ms_per_step_same_blocks": round(o, 4), "speedup": round(e / o, 3),
            "what": "torch.matmul (cuBLAS) GEMMs + eager element-wise SwiGLU forward/backward (grad_h through HBM), "
                    "the pages' unfused drop-h step, alternating blocks of 10 steps with this library's step"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    from bwd_gemm_epilogue_gb300 import binding, ledger, workloads

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws_n > 1 else 0)
    torch.cuda.set_device(dev)

    wl = args.workload
    s, x_h, W1_h, W2_h, dy_h = workloads.make_block(wl)
    M, D, H, Do = s.M, s.D, s.H, s.Dout
    flops = ledger.gemm_flops(M, D, H, Do)

    x, W1, W2, dy = (t.to(dev) for t in (x_h, W1_h, W2_h, dy_h))
    preact = torch.empty(M, 2 * H, dtype=torch.bfloat16, device=dev)
    y = torch.empty(M, Do, dtype=torch.bfloat16, device=dev)
    dx = torch.empty(M, D, dtype=torch.bfloat16, device=dev)
    dW1 = torch.empty(2 * H, D, dtype=torch.bfloat16, device=dev)
    dW2 = torch.empty(Do, H, dtype=torch.bfloat16, device=dev)
    ws_f = torch.empty(binding.swiglu_mlp_fwd_workspace_size(M, D, H, Do), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(binding.swiglu_mlp_bwd_workspace_size(M, D, H, Do), dtype=torch.uint8, device=dev)

    def step():
        binding.swiglu_mlp_fwd(x, W1, W2, preact, y, ws_f, residual=args.residual)
        binding.swiglu_mlp_bwd(x, W1, W2, preact, dy, dx, dW1, dW2, ws_b, residual=args.residual)

    def barrier():
        if ws_n > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    st = binding.swiglu_mlp_device_status(dev)
    if st != 0:
        raise RuntimeError(f"warm-up failed: {binding.swiglu_mlp_strerror(st)}")

    K = args.steps
    trace = binding.LaunchTrace(12 * K)
    barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with trace:
        ev0.record()
        for _ in range(K):
            step()
        ev1.record()
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    st = binding.swiglu_mlp_device_status(dev)
    if st != 0:
        raise RuntimeError(f"timed steps failed: {binding.swiglu_mlp_strerror(st)}")
    ms = max_over_ranks(ev0.elapsed_time(ev1) / K, dev)
    recs = trace.records()
    launches = trace.count

    per_kind = {}
    for kind, kms in recs:
        per_kind.setdefault(kind, []).append(kms)
    kstats = {}
    total_kernel_ms = sum(sum(v) for v in per_kind.values())
    kb = ledger.kernel_bytes(M, D, H, Do)
    if "bwd_dx" in per_kind:   # small-M path: dx runs on its own, the grouped launch is dW2 + dW1
        flops["bwd_gemms"] = flops["bwd_dW2"] + flops["bwd_dW1"]
        kb["bwd_gemms"] = kb["bwd_dW2"] + kb["bwd_dW1"]
    pk, pk_src = peaks()
    tpk, tpk_src = tensor_peak(pk, pk_src, ms * K * 1e-3)
    for kind, v in per_kind.items():
        avg = sum(v) / len(v)
        f_k, b_k = flops.get(kind, 0), kb.get(kind, 0)   # element-wise kernels: not counted
        kstats[kind] = {"launches": len(v), "avg_us": round(avg * 1e3, 2),
                        "tflops": round(f_k / (avg * 1e-3) / 1e12, 1),
                        "frac_of_peak": round(f_k / (avg * 1e-3) / 1e12 / tpk, 3),
                        "hbm_gbs_compulsory": round(b_k / (avg * 1e-3) / 1e9, 1),
                        "share": round(sum(v) / total_kernel_ms, 3)}
    dom = max(kstats, key=lambda k: kstats[k]["share"])
    if wl == "decode":
        # 16 tokens: every kernel streams its weights; the HBM roofline bounds it
        dom_gbs = kstats[dom]["hbm_gbs_compulsory"]
        roofline = {"kernel": dom, "bound": "hbm", "achieved": dom_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": round(dom_gbs / pk["hbm_gbs"], 3), "traffic": measured_traffic(dom, wl if not args.residual else "residual"),
                    "peak_source": f"{pk_src} hbm_gbs"}
        if dom == "bwd_gemms":
            # the weight gradients are almost all writes: their own ceiling is a write-only
            # stream, measured here on the same part (torch fill_ of the same number of bytes)
            wc = write_ceiling_gbs(kb[dom], dev)
            roofline["write_only_ceiling_gbs"] = round(wc, 1)
            roofline["frac_of_write_only_ceiling"] = round(dom_gbs / wc, 3)
    else:
        dom_achieved = kstats[dom]["tflops"]
        roofline = {"kernel": dom, "bound": "tensor", "achieved": dom_achieved,
                    "peak": tpk, "unit": "TFLOP/s",
                    "frac": round(dom_achieved / tpk, 3),
                    "traffic": measured_traffic(dom, wl if not args.residual else "residual"),
                    "peak_source": tpk_src}
    fused = kstats.get("bwd_grad_h", {})
    # forward / backward kernel time per step: every step launches the same sequence, the
    # forward's kernels (element-wise ones included) before the first backward kernel
    per_step = max(1, len(recs) // K)
    nf = next((i for i, (k, _) in enumerate(recs[:per_step]) if k.startswith("bwd")), per_step)
    fwd_ms = sum(t for i, (_, t) in enumerate(recs) if i % per_step < nf) / K
    bwd_ms = max(1e-9, sum(t for i, (_, t) in enumerate(recs) if i % per_step >= nf) / K)

    # ---- end to end: pinned host inputs in, results out, every step; copies of
    # neighbouring steps overlap this step's compute (HostStepRunner)
    from bwd_gemm_epilogue_gb300.pipeline import HostStepRunner
    runner = HostStepRunner(M, D, H, Do, dev, residual=args.residual)
    host_in = {k: t.pin_memory() for k, t in (("x", x_h), ("W1", W1_h), ("W2", W2_h), ("dy", dy_h))}
    host_out = {k: torch.empty(t.shape, dtype=t.dtype).pin_memory()
                for k, t in (("y", y), ("dx", dx), ("dW1", dW1), ("dW2", dW2))}
    bi, bo = runner.bytes_in(host_in), runner.bytes_out(host_out)
    runner.run([host_in] * 2, [host_out] * 2)
    runner.synchronize()
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    runner.run([host_in] * args.e2e_steps, [host_out] * args.e2e_steps)
    runner.synchronize()
    torch.cuda.synchronize(dev)
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps
    barrier()
    e2e_ms = max_over_ranks(e2e_ms, dev)
    st = binding.swiglu_mlp_device_status(dev)
    if st != 0:
        raise RuntimeError(f"e2e steps failed: {binding.swiglu_mlp_strerror(st)}")
    del runner

    graph = None
    if wl == "decode":
        graph = graph_replay_timing(step, dev, K, flops["step"])

    eager = None
    if rank == 0 and ws_n == 1 and wl in ("target", "prefill") and not args.residual:
        eager = eager_comparison(step, x, W1, W2, dy, flops["step"], dev)

    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        pre_h = preact.cpu()
        cpu = cpu_baseline(s, x_h, W1_h, W2_h, dy_h, pre_h, args.cpu_seconds)
        cpu["sample"] = cpu["sample"].replace("target block", f"{wl} block")

    value = job_tflops(flops["step"], ms, ws_n)
    in_bytes = sum(t.numel() * 2 for t in (x_h, W1_h, W2_h, dy_h))
    step_bytes = sum(kb.get(k, 0) * kstats[k]["launches"] / K for k in kstats)
    out = {
        "metric": ("SwiGLU MLP fwd+bwd TFLOP/s (bf16, 11136x3584x14336); fused grad_preact us"
                   if wl == "target" and not args.residual
                   else f"SwiGLU MLP fwd+bwd TFLOP/s (bf16, {M}x{D}x{H}, {wl}{', residual' if args.residual else ''})"),
        "value": round(value, 1),
        "unit": "TFLOP/s",
        "n_gpus": ws_n,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (round(value / ws_n / (flops["step"] / (PAGES_FULL_MS_B200 * 1e-3) / 1e12), 3)
                        if wl == "target" and not args.residual else None),
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations/dy, N(0,1/fan_in) weights, bf16)",
        "config": {"workload": (f"SwiGLU MLP {'residual block y = x + MLP(x)' if args.residual else 'block'} "
                                f"fwd+bwd, M={M} D={D} H={H} Dout={Do}, drop-h, bf16"),
                   "M": M, "D": D, "H": H, "Dout": Do, "parallelism": f"replicas x{ws_n}",
                   "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB per step), no flush"},
        "step_hbm_gbs_compulsory": round(step_bytes / (ms * 1e-3) / 1e9, 1),
        "fused_grad_preact_us": fused.get("avg_us"),
        "fused_grad_preact_tflops": fused.get("tflops"),
        "fwd_ms": round(fwd_ms, 4),
        "bwd_ms": round(bwd_ms, 4),
        "fwd_tflops": round(flops["fwd"] / (fwd_ms * 1e-3) / 1e12, 1),
        "bwd_tflops": round(flops["bwd"] / (bwd_ms * 1e-3) / 1e12, 1),
        "fwd_frac_of_peak": round(flops["fwd"] / (fwd_ms * 1e-3) / 1e12 / tpk, 3),
        "bwd_frac_of_peak": round(flops["bwd"] / (bwd_ms * 1e-3) / 1e12 / tpk, 3),
        "fused_grad_preact_frac_of_peak": fused.get("frac_of_peak"),
        "step_frac_of_peak": round(flops["step"] / (ms * 1e-3) / 1e12 / tpk, 3),
        "peak_tflops": tpk,
        "peak_source": tpk_src,
        "kernels": kstats,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_tflops(flops["step"], e2e_ms, ws_n), 1), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "overlap": "h2d of step i+1 and d2h of step i-1 run during step i (3 streams)"},
        "gpu_launches": launches,
        "clocks": clk,
        "mcycles_per_step": (round(ms * clk["sm_mhz"] / 1e3, 3) if clk.get("sm_mhz") else None),
        "cublas_eager_comparison": eager,
        "cuda_graph": graph,
        "memory_mib": block_memory_mib(M, D, H, Do, ws_b.numel()),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws_n > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    from bwd_gemm_epilogue_gb300 import ledger, workloads
    s, x, W1, W2, dy = workloads.make_block(WORKLOAD)
    preact = workloads.make_preact(s, workloads.CONFIGS[WORKLOAD]["seed"])
    # Each step is a sample of the target step: forward and row-wise backward for some
    # token rows plus the weight gradients for some hidden columns (about a quarter of
    # the time), sized from a calibration so that warm-up + steps take about two minutes.
    import oracle
    nt = max(1, oracle.num_threads())      # the oracle runs rows (columns) in parallel: calibrate on nt of each
    dt_r, _, _ = oracle_sample(s, x, W1, W2, dy, preact, nt, 0, seed=7)
    dt_c, _, _ = oracle_sample(s, x, W1, W2, dy, preact, 0, nt, seed=8)
    per_step_s = 120.0 / max(1, args.steps + args.warmup)
    n_cols = max(1, int(0.25 * per_step_s / max(dt_c / nt, 1e-6)))
    n_rows = max(1, int(0.75 * per_step_s / max(dt_r / nt, 1e-6)))
    for i in range(args.warmup):
        oracle_sample(s, x, W1, W2, dy, preact, n_rows, n_cols, seed=100 + i)
    tot_t, tot_f, threads = 0.0, 0, 0
    for i in range(args.steps):
        dt, f, threads = oracle_sample(s, x, W1, W2, dy, preact, n_rows, n_cols, seed=1000 + i)
        tot_t += dt
        tot_f += f
    value = tot_f / tot_t / 1e12
    flops = ledger.gemm_flops(s.M, s.D, s.H, s.Dout)
    sample = (f"per step: fwd + row-wise bwd for {n_rows} of {s.M} token rows and dW1/dW2 for {n_cols} of {s.H} "
              f"hidden columns of the target block ({tot_f / max(1, args.steps) / 1e9:.1f} GFLOP, fp64 oracle, "
              f"{threads} threads)")
    out = {
        "impl": "reference",
        "metric": "SwiGLU MLP fwd+bwd TFLOP/s (bf16, 11136x3584x14336); fused grad_preact us",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tot_t / max(1, args.steps) * 1e3,
        "ms_per_step_note": "measured seconds of one sampled step (see cpu_baseline.sample), not a full step",
        "extrapolated_full_step_ms": flops["step"] / (value * 1e12) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations/dy, N(0,1/fan_in) weights, bf16)",
        "config": {"workload": f"SwiGLU MLP block fwd+bwd, M={s.M} D={s.D} H={s.H} Dout={s.Dout}, drop-h, bf16",
                   "M": s.M, "D": s.D, "H": s.H, "Dout": s.Dout, "parallelism": "cpu oracle"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def run_stack(args):
    """Four target blocks trained end to end: throughput and saved-activation memory."""
    import torch

    from bwd_gemm_epilogue_gb300 import binding, ledger, workloads
    from bwd_gemm_epilogue_gb300.stack import SwiGLUStack

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s, x_h, dy_h, layers_h = workloads.make_stack("stack4")
    layers = [(W1.to(dev), W2.to(dev)) for W1, W2 in layers_h]
    x, dy = x_h.to(dev), dy_h.to(dev)
    st = SwiGLUStack(layers, s.M)
    for _ in range(args.warmup):
        st.forward(x)
        st.backward(dy)
    torch.cuda.synchronize(dev)
    K = max(1, args.steps // 4)
    clocks = ClockSampler(dev.index)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        st.forward(x)
        st.backward(dy)
    e1.record()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if binding.swiglu_mlp_device_status(dev) != 0:
        raise RuntimeError("stack steps failed")
    ms = e0.elapsed_time(e1) / K
    flops = len(layers) * ledger.gemm_flops(s.M, s.D, s.H, s.Dout)["step"]
    print(json.dumps({
        "metric": "SwiGLU MLP 4-layer stack fwd+bwd TFLOP/s (bf16, 4 x 11136x3584x14336)",
        "value": round(flops / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": "stack4: 4 SwiGLU blocks, M=11136 D=Dout=3584 H=14336"},
        "saved_activation_mib": round(st.saved_activation_bytes() / 2 ** 20, 1),
        "saved_activation_note": "x_0..x_4 and preact_1..4 kept for the backward (h dropped)",
        "bwd_peak_mib": round(st.backward_peak_bytes() / 2 ** 20, 1),
        "bwd_peak_note": "saved activations + one layer's backward workspace (h, grad_preact) + dx ping-pong "
                         "+ all four layers' dW1/dW2; weights, x and dy excluded",
        "gpu_launches_per_step": 4 * (2 + 2), "clocks": clk}), flush=True)


def run_tp2(args):
    """One rank's compute of the target block split over two tensor-parallel ranks: the
    shard's forward with the down projection in row chunks (a CUDA event per chunk, where a
    communication stream would start each chunk's reduction) and backward with dx first (its
    event), against the same shard through the one-piece entry points, in alternating blocks.
    The reductions themselves need the second rank's GPU and are not timed here."""
    import torch

    from bwd_gemm_epilogue_gb300 import binding, ledger, workloads
    from bwd_gemm_epilogue_gb300.tensor_parallel import shard_bounds

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    s, x_h, W1_h, W2_h, dy_h = workloads.make_block("target")
    world, n_chunks = 2, 4
    j0, Hs = shard_bounds(s.H, world, 0)
    x, dy = x_h.to(dev), dy_h.to(dev)
    W1s, W2s = binding.swiglu_mlp_tp_shard_pack(W1_h.to(dev), W2_h.to(dev), j0, Hs)
    M, D, Do = s.M, s.D, s.Dout
    preact = torch.empty(M, 2 * Hs, dtype=torch.bfloat16, device=dev)
    y = torch.empty(M, Do, dtype=torch.bfloat16, device=dev)
    dx = torch.empty(M, D, dtype=torch.bfloat16, device=dev)
    dW1 = torch.empty(2 * Hs, D, dtype=torch.bfloat16, device=dev)
    dW2 = torch.empty(Do, Hs, dtype=torch.bfloat16, device=dev)
    ws_f = torch.empty(binding.swiglu_mlp_fwd_workspace_size(M, D, Hs, Do), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(binding.swiglu_mlp_bwd_workspace_size(M, D, Hs, Do), dtype=torch.uint8, device=dev)
    events = [torch.cuda.Event() for _ in range(n_chunks)]
    dx_ev = torch.cuda.Event()

    def step_tp():
        binding.swiglu_mlp_tp_fwd(x, W1s, W2s, preact, y, ws_f, n_chunks=n_chunks, chunk_events=events)
        binding.swiglu_mlp_tp_bwd(x, W1s, W2s, preact, dy, dx, dW1, dW2, ws_b, dx_event=dx_ev)

    def step_plain():
        binding.swiglu_mlp_fwd(x, W1s, W2s, preact, y, ws_f)
        binding.swiglu_mlp_bwd(x, W1s, W2s, preact, dy, dx, dW1, dW2, ws_b)

    for _ in range(args.warmup):
        step_tp()
        step_plain()
    torch.cuda.synchronize(dev)
    blocks, per = 6, max(1, args.steps // 12)
    t_tp, t_plain = [], []
    clocks = ClockSampler(dev.index)
    for b in range(blocks):
        for name in (("tp", "plain") if b % 2 == 0 else ("plain", "tp")):
            fn = step_tp if name == "tp" else step_plain
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(per):
                fn()
            e1.record()
            torch.cuda.synchronize(dev)
            (t_tp if name == "tp" else t_plain).append(e0.elapsed_time(e1) / per)
    clk = clocks.stop()
    if binding.swiglu_mlp_device_status(dev) != 0:
        raise RuntimeError("tensor-parallel shard steps failed")
    ms_tp, ms_plain = sum(t_tp) / len(t_tp), sum(t_plain) / len(t_plain)
    flops = ledger.gemm_flops(M, D, Hs, Do)["step"]
    ring = 2 * (world - 1) / world   # bytes a ring all-reduce sends per byte of the summed tensor
    print(json.dumps({
        "metric": "SwiGLU MLP tensor-parallel shard fwd+bwd TFLOP/s (bf16, one of 2 ranks of 11136x3584x14336)",
        "value": round(flops / (ms_tp * 1e-3) / 1e12, 1), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": per * blocks, "warmup": args.warmup, "ms_per_step": round(ms_tp, 4), "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"tp2: rank 0 of 2, hidden units [{j0}, {j0 + Hs}) of H={s.H}; M={M} D={D} "
                               f"Dout={Do}; forward in {n_chunks} row chunks with events, backward dx first "
                               f"with an event"},
        "one_piece_ms_per_step": round(ms_plain, 4),
        "chunking_cost": round(ms_tp / ms_plain - 1.0, 4),
        "reductions": {"measured": False,
                       "why": "the partial y and dx are summed across the ranks' GPUs; every run here has one GPU",
                       "bytes_summed_per_step": 2 * M * (Do + D),
                       "ring_all_reduce_bytes_sent_per_rank": round(ring * 2 * M * (Do + D))},
        "gpu_launches_per_step": 1 + n_chunks + 3, "clocks": clk}), flush=True)


def run_moe(args):
    """A mixture-of-experts layer (tokens grouped by expert): forward + backward of
    every expert, each step one grouped launch over all experts."""
    import torch

    from bwd_gemm_epilogue_gb300 import binding, ledger, workloads
    from bwd_gemm_epilogue_gb300.pipeline import HostStepRunner

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = args.workload
    counts, x_h, W1_h, W2_h, dy_h = workloads.make_moe(wl)
    E, D, H, Do = W1_h.shape[0], x_h.shape[1], W2_h.shape[2], W2_h.shape[1]
    T = sum(counts)
    active = sum(1 for c in counts if c)
    flops = ledger.gemm_flops(T, D, H, Do)       # every GEMM is linear in its row (or K) count
    kb = ledger.kernel_bytes(T, D, H, Do, experts=active)
    x, W1, W2, dy = (t.to(dev) for t in (x_h, W1_h, W2_h, dy_h))
    bf = dict(dtype=torch.bfloat16, device=dev)
    preact, y, dx = torch.empty(T, 2 * H, **bf), torch.empty(T, Do, **bf), torch.empty(T, D, **bf)
    dW1, dW2 = torch.empty(E, 2 * H, D, **bf), torch.empty(E, Do, H, **bf)
    ws_f = torch.empty(binding.swiglu_moe_fwd_workspace_size(counts, D, H, Do), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(binding.swiglu_moe_bwd_workspace_size(counts, D, H, Do), dtype=torch.uint8, device=dev)

    def step():
        binding.swiglu_moe_fwd(x, W1, W2, counts, preact, y, ws_f)
        binding.swiglu_moe_bwd(x, W1, W2, preact, dy, counts, dx, dW1, dW2, ws_b)

    for _ in range(args.warmup):
        step()
    if binding.swiglu_mlp_device_status(dev) != 0:
        raise RuntimeError("warm-up failed")
    K = args.steps
    trace = binding.LaunchTrace(8 * K)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with trace:
        ev0.record()
        for _ in range(K):
            step()
        ev1.record()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if binding.swiglu_mlp_device_status(dev) != 0:
        raise RuntimeError("timed steps failed")
    ms = ev0.elapsed_time(ev1) / K
    per_kind = {}
    for kind, kms in trace.records():
        per_kind.setdefault(kind, []).append(kms)
    total = sum(sum(v) for v in per_kind.values())
    pk, pk_src = peaks()
    tpk, tpk_src = tensor_peak(pk, pk_src, ms * K * 1e-3)
    kstats = {}
    for kind, v in per_kind.items():
        avg = sum(v) / len(v)
        f_k = flops.get(kind, 0)
        kstats[kind] = {"launches": len(v), "avg_us": round(avg * 1e3, 2),
                        "tflops": round(f_k / (avg * 1e-3) / 1e12, 1),
                        "frac_of_peak": round(f_k / (avg * 1e-3) / 1e12 / tpk, 3),
                        "hbm_gbs_compulsory": round(kb.get(kind, 0) / (avg * 1e-3) / 1e9, 1),
                        "share": round(sum(v) / total, 3)}
    dom = max(kstats, key=lambda k: kstats[k]["share"])
    roofline = {"kernel": dom, "bound": "tensor", "achieved": kstats[dom]["tflops"],
                "peak": tpk, "unit": "TFLOP/s",
                "frac": round(kstats[dom]["tflops"] / tpk, 3), "traffic": None,
                "peak_source": tpk_src}

    runner = HostStepRunner(T, D, H, Do, dev, counts=counts)
    host_in = {k: t.pin_memory() for k, t in (("x", x_h), ("W1", W1_h), ("W2", W2_h), ("dy", dy_h))}
    host_out = {k: torch.empty(t.shape, dtype=t.dtype).pin_memory()
                for k, t in (("y", y), ("dx", dx), ("dW1", dW1), ("dW2", dW2))}
    bi, bo = runner.bytes_in(host_in), runner.bytes_out(host_out)
    runner.run([host_in] * 2, [host_out] * 2)
    runner.synchronize()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    runner.run([host_in] * args.e2e_steps, [host_out] * args.e2e_steps)
    runner.synchronize()
    torch.cuda.synchronize(dev)
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps
    if binding.swiglu_mlp_device_status(dev) != 0:
        raise RuntimeError("e2e steps failed")
    del runner
    value = flops["step"] / (ms * 1e-3) / 1e12
    cfg = workloads.MOE_CONFIGS[wl]
    print(json.dumps({
        "metric": f"SwiGLU MoE layer fwd+bwd TFLOP/s (bf16, {E} experts, {T} routed rows, D={D} H={H})",
        "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded routed counts, N(0,1) activations/dy, N(0,1/fan_in) weights)",
        "config": {"workload": f"{wl}: MoE SwiGLU layer, E={E} experts ({active} with rows), T={T} rows "
                               f"grouped by expert, D={D} H={H} Dout={Do}",
                   "E": E, "T": T, "D": D, "H": H, "Dout": Do, "seed": cfg["seed"],
                   "rows_per_expert": {"min": min(counts), "max": max(counts)},
                   "l2": "inputs larger than L2, no flush"},
        "kernels": kstats, "roofline": roofline, "cpu_baseline": None,
        "e2e": {"value": round(flops["step"] / (e2e_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
        "gpu_launches": trace.count, "clocks": clk}), flush=True)


def run_fp8(args):
    """The FP8 forward (E4M3 operands, h quantised in the first GEMM's epilogue) at one
    of the block shapes, with the bf16 forward of the same shape timed beside it."""
    import torch

    from bwd_gemm_epilogue_gb300 import binding, ledger, workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    base = args.workload[len("fp8_"):]
    cfg = workloads.CONFIGS[base]
    s = cfg["shape"]
    M, D, H, Do = s.M, s.D, s.H, s.Dout
    x8_h, W1_h, W2_h, sc = workloads.make_fp8_block(s, cfg["seed"])
    x8, W1_8, W2_8 = (t.to(dev) for t in (x8_h, W1_h, W2_h))
    h8 = torch.empty(M, H, dtype=torch.float8_e4m3fn, device=dev)
    y = torch.empty(M, Do, dtype=torch.bfloat16, device=dev)
    flops = ledger.gemm_flops(M, D, H, Do)

    def fp8_step():
        binding.swiglu_mlp_fwd_fp8(x8, W1_8, W2_8, h8=h8, y=y, store_preact=False, **sc)

    # the bf16 forward of the same shape, for comparison
    _, xb_h, W1b_h, W2b_h, _ = workloads.make_block(base)
    xb, W1b, W2b = (t.to(dev) for t in (xb_h, W1b_h, W2b_h))
    pre_b = torch.empty(M, 2 * H, dtype=torch.bfloat16, device=dev)
    ws_f = torch.empty(max(16, binding.swiglu_mlp_fwd_workspace_size(M, D, H, Do)), dtype=torch.uint8, device=dev)

    def bf16_step():
        binding.swiglu_mlp_fwd(xb, W1b, W2b, pre_b, y, ws_f)

    def timed(step, K):
        for _ in range(args.warmup):
            step()
        tr = binding.LaunchTrace(4 * K)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with tr:
            e0.record()
            for _ in range(K):
                step()
            e1.record()
        torch.cuda.synchronize(dev)
        if binding.swiglu_mlp_device_status(dev) != 0:
            raise RuntimeError("fp8 forward steps failed")
        per = {}
        for kind, kms in tr.records():
            per.setdefault(kind, []).append(kms)
        return e0.elapsed_time(e1) / K, {k: sum(v) / len(v) for k, v in per.items()}, tr.count

    K = args.steps
    clocks = ClockSampler(dev.index)
    ms8, k8, launches = timed(fp8_step, K)
    clk = clocks.stop()
    msb, kbf, _ = timed(bf16_step, K)
    pk, pk_src = peaks()
    tpk, tpk_src = tensor_peak(pk, pk_src, ms8 * K * 1e-3)
    peak8 = 2.0 * tpk
    kstats = {k: {"avg_us": round(v * 1e3, 2), "tflops": round(flops.get(k, 0) / (v * 1e-3) / 1e12, 1),
                  "frac_of_fp8_peak": round(flops.get(k, 0) / (v * 1e-3) / 1e12 / peak8, 3)} for k, v in k8.items()}
    dom = max((k for k in k8 if k in flops), key=lambda k: k8[k])
    kb8 = {"fwd_preact": M * D + 2 * H * D + M * H, "fwd_down": M * H + Do * H + 2 * M * Do}   # FP8 bytes
    value = flops["fwd"] / (ms8 * 1e-3) / 1e12
    if base == "decode":
        gbs = kb8[dom] / (k8[dom] * 1e-3) / 1e9
        roofline = {"kernel": dom, "bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": round(gbs / pk["hbm_gbs"], 3), "traffic": None, "peak_source": f"{pk_src} hbm_gbs"}
    else:
        roofline = {"kernel": dom, "bound": "tensor", "achieved": kstats[dom]["tflops"], "peak": round(peak8, 1),
                    "unit": "TFLOP/s", "frac": kstats[dom]["frac_of_fp8_peak"], "traffic": None,
                    "peak_source": f"{tpk_src} x 2 (nominal FP8 / bf16 dense ratio)"}
    print(json.dumps({
        "metric": f"SwiGLU MLP FP8 forward TFLOP/s (E4M3, {M}x{D}x{H})",
        "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms8, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3", "data": "synthetic (the bf16 workload's draws quantised to E4M3, power-of-two scales)",
        "config": {"workload": f"{args.workload}: FP8 forward x8 @ W1_8^T (+SwiGLU, h quantised), h8 @ W2_8^T, "
                               f"M={M} D={D} H={H} Dout={Do}, preact not stored", "scales": sc},
        "kernels": kstats, "roofline": roofline, "cpu_baseline": None,
        "bf16_forward_ms": round(msb, 4), "speedup_vs_bf16_forward": round(msb / ms8, 3),
        "bf16_kernels_us": {k: round(v * 1e3, 2) for k, v in kbf.items()},
        "gpu_launches": launches, "clocks": clk}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "stack4":
        run_stack(args)
    elif args.workload in ("moe8", "moe64"):
        run_moe(args)
    elif args.workload.startswith("fp8_"):
        run_fp8(args)
    elif args.workload == "tp2":
        run_tp2(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
