#!/usr/bin/env python3
"""Benchmark: fused chunked KL forward + backward on one GB300 (or N replicas).

One step = kd_fused_kl_fwd + kd_fused_kl_bwd over the whole workload (every
chunk: teacher prologue, projection + online logsumexp, recompute + dZ, the two
gradient products).  Default workload: the gpt-oss-shaped long context
(B=1, T=32768, d=2880, V=201088, K=100, chunk=4096).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on a bounded sample of the same workload on this host's cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused KL fwd+bwd tokens/s and TFLOP/s vs BF16 peak; peak device GB (1xGB300)"
UNIT = "tokens/s"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(bf16_burst=float(p["bf16_tflops"]), bf16_sustained=float(p["bf16_tflops_sustained"]),
                    hbm=float(p["hbm_gbs"]), source="measured")
    except Exception:
        return dict(bf16_burst=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while open."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of ``kernel`` on ``workload`` from
    profiles/ncu_traffic.json, or None when absent or captured from other sources than the
    ones built now (each record names the source files that define its kernel and their
    digest at capture time)."""
    from sparse_teacher_kl_gb300.build import source_digest
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f)["kernels"][workload][kernel]
        if rec["digest"] != source_digest(rec["sources"]):
            return None
        return rec["bytes_per_launch"]
    except Exception:
        return None


def bench_topk(kd, dev, stream, peaks, steps):
    """kd_topk_cache on the mid workload's dense teacher logits (8192 x 151936 bf16, N(0, 2), K = 100):
    HBM-bound, algorithmic bytes N*V*2 read + N*K*8 written per launch."""
    import torch
    from synth import WORKLOADS, make_dense_teacher_logits
    w = WORKLOADS["mid"]
    N, V, K = w.N, w.V, w.K
    X = make_dense_teacher_logits(N, V, seed=w.seed, device=dev)
    ids = torch.empty((N, K), dtype=torch.int32, device=dev)
    vals = torch.empty((N, K), dtype=torch.float32, device=dev)
    lse = torch.empty((N,), dtype=torch.float32, device=dev)
    ws = kd.workspace(kd._abi.kd_topk_cache_workspace(N, V, K), dev)
    out = {"workload": f"{N}x{V} bf16 N(0,2), K={K}"}
    for name, lp in (("ids+vals", None), ("ids+vals+lse", lse)):
        def run():
            st = kd._abi.kd_topk_cache(X.data_ptr(), N, V, V, K, ids.data_ptr(), vals.data_ptr(),
                                       None if lp is None else lp.data_ptr(), None, ws.data_ptr(), ws.numel(),
                                       stream.cuda_stream)
            assert st == 0
        for _ in range(3):
            run()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            run()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / steps
        byts = N * V * 2 + N * K * 8 + (N * 4 if lp is not None else 0)
        gbs = byts / (ms * 1e-3) / 1e9
        # rows selected a second time after a speculative start (control block word 2), per launch
        resel = int(ws[8:12].view(torch.int32).item()) / (steps + 3)
        ws[8:12].zero_()
        out[name] = {"ms": ms, "achieved_gbs": gbs, "peak_gbs": peaks["hbm"], "frac": gbs / peaks["hbm"],
                     "bytes_per_launch": byts, "reselected_rows_per_launch": resel}
    out["roofline"] = {"bound": "hbm", "achieved": out["ids+vals"]["achieved_gbs"], "peak": peaks["hbm"],
                       "unit": "GB/s", "frac": out["ids+vals"]["frac"], "traffic": ncu_traffic("kd_topk_cache", "mid"),
                       "peak_source": f"{peaks['source']} copy bandwidth"}

    # The same rows with each row's values scaled by 1 + s N(0, 1) (rows of different scales), and
    # with every row's first 4096 values raised by 6 standard deviations (the start taken from a
    # row's first values then misses: the row is selected twice and its warp stops speculating).
    def timed(Xv):
        def run():
            st = kd._abi.kd_topk_cache(Xv.data_ptr(), N, V, V, K, ids.data_ptr(), vals.data_ptr(), None, None,
                                       ws.data_ptr(), ws.numel(), stream.cuda_stream)
            assert st == 0
        for _ in range(3):
            run()
        torch.cuda.synchronize(dev)
        ws[8:12].zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            run()
        b.record(stream)
        torch.cuda.synchronize(dev)
        resel = int(ws[8:12].view(torch.int32).item()) / steps
        ws[8:12].zero_()
        return {"ms": a.elapsed_time(b) / steps, "reselected_rows_per_launch": resel}

    Xs = torch.empty_like(X)
    gen = torch.Generator(device=dev)
    spread = {}
    for sp in (0.05, 0.1, 0.2):
        gen.manual_seed(int(sp * 1000) + 7)
        f = 1.0 + sp * torch.randn((N, 1), generator=gen, device=dev)
        for r0 in range(0, N, 512):
            Xs[r0:r0 + 512] = (X[r0:r0 + 512].float() * f[r0:r0 + 512]).to(torch.bfloat16)
        spread[str(sp)] = timed(Xs)
    out["scale_spread"] = spread
    Xs.copy_(X)
    Xs[:, :4096] = (Xs[:, :4096].float() + 6.0 * math.sqrt(2.0)).to(torch.bfloat16)
    out["prefix_high"] = timed(Xs)
    del X, Xs
    torch.cuda.empty_cache()
    return out


def bench_teacher_topk(kd, dev, stream, peaks, steps):
    """kd_teacher_topk on the gpt-oss shape (32768 teacher positions, dt = 2880, V = 201088,
    K = 100, chunk = 4096): the teacher logits are formed a chunk at a time by the projection
    engine (2*N*dt*V flops, tensor-bound) and reduced to their top K at once (HBM-bound);
    the dense [N, V] teacher logits never exist."""
    import torch
    from synth import WORKLOADS, make_inputs
    w = WORKLOADS["gptoss"]
    N, dt, V, K, c = w.N, w.d, w.V, w.K, w.chunk
    Ht, Wt, _, _, _ = make_inputs(w, device=dev)
    ids = torch.empty((N, K), dtype=torch.int32, device=dev)
    vals = torch.empty((N, K), dtype=torch.float32, device=dev)
    ws = kd.workspace(kd._abi.kd_teacher_topk_workspace(N, dt, V, K, c), dev)

    def run():
        st = kd._abi.kd_teacher_topk(Ht.data_ptr(), Wt.data_ptr(), N, dt, V, K, c, ids.data_ptr(), vals.data_ptr(),
                                     None, None, ws.data_ptr(), ws.numel(), stream.cuda_stream)
        assert st == 0
    for _ in range(2):
        run()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with kd.Profile(capacity=4 * steps * (N // c + 2)) as prof:
        a.record(stream)
        for _ in range(steps):
            run()
        b.record(stream)
        torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    flops = 2.0 * N * dt * V
    kernels = {k: {"launches": n, "avg_ms": t / n, "ms_per_call": t / steps}
               for k, (n, t) in prof.summary().items()}
    # the same calls also returning each row's logsumexp and dropped teacher mass
    lse = torch.empty((N,), dtype=torch.float32, device=dev)
    dropped = torch.empty((N,), dtype=torch.float32, device=dev)

    def run_lse():
        st = kd._abi.kd_teacher_topk(Ht.data_ptr(), Wt.data_ptr(), N, dt, V, K, c, ids.data_ptr(), vals.data_ptr(),
                                     lse.data_ptr(), dropped.data_ptr(), ws.data_ptr(), ws.numel(),
                                     stream.cuda_stream)
        assert st == 0
    run_lse()
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(steps):
        run_lse()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms_lse = a.elapsed_time(b) / steps
    out = {"workload": f"gpt-oss shape: N={N}, dt={dt}, V={V}, K={K}, chunk={c}",
           "ms": ms, "positions_per_s": N / (ms * 1e-3),
           "projection_tflops": flops / (ms * 1e-3) / 1e12,
           "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / peaks["bf16_sustained"],
           "ms_with_lse_and_dropped": ms_lse,
           "peak_source": f"{peaks['source']} bf16 sustained", "kernels": kernels,
           "workspace_gb": ws.numel() / 1e9}
    del Ht, Wt, ids, vals, ws, lse, dropped
    torch.cuda.empty_cache()
    return out


def dense_torch_reference(H, W, ids, tlog, mask, dev):
    """Peak device memory and time of one fwd+bwd of the dense formulation in plain PyTorch
    (full [N, V] student logits and a full-vocabulary teacher grid), for the memory comparison
    only; reports an estimate instead when it does not fit."""
    import torch
    N, V = H.shape[0], W.shape[0]
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    try:
        Hr = H.detach().requires_grad_(True)
        Wr = W.detach().requires_grad_(True)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        logq = torch.log_softmax((Hr @ Wr.T).float(), dim=1)
        grid = torch.full((N, V), float("-inf"), device=dev)
        grid.scatter_(1, ids.long(), tlog)
        logp = torch.log_softmax(grid, dim=1)
        p = logp.exp()
        kl = (p * (torch.where(p > 0, logp, torch.zeros_like(logp)) - logq)).sum(dim=1)
        m = torch.ones(N, device=dev) if mask is None else mask.float()
        loss = (kl * m).sum() / m.sum()
        loss.backward()
        t1.record()
        torch.cuda.synchronize(dev)
        out = {"peak_device_gb": (torch.cuda.max_memory_allocated(dev) - base) / 1e9,
               "ms_per_step": t0.elapsed_time(t1), "fits": True}
        del Hr, Wr, logq, grid, logp, p, kl, loss
    except torch.OutOfMemoryError:
        out = {"fits": False, "estimate_gb": N * V * 4 * 5 / 1e9}
    torch.cuda.empty_cache()
    return out


def config_dict(w, world: int = 1) -> dict:
    """The workload a line measures (both arms print the same dict)."""
    return {"workload": w.name, "B": w.B, "T": w.T, "d": w.d, "V": w.V, "K": w.K, "chunk": w.chunk, "tau": 1.0,
            "teacher": w.teacher, "p_valid": w.p_valid,
            "l2": f"inputs larger than L2 (W is {w.V * w.d * 2 / 1e9:.2f} GB, re-read every chunk)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def dense_estimate_gb(w) -> float:
    """Device memory of the dense formulation's grids alone: bf16 logits plus five fp32 [N, V] grids."""
    return w.N * w.V * (2 + 4 * 5) / 1e9


def bench_fused(kd, dev, stream, w, steps, warmup, peaks, dense=True):
    """kd_fused_kl_fwd + kd_fused_kl_bwd over every chunk of workload ``w``, per step: tokens/s, executed
    TFLOP/s (8 d V per token) and its fraction of the sustained bf16 peak, and the device memory a step
    needs beyond its inputs (the allocator's peak: workspace, gradients, loss and lse) next to the
    workspace alone; with ``dense``, the plain PyTorch dense formulation's peak on the same inputs
    (measured where it fits in memory, else an estimate of its grids)."""
    import torch
    from synth import make_inputs
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    H, W, ids, tlog, mask = make_inputs(w, dev)
    N, d, V, K, c = w.N, w.d, w.V, w.K, w.chunk
    inputs = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    ws = kd.workspace(kd._abi.kd_fused_kl_workspace(N, d, V, K, c), dev)
    grad_H = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    grad_W = torch.zeros((V, d), dtype=torch.float32, device=dev)
    g = torch.ones(1, dtype=torch.float32, device=dev)

    def step():
        loss, lse, _ = kd.fused_kl_forward(H, W, ids, tlog, mask, c, 1.0, ws=ws)
        kd.fused_kl_backward(H, W, ids, tlog, mask, lse, g, c, 1.0, ws=ws, grad_H=grad_H, grad_W=grad_W)
        return loss

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    peak = torch.cuda.max_memory_allocated(dev) - inputs
    st, detail = kd.device_error(ws)
    if st != 0:
        raise SystemExit(f"{w.name}: device error {st} ({detail})")
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    tflops = w.flops_executed() / (ms * 1e-3) / 1e12
    out = {"tokens_per_s": N / (ms * 1e-3), "ms_per_step": ms, "tflops_executed": tflops,
           "tflops_useful": w.flops_useful() / (ms * 1e-3) / 1e12,
           "frac_of_bf16_peak": tflops / peaks["bf16_sustained"], "peak_device_gb": peak / 1e9,
           "workspace_gb": ws.numel() / 1e9, "inputs_gb": inputs / 1e9}
    del ws, grad_H, grad_W
    torch.cuda.empty_cache()
    if dense:
        est = dense_estimate_gb(w)
        free, _ = torch.cuda.mem_get_info(dev)
        if est < 0.8 * free / 1e9:
            out["dense_torch"] = dense_torch_reference(H, W, ids, tlog, mask, dev)
        else:
            out["dense_torch"] = {"fits": False, "estimate_gb": est,
                                  "note": "not run: its grids alone exceed the free device memory"}
    del H, W, ids, tlog, mask
    torch.cuda.empty_cache()
    return out


def aggregate_over_ranks(ms_local: float, tokens_per_rank: int, world: int, all_reduce_max=None):
    """Whole-job step time (max over ranks) and throughput (all ranks' tokens / that time).

    ``all_reduce_max`` maps a float to its maximum over the ranks (identity on one rank).
    """
    ms = float(all_reduce_max(ms_local)) if (all_reduce_max is not None and world > 1) else float(ms_local)
    return ms, world * tokens_per_rank / (ms * 1e-3)


def cpu_oracle_seconds(Hb, Wb, ids, tlog, mask):
    """Wall time of the float64 oracle (fused formulation, fwd + bwd with full grad_W) on these rows."""
    import oracle
    t0 = time.perf_counter()
    oracle.fused_chunked_kl(Hb, Wb, ids, tlog, mask, 1.0, chunk=Hb.shape[0], vtile=8192)
    return time.perf_counter() - t0


def run_reference(args, w):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from synth import bf16_bits, make_inputs
    cores = len(os.sched_getaffinity(0))
    rows = args.ref_rows
    H, W, ids, tlog, mask = make_inputs(w, "cpu", rows=rows)
    Hb, Wb, idn, tln = bf16_bits(H), bf16_bits(W), ids.numpy(), tlog.numpy()
    mn = None if mask is None else mask.numpy()
    times = []
    for i in range(args.warmup + args.steps):
        dt = cpu_oracle_seconds(Hb, Wb, idn, tln, mn)
        if i >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    v = rows / t
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows} positions of {w.name} per step (float64 numpy, fused formulation, "
                                   f"fwd+bwd incl. full grad_W), tokens/s extrapolated per position"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="gptoss")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--cpu-rows", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-modes", action="store_true", help="skip the forward-chunked and dense comparisons")
    ap.add_argument("--no-topk", action="store_true", help="skip the top-K cache measurement")
    ap.add_argument("--topk-only", action="store_true", help="only the top-K cache measurement (profiling)")
    ap.add_argument("--no-teacher", action="store_true", help="skip the teacher projection + top-K measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip the other four workloads")
    ap.add_argument("--rows", type=int, default=None, help="override B*T (profiling a reduced case)")
    ap.add_argument("--vocab", type=int, default=None, help="override V (profiling a reduced case)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import dataclasses
    from synth import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.rows is not None or args.vocab is not None:
        w = dataclasses.replace(w, name=f"{w.name}-reduced", B=1, T=args.rows or w.N, V=args.vocab or w.V)
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from sparse_teacher_kl_gb300.build import build_library
    build_library()
    import sparse_teacher_kl_gb300 as kd
    from synth import make_inputs

    peaks = load_peaks()
    if args.topk_only:
        print(json.dumps({"topk_cache": bench_topk(kd, dev, torch.cuda.current_stream(dev), peaks, args.steps)}))
        return 0
    H, W, ids, tlog, mask = make_inputs(w, dev)
    N, d, V, K, c = w.N, w.d, w.V, w.K, w.chunk
    inputs_alloc = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    ws = kd.workspace(kd._abi.kd_fused_kl_workspace(N, d, V, K, c), dev)
    ws_gb = ws.numel() / 1e9
    grad_H = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    grad_W = torch.zeros((V, d), dtype=torch.float32, device=dev)
    g = torch.ones(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        loss, lse, _ = kd.fused_kl_forward(H, W, ids, tlog, mask, c, 1.0, ws=ws)
        kd.fused_kl_backward(H, W, ids, tlog, mask, lse, g, c, 1.0, ws=ws, grad_H=grad_H, grad_W=grad_W)
        return loss

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    peak_alloc = torch.cuda.max_memory_allocated(dev) - inputs_alloc  # beyond the inputs
    st, detail = kd.device_error(ws)
    if st != 0:
        raise SystemExit(f"device error {st} ({detail}) during warm-up")

    # ---- timed region: inputs resident in HBM (W = V*d*2 bytes, larger than L2)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks, kd.Profile(capacity=64 * (args.steps + 1) * (N // c + 2)) as prof:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    def rank_max(x):
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    ms, tokens_per_s = aggregate_over_ranks(e0.elapsed_time(e1) / args.steps, N, world, rank_max)

    # per-kernel breakdown from the library's own launch events
    summ = prof.summary()
    launches = sum(n for n, _ in summ.values())
    kernels = {k: {"launches": n, "total_ms": t, "avg_ms": t / n, "share": t / max(1e-9, ms * args.steps)}
               for k, (n, t) in sorted(summ.items(), key=lambda kv: -kv[1][1])}
    dom_name = max(summ.items(), key=lambda kv: kv[1][1])[0]
    dom = kernels[dom_name]
    gemm_flops_per_chunk = 2.0 * c * d * V
    if dom_name == "kd_topk_cache":
        raise SystemExit("unexpected dominant kernel")
    achieved = gemm_flops_per_chunk / (dom["avg_ms"] * 1e-3) / 1e12
    peak = peaks["bf16_sustained"]

    tflops_exec = w.flops_executed() / (ms * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        Hh = H.cpu().pin_memory()
        idh = ids.cpu().pin_memory()
        tlh = tlog.cpu().pin_memory()
        mh = None if mask is None else mask.cpu().pin_memory()
        lossh = torch.empty(1, dtype=torch.float32).pin_memory()
        Hd = torch.empty_like(H)
        idd = torch.empty_like(ids)
        tld = torch.empty_like(tlog)
        md = None if mask is None else torch.empty_like(mask)
        h2d = Hh.numel() * 2 + idh.numel() * 4 + tlh.numel() * 4 + (0 if mh is None else mh.numel())

        def e2e_step():
            Hd.copy_(Hh, non_blocking=True)
            idd.copy_(idh, non_blocking=True)
            tld.copy_(tlh, non_blocking=True)
            if md is not None:
                md.copy_(mh, non_blocking=True)
            loss, lse, _ = kd.fused_kl_forward(Hd, W, idd, tld, md, c, 1.0, ws=ws)
            kd.fused_kl_backward(Hd, W, idd, tld, md, lse, g, c, 1.0, ws=ws, grad_H=grad_H, grad_W=grad_W)
            lossh.copy_(loss, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        f1.record(stream)
        torch.cuda.synchronize(dev)
        ems, e2e_rate = aggregate_over_ranks(f0.elapsed_time(f1) / args.steps, N, world, rank_max)
        e2e = {"value": e2e_rate, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": 4, "ms_per_step": ems,
               "note": "pinned host H, teacher cache and mask copied in, loss copied out; W resident"}

    # ---- the pages' other two formulations on the same inputs, for the memory/time trade-off
    fc = None
    if not args.no_modes:
        zb = kd._abi.kd_chunked_kl_logits_bytes(N, V)
        z_store = torch.empty((zb,), dtype=torch.uint8, device=dev)

        def fc_step():
            loss, lse, _, _ = kd.chunked_kl_forward(H, W, ids, tlog, mask, c, 1.0, ws=ws, z_store=z_store)
            kd.chunked_kl_backward(H, W, ids, tlog, mask, lse, g, z_store, c, 1.0, ws=ws, grad_H=grad_H,
                                   grad_W=grad_W)

        for _ in range(2):
            fc_step()
        torch.cuda.synchronize(dev)
        h0 = torch.cuda.Event(enable_timing=True)
        h1 = torch.cuda.Event(enable_timing=True)
        with kd.Profile(capacity=64 * (args.steps + 1) * (N // c + 2)) as fprof:
            h0.record(stream)
            for _ in range(args.steps):
                fc_step()
            h1.record(stream)
            torch.cuda.synchronize(dev)
        fms = h0.elapsed_time(h1) / args.steps
        fk = {k: {"launches": n, "avg_ms": t / n, "share": t / max(1e-9, fms * args.steps)}
              for k, (n, t) in sorted(fprof.summary().items(), key=lambda kv: -kv[1][1])}
        fc = {"ms_per_step": fms, "tokens_per_s": N / (fms * 1e-3),
              "tflops_executed": w.flops_useful() / (fms * 1e-3) / 1e12,
              "kept_logits_gb": zb / 1e9, "workspace_gb": ws.numel() / 1e9, "kernels": fk,
              "note": "forward keeps bf16 logits [N, V]; backward reads them, no recompute (6*d*V flops/token)"}
        if "kd_dz_from_z" in fk:
            # HBM-bound: reads one chunk's kept logits and writes its dZ, bf16 [c, V] each
            zbytes = 2.0 * 2 * c * V
            gbs = zbytes / (fk["kd_dz_from_z"]["avg_ms"] * 1e-3) / 1e9
            fc["dz_from_z_roofline"] = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                                        "frac": gbs / peaks["hbm"], "bytes_per_launch": zbytes,
                                        "peak_source": f"{peaks['source']} copy bandwidth"}
        del z_store
        torch.cuda.empty_cache()
    dense = None
    if not args.no_modes and rank == 0:
        dense = dense_torch_reference(H, W, ids, tlog, mask, dev)

    # ---- offline cache extraction (kd_topk_cache) on the mid workload's dense teacher logits
    topk = None
    if not args.no_topk and rank == 0:
        topk = bench_topk(kd, dev, stream, peaks, args.steps)
    teacher = None
    if not args.no_teacher and rank == 0:
        teacher = bench_teacher_topk(kd, dev, stream, peaks, args.steps)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        from synth import bf16_bits
        r = args.cpu_rows
        dt = cpu_oracle_seconds(bf16_bits(H[:r]), bf16_bits(W), ids[:r].cpu().numpy(), tlog[:r].cpu().numpy(),
                                None if mask is None else mask[:r].cpu().numpy())
        rate = r / dt
        cpu = {"value": rate, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"{args.cpu_rows} positions of {w.name} (float64 numpy, fused formulation, fwd+bwd incl. "
                         f"full grad_W) in {dt:.1f} s, extrapolated per position"}

    # ---- the other four workloads, each measured the same way (the gpt-oss one is the line's value)
    configs = None
    if rank == 0 and not args.no_configs:
        del H, W, ids, tlog, mask, ws, grad_H, grad_W
        torch.cuda.empty_cache()
        configs = {}
        for name in ("tiny", "small", "mid", "gptoss", "headline"):
            if name == w.name:
                configs[name] = {"tokens_per_s": tokens_per_s, "ms_per_step": ms, "tflops_executed": tflops_exec,
                                 "tflops_useful": w.flops_useful() / (ms * 1e-3) / 1e12,
                                 "frac_of_bf16_peak": tflops_exec / peak, "peak_device_gb": peak_alloc / 1e9,
                                 "workspace_gb": ws_gb, "inputs_gb": inputs_alloc / 1e9,
                                 "dense_torch": dense if dense is not None else
                                 {"fits": False, "estimate_gb": dense_estimate_gb(w)}}
            else:
                configs[name] = bench_fused(kd, dev, stream, WORKLOADS[name], args.steps, args.warmup, peaks)

    if rank == 0:
        clk = clocks.summary()

        def brief(x, keys):
            return None if x is None else {k: x[k] for k in keys if k in x}
        topk_brief = None if topk is None else {
            "ms": topk["ids+vals"]["ms"], "achieved_gbs": topk["ids+vals"]["achieved_gbs"],
            "frac_of_hbm": topk["ids+vals"]["frac"], "ms_with_lse": topk["ids+vals+lse"]["ms"],
            "scale_spread_ms": {k: v["ms"] for k, v in topk.get("scale_spread", {}).items()},
            "prefix_high_ms": topk.get("prefix_high", {}).get("ms")}
        teacher_brief = brief(teacher, ("ms", "positions_per_s", "projection_tflops", "frac_of_bf16_peak",
                                        "ms_with_lse_and_dropped"))
        def config_brief(v):
            dt = v["dense_torch"]
            out = {"tokens_per_s": v["tokens_per_s"], "tflops": v["tflops_executed"],
                   "frac_of_bf16_peak": v["frac_of_bf16_peak"], "peak_gb": v["peak_device_gb"],
                   "workspace_gb": v["workspace_gb"]}
            if dt.get("fits"):
                out["dense_torch_gb"] = dt["peak_device_gb"]
            else:
                out["dense_torch_estimate_gb"] = dt.get("estimate_gb")
            return out

        configs_brief = None if configs is None else {k: config_brief(v) for k, v in configs.items()}
        def r4(x):
            """Numbers of the closing summaries to four significant digits."""
            if isinstance(x, float):
                return float(f"{x:.4g}")
            if isinstance(x, dict):
                return {k: r4(v) for k, v in x.items()}
            return x

        # Contract keys first, details next; the short summaries close the line, where a reader
        # keeping only the end of the output still finds them.
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_dict(w, world),
            "roofline": {"bound": "tensor", "kernel": dom_name, "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": ncu_traffic(dom_name, w.name),
                         "peak_source": f"{peaks['source']} bf16 sustained",
                         "flops_per_launch": gemm_flops_per_chunk},
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clk,
            "gpu_launches": launches,
            "kernels": kernels,
            "dense_torch_reference": dense,
            "forward_chunked": fc,
            "topk_cache": topk,
            "teacher_topk": teacher,
            "configs_detail": configs,
            "tflops_executed": tflops_exec,
            "tflops_useful": w.flops_useful() / (ms * 1e-3) / 1e12,
            "frac_of_bf16_peak": tflops_exec / peak,
            "peak_device_gb": peak_alloc / 1e9,
            "workspace_gb": ws_gb,
            "inputs_gb": inputs_alloc / 1e9,
            "clock_normalised": None if not clk.get("sm_mhz") else {
                "ms_per_step_x_ghz": ms * clk["sm_mhz"] / 1000.0,
                "tokens_per_s_per_ghz": tokens_per_s / (clk["sm_mhz"] / 1000.0)},
            "configs": r4(configs_brief),
            "teacher_topk_brief": r4(teacher_brief),
            "topk": r4(topk_brief),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()  # the other ranks wait while rank 0 measures the extra legs, then all leave together
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
