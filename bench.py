"""Benchmark: paged block-sparse prefill on one GB300 (or N independent replicas).

One step = the whole hot path on one batch: plan (host) + metadata upload, page indexer,
top-k, sparse forward (with its page -> row inversion) and LSE combine, on the 8192-token
BF16 prefill workload (32 query / 2 KV heads, head dim 128, 128-token pages, top-16,
permuted physical pages).  Inputs are resident in HBM before timing; L2 is flushed
(256 MB write) between timed steps and each step is timed with CUDA events on the launching
stream.  ``e2e`` repeats the step through the same C-ABI calls starting from pinned host
buffers (H2D of Q/K/V/page table and D2H of the output inside the timed region).

``--impl reference`` times the FP64 CPU oracle instead (a bounded row sample per step).

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-prefill tokens/s on 1 GB300; combine HBM GB/s and fwd tensor-pipe % of peak"
WORKLOAD = "prefill8k"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
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
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def max_over_ranks(values, world: int):
    """Element-wise maximum of per-rank timings over all ranks (identity on one rank)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tokens_per_s(tokens_per_rank: int, world: int, slowest_ms: float) -> float:
    """Whole-job throughput: every rank processed its own batch within the slowest rank's time."""
    return tokens_per_rank * world / (slowest_ms * 1e-3)


def _algorithmic(w, idx_np):
    """Algorithmic bytes / FLOPs of each step for this batch (minimum traffic)."""
    R, K, D, H = w.num_rows, w.top_k, w.head_dim, w.num_q_heads
    tok_pos = np.concatenate([c + np.arange(q) for q, c in zip(w.q_lens, w.ctx_lens)])
    pos = np.repeat(tok_pos, H)  # per row
    o = pos // 128
    n_sel = np.minimum(K, o + 1)
    filled = int(n_sel.sum())
    vis_keys = int((o * 128 + (pos % 128) + 1).sum())
    # keys visible inside the selected pages (own page only to t)
    sel_keys = 0
    if idx_np is not None:
        own_sel = (idx_np == o[:, None]).sum(1)
        sel_keys = int(((idx_np >= 0).sum(1) - own_sel).sum() * 128 + (own_sel * (pos % 128 + 1)).sum())
    kv_bytes = w.num_phys_pages * w.num_kv_heads * 128 * D * 2 * 2
    return {
        "indexer_flops": 2.0 * D * vis_keys,
        "indexer_bytes": R * D * 2 + kv_bytes / 2 + int((o + 1).sum()) * 4,
        "topk_bytes": int((o + 1).sum()) * 4 + R * K * 4,
        "fwd_flops": 4.0 * D * sel_keys,
        "fwd_bytes": filled * D * 4 + R * K * 4 + R * D * 2 + kv_bytes + R * K * 4,
        "combine_bytes": filled * D * 4 + R * K * 4 + R * D * 2 + R * 4,
        "filled_slots": filled,
    }


def _workload(args):
    from paged_top_sparse_gb300 import synth

    if args.tokens == 8192:
        return synth.workload(WORKLOAD, seed=args.seed)
    # same shape with another prefill length (used for profiling captures)
    return synth.workload("custom", seed=args.seed, q_lens=[args.tokens], ctx_lens=[0],
                          num_q_heads=32, num_kv_heads=2, head_dim=128, top_k=16)


def run_gpu(args, rank, world):
    import torch

    from paged_top_sparse_gb300 import binding as B
    from paged_top_sparse_gb300 import build, synth

    build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = _workload(args)
    t = synth.make_tensors(w)
    R, K, D = w.num_rows, w.top_k, w.head_dim

    def todev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    q, kc, vc = todev(t["q"]), todev(t["k"]), todev(t["v"])
    pt = todev(w.page_table.astype(np.int32))
    plan_args = (w.q_lens, w.ctx_lens, w.num_q_heads, w.num_kv_heads, D, K, w.max_pages,
                 w.num_phys_pages)
    plan = B.Plan(*plan_args, softmax_scale=w.sm_scale)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    scores = torch.empty((R, w.max_pages), dtype=torch.float32, device=dev)
    idx = torch.empty((R, K), dtype=torch.int32, device=dev)
    partial = torch.empty((K, R, D), dtype=torch.float32, device=dev)
    lse = torch.empty((K, R), dtype=torch.float32, device=dev)
    out = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(q_, kc_, vc_, pt_, ev=None):
        pl = B.Plan(*plan_args, softmax_scale=w.sm_scale)
        if ev: ev[0].record(stream)
        B.sps_plan_upload(pl, ws)
        B.indexer_scores(pl, q_, 1.0, kc_, None, 1.0, pt_, scores, ws)
        if ev: ev[1].record(stream)
        B.topk_select(pl, scores, idx, ws)
        if ev: ev[2].record(stream)
        B.sparse_prefill_fwd(pl, q_, 1.0, kc_, vc_, None, None, pt_, idx, partial, lse, ws)
        if ev: ev[3].record(stream)
        B.partial_combine(partial, lse, out)
        if ev: ev[4].record(stream)
        return pl

    for _ in range(args.warmup):
        step(q, kc, vc, pt)
    torch.cuda.synchronize()
    assert B.sps_read_device_status(plan, ws) == 0

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    clocks = ClockSampler(dev.index)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        step(q, kc, vc, pt, evs[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    barrier()
    per = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(4)]
                    for i in range(args.steps)])  # ms
    step_ms = float(per.sum(1).mean())

    # ---- end-to-end through the same calls, from pinned host buffers
    hq = torch.from_numpy(np.ascontiguousarray(t["q"]).view(np.int16)).pin_memory()
    hk = torch.from_numpy(np.ascontiguousarray(t["k"]).view(np.int16)).pin_memory()
    hv = torch.from_numpy(np.ascontiguousarray(t["v"]).view(np.int16)).pin_memory()
    hpt = torch.from_numpy(w.page_table.astype(np.int32)).pin_memory()
    hout = torch.empty((R, D), dtype=torch.bfloat16).pin_memory()
    dq, dk, dv, dpt = (torch.empty_like(x, device=dev) for x in (hq, hk, hv, hpt))
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hpt))
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        for d_, h_ in ((dq, hq), (dk, hk), (dv, hv), (dpt, hpt)):
            d_.copy_(h_, non_blocking=True)
        step(dq, dk, dv, dpt)
        hout.copy_(out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for i in range(args.steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e_ms.append(a.elapsed_time(b))
    e2e_ms = float(np.mean(e_ms))
    clk = clocks.stop()

    step_ms, e2e_ms = max_over_ranks([step_ms, e2e_ms], world)

    alg = _algorithmic(w, idx.cpu().numpy())
    hbm, bf16, peak_kind = _peaks()
    k_ms = per.mean(0)
    names = ["indexer", "topk", "fwd", "combine"]
    kern = {
        "indexer": {"us": k_ms[0] * 1e3, "achieved": alg["indexer_flops"] / (k_ms[0] * 1e-3) / 1e12,
                    "unit": "TFLOP/s", "peak": bf16, "bound": "tensor"},
        "topk": {"us": k_ms[1] * 1e3, "achieved": alg["topk_bytes"] / (k_ms[1] * 1e-3) / 1e9,
                 "unit": "GB/s", "peak": hbm, "bound": "hbm"},
        "fwd": {"us": k_ms[2] * 1e3, "achieved": alg["fwd_bytes"] / (k_ms[2] * 1e-3) / 1e9,
                "unit": "GB/s", "peak": hbm, "bound": "hbm",
                "tensor_tflops": alg["fwd_flops"] / (k_ms[2] * 1e-3) / 1e12},
        "combine": {"us": k_ms[3] * 1e3, "achieved": alg["combine_bytes"] / (k_ms[3] * 1e-3) / 1e9,
                    "unit": "GB/s", "peak": hbm, "bound": "hbm"},
    }
    for v in kern.values():
        v["frac"] = v["achieved"] / v["peak"]
        for kk in ("us", "achieved", "frac"):
            v[kk] = round(float(v[kk]), 4)
    kern["fwd"]["tensor_frac"] = round(kern["fwd"]["tensor_tflops"] / bf16, 4)
    dom = names[int(np.argmax(k_ms))]
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            traffic = json.load(f).get(dom)
    except Exception:
        pass
    line = {
        "metric": METRIC,
        "value": round(job_tokens_per_s(w.num_tokens, world, step_ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) BF16 Q/K/V, permuted page table)",
        "config": {"workload": f"prefill {w.num_tokens} tokens, 32 q / 2 kv heads, head_dim 128, "
                               "page 128, top-16, BF16 (permuted physical pages)",
                   "batch": 1, "seq_len": w.num_tokens, "rows": R,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps (256 MB write); per-step CUDA events"},
        "roofline": {"bound": kern[dom]["bound"], "kernel": dom,
                     "achieved": kern[dom]["achieved"], "peak": kern[dom]["peak"],
                     "unit": kern[dom]["unit"], "frac": kern[dom]["frac"],
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json burst)" if peak_kind == "measured" else "fallback",
                     "traffic": traffic},
        "kernels": kern,
        "combine_hbm_gbs": kern["combine"]["achieved"],
        "fwd_tensor_pipe_frac": kern["fwd"]["tensor_frac"],
        "e2e": {"value": round(job_tokens_per_s(w.num_tokens, world, e2e_ms), 1), "unit": "tokens/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 9 * args.steps,
        "clocks": clk,
        "wall_s_timed": round(t_wall, 3),
    }
    return line, w, t


def cpu_baseline(w, t, budget_s: float, seed: int = 7):
    """The oracle as it stands (indexer -> top-k -> forward -> combine) on a random row sample,
    sized to about budget_s of CPU work; returns tokens/s scaled from rows/s."""
    from oracle import oracle as orc
    from tests.helpers import oracle_problem, oracle_tensors

    pb = oracle_problem(w)
    q, k, v, qi, ki = oracle_tensors(w, t)
    rng = np.random.default_rng(seed)
    n = 256
    t0 = time.perf_counter()
    orc.pipeline(pb, q, k, v, w.sm_scale, qi, ki, rows=np.sort(rng.choice(w.num_rows, n, replace=False)))
    dt = time.perf_counter() - t0
    n2 = int(min(w.num_rows, max(n, n * budget_s / max(dt, 1e-3))))
    rows = np.sort(rng.choice(w.num_rows, n2, replace=False))
    t0 = time.perf_counter()
    orc.pipeline(pb, q, k, v, w.sm_scale, qi, ki, rows=rows)
    dt2 = time.perf_counter() - t0
    rows_per_s = n2 / dt2
    return {"value": round(rows_per_s / w.num_q_heads, 2), "unit": "tokens/s",
            "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"{n2} random (token, head) rows of the 8192-token workload, all four steps, "
                      f"{dt2:.1f} s; tokens/s = rows/s / 32 heads"}


def run_reference(args, rank, world):
    """Reference arm: the FP64 CPU oracle on host cores (rank 0 only)."""
    from paged_top_sparse_gb300 import synth

    w = synth.workload(WORKLOAD, seed=args.seed)
    t = synth.make_tensors(w)
    budget = float(os.environ.get("SPS_REF_STEP_S", "8"))
    for _ in range(args.warmup):
        cpu_baseline(w, t, budget_s=0.5)
    vals = [cpu_baseline(w, t, budget_s=budget) for _ in range(args.steps)]
    v = float(np.mean([x["value"] for x in vals]))
    cb = dict(vals[-1])
    cb["value"] = round(v, 2)
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(8192 / v * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill 8192 tokens, 32 q / 2 kv heads, head_dim 128, page 128, "
                               "top-16, BF16 (permuted physical pages)", "batch": 1, "seq_len": 8192},
        "cpu_baseline": cb,
        "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=8192,
                    help="prefill length (8192 = the benchmark workload; others for profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "native" else args.warmup
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            dist.init_process_group("nccl")
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, 1)))
        return
    line, w, t = run_gpu(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, t, budget_s=float(os.environ.get("SPS_CPU_S", "12")))
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
