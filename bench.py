"""Benchmark: paged block-sparse prefill on one GB300 (or N independent replicas).

One step = the whole hot path on one batch: plan (host) + metadata upload, page indexer,
top-k, sparse forward (with its page -> row inversion) and LSE combine, on the 8192-token
BF16 prefill workload (32 query / 2 KV heads, head dim 128, 128-token pages, top-16,
permuted physical pages).  Inputs are resident in HBM before timing; L2 is flushed
(256 MB write) between timed steps and each step is timed with CUDA events on the launching
stream.  ``e2e`` repeats the step through the same C-ABI calls starting from pinned host
buffers (H2D of Q/K/V/page table and D2H of the output inside the timed region), with each
step's copies on their own streams overlapping the neighbouring steps' compute; the serial
form (copy in, step, copy out, one after another) is reported beside it.

The default line (the 8K BF16 prefill with FP32 partials) also carries, under ``configs``, the
same measurement of every other configuration of the method's workloads: the 8K prefill with
FP16 and with BF16 partials, the quantised 8K prefill (exact route and the FP8 route), the
combine stress (a 4.3 GB FP32 partial buffer), the chunked batch (8 x 512 new tokens over
~32K of context) and 512 new tokens at the end of a 1M-token context; ``--no-configs`` skips
them.

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

    def wait_ready(self, timeout_s: float = 10.0):
        """Blocks until nvidia-smi has printed its first sample: starting it (NVML setup) must
        not overlap the timed region."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout_s:
            time.sleep(0.01)

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


def _algorithmic(w, idx_np, partial_bytes=4):
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
    # K and V caches read once: 2 bytes per element, or an NVFP4 nibble plus a scale per 16
    elem = (0.5 + 1.0 / 16) if w.kv_dtype == "nvfp4" else 2.0
    kv_bytes = int(w.num_phys_pages * w.num_kv_heads * 128 * D * elem * 2)
    return {
        "indexer_flops": 2.0 * D * vis_keys,
        "indexer_bytes": R * D * (1 if w.q_dtype == "e4m3" else 2) + kv_bytes // 2
                         + int((o + 1).sum()) * 4,
        "topk_bytes": int((o + 1).sum()) * 4 + R * K * 4,
        "fwd_flops": 4.0 * D * sel_keys,
        "fwd_bytes": filled * D * partial_bytes + R * K * 4 + R * D * (1 if w.q_dtype == "e4m3" else 2)
                     + kv_bytes + R * K * 4,
        "combine_bytes": filled * D * partial_bytes + R * K * 4 + R * D * 2 + R * 4,
        "filled_slots": filled,
    }


WORKLOADS = ("prefill8k", "prefill8k_q", "chunked32k", "combine_stress", "kv_append", "ctx1m")


def _describe(w, name):
    if name == "ctx1m":
        return (f"long context: 512 new tokens after {int(w.ctx_lens[0])} cached (1M tokens, "
                f"{w.max_pages} pages), 32 q / 2 kv heads, head_dim 128, page 128, top-16, BF16 "
                "(permuted physical pages)")
    if name == "chunked32k":
        return (f"chunked prefill: {w.batch} requests x 512 new tokens over {min(w.ctx_lens)}.."
                f"{max(w.ctx_lens)} cached, 32 q / 2 kv heads, head_dim 128, page 128, top-16, "
                "E4M3 indexer q/k, BF16 attention, shared permuted page pool")
    quant = ("E4M3 Q (per-tensor scale), NVFP4 K/V (E4M3 scale per 16)" if w.kv_dtype == "nvfp4"
             else "BF16")
    return (f"prefill {w.num_tokens} tokens, 32 q / 2 kv heads, head_dim 128, page 128, top-16, "
            f"{quant} (permuted physical pages)")


def _host_inputs(w, t):
    """Host arrays one step reads, by name (the end-to-end step copies every one of them)."""
    d = {"q": t["q"], "k": t["k"], "v": t["v"], "pt": w.page_table.astype(np.int32)}
    if w.kv_dtype == "nvfp4":
        d["k_scales"], d["v_scales"] = t["k_scales"], t["v_scales"]
    if w.idx_dtype == "e4m3":
        d["q_idx"], d["k_idx"] = t["q_idx"], t["k_idx"]
    return d


def _pinned(a):
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).pin_memory()


def _timed_loop(args, world, dev, flush, step, nseg):
    """W untimed steps, then K steps each bracketed by nseg+1 events on the launching stream."""
    import torch

    stream = torch.cuda.current_stream()
    clocks = ClockSampler(dev.index)
    clocks.start()
    clocks.wait_ready()
    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nseg + 1)]
           for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        step(evs[i])
    t_enq = time.perf_counter() - t_wall0
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    barrier()
    per = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(nseg)]
                    for i in range(args.steps)])  # ms
    # the same steps with events at their boundaries only: events between the kernels keep
    # each kernel from starting its prologue while the previous one drains (programmatic
    # dependent launch), so the whole-step time comes from this pass
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(float(i))
        bev[i][0].record(stream)
        step(None)
        bev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks.step_ms = np.array([bev[i][0].elapsed_time(bev[i][1]) for i in range(args.steps)])
    # device time between one step's last event and the next step's first (the L2 flush, plus
    # any wait for the host)
    gaps = [evs[i][nseg].elapsed_time(evs[i + 1][0]) for i in range(args.steps - 1)]
    clocks.host = {"enqueue_ms_per_step": round(t_enq * 1e3 / args.steps, 4),
                   "between_steps_ms": round(float(np.mean(gaps)), 4) if gaps else None}
    return per, clocks, t_wall, stream


def _e2e(args, flush, stream, copy_in, step, copy_out):
    import torch

    def e2e_step():
        copy_in()
        step(None)
        copy_out()

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
    return float(np.mean(e_ms))


def _byte_chunks(pairs, chunk_bytes=16 << 20):
    """Split (device dst, pinned host src) tensor pairs into byte slices of at most chunk_bytes."""
    import torch

    out = []
    for d, h in pairs:
        db, hb = d.reshape(-1).view(torch.uint8), h.reshape(-1).view(torch.uint8)
        for i in range(0, hb.numel(), chunk_bytes):
            out.append((db[i:i + chunk_bytes], hb[i:i + chunk_bytes]))
    return out


def _e2e_pipelined(args, flush, stream, in_pairs, step, copy_out, nbuf=2):
    """End-to-end throughput with the copies overlapped: every step's H2D copies run on their
    own streams (`--h2d-streams` of them, the inputs cut into 16 MB slices dealt round-robin,
    into one of `nbuf` device input sets) and its D2H copy on another, while the launching
    stream computes the neighbouring steps.  All copies of the K timed steps are inside the
    timed region (events from the first H2D to the last D2H)."""
    import torch

    nh = max(1, args.h2d_streams)
    h2d_s = [torch.cuda.Stream() for _ in range(nh)]
    d2h_s = torch.cuda.Stream()
    slices = [_byte_chunks(in_pairs(b)) for b in range(nbuf)]
    in_ready = [[torch.cuda.Event() for _ in range(nh)] for _ in range(nbuf)]
    used = [torch.cuda.Event() for _ in range(nbuf)]   # compute of the set's last step done
    read = [torch.cuda.Event() for _ in range(nbuf)]   # D2H of the set's last output done

    def run(n, first=None):
        for i in range(n):
            b = i % nbuf
            if i == 0 and first is not None:
                first.record(h2d_s[0])
                for s_ in h2d_s[1:]:
                    s_.wait_event(first)
            for j, s_ in enumerate(h2d_s):
                if i >= nbuf:
                    s_.wait_event(used[b])
                with torch.cuda.stream(s_):
                    for d_, h_ in slices[b][j::nh]:
                        d_.copy_(h_, non_blocking=True)
                in_ready[b][j].record(s_)
                stream.wait_event(in_ready[b][j])
            if i >= nbuf:
                stream.wait_event(read[b])
            with torch.cuda.stream(stream):
                flush.fill_(float(i))
                step(b)
            used[b].record(stream)
            d2h_s.wait_event(used[b])
            with torch.cuda.stream(d2h_s):
                copy_out(b)
            read[b].record(d2h_s)
        return read[(n - 1) % nbuf]

    run(max(1, args.warmup))
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    last = run(args.steps, first=t0)
    stream.wait_event(last)
    t1.record(stream)
    t1.synchronize()
    return t0.elapsed_time(t1) / args.steps


def _topk_launches(w):
    """Top-k kernels of one call: three (segments' pass 1, the rows, segments' pass 2) when the
    plan splits long rows (top_k <= 16, 64 or more 16-page groups, few enough rows that the
    split pays: the plan's own rule), else one."""
    groups = (w.max_pages + 15) // 16
    if not (1 < w.top_k <= 16 and groups >= 64 and w.num_rows >= 32):
        return 1
    warps = (w.num_rows + 31) // 32
    return 3 if min(groups // 32, -(-(24 * 152) // warps)) >= 2 else 1


def _launches_per_step(w, fp8qk, inv_launches):
    """Kernels of this library one step launches: plan upload, indexer, top-k (one, or three
    over long rows), the inversion (one cooperative launch, or four kernels), forward,
    combine, plus the quantised paths' copies (the indexer's FP16 Q and visible key pages over
    NVFP4 keys; the forward's FP16 Q on the exact route)."""
    n = 4 + _topk_launches(w) + inv_launches
    if w.idx_dtype != "e4m3" and w.kv_dtype == "nvfp4":
        n += 2
    if w.q_dtype == "e4m3" and not fp8qk:
        n += 1
    return n


def run_prefill(args, world, dev, wname, partials="fp32", fp8qk=False, data=None):
    """One workload through the four C-ABI calls: the device-timed step, the end-to-end step
    from pinned host buffers, and the per-kernel roofline fractions.  Returns (line, w, t)."""
    import torch

    from paged_top_sparse_gb300 import binding as B
    from paged_top_sparse_gb300 import synth

    if data is None:
        if wname == "prefill8k" and args.tokens != 8192:
            # same shape with another prefill length (used for profiling captures)
            w = synth.workload("custom", seed=args.seed, q_lens=[args.tokens], ctx_lens=[0],
                               num_q_heads=32, num_kv_heads=2, head_dim=128, top_k=16)
        else:
            w = synth.workload(wname, seed=args.seed)
        t = synth.make_tensors(w)
    else:
        w, t = data
    R, K, D = w.num_rows, w.top_k, w.head_dim
    host = _host_inputs(w, t)
    hin = {k: _pinned(v) for k, v in host.items()}
    din = {k: x.to(dev) for k, x in hin.items()}
    q_scale = float(t.get("q_scale", 1.0))
    idx_fp8 = w.idx_dtype == "e4m3"
    idx_q, idx_k = ("e4m3", "e4m3") if idx_fp8 else (w.q_dtype, w.kv_dtype)
    plan_args = (w.q_lens, w.ctx_lens, w.num_q_heads, w.num_kv_heads, D, K, w.max_pages,
                 w.num_phys_pages)
    plan_kw = dict(q_dtype=w.q_dtype, kv_dtype=w.kv_dtype, idx_q_dtype=idx_q,
                   idx_k_dtype=idx_k, softmax_scale=w.sm_scale)
    plan = B.Plan(*plan_args, **plan_kw)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    # row pitch a multiple of 4 floats (16-byte rows), as indexer_scores asks
    pitch = (w.max_pages + 3) // 4 * 4
    scores = torch.empty((R, pitch), dtype=torch.float32, device=dev)[:, : w.max_pages]
    idx = torch.empty((R, K), dtype=torch.int32, device=dev)
    p16 = partials != "fp32"  # 16-bit partial storage (BF16 or FP16)
    pdt = {"fp32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[partials]
    partial = torch.empty((K, R, D), dtype=pdt, device=dev)
    lse = torch.empty((K, R), dtype=torch.float32, device=dev)
    out = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    fwd_call = {"fp32": B.sparse_prefill_fwd, "bf16": B.sparse_prefill_fwd_bf16,
                "f16": B.sparse_prefill_fwd_f16}[partials]
    if fp8qk:
        if p16 or w.kv_dtype != "nvfp4":
            raise SystemExit("--fp8qk needs the quantised workload (prefill8k_q) and FP32 partials")
        fwd_call = B.sparse_prefill_fwd_fp8qk
    combine_call = {"fp32": B.partial_combine, "bf16": B.partial_combine_bf16,
                    "f16": B.partial_combine_f16}[partials]

    def step(ev, di=din, out_=out):
        pl = B.Plan(*plan_args, **plan_kw)
        if ev: ev[0].record(stream)
        B.sps_plan_upload(pl, ws)
        if idx_fp8:
            B.indexer_scores(pl, di["q_idx"], float(t["q_idx_scale"]), di["k_idx"], None,
                             float(t["k_idx_scale"]), di["pt"], scores, ws)
        else:
            B.indexer_scores(pl, di["q"], q_scale, di["k"], di.get("k_scales"), 1.0, di["pt"],
                             scores, ws)
        if ev: ev[1].record(stream)
        B.topk_select(pl, scores, idx, ws)
        if ev: ev[2].record(stream)
        fwd_call(pl, di["q"], q_scale, di["k"], di["v"], di.get("k_scales"),
                 di.get("v_scales"), di["pt"], idx, partial, lse, ws)
        if ev: ev[3].record(stream)
        combine_call(partial, lse, out_)
        if ev: ev[4].record(stream)
        return pl

    per, clocks, t_wall, stream = _timed_loop(args, world, dev, flush, step, 4)
    assert B.sps_read_device_status(plan, ws) == 0
    step_ms = float(clocks.step_ms.mean())
    step_ms_segmented = float(per.sum(1).mean())

    # ---- end to end through the same calls, from pinned host buffers
    hout = torch.empty((R, D), dtype=torch.bfloat16).pin_memory()
    dcopy = {k: torch.empty_like(x, device=dev) for k, x in hin.items()}
    h2d = sum(x.numel() * x.element_size() for x in hin.values())
    d2h = hout.numel() * hout.element_size()

    def copy_in():
        for k_, h_ in hin.items():
            dcopy[k_].copy_(h_, non_blocking=True)

    e2e_serial_ms = _e2e(args, flush, stream, copy_in, lambda ev: step(ev, dcopy),
                         lambda: hout.copy_(out, non_blocking=True))
    dsets = [{k: torch.empty_like(x, device=dev) for k, x in hin.items()} for _ in range(2)]
    douts = [torch.empty_like(out) for _ in range(2)]

    e2e_ms = _e2e_pipelined(args, flush, stream,
                            lambda b: [(dsets[b][k_], h_) for k_, h_ in hin.items()],
                            lambda b: step(None, dsets[b], douts[b]),
                            lambda b: hout.copy_(douts[b], non_blocking=True))
    assert torch.equal(douts[(args.steps - 1) % 2], out), "pipelined e2e output differs"
    clk = clocks.stop()

    step_ms, step_ms_segmented, e2e_ms, e2e_serial_ms = max_over_ranks(
        [step_ms, step_ms_segmented, e2e_ms, e2e_serial_ms], world)

    alg = _algorithmic(w, idx.cpu().numpy(), partial_bytes=2 if p16 else 4)
    hbm, bf16, peak_kind = _peaks()
    src = "measured (MEASURED_PEAKS.json burst)" if peak_kind == "measured" else "fallback"
    idx_peak = bf16 * 2 if idx_fp8 else bf16  # FP8 tensor rate: the nominal 2x of BF16
    k_ms = per.mean(0)
    names = ["indexer", "topk", "fwd", "combine"]
    # the inversion is one cooperative launch when its 256-row blocks fit on the GPU at once
    # (8 per SM) and no request sees more than 1024 pages, else four kernels
    hg = w.num_q_heads // w.num_kv_heads
    inv_blocks = sum(w.num_kv_heads * -(-(-(-ql * hg // 32)) // 8) for ql in w.q_lens)
    fits = inv_blocks <= 8 * torch.cuda.get_device_properties(dev).multi_processor_count
    inv_launches = 1 if fits and w.max_pages <= 1024 else 4
    kern = {
        "indexer": {"us": k_ms[0] * 1e3, "achieved": alg["indexer_flops"] / (k_ms[0] * 1e-3) / 1e12,
                    "unit": "TFLOP/s", "peak": idx_peak, "bound": "tensor",
                    "peak_source": ("2 x " + src + " BF16 (nominal FP8/BF16 rate ratio)")
                    if idx_fp8 else src + " BF16"},
        "topk": {"us": k_ms[1] * 1e3, "achieved": alg["topk_bytes"] / (k_ms[1] * 1e-3) / 1e9,
                 "unit": "GB/s", "peak": hbm, "bound": "hbm", "peak_source": src + " HBM"},
        "fwd": {"us": k_ms[2] * 1e3, "achieved": alg["fwd_bytes"] / (k_ms[2] * 1e-3) / 1e9,
                "unit": "GB/s", "peak": hbm, "bound": "hbm", "peak_source": src + " HBM",
                "tensor_tflops": alg["fwd_flops"] / (k_ms[2] * 1e-3) / 1e12},
        "combine": {"us": k_ms[3] * 1e3, "achieved": alg["combine_bytes"] / (k_ms[3] * 1e-3) / 1e9,
                    "unit": "GB/s", "peak": hbm, "bound": "hbm", "peak_source": src + " HBM"},
    }
    for v in kern.values():
        v["frac"] = v["achieved"] / v["peak"]
        for kk in ("us", "achieved", "frac"):
            v[kk] = round(float(v[kk]), 4)
    kern["fwd"]["tensor_frac"] = round(kern["fwd"]["tensor_tflops"] / bf16, 4)
    dom = names[int(np.argmax(k_ms))]
    traffic = None
    if wname == "prefill8k" and args.tokens == 8192 and not p16:  # the counters' workload
        try:
            with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
                traffic = json.load(f).get(dom)
        except Exception:
            pass
    storage = {"bf16": ", BF16 partials", "f16": ", FP16 partials"}.get(partials, "")
    line = {
        "metric": METRIC,
        "value": round(job_tokens_per_s(w.num_tokens, world, step_ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "ms_per_step_with_kernel_events": round(step_ms_segmented, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp16" if w.kv_dtype == "nvfp4" else "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, quantised where the workload says; permuted "
                "page table)",
        "config": {"workload": _describe(w, wname) + storage
                               + (", FP8 Q K^T on E4M3-rounded K" if fp8qk else ""),
                   "partials": partials,
                   "batch": int(w.batch), "seq_len": int(max(w.q_lens)), "rows": int(R),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps (256 MB write); CUDA events at step boundaries "
                         "(per-kernel times from a second pass with events between kernels)"},
        "roofline": {"bound": kern[dom]["bound"], "kernel": dom,
                     "achieved": kern[dom]["achieved"], "peak": kern[dom]["peak"],
                     "unit": kern[dom]["unit"], "frac": kern[dom]["frac"],
                     "peak_source": kern[dom]["peak_source"], "traffic": traffic},
        "kernels": kern,
        "combine_hbm_gbs": kern["combine"]["achieved"],
        "fwd_tensor_pipe_frac": kern["fwd"]["tensor_frac"],
        "e2e": {"value": round(job_tokens_per_s(w.num_tokens, world, e2e_ms), 1), "unit": "tokens/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "mode": f"pipelined: each step's H2D ({args.h2d_streams} stream(s)) and D2H on "
                        "their own streams, overlapping the neighbouring steps' compute; all "
                        "copies inside the timed region",
                "serial_ms_per_step": round(e2e_serial_ms, 4),
                "serial_value": round(job_tokens_per_s(w.num_tokens, world, e2e_serial_ms), 1)},
        "gpu_launches": _launches_per_step(w, fp8qk, inv_launches) * args.steps,
        "clocks": clk,
        "wall_s_timed": round(t_wall, 3),
        "host": clocks.host,
    }
    return line, w, t


def run_gpu(args, rank, world):
    import torch

    from paged_top_sparse_gb300 import build

    build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if args.workload == "combine_stress":
        return run_combine_stress(args, rank, world, dev)
    if args.workload == "kv_append":
        return run_kv_append(args, rank, world, dev)
    return run_prefill(args, world, dev, args.workload, args.partials, args.fp8qk)


def _sub(line):
    """The fields of a workload's line that the headline's `configs` key carries."""
    keys = ("value", "unit", "ms_per_step", "dtype", "roofline", "kernels", "e2e",
            "gpu_launches", "clocks")
    d = {k: line[k] for k in keys if k in line}
    d["workload"] = line["config"]["workload"]
    d["tokens_per_s"] = d.pop("value")
    return d


def run_other_configs(args, world, w0, t0):
    """Every other configuration of the method's workloads, each timed like the headline:
    the 8K prefill with 16-bit partials (FP16, BF16), the quantised 8K prefill (exact route
    and the FP8 route), the combine stress, the chunked 8 x 512-over-32K batch and 512 new
    tokens at the end of a 1M-token context."""
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    out = {}
    for key, wname, partials, fp8 in (("prefill8k_f16_partials", "prefill8k", "f16", False),
                                      ("prefill8k_bf16_partials", "prefill8k", "bf16", False)):
        line, _, _ = run_prefill(args, world, dev, wname, partials, fp8, data=(w0, t0))
        out[key] = _sub(line)
        torch.cuda.empty_cache()
    data = None
    for key, fp8 in (("prefill8k_q", False), ("prefill8k_q_fp8qk", True)):
        line, w, t = run_prefill(args, world, dev, "prefill8k_q", "fp32", fp8, data=data)
        data = (w, t)
        out[key] = _sub(line)
        torch.cuda.empty_cache()
    del data
    line, _, _ = run_combine_stress(args, 0, world, dev)
    out["combine_stress"] = _sub(line)
    torch.cuda.empty_cache()
    line, _, _ = run_prefill(args, world, dev, "chunked32k")
    out["chunked32k"] = _sub(line)
    torch.cuda.empty_cache()
    line, _, _ = run_prefill(args, world, dev, "ctx1m")
    out["ctx1m"] = _sub(line)
    torch.cuda.empty_cache()
    return out


def run_combine_stress(args, rank, world, dev):
    """The combine alone on the 16384-token stress buffer: partial [16][16384*32][128] FP32
    N(0,1), LSE N(0, sd 2); tokens/s = 16384 / combine time."""
    import torch

    from paged_top_sparse_gb300 import binding as B
    from paged_top_sparse_gb300 import synth

    T, H, S, D = 16384, 32, 16, 128
    R = T * H
    partial, lse = synth.combine_inputs(R, S, D, seed=args.seed, device=dev)
    out = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(ev, p_=partial, l_=lse):
        if ev: ev[0].record(torch.cuda.current_stream())
        B.partial_combine(p_, l_, out, dev_status=status)
        if ev: ev[1].record(torch.cuda.current_stream())

    per, clocks, t_wall, stream = _timed_loop(args, world, dev, flush, step, 1)
    assert int(status.item()) == 0
    comb_ms = float(per[:, 0].mean())
    # end to end: the partials and LSEs come from pinned host memory, the output goes back
    hp = torch.empty(partial.shape, dtype=torch.float32).pin_memory()
    hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    hp.copy_(partial)
    hl.copy_(lse)
    hout = torch.empty((R, D), dtype=torch.bfloat16).pin_memory()
    dp, dl = torch.empty_like(partial), torch.empty_like(lse)

    def copy_in():
        dp.copy_(hp, non_blocking=True)
        dl.copy_(hl, non_blocking=True)

    e2e_ms = _e2e(args, flush, stream, copy_in, lambda ev: step(ev, dp, dl),
                  lambda: hout.copy_(out, non_blocking=True))
    clk = clocks.stop()
    comb_ms, e2e_ms = max_over_ranks([comb_ms, e2e_ms], world)
    hbm, _, peak_kind = _peaks()
    alg_bytes = R * S * D * 4 + R * S * 4 + R * D * 2
    achieved = alg_bytes / (comb_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(job_tokens_per_s(T, world, comb_ms), 1),
        "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(comb_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) partials, N(0, sd 2) LSEs)",
        "config": {"workload": "combine stress: partial [16][16384*32][128] FP32 (4.3 GB) + LSE "
                               "-> BF16 output", "rows": R, "splits": S, "head_dim": D,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs (4.3 GB) far larger than L2; 256 MB flush between steps"},
        "roofline": {"bound": "hbm", "kernel": "combine", "achieved": round(achieved, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json burst) HBM"
                     if peak_kind == "measured" else "fallback",
                     "traffic": None},
        "kernels": {"combine": {"us": round(comb_ms * 1e3, 4), "achieved": round(achieved, 1),
                                "unit": "GB/s", "peak": hbm, "bound": "hbm",
                                "frac": round(achieved / hbm, 4)}},
        "combine_hbm_gbs": round(achieved, 1),
        "e2e": {"value": round(job_tokens_per_s(T, world, e2e_ms), 1), "unit": "tokens/s",
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": hp.numel() * 4 + hl.numel() * 4,
                "d2h_bytes_per_step": hout.numel() * 2},
        "gpu_launches": args.steps,
        "clocks": clk,
        "wall_s_timed": round(t_wall, 3),
        "host": clocks.host,
    }
    return line, None, None


def run_kv_append(args, rank, world, dev):
    """The chunked-prefill append alone: 8 requests x 512 new tokens (2 KV heads, D 128) into
    an NVFP4 paged cache over ~32K of context; tokens/s = new tokens / append time."""
    import torch

    from paged_top_sparse_gb300 import binding as B
    from paged_top_sparse_gb300 import synth

    base = synth.workload("chunked32k", seed=args.seed)
    w = synth.workload("custom", seed=args.seed, q_lens=list(base.q_lens),
                       ctx_lens=list(base.ctx_lens), num_q_heads=32, num_kv_heads=2,
                       head_dim=128, top_k=16, q_dtype="e4m3", kv_dtype="nvfp4")
    T, G, D, NP = w.num_tokens, w.num_kv_heads, w.head_dim, w.num_phys_pages
    rng = np.random.default_rng(args.seed)
    knew = synth.f32_to_bf16_bits(rng.standard_normal((T, G, D)).astype(np.float32))
    vnew = synth.f32_to_bf16_bits(rng.standard_normal((T, G, D)).astype(np.float32))
    hk, hv = _pinned(knew), _pinned(vnew)
    dk, dv = hk.to(dev), hv.to(dev)
    kc = torch.zeros((NP, G, 128, D // 2), dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    ks = torch.zeros((NP, G, 128, D // 16), dtype=torch.uint8, device=dev)
    vs = torch.zeros_like(ks)
    pt = torch.from_numpy(w.page_table.astype(np.int32)).to(dev)
    plan = B.Plan(w.q_lens, w.ctx_lens, w.num_q_heads, G, D, w.top_k, w.max_pages, NP,
                  q_dtype="e4m3", kv_dtype="nvfp4")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    B.sps_plan_upload(plan, ws)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step(ev, k_=dk, v_=dv):
        if ev: ev[0].record(torch.cuda.current_stream())
        B.sps_kv_append(plan, k_, v_, pt, kc, vc, ks, vs, ws)
        if ev: ev[1].record(torch.cuda.current_stream())

    per, clocks, t_wall, stream = _timed_loop(args, world, dev, flush, step, 1)
    assert B.sps_read_device_status(plan, ws) == 0
    ms = float(per[:, 0].mean())
    ek, ev_ = torch.empty_like(dk), torch.empty_like(dv)

    def copy_in():
        ek.copy_(hk, non_blocking=True)
        ev_.copy_(hv, non_blocking=True)

    e2e_ms = _e2e(args, flush, stream, copy_in, lambda e: step(e, ek, ev_), lambda: None)
    clk = clocks.stop()
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], world)
    hbm, _, peak_kind = _peaks()
    alg = T * G * D * 2 * 2 + T * G * (D // 2 + D // 16) * 2  # read BF16 K/V, write codes + scales
    ach = alg / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(job_tokens_per_s(T, world, ms), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) BF16 K/V)",
        "config": {"workload": f"kv append: {w.batch} requests x 512 new tokens into an NVFP4 "
                               f"paged cache over {min(w.ctx_lens)}..{max(w.ctx_lens)} cached, "
                               "2 KV heads, head_dim 128", "tokens": int(T),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "256 MB flush between steps"},
        "roofline": {"bound": "hbm", "kernel": "kv_append", "achieved": round(ach, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json burst)"
                     if peak_kind == "measured" else "fallback", "traffic": None},
        "e2e": {"value": round(job_tokens_per_s(T, world, e2e_ms), 1), "unit": "tokens/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": hk.numel() * 2 * 2,
                "d2h_bytes_per_step": 0},
        "gpu_launches": args.steps,
        "clocks": clk,
        "wall_s_timed": round(t_wall, 3),
        "host": clocks.host,
    }
    return line, None, None


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
            "sample": f"{n2} random (token, head) rows of the {w.num_tokens}-token workload, all "
                      f"four steps, {dt2:.1f} s; tokens/s = rows/s / {w.num_q_heads} heads"}


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
                               "top-16, BF16 (permuted physical pages)", "batch": 1, "seq_len": 8192,
                   "sampling": "row-sampled: each step runs all four oracle steps on a random "
                               "sample of (token, head) rows (about " + str(int(budget)) + " s of "
                               "CPU work); tokens/s and ms_per_step are scaled from rows/s to the "
                               "whole 8192-token workload"},
        "cpu_baseline": cb,
        "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _json_default(o):
    """numpy scalars in the line print as plain numbers"""
    if isinstance(o, np.generic):
        return o.item()
    raise TypeError(f"{type(o).__name__} is not JSON serializable")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="headline workload only: skip the other configurations that the "
                         "default line carries under `configs`")
    ap.add_argument("--h2d-streams", type=int, default=1,
                    help="streams that share each step's host-to-device input copies in the "
                         "pipelined end-to-end measurement")
    ap.add_argument("--tokens", type=int, default=8192,
                    help="prefill length (8192 = the benchmark workload; others for profiling)")
    ap.add_argument("--workload", default="prefill8k", choices=WORKLOADS,
                    help="prefill8k (default: the headline line), prefill8k_q (E4M3 Q, NVFP4 "
                         "K/V), chunked32k (8 x 512 over 32K context), combine_stress, ctx1m "
                         "(512 new tokens at the end of a 1M-token context)")
    ap.add_argument("--fp8qk", action="store_true",
                    help="quantised workload only: the pages' Q8KV4 route (K rounded to E4M3, "
                         "FP8 Q K^T) through sparse_prefill_fwd_fp8qk")
    ap.add_argument("--partials", default="fp32", choices=["fp32", "bf16", "f16"],
                    help="partial storage: fp32 (the contract; default), or the pages' 16-bit "
                         "storage, bf16 or f16 (sparse_prefill_fwd_{bf16,f16} + "
                         "partial_combine_{bf16,f16})")
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
            print(json.dumps(run_reference(args, rank, 1), default=_json_default))
        return
    line, w, t = run_gpu(args, rank, world)
    default_line = (args.workload == "prefill8k" and args.tokens == 8192
                    and args.partials == "fp32" and not args.fp8qk)
    if default_line and not args.no_configs:
        line["configs"] = run_other_configs(args, world, w, t)
    if rank == 0:
        if not args.no_cpu_baseline and w is not None:
            line["cpu_baseline"] = cpu_baseline(w, t, budget_s=float(os.environ.get("SPS_CPU_S", "12")))
        print(json.dumps(line, default=_json_default))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
