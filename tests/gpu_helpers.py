"""Device-side helpers for the GPU tests: put a synthetic workload on the GPU and run the
four C-ABI calls through the binding."""
from __future__ import annotations

import numpy as np
import torch

from paged_top_sparse_gb300 import binding as B


def _dev(a, dev):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev)


class DeviceRun:
    """Inputs of a workload on ``dev`` plus the plan and its uploaded workspace."""

    def __init__(self, w, t, dev="cuda:0", pitch=None):
        self.w, self.t, self.dev = w, t, dev
        self.q = _dev(t["q"], dev)
        self.k = _dev(t["k"], dev)
        self.v = _dev(t["v"], dev)
        self.k_scales = _dev(t.get("k_scales"), dev)
        self.v_scales = _dev(t.get("v_scales"), dev)
        self.q_scale = float(t.get("q_scale", 1.0))
        if w.idx_dtype == "e4m3":
            self.qi, self.ki = _dev(t["q_idx"], dev), _dev(t["k_idx"], dev)
            self.qi_scale, self.ki_scale = float(t["q_idx_scale"]), float(t["k_idx_scale"])
            self.ki_scales = None
            idx_q, idx_k = "e4m3", "e4m3"
        else:
            self.qi, self.ki, self.ki_scales = self.q, self.k, self.k_scales
            self.qi_scale, self.ki_scale = self.q_scale, 1.0
            idx_q, idx_k = w.q_dtype, w.kv_dtype
        self.page_table = _dev(w.page_table.astype(np.int32), dev)
        self.plan = B.Plan(w.q_lens, w.ctx_lens, w.num_q_heads, w.num_kv_heads, w.head_dim,
                           w.top_k, w.max_pages, w.num_phys_pages, q_dtype=w.q_dtype,
                           kv_dtype=w.kv_dtype, idx_q_dtype=idx_q, idx_k_dtype=idx_k,
                           softmax_scale=w.sm_scale)
        self.ws = torch.zeros(self.plan.workspace_bytes, dtype=torch.uint8, device=dev)
        B.sps_plan_upload(self.plan, self.ws)
        R, K, D = w.num_rows, w.top_k, w.head_dim
        self.pitch = pitch or (w.max_pages + 3) // 4 * 4  # 16-byte rows, as the header asks
        self.scores = torch.full((R, self.pitch), float("nan"), dtype=torch.float32, device=dev)
        self.idx = torch.full((R, K), -7, dtype=torch.int32, device=dev)
        self.partial = torch.full((K, R, D), float("nan"), dtype=torch.float32, device=dev)
        self.lse = torch.full((K, R), float("nan"), dtype=torch.float32, device=dev)
        self.out = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
        self.out_lse = torch.empty((R,), dtype=torch.float32, device=dev)

    def indexer(self):
        B.indexer_scores(self.plan, self.qi, self.qi_scale, self.ki, self.ki_scales,
                         self.ki_scale, self.page_table, self.scores, self.ws)

    def topk(self, scores=None):
        B.topk_select(self.plan, self.scores if scores is None else scores, self.idx, self.ws)

    def forward(self, idx=None):
        B.sparse_prefill_fwd(self.plan, self.q, self.q_scale, self.k, self.v, self.k_scales,
                             self.v_scales, self.page_table, self.idx if idx is None else idx,
                             self.partial, self.lse, self.ws)

    def combine(self):
        B.partial_combine(self.partial, self.lse, self.out, self.out_lse)

    def run_all(self):
        self.indexer()
        self.topk()
        self.forward()
        self.combine()
        torch.cuda.synchronize()

    def status(self) -> int:
        return B.sps_read_device_status(self.plan, self.ws)

    def ws_array(self, off, count, dtype):
        nbytes = count * np.dtype(dtype).itemsize
        return self.ws[off:off + nbytes].cpu().numpy().view(dtype)
