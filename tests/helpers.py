"""Test helpers: turn a synthetic workload into oracle inputs, and compare results."""
from __future__ import annotations

import numpy as np

from oracle import oracle as orc


def oracle_problem(w) -> orc.Problem:
    return orc.Problem(
        q_lens=np.asarray(w.q_lens, np.int32), ctx_lens=np.asarray(w.ctx_lens, np.int32),
        num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
        top_k=w.top_k, page_table=np.asarray(w.page_table, np.int32),
        num_phys_pages=w.num_phys_pages, page_size=w.page_size)


def oracle_tensors(w, t: dict):
    """(q, k, v, q_indexer, k_indexer) as oracle.Tensor objects."""
    q = orc.Tensor(t["q"], w.q_dtype, scale=t.get("q_scale", 1.0))
    k = orc.Tensor(t["k"], w.kv_dtype, scales=t.get("k_scales"))
    v = orc.Tensor(t["v"], w.kv_dtype, scales=t.get("v_scales"))
    if w.idx_dtype == "e4m3":
        qi = orc.Tensor(t["q_idx"], "e4m3", scale=t["q_idx_scale"])
        ki = orc.Tensor(t["k_idx"], "e4m3", scale=t["k_idx_scale"])
    else:
        qi, ki = q, k
    return q, k, v, qi, ki


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def sample_rows(w, n: int, seed: int = 123) -> np.ndarray:
    """Deterministic sample of rows that always includes the first and last rows of each
    request and rows at page boundaries, plus random others."""
    rng = np.random.default_rng(seed)
    H = w.num_q_heads
    picks = set()
    tok0 = 0
    for b in range(w.batch):
        ql, ctx = int(w.q_lens[b]), int(w.ctx_lens[b])
        for i in (0, 1, ql - 1, ql // 2):
            if 0 <= i < ql:
                picks.add((tok0 + i) * H + (i % H))
        # first query token whose position starts a page, and the one before it
        first_boundary = (-ctx) % w.page_size
        for i in (first_boundary - 1, first_boundary):
            if 0 <= i < ql:
                picks.add((tok0 + i) * H + ((i + 1) % H))
        tok0 += ql
    R = w.num_rows
    extra = rng.choice(R, size=min(n, R), replace=False)
    picks.update(int(x) for x in extra)
    return np.array(sorted(picks), dtype=np.int64)
