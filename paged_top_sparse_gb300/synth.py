"""Seeded synthetic inputs for paged block-sparse prefill attention.

This module only *makes inputs*: shapes, seeded random values, page tables and the
quantisation that turns N(0,1) samples into stored E4M3 / NVFP4 codes.  It holds none of the
method's arithmetic (no decode, no dot products, no softmax), so both the CUDA path and the
CPU oracle can consume what it produces without sharing code with each other.

Workloads (shapes of the pages' prefill and chunked-prefill traffic):

* ``tiny``        1 x 1024 tokens, 2 query heads on 1 KV head, D=64, top-4, BF16, identity pages.
* ``prefill8k``   1 x 8192 tokens, 32 query / 2 KV heads, D=128, top-16, BF16, permuted pages.
* ``prefill8k_q`` same shape; Q in E4M3 (per-tensor scale), K/V in NVFP4 (E2M1 code x E4M3
  scale per 16 elements along D).
* ``combine16k``  a [16][16384*32][128] FP32 partial buffer with LSE ~ N(0, sd 2).
* ``chunked32k``  8 requests x 512 new tokens over ~32K cached tokens (jitter +-25 %), E4M3
  indexer q/k with per-tensor scales, BF16 K/V, one shared permuted physical page pool.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

PAGE = 128

E4M3_MAX = 448.0
# the eight non-negative E2M1 magnitudes, indexed by the 3-bit code (exponent:mantissa)
_E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@dataclass
class Workload:
    name: str
    q_lens: np.ndarray
    ctx_lens: np.ndarray
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    top_k: int
    page_table: np.ndarray  # [batch][max_pages] int32, -1 beyond the request's pages
    num_phys_pages: int
    q_dtype: str = "bf16"
    kv_dtype: str = "bf16"
    idx_dtype: str = "same"  # "same" (indexer reads Q/K) or "e4m3" (separate E4M3 copies)
    seed: int = 0
    page_size: int = PAGE

    @property
    def batch(self):
        return len(self.q_lens)

    @property
    def num_tokens(self):
        return int(np.sum(self.q_lens))

    @property
    def num_rows(self):
        return self.num_tokens * self.num_q_heads

    @property
    def max_pages(self):
        return int(self.page_table.shape[1])

    @property
    def sm_scale(self):
        return 1.0 / float(np.sqrt(self.head_dim))


# ------------------------------------------------------------------ fixture encoders

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to BF16 (nearest, ties to even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round to OCP E4M3 (nearest even) with saturation to +-448; returns uint8 codes."""
    import torch

    t = torch.from_numpy(np.clip(np.asarray(x, np.float32), -E4M3_MAX, E4M3_MAX))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e2m1_code(y: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code (ties to the even mantissa), saturating at +-6."""
    a = np.minimum(np.abs(y), 6.0)
    # decision thresholds between neighbouring magnitudes; at a tie the code with mantissa 0
    # wins, which is the even one: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    up = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    tie_goes_up = np.array([False, True, False, True, False, True, False])
    code = np.zeros(a.shape, np.uint8)
    for i, (t, tu) in enumerate(zip(up, tie_goes_up)):
        code = np.where((a > t) | ((a == t) & tu), i + 1, code).astype(np.uint8)
    sign = (np.signbit(y) & (code > 0)).astype(np.uint8) << 3
    return code | sign


def quantize_nvfp4(x: np.ndarray):
    """x [..., D] float32 -> (packed codes [..., D/2] uint8, scales [..., D/16] uint8 E4M3).

    Per 16 consecutive elements: scale = E4M3(absmax / 6), code = E2M1(x / scale); no global
    scale.  Two codes per byte, the even element in the low nibble."""
    import torch

    x = np.asarray(x, np.float32)
    D = x.shape[-1]
    assert D % 16 == 0
    blocks = x.reshape(*x.shape[:-1], D // 16, 16)
    amax = np.abs(blocks).max(axis=-1)
    sc_bits = f32_to_e4m3_bits(amax / 6.0)
    sc = torch.from_numpy(sc_bits).view(torch.float8_e4m3fn).float().numpy()
    safe = np.where(sc > 0, sc, 1.0)[..., None]
    codes = _e2m1_code(np.where(sc[..., None] > 0, blocks / safe, 0.0)).reshape(x.shape)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, sc_bits


def quantize_e4m3_per_tensor(x: np.ndarray):
    """x float32 -> (codes uint8, scale) with scale = absmax / 448."""
    amax = float(np.abs(x).max())
    s = amax / E4M3_MAX if amax > 0 else 1.0
    return f32_to_e4m3_bits(np.asarray(x, np.float32) / np.float32(s)), s


# ------------------------------------------------------------------ workloads

def _pages_needed(ctx, qlen, page=PAGE):
    return (ctx + qlen - 1) // page + 1 if qlen > 0 else 0


def _make_page_table(rng, q_lens, ctx_lens, permute: bool, page=PAGE):
    npages = [_pages_needed(int(c), int(q), page) for q, c in zip(q_lens, ctx_lens)]
    total = int(sum(npages))
    pool = rng.permutation(total).astype(np.int32) if permute else np.arange(total, dtype=np.int32)
    maxp = max(npages) if npages else 1
    pt = np.full((len(q_lens), maxp), -1, np.int32)
    off = 0
    for b, n in enumerate(npages):
        pt[b, :n] = pool[off:off + n]
        off += n
    return pt, total


def workload(name: str, seed: int = 0, **over) -> Workload:
    """Shape, page table and dtypes of a named workload (values come from ``make_tensors``)."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        q_lens, ctx = np.array([1024]), np.array([0])
        H, Hkv, D, k, permute = 2, 1, 64, 4, False
    elif name in ("prefill8k", "prefill8k_q"):
        q_lens, ctx = np.array([8192]), np.array([0])
        H, Hkv, D, k, permute = 32, 2, 128, 16, True
    elif name == "chunked32k":
        ctx = np.round(32768 * rng.uniform(0.75, 1.25, size=8)).astype(np.int64)
        q_lens = np.full(8, 512)
        H, Hkv, D, k, permute = 32, 2, 128, 16, True
    elif name == "ctx1m":  # a 512-token chunk at the end of a 1M-token context (8192 pages)
        q_lens, ctx = np.array([512]), np.array([1048576 - 512])
        H, Hkv, D, k, permute = 32, 2, 128, 16, True
    elif name == "custom":
        q_lens, ctx = np.asarray(over.pop("q_lens")), np.asarray(over.pop("ctx_lens"))
        H, Hkv = over.pop("num_q_heads"), over.pop("num_kv_heads")
        D, k = over.pop("head_dim"), over.pop("top_k")
        permute = over.pop("permute", True)
    else:
        raise ValueError(name)
    pt, nphys = _make_page_table(rng, q_lens, ctx, permute)
    w = Workload(name, np.asarray(q_lens, np.int32), np.asarray(ctx, np.int32), H, Hkv, D, k,
                 pt, nphys, seed=seed)
    if name == "prefill8k_q":
        w.q_dtype, w.kv_dtype = "e4m3", "nvfp4"
    if name == "chunked32k":
        w.idx_dtype = "e4m3"
    for kk, vv in over.items():
        setattr(w, kk, vv)
    return w


def make_tensors(w: Workload) -> dict:
    """Seeded values for a workload, as stored bits on the host.

    Q [T][H][D]; K/V caches [num_phys_pages][H_kv][128][D] (NVFP4: codes [..][D/2] and
    scales [..][D/16]).  Keys of pages that no request owns stay zero."""
    rng = np.random.default_rng(1_000_003 * (w.seed + 1))
    T, H, Hkv, D = w.num_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim
    q32 = rng.standard_normal((T, H, D), dtype=np.float32)
    k32 = rng.standard_normal((w.num_phys_pages, Hkv, w.page_size, D), dtype=np.float32)
    v32 = rng.standard_normal((w.num_phys_pages, Hkv, w.page_size, D), dtype=np.float32)
    out = {}
    if w.q_dtype == "bf16":
        out["q"], out["q_scale"] = f32_to_bf16_bits(q32), 1.0
    else:
        out["q"], out["q_scale"] = quantize_e4m3_per_tensor(q32)
    if w.kv_dtype == "bf16":
        out["k"], out["v"] = f32_to_bf16_bits(k32), f32_to_bf16_bits(v32)
        out["k_scales"] = out["v_scales"] = None
    else:
        out["k"], out["k_scales"] = quantize_nvfp4(k32)
        out["v"], out["v_scales"] = quantize_nvfp4(v32)
    if w.idx_dtype == "e4m3":
        out["q_idx"], out["q_idx_scale"] = quantize_e4m3_per_tensor(q32)
        out["k_idx"], out["k_idx_scale"] = quantize_e4m3_per_tensor(k32)
    return out


def combine_inputs(rows: int, splits: int, head_dim: int, seed: int = 0, device=None):
    """FP32 partials [splits][rows][D] ~ N(0,1) and LSEs [splits][rows] ~ N(0, sd 2).

    Generated with torch's seeded generator on ``device`` (large buffers are made where they
    are used)."""
    import torch

    dev = torch.device(device or "cpu")
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    part = torch.randn((splits, rows, head_dim), generator=g, device=dev, dtype=torch.float32)
    lse = 2.0 * torch.randn((splits, rows), generator=g, device=dev, dtype=torch.float32)
    return part, lse
