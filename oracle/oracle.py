"""ctypes front end of the FP64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's CPU
baseline may use this module; the product path never does.  It imports nothing from the
CUDA package.  Each function names the definition it follows; the arithmetic lives in
``oracle.c`` and is commented there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")

DTYPES = {"bf16": 0, "fp16": 1, "e4m3": 2, "nvfp4": 3, "fp32": 4, "nvfp4_e4m3": 5}


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (-O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _SO)
    return _SO


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("q_lens", ctypes.c_void_p),
        ("ctx_lens", ctypes.c_void_p),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("num_phys_pages", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
    ]


class _Tensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("scale", ctypes.c_double),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P, T = ctypes.POINTER(_Problem), _Tensor
        vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        _lib.orc_decode_bf16.restype = dbl
        _lib.orc_decode_fp16.restype = dbl
        _lib.orc_decode_e4m3.restype = dbl
        _lib.orc_decode_e2m1.restype = dbl
        _lib.orc_decode_bf16.argtypes = [ctypes.c_uint16]
        _lib.orc_decode_fp16.argtypes = [ctypes.c_uint16]
        _lib.orc_decode_e4m3.argtypes = [ctypes.c_uint8]
        _lib.orc_decode_e2m1.argtypes = [ctypes.c_uint8]
        _lib.orc_decode.argtypes = [T, i64, i64, vp]
        _lib.orc_token_meta.argtypes = [P, vp, vp]
        _lib.orc_token_meta.restype = i64
        _lib.orc_indexer.argtypes = [P, T, T, vp, i64, vp, i64]
        _lib.orc_topk.argtypes = [P, vp, i64, vp, i64, vp]
        _lib.orc_inversion.argtypes = [P, vp, vp, vp, vp]
        _lib.orc_inversion.restype = i64
        _lib.orc_forward.argtypes = [P, T, T, T, dbl, vp, vp, i64, vp, vp]
        _lib.orc_combine.argtypes = [i64, i32, i32, vp, i64, i64, vp, i64, vp, vp]
        _lib.orc_dense.argtypes = [P, T, T, T, dbl, vp, vp, i64, vp, vp]
        _lib.orc_num_threads.restype = ctypes.c_int
        _lib.orc_round_e4m3_n.argtypes = [vp, i64, vp]
        _lib.orc_round_e2m1_n.argtypes = [vp, i64, vp]
        _lib.orc_quantize_nvfp4_block.argtypes = [vp, vp, vp]
        _lib.orc_quantize_e4m3.argtypes = [vp, i64, ctypes.c_float, vp]
        _lib.orc_kv_append.argtypes = [P, i32, vp, vp, vp]
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Tensor:
    """Raw element bits plus how to decode them.

    ``data``: uint16 (bf16/fp16), uint8 (e4m3), packed uint8 codes (nvfp4, even element in
    the low nibble) or float32.  ``scales``: uint8 E4M3, one per 16 elements (nvfp4 only).
    ``nvfp4_e4m3``: NVFP4 whose code x scale products are rounded to E4M3 (the pages' QMUL4).
    ``scale``: per-tensor multiplier applied after decoding.
    """

    data: np.ndarray
    dtype: str
    scales: np.ndarray | None = None
    scale: float = 1.0

    def c(self):
        d = np.ascontiguousarray(self.data)
        s = None if self.scales is None else np.ascontiguousarray(self.scales)
        self._keep = (d, s)
        return _Tensor(_ptr(d), _ptr(s), DTYPES[self.dtype], float(self.scale))


@dataclass
class Problem:
    """Shapes and the page table of one batch (``[batch][max_pages]`` int32)."""

    q_lens: np.ndarray
    ctx_lens: np.ndarray
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    top_k: int
    page_table: np.ndarray
    num_phys_pages: int
    page_size: int = 128
    _keep: tuple = field(default=(), repr=False)

    @property
    def batch(self):
        return len(self.q_lens)

    @property
    def max_pages(self):
        return int(self.page_table.shape[1])

    @property
    def num_tokens(self):
        return int(np.sum(self.q_lens))

    @property
    def num_rows(self):
        return self.num_tokens * self.num_q_heads

    def c(self):
        ql = np.ascontiguousarray(self.q_lens, dtype=np.int32)
        cl = np.ascontiguousarray(self.ctx_lens, dtype=np.int32)
        pt = np.ascontiguousarray(self.page_table, dtype=np.int32)
        self._keep = (ql, cl, pt)
        return _Problem(
            len(ql), _ptr(ql), _ptr(cl), self.num_q_heads, self.num_kv_heads, self.head_dim,
            self.page_size, self.top_k, pt.shape[1], self.num_phys_pages, _ptr(pt),
        )


def _rows(pb: Problem, rows):
    if rows is None:
        rows = np.arange(pb.num_rows, dtype=np.int64)
    return np.ascontiguousarray(rows, dtype=np.int64)


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """binary32 -> E4M3 codes: nearest, ties to the even code, saturating at +-448."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_round_e4m3_n(_ptr(x), x.size, _ptr(out))
    return out


def round_e2m1(x: np.ndarray) -> np.ndarray:
    """binary32 -> E2M1 nibbles: nearest, ties to the even code, saturating at +-6."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_round_e2m1_n(_ptr(x), x.size, _ptr(out))
    return out


def quantize_nvfp4(x_bf16: np.ndarray):
    """BF16 bits [..., 16 m] -> (codes [..., 8 m] uint8, scales [..., m] uint8), block by
    block: scale = E4M3(absmax / 6), code = E2M1(x / scale)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    n = x.size // 16
    codes = np.empty(n * 8, np.uint8)
    scales = np.empty(n, np.uint8)
    flat = x.reshape(-1)
    L = lib()
    for b in range(n):
        blk = flat[16 * b: 16 * b + 16]
        L.orc_quantize_nvfp4_block(_ptr(blk), _ptr(codes[8 * b:]), _ptr(scales[b:]))
    return codes.reshape(x.shape[:-1] + (x.shape[-1] // 2,)), scales.reshape(x.shape[:-1] + (x.shape[-1] // 16,))


def quantize_e4m3(x_bf16: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes of BF16 values with a per-tensor scale: E4M3(x / scale) in binary32."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    out = np.empty(x.shape, np.uint8)
    lib().orc_quantize_e4m3(_ptr(x), x.size, ctypes.c_float(scale), _ptr(out))
    return out


def kv_append(pb: Problem, kv_dtype: str, new_bf16: np.ndarray, cache: np.ndarray,
              scales: np.ndarray | None = None):
    """Writes the batch's new tokens ``new_bf16`` [T][H_kv][D] (BF16 bits) into ``cache`` in
    place: BF16 bits [phys][H_kv][P][D], or NVFP4 codes [phys][H_kv][P][D/2] with ``scales``
    [phys][H_kv][P][D/16]."""
    x = np.ascontiguousarray(new_bf16, dtype=np.uint16)
    assert cache.flags.c_contiguous and (scales is None or scales.flags.c_contiguous)
    lib().orc_kv_append(ctypes.byref(pb.c()), DTYPES[kv_dtype], _ptr(x), _ptr(cache), _ptr(scales))


def num_threads() -> int:
    return lib().orc_num_threads()


def decode(t: Tensor, first: int = 0, n: int | None = None) -> np.ndarray:
    """Decoded values (times the per-tensor scale) of n elements starting at ``first``."""
    if n is None:
        n = t.data.size * (2 if t.dtype.startswith("nvfp4") else 1) - first
    out = np.empty(n, dtype=np.float64)
    lib().orc_decode(t.c(), first, n, _ptr(out))
    return out


def token_meta(pb: Problem):
    """(request, absolute position) of every flat token."""
    T = pb.num_tokens
    req = np.empty(T, np.int32)
    pos = np.empty(T, np.int32)
    lib().orc_token_meta(ctypes.byref(pb.c()), _ptr(req), _ptr(pos))
    return req, pos


def indexer(pb: Problem, q: Tensor, k: Tensor, rows=None) -> np.ndarray:
    """Page scores S[row][p] = max_{visible j in page p} q.k_j (FP64); NaN where p > o."""
    rows = _rows(pb, rows)
    out = np.full((len(rows), pb.max_pages), np.nan, dtype=np.float64)
    lib().orc_indexer(ctypes.byref(pb.c()), q.c(), k.c(), _ptr(rows), len(rows), _ptr(out),
                      pb.max_pages)
    return out


def topk(pb: Problem, scores: np.ndarray, rows=None) -> np.ndarray:
    """Per-row page selection from ``scores`` ([nrows][>= o+1], any float dtype, converted
    exactly to FP64): own page forced, best others by (score desc, page asc), ascending."""
    rows = _rows(pb, rows)
    s = np.ascontiguousarray(scores, dtype=np.float64)
    assert s.shape[0] == len(rows)
    idx = np.empty((len(rows), pb.top_k), np.int32)
    lib().orc_topk(ctypes.byref(pb.c()), _ptr(s), s.shape[1], _ptr(rows), len(rows), _ptr(idx))
    return idx


def inversion(pb: Problem, idx_all: np.ndarray):
    """(offsets [nbuckets+1], entry_row, entry_slot) of the page -> (row, slot) inversion."""
    idx = np.ascontiguousarray(idx_all, dtype=np.int32)
    assert idx.shape == (pb.num_rows, pb.top_k)
    n_entries = int(np.count_nonzero(idx >= 0))
    last = np.asarray(pb.ctx_lens, np.int64) + np.asarray(pb.q_lens, np.int64) - 1
    npages = np.where(np.asarray(pb.q_lens) > 0, last // pb.page_size + 1, 0)
    nb = int(npages.sum()) * pb.num_kv_heads
    offsets = np.empty(nb + 1, np.int64)
    er = np.empty(max(n_entries, 1), np.int32)
    es = np.empty(max(n_entries, 1), np.int32)
    got = lib().orc_inversion(ctypes.byref(pb.c()), _ptr(idx), _ptr(offsets), _ptr(er), _ptr(es))
    assert got == nb
    return offsets, er[:n_entries], es[:n_entries]


def forward(pb: Problem, q: Tensor, k: Tensor, v: Tensor, sm_scale: float, idx: np.ndarray,
            rows=None):
    """Per (row, slot) page softmax: partial [nrows][k][D] (FP64) and lse [nrows][k]."""
    rows = _rows(pb, rows)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    assert idx.shape == (len(rows), pb.top_k)
    part = np.empty((len(rows), pb.top_k, pb.head_dim), np.float64)
    lse = np.empty((len(rows), pb.top_k), np.float64)
    lib().orc_forward(ctypes.byref(pb.c()), q.c(), k.c(), v.c(), float(sm_scale), _ptr(idx),
                      _ptr(rows), len(rows), _ptr(part), _ptr(lse))
    return part, lse


def combine(partial: np.ndarray, lse: np.ndarray):
    """LSE merge.  ``partial`` [splits][rows][D] and ``lse`` [splits][rows] (any float dtype,
    converted exactly to FP64).  Returns out [rows][D] and out_lse [rows] in FP64."""
    p = np.ascontiguousarray(partial, dtype=np.float64)
    l = np.ascontiguousarray(lse, dtype=np.float64)
    S, R, D = p.shape
    out = np.empty((R, D), np.float64)
    olse = np.empty(R, np.float64)
    lib().orc_combine(R, S, D, _ptr(p), R * D, D, _ptr(l), R, _ptr(out), _ptr(olse))
    return out, olse


def dense(pb: Problem, q: Tensor, k: Tensor, v: Tensor, sm_scale: float, idx: np.ndarray,
          rows=None):
    """Direct definition: one softmax over the union of the selected pages' visible keys."""
    rows = _rows(pb, rows)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    out = np.empty((len(rows), pb.head_dim), np.float64)
    olse = np.empty(len(rows), np.float64)
    lib().orc_dense(ctypes.byref(pb.c()), q.c(), k.c(), v.c(), float(sm_scale), _ptr(idx),
                    _ptr(rows), len(rows), _ptr(out), _ptr(olse))
    return out, olse


def pipeline(pb: Problem, q: Tensor, k: Tensor, v: Tensor, sm_scale: float, qi: Tensor = None,
             ki: Tensor = None, rows=None):
    """The four steps on the oracle alone (indexer -> top-k -> forward -> combine) for a row
    subset; ``qi``/``ki`` are the indexer's inputs (default: the attention Q/K)."""
    rows = _rows(pb, rows)
    s = indexer(pb, qi or q, ki or k, rows)
    idx = topk(pb, np.nan_to_num(s, nan=-np.inf), rows)
    part, lse = forward(pb, q, k, v, sm_scale, idx, rows)
    out, olse = combine(part.transpose(1, 0, 2), lse.T)
    return dict(scores=s, idx=idx, partial=part, lse=lse, out=out, out_lse=olse)
