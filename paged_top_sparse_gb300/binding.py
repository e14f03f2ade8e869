"""Thin ctypes binding of libsps (``include/sparse_prefill.h``).

Argument marshalling only: every function takes torch tensors (device memory supplied by
the caller), derives pointers, pitches and strides from them, calls the C entry point of the
same name and raises ``SpsError`` on a non-OK status.  No computation happens here, and
there is no fallback: if the library is missing, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

BF16, FP16, E4M3, NVFP4 = 0, 1, 2, 3
DTYPE_CODES = {"bf16": BF16, "fp16": FP16, "e4m3": E4M3, "nvfp4": NVFP4}
STATUS = {0: "SPS_OK", 1: "SPS_EINVAL", 2: "SPS_EUNSUPPORTED", 3: "SPS_ENOSPACE",
          4: "SPS_ECUDA", 5: "SPS_EDEVICE"}
HEADER = os.path.join(os.path.dirname(_build.HERE), "include", "sparse_prefill.h")


class SpsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("q_lens", ctypes.POINTER(ctypes.c_int32)),
        ("ctx_lens", ctypes.POINTER(ctypes.c_int32)),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("max_pages_per_req", ctypes.c_int32),
        ("num_phys_pages", ctypes.c_int32),
        ("q_dtype", ctypes.c_int),
        ("kv_dtype", ctypes.c_int),
        ("idx_q_dtype", ctypes.c_int),
        ("idx_k_dtype", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "num_tokens", "num_rows", "num_buckets", "max_entries", "indexer_tasks", "max_fwd_tasks",
        "workspace_bytes", "off_status", "off_tok_pos", "off_tok_req", "off_bucket_offsets",
        "off_entries", "off_fwd_task_count")]


_lib = None


def header_functions() -> list[str]:
    """Names of the functions declared in include/sparse_prefill.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, re.M))
                  - {"if", "while"})


def lib(path: str | None = None):
    """Load libsps.so (built in-tree by ``build.build()``, or the file named by $SPS_LIB);
    raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("SPS_LIB") or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libsps.so not built ({path}); run paged_top_sparse_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    L.sparse_prefill_plan.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(vp),
                                      ctypes.POINTER(ctypes.c_size_t)]
    L.sps_plan_destroy.argtypes = [vp]
    L.sps_plan_destroy.restype = None
    L.sps_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
    L.sps_plan_upload.argtypes = [vp, vp, ctypes.c_size_t, vp]
    L.indexer_scores.argtypes = [vp, vp, f32, vp, vp, f32, vp, vp, i64, vp, vp]
    L.topk_select.argtypes = [vp, vp, i64, vp, vp, vp]
    L.sparse_prefill_fwd.argtypes = [vp, vp, f32, vp, vp, vp, vp, vp, vp, vp, i64, vp, i64, vp, vp]
    L.partial_combine.argtypes = [i64, i32, i32, vp, i64, vp, i64, vp, i64, vp, vp, vp]
    L.sparse_prefill_fwd_bf16.argtypes = L.sparse_prefill_fwd.argtypes
    L.sparse_prefill_fwd_fp8qk.argtypes = L.sparse_prefill_fwd.argtypes
    L.sparse_prefill_fwd_f16.argtypes = L.sparse_prefill_fwd.argtypes
    L.sps_kv_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.sps_quantize_e4m3.argtypes = [vp, i64, f32, vp, vp]
    L.sps_absmax_bf16.argtypes = [vp, i64, vp, vp]
    L.partial_combine_bf16.argtypes = L.partial_combine.argtypes
    L.partial_combine_f16.argtypes = L.partial_combine.argtypes
    L.sparse_prefill_fwd_noalloc.argtypes = [vp, vp, f32, vp, vp, vp, vp, vp, vp, vp, i64, vp, i64,
                                             vp, vp]
    L.sps_read_device_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
    L.sps_dequantize.argtypes = [ctypes.c_int, vp, vp, i64, vp, vp]
    L.sps_check_wait_timeout.argtypes = [i64, vp, vp]
    L.sps_check_barrier_timeout.argtypes = [i64, vp, vp, vp]
    L.sps_last_error.restype = ctypes.c_char_p
    for name in ("sparse_prefill_plan", "sps_plan_get_info", "sps_plan_upload", "indexer_scores",
                 "topk_select", "sparse_prefill_fwd", "partial_combine", "sps_read_device_status",
                 "sparse_prefill_fwd_noalloc", "sps_dequantize", "sps_check_wait_timeout",
                 "sps_check_barrier_timeout"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(st: int):
    if st != 0:
        raise SpsError(st, lib().sps_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """Owns an sps_plan; ``workspace_bytes`` is the device workspace its calls need."""

    def __init__(self, q_lens, ctx_lens, num_q_heads, num_kv_heads, head_dim, top_k,
                 max_pages_per_req, num_phys_pages, q_dtype="bf16", kv_dtype="bf16",
                 idx_q_dtype=None, idx_k_dtype=None, softmax_scale=None, page_size=128):
        L = lib()
        n = len(q_lens)
        self._ql = (ctypes.c_int32 * n)(*[int(x) for x in q_lens])
        self._cl = (ctypes.c_int32 * n)(*[int(x) for x in ctx_lens])
        self.problem = Problem(
            n, self._ql, self._cl, num_q_heads, num_kv_heads, head_dim, page_size, top_k,
            max_pages_per_req, num_phys_pages, DTYPE_CODES[q_dtype], DTYPE_CODES[kv_dtype],
            DTYPE_CODES[idx_q_dtype or q_dtype], DTYPE_CODES[idx_k_dtype or kv_dtype],
            float(softmax_scale if softmax_scale is not None else head_dim ** -0.5))
        self.handle = ctypes.c_void_p()
        ws = ctypes.c_size_t()
        _check(L.sparse_prefill_plan(ctypes.byref(self.problem), ctypes.byref(self.handle),
                                     ctypes.byref(ws)))
        self.workspace_bytes = ws.value
        self.head_dim, self.top_k = head_dim, top_k

    def info(self) -> PlanInfo:
        inf = PlanInfo()
        _check(lib().sps_plan_get_info(self.handle, ctypes.byref(inf)))
        return inf

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.sps_plan_destroy(h)
            self.handle = None


def sparse_prefill_plan(*args, **kw) -> Plan:
    return Plan(*args, **kw)


def sps_plan_upload(plan: Plan, workspace, stream=None):
    _check(lib().sps_plan_upload(plan.handle, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))


def indexer_scores(plan: Plan, q_idx, q_scale, k_idx_cache, k_idx_scales, k_scale, page_table,
                   scores, workspace, stream=None):
    _check(lib().indexer_scores(plan.handle, _ptr(q_idx), float(q_scale), _ptr(k_idx_cache),
                                _ptr(k_idx_scales), float(k_scale), _ptr(page_table), _ptr(scores),
                                scores.stride(0), _ptr(workspace), _stream(stream)))


def topk_select(plan: Plan, scores, idx, workspace, stream=None):
    _check(lib().topk_select(plan.handle, _ptr(scores), scores.stride(0), _ptr(idx),
                             _ptr(workspace), _stream(stream)))


def sparse_prefill_fwd(plan: Plan, q, q_scale, k_cache, v_cache, k_scales, v_scales, page_table,
                       idx, partial, lse, workspace, stream=None):
    """``partial`` is a [splits][rows][D] view (its stride(0) is the split stride); ``lse`` is
    [splits][rows] (stride(0) is the LSE split stride)."""
    _check(lib().sparse_prefill_fwd(plan.handle, _ptr(q), float(q_scale), _ptr(k_cache),
                                    _ptr(v_cache), _ptr(k_scales), _ptr(v_scales), _ptr(page_table),
                                    _ptr(idx), _ptr(partial), partial.stride(0), _ptr(lse),
                                    lse.stride(0), _ptr(workspace), _stream(stream)))


def sparse_prefill_fwd_bf16(plan: Plan, q, q_scale, k_cache, v_cache, k_scales, v_scales,
                            page_table, idx, partial, lse, workspace, stream=None):
    """As ``sparse_prefill_fwd`` with ``partial`` a BF16 [splits][rows][D] view."""
    _check(lib().sparse_prefill_fwd_bf16(plan.handle, _ptr(q), float(q_scale), _ptr(k_cache),
                                         _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
                                         _ptr(page_table), _ptr(idx), _ptr(partial),
                                         partial.stride(0), _ptr(lse), lse.stride(0),
                                         _ptr(workspace), _stream(stream)))


def sparse_prefill_fwd_f16(plan: Plan, q, q_scale, k_cache, v_cache, k_scales, v_scales,
                           page_table, idx, partial, lse, workspace, stream=None):
    """As ``sparse_prefill_fwd`` with ``partial`` an FP16 [splits][rows][D] view."""
    _check(lib().sparse_prefill_fwd_f16(plan.handle, _ptr(q), float(q_scale), _ptr(k_cache),
                                        _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
                                        _ptr(page_table), _ptr(idx), _ptr(partial),
                                        partial.stride(0), _ptr(lse), lse.stride(0),
                                        _ptr(workspace), _stream(stream)))


def sparse_prefill_fwd_fp8qk(plan: Plan, q, q_scale, k_cache, v_cache, k_scales, v_scales,
                             page_table, idx, partial, lse, workspace, stream=None):
    """As ``sparse_prefill_fwd``: E4M3 Q, NVFP4 K rounded to E4M3, FP8 Q K^T (the pages' route)."""
    _check(lib().sparse_prefill_fwd_fp8qk(plan.handle, _ptr(q), float(q_scale), _ptr(k_cache),
                                          _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
                                          _ptr(page_table), _ptr(idx), _ptr(partial),
                                          partial.stride(0), _ptr(lse), lse.stride(0),
                                          _ptr(workspace), _stream(stream)))


def sparse_prefill_fwd_noalloc(plan: Plan, q, q_scale, k_cache, v_cache, k_scales, v_scales,
                               page_table, idx, partial, lse, dev_status=None, stream=None):
    """sparse_prefill_fwd without a workspace: the library's own fixed scratch array is used
    (for callers that cannot allocate device memory; see the header for the rules)."""
    _check(lib().sparse_prefill_fwd_noalloc(
        plan.handle, _ptr(q), float(q_scale), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales),
        _ptr(v_scales), _ptr(page_table), _ptr(idx), _ptr(partial), partial.stride(0), _ptr(lse),
        lse.stride(0), _ptr(dev_status), _stream(stream)))


def partial_combine(partial, lse, out, out_lse=None, dev_status=None, stream=None):
    """partial [splits][rows][D] FP32 (rows contiguous), lse [splits][rows], out [rows][D] BF16."""
    S, R, D = partial.shape
    _check(lib().partial_combine(R, S, D, _ptr(partial), partial.stride(0), _ptr(lse),
                                 lse.stride(0), _ptr(out), out.stride(0), _ptr(out_lse),
                                 _ptr(dev_status), _stream(stream)))


def partial_combine_bf16(partial, lse, out, out_lse=None, dev_status=None, stream=None):
    """As ``partial_combine`` with ``partial`` BF16 [splits][rows][D] (rows contiguous)."""
    S, R, D = partial.shape
    _check(lib().partial_combine_bf16(R, S, D, _ptr(partial), partial.stride(0), _ptr(lse),
                                      lse.stride(0), _ptr(out), out.stride(0), _ptr(out_lse),
                                      _ptr(dev_status), _stream(stream)))


def partial_combine_f16(partial, lse, out, out_lse=None, dev_status=None, stream=None):
    """As ``partial_combine`` with ``partial`` FP16 [splits][rows][D] (rows contiguous)."""
    S, R, D = partial.shape
    _check(lib().partial_combine_f16(R, S, D, _ptr(partial), partial.stride(0), _ptr(lse),
                                     lse.stride(0), _ptr(out), out.stride(0), _ptr(out_lse),
                                     _ptr(dev_status), _stream(stream)))


def sps_kv_append(plan: Plan, k_new, v_new, page_table, k_cache, v_cache, k_scales, v_scales,
                  workspace, stream=None):
    """New tokens' K/V [T][H_kv][D] BF16 into the paged cache (the plan's kv dtype)."""
    _check(lib().sps_kv_append(plan.handle, _ptr(k_new), _ptr(v_new), _ptr(page_table),
                               _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
                               _ptr(workspace), _stream(stream)))


def sps_quantize_e4m3(x_bf16, scale: float, codes, stream=None):
    """E4M3 codes of ``x_bf16`` (any shape, n % 16 == 0) with a per-tensor scale."""
    _check(lib().sps_quantize_e4m3(_ptr(x_bf16), x_bf16.numel(), float(scale), _ptr(codes),
                                   _stream(stream)))


def sps_absmax_bf16(x_bf16, out_f32, stream=None):
    """out_f32[0] = max |x| over ``x_bf16`` (device)."""
    _check(lib().sps_absmax_bf16(_ptr(x_bf16), x_bf16.numel(), _ptr(out_f32), _stream(stream)))


def sps_dequantize(in_dtype: str, data, scales, n: int, out_f16, stream=None):
    """Exact E4M3 / NVFP4 -> FP16 of n elements into ``out_f16`` (see the header)."""
    _check(lib().sps_dequantize(DTYPE_CODES[in_dtype], _ptr(data), _ptr(scales), int(n),
                                _ptr(out_f16), _stream(stream)))


def sps_check_wait_timeout(limit_ns: int, dev_status, stream=None):
    """Launch the bounded-wait self-check; *dev_status becomes SPS_DEV_TIMEOUT (1)."""
    _check(lib().sps_check_wait_timeout(int(limit_ns), _ptr(dev_status), _stream(stream)))


def sps_check_barrier_timeout(limit_ns: int, dev_barrier, dev_status, stream=None):
    """Grid-barrier timeout self-check: dev_barrier is a zeroed device int32 tensor of 2."""
    _check(lib().sps_check_barrier_timeout(int(limit_ns), _ptr(dev_barrier), _ptr(dev_status),
                                           _stream(stream)))


def sps_read_device_status(plan: Plan, workspace) -> int:
    code = ctypes.c_int32()
    st = lib().sps_read_device_status(plan.handle, _ptr(workspace), ctypes.byref(code))
    if st not in (0, 5):
        _check(st)
    return code.value
