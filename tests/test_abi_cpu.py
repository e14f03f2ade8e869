"""C-ABI checks that need no GPU: the library builds and loads, exports every function that
include/sparse_prefill.h declares, and the host-only planning / validation behaves."""
import numpy as np
import pytest

from paged_top_sparse_gb300 import binding as B
from paged_top_sparse_gb300 import build


@pytest.fixture(scope="module")
def L():
    build.build()
    return B.lib()


def test_every_header_function_is_exported(L):
    names = B.header_functions()
    assert {"sparse_prefill_plan", "indexer_scores", "topk_select", "sparse_prefill_fwd",
            "partial_combine", "sps_read_device_status", "sps_last_error"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def _plan(**kw):
    args = dict(q_lens=[8192], ctx_lens=[0], num_q_heads=32, num_kv_heads=2, head_dim=128,
                top_k=16, max_pages_per_req=64, num_phys_pages=64)
    args.update(kw)
    return B.Plan(**args)


def test_plan_sizes(L):
    p = _plan()
    info = p.info()
    assert info.num_tokens == 8192 and info.num_rows == 8192 * 32
    assert info.num_buckets == 64 * 2
    assert info.max_entries == 8192 * 32 * 16
    assert info.workspace_bytes == p.workspace_bytes and p.workspace_bytes % 256 == 0
    assert info.indexer_tasks >= 4 * 152 or info.indexer_tasks > 0
    # offsets are ordered, aligned and inside the workspace
    offs = [info.off_status, info.off_tok_pos, info.off_tok_req, info.off_bucket_offsets,
            info.off_entries]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert info.off_entries + 8 * info.max_entries <= p.workspace_bytes


def test_chunked_plan_counts_pages_per_request(L):
    ctx = [1000, 0, 255]
    ql = [300, 128, 1]
    p = _plan(q_lens=ql, ctx_lens=ctx, max_pages_per_req=16, num_phys_pages=40, head_dim=64)
    pages = [(c + q - 1) // 128 + 1 for c, q in zip(ctx, ql)]
    assert p.info().num_buckets == sum(pages) * 2


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 2),
    (dict(num_kv_heads=3), 1),
    (dict(top_k=0), 1),
    (dict(top_k=65), 1),
    (dict(max_pages_per_req=63), 1),
    (dict(page_size=64), 2),
    (dict(q_lens=[0], ctx_lens=[0]), 1),
    (dict(q_lens=[5], ctx_lens=[-1]), 1),
    (dict(softmax_scale=float("nan")), 1),
    (dict(q_dtype="e4m3", kv_dtype="bf16"), 2),
    (dict(idx_q_dtype="bf16", idx_k_dtype="e4m3"), 2),
])
def test_plan_rejects_invalid_problems(L, kw, status):
    with pytest.raises(B.SpsError) as e:
        _plan(**kw)
    assert e.value.status == status
    assert L.sps_last_error().decode()


def test_combine_validation_needs_no_device(L):
    import ctypes
    # rows = 0 is a no-op; bad splits / head_dim rejected before any CUDA call
    assert L.partial_combine(0, 16, 128, None, 0, None, 0, None, 128, None, None, None) == 0
    assert L.partial_combine(10, 0, 128, None, 0, None, 0, None, 128, None, None, None) == 1
    assert L.partial_combine(10, 4, 96, None, 0, None, 0, None, 128, None, None, None) == 2
    # a split stride below rows * head_dim: real buffers large enough for every element the
    # declared strides reach, so the call stays in bounds whatever the order of the checks
    rows, splits, d, stride = 10, 4, 128, 100
    part = np.zeros((splits - 1) * stride + rows * d, dtype=np.float32)
    lse = np.zeros(splits * rows, dtype=np.float32)
    out = np.zeros(rows * d, dtype=np.uint16)
    ptr = lambda a: ctypes.c_void_p(a.ctypes.data)
    assert L.partial_combine(rows, splits, d, ptr(part), stride, ptr(lse), rows, ptr(out), d,
                             None, None, None) == 1
    assert b"split_stride" in L.sps_last_error()


def test_plan_page_limits(L):
    """With top_k <= 16 a request may see up to 8192 pages (1M tokens of context: the
    inversion packs a page into 16 bits); with top_k > 16 up to 1024 (128K tokens: the
    warp-per-row top-k holds at most 32 pages per lane).  A plan beyond its limit is refused
    with a message naming it."""
    _plan(q_lens=[16], ctx_lens=[1048560], max_pages_per_req=8192, num_phys_pages=8192,
          num_q_heads=2, num_kv_heads=1, head_dim=64)
    with pytest.raises(B.SpsError) as e:
        _plan(q_lens=[16], ctx_lens=[1048570], max_pages_per_req=8193, num_phys_pages=8193,
              num_q_heads=2, num_kv_heads=1, head_dim=64)
    assert e.value.status == 2
    assert "8192" in str(e.value)
    _plan(q_lens=[200], ctx_lens=[130800], max_pages_per_req=1024, num_phys_pages=1024, top_k=17)
    with pytest.raises(B.SpsError) as e:
        _plan(q_lens=[200], ctx_lens=[130900], max_pages_per_req=1025, num_phys_pages=1025,
              top_k=17)
    assert e.value.status == 2
    assert "1024" in str(e.value) and "top_k 17" in str(e.value)
    # a 1025-page request with top_k <= 16 is a valid plan
    _plan(q_lens=[200], ctx_lens=[130900], max_pages_per_req=1025, num_phys_pages=1025)
