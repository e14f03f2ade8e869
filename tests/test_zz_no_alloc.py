"""sparse_prefill_fwd_noalloc: the forward for callers that cannot allocate device memory
(their scratch lives in a fixed array inside the library).  Checked through the C ABI against
the workspace-based sparse_prefill_fwd on the same inputs: two calls in a row on one plan,
then plans of other sizes, top_k and dtypes through the same array (it keeps the previous
call's contents, so every call must clear and rebuild what it needs), and a call without a
status word.  This file is named to run after every other test file."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from paged_top_sparse_gb300 import synth

pytestmark = pytest.mark.gpu

PARTIAL_RL2 = 1e-3  # the tolerance the forward's parity tests use
LSE_ATOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_top_sparse_gb300 import build

    build.build()


def _rel_l2(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _workspace_reference(w):
    """The whole path with a workspace: the selection, and the forward's partials and LSEs."""
    from tests.gpu_helpers import DeviceRun

    run = DeviceRun(w, synth.make_tensors(w))
    run.indexer()
    run.topk()
    run.forward()
    torch.cuda.synchronize()
    assert run.status() == 0
    return run, run.partial.cpu().numpy(), run.lse.cpu().numpy()


def _noalloc_matches(run, ref_p, ref_l, status, label):
    from paged_top_sparse_gb300 import binding as B

    partial = torch.full_like(run.partial, float("nan"))
    lse = torch.full_like(run.lse, float("nan"))
    B.sparse_prefill_fwd_noalloc(run.plan, run.q, run.q_scale, run.k, run.v, run.k_scales,
                                 run.v_scales, run.page_table, run.idx, partial, lse,
                                 dev_status=status)
    torch.cuda.synchronize()
    if status is not None:
        assert int(status.item()) == 0, f"{label}: device status {int(status.item())}"
    filled = (run.idx.cpu().numpy() >= 0).T  # [slot][row]
    got_p = partial.cpu().numpy()
    got_l = lse.cpu().numpy()
    assert np.all(got_l[~filled] == -np.inf), label
    assert np.all(np.isnan(got_p[~filled])), label
    assert _rel_l2(got_p[filled], ref_p[filled]) <= PARTIAL_RL2, label
    assert np.max(np.abs(got_l[filled] - ref_l[filled])) <= LSE_ATOL, label
    # the same kernels on the same inputs: expect identical bits
    assert np.array_equal(got_p[filled].view(np.uint32), ref_p[filled].view(np.uint32)), label
    assert np.array_equal(got_l[filled].view(np.uint32), ref_l[filled].view(np.uint32)), label


def test_noalloc_forward_matches_workspace_forward_on_two_calls():
    w = synth.workload("custom", seed=21, q_lens=[300, 77, 129], ctx_lens=[0, 1000, 250],
                       num_q_heads=4, num_kv_heads=2, head_dim=128, top_k=5)
    run, ref_p, ref_l = _workspace_reference(w)
    status = torch.zeros(1, dtype=torch.int32, device=run.dev)
    for call in range(2):
        _noalloc_matches(run, ref_p, ref_l, status, f"call {call}")


def test_noalloc_after_larger_plan_other_top_k_quantised_and_without_status():
    """A large plan (2048 tokens x 32 heads, top-16) fills much of the array; then a small plan
    with top-3, an E4M3 / NVFP4 plan and a call with no status word run through the same array
    and must each equal the workspace forward bit for bit."""
    big = synth.workload("custom", seed=22, q_lens=[2048], ctx_lens=[900], num_q_heads=32,
                         num_kv_heads=2, head_dim=128, top_k=16)
    small = synth.workload("custom", seed=23, q_lens=[130, 61], ctx_lens=[0, 300], num_q_heads=4,
                           num_kv_heads=2, head_dim=64, top_k=3)
    quant = synth.workload("custom", seed=24, q_lens=[300, 77], ctx_lens=[0, 1000],
                           num_q_heads=4, num_kv_heads=2, head_dim=128, top_k=5,
                           q_dtype="e4m3", kv_dtype="nvfp4")
    refs = [(name, *_workspace_reference(w)) for name, w in
            (("big", big), ("small", small), ("quant", quant))]
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    for name, run, ref_p, ref_l in refs:
        _noalloc_matches(run, ref_p, ref_l, status, name)
    name, run, ref_p, ref_l = refs[1]
    _noalloc_matches(run, ref_p, ref_l, None, "small, no status word")


def test_noalloc_long_context():
    """16 tokens after 1,048,560 cached (8192 pages): the inversion runs its multi-kernel form
    in the array (one scan block per eight of the 8192 buckets), and the top-k's segment lists,
    which only topk_select uses, are not part of the array's need."""
    w = synth.workload("custom", seed=25, q_lens=[16], ctx_lens=[1048560], num_q_heads=2,
                       num_kv_heads=1, head_dim=64, top_k=16)
    run, ref_p, ref_l = _workspace_reference(w)
    status = torch.zeros(1, dtype=torch.int32, device=run.dev)
    _noalloc_matches(run, ref_p, ref_l, status, "1M-token context")


def test_noalloc_rejects_a_batch_larger_than_its_scratch():
    """4096 tokens x 32 heads x top-64 needs more scratch than the array holds: the call is
    refused before any launch.  Every buffer is real and of the size the arguments declare (the
    selection empty), so the call would stay in bounds whatever the order of its checks."""
    from paged_top_sparse_gb300 import binding as B

    T, H, G, D, K = 4096, 32, 2, 128, 64
    pages = T // 128
    plan = B.Plan([T], [0], H, G, D, K, pages, pages)
    assert plan.workspace_bytes > 48 << 20
    dev = "cuda:0"
    R = T * H
    q = torch.zeros((T, H, D), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((pages, G, 128, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    pt = torch.arange(pages, dtype=torch.int32, device=dev).view(1, pages)
    idx = torch.full((R, K), -1, dtype=torch.int32, device=dev)
    partial = torch.empty((K, R, D), dtype=torch.float32, device=dev)
    lse = torch.empty((K, R), dtype=torch.float32, device=dev)
    with pytest.raises(B.SpsError) as e:
        B.sparse_prefill_fwd_noalloc(plan, q, 1.0, kc, vc, None, None, pt, idx, partial, lse)
    assert e.value.status == 3  # SPS_ENOSPACE
    assert "scratch" in str(e.value)
    del partial
