"""sparse_prefill_fwd_noalloc: the forward for callers that cannot allocate device memory
(their scratch lives in a fixed array inside the library).  Checked through the C ABI against
the workspace-based sparse_prefill_fwd on the same inputs, on two calls in a row (the array
keeps the previous call's contents, so the second call must clear what it needs).  This file
is named to run after every other test file."""
import ctypes

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


def test_noalloc_forward_matches_workspace_forward_on_two_calls():
    from paged_top_sparse_gb300 import binding as B
    from tests.gpu_helpers import DeviceRun

    w = synth.workload("custom", seed=21, q_lens=[300, 77, 129], ctx_lens=[0, 1000, 250],
                       num_q_heads=4, num_kv_heads=2, head_dim=128, top_k=5)
    run = DeviceRun(w, synth.make_tensors(w))
    run.indexer()
    run.topk()
    run.forward()
    torch.cuda.synchronize()
    assert run.status() == 0
    ref_p = run.partial.cpu().numpy()
    ref_l = run.lse.cpu().numpy()
    filled = (run.idx.cpu().numpy() >= 0).T  # [slot][row]
    status = torch.zeros(1, dtype=torch.int32, device=run.dev)
    for call in range(2):
        partial = torch.full_like(run.partial, float("nan"))
        lse = torch.full_like(run.lse, float("nan"))
        B.sparse_prefill_fwd_noalloc(run.plan, run.q, run.q_scale, run.k, run.v, run.k_scales,
                                     run.v_scales, run.page_table, run.idx, partial, lse,
                                     dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        got_p = partial.cpu().numpy()
        got_l = lse.cpu().numpy()
        assert np.all(got_l[~filled] == -np.inf)
        assert np.all(np.isnan(got_p[~filled]))
        assert _rel_l2(got_p[filled], ref_p[filled]) <= PARTIAL_RL2
        assert np.max(np.abs(got_l[filled] - ref_l[filled])) <= LSE_ATOL
        # the same kernels on the same inputs: expect identical bits
        assert np.array_equal(got_p[filled].view(np.uint32), ref_p[filled].view(np.uint32))


def test_noalloc_rejects_a_batch_larger_than_its_scratch():
    from paged_top_sparse_gb300 import binding as B

    plan = B.Plan([16384], [0], 32, 2, 128, 16, 128, 128)
    assert plan.workspace_bytes > 48 << 20
    L = B.lib()
    R = 16384 * 32
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = L.sparse_prefill_fwd_noalloc(plan.handle, fake, 1.0, fake, fake, None, None, fake, fake,
                                      fake, R * 128, fake, R, None, None)
    assert st == 3  # SPS_ENOSPACE
    assert b"scratch" in L.sps_last_error()
