"""GPU parity: every step through the C ABI against the FP64 oracle on the same seeded inputs.

Tolerances (the method's stated bar):
  * plan metadata, page selection and the page -> row inversion: bit-exact;
  * scores: |s_gpu - s_ref| <= 1e-5 * max(|s_ref|, A), A = max over the page's visible keys of
    sum_i |q_i k_ji| (the second term covers near-cancelling dot products);
  * partials: relative L2 <= 1e-3 per checked set, LSE: abs <= 1e-4;
  * output: relative L2 <= 2e-3 and max abs <= 1e-2 for BF16 inputs, 5e-3 / 2e-2 for
    E4M3/NVFP4 inputs (against the oracle on the dequantised values).
Top-k is checked on the shared GPU score buffer and the forward on the shared GPU selection,
so each step is compared on identical inputs.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import oracle as orc
from paged_top_sparse_gb300 import synth
from tests.helpers import oracle_problem, oracle_tensors, rel_l2, sample_rows

pytestmark = pytest.mark.gpu

SCORE_RTOL = 1e-5
PARTIAL_RL2 = 1e-3
LSE_ATOL = 1e-4
OUT_TOL = {"bf16": (2e-3, 1e-2), "quant": (5e-3, 2e-2)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_top_sparse_gb300 import build

    build.build()


def _workload(name):
    if name == "ragged":
        return synth.workload("custom", seed=11, q_lens=[300, 77, 129], ctx_lens=[0, 1000, 250],
                              num_q_heads=4, num_kv_heads=2, head_dim=128, top_k=5)
    if name == "mha_d64":
        return synth.workload("custom", seed=12, q_lens=[200], ctx_lens=[130], num_q_heads=3,
                              num_kv_heads=3, head_dim=64, top_k=2)
    if name == "k1":
        return synth.workload("custom", seed=13, q_lens=[257], ctx_lens=[0], num_q_heads=2,
                              num_kv_heads=1, head_dim=128, top_k=1)
    if name == "quant_small":  # E4M3 Q, NVFP4 K/V (attention and indexer)
        return synth.workload("custom", seed=15, q_lens=[300, 77], ctx_lens=[0, 1000],
                              num_q_heads=4, num_kv_heads=2, head_dim=128, top_k=5,
                              q_dtype="e4m3", kv_dtype="nvfp4")
    if name == "quant_d64":
        return synth.workload("custom", seed=16, q_lens=[190], ctx_lens=[70], num_q_heads=2,
                              num_kv_heads=1, head_dim=64, top_k=2, q_dtype="e4m3",
                              kv_dtype="nvfp4")
    if name == "maxctx":  # 512 pages, 64K tokens
        return synth.workload("custom", seed=41, q_lens=[200], ctx_lens=[65300], num_q_heads=4,
                              num_kv_heads=2, head_dim=128, top_k=16)
    if name == "ctx128k":  # 1024 pages, 128K tokens: the single-launch inversion's widest case
        return synth.workload("custom", seed=43, q_lens=[200], ctx_lens=[130800],
                              num_q_heads=4, num_kv_heads=2, head_dim=128, top_k=16)
    if name == "ctx1m":  # 8192 pages, 1M tokens: the largest page count a plan takes (top_k 16);
        # 32 rows, so top-k runs its TMA form; the inversion runs its multi-kernel form
        return synth.workload("custom", seed=44, q_lens=[16], ctx_lens=[1048560],
                              num_q_heads=2, num_kv_heads=1, head_dim=64, top_k=16)
    if name == "ctx1m_q":  # the same limit with E4M3 Q and NVFP4 K/V (the indexer's key-page
        # conversion over 8192 pages, the forward's loader dequant), top-8
        return synth.workload("custom", seed=45, q_lens=[16], ctx_lens=[1048560],
                              num_q_heads=2, num_kv_heads=1, head_dim=64, top_k=8,
                              q_dtype="e4m3", kv_dtype="nvfp4")
    if name == "with_empty":  # requests without new tokens between others
        return synth.workload("custom", seed=42, q_lens=[0, 150, 0, 33],
                              ctx_lens=[500, 700, 0, 1000], num_q_heads=4, num_kv_heads=2,
                              head_dim=64, top_k=4)
    if name == "chunked_fp8_small":  # chunked prefill, E4M3 indexer q/k, BF16 attention
        return synth.workload("custom", seed=14, q_lens=[200, 64, 131], ctx_lens=[1000, 2900, 555],
                              num_q_heads=4, num_kv_heads=2, head_dim=128, top_k=6,
                              idx_dtype="e4m3")
    return synth.workload(name, seed=0)


SMALL = ["tiny", "ragged", "mha_d64", "k1", "chunked_fp8_small", "quant_small", "quant_d64",
         "maxctx", "ctx128k", "ctx1m", "ctx1m_q", "with_empty"]
FULL = ["prefill8k", "prefill8k_q", "chunked32k"]
_cache = {}


def _run(name):
    """Run the whole path once per workload (module cache) and return everything."""
    if name in _cache:
        return _cache[name]
    from tests.gpu_helpers import DeviceRun

    w = _workload(name)
    t = synth.make_tensors(w)
    run = DeviceRun(w, t)
    run.run_all()
    assert run.status() == 0
    full = w.num_rows <= 20000
    rows = np.arange(w.num_rows, dtype=np.int64) if full else sample_rows(w, 192)
    rows_t = torch.from_numpy(rows).to(run.dev)
    res = dict(
        w=w, t=t, run=run, rows=rows,
        scores=run.scores[rows_t].cpu().numpy(),
        idx=run.idx[rows_t].cpu().numpy(),
        partial=run.partial[:, rows_t].cpu().numpy(),
        lse=run.lse[:, rows_t].cpu().numpy(),
        out=run.out[rows_t].float().cpu().numpy(),
        out_lse=run.out_lse[rows_t].cpu().numpy(),
    )
    _cache[name] = res
    return res


def _abs_tensor(tn: orc.Tensor) -> orc.Tensor:
    """Same tensor with every element's sign cleared (for the |q|.|k| bound)."""
    mask = {"bf16": 0x7FFF, "fp16": 0x7FFF, "e4m3": 0x7F, "nvfp4": 0x77}[tn.dtype]
    data = tn.data & np.array(mask, dtype=tn.data.dtype)
    return orc.Tensor(data, tn.dtype, scales=tn.scales, scale=abs(tn.scale))


@pytest.mark.parametrize("name", SMALL + FULL)
def test_plan_metadata_bit_exact(name):
    r = _run(name)
    run, w = r["run"], r["w"]
    info = run.plan.info()
    pos = run.ws_array(info.off_tok_pos, w.num_tokens, np.int32)
    req = run.ws_array(info.off_tok_req, w.num_tokens, np.int32)
    oreq, opos = orc.token_meta(oracle_problem(w))
    assert np.array_equal(pos, opos) and np.array_equal(req, oreq)


@pytest.mark.parametrize("name", SMALL + FULL)
def test_indexer_scores(name):
    r = _run(name)
    w, rows = r["w"], r["rows"]
    pb = oracle_problem(w)
    q, k, v, qi, ki = oracle_tensors(w, r["t"])
    ref = orc.indexer(pb, qi, ki, rows)
    bound = orc.indexer(pb, _abs_tensor(qi), _abs_tensor(ki), rows)
    got = r["scores"][:, : w.max_pages].astype(np.float64)
    vis = ~np.isnan(ref)
    assert np.array_equal(vis, ~np.isnan(got)), "written entries must be exactly p <= o"
    err = np.abs(got[vis] - ref[vis])
    tol = SCORE_RTOL * np.maximum(np.abs(ref[vis]), bound[vis])
    assert np.all(err <= tol), f"max err/tol {np.max(err / tol):.3g}"


@pytest.mark.parametrize("name", SMALL + FULL)
def test_topk_bit_exact_on_shared_scores(name):
    r = _run(name)
    w, rows = r["w"], r["rows"]
    ref = orc.topk(oracle_problem(w), np.nan_to_num(r["scores"].astype(np.float64), nan=-np.inf),
                   rows)
    assert np.array_equal(r["idx"], ref)


@pytest.mark.parametrize("q_lens,ctx_lens,k", [
    ([1024], [0], 4),            # 8 pages
    ([601, 334], [4500, 0], 16),  # up to 41 pages, two requests, ragged rows
    ([500], [7600], 16),          # 64 pages
    ([256], [12000], 7),          # 96 pages
    ([64], [20000], 16),          # 157 pages
    ([200], [3000], 32),          # 25 pages, k above the page count for most rows
    ([130], [38000], 64),         # 298 pages, the largest k
    ([300], [40000], 16),         # 315 pages
    ([100], [44000], 16),         # 345 pages
    ([50], [65000], 16),          # 508 pages
    ([40], [89000], 16),          # 696 pages
    ([30], [127900], 16),         # 1000 pages
    ([20], [130900], 64),         # 1023 pages, the largest k
    ([20], [200000], 16),         # 1563 pages: pass 1 in segments merged per row
    ([12], [500000], 5),          # 3907 pages, segments
    ([8], [1048000], 16),         # 8192 pages (the limit), sixteen segments
])
def test_topk_ties_and_signed_zeros(q_lens, ctx_lens, k):
    """Scores drawn from {-1.5, ..., 1.5} with signed zeros: most pages tie with others, so
    the (score desc, page asc) order and -0.0 == +0.0 decide most selections."""
    from paged_top_sparse_gb300 import binding as B

    w = synth.workload("custom", seed=21, q_lens=q_lens, ctx_lens=ctx_lens, num_q_heads=4,
                       num_kv_heads=2, head_dim=128, top_k=k)
    plan = B.Plan(w.q_lens, w.ctx_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.top_k,
                  w.max_pages, w.num_phys_pages)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda:0")
    B.sps_plan_upload(plan, ws)
    rng = np.random.default_rng(5)
    R, P = w.num_rows, w.max_pages
    s = (rng.integers(-3, 4, size=(R, P)) * 0.5).astype(np.float32)
    s[rng.random((R, P)) < 0.2] = -0.0
    s[:7] = 1.0  # whole rows of equal scores
    _, tok_pos = orc.token_meta(oracle_problem(w))
    own = (tok_pos[np.arange(R) // w.num_q_heads] // 128)[:, None]
    s[np.arange(P)[None, :] > own] = np.nan  # never read by the selection
    idx = torch.full((R, k), -7, dtype=torch.int32, device="cuda:0")
    B.topk_select(plan, torch.from_numpy(s).cuda(), idx, ws)
    torch.cuda.synchronize()
    ref = orc.topk(oracle_problem(w), np.nan_to_num(s.astype(np.float64), nan=-np.inf))
    assert np.array_equal(idx.cpu().numpy(), ref)


@pytest.mark.parametrize("k", [16, 9, 2])
def test_topk_long_rows_by_segments(k):
    """Rows of ~4700 pages in a batch of 128 rows: pass 1 runs in segments, and pass 2 by
    segments for the warps whose rows all have an unshared threshold (warps 1 and 3, N(0,1)
    scores) and row by row for the others (warps 0 and 2, scores from {-1, ..., 1} with signed
    zeros, so thresholds are shared)."""
    from paged_top_sparse_gb300 import binding as B

    w = synth.workload("custom", seed=23, q_lens=[32], ctx_lens=[600000], num_q_heads=4,
                       num_kv_heads=2, head_dim=128, top_k=k)
    plan = B.Plan(w.q_lens, w.ctx_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.top_k,
                  w.max_pages, w.num_phys_pages)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda:0")
    B.sps_plan_upload(plan, ws)
    rng = np.random.default_rng(7)
    R, P = w.num_rows, w.max_pages
    assert R == 128
    s = rng.standard_normal((R, P)).astype(np.float32)
    for wp in (0, 2):
        t = (rng.integers(-2, 3, size=(32, P)) * 0.5).astype(np.float32)
        t[rng.random((32, P)) < 0.2] = -0.0
        s[32 * wp:32 * wp + 32] = t
    _, tok_pos = orc.token_meta(oracle_problem(w))
    own = (tok_pos[np.arange(R) // w.num_q_heads] // 128)[:, None]
    s[np.arange(P)[None, :] > own] = np.nan
    idx = torch.full((R, k), -7, dtype=torch.int32, device="cuda:0")
    B.topk_select(plan, torch.from_numpy(s).cuda(), idx, ws)
    torch.cuda.synchronize()
    assert B.sps_read_device_status(plan, ws) == 0
    ref = orc.topk(oracle_problem(w), np.nan_to_num(s.astype(np.float64), nan=-np.inf))
    got = idx.cpu().numpy()
    bad = np.nonzero(~np.all(got == ref, axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:5]}"


def test_topk_long_and_short_rows_in_one_warp():
    """A plan whose long request (5469 pages) splits the top-k into segments, with a second
    request of one or two pages: the first warp holds 24 long rows and 8 short ones (fewer
    visible pages than k: every page, then -1), so the segment kernels skip rows the row kernel
    writes whole."""
    from paged_top_sparse_gb300 import binding as B

    w = synth.workload("custom", seed=26, q_lens=[6, 40], ctx_lens=[700000, 100], num_q_heads=4,
                       num_kv_heads=2, head_dim=128, top_k=16)
    plan = B.Plan(w.q_lens, w.ctx_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.top_k,
                  w.max_pages, w.num_phys_pages)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda:0")
    B.sps_plan_upload(plan, ws)
    rng = np.random.default_rng(8)
    R, P = w.num_rows, w.max_pages
    s = rng.standard_normal((R, P)).astype(np.float32)
    _, tok_pos = orc.token_meta(oracle_problem(w))
    own = (tok_pos[np.arange(R) // w.num_q_heads] // 128)[:, None]
    s[np.arange(P)[None, :] > own] = np.nan
    idx = torch.full((R, w.top_k), -7, dtype=torch.int32, device="cuda:0")
    B.topk_select(plan, torch.from_numpy(s).cuda(), idx, ws)
    torch.cuda.synchronize()
    assert B.sps_read_device_status(plan, ws) == 0
    ref = orc.topk(oracle_problem(w), np.nan_to_num(s.astype(np.float64), nan=-np.inf))
    assert np.array_equal(idx.cpu().numpy(), ref)


@pytest.mark.parametrize("pad", [0, 1, 4])
@pytest.mark.parametrize("q_lens,ctx_lens,k", [
    ([150, 90, 301], [2100, 700, 0], 16),  # three requests: rows of a warp see different pages
    ([200], [7000], 15),
    ([100], [9000], 2),
    ([120], [5000], 1),
    ([64], [40000], 16),                   # 313 pages: twenty groups of 16
    ([5], [2100], 16),                     # 20 rows (< 32: per-thread loads), 17 pages
    ([40], [300000], 16),                  # 2345 pages: pass 1 in segments (16-byte pitch)
])
def test_topk_strided_scores(q_lens, ctx_lens, k, pad):
    """The score buffer as a view whose row pitch exceeds max_pages (pad 0 and 4: a pitch that
    is a multiple of 4, read with 16-byte loads; pad 1: an odd pitch, read element by element).
    Half the rows hold N(0,1) scores, half scores from {-1, -0.5, 0, 0.5, 1} (ties); every entry
    past the own page and the pitch padding hold NaN."""
    from paged_top_sparse_gb300 import binding as B

    w = synth.workload("custom", seed=22, q_lens=q_lens, ctx_lens=ctx_lens, num_q_heads=4,
                       num_kv_heads=2, head_dim=128, top_k=k)
    plan = B.Plan(w.q_lens, w.ctx_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, w.top_k,
                  w.max_pages, w.num_phys_pages)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda:0")
    B.sps_plan_upload(plan, ws)
    rng = np.random.default_rng(6)
    R, P = w.num_rows, w.max_pages
    s = rng.standard_normal((R, P)).astype(np.float32)
    tie_rows = rng.random(R) < 0.5
    s[tie_rows] = (rng.integers(-2, 3, size=(int(tie_rows.sum()), P)) * 0.5).astype(np.float32)
    _, tok_pos = orc.token_meta(oracle_problem(w))
    own = (tok_pos[np.arange(R) // w.num_q_heads] // 128)[:, None]
    s[np.arange(P)[None, :] > own] = np.nan
    pitch = (P + 3) // 4 * 4 + pad
    buf = torch.full((R, pitch), float("nan"), dtype=torch.float32, device="cuda:0")
    buf[:, :P] = torch.from_numpy(s).cuda()
    view = buf[:, :P]
    assert view.stride(0) == pitch
    idx = torch.full((R, k), -7, dtype=torch.int32, device="cuda:0")
    B.topk_select(plan, view, idx, ws)
    torch.cuda.synchronize()
    ref = orc.topk(oracle_problem(w), np.nan_to_num(s.astype(np.float64), nan=-np.inf))
    got = idx.cpu().numpy()
    bad = np.nonzero(~np.all(got == ref, axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:5]}"


@pytest.mark.parametrize("name", SMALL + FULL)
def test_forward_partials_and_lse(name):
    r = _run(name)
    w, rows = r["w"], r["rows"]
    q, k, v, qi, ki = oracle_tensors(w, r["t"])
    part, lse = orc.forward(oracle_problem(w), q, k, v, w.sm_scale, r["idx"], rows)
    got_p = r["partial"].transpose(1, 0, 2)  # [rows][slot][D]
    got_l = r["lse"].T
    filled = r["idx"] >= 0
    assert np.all(got_l[~filled] == -np.inf)
    assert np.all(np.isnan(got_p[~filled])), "empty slots must not be written"
    assert rel_l2(got_p[filled], part[filled]) <= PARTIAL_RL2
    assert np.max(np.abs(got_l[filled] - lse[filled])) <= LSE_ATOL


@pytest.mark.parametrize("name", SMALL + FULL)
def test_output_matches_oracle(name):
    r = _run(name)
    w, rows = r["w"], r["rows"]
    q, k, v, qi, ki = oracle_tensors(w, r["t"])
    ref, ref_lse = orc.dense(oracle_problem(w), q, k, v, w.sm_scale, r["idx"], rows)
    rl2_tol, abs_tol = OUT_TOL["bf16" if w.kv_dtype == "bf16" else "quant"]
    err, mx = rel_l2(r["out"], ref), float(np.max(np.abs(r["out"] - ref)))
    print(f"{name}: output rel L2 {err:.3e}, max abs {mx:.3e}")
    assert err <= rl2_tol and mx <= abs_tol, (name, err, mx)
    assert np.max(np.abs(r["out_lse"] - ref_lse)) <= LSE_ATOL


@pytest.mark.parametrize("name", SMALL + FULL)
def test_inversion_bit_exact(name):
    r = _run(name)
    run, w = r["run"], r["w"]
    if w.num_rows > 20000:
        idx_all = run.idx.cpu().numpy()
    else:
        idx_all = r["idx"]
    offsets, er, es = orc.inversion(oracle_problem(w), idx_all)
    info = run.plan.info()
    nb = len(offsets) - 1
    got_off = run.ws_array(info.off_bucket_offsets, nb + 1, np.int32)
    assert np.array_equal(got_off, offsets.astype(np.int32))
    ent = run.ws_array(info.off_entries, 2 * len(er), np.int32).reshape(-1, 2)
    _, tok_pos = orc.token_meta(oracle_problem(w))
    assert np.array_equal(ent[:, 0], er)
    assert np.array_equal(ent[:, 1] & 63, es)
    assert np.array_equal(ent[:, 1] >> 6, tok_pos[er // w.num_q_heads])


def test_determinism_three_runs():
    from tests.gpu_helpers import DeviceRun

    w = _workload("ragged")
    t = synth.make_tensors(w)
    outs = []
    for _ in range(3):
        run = DeviceRun(w, t)
        run.run_all()
        outs.append([x.cpu().clone() for x in (run.scores, run.idx, run.partial, run.lse, run.out)])
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                               b.view(torch.uint8) if b.dtype != torch.int32 else b)


def test_wide_score_pitch_and_untouched_entries():
    from tests.gpu_helpers import DeviceRun

    w = _workload("ragged")
    t = synth.make_tensors(w)
    narrow = DeviceRun(w, t)
    narrow.indexer()
    wide = DeviceRun(w, t, pitch=8192)
    wide.indexer()
    torch.cuda.synchronize()
    a = narrow.scores.cpu().numpy()
    b = wide.scores.cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b[:, : a.shape[1]].view(np.uint32))
    assert np.all(np.isnan(b[:, a.shape[1]:]))


def test_cuda_graph_replay_matches_eager():
    from paged_top_sparse_gb300 import binding as B
    from tests.gpu_helpers import DeviceRun

    w = _workload("ragged")
    t = synth.make_tensors(w)
    run = DeviceRun(w, t)
    run.run_all()
    eager = [x.clone() for x in (run.scores, run.idx, run.partial, run.lse, run.out)]
    for x in (run.scores, run.partial, run.lse):
        x.fill_(float("nan"))
    run.out.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            B.indexer_scores(run.plan, run.qi, run.qi_scale, run.ki, run.ki_scales, run.ki_scale,
                             run.page_table, run.scores, run.ws, stream=s)
            B.topk_select(run.plan, run.scores, run.idx, run.ws, stream=s)
            B.sparse_prefill_fwd(run.plan, run.q, run.q_scale, run.k, run.v, run.k_scales,
                                 run.v_scales, run.page_table, run.idx, run.partial, run.lse,
                                 run.ws, stream=s)
            B.partial_combine(run.partial, run.lse, run.out, run.out_lse, stream=s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (run.scores, run.idx, run.partial, run.lse, run.out)):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                           b.view(torch.uint8) if b.dtype != torch.int32 else b)


@pytest.mark.parametrize("D,S,R,pad", [(128, 16, 1000, 0), (64, 5, 77, 12), (128, 1, 33, 4),
                                       (128, 64, 129, 0)])
def test_combine_direct(D, S, R, pad):
    """Plan-free combine on random partials: empty slots (lse = -inf) hold NaN garbage that
    must not leak, one row has no valid slot, split stride padded."""
    from paged_top_sparse_gb300 import binding as B

    g = torch.Generator().manual_seed(D * 1000 + S * 10 + R)
    base = torch.randn((S, R * D + pad * 4), generator=g, dtype=torch.float32)
    lse = 2.0 * torch.randn((S, R), generator=g)
    drop = torch.rand((S, R), generator=g) < 0.3
    lse[drop] = float("-inf")
    lse[:, R // 2] = float("-inf")
    partial_full = base.clone()
    pview = partial_full[:, : R * D].view(S, R, D)
    pview[drop] = float("nan")
    pv = pview.clone()
    dev = "cuda:0"
    pd = partial_full.to(dev)
    partial = pd.as_strided((S, R, D), (R * D + pad * 4, D, 1))
    ld = lse.to(dev)
    out = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty(R, dtype=torch.float32, device=dev)
    B.partial_combine(partial, ld, out, out_lse)
    torch.cuda.synchronize()
    ref, ref_lse = orc.combine(np.nan_to_num(pv.numpy(), nan=0.0), lse.numpy())
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert rel_l2(got, ref) <= 2e-3 and np.max(np.abs(got - ref)) <= 1e-2
    gl = out_lse.cpu().numpy()
    assert gl[R // 2] == -np.inf and np.all(got[R // 2] == 0)
    fin = np.isfinite(ref_lse)
    assert np.max(np.abs(gl[fin] - ref_lse[fin])) <= LSE_ATOL


@pytest.mark.parametrize("D,S,R,pad", [(128, 16, 1000, 0), (64, 5, 77, 16), (128, 1, 33, 8),
                                       (128, 64, 129, 0), (64, 16, 300, 0)])
def test_combine_bf16_direct(D, S, R, pad):
    """Plan-free combine over BF16 partials: the same cases as the FP32 combine, the oracle
    merging the identical (exactly widened) BF16 values."""
    from paged_top_sparse_gb300 import binding as B

    g = torch.Generator().manual_seed(D * 1000 + S * 10 + R + 7)
    base = torch.randn((S, R * D + pad * 8), generator=g).to(torch.bfloat16)
    lse = 2.0 * torch.randn((S, R), generator=g)
    drop = torch.rand((S, R), generator=g) < 0.3
    lse[drop] = float("-inf")
    lse[:, R // 2] = float("-inf")
    pview = base[:, : R * D].view(S, R, D)
    pview[drop] = float("nan")
    pv = pview.float().clone()
    dev = "cuda:0"
    pd = base.to(dev)
    partial = pd.as_strided((S, R, D), (R * D + pad * 8, D, 1))
    ld = lse.to(dev)
    out = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty(R, dtype=torch.float32, device=dev)
    B.partial_combine_bf16(partial, ld, out, out_lse)
    torch.cuda.synchronize()
    ref, ref_lse = orc.combine(np.nan_to_num(pv.numpy(), nan=0.0), lse.numpy())
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert rel_l2(got, ref) <= 2e-3 and np.max(np.abs(got - ref)) <= 1e-2
    gl = out_lse.cpu().numpy()
    assert gl[R // 2] == -np.inf and np.all(got[R // 2] == 0)
    fin = np.isfinite(ref_lse)
    assert np.max(np.abs(gl[fin] - ref_lse[fin])) <= LSE_ATOL


P16_WORKLOADS = ["tiny", "ragged", "mha_d64", "k1", "quant_small", "chunked_fp8_small",
                 "ctx1m", "prefill8k"]


@pytest.mark.parametrize("storage", ["f16", "bf16"])
@pytest.mark.parametrize("name", P16_WORKLOADS)
def test_16bit_partials_path(name, storage):
    """sparse_prefill_fwd_{f16,bf16} + partial_combine_{f16,bf16} on the FP32 run's selection:
    each 16-bit partial is the FP32 path's partial rounded to nearest even (bit-exact), the
    LSEs are the FP32 path's bit for bit, the combine matches the oracle merge of those 16-bit
    values, and the output matches the oracle's partials stored in the same 16-bit format and
    merged.  FP16 storage (11 significant bits) also holds the direct definition within the
    contract's output bound; BF16 storage (8 bits) adds a second BF16 rounding of about 1.1e-3
    relative per partial, which rows that merge one or two partials cannot average away, so its
    distance to the direct definition is reported, not bounded."""
    from paged_top_sparse_gb300 import binding as B

    r = _run(name)
    w, run, rows = r["w"], r["run"], r["rows"]
    R, K, D = w.num_rows, w.top_k, w.head_dim
    dev = run.dev
    tdt = torch.float16 if storage == "f16" else torch.bfloat16
    fwd = B.sparse_prefill_fwd_f16 if storage == "f16" else B.sparse_prefill_fwd_bf16
    comb = B.partial_combine_f16 if storage == "f16" else B.partial_combine_bf16
    pb = torch.full((K, R, D), float("nan"), dtype=tdt, device=dev)
    lse = torch.full((K, R), float("nan"), dtype=torch.float32, device=dev)
    fwd(run.plan, run.q, run.q_scale, run.k, run.v, run.k_scales, run.v_scales, run.page_table,
        run.idx, pb, lse, run.ws)
    out = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
    olse = torch.empty((R,), dtype=torch.float32, device=dev)
    comb(pb, lse, out, olse)
    torch.cuda.synchronize()
    assert run.status() == 0
    rows_t = torch.from_numpy(rows).to(dev)
    live = torch.from_numpy((r["idx"] >= 0).T.copy()).to(dev)  # [K][rows]
    got_p = pb[:, rows_t]
    want_p = run.partial[:, rows_t].to(tdt)
    assert torch.equal(got_p[live].view(torch.int16), want_p[live].view(torch.int16))
    assert torch.equal(lse[:, rows_t], run.lse[:, rows_t])
    # the combine against the oracle on the same 16-bit partials
    pnp = got_p.float().cpu().numpy().astype(np.float64)
    lnp = lse[:, rows_t].cpu().numpy().astype(np.float64)
    ref_c, _ = orc.combine(np.where(np.isfinite(pnp), pnp, 0.0), lnp)
    got = out[rows_t].float().cpu().numpy()
    rl2_tol, abs_tol = OUT_TOL["bf16" if w.kv_dtype == "bf16" else "quant"]
    assert rel_l2(got, ref_c) <= 2e-3 and np.max(np.abs(got - ref_c)) <= 1e-2
    # against the oracle's own partials, stored in the same format and merged
    q, k, v, qi, ki = oracle_tensors(w, r["t"])
    opart, olse_ = orc.forward(oracle_problem(w), q, k, v, w.sm_scale, r["idx"], rows)
    opart16 = torch.from_numpy(opart).to(tdt).double().numpy()  # [rows][slot][D]
    ref_s, _ = orc.combine(np.nan_to_num(opart16.transpose(1, 0, 2), nan=0.0), olse_.T)
    err_s, mx_s = rel_l2(got, ref_s), float(np.max(np.abs(got - ref_s)))
    # against the direct definition
    ref, _ = orc.dense(oracle_problem(w), q, k, v, w.sm_scale, r["idx"], rows)
    err, mx = rel_l2(got, ref), float(np.max(np.abs(got - ref)))
    print(f"{name}: {storage} partials, output rel L2 {err:.3e} (max abs {mx:.3e}) against the "
          f"definition, {err_s:.3e} (max abs {mx_s:.3e}) against {storage}-stored oracle partials")
    assert err_s <= rl2_tol and mx_s <= abs_tol, (name, storage, err_s, mx_s)
    if storage == "f16":
        assert err <= rl2_tol and mx <= abs_tol, (name, err, mx)


@pytest.mark.parametrize("name", ["quant_small", "prefill8k_q"])
def test_fp8qk_route_matches_oracle_on_e4m3_rounded_keys(name):
    """sparse_prefill_fwd_fp8qk (the pages' Q8KV4 route: K products rounded to E4M3, FP8 Q K^T)
    against the oracle decoding K the same way (the 'nvfp4_e4m3' tensor): partials and LSE at
    the exact path's tolerances, the combined output at the quantised-input bound.  The
    distance to the exact-product oracle is reported by the second check, whose bound is the
    rounding of K to E4M3 (3 mantissa bits) seen through the softmax."""
    from paged_top_sparse_gb300 import binding as B

    r = _run(name)
    w, run, rows = r["w"], r["run"], r["rows"]
    R, K, D = w.num_rows, w.top_k, w.head_dim
    dev = run.dev
    part = torch.full((K, R, D), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((K, R), float("nan"), dtype=torch.float32, device=dev)
    B.sparse_prefill_fwd_fp8qk(run.plan, run.q, run.q_scale, run.k, run.v, run.k_scales,
                               run.v_scales, run.page_table, run.idx, part, lse, run.ws)
    out = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
    B.partial_combine(part, lse, out)
    torch.cuda.synchronize()
    assert run.status() == 0
    rows_t = torch.from_numpy(rows).to(dev)
    q, k, v, qi, ki = oracle_tensors(w, r["t"])
    kr = orc.Tensor(k.data, "nvfp4_e4m3", scales=k.scales, scale=k.scale)
    pb = oracle_problem(w)
    ref_p, ref_l = orc.forward(pb, q, kr, v, w.sm_scale, r["idx"], rows)
    got_p = part[:, rows_t].cpu().numpy().transpose(1, 0, 2)
    got_l = lse[:, rows_t].cpu().numpy().T
    live = r["idx"] >= 0
    assert rel_l2(got_p[live], ref_p[live]) <= PARTIAL_RL2
    assert np.max(np.abs(got_l[live] - ref_l[live])) <= LSE_ATOL
    got = out[rows_t].float().cpu().numpy()
    ref, _ = orc.dense(pb, q, kr, v, w.sm_scale, r["idx"], rows)
    tol = OUT_TOL["quant"]
    assert rel_l2(got, ref) <= tol[0] and np.max(np.abs(got - ref)) <= tol[1]
    exact, _ = orc.dense(pb, q, k, v, w.sm_scale, r["idx"], rows)
    assert rel_l2(got, exact) <= 5e-2


def test_bad_page_table_entry_sets_status():
    """An out-of-range physical page is caught on the device: status, no fault."""
    from tests.gpu_helpers import DeviceRun

    w = _workload("ragged")
    t = synth.make_tensors(w)
    run = DeviceRun(w, t)
    run.page_table[0, 1] = w.num_phys_pages + 5
    run.indexer()
    assert run.status() == 2  # SPS_DEV_BAD_PAGE


def test_host_rejects_invalid_arguments():
    from paged_top_sparse_gb300 import binding as B
    from tests.gpu_helpers import DeviceRun

    w = _workload("ragged")
    t = synth.make_tensors(w)
    run = DeviceRun(w, t)
    bad = torch.empty((w.num_rows, w.max_pages - 1), dtype=torch.float32, device="cuda:0")
    with pytest.raises(B.SpsError) as e:
        B.indexer_scores(run.plan, run.qi, 1.0, run.ki, None, 1.0, run.page_table, bad, run.ws)
    assert e.value.status == 1
    small_ws = run.ws[: run.plan.workspace_bytes // 2]
    with pytest.raises(B.SpsError) as e:
        B.sps_plan_upload(run.plan, small_ws)
    assert e.value.status == 3


def test_combine_stress_full_size():
    """The combine-stress workload at full size: partial [16][16384*32][128] FP32 (4.3 GB) and
    LSE ~ N(0, sd 2), generated on the device; sampled rows against the oracle."""
    from paged_top_sparse_gb300 import binding as B

    S, R, D = 16, 16384 * 32, 128
    part, lse = synth.combine_inputs(R, S, D, seed=5, device="cuda:0")
    lse[3, ::7] = float("-inf")  # some empty slots
    out = torch.empty((R, D), dtype=torch.bfloat16, device="cuda:0")
    out_lse = torch.empty(R, dtype=torch.float32, device="cuda:0")
    B.partial_combine(part, lse, out, out_lse)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, R - 1], rng.choice(R, 2000, replace=False)]))
    rt = torch.from_numpy(rows).cuda()
    ref, ref_lse = orc.combine(part[:, rt].cpu().numpy(), lse[:, rt].cpu().numpy())
    got = out[rt].float().cpu().numpy()
    assert rel_l2(got, ref) <= 2e-3 and np.max(np.abs(got - ref)) <= 1e-2
    assert np.max(np.abs(out_lse[rt].cpu().numpy() - ref_lse)) <= LSE_ATOL
    del part, lse


def test_dequant_exhaustive_bit_exact():
    """sps_dequantize against the oracle's decode: every E4M3 code, and every E2M1 code under
    every E4M3 scale (NaN scales give NaN), bit for bit in FP16."""
    from paged_top_sparse_gb300 import binding as B

    codes = np.tile(np.arange(256, dtype=np.uint8), 16)
    out = torch.empty(codes.size, dtype=torch.float16, device="cuda:0")
    B.sps_dequantize("e4m3", torch.from_numpy(codes).cuda(), None, codes.size, out)
    ref = orc.decode(orc.Tensor(codes, "e4m3"))
    got = out.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))

    nib = np.tile(np.arange(16, dtype=np.uint8), 256)          # block b holds codes 0..15
    packed = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    scales = np.arange(256, dtype=np.uint8)                     # block b has scale code b
    out = torch.empty(nib.size, dtype=torch.float16, device="cuda:0")
    B.sps_dequantize("nvfp4", torch.from_numpy(packed).cuda(), torch.from_numpy(scales).cuda(),
                     nib.size, out)
    ref = orc.decode(orc.Tensor(packed, "nvfp4", scales=scales))
    got = out.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_bounded_wait_times_out_without_hanging():
    """A wait on an mbarrier that never completes ends after its limit with SPS_DEV_TIMEOUT in
    the status word; the context stays usable for the next launch."""
    import time

    from paged_top_sparse_gb300 import binding as B

    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    t0 = time.perf_counter()
    B.sps_check_wait_timeout(200_000_000, st)  # 0.2 s
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == 1  # SPS_DEV_TIMEOUT
    assert 0.15 < dt < 5.0
    # the context still works
    part = torch.randn((2, 64, 128), device="cuda:0")
    lse = torch.zeros((2, 64), device="cuda:0")
    out = torch.empty((64, 128), dtype=torch.bfloat16, device="cuda:0")
    B.partial_combine(part, lse, out)
    torch.cuda.synchronize()
    assert torch.allclose(out.float(), part.mean(0), atol=2e-2)


def test_grid_barrier_times_out_without_hanging():
    """The cooperative inversion's grid barrier: one of two blocks leaves without arriving, the
    other's wait ends after its limit with SPS_DEV_TIMEOUT, and the context stays usable."""
    import time

    from paged_top_sparse_gb300 import binding as B

    bar = torch.zeros(2, dtype=torch.int32, device="cuda:0")
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    t0 = time.perf_counter()
    B.sps_check_barrier_timeout(200_000_000, bar, st)  # 0.2 s
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == 1  # SPS_DEV_TIMEOUT
    assert 0.15 < dt < 5.0
    part = torch.randn((2, 64, 128), device="cuda:0")
    lse = torch.zeros((2, 64), device="cuda:0")
    out = torch.empty((64, 128), dtype=torch.bfloat16, device="cuda:0")
    B.partial_combine(part, lse, out)
    torch.cuda.synchronize()
    assert torch.allclose(out.float(), part.mean(0), atol=2e-2)


@pytest.mark.parametrize("q_len,ctx,H", [
    (12000, 0, 32),      # 94 pages: one group of two 64-page windows (shared-memory ORs)
    (8100, 0, 64),       # 64 pages: a single window (ballots)
    (12000, 60000, 32),  # 563 pages: a group of eight windows and a single ninth
])
def test_inversion_when_the_single_launch_does_not_fit(q_len, ctx, H):
    """Over 1216 inversion chunks (e.g. 12000 tokens x 16 heads per KV group: 1500), more
    blocks than the GPU holds at once, so the inversion takes its multi-kernel path; the CSR
    offsets and entries must still match the oracle bit for bit (and the 8K workloads above
    cover the single-launch path)."""
    from tests.gpu_helpers import DeviceRun

    w = synth.workload("custom", seed=31, q_lens=[q_len], ctx_lens=[ctx], num_q_heads=H,
                       num_kv_heads=2, head_dim=128, top_k=16)
    run = DeviceRun(w, synth.make_tensors(w))
    run.run_all()
    assert run.status() == 0
    idx_all = run.idx.cpu().numpy()
    offsets, er, es = orc.inversion(oracle_problem(w), idx_all)
    info = run.plan.info()
    nb = len(offsets) - 1
    got_off = run.ws_array(info.off_bucket_offsets, nb + 1, np.int32)
    assert np.array_equal(got_off, offsets.astype(np.int32))
    ent = run.ws_array(info.off_entries, 2 * len(er), np.int32).reshape(-1, 2)
    assert np.array_equal(ent[:, 0], er)
    assert np.array_equal(ent[:, 1] & 63, es)


@pytest.mark.parametrize("q_len", [300, 12000])
def test_repeated_forward_after_one_upload(q_len):
    """Three forward calls on one uploaded workspace give bit-identical partials, LSEs and
    outputs: the inversion's grid barrier returns to zero after each call, so no
    call clears counters.  300 tokens take the single cooperative inversion launch, 12000 tokens
    x 32 heads the multi-kernel path."""
    from tests.gpu_helpers import DeviceRun

    w = synth.workload("custom", seed=32, q_lens=[q_len], ctx_lens=[200], num_q_heads=32,
                       num_kv_heads=2, head_dim=128, top_k=16)
    run = DeviceRun(w, synth.make_tensors(w))
    run.indexer()
    run.topk()
    ref = None
    for _ in range(3):
        run.partial.fill_(float("nan"))
        run.lse.fill_(float("nan"))
        run.forward()
        run.combine()
        torch.cuda.synchronize()
        assert run.status() == 0
        got = [run.partial.view(torch.int32).clone(), run.lse.view(torch.int32).clone(),
               run.out.view(torch.int16).clone()]
        if ref is None:
            ref = got
        else:
            for a, b in zip(ref, got):
                assert torch.equal(a, b)
    idx_all = run.idx.cpu().numpy()
    offsets, er, es = orc.inversion(oracle_problem(w), idx_all)
    info = run.plan.info()
    got_off = run.ws_array(info.off_bucket_offsets, len(offsets), np.int32)
    assert np.array_equal(got_off, offsets.astype(np.int32))
    ent = run.ws_array(info.off_entries, 2 * len(er), np.int32).reshape(-1, 2)
    assert np.array_equal(ent[:, 0], er)


def test_plan_upload_does_not_wait_for_other_streams_copies():
    """The plan upload is a kernel reading the library's mapped page-locked ring, so it does not
    queue behind a large host-to-device copy running on another stream; the uploaded plan is
    the one the next calls use."""
    from paged_top_sparse_gb300 import binding as B
    from tests.gpu_helpers import DeviceRun

    w = _workload("ragged")
    run = DeviceRun(w, synth.make_tensors(w))
    run.run_all()
    ref = run.out.view(torch.int16).clone()

    big_h = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    big_d = torch.empty(1 << 30, dtype=torch.uint8, device="cuda:0")
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    torch.cuda.synchronize()
    ev[0].record(main)
    side.wait_event(ev[0])
    with torch.cuda.stream(side):
        big_d.copy_(big_h, non_blocking=True)
    ev[2].record(side)
    run.ws.zero_()
    B.sps_plan_upload(run.plan, run.ws)
    ev[1].record(main)
    run.out.zero_()
    run.indexer()
    run.topk()
    run.forward()
    run.combine()
    torch.cuda.synchronize()
    assert run.status() == 0
    assert torch.equal(run.out.view(torch.int16), ref)
    upload_ms, copy_ms = ev[0].elapsed_time(ev[1]), ev[0].elapsed_time(ev[2])
    assert copy_ms > 1.0  # 1 GiB over the host link takes milliseconds
    assert upload_ms < 0.5 * copy_ms, (upload_ms, copy_ms)
