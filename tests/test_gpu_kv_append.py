"""GPU parity of the chunked-prefill append step: sps_kv_append (BF16 and NVFP4 caches),
sps_quantize_e4m3 and sps_absmax_bf16 through the C ABI, byte-exact against the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import oracle as orc
from paged_top_sparse_gb300 import synth
from tests.helpers import oracle_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_top_sparse_gb300 import build

    build.build()


def _edge_rows(rng, T, G, D):
    """New K/V rows with the blocks that decide the rounding: all-zero blocks, signed zeros,
    tiny blocks whose scale rounds to zero, huge blocks that saturate the scale, exact E2M1
    midpoints at scale 1, and ordinary N(0,1) values."""
    x = rng.standard_normal((T, G, D)).astype(np.float32)
    flat = x.reshape(-1, 16)
    n = flat.shape[0]
    flat[0::7] = 0.0
    flat[1::7, ::2] = -0.0
    flat[2::7] *= 1e-6
    flat[3::7] *= 3e3
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    flat[4::7] = np.concatenate([mids, -mids])[None, :]
    return synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("kv_dtype,D", [("bf16", 128), ("nvfp4", 128), ("nvfp4", 64), ("bf16", 64)])
def test_kv_append_bytes_match_oracle(kv_dtype, D):
    from paged_top_sparse_gb300 import binding as B

    w = synth.workload("custom", seed=51, q_lens=[200, 64, 131, 1], ctx_lens=[1000, 2900, 555, 127],
                       num_q_heads=4, num_kv_heads=2, head_dim=D, top_k=4, kv_dtype=kv_dtype,
                       q_dtype="e4m3" if kv_dtype == "nvfp4" else "bf16")
    rng = np.random.default_rng(52)
    T, G, NP = w.num_tokens, w.num_kv_heads, w.num_phys_pages
    knew, vnew = _edge_rows(rng, T, G, D), _edge_rows(rng, T, G, D)
    if kv_dtype == "bf16":
        kc = rng.integers(0, 1 << 16, (NP, G, 128, D), dtype=np.uint16)
        vc = rng.integers(0, 1 << 16, (NP, G, 128, D), dtype=np.uint16)
        ks = vs = None
    else:
        kc = rng.integers(0, 256, (NP, G, 128, D // 2), dtype=np.uint8)
        vc = rng.integers(0, 256, (NP, G, 128, D // 2), dtype=np.uint8)
        ks = rng.integers(0, 0x7F, (NP, G, 128, D // 16), dtype=np.uint8)
        vs = rng.integers(0, 0x7F, (NP, G, 128, D // 16), dtype=np.uint8)
    dev = "cuda:0"

    def td(a):
        if a is None:
            return None
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    plan = B.Plan(w.q_lens, w.ctx_lens, w.num_q_heads, G, D, w.top_k, w.max_pages, NP,
                  q_dtype=w.q_dtype, kv_dtype=kv_dtype)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    B.sps_plan_upload(plan, ws)
    dk, dv, dks, dvs = td(kc.copy()), td(vc.copy()), td(None if ks is None else ks.copy()), td(None if vs is None else vs.copy())
    pt = torch.from_numpy(w.page_table.astype(np.int32)).to(dev)
    B.sps_kv_append(plan, td(knew), td(vnew), pt, dk, dv, dks, dvs, ws)
    torch.cuda.synchronize()
    assert B.sps_read_device_status(plan, ws) == 0
    pb = oracle_problem(w)
    for new, cache, scl, dc, dsc in ((knew, kc, ks, dk, dks), (vnew, vc, vs, dv, dvs)):
        orc.kv_append(pb, kv_dtype, new, cache, scl)
        got = dc.cpu().numpy().view(cache.dtype)
        assert np.array_equal(got, cache)
        if scl is not None:
            assert np.array_equal(dsc.cpu().numpy(), scl)


def test_quantize_e4m3_and_absmax_match_oracle():
    from paged_top_sparse_gb300 import binding as B

    rng = np.random.default_rng(53)
    x = (rng.standard_normal(1 << 16) * np.exp(rng.uniform(-12, 10, 1 << 16))).astype(np.float32)
    x[:64] = [0.0, -0.0] * 32
    bits = synth.f32_to_bf16_bits(x)
    xd = torch.from_numpy(bits.view(np.int16)).cuda()
    amax = torch.zeros(1, dtype=torch.float32, device="cuda:0")
    B.sps_absmax_bf16(xd, amax)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    torch.cuda.synchronize()
    assert amax.item() == np.abs(xb).max()
    for scale in (float(np.abs(xb).max()) / 448.0, 1.0, 0.0078125, 3.0):
        codes = torch.empty(bits.size, dtype=torch.uint8, device="cuda:0")
        B.sps_quantize_e4m3(xd, scale, codes)
        torch.cuda.synchronize()
        want = orc.quantize_e4m3(bits, np.float32(scale))
        assert np.array_equal(codes.cpu().numpy(), want), scale
