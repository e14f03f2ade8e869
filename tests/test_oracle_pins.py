"""Pins for the FP64 oracle: each test ties it to something other than itself.

* decode: library routines (torch bfloat16 / float8_e4m3fn, numpy float16) and the
  published code tables under tests/golden/;
* NVFP4 product exactness: exhaustive over all E2M1 x E4M3 pairs;
* indexer: a dense matrix formulation in numpy (matmul + masked max), brute force;
* top-k: numpy lexsort on (score desc, page asc);
* forward + combine: a dense masked-softmax attention in numpy, and with top-k >= pages the
  plain full causal attention;
* combine: associativity, permutation invariance, empty slots, half-page splitting;
* single-key own page: closed form (partial = v_t, lse = scale q.k_t);
* inversion: a dict-of-lists bucket build.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_top_sparse_gb300 import synth
from tests.helpers import oracle_problem, oracle_tensors, rel_l2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((int(parts[0], 16), float(parts[1])))
    return rows


# ------------------------------------------------------------------ decode pins

def test_bf16_decode_matches_torch_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.decode(orc.Tensor(bits, "bf16"))
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_fp16_decode_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.decode(orc.Tensor(bits, "fp16"))
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_matches_torch_and_golden():
    bits = np.arange(256, dtype=np.uint8)
    got = orc.decode(orc.Tensor(bits, "e4m3"))
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    for code, val in _golden("e4m3_special.txt"):
        g = orc.lib().orc_decode_e4m3(code)
        if math.isnan(val):
            assert math.isnan(g)
        else:
            assert g == val and math.copysign(1, g) == math.copysign(1, val), hex(code)


def test_e2m1_decode_matches_golden_table():
    table = _golden("e2m1_values.txt")
    assert len(table) == 16
    for code, val in table:
        g = orc.lib().orc_decode_e2m1(code)
        assert g == val and math.copysign(1, g) == math.copysign(1, val), hex(code)


def test_nvfp4_element_layout_and_products_exact():
    """Every E2M1 code x every finite E4M3 scale: the oracle's NVFP4 element equals the product
    of the two library/golden decodes, and that product is exact in FP16 and BF16 (so the
    kernels may dequantise to 16-bit without rounding)."""
    e2m1 = np.array([v for _, v in _golden("e2m1_values.txt")])
    e4m3 = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    finite_scales = np.nonzero(np.isfinite(e4m3))[0].astype(np.uint8)
    # one 16-element block per scale: element i holds code (i % 16); packed low nibble first
    nblk = len(finite_scales)
    codes = np.tile(np.arange(16, dtype=np.uint8), nblk)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    got = orc.decode(orc.Tensor(packed, "nvfp4", scales=finite_scales))
    ref = (e2m1[codes] * np.repeat(e4m3[finite_scales], 16))
    assert np.array_equal(got, ref)
    assert np.array_equal(got.astype(np.float16).astype(np.float64), got)
    bf = torch.from_numpy(got).to(torch.bfloat16).double().numpy()
    assert np.array_equal(bf, got)
    # significant bits of the nonzero products: at most 6 (e.g. 1.5 x 1.875 = 2.8125)
    nz = np.abs(got[got != 0])
    m, _ = np.frexp(nz)
    sig = np.array([len(bin(int(x * 2 ** 53)).rstrip("0")) - 2 for x in m])
    assert sig.max() == 6
    assert 1.5 * 1.875 in set(got.tolist())
    # the 4064 signed pairs: 16 codes x 254 finite scales
    assert len(got) == 16 * 254 == 4064


# ------------------------------------------------------------------ small problems

def _small(seed=0, q_lens=(300, 77), ctx=(0, 257), H=4, Hkv=2, D=32, k=3, dtype="bf16"):
    w = synth.workload("custom", seed=seed, q_lens=list(q_lens), ctx_lens=list(ctx),
                       num_q_heads=H, num_kv_heads=Hkv, head_dim=D, top_k=k)
    if dtype != "bf16":
        w.q_dtype, w.kv_dtype = "e4m3", "nvfp4"
    t = synth.make_tensors(w)
    return w, t


def _dense_inputs(w, t):
    """Dense FP64 arrays via the library decoders (torch), independent of the oracle:
    q [T][H][D], and per request the K/V of its logical key positions [n_keys][H_kv][D]."""
    def dec(bits, dtype, scales=None, scale=1.0):
        if dtype == "bf16":
            return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy() * scale
        if dtype == "e4m3":
            return torch.from_numpy(bits).view(torch.float8_e4m3fn).double().numpy() * scale
        if dtype == "nvfp4":
            e2m1 = np.array([v for _, v in _golden("e2m1_values.txt")])
            lo, hi = bits & 0xF, bits >> 4
            codes = np.stack([lo, hi], axis=-1).reshape(*bits.shape[:-1], bits.shape[-1] * 2)
            sc = torch.from_numpy(scales).view(torch.float8_e4m3fn).double().numpy()
            return e2m1[codes] * np.repeat(sc, 16, axis=-1)
        raise ValueError(dtype)

    q = dec(t["q"], w.q_dtype, scale=t.get("q_scale", 1.0))
    kc = dec(t["k"], w.kv_dtype, t.get("k_scales"))
    vc = dec(t["v"], w.kv_dtype, t.get("v_scales"))
    Ks, Vs = [], []
    for b in range(w.batch):
        n_keys = int(w.ctx_lens[b] + w.q_lens[b])
        pos = np.arange(n_keys)
        phys = w.page_table[b][pos // w.page_size]
        Ks.append(kc[phys, :, pos % w.page_size, :])  # [n_keys][H_kv][D]
        Vs.append(vc[phys, :, pos % w.page_size, :])
    return q, Ks, Vs


def _rows_of(w):
    """(row, request, position, kv head) of every row, computed independently."""
    out = []
    tok = 0
    H, g = w.num_q_heads, w.num_q_heads // w.num_kv_heads
    for b in range(w.batch):
        for i in range(int(w.q_lens[b])):
            for h in range(H):
                out.append((tok * H + h, b, int(w.ctx_lens[b]) + i, h // g))
            tok += 1
    return out


def test_token_meta_positions():
    w, _ = _small()
    req, pos = orc.token_meta(oracle_problem(w))
    assert list(req[:300]) == [0] * 300 and list(req[300:]) == [1] * 77
    assert list(pos[:3]) == [0, 1, 2] and pos[300] == 257 and pos[-1] == 257 + 76


def test_indexer_matches_dense_matmul_bruteforce():
    w, t = _small()
    pb = oracle_problem(w)
    q, k, v, qi, ki = oracle_tensors(w, t)
    got = orc.indexer(pb, qi, ki)
    qd, Ks, _ = _dense_inputs(w, t)
    P = w.page_size
    for (r, b, tpos, g) in _rows_of(w):
        h = r % w.num_q_heads
        s = Ks[b][:, g, :] @ qd[r // w.num_q_heads, h]  # all keys of the request
        s = np.where(np.arange(len(s)) <= tpos, s, -np.inf)
        o = tpos // P
        for p in range(w.max_pages):
            if p <= o:
                ref = s[p * P:(p + 1) * P].max()
                assert abs(got[r, p] - ref) <= 1e-12 * max(1.0, abs(ref)), (r, p)
            else:
                assert np.isnan(got[r, p])


def _lexsort_topk(scores_row, o, k):
    """Reference selection by numpy lexsort: own page, then best others by (-score, page)."""
    pages = np.arange(o + 1)
    others = pages[pages != o]
    order = others[np.lexsort((others, -scores_row[others]))]
    chosen = sorted([o] + list(order[: min(k, o + 1) - 1]))
    return chosen + [-1] * (k - len(chosen))


def test_topk_matches_lexsort_with_ties_and_signed_zero():
    w, _ = _small(k=3, ctx=(0, 900))  # up to 9 visible pages, so selection really happens
    pb = oracle_problem(w)
    rng = np.random.default_rng(7)
    rows = np.arange(w.num_rows, dtype=np.int64)
    scores = rng.standard_normal((len(rows), w.max_pages))
    # heavy ties: quantise most rows to a few levels, sprinkle -0.0 and +0.0
    scores[::3] = np.round(scores[::3])
    scores[1::7, ::2] = -0.0
    scores[1::7, 1::2] = 0.0
    idx = orc.topk(pb, scores, rows)
    n_real = 0
    for (r, b, tpos, g) in _rows_of(w):
        n_real += (tpos // w.page_size + 1) > w.top_k
        o = tpos // w.page_size
        assert list(idx[r]) == _lexsort_topk(scores[r] + 0.0, o, w.top_k), r
    assert n_real > 100


def test_topk_invariants():
    w, t = _small(k=3, ctx=(0, 900))
    pb = oracle_problem(w)
    q, k, v, qi, ki = oracle_tensors(w, t)
    s = orc.indexer(pb, qi, ki)
    idx = orc.topk(pb, np.nan_to_num(s, nan=-np.inf))
    for (r, b, tpos, g) in _rows_of(w):
        o = tpos // w.page_size
        sel = [p for p in idx[r] if p >= 0]
        assert o in sel
        assert len(sel) == min(w.top_k, o + 1)
        assert sel == sorted(sel) and len(set(sel)) == len(sel)
        assert all(0 <= p <= o for p in sel)
        assert all(p == -1 for p in idx[r][len(sel):])


def _numpy_sparse_attention(w, t, idx):
    """Dense masked softmax attention: each row attends to the keys of its selected pages
    that are causally visible (matrix formulation, numpy)."""
    qd, Ks, Vs = _dense_inputs(w, t)
    P = w.page_size
    out = np.zeros((w.num_rows, w.head_dim))
    for (r, b, tpos, g) in _rows_of(w):
        h = r % w.num_q_heads
        n_keys = len(Ks[b])
        allowed = np.zeros(n_keys, bool)
        for p in idx[r]:
            if p >= 0:
                allowed[p * P:(p + 1) * P] = True
        allowed &= np.arange(n_keys) <= tpos
        logits = (Ks[b][:, g, :] @ qd[r // w.num_q_heads, h]) * w.sm_scale
        logits = np.where(allowed, logits, -np.inf)
        e = np.exp(logits - logits.max())
        out[r] = (e / e.sum()) @ Vs[b][:, g, :]
    return out


@pytest.mark.parametrize("dtype", ["bf16", "q8kv4"])
def test_pipeline_matches_dense_masked_attention(dtype):
    w, t = _small(dtype=dtype)
    pb = oracle_problem(w)
    q, k, v, qi, ki = oracle_tensors(w, t)
    res = orc.pipeline(pb, q, k, v, w.sm_scale, qi, ki)
    ref = _numpy_sparse_attention(w, t, res["idx"])
    assert rel_l2(res["out"], ref) < 1e-12
    # and the oracle's own direct definition agrees too
    d_out, d_lse = orc.dense(pb, q, k, v, w.sm_scale, res["idx"])
    assert rel_l2(res["out"], d_out) < 1e-12
    assert np.allclose(res["out_lse"], d_lse, rtol=0, atol=1e-10)


def test_topk_all_pages_equals_full_causal_attention():
    w, t = _small(k=8)  # every request here has at most 5 visible pages
    pb = oracle_problem(w)
    q, k, v, qi, ki = oracle_tensors(w, t)
    res = orc.pipeline(pb, q, k, v, w.sm_scale)
    qd, Ks, Vs = _dense_inputs(w, t)
    out = np.zeros_like(res["out"])
    for (r, b, tpos, g) in _rows_of(w):
        h = r % w.num_q_heads
        logits = Ks[b][: tpos + 1, g, :] @ qd[r // w.num_q_heads, h] * w.sm_scale
        e = np.exp(logits - logits.max())
        out[r] = (e / e.sum()) @ Vs[b][: tpos + 1, g, :]
    assert rel_l2(res["out"], out) < 1e-12


def test_single_key_own_page_closed_form():
    """A token at the first position of its page that keeps only its own page attends to
    exactly one key: the partial is v_t and the LSE is scale * q.k_t."""
    w, t = _small(q_lens=(260,), ctx=(0,), H=2, Hkv=1, D=64, k=1)
    pb = oracle_problem(w)
    q, k, v, qi, ki = oracle_tensors(w, t)
    qd, Ks, Vs = _dense_inputs(w, t)
    for tok in (128, 256):
        for h in range(2):
            r = tok * 2 + h
            idx = np.array([[tok // 128]], np.int32)
            part, lse = orc.forward(pb, q, k, v, w.sm_scale, idx, rows=[r])
            assert np.array_equal(part[0, 0], Vs[0][tok, 0])
            assert abs(lse[0, 0] - w.sm_scale * float(qd[tok, h] @ Ks[0][tok, 0])) < 1e-12


def test_combine_associative_permutation_and_empty_slots():
    rng = np.random.default_rng(3)
    S, R, D = 6, 9, 16
    part = rng.standard_normal((S, R, D))
    lse = 2 * rng.standard_normal((S, R))
    lse[2, :4] = -np.inf
    part[2, :4] = np.nan  # garbage in empty slots must not leak
    lse[:, 8] = -np.inf    # a row with no valid slot
    out, olse = orc.combine(part, lse)
    assert np.all(np.isfinite(out))
    assert np.array_equal(out[8], np.zeros(D)) and olse[8] == -np.inf
    perm = rng.permutation(S)
    out_p, olse_p = orc.combine(part[perm], lse[perm])
    assert np.allclose(out_p, out, rtol=1e-13, atol=1e-13)
    # merge in two halves, then merge the halves
    a, la = orc.combine(part[:3], lse[:3])
    b, lb = orc.combine(part[3:], lse[3:])
    ab, lab = orc.combine(np.stack([a, b]), np.stack([la, lb]))
    assert np.allclose(ab[:8], out[:8], rtol=1e-13, atol=1e-13)
    assert np.allclose(lab[:8], olse[:8], rtol=0, atol=1e-13)


def test_combine_of_half_pages_equals_whole_page():
    """Softmax over 128 keys equals the LSE merge of the softmaxes over its two halves."""
    rng = np.random.default_rng(5)
    D = 32
    logits = rng.standard_normal(128) * 3
    V = rng.standard_normal((128, D))

    def sm(lg, vv):
        m = lg.max()
        e = np.exp(lg - m)
        return (e @ vv) / e.sum(), m + np.log(e.sum())

    whole, lwhole = sm(logits, V)
    h1, l1 = sm(logits[:64], V[:64])
    h2, l2 = sm(logits[64:], V[64:])
    out, olse = orc.combine(np.stack([h1, h2])[:, None, :], np.array([[l1], [l2]]))
    assert np.allclose(out[0], whole, rtol=1e-13, atol=1e-13)
    assert abs(olse[0] - lwhole) < 1e-12


def test_inversion_matches_dict_buckets():
    w, t = _small(k=3)
    pb = oracle_problem(w)
    q, k, v, qi, ki = oracle_tensors(w, t)
    s = orc.indexer(pb, qi, ki)
    idx = orc.topk(pb, np.nan_to_num(s, nan=-np.inf))
    offsets, er, es = orc.inversion(pb, idx)
    npages = [(int(c) + int(ql) - 1) // 128 + 1 for c, ql in zip(w.ctx_lens, w.q_lens)]
    base = np.concatenate([[0], np.cumsum(npages)])
    buckets = {}
    for (r, b, tpos, g) in _rows_of(w):
        for s_, p in enumerate(idx[r]):
            if p >= 0:
                buckets.setdefault((int(base[b]) + int(p)) * w.num_kv_heads + g, []).append((r, s_))
    nb = int(base[-1]) * w.num_kv_heads
    assert len(offsets) == nb + 1
    for bk in range(nb):
        lst = list(zip(er[offsets[bk]:offsets[bk + 1]], es[offsets[bk]:offsets[bk + 1]]))
        assert lst == sorted(buckets.get(bk, [])), bk


# ---------------------------------------------------------------- quantisation / append

def _e4m3_ties_and_edges(rng):
    """Random finite values plus every exact midpoint between neighbouring E4M3 values, the
    subnormal range and values just beside the midpoints."""
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    dec = np.array([orc.lib().orc_decode_e4m3(int(c)) for c in codes])
    mids = (dec[:-1] + dec[1:]) / 2.0
    near = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                           np.nextafter(mids.astype(np.float32), np.float32(1e9))])
    rnd = rng.standard_normal(20000) * np.exp(rng.uniform(-9, 6, 20000))
    allv = np.concatenate([dec, near, rnd])
    allv = allv[np.abs(allv) <= 448]
    return np.concatenate([allv, -allv]).astype(np.float32)


def test_e4m3_rounding_matches_torch_ties_to_even():
    """orc.round_e4m3 against torch's float8_e4m3fn conversion (round to nearest even) on every
    midpoint, the subnormals and random values; beyond 448 it saturates to the 0x7E code."""
    rng = np.random.default_rng(41)
    x = _e4m3_ties_and_edges(rng)
    got = orc.round_e4m3(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # -0.0 and +0.0 may differ only in the sign bit for inputs that are zero
    assert np.array_equal(got, want)
    big = np.array([448.0, 449.0, 464.0, 480.0, 1e6, -500.0], np.float32)
    assert list(orc.round_e4m3(big)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_e2m1_rounding_matches_bruteforce_nearest():
    """orc.round_e2m1 against a direct search over the eight magnitudes (nearest value, ties
    to the even code, saturating at 6) on a dense grid including every midpoint."""
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    grid = np.concatenate([np.arange(0, 8.0, 1 / 64), (mags[:-1] + mags[1:]) / 2, [6.0, 7.0, 1e3]])
    x = np.concatenate([grid, -grid]).astype(np.float32)
    want = []
    for v in x.astype(np.float64):
        a = abs(v)
        d = np.abs(mags - a)
        best = np.flatnonzero(d == d.min())
        code = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        want.append(code | (8 if np.signbit(v) else 0))
    assert np.array_equal(orc.round_e2m1(x), np.array(want, np.uint8))


def test_nvfp4_block_quantisation_worked_example():
    """A block whose absmax is 6 has scale 1 (E4M3 0x38) and its codes are the E2M1 roundings
    of the values themselves; doubling every value doubles the scale and keeps the codes; a
    zero block gets scale 0 and zero codes."""
    vals = np.array([6, -6, 0.25, 0.75, 1.25, 2.5, 5, -3, 0.5, 1, 1.5, 2, 3, 4, -0.5, 0],
                    np.float32)
    bits = synth.f32_to_bf16_bits(vals)
    codes, scales = orc.quantize_nvfp4(bits[None, :])
    assert scales[0, 0] == 0x38
    nib = np.stack([codes[0] & 0xF, codes[0] >> 4], 1).reshape(-1)
    assert np.array_equal(nib, orc.round_e2m1(vals))
    codes2, scales2 = orc.quantize_nvfp4(synth.f32_to_bf16_bits(vals * 2)[None, :])
    assert orc.lib().orc_decode_e4m3(int(scales2[0, 0])) == 2.0 and np.array_equal(codes2, codes)
    codes0, scales0 = orc.quantize_nvfp4(synth.f32_to_bf16_bits(np.zeros(16, np.float32))[None, :])
    assert scales0[0, 0] == 0 and not codes0.any()


def test_nvfp4_quantisation_error_bound_and_decode_roundtrip():
    """On random blocks: the scale is E4M3(absmax/6); every decoded element is within half an
    E2M1 step of x (at the block's scale), or clipped at 6 x scale; decoding then
    re-quantising reproduces the codes when the block keeps its scale."""
    rng = np.random.default_rng(43)
    x = (rng.standard_normal((300, 16)) * np.exp(rng.uniform(-6, 6, (300, 1)))).astype(np.float32)
    bits = synth.f32_to_bf16_bits(x)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    codes, scales = orc.quantize_nvfp4(bits)
    amax = np.abs(xb).max(1)
    assert np.array_equal(scales[:, 0], orc.round_e4m3((amax / np.float32(6)).astype(np.float32)))
    t = orc.Tensor(codes, "nvfp4", scales=scales)
    dec = orc.decode(t).reshape(300, 16)
    sv = np.array([orc.lib().orc_decode_e4m3(int(s)) for s in scales[:, 0]])
    # E2M1 spacing at |x|/s: 0.5 below 2, 1 up to 4, 2 up to 6
    with np.errstate(divide="ignore"):  # a block whose scale rounds to 0 has zero codes
        q = np.abs(xb) / sv[:, None]
    half_step = np.where(q < 2, 0.25, np.where(q < 4, 0.5, 1.0)) * sv[:, None]
    clipped = q > 6
    assert np.all((np.abs(dec - xb) <= half_step + 1e-12) | clipped)
    assert np.all(np.abs(dec[clipped]) == 6 * np.repeat(sv[:, None], 16, 1)[clipped])


def test_kv_append_places_tokens_through_page_table():
    """BF16 append: decoding the cache at (page_table[b][t/P], g, t%P) gives back every new
    token's row; every other slot keeps its previous bits.  NVFP4 append: the slot holds the
    block quantisation of the row and nothing else changes."""
    w = synth.workload("custom", seed=44, q_lens=[130, 5, 256], ctx_lens=[100, 383, 0],
                       num_q_heads=4, num_kv_heads=2, head_dim=64, top_k=2)
    pb = oracle_problem(w)
    rng = np.random.default_rng(45)
    T, G, D, P = w.num_tokens, w.num_kv_heads, w.head_dim, 128
    new = synth.f32_to_bf16_bits(rng.standard_normal((T, G, D)).astype(np.float32))
    cache = synth.f32_to_bf16_bits(rng.standard_normal((w.num_phys_pages, G, P, D)).astype(np.float32))
    before = cache.copy()
    orc.kv_append(pb, "bf16", new, cache)
    written = np.zeros((w.num_phys_pages, G, P), bool)
    tk = 0
    for b, (ql, cl) in enumerate(zip(w.q_lens, w.ctx_lens)):
        for i in range(ql):
            t = cl + i
            phys = w.page_table[b, t // P]
            assert np.array_equal(cache[phys, :, t % P], new[tk])
            written[phys, :, t % P] = True
            tk += 1
    assert np.array_equal(cache[~written], before[~written])
    codes = np.zeros((w.num_phys_pages, G, P, D // 2), np.uint8)
    scl = np.zeros((w.num_phys_pages, G, P, D // 16), np.uint8)
    orc.kv_append(pb, "nvfp4", new, codes, scl)
    qc, qs = orc.quantize_nvfp4(new)
    tk = 0
    for b, (ql, cl) in enumerate(zip(w.q_lens, w.ctx_lens)):
        for i in range(ql):
            t = cl + i
            phys = w.page_table[b, t // P]
            assert np.array_equal(codes[phys, :, t % P], qc[tk])
            assert np.array_equal(scl[phys, :, t % P], qs[tk])
            tk += 1
    assert not codes[~written].any() and not scl[~written].any()


def test_nvfp4_e4m3_rounded_decode_is_nearest_e4m3_of_the_product():
    """The 'nvfp4_e4m3' decode (the pages' QMUL4 dequant) gives, for every one of the 16 x 127
    (code, scale) pairs, torch's float8_e4m3fn rounding of the exact product, and +-448 where
    the product lies beyond the E4M3 range (saturating conversion)."""
    scale_codes = np.arange(0, 0x7F, dtype=np.uint8)
    nibs = np.arange(16, dtype=np.uint8)
    codes = np.repeat((nibs[0::2] | (nibs[1::2] << 4))[None, :], len(scale_codes), 0).reshape(-1)
    scales = np.repeat(scale_codes, 1)  # one scale per 16-element block = per row of 8 bytes
    exact = orc.decode(orc.Tensor(codes, "nvfp4", scales=scales))
    rounded = orc.decode(orc.Tensor(codes, "nvfp4_e4m3", scales=scales))
    inr = np.abs(exact) <= 448  # torch's cast gives NaN beyond the E4M3 range; ours saturates
    want = torch.from_numpy(exact[inr].astype(np.float32)).to(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(rounded[inr], want.astype(np.float64))
    assert np.all(rounded[~inr] == np.sign(exact[~inr]) * 448.0) and (~inr).any()
    assert np.any(rounded[inr] != exact[inr])  # some products need rounding (6 significant bits)
