"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test fixes the oracle to something the pages or plain mathematics decide:
hand-derived closed forms (tests/golden), pure-Python brute force on tiny
inputs, invariants of the paged layout (paging is pure indirection, NHD and
HND hold the same values), special cases with a closed form, and an
independent library routine (torch's scaled_dot_product_attention in float64)
on a densely gathered copy. The mutation tests at the bottom plant plausible
mistakes in the oracle and check that some pin catches each one.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as OA
from paged_kv_attention_27_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def _bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def brute_force(q, k, v, scale, vis):
    """Two-pass softmax in pure Python: materialise every score, take the max,
    exponentiate, normalise, weight the V rows."""
    n, T, dv = len(q), len(k), len(v[0]) if len(v) else 0
    outs, lses = [], []
    for r in range(n):
        scores = []
        for t in range(T):
            if vis[r][t]:
                scores.append((t, scale * sum(a * b for a, b in zip(q[r], k[t]))))
        if not scores:
            outs.append([0.0] * dv)
            lses.append(-math.inf)
            continue
        m = max(s for _, s in scores)
        e = [(t, math.exp(s - m)) for t, s in scores]
        z = sum(x for _, x in e)
        o = [0.0] * dv
        for t, x in e:
            for j in range(dv):
                o[j] += (x / z) * v[t][j]
        outs.append(o)
        lses.append(m + math.log(z))
    return np.array(outs), np.array(lses)


# --------------------------------------------------------------------------
# reading inputs
# --------------------------------------------------------------------------

def test_bf16_bit_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3E00, 0x7F80, 0xFF80, 0x0001, 0x4049, 0x0000, 0x8000],
                    dtype=np.uint16)
    want = [1.0, -2.0, 0.125, math.inf, -math.inf, 2.0 ** -133, 3.140625, 0.0, -0.0]
    got = oracle.bf16_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w
    assert math.copysign(1.0, got[-1]) == -1.0


def test_fp16_bit_patterns():
    """Hand-decoded IEEE binary16 values, then every pattern against numpy's
    own float16 type (an independent decoder)."""
    bits = np.array([0x3C00, 0xC000, 0x3555, 0x7BFF, 0x0001, 0x03FF, 0x0400, 0x7C00, 0xFC00,
                     0x0000, 0x8000], dtype=np.uint16)
    want = [1.0, -2.0, 0.333251953125, 65504.0, 2.0 ** -24, 1023 * 2.0 ** -24, 2.0 ** -14,
            math.inf, -math.inf, 0.0, -0.0]
    got = oracle.f16_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w
    assert math.copysign(1.0, got[-1]) == -1.0
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    mine = oracle.f16_to_f64(allbits)
    same = (mine == ref) | (np.isnan(mine) & np.isnan(ref))
    assert same.all()


def test_fp16_inputs_match_torch_sdpa_float64():
    """A prefill batch in fp16 against torch SDPA in float64 on tensors that
    torch decodes from the same bits itself."""
    torch = pytest.importorskip("torch")
    b = synth.make_batch("fp16", [40, 130], [40, 33], 8, 2, 32, 16, synth.NHD, None, True, 23,
                         dtype="fp16")
    out, lse = _run(b)
    g = b.num_qo_heads // b.num_kv_heads
    for r in range(b.batch):
        kv, qo = int(b.kv_lens[r]), int(b.qo_lens[r])
        pages = b.page_indices[int(b.page_indptr[r]):int(b.page_indptr[r + 1])]
        to = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(
            torch.float16).to(torch.float64)
        kt = to(np.concatenate([b.k_cache[p] for p in pages], axis=0)[:kv]).transpose(0, 1)
        vt = to(np.concatenate([b.v_cache[p] for p in pages], axis=0)[:kv]).transpose(0, 1)
        qt = to(b.q[int(b.qo_indptr[r]):int(b.qo_indptr[r + 1])]).transpose(0, 1)
        kt, vt = kt.repeat_interleave(g, 0), vt.repeat_interleave(g, 0)
        mask = torch.ones(qo, kv, dtype=torch.bool).tril(kv - qo)
        so = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                              scale=b.sm_scale)
        rows = slice(int(b.qo_indptr[r]), int(b.qo_indptr[r + 1]))
        np.testing.assert_allclose(out[rows], so.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
    # the same draws rounded to bf16 give a different (but close) answer
    b16 = synth.make_batch("bf16", [40, 130], [40, 33], 8, 2, 32, 16, synth.NHD, None, True, 23)
    o16, _ = _run(b16)
    assert not np.array_equal(o16, out) and np.abs(o16 - out).max() < 0.05


def test_e4m3_bit_patterns():
    """Hand-decoded OCP FP8 E4M3 values, then all 256 patterns against
    torch's float8_e4m3fn (an independent decoder)."""
    bits = np.array([0x38, 0xB8, 0x7E, 0x01, 0x07, 0x08, 0x3C, 0x7F, 0xFF, 0x00, 0x80], np.uint8)
    want = [1.0, -1.0, 448.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.5, math.nan, math.nan,
            0.0, -0.0]
    got = oracle.e4m3_to_f64(bits)
    for g, w in zip(got, want):
        assert (math.isnan(g) and math.isnan(w)) or g == w
    assert math.copysign(1.0, got[-1]) == -1.0
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    allb = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(allb).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.e4m3_to_f64(allb)
    assert ((mine == ref) | (np.isnan(mine) & np.isnan(ref))).all()


def test_kv_scales_fold_into_the_score_scale_and_the_output():
    """k_scale multiplies every score, so it is the same as multiplying
    sm_scale; v_scale multiplies the output and leaves lse unchanged."""
    b = synth.make_batch("fp8", [70, 130, 1], [1, 1, 1], 8, 2, 64, 16, synth.NHD, 0.125, False,
                         24, kv_dtype="e4m3")
    o1, l1 = _run(b)
    b.k_scale = 0.5
    o2, l2 = _run(b)
    b.k_scale, b.sm_scale = 1.0, 0.0625
    o3, l3 = _run(b)
    np.testing.assert_allclose(o2, o3, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l3, rtol=0, atol=1e-13)
    assert np.abs(o1 - o2).max() > 1e-3                     # the scale matters
    b.sm_scale, b.v_scale = 0.125, 0.25
    o4, l4 = _run(b)
    np.testing.assert_allclose(o4, 0.25 * o1, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(l4, l1)


def test_fp8_cache_matches_torch_sdpa_float64():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    b = synth.make_batch("fp8 sdpa", [45, 300], [1, 1], 8, 2, 32, 16, synth.HND, None, False, 25,
                         kv_dtype="e4m3", kv_scale=1 / 16)
    assert b.k_cache.dtype == np.uint8 and b.k_scale == 1 / 16
    out, lse = _run(b)
    g = b.num_qo_heads // b.num_kv_heads
    for r in range(b.batch):
        kv = int(b.kv_lens[r])
        pages = b.page_indices[int(b.page_indptr[r]):int(b.page_indptr[r + 1])]
        dec = lambda x: torch.from_numpy(np.ascontiguousarray(x)).view(torch.float8_e4m3fn).to(
            torch.float64)
        kt = dec(np.concatenate([b.k_cache[p] for p in pages], axis=1)[:, :kv]) * b.k_scale
        vt = dec(np.concatenate([b.v_cache[p] for p in pages], axis=1)[:, :kv]) * b.v_scale
        qt = torch.from_numpy(b.q[r:r + 1].view(np.int16)).view(torch.bfloat16).to(
            torch.float64).transpose(0, 1)                               # [Hq, 1, d]
        kt, vt = kt.repeat_interleave(g, 0), vt.repeat_interleave(g, 0)
        so = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=b.sm_scale)
        np.testing.assert_allclose(out[r], so[:, 0].numpy(), rtol=0, atol=1e-12)


def test_fp8_cache_with_per_head_scales_matches_torch_sdpa_float64():
    """Each kv head with its own K and V scale (the cache holds K / (k_scale
    s_h) and V / (v_scale t_h)): torch decodes the codes, applies the scale
    of each head and computes attention in float64."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    ks = [0.5, 2.0, 0.125]
    vs = [4.0, 0.25, 1.0]
    b = synth.make_batch("fp8 per-head", [45, 300, 7], [1, 1, 1], 6, 3, 32, 16, synth.NHD, None,
                         False, 26, kv_dtype="e4m3", kv_scale=1 / 16, head_scales=(ks, vs))
    np.testing.assert_array_equal(b.k_head_scale, np.float32(ks))
    out, lse = _run(b)
    g = b.num_qo_heads // b.num_kv_heads
    dec = lambda x: torch.from_numpy(np.ascontiguousarray(x)).view(torch.float8_e4m3fn).to(
        torch.float64)
    for r in range(b.batch):
        kv = int(b.kv_lens[r])
        pages = b.page_indices[int(b.page_indptr[r]):int(b.page_indptr[r + 1])]
        kt = dec(np.concatenate([b.k_cache[p] for p in pages], axis=0)[:kv])   # [kv, Hkv, d]
        vt = dec(np.concatenate([b.v_cache[p] for p in pages], axis=0)[:kv])
        kt = (kt * torch.tensor(ks, dtype=torch.float64)[None, :, None] / 16).transpose(0, 1)
        vt = (vt * torch.tensor(vs, dtype=torch.float64)[None, :, None] / 16).transpose(0, 1)
        qt = torch.from_numpy(b.q[r:r + 1].view(np.int16)).view(torch.bfloat16).to(
            torch.float64).transpose(0, 1)                               # [Hq, 1, d]
        kt, vt = kt.repeat_interleave(g, 0), vt.repeat_interleave(g, 0)
        so = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=b.sm_scale)
        np.testing.assert_allclose(out[r], so[:, 0].numpy(), rtol=0, atol=1e-12)
    # the scales matter: one number for every head gives another result
    b1 = synth.PagedBatch(**{**b.__dict__, "k_head_scale": None, "v_head_scale": None})
    assert np.abs(_run(b1)[0] - out).max() > 1e-2
    # the attended values are close to the unscaled normal draws
    assert 0.3 < np.abs(dec(b.k_cache).numpy()[:, :, 1] * ks[1] / 16).mean() < 1.5


def test_kv_lengths_of_tiny_config():
    b = synth.tiny_decode()
    # pages {1,2,4,7}, last page lengths {1,1,16,4} for KV lengths {1,17,64,100}
    assert list(np.diff(b.page_indptr)) == [1, 2, 4, 7]
    assert list(b.last_page_len) == [1, 1, 16, 4]
    assert list(oracle.kv_lengths(b.page_indptr, b.last_page_len, 16)) == [1, 17, 64, 100]
    # a request with no pages holds no tokens, whatever last_page_len says
    assert list(oracle.kv_lengths([0, 0, 3], [5, 2], 16)) == [0, 34]


@pytest.mark.parametrize("layout", [synth.NHD, synth.HND])
def test_gather_inverts_page_placement(layout):
    """Build a cache by placing logical page j of a request on physical page
    perm[j]; gathering through the page table must give back the logical rows."""
    rng = np.random.default_rng(7)
    P, Hkv, d, T = 4, 3, 5, 23
    npages = (T + P - 1) // P
    perm = rng.permutation(npages + 2)[:npages]          # some physical pages unused
    logical = rng.integers(0, 2 ** 15, size=(Hkv, npages * P, d)).astype(np.uint16)
    shape = (npages + 2, P, Hkv, d) if layout == synth.NHD else (npages + 2, Hkv, P, d)
    cache = np.zeros(shape, dtype=np.uint16)
    for j in range(npages):
        for s in range(P):
            for h in range(Hkv):
                if layout == synth.NHD:
                    cache[perm[j], s, h] = logical[h, j * P + s]
                else:
                    cache[perm[j], h, s] = logical[h, j * P + s]
    page_indptr = np.array([0, npages])
    for h in range(Hkv):
        got = oracle.gather_kv(cache, layout, page_indptr, perm, 0, h, T, P)
        np.testing.assert_array_equal(got, oracle.bf16_to_f64(logical[h, :T]))


# --------------------------------------------------------------------------
# the definition against hand-derived values and brute force
# --------------------------------------------------------------------------

def test_closed_form_golden_cases():
    g = json.load(open(GOLDEN))
    for case in g["cases"]:
        q = np.array([case["q"]])
        k = np.array(case["k"])
        v = np.array(case["v"])
        vis = np.ones((1, len(k)), dtype=bool)
        for fn in (lambda: oracle.softmax_attention(q, k, v, case["scale"], vis),
                   lambda: oracle.online_softmax_attention(q, k, v, case["scale"], vis, 1),
                   lambda: oracle.masked_attention(q, k, v, case["scale"], np.zeros((1, len(k))))):
            o, lse = fn()
            np.testing.assert_allclose(o[0], case["o"], rtol=0, atol=1e-14)
            assert abs(lse[0] - case["lse"]) < 1e-14
    ds = g["default_scale"]
    for d in (64, 128, 256):
        assert synth.make_batch("x", [1], [1], 1, 1, d, 16, synth.NHD, None, False, 0).sm_scale \
            == pytest.approx(ds[f"head_dim_{d}"], rel=1e-15)


@pytest.mark.parametrize("seed", range(6))
def test_definition_and_online_form_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    n, T, d = rng.integers(1, 5), rng.integers(1, 12), rng.integers(1, 6)
    q, k, v = rng.normal(size=(n, d)), rng.normal(size=(T, d)), rng.normal(size=(T, d))
    scale = float(rng.uniform(0.1, 2.0))
    vis = rng.random((n, T)) < 0.7
    vis[0, :] = False                       # one empty row
    bo, bl = brute_force(q.tolist(), k.tolist(), v.tolist(), scale, vis.tolist())
    o, l = oracle.softmax_attention(q, k, v, scale, vis)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, bl, rtol=0, atol=1e-12)
    for chunk in (1, 2, 3, 7, 100):
        oo, ol = oracle.online_softmax_attention(q, k, v, scale, vis, chunk)
        np.testing.assert_allclose(oo, bo, rtol=0, atol=1e-12)
        np.testing.assert_allclose(ol, bl, rtol=0, atol=1e-12)


def test_single_key_returns_its_value_row():
    b = synth.make_batch("one", [1], [1], 4, 2, 32, 16, synth.NHD, 0.3, False, 11)
    out, lse = oracle.batch_decode(b.q, b.k_cache, b.v_cache, b.layout, b.page_indptr,
                                   b.page_indices, b.last_page_len, 4, 2, 16, 0.3)
    p = b.page_indices[0]
    for h in range(4):
        kh = h // 2
        np.testing.assert_array_equal(out[0, h], oracle.bf16_to_f64(b.v_cache[p, 0, kh]))
        s0 = 0.3 * float(oracle.bf16_to_f64(b.q[0, h]) @ oracle.bf16_to_f64(b.k_cache[p, 0, kh]))
        assert lse[0, h] == pytest.approx(s0, abs=1e-13)


def test_constant_values_give_that_constant():
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=(3, 8)), rng.normal(size=(40, 8)) * 3
    v = np.tile(np.array([0.5, -1.25, 2.0, 0.0, 7.0, 1.0, -3.0, 0.125]), (40, 1))
    o, _ = oracle.softmax_attention(q, k, v, 0.7, np.ones((3, 40), bool))
    np.testing.assert_allclose(o, v[:3], rtol=0, atol=1e-13)


def test_zero_keys_or_zero_scale_give_mean_and_log_count():
    rng = np.random.default_rng(4)
    q, k, v = rng.normal(size=(2, 6)), rng.normal(size=(9, 6)), rng.normal(size=(9, 6))
    vis = np.ones((2, 9), bool)
    vis[1, 5:] = False
    for kk, sc in ((np.zeros_like(k), 0.9), (k, 0.0)):
        o, l = oracle.softmax_attention(q, kk, v, sc, vis)
        np.testing.assert_allclose(o[0], v.mean(axis=0), atol=1e-14)
        np.testing.assert_allclose(o[1], v[:5].mean(axis=0), atol=1e-14)
        np.testing.assert_allclose(l, [math.log(9), math.log(5)], atol=1e-14)


def test_one_dominant_score_is_overflow_safe():
    """Scores far beyond exp's float64 range (the pages warn about overflow
    under fast exp, FlashAttention-3 page section 4) still give that row."""
    d = 4
    q = np.array([[1.0, 0, 0, 0]])
    k = np.array([[800.0, 0, 0, 0], [750.0, 0, 0, 0], [0.0, 0, 0, 0]])
    v = np.array([[1.0, 2, 3, 4], [5.0, 6, 7, 8], [9.0, 9, 9, 9]])
    o, l = oracle.softmax_attention(q, k, v, 1.0, np.ones((1, 3), bool))
    assert np.all(np.isfinite(o))
    np.testing.assert_allclose(o[0], v[0], atol=1e-20)
    assert l[0] == pytest.approx(800.0 + math.log1p(math.exp(-50.0)), abs=1e-12)
    # boosted by +50 relative to a plain batch: o equals that V row to ~e^-50
    rng = np.random.default_rng(5)
    q = rng.normal(size=(1, d)) * 0.01
    kk = rng.normal(size=(6, d)) * 0.01
    kk[2] = q[0] / np.dot(q[0], q[0]) * 50.0
    vv = rng.normal(size=(6, d))
    o, _ = oracle.softmax_attention(q, kk, vv, 1.0, np.ones((1, 6), bool))
    np.testing.assert_allclose(o[0], vv[2], atol=1e-19)


# --------------------------------------------------------------------------
# invariants of the paged layout
# --------------------------------------------------------------------------

def _run(b, requests=None):
    return oracle.batch_attention(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.layout, b.page_indptr,
                                  b.page_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                                  b.page_size, b.sm_scale, b.causal, requests=requests,
                                  window_left=b.window_left, dtype=b.dtype,
                                  kv_dtype=b.cache_dtype, k_scale=b.k_scales, v_scale=b.v_scales)


def test_permuting_physical_pages_changes_nothing():
    b = synth.make_batch("perm", [37, 5, 64, 0, 90], [3, 1, 7, 0, 90], 4, 2, 16, 16, synth.NHD,
                         None, True, 12, extra_pages=3)
    out, lse = _run(b)
    rng = np.random.default_rng(0)
    sigma = rng.permutation(b.num_pages)               # new physical id of old page p
    k2 = np.empty_like(b.k_cache)
    v2 = np.empty_like(b.v_cache)
    k2[sigma] = b.k_cache
    v2[sigma] = b.v_cache
    b2 = synth.PagedBatch(**{**b.__dict__, "k_cache": k2, "v_cache": v2,
                             "page_indices": sigma[b.page_indices].astype(np.int32)})
    out2, lse2 = _run(b2)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_nhd_equals_hnd():
    b = synth.make_batch("nhd", [37, 5, 64, 90], [3, 1, 7, 90], 8, 2, 16, 16, synth.NHD,
                         None, True, 13)
    out, lse = _run(b)
    b2 = synth.PagedBatch(**{**b.__dict__, "layout": synth.HND,
                             "k_cache": np.ascontiguousarray(b.k_cache.transpose(0, 2, 1, 3)),
                             "v_cache": np.ascontiguousarray(b.v_cache.transpose(0, 2, 1, 3))})
    out2, lse2 = _run(b2)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_decode_is_prefill_with_one_row_and_gqa_is_replicated_mha():
    b = synth.make_batch("gqa", [33, 1, 70], [1, 1, 1], 8, 2, 16, 16, synth.HND, None, False, 14)
    d_out, d_lse = oracle.batch_decode(b.q, b.k_cache, b.v_cache, b.layout, b.page_indptr,
                                       b.page_indices, b.last_page_len, 8, 2, 16, b.sm_scale)
    for causal in (False, True):
        p_out, p_lse = oracle.batch_attention(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.layout,
                                              b.page_indptr, b.page_indices, b.last_page_len,
                                              8, 2, 16, b.sm_scale, causal)
        np.testing.assert_array_equal(d_out, p_out)
        np.testing.assert_array_equal(d_lse, p_lse)
    # replicate each kv head 4 times -> MHA with 8 kv heads
    kr = np.repeat(b.k_cache, 4, axis=1)
    vr = np.repeat(b.v_cache, 4, axis=1)
    m_out, m_lse = oracle.batch_decode(b.q, kr, vr, b.layout, b.page_indptr, b.page_indices,
                                       b.last_page_len, 8, 8, 16, b.sm_scale)
    np.testing.assert_array_equal(d_out, m_out)
    np.testing.assert_array_equal(d_lse, m_lse)


# --------------------------------------------------------------------------
# split-KV + merge, causal mask
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(5))
def test_split_kv_merge_equals_unsplit(seed):
    rng = np.random.default_rng(100 + seed)
    n, T, d = 4, int(rng.integers(2, 80)), 8
    q, k, v = rng.normal(size=(n, d)), rng.normal(size=(T, d)), rng.normal(size=(T, d))
    vis = oracle.visible_keys(n, T, True) if T >= n else np.ones((n, T), bool)
    o, l = oracle.softmax_attention(q, k, v, 0.4, vis)
    cuts = sorted(set(rng.integers(0, T + 1, size=int(rng.integers(1, 6))).tolist()) | {0, T})
    if seed == 0:
        cuts = [0, 0, T // 2, T // 2, T]      # empty parts merge as nothing
    po, pl = oracle.split_kv_states(q, k, v, 0.4, vis, cuts)
    mo, ml = oracle.merge_states(po, pl)
    np.testing.assert_allclose(mo, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, l, rtol=0, atol=1e-12)


def test_merge_states_closed_forms():
    o1 = np.array([[1.0, 2.0]])
    o2 = np.array([[3.0, -2.0]])
    # equal lse: plain average, lse + ln 2
    mo, ml = oracle.merge_states(np.stack([o1, o2]), np.array([[0.5], [0.5]]))
    np.testing.assert_allclose(mo, [[2.0, 0.0]], atol=1e-15)
    np.testing.assert_allclose(ml, [0.5 + math.log(2)], atol=1e-15)
    # lse apart by ln 3: weights 3/4 and 1/4
    mo, ml = oracle.merge_states(np.stack([o1, o2]), np.array([[math.log(3)], [0.0]]))
    np.testing.assert_allclose(mo, [[1.5, 1.0]], atol=1e-15)
    np.testing.assert_allclose(ml, [math.log(4)], atol=1e-15)
    # an empty part weighs nothing; all empty gives 0 / -inf
    mo, ml = oracle.merge_states(np.stack([o1, o2]), np.array([[-np.inf], [0.25]]))
    np.testing.assert_array_equal(mo, o2)
    assert ml[0] == 0.25
    mo, ml = oracle.merge_states(np.stack([o1, o2]), np.array([[-np.inf], [-np.inf]]))
    np.testing.assert_array_equal(mo, [[0.0, 0.0]])
    assert np.isneginf(ml[0])


@pytest.mark.parametrize("qo,kv", [(1, 1), (5, 5), (3, 11), (8, 30), (16, 16)])
def test_causal_matches_explicit_mask(qo, kv):
    rng = np.random.default_rng(qo * 100 + kv)
    q, k, v = rng.normal(size=(qo, 8)), rng.normal(size=(kv, 8)), rng.normal(size=(kv, 8))
    o, l = oracle.softmax_attention(q, k, v, 0.3, oracle.visible_keys(qo, kv, True))
    mo, ml = oracle.masked_attention(q, k, v, 0.3, oracle.causal_mask(qo, kv))
    np.testing.assert_allclose(o, mo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ml, rtol=0, atol=1e-12)
    # the last row always sees every key; the first sees kv-qo+1 of them
    assert oracle.visible_keys(qo, kv, True)[-1].all()
    assert oracle.visible_keys(qo, kv, True)[0].sum() == kv - qo + 1


# --------------------------------------------------------------------------
# the left attention window (window_size of the FlashAttention-3 page's
# varlen call, section 2): closed forms and reductions
# --------------------------------------------------------------------------

@pytest.mark.parametrize("qo,kv", [(1, 1), (4, 9), (12, 12), (5, 40)])
def test_window_zero_sees_only_its_own_position(qo, kv):
    """Causal with window_left = 0: row i sees exactly key kv-qo+i, so its
    output is that V row and its lse that one scaled score."""
    rng = np.random.default_rng(qo * 7 + kv)
    q, k, v = rng.normal(size=(qo, 8)), rng.normal(size=(kv, 8)), rng.normal(size=(kv, 8))
    o, l = oracle.softmax_attention(q, k, v, 0.7, oracle.visible_keys(qo, kv, True, 0))
    for i in range(qo):
        t = kv - qo + i
        np.testing.assert_allclose(o[i], v[t], rtol=0, atol=1e-14)
        assert abs(l[i] - 0.7 * float(q[i] @ k[t])) < 1e-12


@pytest.mark.parametrize("w", [0, 1, 15, 16, 17, 63, 99, 100, 5000])
def test_windowed_decode_is_attention_over_the_last_keys(w):
    """Decode with window_left = w equals plain (unwindowed) attention over
    the last min(w+1, kv_len) keys, sliced out of a dense copy made by
    walking the pages in order (no page arithmetic shared with the oracle)."""
    b = synth.tiny_decode()
    b.window_left = w
    out, lse = _run(b)
    g = b.num_qo_heads // b.num_kv_heads
    for r in range(b.batch):
        kv = int(b.kv_lens[r])
        pages = b.page_indices[int(b.page_indptr[r]):int(b.page_indptr[r + 1])]
        dk = np.concatenate([b.k_cache[p] for p in pages], axis=0)[:kv]   # NHD: [t, Hkv, d]
        dv = np.concatenate([b.v_cache[p] for p in pages], axis=0)[:kv]
        keep = min(w + 1, kv)
        for h in range(b.num_qo_heads):
            kh = h // g
            k = oracle.bf16_to_f64(dk[kv - keep:, kh])
            v = oracle.bf16_to_f64(dv[kv - keep:, kh])
            q = oracle.bf16_to_f64(b.q[r, h])[None]
            ro, rl = brute_force(q.tolist(), k.tolist(), v.tolist(), b.sm_scale,
                                 [[True] * keep])
            np.testing.assert_allclose(out[r, h], ro[0], rtol=0, atol=1e-12)
            assert abs(lse[r, h] - rl[0]) < 1e-12


def test_window_wider_than_the_context_changes_nothing():
    b = synth.make_batch("w", [40, 130, 17], [40, 33, 1], 8, 2, 32, 16, synth.NHD, None, True, 31)
    o0, l0 = _run(b)
    b.window_left = 129
    o1, l1 = _run(b)
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("w", [0, 3, 31, 32])
def test_window_matches_torch_band_mask(causal, w):
    """torch SDPA in float64 with a band mask built by torch.tril/triu
    diagonals (an independent construction of the same visibility)."""
    torch = pytest.importorskip("torch")
    b = synth.make_batch("band", [70, 45], [20, 45], 4, 2, 32, 16, synth.NHD, None, causal, 32,
                         window_left=w)
    out, lse = _run(b)
    g = b.num_qo_heads // b.num_kv_heads
    for r in range(b.batch):
        kv, qo = int(b.kv_lens[r]), int(b.qo_lens[r])
        pages = b.page_indices[int(b.page_indptr[r]):int(b.page_indptr[r + 1])]
        to = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(
            torch.bfloat16).to(torch.float64)
        dk = to(np.concatenate([b.k_cache[p] for p in pages], axis=0)[:kv]).transpose(0, 1)
        dv = to(np.concatenate([b.v_cache[p] for p in pages], axis=0)[:kv]).transpose(0, 1)
        qt = to(b.q[int(b.qo_indptr[r]):int(b.qo_indptr[r + 1])]).transpose(0, 1)
        ones = torch.ones(qo, kv, dtype=torch.bool)
        # diagonal kv-qo of an (qo x kv) matrix is the key aligned with each row
        mask = ones.tril(kv - qo) if causal else ones.clone()
        mask &= ones.triu(kv - qo - w)
        kt, vt = dk.repeat_interleave(g, 0), dv.repeat_interleave(g, 0)
        so = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                              scale=b.sm_scale)
        sc = (qt @ kt.transpose(-1, -2)) * b.sm_scale
        sl = torch.logsumexp(sc.masked_fill(~mask, -math.inf), dim=-1)
        rows = slice(int(b.qo_indptr[r]), int(b.qo_indptr[r + 1]))
        np.testing.assert_allclose(out[rows], so.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[rows], sl.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# an independent library routine on a densely gathered copy
# --------------------------------------------------------------------------

def _sdpa_dense(b):
    torch = pytest.importorskip("torch")
    g = b.num_qo_heads // b.num_kv_heads
    outs, lses = [], []
    for r in range(b.batch):
        kv, qo = int(b.kv_lens[r]), int(b.qo_lens[r])
        lo = int(b.page_indptr[r])
        # dense [Hkv, kv, d] by walking logical pages in order (no page arithmetic shared)
        pages = b.page_indices[lo:int(b.page_indptr[r + 1])]
        if b.layout == synth.NHD:
            dense_k = np.concatenate([b.k_cache[p] for p in pages], axis=0)[:kv].transpose(1, 0, 2)
            dense_v = np.concatenate([b.v_cache[p] for p in pages], axis=0)[:kv].transpose(1, 0, 2)
        else:
            dense_k = np.concatenate([b.k_cache[p] for p in pages], axis=1)[:, :kv]
            dense_v = np.concatenate([b.v_cache[p] for p in pages], axis=1)[:, :kv]
        to = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(torch.float64)
        qt = to(b.q[int(b.qo_indptr[r]):int(b.qo_indptr[r + 1])]).transpose(0, 1)   # [Hq, qo, d]
        kt = to(np.ascontiguousarray(dense_k)).repeat_interleave(g, dim=0)
        vt = to(np.ascontiguousarray(dense_v)).repeat_interleave(g, dim=0)
        mask = None
        if b.causal:
            i = torch.arange(qo)[:, None]
            t = torch.arange(kv)[None, :]
            mask = t <= kv - qo + i
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                             scale=b.sm_scale)
        s = (qt @ kt.transpose(-1, -2)) * b.sm_scale
        if mask is not None:
            s = s.masked_fill(~mask, -math.inf)
        lses.append(torch.logsumexp(s, dim=-1).transpose(0, 1).numpy())
        outs.append(o.transpose(0, 1).numpy())
    return np.concatenate(outs), np.concatenate(lses)


@pytest.mark.parametrize("which", ["tiny", "7b_sample", "prefill_small", "gqa_hnd"])
def test_oracle_matches_torch_sdpa_float64(which):
    if which == "tiny":
        b = synth.tiny_decode()
    elif which == "7b_sample":
        b = synth.sub_batch(synth.llama7b_decode(batch=6), range(3))
    elif which == "prefill_small":
        b = synth.make_batch("pf", [40, 130, 17], [40, 33, 17], 8, 2, 32, 16, synth.NHD, None,
                             True, 21)
    else:
        b = synth.make_batch("gqa", [300, 70], [1, 1], 16, 2, 64, 16, synth.HND, None, False, 22)
    out, lse = _run(b)
    so, sl = _sdpa_dense(b)
    np.testing.assert_allclose(out, so, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, sl, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# mutation tests: plant a plausible mistake in the oracle, on the CPU, and
# check that one of the pins above notices
# --------------------------------------------------------------------------

def _raises(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught(monkeypatch):
    # 1. page and slot swapped in the gather
    def bad_gather(cache_bits, layout, page_indptr, page_indices, b, kv_head, kv_len, P):
        t = np.arange(kv_len)
        pages = np.asarray(page_indices)[int(page_indptr[b]) + t % P % max(1, len(page_indices))]
        rows = cache_bits[pages, (t // P) % P, kv_head] if layout == OA.NHD else \
            cache_bits[pages, kv_head, (t // P) % P]
        return OA.bf16_to_f64(rows)
    with monkeypatch.context() as m:
        m.setattr(OA, "gather_kv", bad_gather)
        m.setattr(oracle, "gather_kv", bad_gather)
        assert _raises(lambda: test_gather_inverts_page_placement(synth.NHD))

    # 2. causal bound off by one
    def bad_visible(qo_len, kv_len, causal):
        i = np.arange(qo_len)[:, None]
        t = np.arange(kv_len)[None, :]
        return (t < kv_len - qo_len + i) if causal else np.ones((qo_len, kv_len), bool)
    with monkeypatch.context() as m:
        m.setattr(oracle, "visible_keys", bad_visible)
        assert _raises(lambda: test_causal_matches_explicit_mask(8, 30))

    # 3. the scale dropped from the scores
    real = OA.softmax_attention

    def no_scale(q, k, v, sm_scale, visible):
        return real(q, k, v, 1.0, visible)
    with monkeypatch.context() as m:
        m.setattr(oracle, "softmax_attention", no_scale)
        assert _raises(lambda: test_definition_and_online_form_match_brute_force(1))

    # 4. lse returned without the running max
    def lse_no_max(q, k, v, sm_scale, visible):
        o, l = real(q, k, v, sm_scale, visible)
        s = sm_scale * (q @ k.T)
        return o, np.array([l[r] - np.max(s[r, visible[r]]) if visible[r].any() else l[r]
                            for r in range(len(l))])
    with monkeypatch.context() as m:
        m.setattr(oracle, "softmax_attention", lse_no_max)
        assert _raises(test_closed_form_golden_cases)

    # 5. merge weights not normalised
    def bad_merge(o_parts, lse_parts):
        M = lse_parts.max(axis=0)
        w = np.exp(lse_parts - M)
        return (w[..., None] * o_parts).sum(axis=0), M
    with monkeypatch.context() as m:
        m.setattr(oracle, "merge_states", bad_merge)
        assert _raises(lambda: test_split_kv_merge_equals_unsplit(2))

    # 7. window bound off by one (one key too many on the left)
    real_vis = OA.visible_keys

    def wide_window(qo_len, kv_len, causal, window_left=-1):
        return real_vis(qo_len, kv_len, causal, window_left + 1 if window_left >= 0 else -1)
    with monkeypatch.context() as m:
        m.setattr(oracle, "visible_keys", wide_window)
        m.setattr(OA, "visible_keys", wide_window)
        assert _raises(lambda: test_window_zero_sees_only_its_own_position(4, 9))
        assert _raises(lambda: test_windowed_decode_is_attention_over_the_last_keys(15))

    # 6. K and V swapped (transposed operand roles)
    def kv_swapped(q, k, v, sm_scale, visible):
        return real(q, v, k, sm_scale, visible)
    with monkeypatch.context() as m:
        m.setattr(OA, "softmax_attention", kv_swapped)
        assert _raises(lambda: test_oracle_matches_torch_sdpa_float64("tiny"))
