"""GPU parity of batch decode (and merge_states) against the fp64 oracle,
through the C ABI. Same seeded inputs on both sides; bf16 outputs within
max-abs 1e-2 / mean-abs 1e-3 of the unrounded oracle, lse within 1e-3."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from paged_kv_attention_27_gb300 import binding as B  # noqa: E402
from paged_kv_attention_27_gb300 import synth  # noqa: E402

from ._gpu import compare, ensure_built, oracle_parallel, scale_v  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    B.lib()


def _dev(b, **kw):
    from paged_kv_attention_27_gb300.device import DeviceBatch
    return DeviceBatch(b, **kw)


def _oracle(b, requests=None):
    return oracle.batch_attention(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.layout, b.page_indptr,
                                  b.page_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                                  b.page_size, b.sm_scale, b.causal, requests=requests,
                                  window_left=b.window_left, dtype=b.dtype,
                                  kv_dtype=b.cache_dtype, k_scale=b.k_scales, v_scale=b.v_scales)


def _rows(b, requests):
    return np.concatenate([np.arange(b.qo_indptr[r], b.qo_indptr[r + 1]) for r in requests])


def check(b, requests=None, sms=None, what=None):
    db = _dev(b, sms=sms)
    out, lse = db.run()
    torch.cuda.synchronize()
    assert db.status() == B.FI_OK
    ref_o, ref_l = _oracle(b, requests)
    rows = None if requests is None else _rows(b, requests)
    return compare(out, lse, ref_o, ref_l, rows=rows, what=what or b.name), db


def test_tiny_decode():
    check(synth.tiny_decode())


def check_all(b):
    """The whole batch against the oracle (run over the requests in parallel)."""
    db = _dev(b)
    out, lse = db.run()
    torch.cuda.synchronize()
    assert db.status() == B.FI_OK
    ref_o, ref_l = oracle_parallel(b)
    return compare(out, lse, ref_o, ref_l, what=b.name), db


def test_llama7b_decode_full_size_every_request():
    # the benchmark's batch as the benchmark launches it: every request, every
    # split chunk and every merge of the plan
    check_all(synth.llama7b_decode())


def test_llama70b_gqa_decode_full_size_every_request():
    b = synth.llama70b_gqa_decode()
    (_, _), db = check_all(b)
    info = B.fi_plan_get_info(db.plan)
    assert info["num_split_requests"] > 0        # long requests really were split


def test_gqa_decode_d256_full_size_sampled():
    """The d = 256, 8-heads-per-kv-head benchmark batch on the tensor-core
    consumer: 16 of its 64 requests (the longest, the shortest and a spread)
    against the oracle, computed in parallel."""
    b = synth.gqa_decode_d256()
    order = np.argsort(-b.kv_lens)
    sample = sorted(set(order[:4].tolist() + order[-4:].tolist() + list(range(0, 64, 8))))
    db = _dev(b)
    out, lse = db.run()
    torch.cuda.synchronize()
    assert db.status() == B.FI_OK
    ref_o, ref_l = oracle_parallel(b, requests=sample)
    compare(out, lse, ref_o, ref_l, rows=np.array(sample), what=b.name)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("P", [16, 32])
def test_shapes(d, g, P):
    hkv = 2
    kv = [0, 1, P - 1, P, P + 1, 3 * P + 5, 700, 2049]
    b = synth.make_batch(f"shape d{d} g{g} P{P}", kv, [1] * len(kv), g * hkv, hkv, d, P,
                         synth.NHD if (d + g) % 2 == 0 else synth.HND, None, False, d * 31 + g + P)
    check(b)


@pytest.mark.parametrize("sms", [1, 3, 2000])
def test_split_kv_matches_oracle_for_any_split(sms):
    kv = [5000, 33, 1, 0, 2600, 17000]
    b = synth.make_batch("splits", kv, [1] * len(kv), 16, 4, 128, 16, synth.HND, None, False, 77)
    (_, _), db = check(b, sms=sms)
    if sms == 2000:
        assert B.fi_plan_get_info(db.plan)["num_split_requests"] >= 3


def test_nan_in_unused_tail_slots_is_never_read():
    kv = [3, 17, 45, 100, 513]
    b = synth.make_batch("nan tail", kv, [1] * len(kv), 8, 2, 128, 16, synth.NHD, None, False, 5,
                         tail_fill="nan")
    check(b)
    b = synth.make_batch("nan tail HND", kv, [1] * len(kv), 8, 8, 64, 32, synth.HND, None, False,
                         6, tail_fill="nan")
    check(b)


def test_deterministic_run_to_run():
    b = synth.make_batch("det", [9000, 300, 4100], [1, 1, 1], 32, 8, 128, 16, synth.NHD, None,
                         False, 8)
    db = _dev(b, sms=200)
    o1 = db.run()[0].clone()
    l1 = db.lse.clone()
    o2, l2 = db.run()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_layouts_agree_and_page_stride_views():
    b = synth.make_batch("nhd", [70, 300, 1], [1, 1, 1], 8, 2, 128, 16, synth.NHD, None, False, 9)
    db = _dev(b)
    o_nhd = db.run()[0].clone()
    bh = synth.PagedBatch(**{**b.__dict__, "layout": synth.HND,
                             "k_cache": np.ascontiguousarray(b.k_cache.transpose(0, 2, 1, 3)),
                             "v_cache": np.ascontiguousarray(b.v_cache.transpose(0, 2, 1, 3))})
    o_hnd = _dev(bh).run()[0]
    torch.cuda.synchronize()
    assert torch.equal(o_nhd, o_hnd)
    # K and V interleaved in one [num_pages][2][P][Hkv][d] buffer
    from paged_kv_attention_27_gb300.device import bf16_tensor
    kv = np.stack([b.k_cache, b.v_cache], axis=1)
    kvt = bf16_tensor(kv)
    page_elems = 16 * 2 * 128
    out = torch.empty_like(db.out)
    B.fi_batch_decode_paged(db.plan, db.q, kvt[:, 0], kvt[:, 1], B.FI_LAYOUT_NHD, 2 * page_elems,
                            b.num_pages, db.page_indptr, db.page_indices, db.last_page_len,
                            b.sm_scale, 1.0, 1.0, out, None, db.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out, o_nhd)


@pytest.mark.parametrize("n,S,H,d", [(5, 3, 4, 128), (2, 1, 8, 64), (3, 7, 2, 256), (1, 0, 2, 64)])
def test_merge_states_abi(n, S, H, d):
    rng = np.random.default_rng(n * 1000 + S)
    # |o| ~ 0.25: at |o| ~ 1 the bf16 rounding of the output alone would use
    # up the mean-abs budget (2^-9 relative), hiding any real error
    v = (0.25 * rng.normal(size=(n, S, H, d))).astype(np.float32)
    s = (rng.normal(size=(n, S, H)) * 4).astype(np.float32)
    if S >= 2:
        s[0, 1, :] = -np.inf             # an empty state
        s[-1, :, 0] = -np.inf            # a row with every state empty
    if S == 0:     # no states at all: the empty merge, o = 0 and lse = -inf
        ref_o, ref_l = np.zeros((n, H, d)), np.full((n, H), -np.inf)
    else:
        ref_o, ref_l = oracle.merge_states(np.moveaxis(v.astype(np.float64), 1, 0),
                                           np.moveaxis(s.astype(np.float64), 1, 0))
    vt = torch.from_numpy(v).cuda()
    st = torch.from_numpy(s).cuda()
    out = torch.empty((n, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((n, H), dtype=torch.float32, device="cuda")
    B.fi_merge_states(vt, st, n, S, H, d, B.FI_DTYPE_BF16, out, lse)
    torch.cuda.synchronize()
    compare(out, lse, ref_o, ref_l, what="merge_states")


@pytest.mark.parametrize("hq", [8, 2])
def test_bounded_wait_times_out_and_context_survives(hq):
    """4 heads per kv head: one item per CTA (tensor-core consumer); 1 head:
    the persistent launch (SIMT consumer), where the CTA that times out holds
    further items from the counter."""
    b = synth.make_batch(f"timeout hq{hq}", [4000, 100, 9000, 1], [1, 1, 1, 1], hq, 2, 128, 16,
                         synth.NHD, None, False, 10)
    db = _dev(b, sms=2)
    B.fi_debug_set_fault(1, 2_000_000)          # 2 ms bound; producer skips one load
    try:
        db.run()
        assert db.status() == B.FI_ERR_DEVICE_TIMEOUT
    finally:
        B.fi_debug_set_fault(0, 0)
    out, lse = db.run()                          # same context, normal run
    torch.cuda.synchronize()
    assert db.status() == B.FI_OK
    ref_o, ref_l = _oracle(b)
    compare(out, lse, ref_o, ref_l, what="after timeout")


@pytest.mark.parametrize("hq", [8, 2])
def test_out_of_range_page_index_is_reported_not_read(hq):
    b = synth.make_batch(f"bounds hq{hq}", [40, 40], [1, 1], hq, 2, 64, 16, synth.NHD, None,
                         False, 11)
    db = _dev(b)
    bad = b.page_indices.copy()
    bad[1] = b.num_pages + 1000
    db.page_indices.copy_(torch.from_numpy(bad))
    db.run()
    assert db.status() == B.FI_ERR_DEVICE_BOUNDS
    # request 1 is untouched by the bad index
    torch.cuda.synchronize()
    ref_o, ref_l = _oracle(b, [1])
    compare(db.out, db.lse, ref_o, ref_l, rows=np.array([1]), what="bounds, clean request")


@pytest.mark.parametrize("g,d", [(1, 128), (8, 128), (2, 256), (4, 64)])
@pytest.mark.parametrize("w", [0, 1, 15, 16, 17, 300, 5000])
def test_sliding_window_decode(g, d, w):
    """Left window: a decode row sees its last w+1 keys. Covers a window
    start inside a page, on a page boundary, inside the first chunk of a
    split request, and wider than the context."""
    hkv = 2
    kv = [1, 16, 17, 40, 700, 9000]
    b = synth.make_batch(f"window {w} g{g} d{d}", kv, [1] * len(kv), g * hkv, hkv, d, 16,
                         synth.NHD if g % 2 else synth.HND, None, False, 200 + w + g,
                         window_left=w)
    check(scale_v(b), sms=8)


@pytest.mark.parametrize("g,d", [(1, 128), (8, 128), (2, 256), (4, 64), (1, 64), (8, 256)])
def test_fp16_decode(g, d):
    """fp16 q/K/V/out through the same kernels (fp16 MMAs and conversions)."""
    hkv = 2
    kv = [1, 16, 17, 300, 2049, 9000]
    b = synth.make_batch(f"fp16 g{g} d{d}", kv, [1] * len(kv), g * hkv, hkv, d, 16,
                         synth.NHD if g % 2 else synth.HND, None, False, 500 + g + d,
                         dtype="fp16", tail_fill="nan")
    (_, _), db = check(b, sms=8)
    assert db.out.dtype == torch.float16


def test_fp16_merge_states_abi():
    rng = np.random.default_rng(5)
    n, S, H, d = 4, 3, 4, 128
    v = (0.25 * rng.normal(size=(n, S, H, d))).astype(np.float32)
    s = (rng.normal(size=(n, S, H)) * 4).astype(np.float32)
    ref_o, ref_l = oracle.merge_states(np.moveaxis(v.astype(np.float64), 1, 0),
                                       np.moveaxis(s.astype(np.float64), 1, 0))
    out = torch.empty((n, H, d), dtype=torch.float16, device="cuda")
    lse = torch.empty((n, H), dtype=torch.float32, device="cuda")
    B.fi_merge_states(torch.from_numpy(v).cuda(), torch.from_numpy(s).cuda(), n, S, H, d,
                      B.FI_DTYPE_FP16, out, lse)
    torch.cuda.synchronize()
    compare(out, lse, ref_o, ref_l, what="merge_states fp16")


# ---- FP8 (E4M3) cache --------------------------------------------------------

@pytest.mark.parametrize("g,d", [(1, 128), (8, 128), (4, 64), (2, 256), (1, 64), (8, 256)])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp8_cache_decode(g, d, dtype):
    """An E4M3 cache (stored values times 16) with the per-tensor scales
    passed to the run call; SIMT and tensor-core consumers; splits; NaN in
    the unused tail slots."""
    hkv = 2
    kv = [1, 16, 17, 300, 2049, 9000]
    b = synth.make_batch(f"fp8 g{g} d{d} {dtype}", kv, [1] * len(kv), g * hkv, hkv, d, 16,
                         synth.NHD if g % 2 else synth.HND, None, False, 700 + g + d,
                         dtype=dtype, kv_dtype="e4m3", kv_scale=1 / 16, tail_fill="nan")
    assert b.k_cache.dtype == np.uint8
    check(b, sms=8)


def test_fp8_cache_scales_and_window():
    b = synth.make_batch("fp8 scales window", [5000, 77, 1300], [1, 1, 1], 16, 2, 128, 32,
                         synth.HND, None, False, 710, kv_dtype="e4m3", kv_scale=1 / 8,
                         window_left=1000)
    b.k_scale, b.v_scale = 0.1, 0.3      # any positive scales: the kernel folds them
    check(b, sms=16)


@pytest.mark.parametrize("g,d", [(1, 128), (2, 64), (4, 256), (8, 128), (8, 64), (2, 256)])
def test_fp8_cache_per_head_scales(g, d):
    """Every kv head quantised on its own K and V scale (device arrays of
    the run call, on top of the per-tensor scales): the kernel must take
    each head's factor, not its neighbour's; splits and windows included."""
    hkv = 4
    kv = [1, 17, 300, 2049, 9000]
    ks = [0.5, 2.0, 1.0, 0.25]
    vs = [1.0, 0.5, 4.0, 2.0]
    b = synth.make_batch(f"fp8 per-head g{g} d{d}", kv, [1] * len(kv), g * hkv, hkv, d, 16,
                         synth.HND if g % 2 else synth.NHD, None, False, 720 + g + d,
                         kv_dtype="e4m3", kv_scale=1 / 16, head_scales=(ks, vs),
                         window_left=-1 if g != 8 else 2000)
    check(b, sms=8)


@pytest.mark.parametrize("g", [1, 4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp8_cache_q_dynamic_range(g, dtype):
    """With an FP8 cache at head_dim 128 and bf16 q, K Q^T runs as e4m3 MMAs
    with q as a sum of two e4m3 terms under power-of-two scales per head
    (fp16 q keeps fp16 MMAs). Elements spread over 2^-10..2^2 inside a head,
    heads scaled by 2^-12, 1 or 2^6, one head all zeros, fp16 q using all 11
    bits: the scores must still be those of the exact q."""
    hkv = 2
    kv = [1, 16, 300, 2049, 9000]
    b = synth.make_batch(f"fp8 q range g{g} {dtype}", kv, [1] * len(kv), g * hkv, hkv, 128, 16,
                         synth.NHD, None, False, 730 + g, dtype=dtype, kv_dtype="e4m3",
                         kv_scale=1 / 16)
    gen = synth.philox(731 + g)
    shape = b.q.shape
    q = gen.standard_normal(shape) * np.exp2(gen.uniform(-10, 2, shape))
    q *= np.exp2(np.array([-12.0, 0.0, 6.0])[gen.integers(0, 3, shape[:2])])[..., None]
    q[1, 0] = 0.0
    b.q = synth.to_bits(q.astype(np.float32), dtype)
    check(b, sms=8)


def test_fp8_cache_70b_full_size_every_request():
    # the bench's FP8 batch: a per-head K and V scale on each of the 8 kv heads
    b = synth.llama70b_gqa_decode(kv_dtype="e4m3")
    assert b.k_head_scale is not None and len(set(b.k_head_scale.tolist())) > 1
    check_all(b)


# ---- shared-prefix (cascade) decode ------------------------------------------

@pytest.mark.parametrize("g,d,P", [(8, 128, 16), (1, 128, 16), (4, 64, 32), (2, 256, 16)])
def test_shared_prefix_decode(g, d, P):
    """The first four requests share a 3-page prefix (one of them is exactly
    the prefix); the others decode as usual; splits forced by few SMs."""
    hkv = 2
    kv = [3 * P, 3 * P + 1, 200, 9000, 77, 1, 2500]
    b = synth.make_batch(f"cascade g{g} d{d} P{P}", kv, [1] * len(kv), g * hkv, hkv, d, P,
                         synth.HND if g % 2 else synth.NHD, None, False, 800 + g + d + P,
                         shared_prefix_requests=4, shared_prefix_tokens=3 * P)
    b.cascade = True
    (_, _), db = check(b, sms=8)
    info = B.fi_plan_get_info(db.plan)
    assert info["num_prefix_groups"] == 1 and info["num_prefix_items"] > 0


def test_shared_prefix_decode_long_prefix_many_chunks():
    b = synth.shared_prefix_decode(batch=12, prefix_tokens=20000 // 16 * 16)
    (_, _), db = check(b, requests=[0, 5, 11])
    assert B.fi_plan_get_info(db.plan)["num_prefix_items"] > 64   # the prefix was cut in chunks


def test_shared_prefix_decode_70b_batch_sampled():
    b = synth.llama70b_gqa_decode()
    b.cascade = True                                 # its first 32 requests share 1024 tokens
    check(b, requests=[0, 7, 31, 32, 100])
