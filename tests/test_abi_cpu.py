"""CPU-only checks of the C ABI: the library loads and exports every symbol
include/fi.h declares; the host planner's work lists cover every
(request, head, key) exactly once with page-aligned splits; argument
validation returns the documented status codes. No kernel is launched."""
import os
import re

import numpy as np
import pytest

from paged_kv_attention_27_gb300 import binding as B
from paged_kv_attention_27_gb300 import synth
from paged_kv_attention_27_gb300.device import plan_options

from ._gpu import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    return B.lib()


def test_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "fi.h")).read()
    declared = set(re.findall(r"^\s*(?:fi_status|const char\*)\s+(fi_\w+)\s*\(", header, re.M))
    assert declared, "no declarations parsed"
    assert declared == set(B.EXPORTED)
    L = B.lib()
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings():
    for code in range(8):
        assert B.status_string(code) != "unknown status"
    assert B.status_string(99) == "unknown status"


def _plan(b, mode=None, sms=152):
    if mode is None:
        mode = B.FI_MODE_DECODE if (b.is_decode and not b.causal) else B.FI_MODE_PREFILL
    return B.fi_plan(mode, b.batch, b.qo_indptr if mode == B.FI_MODE_PREFILL else None,
                     b.page_indptr, b.last_page_len, b.num_qo_heads, b.num_kv_heads, b.head_dim,
                     b.page_size, b.causal, plan_options(b), sms)


def _check_decode_cover(b, plan):
    """Each visible (request, kv head, key) exactly once; chunks start on
    page boundaries (the first one of a windowed request inside its first
    page); pages named are the request's own."""
    info = B.fi_plan_get_info(plan)
    work = B.fi_plan_get_work(plan)
    dec = work[:info["num_decode_items"]]
    seen = {}
    for req, kh, pb, npg, t0, t1, slot, qrow in dec.tolist():
        a = t0 - t0 % b.page_size                   # start of the page holding t0
        assert pb == b.page_indptr[req] + a // b.page_size
        assert npg == -(-(t1 - a) // b.page_size)
        assert pb + npg <= b.page_indptr[req + 1]
        assert qrow == b.qo_indptr[req]
        for t in range(t0, t1):
            seen[(req, kh, t)] = seen.get((req, kh, t), 0) + 1

    def first(r):      # first visible key of a decode row
        return 0 if b.window_left < 0 else max(0, int(b.kv_lens[r]) - 1 - b.window_left)
    want = {(r, h, t) for r in range(b.batch) if b.qo_lens[r] == 1
            for h in range(b.num_kv_heads) for t in range(first(r), int(b.kv_lens[r]))}
    assert set(seen) == want
    assert all(c == 1 for c in seen.values())
    # every decode request appears for every kv head (also empty ones)
    per = {}
    for req, kh, *_ in dec.tolist():
        per.setdefault(req, set()).add(kh)
    for r in range(b.batch):
        if b.qo_lens[r] == 1:
            assert per[r] == set(range(b.num_kv_heads))
    # longest items first
    lens = dec[:, 5] - dec[:, 4]
    assert np.all(np.diff(lens) <= 0)
    # split requests own consecutive slots, one per chunk
    slots = dec[dec[:, 6] >= 0]
    if len(slots):
        assert info["num_partial_slots"] == len(set(slots[:, 6].tolist()))
    return info


@pytest.mark.parametrize("name", ["tiny", "7b", "70b"])
def test_decode_plans_cover_every_key_once(name):
    if name == "tiny":
        b = synth.tiny_decode()
    elif name == "7b":
        g = synth.philox(1001)
        b = _table_only(g.integers(512, 4097, size=64), 32, 32, 128, 16)
    else:
        g = synth.philox(1002)
        b = _table_only(synth.lognormal_lengths(g, 128), 64, 8, 128, 16)
    plan = _plan(b)
    info = _check_decode_cover(b, plan)
    assert info["workspace_bytes"] >= 256
    if name == "70b":
        assert info["num_split_requests"] > 0


def _table_only(kv, hq, hkv, d, P, qo=None):
    """A batch with a page table but a one-page dummy cache (planning only)."""
    kv = np.asarray(kv, np.int64)
    qo = np.ones_like(kv) if qo is None else np.asarray(qo, np.int64)
    npg = np.where(kv > 0, (kv + P - 1) // P, 0)
    indptr = np.zeros(len(kv) + 1, np.int32)
    indptr[1:] = np.cumsum(npg)
    qo_indptr = np.zeros(len(kv) + 1, np.int32)
    qo_indptr[1:] = np.cumsum(qo)
    last = np.where(kv > 0, kv - (npg - 1) * P, 0).astype(np.int32)
    z = np.zeros((1, P, hkv, d), np.uint16)
    return synth.PagedBatch("table", hq, hkv, d, P, synth.NHD, 0.1, bool((qo > 1).any()), kv, qo,
                            qo_indptr, indptr, np.arange(int(npg.sum()), dtype=np.int32), last,
                            np.zeros((int(qo.sum()), hq, d), np.uint16), z, z)


@pytest.mark.parametrize("sms", [1, 7, 152])
def test_split_decisions_scale_with_sm_count(sms):
    b = _table_only([1, 0, 33, 4096, 32768, 700], 32, 8, 128, 16)
    plan = _plan(b, sms=sms)
    info = _check_decode_cover(b, plan)
    assert info["chunk_tokens"] % 16 == 0
    assert info["chunk_tokens"] >= 512


@pytest.mark.parametrize("hq,hkv", [(8, 2), (8, 8), (16, 2)])
def test_prefill_plan_tiles_and_causal_bounds(hq, hkv):
    """Prefill items are (128 rows, query head); every (request, query
    head, row) exactly once."""
    kv = [300, 1, 129, 77, 5000]
    qo = [300, 1, 100, 77, 4]
    b = _table_only(kv, hq, hkv, 128, 16, qo)
    plan = _plan(b, B.FI_MODE_PREFILL)
    info = B.fi_plan_get_info(plan)
    work = B.fi_plan_get_work(plan)
    pre = work[info["num_decode_items"]:]
    rows = {}
    for req, h, pb, npg, t0, t1, slot, qrow in pre.tolist():
        qo_len, kv_len = qo[req], kv[req]
        r0 = qrow - b.qo_indptr[req]
        r_last = min(qo_len, r0 + 128) - 1
        assert t0 == 0 and slot == -1 and 0 <= h < hq
        assert t1 == min(kv_len, kv_len - qo_len + r_last + 1)   # causal bound of the last row
        assert npg == -(-t1 // 16)
        for r in range(r0, r_last + 1):
            rows[(req, h, r)] = rows.get((req, h, r), 0) + 1
    want = {(r, h, i) for r in range(len(kv)) if qo[r] >= 2 for h in range(hq)
            for i in range(qo[r])}
    assert set(rows) == want and all(c == 1 for c in rows.values())
    # the single-row request is decode work
    _check_decode_cover(b, plan)
    assert np.all(np.diff(pre[:, 5]) <= 0)


@pytest.mark.parametrize("w", [0, 1, 15, 16, 17, 600, 5000])
def test_windowed_decode_plans_cover_the_window_once(w):
    b = _table_only([1, 0, 33, 4096, 32768, 700, 17], 32, 8, 128, 16)
    b.window_left = w
    for sms in (1, 152):
        _check_decode_cover(b, _plan(b, sms=sms))


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("w", [0, 100, 127, 128, 1000])
def test_windowed_prefill_items_start_on_the_page_of_the_first_row_window(causal, w):
    kv = [300, 129, 77, 5000, 2000]
    qo = [300, 100, 77, 4, 700]
    b = _table_only(kv, 8, 2, 128, 16, qo)
    b.causal = causal
    b.window_left = w
    for sms in (152, 4):   # split tiles (few work units for 152 SMs) and whole ones
        _check_prefill_cover(b, _plan(b, B.FI_MODE_PREFILL, sms=sms))


@pytest.mark.parametrize("case,status", [
    ("last_page_len_zero", B.FI_ERR_INVALID_ARG),
    ("last_page_len_big", B.FI_ERR_INVALID_ARG),
    ("decreasing_indptr", B.FI_ERR_INVALID_ARG),
    ("causal_qo_gt_kv", B.FI_ERR_INVALID_ARG),
    ("heads_not_multiple", B.FI_ERR_INVALID_ARG),
    ("head_dim_96", B.FI_ERR_UNSUPPORTED),
    ("page_size_8", B.FI_ERR_UNSUPPORTED),
    ("group_3", B.FI_ERR_UNSUPPORTED),
    ("decode_with_qo_indptr", B.FI_ERR_INVALID_ARG),
    ("prefill_without_qo_indptr", B.FI_ERR_INVALID_ARG),
    ("qo_indptr_not_zero_based", B.FI_ERR_INVALID_ARG),
    ("no_sms", B.FI_ERR_INVALID_ARG),
    ("window_below_minus_one", B.FI_ERR_INVALID_ARG),
    ("dtype_unknown", B.FI_ERR_INVALID_ARG),
    ("q_dtype_e4m3", B.FI_ERR_INVALID_ARG),
    ("kv_dtype_other_16bit", B.FI_ERR_INVALID_ARG),
    ("fp8_cache_prefill_plan", B.FI_ERR_UNSUPPORTED),
])
def test_plan_validation(case, status):
    args = dict(mode=B.FI_MODE_DECODE, batch_size=2, qo_indptr_h=None,
                page_indptr_h=[0, 2, 3], last_page_len_h=[5, 16], num_qo_heads=8,
                num_kv_heads=2, head_dim=128, page_size=16, causal=0, options=None,
                num_sms=152)
    if case == "last_page_len_zero":
        args["last_page_len_h"] = [0, 16]
    elif case == "last_page_len_big":
        args["last_page_len_h"] = [17, 16]
    elif case == "decreasing_indptr":
        args["page_indptr_h"] = [0, 3, 2]
    elif case == "causal_qo_gt_kv":
        args.update(mode=B.FI_MODE_PREFILL, qo_indptr_h=[0, 22, 23], causal=1)
    elif case == "heads_not_multiple":
        args["num_qo_heads"] = 7
    elif case == "head_dim_96":
        args["head_dim"] = 96
    elif case == "page_size_8":
        args["page_size"] = 8
    elif case == "group_3":
        args.update(num_qo_heads=6, num_kv_heads=2)
    elif case == "decode_with_qo_indptr":
        args["qo_indptr_h"] = [0, 1, 2]
    elif case == "prefill_without_qo_indptr":
        args["mode"] = B.FI_MODE_PREFILL
    elif case == "qo_indptr_not_zero_based":
        args.update(mode=B.FI_MODE_PREFILL, qo_indptr_h=[1, 2, 3])
    elif case == "no_sms":
        args["num_sms"] = 0
    elif case == "window_below_minus_one":
        args["options"] = {"window_left": -2}
    elif case == "dtype_unknown":
        args["options"] = {"dtype": 7}
    elif case == "q_dtype_e4m3":
        args["options"] = {"dtype": B.FI_DTYPE_E4M3}
    elif case == "kv_dtype_other_16bit":
        args["options"] = {"dtype": B.FI_DTYPE_BF16, "kv_dtype": B.FI_DTYPE_FP16}
    elif case == "fp8_cache_prefill_plan":
        args.update(mode=B.FI_MODE_PREFILL, qo_indptr_h=[0, 2, 3],
                    options={"kv_dtype": B.FI_DTYPE_E4M3})
    with pytest.raises(B.FiError) as e:
        B.fi_plan(**args)
    assert e.value.status == status


def test_valid_edge_plans():
    # empty batch; a request without pages (last_page_len ignored in [0, P])
    p = B.fi_plan(B.FI_MODE_DECODE, 0, None, [0], [], 8, 2, 64, 16, 0, None, 4)
    assert B.fi_plan_get_info(p)["num_items"] == 0
    p = B.fi_plan(B.FI_MODE_DECODE, 2, None, [0, 0, 1], [0, 3], 8, 2, 64, 16, 0, None, 4)
    info = B.fi_plan_get_info(p)
    assert info["total_kv_tokens"] == 3 and info["num_decode_items"] == 4


def test_longest_request_plans_and_one_page_more_is_rejected():
    # a request may hold up to INT32_MAX / 2 keys (key positions and their
    # sums stay in int32 on the device); the split covers it with bounded
    # work lists
    npg = (2**31 - 1) // 2 // 16
    p = B.fi_plan(B.FI_MODE_DECODE, 1, None, [0, npg], [15], 8, 2, 128, 16, 0, None, 152)
    info = B.fi_plan_get_info(p)
    assert info["total_kv_tokens"] == (npg - 1) * 16 + 15
    assert info["num_split_requests"] == 1
    assert info["num_decode_items"] <= 4 * 152 * 2       # a few waves, not one per page
    chunks = info["num_decode_items"] // 2                 # items: (chunk, kv head), 2 kv heads
    assert info["chunk_tokens"] * chunks >= info["total_kv_tokens"]
    with pytest.raises(B.FiError) as e:
        B.fi_plan(B.FI_MODE_DECODE, 1, None, [0, npg + 1], [16], 8, 2, 128, 16, 0, None, 152)
    assert e.value.status == B.FI_ERR_INVALID_ARG


def test_workspace_too_small_and_bad_args_return_before_any_launch():
    """Host-side checks happen before the device is touched; on a machine
    without a GPU, a well-formed call reports that there is no device."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("uses fake device addresses; only meaningful without a GPU")
    p = B.fi_plan(B.FI_MODE_DECODE, 2, None, [0, 2, 3], [5, 16], 8, 2, 128, 16, 0, None, 4)
    fake = 1 << 20   # aligned, never dereferenced: every call below returns first
    args = [p, fake, fake, fake, B.FI_LAYOUT_NHD, 0, 4, fake, fake, fake, 0.1, 1.0, 1.0, fake,
            fake, fake]
    with pytest.raises(B.FiError) as e:
        B.fi_batch_decode_paged(*args, workspace_bytes=16, stream=0)
    assert e.value.status == B.FI_ERR_WORKSPACE_TOO_SMALL
    bad = list(args)
    bad[1] = fake + 2          # misaligned q
    with pytest.raises(B.FiError) as e:
        B.fi_batch_decode_paged(*bad, stream=0)
    assert e.value.status == B.FI_ERR_INVALID_ARG
    bad = list(args)
    bad[4] = 7                 # unknown layout
    with pytest.raises(B.FiError) as e:
        B.fi_batch_decode_paged(*bad, stream=0)
    assert e.value.status == B.FI_ERR_INVALID_ARG
    with pytest.raises(B.FiError) as e:      # prefill call with a decode plan
        B.fi_batch_prefill_paged(p, fake, fake, fake, fake, 0, 0, 4, fake, fake, fake, 0.1, 1.0,
                                 1.0, fake, fake, fake, stream=0)
    assert e.value.status == B.FI_ERR_INVALID_ARG
    for bad_scale in (-0.1, float("nan"), float("inf")):
        bad = list(args)
        bad[10] = bad_scale    # sm_scale must be finite and >= 0
        with pytest.raises(B.FiError) as e:
            B.fi_batch_decode_paged(*bad, stream=0)
        assert e.value.status == B.FI_ERR_INVALID_ARG
    for pos, bad_scale in ((11, 0.0), (11, float("nan")), (12, -1.0), (12, float("inf"))):
        bad = list(args)
        bad[pos] = bad_scale   # k_scale and v_scale must be finite and > 0
        with pytest.raises(B.FiError) as e:
            B.fi_batch_decode_paged(*bad, stream=0)
        assert e.value.status == B.FI_ERR_INVALID_ARG
    for kw in ({"k_head_scale": fake + 2}, {"v_head_scale": fake + 1}):
        with pytest.raises(B.FiError) as e:   # per-head scale arrays: fp32, 4-byte aligned
            B.fi_batch_decode_paged(*args, stream=0, **kw)
        assert e.value.status == B.FI_ERR_INVALID_ARG
    with pytest.raises(B.FiError) as e:
        B.fi_batch_decode_paged(*args, stream=0)
    assert e.value.status == B.FI_ERR_NO_DEVICE
    with pytest.raises(B.FiError) as e:      # aligned per-head scales pass the host checks
        B.fi_batch_decode_paged(*args, stream=0, k_head_scale=fake, v_head_scale=fake + 4)
    assert e.value.status == B.FI_ERR_NO_DEVICE
    with pytest.raises(B.FiError) as e:
        B.fi_merge_states(fake, fake, 2, 3, 4, 6, B.FI_DTYPE_BF16, fake, None, stream=0)  # d % 4
    assert e.value.status == B.FI_ERR_INVALID_ARG
    with pytest.raises(B.FiError) as e:
        B.fi_merge_states(fake, fake, 2, 3, 4, 8, 5, fake, None, stream=0)   # unknown dtype
    assert e.value.status == B.FI_ERR_INVALID_ARG


def _check_prefix_cover(b, gi, pages, sms):
    """Shared-prefix decode: the prefix items cover every (row of a group,
    query head, prefix key) once; the decode items cover each grouped
    request's keys after the prefix once (the rest as usual); every grouped
    request goes through a merge. Returns the number of prefix chunks of the
    longest group."""
    P, hq, hkv = b.page_size, b.num_qo_heads, b.num_kv_heads
    g = hq // hkv
    rows_per_tile = 128 // g                       # a tile packs the g heads of a kv head
    G = len(gi) - 1
    p = B.fi_plan(B.FI_MODE_DECODE, b.batch, None, b.page_indptr, b.last_page_len, hq, hkv,
                  b.head_dim, P, 0, {"prefix_group_indptr": gi, "prefix_pages": pages}, sms)
    info = B.fi_plan_get_info(p)
    work = B.fi_plan_get_work(p)
    nd = info["num_decode_items"]
    assert info["num_prefix_groups"] == G
    dec, pre = work[:nd], work[nd:]
    # counts[r, h, t]: row r of q (a grouped request), query head h, prefix key t
    counts = {grp: np.zeros((gi[grp + 1] - gi[grp], hq, pages[grp] * P), np.int32)
              for grp in range(G)}
    chunks = {}
    for req, kh, pb, npg, t0, t1, slot, qrow in pre.tolist():
        grp = req // 2
        assert req % 2 == 0 and pb == b.page_indptr[gi[grp]] + t0 // P
        assert 0 <= t0 < t1 <= pages[grp] * P and t0 % 128 == 0
        assert npg == -(-(t1 - t0) // P)
        r0 = qrow - gi[grp]
        counts[grp][r0:r0 + rows_per_tile, kh * g:(kh + 1) * g, t0:t1] += 1
        chunks.setdefault(grp, set()).add(t0)
    for grp in range(G):
        assert np.all(counts[grp] == 1)
    prefix = {r: pages[grp] * P for grp in range(G) for r in range(gi[grp], gi[grp + 1])}
    cover = [np.zeros((hkv, int(k)), np.int32) for k in b.kv_lens]
    for req, kh, pb, npg, t0, t1, slot, qrow in dec.tolist():
        assert t0 >= prefix.get(req, 0)
        if req in prefix:
            assert slot >= 0            # grouped rows always go through a merge
        cover[req][kh, t0:t1] += 1
    for r in range(b.batch):
        k0 = prefix.get(r, 0)
        assert np.all(cover[r][:, :k0] == 0) and np.all(cover[r][:, k0:] == 1)
    return max((len(c) for c in chunks.values()), default=0)


def test_shared_prefix_plan_covers_prefix_and_suffixes():
    kv = [100, 48, 300, 5000, 64, 17, 900]
    b = _table_only(kv, 16, 2, 128, 16)
    gi, pages = [0, 3, 3, 5], [3, 1, 4]            # group 1 is empty
    for sms in (4, 152):
        _check_prefix_cover(b, gi, pages, sms)


@pytest.mark.parametrize("seed", range(20))
def test_random_shared_prefix_plans(seed):
    """Seeded random groups of consecutive requests (some empty), prefixes
    of whole shared pages, every supported group size, 1 to 300 SMs."""
    rng = np.random.default_rng(2000 + seed)
    P = int(rng.choice([16, 32]))
    hkv = int(rng.choice([1, 2]))
    hq = hkv * int(rng.choice([1, 2, 4, 8]))
    batch = int(rng.integers(2, 10))
    cuts = np.sort(rng.choice(np.arange(batch + 1), size=int(rng.integers(2, 5)), replace=True))
    gi = [int(x) for x in cuts]
    # short prefixes (one chunk) and long ones (cut into several chunks)
    pages = [int(rng.integers(1, 12)) if rng.random() < 0.5 else int(rng.integers(64, 400))
             for _ in range(len(gi) - 1)]
    kv = rng.integers(0, 1500, size=batch)
    for grp in range(len(gi) - 1):                 # grouped requests hold the prefix pages
        for r in range(gi[grp], gi[grp + 1]):
            kv[r] = pages[grp] * P + int(rng.choice([0, 1, int(rng.integers(1, 600))]))
    b = _table_only(kv, hq, hkv, 128, P)
    _check_prefix_cover(b, gi, pages, int(rng.integers(1, 300)))


def test_long_shared_prefix_is_cut_into_chunks():
    kv = [9000, 8200, 8193, 5000]
    b = _table_only(kv, 8, 1, 128, 16)
    assert _check_prefix_cover(b, [0, 3], [512], 152) > 1


@pytest.mark.parametrize("case,status", [
    ("prefix_longer_than_request", B.FI_ERR_INVALID_ARG),
    ("prefix_not_full_pages", B.FI_ERR_INVALID_ARG),
    ("zero_pages", B.FI_ERR_INVALID_ARG),
    ("decreasing_groups", B.FI_ERR_INVALID_ARG),
    ("past_the_batch", B.FI_ERR_INVALID_ARG),
    ("prefill_plan", B.FI_ERR_UNSUPPORTED),
    ("with_window", B.FI_ERR_UNSUPPORTED),
    ("with_fp8_cache", B.FI_ERR_UNSUPPORTED),
])
def test_shared_prefix_validation(case, status):
    kv = [40, 40, 100]           # pages 3, 3, 7; the 40-token requests end mid-page
    b = _table_only(kv, 8, 2, 128, 16)
    opts = {"prefix_group_indptr": [0, 2], "prefix_pages": [2]}
    mode, qo = B.FI_MODE_DECODE, None
    if case == "prefix_longer_than_request":
        opts["prefix_pages"] = [4]
    elif case == "prefix_not_full_pages":
        opts["prefix_pages"] = [3]              # page 3 of a 40-token request holds 8 tokens
    elif case == "zero_pages":
        opts["prefix_pages"] = [0]
    elif case == "decreasing_groups":
        opts = {"prefix_group_indptr": [0, 2, 1], "prefix_pages": [2, 2]}
    elif case == "past_the_batch":
        opts["prefix_group_indptr"] = [0, 4]
    elif case == "prefill_plan":
        mode, qo = B.FI_MODE_PREFILL, [0, 1, 2, 3]
    elif case == "with_window":
        opts["window_left"] = 10
    elif case == "with_fp8_cache":
        opts["kv_dtype"] = B.FI_DTYPE_E4M3
    with pytest.raises(B.FiError) as e:
        B.fi_plan(mode, 3, qo, b.page_indptr, b.last_page_len, 8, 2, 128, 16, 0, opts, 152)
    assert e.value.status == status


def test_host_buffer_call_sizes_its_region_and_checks_before_any_copy():
    """fi_batch_attention_host: the plan reports the workspace part that holds
    the step's q, out and lse (each region 256-byte aligned; the page table
    sits in the run calls' part, right after the work lists, and crosses the
    link with them); bad arguments and a short workspace are refused before
    anything is copied, and a well-formed call on a machine without a GPU
    reports that."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("uses fake device addresses; only meaningful without a GPU")
    rnd = lambda n: (n + 255) // 256 * 256
    # decode: 2 rows x 8 heads x d128 (bf16) for q and out, fp32 lse
    p = B.fi_plan(B.FI_MODE_DECODE, 2, None, [0, 2, 3], [5, 16], 8, 2, 128, 16, 0, None, 4)
    info = B.fi_plan_get_info(p)
    assert info["host_io_bytes"] == 2 * rnd(2 * 8 * 128 * 2) + rnd(2 * 8 * 4)
    # the page table (3 + 3 + 2 int32) is part of the run calls' workspace
    p0 = B.fi_plan(B.FI_MODE_DECODE, 0, None, [0], [], 8, 2, 128, 16, 0, None, 4)
    # prefill: 4 rows; the page table gains qo_indptr (3 more int32)
    pf = B.fi_plan(B.FI_MODE_PREFILL, 2, [0, 3, 4], [0, 2, 3], [5, 16], 8, 2, 128, 16, 1,
                   None, 4)
    info_f = B.fi_plan_get_info(pf)
    assert info_f["host_io_bytes"] == 2 * rnd(4 * 8 * 128 * 2) + rnd(4 * 8 * 4)
    del p0

    fake = 1 << 20    # aligned device address, never dereferenced here
    q_h = np.zeros((2, 8, 128), np.uint16)
    out_h = np.zeros_like(q_h)
    lse_h = np.zeros((2, 8), np.float32)
    indptr, indices, last = (np.array(a, np.int32) for a in ([0, 2, 3], [0, 1, 2], [5, 16]))
    need = info["workspace_bytes"] + info["host_io_bytes"]
    args = [p, q_h, None, fake, fake, B.FI_LAYOUT_NHD, 0, 4, indptr, indices, last, 0.1, 1.0,
            1.0, out_h, lse_h, fake, need]
    with pytest.raises(B.FiError) as e:
        B.fi_batch_attention_host(*args[:-1], info["workspace_bytes"], stream=0)
    assert e.value.status == B.FI_ERR_WORKSPACE_TOO_SMALL
    for pos, bad_value in ((1, None), (14, None), (8, None), (3, None), (5, 7), (11, -1.0),
                           (12, 0.0), (16, fake + 8)):
        bad = list(args)
        bad[pos] = bad_value   # q_h, out_h, page_indptr_h, k_cache, layout, scales, alignment
        with pytest.raises(B.FiError) as e:
            B.fi_batch_attention_host(*bad, stream=0)
        assert e.value.status == B.FI_ERR_INVALID_ARG, pos
    with pytest.raises(B.FiError) as e:      # a prefill plan needs qo_indptr_h
        B.fi_batch_attention_host(pf, np.zeros((4, 8, 128), np.uint16), None, fake, fake,
                                  B.FI_LAYOUT_NHD, 0, 4, indptr, indices, last, 0.1, 1.0, 1.0,
                                  np.zeros((4, 8, 128), np.uint16), None, fake,
                                  info_f["workspace_bytes"] + info_f["host_io_bytes"], stream=0)
    assert e.value.status == B.FI_ERR_INVALID_ARG
    with pytest.raises(B.FiError) as e:
        B.fi_batch_attention_host(*args, stream=0)
    assert e.value.status == B.FI_ERR_NO_DEVICE
    # the asynchronous form checks the same way, before a ticket exists
    with pytest.raises(B.FiError) as e:
        B.fi_batch_attention_host_async(*args[:-1], info["workspace_bytes"], stream=0)
    assert e.value.status == B.FI_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(B.FiError) as e:
        B.fi_batch_attention_host_async(*args, stream=0)
    assert e.value.status == B.FI_ERR_NO_DEVICE


def test_plans_without_query_rows_run_nothing():
    """A plan without query rows (every request's qo_len 0, keys or not) makes
    the run calls return FI_OK at once, reading no argument but the plan."""
    for kv in ([0, 0], [0, 37]):
        p = B.fi_plan(B.FI_MODE_PREFILL, 2, [0, 0, 0], [0, 0, -(-kv[1] // 16)],
                      [0, kv[1] - 16 * (-(-kv[1] // 16) - 1) if kv[1] else 0], 8, 2, 128, 16,
                      1, None, 152)
        assert B.fi_plan_get_info(p)["num_items"] == 0
        B.fi_batch_prefill_paged(p, None, None, None, None, B.FI_LAYOUT_NHD, 0, 0, None, None,
                                 None, 0.1, 1.0, 1.0, None, None, None, 0, stream=0)
        t = B.fi_batch_attention_host_async(p, None, None, None, None, B.FI_LAYOUT_NHD, 0, 0,
                                            None, None, None, 0.1, 1.0, 1.0, None, None, None,
                                            0, stream=0)
        assert t == 0


def test_host_step_tickets_without_a_device():
    """An empty plan's step has ticket 0, which is always complete; a ticket
    that was never issued is refused."""
    p0 = B.fi_plan(B.FI_MODE_DECODE, 0, None, [0], [], 8, 2, 128, 16, 0, None, 4)
    t = B.fi_batch_attention_host_async(p0, None, None, None, None, B.FI_LAYOUT_NHD, 0, 0,
                                        None, None, None, 0.1, 1.0, 1.0, None, None, None, 0,
                                        stream=0)
    assert t == 0
    B.fi_host_step_wait(0)
    for bogus in (1, 9, 2**63 + 5):
        with pytest.raises(B.FiError) as e:
            B.fi_host_step_wait(bogus)
        assert e.value.status == B.FI_ERR_INVALID_ARG


def _check_prefill_cover(b, plan):
    """Each (request, query head, row) of a multi-row request in exactly one
    prefill tile, whose page-aligned key range holds every key its rows may
    see: from the page of its first row's first visible key to the causal
    bound of its last row (or the end of the keys). A tile is one item, or
    (a split tile) pieces of whole KV tiles that cover its range once, in
    order, each with its own state slots (row r of piece j: slot s0 + r * k
    + j, k pieces), disjoint from every other tile's."""
    info = B.fi_plan_get_info(plan)
    pre = B.fi_plan_get_work(plan)[info["num_decode_items"]:][:info["num_prefill_items"]]
    P, w = b.page_size, b.window_left
    kv_tile = 128 if b.head_dim <= 128 else 64
    tiles = {}
    for req, h, pb, npg, t0, t1, slot, qrow in pre.tolist():
        assert 0 <= h < b.num_qo_heads
        assert pb == b.page_indptr[req] + t0 // P and npg == -(-(t1 - t0) // P)
        assert pb + npg <= b.page_indptr[req + 1]
        tiles.setdefault((req, h, qrow), []).append((t0, t1, slot))
    rows, slots = {}, set()
    for (req, h, qrow), pieces in tiles.items():
        qo_len, kv_len = int(b.qo_lens[req]), int(b.kv_lens[req])
        r0 = qrow - int(b.qo_indptr[req])
        r_last = min(qo_len, r0 + 128) - 1
        end = min(kv_len, kv_len - qo_len + r_last + 1) if b.causal else kv_len
        first = 0 if w < 0 else max(0, kv_len - qo_len + r0 - w)
        pieces.sort()
        t0 = pieces[0][0]
        assert t0 % P == 0 and t0 <= min(first, end) < t0 + P or t0 == pieces[-1][1]
        assert pieces[-1][1] == end
        k = len(pieces)
        if k == 1:
            assert pieces[0][2] == -1
        else:
            s0 = pieces[0][2]
            for j, (a, z, slot) in enumerate(pieces):
                assert (a - t0) % kv_tile == 0 and a < z and slot == s0 + j
                assert j == 0 or a == pieces[j - 1][1]
            if h == 0:
                for r in range(r_last + 1 - r0):
                    for j in range(k):
                        assert s0 + r * k + j not in slots
                        slots.add(s0 + r * k + j)
        for r in range(r0, r_last + 1):
            rows[(req, h, r)] = rows.get((req, h, r), 0) + 1
    assert all(0 <= s < info["num_partial_slots"] for s in slots)
    want = {(r, h, i) for r in range(b.batch) if b.qo_lens[r] >= 2
            for h in range(b.num_qo_heads) for i in range(int(b.qo_lens[r]))}
    assert set(rows) == want and all(c == 1 for c in rows.values())
    lens = pre[:, 5] - pre[:, 4]
    assert np.all(np.diff(lens) <= 0)                 # longest first
    if b.num_qo_heads % 2 == 0:
        # items 2p and 2p + 1: heads h, h + 1 of one tile (the two-tile kernel's pairs)
        assert np.all(pre[0::2, 1] % 2 == 0) and np.all(pre[0::2, 1] + 1 == pre[1::2, 1])
        same = [0, 2, 3, 4, 5, 6, 7]                   # every field but the head
        assert np.array_equal(pre[0::2][:, same], pre[1::2][:, same])
    return tiles


def test_short_prefill_launches_split_their_long_tiles():
    """Under two waves of work units, long tiles are cut into pieces when the
    estimate gains enough: a 512-row chunk on 32K keys with 32/8 heads (4
    tiles x 16 head pairs = 64 units on 152 SMs) is split; with 64/8 heads
    (128 units) the estimated gain is too small; with two waves or more, with
    decode rows in the plan, or with short tiles nothing is split."""
    b = _table_only([32768], 32, 8, 128, 16, [512])
    b.causal = True
    plan = _plan(b, B.FI_MODE_PREFILL, sms=152)
    tiles = _check_prefill_cover(b, plan)
    ks = {len(p) for p in tiles.values()}
    assert len(ks) == 1 and min(ks) > 1
    k = ks.pop()
    # 64 units of ~256 KV tiles: k minimises ceil(64 k / 152) (256 / k + 5)
    f = lambda k: -(-64 * k // 152) * (256 / k + 5)
    assert f(k) == min(f(j) for j in range(1, 17)) and f(k) <= 0.85 * f(1)
    info = B.fi_plan_get_info(plan)
    assert info["num_partial_slots"] == 512 * k
    for hq, sms in ((64, 152), (32, 32)):   # a small gain; two waves of units
        b1 = _table_only([32768], hq, 8, 128, 16, [512])
        b1.causal = True
        tiles = _check_prefill_cover(b1, _plan(b1, B.FI_MODE_PREFILL, sms=sms))
        assert all(len(p) == 1 for p in tiles.values())
    # a decode row in the batch: whole tiles
    b2 = _table_only([32768, 900], 32, 8, 128, 16, [512, 1])
    b2.causal = True
    tiles = _check_prefill_cover(b2, _plan(b2, B.FI_MODE_PREFILL, sms=152))
    assert all(len(p) == 1 for p in tiles.values())
    # short tiles (under 16 KV tiles) stay whole
    b3 = _table_only([1900], 8, 2, 128, 16, [300])
    b3.causal = True
    tiles = _check_prefill_cover(b3, _plan(b3, B.FI_MODE_PREFILL, sms=152))
    assert all(len(p) == 1 for p in tiles.values())


@pytest.mark.parametrize("seed", range(40))
def test_random_plans_cover_every_visible_key_once(seed):
    """Seeded random page tables (empty requests, lengths on and off page
    boundaries, decode rows mixed into prefill batches, left windows, 1 to
    300 SMs) against the coverage rules of the decode and prefill work."""
    g = np.random.default_rng(1000 + seed)
    P = int(g.choice([16, 32]))
    hkv = int(g.choice([1, 2, 4]))
    hq = hkv * int(g.choice([1, 2, 4, 8]))
    batch = int(g.integers(1, 12))
    kv = g.integers(0, 2500, size=batch)
    kv[g.random(batch) < 0.2] = 0
    edge = g.random(batch) < 0.3
    kv[edge] = (g.integers(1, 40, size=int(edge.sum())) * P + g.choice([-1, 0, 1])).clip(0)
    prefill = bool(g.random() < 0.6)
    if prefill:
        qo = np.where(g.random(batch) < 0.3, 1, g.integers(1, 400, size=batch))
        qo = np.minimum(qo, np.maximum(kv, 1))
        qo[kv == 0] = 0                               # causal plans need qo_len <= kv_len
    else:
        qo = np.ones(batch, np.int64)
    b = _table_only(kv, hq, hkv, 128, P, qo)
    b.causal = prefill and bool(g.random() < 0.8)
    b.window_left = int(g.choice([-1, -1, 0, 1, P - 1, P, 100, 1000]))
    sms = int(g.integers(1, 300))
    plan = _plan(b, B.FI_MODE_PREFILL if prefill else B.FI_MODE_DECODE, sms=sms)
    _check_decode_cover(b, plan)
    if prefill:
        _check_prefill_cover(b, plan)
