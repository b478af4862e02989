"""GPU parity of causal variable-length prefill (and mixed prefill + decode
batches) against the fp64 oracle, through fi_batch_prefill_paged. Small
cases are compared on every row; the full-size workloads on sampled rows
(first/last rows, tile and page boundaries, random rows) that the oracle
computes one by one."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from paged_kv_attention_27_gb300 import binding as B  # noqa: E402
from paged_kv_attention_27_gb300 import synth  # noqa: E402

from ._gpu import compare, ensure_built, scale_v  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    B.lib()


def _run(b, sms=None):
    from paged_kv_attention_27_gb300.device import DeviceBatch
    db = DeviceBatch(b, mode=B.FI_MODE_PREFILL, sms=sms)
    out, lse = db.run()
    torch.cuda.synchronize()
    assert db.status() == B.FI_OK
    return db, out, lse


def _oracle(b, rows=None, requests=None):
    return oracle.batch_attention(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.layout, b.page_indptr,
                                  b.page_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                                  b.page_size, b.sm_scale, b.causal, requests=requests, rows=rows,
                                  window_left=b.window_left, dtype=b.dtype,
                                  kv_dtype=b.cache_dtype, k_scale=b.k_scales, v_scale=b.v_scales)


def check_full(b, what=None):
    db, out, lse = _run(b)
    ref_o, ref_l = _oracle(b)
    compare(out, lse, ref_o, ref_l, what=what or b.name)
    return db


def sample_rows(b, per_request=24, seed=0):
    """Rows per request: first, last, around 128-row tile boundaries and the
    first page boundary, plus random rows."""
    rng = np.random.default_rng(seed)
    rows = {}
    for r in range(b.batch):
        n = int(b.qo_lens[r])
        if n == 0:
            continue
        s = {0, n - 1, min(n - 1, 1)}
        for t in range(127, n, 128):
            s.update({t, min(n - 1, t + 1)})
            if len(s) > per_request // 2:
                break
        s.update({min(n - 1, b.page_size - 1), min(n - 1, b.page_size)})
        if b.window_left >= 0:       # rows where the window starts to cut keys off
            w = b.window_left
            s.update({min(n - 1, x) for x in (w, w + 1, w + 127, w + 128, w + 129)})
        s.update(rng.integers(0, n, size=per_request // 2).tolist())
        rows[r] = sorted(s)
    return rows


def check_sampled(b, per_request=24, requests=None):
    db, out, lse = _run(b)
    rows = sample_rows(b, per_request)
    if requests is not None:
        rows = {r: v for r, v in rows.items() if r in requests}
    ref_o, ref_l = _oracle(b, rows=rows, requests=sorted(rows))
    flat = np.concatenate([b.qo_indptr[r] + np.asarray(v) for r, v in rows.items()])
    compare(out, lse, ref_o, ref_l, rows=flat, what=b.name)
    return db


@pytest.mark.parametrize("d,P", [(128, 16), (64, 16), (256, 32), (128, 32), (64, 32), (256, 16)])
def test_causal_prefill_small(d, P):
    kv = [1, 2, 17, 128, 129, 300, 513]
    b = synth.make_batch(f"prefill d{d} P{P}", kv, kv, 8, 2, d, P,
                         synth.NHD if d != 64 else synth.HND, None, True, 100 + d + P)
    check_full(b)


@pytest.mark.parametrize("case", ["pair_d128", "pair_d64_fp16", "one_tile_d256", "one_tile_g1",
                                  "window", "non_causal", "ragged"])
def test_split_prefill_tiles(case):
    """A launch of under two waves of work units cuts its long tiles into
    pieces of whole KV tiles; each piece writes fp32 states and one merge
    launch combines a row's pieces by log-sum-exp. Every row against the
    oracle, on the two-tile and the one-tile kernel, with a window, without
    the causal mask, and with tiles of different lengths."""
    mk = synth.make_batch
    if case == "pair_d128":
        b = mk("split pair d128", [9000], [300], 8, 2, 128, 16, synth.NHD, None, True, 901)
    elif case == "pair_d64_fp16":
        b = mk("split pair d64 fp16", [7000], [200], 8, 2, 64, 16, synth.HND, None, True, 902,
               dtype="fp16")
    elif case == "one_tile_d256":
        b = mk("split d256", [5000], [200], 16, 8, 256, 32, synth.HND, None, True, 903)
    elif case == "one_tile_g1":
        b = mk("split g1", [6000], [256], 4, 4, 128, 16, synth.NHD, None, True, 904)
    elif case == "window":
        b = mk("split window", [9000], [300], 8, 2, 128, 16, synth.NHD, None, True, 905,
               window_left=2500)
    elif case == "non_causal":
        b = mk("split non-causal", [8000], [200], 8, 2, 128, 16, synth.NHD, None, False, 906)
    else:
        b = mk("split ragged", [9000, 300, 4000, 2500], [300, 300, 129, 2], 8, 2, 128, 16,
               synth.NHD, None, True, 907)
    db = check_full(b)
    info = B.fi_plan_get_info(db.plan)
    assert info["num_partial_slots"] > 0   # the plan did split


def test_chunked_prefill_bottom_right_causal():
    kv = [700, 200, 129, 1000]
    qo = [37, 200, 128, 300]          # chunks appended to existing KV
    b = synth.make_batch("chunks", kv, qo, 16, 4, 128, 16, synth.HND, None, True, 7)
    check_full(b)


def test_non_causal_prefill_including_empty_kv():
    kv = [0, 50, 300, 5]
    qo = [3, 80, 17, 130]
    b = synth.make_batch("full attention", kv, qo, 8, 8, 128, 16, synth.NHD, None, False, 8)
    check_full(b)


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_group_sizes(g):
    """Even groups run on the two-tile kernel (two query heads per CTA), g = 1
    on the one-tile kernel."""
    kv = [255, 64, 390]
    b = synth.make_batch(f"prefill g{g}", kv, kv, 2 * g, 2, 128, 16, synth.NHD, None, True, 9 + g)
    check_full(b)


@pytest.mark.parametrize("g", [1, 2])
def test_group_sizes_d64(g):
    kv = [200, 17, 333]
    b = synth.make_batch(f"prefill g{g} d64", kv, kv, 3 * g, 3, 64, 16, synth.HND, None, True,
                         20 + g)
    check_full(b)


def test_nan_tail_slots_never_reach_the_output():
    kv = [3, 17, 45, 100, 200]
    b = synth.make_batch("prefill nan tail", kv, kv, 8, 2, 128, 16, synth.NHD, None, True, 12,
                         tail_fill="nan")
    check_full(b)
    b = synth.make_batch("prefill nan tail d256", kv, kv, 4, 2, 256, 32, synth.HND, None, True,
                         13, tail_fill="nan")
    check_full(b)


def test_small_mixed_batch_one_call():
    b = synth.small_mixed()
    db = check_full(b)
    info = B.fi_plan_get_info(db.plan)
    assert info["num_decode_items"] > 0 and info["num_prefill_items"] > 0


def test_deterministic():
    kv = [900, 300]
    b = synth.make_batch("det", kv, kv, 8, 2, 128, 16, synth.NHD, None, True, 14)
    db, out, lse = _run(b)
    o1, l1 = out.clone(), lse.clone()
    o2, l2 = db.run()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_large_scores_stay_finite_with_rescale():
    """Keys scaled page by page from 0x to 6x (sm_scale 1): scores span
    hundreds of log2 units, the running max jumps many times (the lazy
    rescale fires), yet outputs match the oracle."""
    kv = [600, 1000]
    b = synth.make_batch("big scores", kv, kv, 4, 2, 128, 16, synth.NHD, 1.0, True, 15)
    ramp = np.linspace(0, 6, b.k_cache.shape[0] * 16, dtype=np.float32).reshape(-1, 16)
    kf = oracle.bf16_to_f64(b.k_cache).astype(np.float32) * ramp[:, :, None, None]
    b.k_cache = synth.f32_to_bf16_bits(kf)
    # |o| ~ 0.25 keeps the bf16 rounding of the nearly one-hot outputs well
    # inside the mean-abs budget
    b.v_cache = synth.f32_to_bf16_bits(oracle.bf16_to_f64(b.v_cache).astype(np.float32) * 0.25)
    check_full(b)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("w", [0, 1, 63, 127, 128, 129, 500])
def test_sliding_window_causal_prefill(d, w):
    kv = [1, 17, 200, 700, 1000]
    qo = [1, 17, 200, 300, 1000]      # one decode row, full prefills and a chunk
    b = synth.make_batch(f"window {w} d{d}", kv, qo, 8, 2, d, 16 if d < 256 else 32,
                         synth.NHD, None, True, 300 + w + d, window_left=w)
    check_full(scale_v(b))


@pytest.mark.parametrize("w", [0, 40, 260])
def test_sliding_window_non_causal_prefill(w):
    kv = [0, 50, 300, 600]
    qo = [3, 80, 17, 130]
    b = synth.make_batch(f"window {w} non-causal", kv, qo, 8, 8, 128, 16, synth.HND, None, False,
                         400 + w, window_left=w)
    check_full(scale_v(b))


def test_sliding_window_mixed_batch():
    b = synth.small_mixed()
    b.window_left = 100
    check_full(b)


# ---- full-size workloads, sampled rows ------------------------------------

@pytest.mark.parametrize("L", [1024, 4096, 16384])
def test_causal_prefill_70b_full_size(L):
    check_sampled(synth.causal_prefill(L), per_request=16 if L > 4096 else 24)


def test_causal_prefill_32k_sampled():
    # two 32K-token requests: 256 query tiles each, up to 256 KV tiles per item
    check_sampled(synth.causal_prefill(32768, batch=2), per_request=12)


def test_ragged_prefill_full_size():
    check_sampled(synth.ragged_prefill(), per_request=16)


def test_mixed_chunk_decode_full_size():
    b = synth.mixed_chunk_decode()
    check_sampled(b, per_request=16, requests=set(range(8)) | {8, 9, 20, 33, 63})


@pytest.mark.parametrize("d,w", [(128, -1), (128, 100), (256, -1), (64, 33)])
def test_zero_score_scale_with_masked_tiles(d, w):
    """sm_scale = 0: every visible key weighs the same, hidden keys nothing,
    in tiles that cross the causal bound or the window too (the kernels hide
    a key by giving it a score of -inf, which must not meet a zero scale)."""
    kv = [300, 129, 17]
    b = synth.make_batch(f"zero scale d{d} w{w}", kv, kv, 4, 2, d, 16, synth.NHD, 0.0, True,
                         40 + d, window_left=w)
    scale_v(b)
    check_full(b)


@pytest.mark.parametrize("case", ["pair", "one-tile d256", "mixed"])
def test_per_head_scales_in_prefill_and_mixed_calls(case):
    """The per-kv-head scale arrays apply to every kernel: a 16-bit cache
    with K and V scaled per head (the two-tile and one-tile prefill kernels
    and the mixed launch)."""
    hkv = 2
    ks, vs = [0.5, 2.0], [2.0, 0.25]
    if case == "pair":
        kv = [300, 129, 700]
        b = synth.make_batch("per-head pair", kv, kv, 8, hkv, 128, 16, synth.NHD, None, True, 31,
                             head_scales=(ks, vs))
    elif case == "one-tile d256":
        kv = [300, 129]
        b = synth.make_batch("per-head d256", kv, kv, 2, hkv, 256, 32, synth.HND, None, True, 32,
                             head_scales=(ks, vs))
    else:
        kv, qo = [400, 150, 900, 3000], [96, 1, 1, 64]
        b = synth.make_batch("per-head mixed", kv, qo, 4, hkv, 256, 32, synth.NHD, None, True, 33,
                             head_scales=(ks, vs))
    check_full(b)


# ---- failure path: a bounded wait that runs out ----------------------------

@pytest.mark.parametrize("case", ["d128", "d256", "mixed"])
def test_bounded_wait_times_out_and_context_survives(case):
    """The test hook makes the first CTA's K producer skip its first tile, so
    the MMA issuer's bounded wait on that tile runs out: the call must report
    FI_ERR_DEVICE_TIMEOUT (no hang, no fault), and the next call in the same
    context must be correct."""
    from paged_kv_attention_27_gb300.device import DeviceBatch
    if case == "mixed":
        b = synth.small_mixed()
    else:
        d = int(case[1:])
        kv = [900, 300]
        b = synth.make_batch(f"timeout {case}", kv, kv, 8, 2, d, 16, synth.NHD, None, True, 16)
    db = DeviceBatch(b, mode=B.FI_MODE_PREFILL)
    B.fi_debug_set_fault(1, 2_000_000)          # 2 ms bound
    try:
        db.run()
        assert db.status() == B.FI_ERR_DEVICE_TIMEOUT
    finally:
        B.fi_debug_set_fault(0, 0)
    out, lse = db.run()
    torch.cuda.synchronize()
    assert db.status() == B.FI_OK
    ref_o, ref_l = _oracle(b)
    compare(out, lse, ref_o, ref_l, what=f"after timeout ({case})")


def test_sliding_window_prefill_16k_full_size():
    check_sampled(synth.causal_prefill(16384, window_left=4095), per_request=16)


# ---- fp16 inputs -----------------------------------------------------------

@pytest.mark.parametrize("d,P", [(64, 16), (128, 16), (256, 32)])
def test_fp16_causal_prefill(d, P):
    kv = [1, 2, 17, 128, 129, 300, 513]
    b = synth.make_batch(f"fp16 prefill d{d}", kv, kv, 8, 2, d, P, synth.HND, None, True,
                         600 + d, dtype="fp16", tail_fill="nan")
    db = check_full(b)
    assert db.out.dtype == torch.float16


def test_fp16_mixed_batch_with_window():
    b = synth.small_mixed()
    b = synth.make_batch("fp16 mixed window", b.kv_lens, b.qo_lens, 16, 8, 256, 32, synth.NHD,
                         None, True, 601, dtype="fp16", window_left=200)
    check_full(b)


def test_fp16_prefill_4k_full_size():
    b = synth.causal_prefill(4096, batch=2)
    b = synth.make_batch("fp16 causal prefill B2 L4096", b.kv_lens, b.qo_lens, 64, 8, 128, 16,
                         synth.NHD, None, True, 602, dtype="fp16")
    check_sampled(b, per_request=16)


@pytest.mark.parametrize("which", ["decode", "mixed", "prefill"])
def test_host_buffer_call_matches_device_call(which):
    """fi_batch_attention_host copies q and the page table in, runs the same
    kernels and copies out and lse back: bitwise the device-buffer call's
    results, and within the oracle's tolerances."""
    from paged_kv_attention_27_gb300.device import DeviceBatch
    if which == "decode":
        b, mode = synth.tiny_decode(), B.FI_MODE_DECODE
    elif which == "mixed":
        b, mode = synth.small_mixed(), B.FI_MODE_PREFILL
    else:
        kv = [1, 17, 129, 300]
        b = synth.make_batch("host-call prefill d128 P16", kv, kv, 8, 2, 128, 16, synth.NHD, None,
                             True, 41)
        mode = B.FI_MODE_PREFILL
    db = DeviceBatch(b, mode=mode)
    out_d, lse_d = db.run()
    torch.cuda.synchronize()
    assert db.status() == B.FI_OK
    out_h, lse_h = db.run_host()
    assert torch.equal(out_h.view(torch.int16), out_d.cpu().view(torch.int16))
    assert torch.equal(lse_h, lse_d.cpu())
    ref_o, ref_l = _oracle(b)
    compare(out_h, lse_h, ref_o, ref_l, what=f"host call, {b.name}")


def test_async_host_steps_in_flight():
    """fi_batch_attention_host_async: eight steps with their own q and
    outputs in flight on one workspace; a ninth is refused while they are;
    waiting for each in issue order gives, bitwise, what the device-buffer
    call gives for that step's q; a ticket waited for twice is refused."""
    from paged_kv_attention_27_gb300.device import DeviceBatch
    b = synth.tiny_decode()
    db = DeviceBatch(b)
    info = B.fi_plan_get_info(db.plan)
    ws_bytes = info["workspace_bytes"] + info["host_io_bytes"]
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=db.device)
    g = torch.Generator().manual_seed(77)
    qs = [torch.randn(db.q.shape, generator=g).to(db.q.dtype).pin_memory() for _ in range(8)]
    outs = [(torch.empty(db.out.shape, dtype=db.out.dtype).pin_memory(),
             torch.empty(db.lse.shape, dtype=torch.float32).pin_memory()) for _ in range(8)]
    tables = (b.page_indptr.astype(np.int32), b.page_indices.astype(np.int32),
              b.last_page_len.astype(np.int32))

    def issue(q_h, out_h, lse_h):
        return B.fi_batch_attention_host_async(
            db.plan, q_h, None, db.k, db.v, B.LAYOUTS[b.layout], 0, b.num_pages, *tables,
            b.sm_scale, b.k_scale, b.v_scale, out_h, lse_h, ws, ws_bytes,
            k_head_scale=db.k_head_scale, v_head_scale=db.v_head_scale)

    tickets = [issue(q, *o) for q, o in zip(qs, outs)]
    assert len(set(tickets)) == 8 and 0 not in tickets
    with pytest.raises(B.FiError) as e:
        issue(qs[0], *outs[0])
    assert e.value.status == B.FI_ERR_INVALID_ARG
    for t in tickets:
        B.fi_host_step_wait(t)
    with pytest.raises(B.FiError) as e:
        B.fi_host_step_wait(tickets[0])
    assert e.value.status == B.FI_ERR_INVALID_ARG
    for q_h, (out_h, lse_h) in zip(qs, outs):
        db.q.copy_(q_h)
        out_d, lse_d = db.run()
        torch.cuda.synchronize()
        assert torch.equal(out_h.view(torch.int16), out_d.cpu().view(torch.int16))
        assert torch.equal(lse_h, lse_d.cpu())
