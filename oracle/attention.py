"""fp64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline may import this module; the library path never does. It shares no
code with the CUDA side: it reads bf16 bit patterns itself, walks the page
table itself and computes everything in float64 from the plain definition.

What it computes, per request ``b``, query row ``i`` and query head ``h``
(the "FlashAttention-3 kernel integration in inference engines" page draws
attention as Q K^T -> softmax -> times V in its section 1 diagram; the
FlashInfer deep-dive page, section "PageAttention", stores K/V in fixed-size
pages reached through a page table; the same two pages name the default
scale ``1/sqrt(head_dim)``, section 3.1 of the FlashInfer analysis page and
the varlen wrapper of section 2 of the FlashAttention-3 page):

* ``kv_len[b] = (page_indptr[b+1]-page_indptr[b]-1)*P + last_page_len[b]``
  when the request owns pages, else 0;
* key ``t`` of request ``b`` lives on physical page
  ``page_indices[page_indptr[b] + t // P]`` in slot ``t % P``;
* GQA: query head ``h`` reads kv head ``h // (Hq/Hkv)``;
* causal varlen: row ``i`` of a request with ``qo_len`` rows sees keys
  ``t <= kv_len - qo_len + i`` (bottom-right alignment: a chunk's queries
  are the last ``qo_len`` positions of its KV);
* ``s_t = sm_scale * <q, k_t>``; ``lse = log(sum_visible exp(s_t))``
  (natural log of the scaled scores); ``o = sum_visible exp(s_t - lse) v_t``;
* a row with no visible key gives ``o = 0`` and ``lse = -inf``.

Besides this definition the module holds, as separate plain functions, the
three restatements the pins compare it against: the online (streaming)
softmax recurrence of FlashAttention-1/2 tiling (section 1 of the
FlashAttention-3 page: the softmax statistics are kept on chip and the output
is accumulated tile by tile), split-KV partial states combined by log-sum-exp
(``merge_states``), and an explicit additive-mask form
``softmax(scale*QK^T + mask) V``.
"""
from __future__ import annotations

import math

import numpy as np

NHD = "NHD"
HND = "HND"


# --------------------------------------------------------------------------
# reading the inputs
# --------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of IEEE binary16 bit patterns (uint16) as float64, from
    the format's definition: sign bit, 5 exponent bits (bias 15), 10
    fraction bits; exponent 0 is subnormal (2^-14 * f/1024), 31 is inf/NaN."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    normal = sign * np.ldexp(1.0 + f / 1024.0, (e - 15).astype(np.int32))
    sub = sign * np.ldexp(f / 1024.0, -14)
    special = np.where(f == 0, sign * np.inf, np.nan)
    return np.where(e == 0, sub, np.where(e == 31, special, normal))


def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of FP8 E4M3 bit patterns (uint8) as float64, from the OCP
    8-bit floating-point definition: sign bit, 4 exponent bits (bias 7), 3
    fraction bits; exponent 0 is subnormal (2^-6 * f/8); no infinities, and
    exponent 15 with fraction 7 is NaN (largest finite value 448)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    f = (b & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + f / 8.0, (e - 7).astype(np.int32))
    sub = sign * np.ldexp(f / 8.0, -6)
    val = np.where(e == 0, sub, normal)
    return np.where((e == 15) & (f == 7), np.nan, val)


def to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact value of bf16, fp16 or e4m3 bit patterns as float64."""
    if dtype == "bf16":
        return bf16_to_f64(bits)
    if dtype == "fp16":
        return f16_to_f64(bits)
    if dtype == "e4m3":
        return e4m3_to_f64(bits)
    raise ValueError(dtype)


def kv_lengths(page_indptr, last_page_len, page_size: int) -> np.ndarray:
    """Tokens held by each request's pages (all pages full but the last)."""
    page_indptr = np.asarray(page_indptr, dtype=np.int64)
    last_page_len = np.asarray(last_page_len, dtype=np.int64)
    n = page_indptr[1:] - page_indptr[:-1]
    return np.where(n > 0, (n - 1) * page_size + last_page_len, 0)


def gather_kv(cache_bits: np.ndarray, layout: str, page_indptr, page_indices,
              b: int, kv_head: int, kv_len: int, page_size: int,
              dtype: str = "bf16") -> np.ndarray:
    """Rows 0..kv_len-1 of kv head ``kv_head`` of request ``b``, in token
    order, as float64 ``[kv_len, d]`` (cache elements of ``dtype``)."""
    t = np.arange(kv_len, dtype=np.int64)
    pages = np.asarray(page_indices, dtype=np.int64)[int(page_indptr[b]) + t // page_size]
    slots = t % page_size
    if layout == NHD:      # [page][slot][head][dim]
        rows = cache_bits[pages, slots, kv_head, :]
    elif layout == HND:    # [page][head][slot][dim]
        rows = cache_bits[pages, kv_head, slots, :]
    else:
        raise ValueError(layout)
    return to_f64(rows, dtype)


def visible_keys(qo_len: int, kv_len: int, causal: bool, window_left: int = -1) -> np.ndarray:
    """Boolean ``[qo_len, kv_len]``: may query row i see key t?

    Row i stands at key position ``pos = kv_len - qo_len + i`` (bottom-right
    alignment). Causal: ``t <= pos``. A left window (``window_left >= 0``,
    the left half of the ``window_size`` pair of the FlashAttention-3 page's
    varlen call, section 2; -1 = unbounded) also hides ``t < pos -
    window_left``, so a causal row sees at most ``window_left + 1`` keys.
    """
    i = np.arange(qo_len)[:, None]
    t = np.arange(kv_len)[None, :]
    pos = kv_len - qo_len + i
    vis = (t <= pos) if causal else np.ones((qo_len, kv_len), dtype=bool)
    if window_left >= 0:
        vis = vis & (t >= pos - window_left)
    return vis


# --------------------------------------------------------------------------
# the definition
# --------------------------------------------------------------------------

def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float,
                      visible: np.ndarray):
    """Rows of ``softmax(sm_scale * q k^T restricted to visible keys) v``.

    q ``[n, d]``, k/v ``[T, d]``, visible ``[n, T]`` (bool). Returns
    ``o [n, d]`` and ``lse [n]`` (natural log of the sum of exp of the scaled
    visible scores). Rows with nothing visible: o = 0, lse = -inf.
    """
    n, d = q.shape
    o = np.zeros((n, v.shape[1]), dtype=np.float64)
    lse = np.full(n, -np.inf, dtype=np.float64)
    if k.shape[0] == 0:
        return o, lse
    s = sm_scale * (q @ k.T)                                    # [n, T]
    for r in range(n):
        vis = visible[r]
        if not vis.any():
            continue
        sv = s[r, vis]
        m = sv.max()
        z = np.exp(sv - m).sum()
        lse[r] = m + math.log(z)
        w = np.exp(sv - lse[r])                                 # weights, sum to 1
        o[r] = w @ v[vis]
    return o, lse


def batch_attention(q_bits, qo_indptr, k_cache_bits, v_cache_bits, layout: str,
                    page_indptr, page_indices, last_page_len, num_qo_heads: int,
                    num_kv_heads: int, page_size: int, sm_scale: float, causal: bool,
                    requests=None, rows=None, window_left: int = -1, dtype: str = "bf16",
                    kv_dtype: str | None = None, k_scale=1.0, v_scale=1.0):
    """Paged attention for a packed batch.

    q_bits ``[sum qo_len, Hq, d]`` bit patterns of ``dtype`` ("bf16" or
    "fp16"); caches as laid out by ``layout``, of ``kv_dtype`` (default:
    ``dtype``; "e4m3" for an FP8 cache). A quantised cache holds K / k_scale
    and V / v_scale: the keys and values attended to are ``k_scale`` and
    ``v_scale`` times the stored ones. Either scale is one number for the
    whole cache or a sequence of ``num_kv_heads`` numbers, one per kv head.
    Returns ``out [sum qo_len, Hq, d]`` and ``lse [sum qo_len, Hq]`` in
    float64. ``requests`` limits the work to some requests (other rows stay
    NaN); ``rows`` maps a request to the list of its row indices to compute
    (for sampled checks of large batches); ``window_left`` as in
    ``visible_keys``.
    """
    if num_qo_heads % num_kv_heads:
        raise ValueError("num_qo_heads must be a multiple of num_kv_heads")
    group = num_qo_heads // num_kv_heads
    qo_indptr = np.asarray(qo_indptr, dtype=np.int64)
    kv_len = kv_lengths(page_indptr, last_page_len, page_size)
    total, _, d = q_bits.shape
    out = np.full((total, num_qo_heads, d), np.nan)
    lse = np.full((total, num_qo_heads), np.nan)
    B = len(qo_indptr) - 1
    for b in (range(B) if requests is None else requests):
        q0, q1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
        qo_len = q1 - q0
        if qo_len == 0:
            continue
        sel = np.arange(qo_len) if rows is None or b not in rows else np.asarray(rows[b])
        vis = visible_keys(qo_len, int(kv_len[b]), causal, window_left)[sel]
        for kh in range(num_kv_heads):
            ks = float(k_scale[kh]) if np.ndim(k_scale) else float(k_scale)
            vs = float(v_scale[kh]) if np.ndim(v_scale) else float(v_scale)
            k = ks * gather_kv(k_cache_bits, layout, page_indptr, page_indices, b, kh,
                               int(kv_len[b]), page_size, kv_dtype or dtype)
            v = vs * gather_kv(v_cache_bits, layout, page_indptr, page_indices, b, kh,
                               int(kv_len[b]), page_size, kv_dtype or dtype)
            for h in range(kh * group, (kh + 1) * group):
                qh = to_f64(q_bits[q0 + sel, h, :], dtype)
                o, l = softmax_attention(qh, k, v, sm_scale, vis)
                out[q0 + sel, h] = o
                lse[q0 + sel, h] = l
    return out, lse


def batch_decode(q_bits, k_cache_bits, v_cache_bits, layout: str, page_indptr,
                 page_indices, last_page_len, num_qo_heads: int, num_kv_heads: int,
                 page_size: int, sm_scale: float, requests=None, window_left: int = -1,
                 dtype: str = "bf16", kv_dtype: str | None = None, k_scale=1.0,
                 v_scale=1.0):
    """One query token per request: q_bits ``[B, Hq, d]``; out ``[B, Hq, d]``,
    lse ``[B, Hq]``. Every key of the request is visible, or with a left
    window only the last ``window_left + 1``."""
    B = q_bits.shape[0]
    return batch_attention(q_bits, np.arange(B + 1), k_cache_bits, v_cache_bits, layout,
                           page_indptr, page_indices, last_page_len, num_qo_heads,
                           num_kv_heads, page_size, sm_scale, False, requests=requests,
                           window_left=window_left, dtype=dtype, kv_dtype=kv_dtype,
                           k_scale=k_scale, v_scale=v_scale)


# --------------------------------------------------------------------------
# restatements used as cross-checks
# --------------------------------------------------------------------------

def online_softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float,
                             visible: np.ndarray, chunk: int):
    """The streaming form: keys in chunks of ``chunk``; a running max ``m``,
    running denominator ``l`` and unnormalised accumulator are rescaled by
    ``exp(m_old - m_new)`` whenever the max grows; one division at the end."""
    n, d = q.shape
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    acc = np.zeros((n, v.shape[1]))
    for c0 in range(0, k.shape[0], chunk):
        c1 = min(c0 + chunk, k.shape[0])
        s = sm_scale * (q @ k[c0:c1].T)
        s = np.where(visible[:, c0:c1], s, -np.inf)
        m_new = np.maximum(m, s.max(axis=1))
        # a row that has seen no visible key yet keeps m = -inf; measure from 0
        # instead so that exp() never sees (-inf) - (-inf)
        ref = np.where(np.isneginf(m_new), 0.0, m_new)
        alpha = np.exp(m - ref)
        p = np.exp(s - ref[:, None])
        l = l * alpha + p.sum(axis=1)
        acc = acc * alpha[:, None] + p @ v[c0:c1]
        m = m_new
    o = np.zeros_like(acc)
    lse = np.full(n, -np.inf)
    ok = l > 0
    o[ok] = acc[ok] / l[ok, None]
    lse[ok] = m[ok] + np.log(l[ok])
    return o, lse


def split_kv_states(q, k, v, sm_scale: float, visible, boundaries):
    """Attention of q over each key range ``[boundaries[j], boundaries[j+1])``
    on its own: the partial states (o_j, lse_j) of split-KV."""
    os_, ls_ = [], []
    for a, b in zip(boundaries[:-1], boundaries[1:]):
        o, l = softmax_attention(q, k[a:b], v[a:b], sm_scale, visible[:, a:b])
        os_.append(o)
        ls_.append(l)
    return np.stack(os_), np.stack(ls_)


def merge_states(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Combine partial states over disjoint key sets.

    o_parts ``[S, ..., d]``, lse_parts ``[S, ...]``. With ``M = max_j lse_j``
    and ``w_j = exp(lse_j - M)``: ``o = sum_j w_j o_j / sum_j w_j``,
    ``lse = M + log sum_j w_j``. A part with lse = -inf weighs nothing; if
    every part is -inf the result is o = 0, lse = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    M = lse_parts.max(axis=0)
    empty = np.isneginf(M)
    Ms = np.where(empty, 0.0, M)
    w = np.where(np.isneginf(lse_parts), 0.0, np.exp(lse_parts - Ms))
    sw = w.sum(axis=0)
    o = np.where(empty[..., None], 0.0,
                 (w[..., None] * o_parts).sum(axis=0) / np.where(empty, 1.0, sw)[..., None])
    lse = np.where(empty, -np.inf, Ms + np.log(np.where(empty, 1.0, sw)))
    return o, lse


def masked_attention(q, k, v, sm_scale: float, mask: np.ndarray):
    """``softmax(sm_scale * q k^T + mask) v`` for an explicit additive mask
    whose entries are 0 or -inf. Fully masked rows give o = 0, lse = -inf."""
    s = sm_scale * (q @ k.T) + mask
    n = q.shape[0]
    o = np.zeros((n, v.shape[1]))
    lse = np.full(n, -np.inf)
    for r in range(n):
        if np.all(np.isneginf(s[r])):
            continue
        m = s[r].max()
        e = np.exp(s[r] - m)
        lse[r] = m + math.log(e.sum())
        o[r] = (e / e.sum()) @ v
    return o, lse


def causal_mask(qo_len: int, kv_len: int) -> np.ndarray:
    """Additive bottom-right causal mask: 0 where row i may see key t, -inf else."""
    m = np.zeros((qo_len, kv_len))
    for i in range(qo_len):
        m[i, max(0, kv_len - qo_len + i + 1):] = -np.inf
    return m
