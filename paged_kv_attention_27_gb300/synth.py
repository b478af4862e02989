"""Seeded synthetic paged-KV batches: the one input source shared by the oracle
side and the CUDA side of every test and of the benchmark.

This module builds inputs only. It holds none of the attention arithmetic:
no scores, no softmax, no merge. Everything it returns is plain numpy:

* values are standard normal draws from numpy's counter-based Philox
  generator, rounded to bf16 or fp16 (round-to-nearest-even) and stored as
  raw ``uint16`` bit patterns;
* the page table is the CSR triple ``page_indptr`` / ``page_indices`` /
  ``last_page_len`` of a paged KV cache (pages of ``page_size`` token slots,
  allocated on demand, "FlashInfer kernel library deep-dive", section
  "PageAttention"), with the physical pages handed out in a seeded random
  order so that no request's pages are contiguous;
* the two cache layouts are named as on that page (section "KV cache layout"):
  NHD = ``[page][slot][kv_head][dim]``, HND = ``[page][kv_head][slot][dim]``;
* query rows of all requests are packed back to back (``qo_indptr``), the
  variable-length form with prefix-sum offsets used by the varlen prefill
  wrapper in "FlashAttention-3 kernel integration in inference engines",
  section 2.

The workload builders at the bottom give the shapes of the pages' workloads
(Llama-7B and Llama2-70B head shapes, 1K-32K contexts); no model weights or
datasets are involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

NHD = "NHD"
HND = "HND"


def philox(seed: int) -> np.random.Generator:
    """numpy Generator over the Philox-4x64 counter-based bit generator."""
    return np.random.Generator(np.random.Philox(key=int(seed)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even).

    Returns the bf16 bit patterns as uint16. NaN stays a quiet NaN.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE fp16 (numpy's conversion: round to
    nearest, ties to even; overflow to inf). Returns uint16 bit patterns."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _e4m3_grid() -> np.ndarray:
    """The 127 non-negative finite FP8 E4M3 values, indexed by their code
    (0x00..0x7E): 2^-6 * m/8 for exponent field 0, 2^(e-7) * (1 + m/8) else."""
    codes = np.arange(127)
    e, m = codes >> 3, codes & 7
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e - 7.0))


_E4M3 = _e4m3_grid()


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to FP8 E4M3 (nearest, ties to the even code),
    saturating at +-448; NaN becomes 0x7F. Returns uint8 codes."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(_E4M3, a, side="left"), 1, 126)   # _E4M3[hi-1] < a <= _E4M3[hi]
    lo = hi - 1
    dlo, dhi = a - _E4M3[lo], _E4M3[hi] - a
    code = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a <= 0, 0, code)
    out = (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)
    out[np.isnan(x)] = 0x7F
    return out


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> bit patterns of ``dtype`` ("bf16" or "fp16")."""
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "fp16":
        return f32_to_f16_bits(x)
    if dtype == "e4m3":
        return f32_to_e4m3_bits(x)
    raise ValueError(dtype)


QNAN_BITS = {"bf16": 0x7FC0, "fp16": 0x7E00, "e4m3": 0x7F}

_CHUNK = 1 << 22


def normal_bf16(seed: int, stream: int, shape, dtype: str = "bf16",
                scale: float = 1.0, axis_scale=None) -> np.ndarray:
    """Standard normal values (times ``scale``) of ``shape`` as bit patterns
    of ``dtype``: bf16 (default) or fp16 as uint16, e4m3 as uint8.
    ``axis_scale`` = (axis, factors): the values at index i along ``axis``
    are also multiplied by factors[i] (per-head scales of a cache).

    Element block j (of 2^22 elements) is drawn from its own Philox stream
    keyed by (seed, stream, j), so the values do not depend on how many
    threads fill the array; blocks are filled in parallel.
    """
    import concurrent.futures as cf
    import os
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint8 if dtype == "e4m3" else np.uint16)
    if axis_scale is not None:
        axis, factors = axis_scale
        inner = int(np.prod(shape[axis + 1:], dtype=np.int64))
        factors = np.asarray(factors, dtype=np.float32)

    def fill(j):
        s = j * _CHUNK
        c = min(_CHUNK, n - s)
        g = np.random.Generator(np.random.Philox(key=[int(seed) * 64 + int(stream), j]))
        x = g.standard_normal(c, dtype=np.float32)
        if scale != 1.0:
            x = x * np.float32(scale)
        if axis_scale is not None:
            idx = (np.arange(s, s + c, dtype=np.int64) // inner) % shape[axis]
            x = x * factors[idx]
        out[s:s + c] = to_bits(x, dtype)

    blocks = range((n + _CHUNK - 1) // _CHUNK)
    with cf.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, blocks))
    return out.reshape(shape)


@dataclass
class PagedBatch:
    """One batch of requests over a paged KV cache (all arrays host numpy)."""

    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    layout: str                  # NHD or HND
    sm_scale: float
    causal: bool
    kv_lens: np.ndarray          # int64 [B]   (what the page table encodes)
    qo_lens: np.ndarray          # int64 [B]
    qo_indptr: np.ndarray        # int32 [B+1]
    page_indptr: np.ndarray      # int32 [B+1]
    page_indices: np.ndarray     # int32 [nnz]
    last_page_len: np.ndarray    # int32 [B]
    q: np.ndarray                # uint16 bf16 bits [sum qo, Hq, d]
    k_cache: np.ndarray          # uint16 bf16 bits, layout-dependent 4-D
    v_cache: np.ndarray
    shared_prefix_pages: int = 0
    meta: dict = field(default_factory=dict)
    window_left: int = -1        # left attention window (-1 = unbounded)
    dtype: str = "bf16"          # element type of q and out ("bf16" or "fp16")
    kv_dtype: str = ""           # element type of the caches ("" = dtype; "e4m3")
    k_scale: float = 1.0         # attended keys / values = scale * stored ones
    v_scale: float = 1.0
    cascade: bool = False        # plan the shared prefix as one group (shared-prefix decode)
    # per-kv-head factors on top of k_scale / v_scale (float32 [Hkv]; None = 1)
    k_head_scale: np.ndarray | None = None
    v_head_scale: np.ndarray | None = None

    @property
    def k_scales(self):
        """The key scale the oracle applies: one number, or one per kv head."""
        if self.k_head_scale is None:
            return self.k_scale
        return self.k_scale * self.k_head_scale.astype(np.float64)

    @property
    def v_scales(self):
        if self.v_head_scale is None:
            return self.v_scale
        return self.v_scale * self.v_head_scale.astype(np.float64)

    @property
    def cache_dtype(self) -> str:
        return self.kv_dtype or self.dtype

    @property
    def batch(self) -> int:
        return int(self.kv_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def is_decode(self) -> bool:
        return bool(np.all(self.qo_lens == 1))


def make_batch(name: str, kv_lens, qo_lens, num_qo_heads: int, num_kv_heads: int,
               head_dim: int, page_size: int, layout: str, sm_scale: float | None,
               causal: bool, seed: int, shared_prefix_requests: int = 0,
               shared_prefix_tokens: int = 0, tail_fill: str = "normal",
               extra_pages: int = 0, window_left: int = -1,
               dtype: str = "bf16", kv_dtype: str = "", kv_scale: float = 1.0,
               head_scales=None) -> PagedBatch:
    """Build a paged batch with seeded values and a shuffled page table.

    ``shared_prefix_requests`` requests (the first ones) map their first
    ``shared_prefix_tokens // page_size`` logical pages onto the same physical
    pages. ``tail_fill`` chooses what sits in the unused slots of every last
    page: "normal" (more random values) or "nan" (quiet NaN bits, to show that
    nothing past ``last_page_len`` is read). ``extra_pages`` physical pages that
    no request uses are added to the pool. ``head_scales`` (two sequences of
    ``num_kv_heads`` factors, for K and V) gives each kv head its own scale on
    top of ``kv_scale``: the cache stores the draws divided by both.
    """
    gen = philox(seed)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    qo_lens = np.asarray(qo_lens, dtype=np.int64)
    B = kv_lens.shape[0]
    assert qo_lens.shape == (B,)
    P = page_size
    npages = np.where(kv_lens > 0, (kv_lens + P - 1) // P, 0)
    last = np.where(kv_lens > 0, kv_lens - (npages - 1) * P, 0)

    prefix_pages = shared_prefix_tokens // P if shared_prefix_requests else 0
    if prefix_pages:
        assert shared_prefix_tokens % P == 0
        assert np.all(kv_lens[:shared_prefix_requests] >= shared_prefix_tokens)
    own = npages.copy()
    own[:shared_prefix_requests] -= prefix_pages
    num_phys = int(prefix_pages + own.sum()) + int(extra_pages)
    perm = gen.permutation(num_phys).astype(np.int32)

    page_lists = []
    cursor = prefix_pages
    for b in range(B):
        pl = []
        if b < shared_prefix_requests and prefix_pages:
            pl.extend(perm[:prefix_pages].tolist())
        pl.extend(perm[cursor:cursor + own[b]].tolist())
        cursor += int(own[b])
        page_lists.append(pl)
    page_indptr = np.zeros(B + 1, dtype=np.int32)
    page_indptr[1:] = np.cumsum([len(p) for p in page_lists])
    page_indices = np.array([p for pl in page_lists for p in pl], dtype=np.int32)
    qo_indptr = np.zeros(B + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)

    Hkv, d = num_kv_heads, head_dim
    shape = (num_phys, P, Hkv, d) if layout == NHD else (num_phys, Hkv, P, d)
    # an FP8 cache stores the draws divided by the per-tensor scale
    cdt = kv_dtype or dtype
    head_axis = 2 if layout == NHD else 1
    ks_h = vs_h = None
    if head_scales is not None:
        ks_h = np.asarray(head_scales[0], dtype=np.float32)
        vs_h = np.asarray(head_scales[1], dtype=np.float32)
        assert ks_h.shape == (Hkv,) and vs_h.shape == (Hkv,)
    k_cache = normal_bf16(seed, 1, shape, cdt, 1.0 / kv_scale,
                          None if ks_h is None else (head_axis, 1.0 / ks_h))
    v_cache = normal_bf16(seed, 2, shape, cdt, 1.0 / kv_scale,
                          None if vs_h is None else (head_axis, 1.0 / vs_h))
    q = normal_bf16(seed, 3, (int(qo_lens.sum()), num_qo_heads, d), dtype)
    if tail_fill == "nan":
        for b in range(B):
            if npages[b] == 0 or last[b] == P:
                continue
            p = page_lists[b][-1]
            for cache in (k_cache, v_cache):
                if layout == NHD:
                    cache[p, last[b]:, :, :] = QNAN_BITS[cdt]
                else:
                    cache[p, :, last[b]:, :] = QNAN_BITS[cdt]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    return PagedBatch(name=name, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, page_size=P, layout=layout, sm_scale=float(sm_scale),
                      causal=bool(causal), kv_lens=kv_lens, qo_lens=qo_lens, qo_indptr=qo_indptr,
                      page_indptr=page_indptr, page_indices=page_indices,
                      last_page_len=last.astype(np.int32), q=q, k_cache=k_cache, v_cache=v_cache,
                      shared_prefix_pages=int(prefix_pages),
                      meta={"seed": seed, "shared_prefix_requests": shared_prefix_requests},
                      window_left=int(window_left), dtype=dtype, kv_dtype=kv_dtype,
                      k_scale=float(kv_scale), v_scale=float(kv_scale),
                      k_head_scale=ks_h, v_head_scale=vs_h)


# ----------------------------------------------------------------------------
# Workloads shaped like the pages' (head shapes of Llama-7B / Llama2-70B,
# contexts from 1K to 32K).
# ----------------------------------------------------------------------------

def tiny_decode(seed: int = 0) -> PagedBatch:
    """4 requests, 8 q / 2 kv heads, d=64, P=16, KV lengths {1,17,64,100}, NHD, scale 1/8."""
    return make_batch("tiny batch decode B4 Hq8 Hkv2 d64 P16 kv{1,17,64,100} NHD",
                      [1, 17, 64, 100], [1, 1, 1, 1], 8, 2, 64, 16, NHD, 1.0 / 8, False, seed)


def _fp8_scale(kv_dtype: str) -> float:
    # an FP8 cache stores N(0,1) draws times 16 (|x| < 448 for any practical
    # draw), so that the small values keep their 3 mantissa bits
    return 1.0 / 16 if kv_dtype == "e4m3" else 1.0


def fp8_head_scales(num_kv_heads: int, kv_dtype: str):
    """Per-kv-head K and V factors of the synthetic FP8 caches: powers of two
    from 1/2 to 2 in a fixed pattern (K and V differ), so that every head is
    quantised on its own scale; None for 16-bit caches."""
    if kv_dtype != "e4m3":
        return None
    h = np.arange(num_kv_heads)
    return (2.0 ** ((h % 3) - 1), 2.0 ** (((h + 1) % 3) - 1))


def llama7b_decode(seed: int = 1, batch: int = 64, dtype: str = "bf16",
                   kv_dtype: str = "") -> PagedBatch:
    """Llama-7B-shaped decode: 32/32 heads, d=128, P=16, KV ~ U[512,4096], NHD."""
    g = philox(seed + 1000)
    kv = g.integers(512, 4097, size=batch)
    tname = ("" if dtype == "bf16" else f" {dtype}") + (f" {kv_dtype} cache" if kv_dtype else "")
    return make_batch(f"Llama-7B-shaped batch decode B{batch} Hq32 Hkv32 d128 P16 kv~U[512,4096] "
                      f"NHD{tname}",
                      kv, np.ones(batch, np.int64), 32, 32, 128, 16, NHD, None, False, seed,
                      dtype=dtype, kv_dtype=kv_dtype, kv_scale=_fp8_scale(kv_dtype),
                      head_scales=fp8_head_scales(32, kv_dtype))


def lognormal_lengths(gen, n, median=2048, sigma=1.0, lo=1, hi=32768):
    x = np.exp(math.log(median) + sigma * gen.standard_normal(n))
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def llama70b_gqa_decode(seed: int = 2, batch: int = 128, shared: int = 32,
                        window_left: int = -1, kv_dtype: str = "") -> PagedBatch:
    """Llama2-70B-shaped GQA decode: 64/8 heads, d=128, P=16, HND,
    KV ~ lognormal(median 2048, sigma 1) clipped to [1,32768]; the first 32
    requests share the physical pages of one 1024-token prefix. Optionally a
    left window of ``window_left`` keys."""
    g = philox(seed + 1000)
    kv = lognormal_lengths(g, batch)
    kv[:shared] = np.maximum(kv[:shared], 1024)
    wname = f" window {window_left + 1}" if window_left >= 0 else ""
    wname += f" {kv_dtype} cache" if kv_dtype else ""
    return make_batch(f"Llama2-70B-shaped GQA decode B{batch} Hq64 Hkv8 d128 P16 HND lognormal(2048) "
                      f"{shared} share a 1024-token prefix{wname}",
                      kv, np.ones(batch, np.int64), 64, 8, 128, 16, HND, None, False, seed,
                      shared_prefix_requests=shared, shared_prefix_tokens=1024,
                      window_left=window_left, kv_dtype=kv_dtype,
                      kv_scale=_fp8_scale(kv_dtype), head_scales=fp8_head_scales(8, kv_dtype))


def gqa_decode_d256(seed: int = 9, batch: int = 64) -> PagedBatch:
    """GQA decode at the mixed batch's head_dim with a Llama2-70B-style group:
    64 q / 8 kv heads (8 per kv head), head_dim 256, P=32, HND, KV ~ U[1,32768]
    (the decode rows' length distribution of the mixed batch)."""
    g = philox(seed + 1000)
    kv = g.integers(1, 32769, size=batch)
    return make_batch(f"GQA decode d256 B{batch} Hq64 Hkv8 P32 HND kv~U[1,32K]",
                      kv, np.ones(batch, np.int64), 64, 8, 256, 32, HND, None, False, seed)


def shared_prefix_decode(seed: int = 7, batch: int = 64, prefix_tokens: int = 32768,
                         cascade: bool = True) -> PagedBatch:
    """Decode of ``batch`` requests that share one long prefix (a system
    prompt or document, ``prefix_tokens`` tokens on the same physical pages)
    followed by their own U[1, 2048] tokens; Llama2-70B head shape (64/8,
    d=128, P=16, HND). ``cascade`` plans the prefix as one shared-prefix
    group."""
    g = philox(seed + 1000)
    kv = prefix_tokens + g.integers(1, 2049, size=batch)
    b = make_batch(f"shared-prefix decode B{batch} prefix {prefix_tokens} + U[1,2048] Hq64 Hkv8 "
                   f"d128 P16 HND{' (cascade)' if cascade else ' (flat)'}",
                   kv, np.ones(batch, np.int64), 64, 8, 128, 16, HND, None, False, seed,
                   shared_prefix_requests=batch, shared_prefix_tokens=prefix_tokens)
    b.cascade = cascade
    return b


def causal_prefill(seq_len: int, batch: int = 8, seed: int = 3,
                   window_left: int = -1, dtype: str = "bf16") -> PagedBatch:
    """Causal prefill, 70B shape: 64/8 heads, d=128, P=16, qo_len = kv_len =
    seq_len; optionally a left window of ``window_left`` keys."""
    L = np.full(batch, seq_len, np.int64)
    wname = f" window {window_left + 1}" if window_left >= 0 else ""
    tname = "" if dtype == "bf16" else f" {dtype}"
    return make_batch(f"causal prefill B{batch} L{seq_len} Hq64 Hkv8 d128 P16 NHD{wname}{tname}",
                      L, L, 64, 8, 128, 16, NHD, None, True, seed + seq_len,
                      window_left=window_left, dtype=dtype)


def long_context_chunk(seed: int = 11, batch: int = 1, chunk_len: int = 512,
                       context: int = 32768, num_qo_heads: int = 64) -> PagedBatch:
    """Chunked prefill of a long prompt (8 kv heads, d=128, P=16; 64 query
    heads: the 70B shape, 32: an 8B-class shape): each request appends
    ``chunk_len`` causal rows to a context of ``context`` keys in all (the
    chunk's own keys included)."""
    kv = np.full(batch, context, np.int64)
    qo = np.full(batch, chunk_len, np.int64)
    return make_batch(f"long-context chunk B{batch} {chunk_len} rows on {context} keys "
                      f"Hq{num_qo_heads} Hkv8 d128 P16 NHD", kv, qo, num_qo_heads, 8, 128, 16,
                      NHD, None, True, seed)


def ragged_prefill(seed: int = 4, batch: int = 16) -> PagedBatch:
    """Causal varlen prefill, 70B shape, 16 requests with L ~ U[128,8192]."""
    g = philox(seed + 1000)
    L = g.integers(128, 8193, size=batch)
    return make_batch(f"ragged causal prefill B{batch} L~U[128,8192] Hq64 Hkv8 d128 P16 NHD",
                      L, L, 64, 8, 128, 16, NHD, None, True, seed)


def mixed_chunk_decode(seed: int = 5, chunks: int = 8, decodes: int = 56,
                       chunk_len: int = 512, batch: int | None = None) -> PagedBatch:
    """Chunked prefill + decode in one batch: 16/8 heads, d=256, P=32.

    ``chunks`` requests each append a ``chunk_len``-token causal chunk to an
    existing KV of U[4096,32768] tokens; ``decodes`` requests decode one token
    against KV ~ U[1,32768]. ``batch`` (for smaller profiling cases) sets the
    chunk count and keeps seven decodes per chunk."""
    if batch is not None:
        chunks, decodes = batch, 7 * batch
    g = philox(seed + 1000)
    existing = g.integers(4096, 32769, size=chunks)
    dec_kv = g.integers(1, 32769, size=decodes)
    kv = np.concatenate([existing + chunk_len, dec_kv])
    qo = np.concatenate([np.full(chunks, chunk_len, np.int64), np.ones(decodes, np.int64)])
    return make_batch(f"mixed chunked-prefill+decode {chunks}x{chunk_len}-token chunks on U[4K,32K] "
                      f"+ {decodes} decodes kv~U[1,32K] Hq16 Hkv8 d256 P32 NHD",
                      kv, qo, 16, 8, 256, 32, NHD, None, True, seed)


def small_mixed(seed: int = 6) -> PagedBatch:
    """The mixed batch at a size the oracle finishes in seconds (same shape rules)."""
    g = philox(seed + 1000)
    existing = g.integers(100, 700, size=3)
    dec_kv = g.integers(1, 900, size=5)
    kv = np.concatenate([existing + 96, dec_kv])
    qo = np.concatenate([np.full(3, 96, np.int64), np.ones(5, np.int64)])
    return make_batch("small mixed chunked-prefill+decode Hq16 Hkv8 d256 P32 NHD",
                      kv, qo, 16, 8, 256, 32, NHD, None, True, seed)


def small_gqa_prefill(seed: int = 17) -> PagedBatch:
    """Causal prefill with the 70B head ratio (8 query heads per kv head,
    d = 128, P = 16) at a size the oracle finishes in seconds: three requests
    of 255, 64 and 390 tokens (ragged row tiles, one shorter than a tile)."""
    kv = [255, 64, 390]
    return make_batch("small causal prefill Hq16 Hkv2 d128 P16 NHD", kv, kv, 16, 2, 128, 16,
                      NHD, None, True, seed)


def sub_batch(src: PagedBatch, requests) -> PagedBatch:
    """Copy the listed requests of ``src`` into a compact batch of their own
    (pages renumbered densely, order kept). Used to draw bounded samples."""
    requests = list(requests)
    pages, pl_lens = [], []
    for b in requests:
        lo, hi = int(src.page_indptr[b]), int(src.page_indptr[b + 1])
        pages.extend(src.page_indices[lo:hi].tolist())
        pl_lens.append(hi - lo)
    uniq = sorted(set(pages))
    remap = {p: i for i, p in enumerate(uniq)}
    page_indices = np.array([remap[p] for p in pages], dtype=np.int32)
    page_indptr = np.zeros(len(requests) + 1, np.int32)
    page_indptr[1:] = np.cumsum(pl_lens)
    qo_lens = src.qo_lens[requests]
    qo_indptr = np.zeros(len(requests) + 1, np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)
    q = np.concatenate([src.q[src.qo_indptr[b]:src.qo_indptr[b + 1]] for b in requests], axis=0)
    idx = np.array(uniq, dtype=np.int64)
    return PagedBatch(name=src.name + f" [sample of {len(requests)} requests]",
                      num_qo_heads=src.num_qo_heads, num_kv_heads=src.num_kv_heads,
                      head_dim=src.head_dim, page_size=src.page_size, layout=src.layout,
                      sm_scale=src.sm_scale, causal=src.causal, kv_lens=src.kv_lens[requests].copy(),
                      qo_lens=qo_lens.copy(), qo_indptr=qo_indptr, page_indptr=page_indptr,
                      page_indices=page_indices, last_page_len=src.last_page_len[requests].copy(),
                      q=q, k_cache=src.k_cache[idx], v_cache=src.v_cache[idx],
                      meta=dict(src.meta, sample=requests), window_left=src.window_left,
                      dtype=src.dtype, kv_dtype=src.kv_dtype, k_scale=src.k_scale,
                      v_scale=src.v_scale, k_head_scale=src.k_head_scale,
                      v_head_scale=src.v_head_scale)   # the sample's pages are renumbered: no cascade
