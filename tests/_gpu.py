"""Helpers shared by the GPU parity tests: build/load the library, compare
GPU results with the fp64 oracle under the stated tolerances, and run the
oracle over a batch's requests on a thread pool.

Every comparison also reports the rounding floor: the error of the oracle
itself once rounded to the output type. A kernel cannot get below it, so the
distance between the two shows how much of the budget the kernel's own
arithmetic uses. With FI_PARITY_LOG set to a file path, each comparison
appends one line (what, max and mean error, floor max and mean) to it."""
import concurrent.futures as cf
import os

import numpy as np

# bf16 (or fp16) outputs against the unrounded fp64 oracle; fp32 lse absolute
OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def scale_v(b, factor=0.25):
    """Scale V by a power of two (exact in bf16; in fp16 exact above the
    subnormal range). Rows that average only a few V rows (small windows,
    short contexts) have |o| of a few units, where the bf16 rounding of the
    output alone (half an ulp: 2^-6 at 4) exceeds the max-abs budget; a
    factor of 1/4 keeps |o| in the range the budget is stated for."""
    from paged_kv_attention_27_gb300.synth import to_bits
    if b.dtype == "fp16":
        v = b.v_cache.view(np.float16).astype(np.float32) * np.float32(factor)
    else:
        v = (b.v_cache.astype(np.uint32) << 16).view(np.float32) * np.float32(factor)
    b.v_cache = to_bits(v, b.dtype)
    return b


def ensure_built():
    from paged_kv_attention_27_gb300 import build
    build.build()


def oracle_parallel(b, requests=None, threads=None):
    """oracle.batch_attention over the batch's requests (all, or those
    given), one request per task on a thread pool; rows of other requests
    stay NaN, as in the oracle itself."""
    import oracle
    reqs = list(range(b.batch)) if requests is None else list(requests)
    total, hq, d = b.q.shape
    out = np.full((total, hq, d), np.nan)
    lse = np.full((total, hq), np.nan)

    def one(r):
        o, l = oracle.batch_attention(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.layout,
                                      b.page_indptr, b.page_indices, b.last_page_len,
                                      b.num_qo_heads, b.num_kv_heads, b.page_size, b.sm_scale,
                                      b.causal, requests=[r], window_left=b.window_left,
                                      dtype=b.dtype, kv_dtype=b.cache_dtype, k_scale=b.k_scales,
                                      v_scale=b.v_scales)
        r0, r1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        return r0, r1, o[r0:r1], l[r0:r1]

    with cf.ThreadPoolExecutor(max_workers=threads or os.cpu_count() or 1) as ex:
        for r0, r1, o, l in ex.map(one, reqs):
            out[r0:r1] = o
            lse[r0:r1] = l
    return out, lse


def rounding_floor(out_ref, half: bool):
    """|oracle rounded to the output type - oracle|: bf16 (RNE) or fp16."""
    from paged_kv_attention_27_gb300.synth import f32_to_bf16_bits
    if half:
        rounded = out_ref.astype(np.float16).astype(np.float64)
    else:
        rounded = (f32_to_bf16_bits(out_ref.astype(np.float32)).astype(np.uint32) << 16) \
            .view(np.float32).astype(np.float64)
    return np.abs(rounded - out_ref), rounded


def compare(out_gpu, lse_gpu, out_ref, lse_ref, rows=None, what=""):
    """Element-wise comparison on the rows given (all rows if None)."""
    import torch
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64) if lse_gpu is not None else None
    if rows is not None:
        o, out_ref = o[rows], out_ref[rows]
        if l is not None:
            l, lse_ref = l[rows], lse_ref[rows]
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - out_ref)
    floor, rounded = rounding_floor(out_ref, out_gpu.dtype == torch.float16)
    margin = (f"{what}: max-abs {err.max():.3e} mean-abs {err.mean():.3e} | rounding floor "
              f"max {floor.max():.3e} mean {floor.mean():.3e}")
    print(margin)
    log = os.environ.get("FI_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(margin + "\n")
    detail = ""
    if err.max() > OUT_MAX_ABS or err.mean() > OUT_MEAN_ABS:
        i = np.unravel_index(np.argmax(err), err.shape)
        detail = (f"; worst at {i}: gpu {o[i]:.6f} oracle {out_ref[i]:.6f} "
                  f"(rounded oracle {rounded[i]:.6f}); rounding floor max "
                  f"{floor.max():.3e} mean {floor.mean():.3e}")
    assert err.max() <= OUT_MAX_ABS, f"{what}: max-abs {err.max():.3e}{detail}"
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}{detail}"
    if l is not None:
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(l), inf_ref), f"{what}: -inf lse pattern differs"
        fin = ~inf_ref
        if fin.any():
            le = np.abs(l[fin] - lse_ref[fin])
            assert le.max() <= LSE_MAX_ABS, f"{what}: lse max-abs {le.max():.3e}"
    return float(err.max()), float(err.mean())
