"""Helpers shared by the GPU parity tests: build/load the library, compare
GPU results with the fp64 oracle under the stated tolerances."""
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


def compare(out_gpu, lse_gpu, out_ref, lse_ref, rows=None, what=""):
    """Element-wise comparison on the rows given (all rows if None)."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64) if lse_gpu is not None else None
    if rows is not None:
        o, out_ref = o[rows], out_ref[rows]
        if l is not None:
            l, lse_ref = l[rows], lse_ref[rows]
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - out_ref)
    detail = ""
    if err.max() > OUT_MAX_ABS or err.mean() > OUT_MEAN_ABS:
        # diagnostic: how much of the error is the rounding of the output itself
        from paged_kv_attention_27_gb300.synth import f32_to_bf16_bits
        import torch
        if out_gpu.dtype == torch.float16:
            rounded = out_ref.astype(np.float16).astype(np.float64)
        else:
            rounded = (f32_to_bf16_bits(out_ref.astype(np.float32)).astype(np.uint32) << 16) \
                .view(np.float32).astype(np.float64)
        floor = np.abs(rounded - out_ref)
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
