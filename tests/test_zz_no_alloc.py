"""fi_batch_decode_paged_noalloc against fi_batch_decode_paged and the oracle.

The no-allocation variant serves callers that cannot give the library a
workspace (an engine plugin whose framework owns all device memory, or a hot
loop where cudaMalloc is not acceptable); it keeps its scratch in a static
device array inside libfi.so. This file is named so that pytest collects it
last. Two calls in a row, on different batches (the second one with split-KV
partials in the shared scratch), must each match the workspace entry point
and the fp64 oracle within the parity tolerance; a further call on the same
batch must leave the device's allocations as they were.
"""
import gc

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from paged_kv_attention_27_gb300 import binding as B  # noqa: E402
from paged_kv_attention_27_gb300 import synth  # noqa: E402

from ._gpu import (LSE_MAX_ABS, OUT_MAX_ABS, OUT_MEAN_ABS, compare, ensure_built,  # noqa: E402
                   oracle_parallel)

pytestmark = pytest.mark.gpu


def _both(b):
    from paged_kv_attention_27_gb300.device import DeviceBatch
    db = DeviceBatch(b)
    ref_out, ref_lse = db.run()
    torch.cuda.synchronize()
    assert db.status() == B.FI_OK
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    out = torch.full_like(db.out, float("nan"))
    lse = torch.full_like(db.lse, float("nan"))
    B.fi_batch_decode_paged_noalloc(db.plan, db.q, db.k, db.v, B.LAYOUTS[b.layout], 0,
                                    b.num_pages, db.page_indptr, db.page_indices,
                                    db.last_page_len, b.sm_scale, 1.0, 1.0, out, lse)
    torch.cuda.synchronize()
    return db, out, lse, ref_out, ref_lse


def _close(out, lse, ref_out, ref_lse):
    o = out.float().cpu().numpy().astype(np.float64)
    r = ref_out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o))
    err = np.abs(o - r)
    assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS, (err.max(), err.mean())
    l = lse.cpu().numpy().astype(np.float64)
    rl = ref_lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.abs(l[fin] - rl[fin]).max() <= LSE_MAX_ABS


def test_noalloc_decode_matches_workspace_decode_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    B.lib()
    # call 1: the tiny batch (no splits)
    _, out, lse, ref_out, ref_lse = _both(synth.tiny_decode())
    _close(out, lse, ref_out, ref_lse)
    # call 2: a batch whose long requests are split, so partial states and
    # merge tasks go through the shared static scratch
    b = synth.make_batch("noalloc splits", [20000, 300, 1, 0, 9000], [1] * 5, 32, 8, 128, 16,
                         synth.HND, None, False, 41)
    db, out, lse, ref_out, ref_lse = _both(b)
    assert B.fi_plan_get_info(db.plan)["num_split_requests"] >= 2
    _close(out, lse, ref_out, ref_lse)
    o_ref, l_ref = oracle_parallel(b)
    compare(out, lse, o_ref, l_ref, what="noalloc splits vs oracle")
    # the call exists for callers that cannot allocate: once the kernel is
    # loaded, another call changes neither torch's allocations nor the
    # device's free memory
    # (Python's garbage collector is kept from freeing unrelated tensors
    # meanwhile)
    out2 = torch.full_like(out, float("nan"))
    lse2 = torch.full_like(lse, float("nan"))
    gc.collect()
    gc.disable()
    try:
        torch.cuda.synchronize()
        alloc1 = torch.cuda.memory_allocated()
        free1, _ = torch.cuda.mem_get_info()
        B.fi_batch_decode_paged_noalloc(db.plan, db.q, db.k, db.v, B.LAYOUTS[b.layout], 0,
                                        b.num_pages, db.page_indptr, db.page_indices,
                                        db.last_page_len, b.sm_scale, 1.0, 1.0, out2, lse2)
        torch.cuda.synchronize()
        alloc2 = torch.cuda.memory_allocated()
        free2, _ = torch.cuda.mem_get_info()
    finally:
        gc.enable()
    # nothing grew (torch may release an unrelated cached block meanwhile)
    assert alloc2 <= alloc1, (alloc1, alloc2)
    assert free2 >= free1, (free1, free2)
    assert torch.equal(out2, out) and torch.equal(lse2, lse)   # same plan: bitwise the same


def test_noalloc_rejects_plans_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()
    # 512 requests of 32K tokens planned for a huge SM count: every request is
    # cut into 64 chunks, and the fp32 partials need far more than 16 MiB
    kv = np.full(512, 32768)
    pi = np.zeros(513, np.int32)
    pi[1:] = np.cumsum(np.full(512, 32768 // 32))
    plan = B.fi_plan(B.FI_MODE_DECODE, 512, None, pi, np.full(512, 32, np.int32), 16, 8, 256, 32,
                     0, None, 100000)
    assert plan.workspace_bytes > (16 << 20)
    x = torch.empty(16, device="cuda")
    with pytest.raises(B.FiError) as e:
        B.fi_batch_decode_paged_noalloc(plan, x, x, x, 0, 0, 1, x, x, x, 0.1, 1.0, 1.0, x, None)
    assert e.value.status == B.FI_ERR_WORKSPACE_TOO_SMALL
    del kv
