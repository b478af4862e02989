"""The host side of __graft_entry__.smoke(): every case builds, plans in
the mode the device run uses, and the oracle gives finite results for it;
the 70B-ratio prefill case plans work the two-tile kernel takes (an even
group at head_dim 128, query heads in adjacent pairs)."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import __graft_entry__ as entry  # noqa: E402
import oracle  # noqa: E402
from paged_kv_attention_27_gb300 import binding as B  # noqa: E402
from paged_kv_attention_27_gb300.device import plan_options  # noqa: E402

from ._gpu import ensure_built  # noqa: E402


def test_smoke_cases_plan_and_have_finite_oracle_results():
    ensure_built()
    cases = entry.smoke_cases()
    assert len(cases) == 3
    for b in cases:
        decode = b.is_decode and not b.causal
        p = B.fi_plan(B.FI_MODE_DECODE if decode else B.FI_MODE_PREFILL, b.batch,
                      None if decode else b.qo_indptr, b.page_indptr, b.last_page_len,
                      b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.causal,
                      plan_options(b), 152)
        info = B.fi_plan_get_info(p)
        assert info["num_items"] > 0
        o, l = oracle.batch_attention(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.layout,
                                      b.page_indptr, b.page_indices, b.last_page_len,
                                      b.num_qo_heads, b.num_kv_heads, b.page_size, b.sm_scale,
                                      b.causal)
        assert o.shape == (int(b.qo_indptr[-1]), b.num_qo_heads, b.head_dim)
        assert np.isfinite(o).all() and np.isfinite(l).all()
    gqa = cases[2]
    g = gqa.num_qo_heads // gqa.num_kv_heads
    assert (gqa.head_dim, g, gqa.causal) == (128, 8, True)
    p = B.fi_plan(B.FI_MODE_PREFILL, gqa.batch, gqa.qo_indptr, gqa.page_indptr,
                  gqa.last_page_len, gqa.num_qo_heads, gqa.num_kv_heads, gqa.head_dim,
                  gqa.page_size, True, None, 152)
    info = B.fi_plan_get_info(p)
    assert info["num_decode_items"] == 0 and info["num_prefill_items"] % 2 == 0
    items = B.fi_plan_get_work(p)
    heads = items[:, 1]
    assert np.all(heads[0::2] % 2 == 0) and np.all(heads[1::2] == heads[0::2] + 1)
