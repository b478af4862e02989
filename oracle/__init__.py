"""fp64 CPU oracle for paged-KV attention.

TEST INFRASTRUCTURE, not part of the library: only ``tests/``, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` import it. It
shares no code with the CUDA path. Every function cites the passage of the
source pages it restates; see ``oracle.attention``.
"""
from .attention import (  # noqa: F401
    HND, NHD, batch_attention, batch_decode, bf16_to_f64, causal_mask, e4m3_to_f64, f16_to_f64,
    gather_kv,
    kv_lengths, masked_attention, merge_states, online_softmax_attention,
    softmax_attention, split_kv_states, to_f64, visible_keys,
)
