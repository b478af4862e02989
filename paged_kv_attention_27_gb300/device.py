"""Moving a synthetic PagedBatch to the GPU and calling the C ABI on it.

Marshalling only: numpy bf16 / fp16 bit patterns become torch bfloat16 /
float16 tensors on the device, outputs and the workspace are allocated with
torch, and the calls go through ``binding`` (libfi.so). No attention
arithmetic happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .synth import PagedBatch


TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}
FI_DTYPES = {"bf16": B.FI_DTYPE_BF16, "fp16": B.FI_DTYPE_FP16, "e4m3": B.FI_DTYPE_E4M3}


def bf16_tensor(bits: np.ndarray, device="cuda", dtype: str = "bf16") -> torch.Tensor:
    """Bit patterns of `dtype` -> a torch tensor on `device`: bf16 / fp16
    (uint16 patterns) as torch.bfloat16 / torch.float16, e4m3 (uint8 codes)
    as raw uint8 bytes."""
    if dtype == "e4m3":
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).to(device)
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_DTYPES[dtype])
    return t.to(device)


def i32_tensor(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def plan_options(b: PagedBatch):
    """fi_plan options of a batch (None = the defaults). A batch marked
    `cascade` plans its shared prefix (the first requests' common leading
    pages) as one shared-prefix group."""
    cascade = b.cascade and b.shared_prefix_pages > 0
    if b.window_left < 0 and b.dtype == "bf16" and b.cache_dtype == "bf16" and not cascade:
        return None
    opt = {"window_left": int(b.window_left), "dtype": FI_DTYPES[b.dtype],
           "kv_dtype": FI_DTYPES[b.cache_dtype]}
    if cascade:
        opt["prefix_group_indptr"] = [0, int(b.meta["shared_prefix_requests"])]
        opt["prefix_pages"] = [int(b.shared_prefix_pages)]
    return opt


def num_sms(device="cuda") -> int:
    return torch.cuda.get_device_properties(device).multi_processor_count


class DeviceBatch:
    """A PagedBatch resident on the GPU, with its plan, outputs and workspace."""

    def __init__(self, b: PagedBatch, device="cuda", mode=None, sms=None, lse=True):
        self.b = b
        self.device = device
        self.q = bf16_tensor(b.q, device, b.dtype)
        self.k = bf16_tensor(b.k_cache, device, b.cache_dtype)
        self.v = bf16_tensor(b.v_cache, device, b.cache_dtype)
        self.page_indptr = i32_tensor(b.page_indptr, device)
        self.page_indices = i32_tensor(b.page_indices if b.page_indices.size else np.zeros(1),
                                       device)
        self.last_page_len = i32_tensor(b.last_page_len, device)
        self.qo_indptr = i32_tensor(b.qo_indptr, device)
        # per-kv-head cache scales (device fp32), when the batch has them
        f32 = lambda a: None if a is None else torch.from_numpy(
            np.ascontiguousarray(a, dtype=np.float32)).to(device)
        self.k_head_scale = f32(b.k_head_scale)
        self.v_head_scale = f32(b.v_head_scale)
        if mode is None:
            mode = B.FI_MODE_DECODE if (b.is_decode and not b.causal) else B.FI_MODE_PREFILL
        self.mode = mode
        self.plan = B.fi_plan(mode, b.batch, b.qo_indptr if mode == B.FI_MODE_PREFILL else None,
                              b.page_indptr, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                              b.head_dim, b.page_size, b.causal, plan_options(b),
                              sms or num_sms(device))
        self.workspace = torch.empty(max(self.plan.workspace_bytes, 256), dtype=torch.uint8,
                                     device=device)
        rows = int(b.qo_lens.sum())
        self.out = torch.empty((rows, b.num_qo_heads, b.head_dim), dtype=TORCH_DTYPES[b.dtype],
                               device=device)
        self.lse = torch.empty((rows, b.num_qo_heads), dtype=torch.float32,
                               device=device) if lse else None

    def run(self, stream=None):
        b = self.b
        layout = B.LAYOUTS[b.layout]
        if self.mode == B.FI_MODE_DECODE:
            B.fi_batch_decode_paged(self.plan, self.q, self.k, self.v, layout, 0, b.num_pages,
                                    self.page_indptr, self.page_indices, self.last_page_len,
                                    b.sm_scale, b.k_scale, b.v_scale, self.out, self.lse,
                                    self.workspace, stream=stream, k_head_scale=self.k_head_scale,
                                    v_head_scale=self.v_head_scale)
        else:
            B.fi_batch_prefill_paged(self.plan, self.q, self.qo_indptr, self.k, self.v, layout, 0,
                                     b.num_pages, self.page_indptr, self.page_indices,
                                     self.last_page_len, b.sm_scale, b.k_scale, b.v_scale,
                                     self.out, self.lse, self.workspace, stream=stream,
                                     k_head_scale=self.k_head_scale,
                                     v_head_scale=self.v_head_scale)
        return self.out, self.lse

    def run_host(self, stream=None):
        """The same step through fi_batch_attention_host: q and the page table
        from (pinned) host memory, out and lse back into host memory; returns
        the host (CPU) out and lse tensors. Uses its own workspace with room
        for the call's host-IO part."""
        b = self.b
        info = B.fi_plan_get_info(self.plan)
        ws_bytes = info["workspace_bytes"] + info["host_io_bytes"]
        if getattr(self, "_ws_host", None) is None or self._ws_host.numel() < ws_bytes:
            self._ws_host = torch.empty(max(ws_bytes, 256), dtype=torch.uint8,
                                        device=self.device)
        q_h = self.q.cpu().pin_memory()
        out_h = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        lse_h = (torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()
                 if self.lse is not None else None)
        prefill = self.mode == B.FI_MODE_PREFILL
        B.fi_batch_attention_host(self.plan, q_h,
                                  b.qo_indptr.astype(np.int32) if prefill else None,
                                  self.k, self.v, B.LAYOUTS[b.layout], 0, b.num_pages,
                                  b.page_indptr.astype(np.int32),
                                  b.page_indices.astype(np.int32), b.last_page_len.astype(np.int32),
                                  b.sm_scale, b.k_scale, b.v_scale, out_h, lse_h, self._ws_host,
                                  ws_bytes, stream=stream, k_head_scale=self.k_head_scale,
                                  v_head_scale=self.v_head_scale)
        return out_h, lse_h

    def status(self, stream=None) -> int:
        return B.fi_check_device_status(self.workspace, stream)
