#!/usr/bin/env python3
"""Benchmark of the paged-KV attention path on one GB300 (or N, one rank each).

Default workload: Llama-7B-shaped batch decode (64 requests, 32 q / 32 kv
heads, head_dim 128, page size 16, KV lengths uniform in [512, 4096], NHD,
shuffled page table), the configuration the headline metric is quoted on.
The default line also carries, under "workloads", every other configuration
of the hot path timed the same way (Llama2-70B GQA decode, causal prefill at
1K / 4K / 16K / 32K, the ragged prefill batch and the mixed chunked-prefill +
decode batch), each with its own roofline and clock record.
One step = one pass of the hot path over that batch through the C ABI: the
stream-ordered work-list upload and the decode kernel (which also merges the
partial states of split requests). The plan itself is host work done once per
batch composition; it is inside the end-to-end number (`e2e`), which also
copies the step's inputs from pinned host memory and its outputs back.

Prints one JSON line. `value` is KV bytes read per step (each request's
K and V rows, bf16) over the device time of the step, in GB/s, summed over
ranks. `roofline` compares the decode kernel's own time (CUDA events around
that launch, on its stream) with the measured HBM copy bandwidth.
`cpu_baseline` times the fp64 oracle on a bounded sample of the same batch.

`--impl reference` times the oracle itself (there is no other implementation
to run), on the host cores, each step a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s & prefill TFLOPS on 1 GB300, as % of HBM / bf16 tensor peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 8000.0      # HBM3e data-sheet figure (about 8 TB/s)

# every other configuration of the hot path, timed after the headline on the
# default line: (workload, cap on the timed steps)
SECONDARY = [("llama70b_gqa_decode", 200), ("causal_prefill_1k", 200),
             ("causal_prefill_4k", 100), ("causal_prefill_16k", 30),
             ("causal_prefill_32k", 30), ("ragged_prefill", 60), ("mixed_chunk_decode", 100),
             ("gqa_decode_d256", 100), ("long_context_chunk", 100),
             ("long_context_chunk_hq32", 100)]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama7b_decode", choices=sorted(WORKLOADS))
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other workloads added to the default line")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's request count (smaller profiling cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


WORKLOADS = {
    "llama7b_decode": ("llama7b_decode", {}),
    "llama70b_gqa_decode": ("llama70b_gqa_decode", {}),
    "llama70b_gqa_decode_window4k": ("llama70b_gqa_decode", {"window_left": 4095}),
    "tiny_decode": ("tiny_decode", {}),
    "causal_prefill_1k": ("causal_prefill", {"seq_len": 1024}),
    "causal_prefill_4k": ("causal_prefill", {"seq_len": 4096}),
    "causal_prefill_16k": ("causal_prefill", {"seq_len": 16384}),
    "causal_prefill_32k": ("causal_prefill", {"seq_len": 32768, "batch": 2}),
    "causal_prefill_16k_window4k": ("causal_prefill", {"seq_len": 16384, "window_left": 4095}),
    "causal_prefill_4k_fp16": ("causal_prefill", {"seq_len": 4096, "dtype": "fp16"}),
    "llama7b_decode_fp16": ("llama7b_decode", {"dtype": "fp16"}),
    "llama7b_decode_fp8kv": ("llama7b_decode", {"kv_dtype": "e4m3"}),
    "shared_prefix_decode": ("shared_prefix_decode", {}),
    "shared_prefix_decode_flat": ("shared_prefix_decode", {"cascade": False}),
    "llama70b_gqa_decode_fp8kv": ("llama70b_gqa_decode", {"kv_dtype": "e4m3"}),
    "ragged_prefill": ("ragged_prefill", {}),
    "mixed_chunk_decode": ("mixed_chunk_decode", {}),
    "gqa_decode_d256": ("gqa_decode_d256", {}),
    "long_context_chunk": ("long_context_chunk", {}),
    "long_context_chunk_hq32": ("long_context_chunk", {"num_qo_heads": 32}),
}


def make_workload(name, batch=None):
    from paged_kv_attention_27_gb300 import synth
    fn_name, kw = WORKLOADS[name]
    kw = dict(kw)
    if batch is not None:
        kw["batch"] = batch
    return getattr(synth, fn_name)(**kw)


def visible_pairs(b):
    """(query row, key) pairs the mask leaves visible, summed over requests.
    Row i stands at key position pos = kv - qo + i; causal rows see keys up
    to pos, and a left window hides keys below pos - window_left."""
    import numpy as np
    total = 0
    for qo, kv in zip(b.qo_lens.tolist(), b.kv_lens.tolist()):
        pos = kv - qo + np.arange(qo, dtype=np.int64)
        hi = np.minimum(pos, kv - 1) if (b.causal and qo > 1) else np.full(qo, kv - 1)
        lo = np.maximum(0, pos - b.window_left) if b.window_left >= 0 else np.zeros(qo, np.int64)
        total += int(np.maximum(0, hi - lo + 1).sum())
    return total


def attention_flops(b):
    """Causal-triangle FLOPs: 2*d for QK^T plus 2*d for PV per visible pair per head."""
    return 4 * b.head_dim * b.num_qo_heads * visible_pairs(b)


def cache_elem_bytes(b):
    return 1 if b.cache_dtype == "e4m3" else 2


def kv_bytes(b):
    """K+V bytes a pass reads: the rows of K and V that some query row of a
    request may see (all kv_len of them without a left window), for every
    kv head (bf16). A page slot shared by several requests counts once."""
    seen = set()
    for r in range(b.batch):
        kv, qo = int(b.kv_lens[r]), int(b.qo_lens[r])
        first = max(0, kv - qo - b.window_left) if b.window_left >= 0 else 0
        lo = int(b.page_indptr[r])
        for t in range(first, kv):
            seen.add((int(b.page_indices[lo + t // b.page_size]), t % b.page_size))
    return len(seen) * 2 * b.num_kv_heads * b.head_dim * cache_elem_bytes(b)


def io_bytes(b):
    """q + out (bf16) + lse (fp32) bytes of a pass."""
    rows = int(b.qo_lens.sum())
    return rows * b.num_qo_heads * (b.head_dim * 2 * 2 + 4)


KERNEL_SOURCES = {
    "decode_kernel": ["decode.cu", "decode_roles.cuh", "ptx.cuh", "kernels.cuh", "fi_internal.h"],
    "prefill_kernel": ["prefill.cu", "decode_roles.cuh", "ptx.cuh", "kernels.cuh",
                       "fi_internal.h"],
    "mixed_kernel": ["prefill.cu", "decode_roles.cuh", "ptx.cuh", "kernels.cuh",
                     "fi_internal.h"],
    "prefill_pair_kernel": ["prefill_pair.cu", "ptx.cuh", "kernels.cuh", "fi_internal.h"],
    "merge_kernel": ["merge.cu", "kernels.cuh", "fi_internal.h"],
}


def source_digest(kernel):
    """Hash of the sources a kernel is compiled from, blind to comments and
    whitespace (re-indenting a file or rewording a comment does not change the
    kernel its counters describe; the hashed files hold no comment markers
    inside string literals)."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_attention_27_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        src = open(os.path.join(csrc, f), "rb").read()
        src = re.sub(rb"/\*.*?\*/", b"", src, flags=re.S)
        src = re.sub(rb"//[^\n]*", b"", src)
        h.update(re.sub(rb"\s+", b"", src))
    return h.hexdigest()[:16]


def committed_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    e = d.get(f"{workload}:{kernel}")
    if not e or e.get("source_digest") != source_digest(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None
        self.windows = []       # (t0, t1) of every timed region, in order

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._reader, daemon=True).start()

    def _reader(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        self.windows.append((self.t0, self.t1))

    def stop(self):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, window_index=-1):
        """Clocks over one timed region (the last by default); the whole run
        when no sample fell inside it."""
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        t0, t1 = self.windows[window_index] if self.windows else (None, None)
        inside = [s for t, s in self.samples if t0 and t1 and t0 - 0.1 <= t <= t1 + 0.1]
        window = "timed region"
        if not inside:
            inside = [s for _, s in self.samples]
            window = "whole run (timed region shorter than the 100 ms sampling period)"
        sm = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ----------------------------------------------------------------------------

def oracle_sample(b, budget_s=12.0, threads=None):
    """Run the fp64 oracle request by request (a thread pool over requests,
    in batch order) until about `budget_s` of wall time has passed. Returns
    (KV GB/s over the completed requests, seconds, threads, requests done)."""
    import oracle
    threads = threads or (os.cpu_count() or 1)

    def one(r):
        oracle.batch_attention(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.layout, b.page_indptr,
                               b.page_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                               b.page_size, b.sm_scale, b.causal, requests=[r],
                               window_left=b.window_left, dtype=b.dtype,
                               kv_dtype=b.cache_dtype, k_scale=b.k_scales, v_scale=b.v_scales)
        return r

    done = []
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        pending = set()
        nxt = 0
        while nxt < b.batch and len(pending) < threads:
            pending.add(ex.submit(one, nxt))
            nxt += 1
        while pending:
            fin, pending = cf.wait(pending, return_when=cf.FIRST_COMPLETED)
            done.extend(f.result() for f in fin)
            if nxt < b.batch and time.perf_counter() - t0 < budget_s:
                pending.add(ex.submit(one, nxt))
                nxt += 1
    dt = time.perf_counter() - t0
    w = b.window_left
    keys = [int(b.kv_lens[r]) if w < 0 else min(int(b.kv_lens[r]), w + 1) for r in done]
    kvb = sum(keys) * 2 * b.num_kv_heads * b.head_dim * cache_elem_bytes(b)
    return kvb / dt / 1e9, dt, threads, sorted(done)


def run_reference(args, rank, world, budget_s=150.0):
    """The oracle as the reference arm, on the host cores. One untimed pass
    over the whole batch measures its cost; every step is then the whole
    batch when the K + W steps fit in about `budget_s`, else the first
    requests of the batch in the number that fits."""
    if rank != 0:
        return
    b = make_workload(args.workload, args.batch)
    from paged_kv_attention_27_gb300 import synth
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle_sample(b, budget_s=1e9, threads=threads)
    t_full = time.perf_counter() - t0
    runs = max(1, args.steps + args.warmup - 1)
    if t_full * runs <= budget_s:
        n = b.batch
    else:
        n = max(min(b.batch, threads), int(b.batch * budget_s / (t_full * runs)))
        n = min(n, b.batch)
    sample = list(range(n))
    sb = b if n == b.batch else synth.sub_batch(b, sample)
    for _ in range(args.warmup - 1):
        oracle_sample(sb, budget_s=1e9, threads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_sample(sb, budget_s=1e9, threads=threads)
        times.append(time.perf_counter() - t0)
    kvb = kv_bytes(sb)
    step_s = sum(times) / len(times)
    value = kvb / step_s / 1e9
    if n == b.batch:
        desc = (f"fp64 oracle over the whole batch ({int(sb.kv_lens.sum())} KV tokens per step), "
                f"{threads} threads")
    else:
        desc = (f"fp64 oracle over requests 0..{n - 1} of the batch ({int(sb.kv_lens.sum())} KV "
                f"tokens per step; the whole batch took {t_full:.1f} s, too long for "
                f"{runs + 1} steps), {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(config_of(b, None, kv_bytes(b), attention_flops(b)), sample=desc),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def reduce_max(x, dist, device="cpu"):
    """Max of a per-rank scalar over all ranks (the step time the whole job
    waits for); identity when running alone. Timing plumbing only: no data
    of the attention path crosses ranks."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms_per_step_max):
    """Units per second for the whole job: every rank processes its own batch
    (weak scaling), and the job takes as long as its slowest rank."""
    return units_per_rank * world / (ms_per_step_max / 1e3)


L2_BYTES = 129 * 2**20


def time_steps(db, K, W, dist=None, sampler=None, flush_l2=False):
    """W untimed steps, then K steps bracketed by a barrier and a device
    synchronisation on both sides, timed with CUDA events on the launching
    stream. Returns (ms for the K steps, mean ms of the attention kernels
    alone, from events the library records around them).

    flush_l2: before every timed step, overwrite a buffer twice the L2 size
    so that the step starts with none of its K/V in the L2; the step time is
    then the sum of per-step events around each step alone (the flush is
    not timed)."""
    import torch
    from paged_kv_attention_27_gb300 import binding as B

    stream = torch.cuda.current_stream()
    for _ in range(max(W, 1)):
        db.run()
    torch.cuda.synchronize()
    st = db.status()
    assert st == B.FI_OK, B.status_string(st)
    ks = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ss = [torch.cuda.Event(enable_timing=True) for _ in range(K)] if flush_l2 else []
    se = [torch.cuda.Event(enable_timing=True) for _ in range(K)] if flush_l2 else []
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    for ev in ks + ke + ss + se:   # create the CUDA events (torch creates them on first record)
        ev.record(stream)
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=db.device) \
        if flush_l2 else None
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    t_start.record(stream)
    for i in range(K):
        if flush_l2:
            scrub.fill_(float(i))
            ss[i].record(stream)
        B.fi_profile_next_launch(ks[i], ke[i])
        db.run()
        if flush_l2:
            se[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    if dist:
        dist.barrier()
    st = db.status()
    assert st == B.FI_OK, B.status_string(st)
    if flush_l2:
        ms_total = sum(a.elapsed_time(e) for a, e in zip(ss, se))
    else:
        ms_total = t_start.elapsed_time(t_end)
    kern_ms = sum(a.elapsed_time(e) for a, e in zip(ks, ke)) / K
    ms_total = reduce_max(ms_total, dist, "cuda")
    return ms_total, kern_ms


def config_of(b, info, kvb, flops):
    """The JSON line's config: the workload and its sizes (and, with a plan
    summary, the plan's work split)."""
    cfg = {"workload": b.name, "batch": b.batch, "num_qo_heads": b.num_qo_heads,
            "num_kv_heads": b.num_kv_heads, "head_dim": b.head_dim, "page_size": b.page_size,
            "layout": b.layout, "causal": b.causal, "kv_tokens": int(b.kv_lens.sum()),
            "q_rows": int(b.qo_lens.sum()), "kv_bytes_per_step": kvb,
            "attention_flops_per_step": flops, "io_bytes_per_step": io_bytes(b),
            "l2": (f"inputs larger than L2 ({(kvb + io_bytes(b)) / 1e9:.2f} GB of KV, q and out "
                   "per step vs 129 MB L2): no flush") if kvb > 2 * L2_BYTES else
                  (f"K/V ({kvb / 1e6:.0f} MB) could stay in the 129 MB L2: L2 flushed before "
                   "every timed step (a 258 MB write, not timed)")}
    if info is not None:
        cfg["plan"] = {k: info[k] for k in ("num_decode_items", "num_prefill_items",
                                            "chunk_tokens", "num_split_requests",
                                            "num_partial_slots")}
    return cfg


def roofline_of(b, kvb, flops, kern_ms, kernel_names, workload):
    hbm, bf16, src = peaks()
    try:
        bf16_sus = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
                         ["bf16_tflops_sustained"])
    except Exception:
        bf16_sus = 1700.0
    gbs = kvb / (kern_ms / 1e3) / 1e9
    tfs = flops / (kern_ms / 1e3) / 1e12
    f_hbm, f_tc = gbs / hbm, tfs / bf16_sus
    label = "of measured" if src == "measured" else "of fallback"
    if f_hbm >= f_tc:
        r = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": f_hbm,
             "peak_source": f"hbm_gbs {label} (MEASURED_PEAKS.json)"}
    else:
        r = {"bound": "tensor", "achieved": tfs, "peak": bf16_sus, "unit": "TFLOP/s",
             "frac": f_tc, "peak_source": f"bf16_tflops_sustained {label} (the kernel runs back "
                                          "to back for the whole timed loop)"}
    r["traffic"] = committed_traffic(workload, kernel_names[0]) if kernel_names else None
    r["kernel"] = "+".join(kernel_names)
    r["kernel_ms"] = kern_ms
    r["hbm_frac"] = f_hbm
    r["hbm_frac_of_nominal"] = gbs / NOMINAL_HBM_GBS
    r["tensor_frac"] = f_tc
    return r


def mixed_fused(b, info):
    """Whether a plan's prefill and decode work run as one persistent mixed
    launch (head_dim 256, 1, 2 or 4 query heads per kv head, a 16-bit cache)."""
    g = b.num_qo_heads // b.num_kv_heads
    return (bool(info["num_prefill_items"]) and bool(info["num_decode_items"]) and
            b.head_dim == 256 and g in (1, 2, 4) and b.cache_dtype == b.dtype)


def prefill_split(info):
    """Whether a plan cut its prefill tiles into pieces (a launch of under two
    waves; only plans without decode rows): one merge launch follows."""
    return (bool(info["num_prefill_items"]) and not info["num_decode_items"] and
            info["num_partial_slots"] > 0)


def launches_per_step(b, info):
    if mixed_fused(b, info):
        return 1
    return ((1 if info["num_decode_items"] else 0) + (1 if info["num_prefill_items"] else 0) +
            (1 if prefill_split(info) else 0))


def kernels_of(b, info):
    """The kernels a plan launches (the two-tile prefill kernel takes plain
    prefill work at head_dim 64 and 128 with an even number of query heads
    per kv head; the one-tile kernel the rest; a mixed batch at head_dim 256
    runs as one mixed kernel)."""
    if mixed_fused(b, info):
        return ["mixed_kernel"]
    names = []
    if info["num_prefill_items"]:
        pair = b.head_dim in (64, 128) and (b.num_qo_heads // b.num_kv_heads) % 2 == 0
        names.append("prefill_pair_kernel" if pair else "prefill_kernel")
    if info["num_decode_items"]:
        names.append("decode_kernel")
    if prefill_split(info):
        names.append("merge_kernel")
    return names


def run_ours(args, rank, world, local_rank):
    import torch

    from paged_kv_attention_27_gb300 import binding as B
    from paged_kv_attention_27_gb300 import build as _build
    from paged_kv_attention_27_gb300.device import DeviceBatch

    torch.cuda.set_device(local_rank)
    _build.build()
    B.lib()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    b = make_workload(args.workload, args.batch)
    db = DeviceBatch(b, device=f"cuda:{local_rank}")
    info = B.fi_plan_get_info(db.plan)
    kvb = kv_bytes(b)
    flops = attention_flops(b)

    # CPU baseline first (rank 0, N = 1 only), before the device is busy
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(b)

    from paged_kv_attention_27_gb300.device import num_sms
    plan_host = time_plan(b, num_sms(f"cuda:{local_rank}"))

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    ms_total, kern_ms = time_steps(db, K, args.warmup, dist, sampler,
                                   flush_l2=kvb <= 2 * L2_BYTES)
    clocks = sampler.summary()
    ms_step = ms_total / K
    if info["num_decode_items"]:          # decode or mixed: HBM-bound, KV GB/s
        value, unit = whole_job_rate(kvb, world, ms_step) / 1e9, "GB/s"
    else:                                 # prefill: tensor-bound, TFLOP/s
        value, unit = whole_job_rate(flops, world, ms_step) / 1e12, "TFLOP/s"

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(b, db, K, local_rank, unit)

    workloads = None
    if args.workload == "llama7b_decode" and args.batch is None and not args.no_secondary:
        del db
        torch.cuda.empty_cache()
        workloads = {}
        for name, cap in SECONDARY:
            workloads[name] = measure_secondary(name, max(5, min(K, cap)), max(3, args.warmup),
                                                dist, sampler, world)
            torch.cuda.empty_cache()
    sampler.stop()

    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": b.dtype if b.cache_dtype == b.dtype else f"{b.dtype} (cache {b.cache_dtype})",
        "data": f"synthetic (seeded Philox normals rounded to {b.cache_dtype}, shuffled page table)",
        "config": config_of(b, info, kvb, flops),
        "roofline": roofline_of(b, kvb, flops, kern_ms, kernels_of(b, info), args.workload),
        "tflops": flops * world / (ms_step / 1e3) / 1e12,
        "kv_gbs": kvb * world / (ms_step / 1e3) / 1e9,
        "tokens_per_s": int(b.qo_lens.sum()) * world / (ms_step / 1e3),
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step(b, info) * K,
        "plan_host_us": plan_host,
        "clocks": clocks,
    }
    if workloads:
        line["workloads"] = workloads
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def measure_secondary(workload, K, W, dist, sampler, world):
    """Another configuration of the hot path, timed like the headline (no CPU
    baseline, no e2e): whole-job rate in its own unit (KV GB/s when the batch
    has decode rows, TFLOP/s of the causal triangle otherwise), the attention
    kernels' own time, the roofline of that time, and the clocks seen while it
    ran."""
    import torch
    from paged_kv_attention_27_gb300 import binding as B
    from paged_kv_attention_27_gb300.device import DeviceBatch
    b = make_workload(workload)
    db = DeviceBatch(b, device=f"cuda:{torch.cuda.current_device()}")
    info = B.fi_plan_get_info(db.plan)
    kvb, flops = kv_bytes(b), attention_flops(b)
    flush = kvb <= 2 * L2_BYTES     # K/V that the L2 could hold between steps
    ms_total, kern_ms = time_steps(db, K, W, dist, sampler, flush_l2=flush)
    ms_step = ms_total / K
    if info["num_decode_items"]:
        value, unit = whole_job_rate(kvb, world, ms_step) / 1e9, "GB/s"
    else:
        value, unit = whole_job_rate(flops, world, ms_step) / 1e12, "TFLOP/s"
    launches = launches_per_step(b, info)
    out = {"workload": b.name, "value": value, "unit": unit, "steps": K, "warmup": W,
           "ms_per_step": ms_step, "kernel_ms": kern_ms,
           "kv_bytes_per_step": kvb, "attention_flops_per_step": flops,
           "tokens_per_s": int(b.qo_lens.sum()) * world / (ms_step / 1e3),
           "kv_tokens": int(b.kv_lens.sum()), "q_rows": int(b.qo_lens.sum()),
           "gpu_launches": launches * K,
           "l2": (f"K/V ({kvb / 1e6:.0f} MB) could stay in the 129 MB L2: L2 flushed before "
                  "every timed step (a 258 MB write, not timed)") if flush else
                 f"inputs larger than L2 ({kvb / 1e9:.2f} GB of K/V per step): no flush",
           "roofline": roofline_of(b, kvb, flops, kern_ms, kernels_of(b, info), workload),
           "clocks": sampler.summary()}
    del db
    return out


def cpu_baseline(b):
    """The fp64 oracle on a bounded sample of the same batch."""
    if b.is_decode and not b.causal:
        v, dt, thr, done = oracle_sample(b)
        return {"value": v, "unit": "GB/s", "cores": thr, "kind": "oracle",
                "sample": f"fp64 oracle over {len(done)} of {b.batch} requests of the same batch "
                          f"(batch order, {thr} threads, {dt:.1f} s)"}
    v, dt, thr, nrows = oracle_rows_sample(b)
    return {"value": v, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
            "sample": f"fp64 oracle over {nrows} query rows (the last rows of each request, "
                      f"which see the most keys; {thr} threads, {dt:.1f} s)"}


def oracle_rows_sample(b, budget_s=12.0):
    """TFLOP/s of the oracle on sampled query rows: the visible pairs of the
    rows it completed within the budget, over the wall time."""
    import oracle
    threads = os.cpu_count() or 1
    tasks = []
    for r in range(b.batch):
        n = int(b.qo_lens[r])
        for i in range(max(0, n - 64), n):
            tasks.append((r, i))

    def one(task):
        r, i = task
        oracle.batch_attention(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.layout, b.page_indptr,
                               b.page_indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                               b.page_size, b.sm_scale, b.causal, requests=[r], rows={r: [i]},
                               window_left=b.window_left, dtype=b.dtype,
                               kv_dtype=b.cache_dtype, k_scale=b.k_scales, v_scale=b.v_scales)
        qo, kv = int(b.qo_lens[r]), int(b.kv_lens[r])
        pos = kv - qo + i
        hi = min(kv - 1, pos) if b.causal else kv - 1
        lo = max(0, pos - b.window_left) if b.window_left >= 0 else 0
        return 4 * b.head_dim * b.num_qo_heads * max(hi - lo + 1, 0)

    done_flops, n = 0, 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        nxt = 0
        pending = set()
        while nxt < len(tasks) and len(pending) < threads:
            pending.add(ex.submit(one, tasks[nxt]))
            nxt += 1
        while pending:
            fin, pending = cf.wait(pending, return_when=cf.FIRST_COMPLETED)
            for f in fin:
                done_flops += f.result()
                n += 1
            while nxt < len(tasks) and len(pending) < threads and \
                    time.perf_counter() - t0 < budget_s:
                pending.add(ex.submit(one, tasks[nxt]))
                nxt += 1
    dt = time.perf_counter() - t0
    return done_flops / dt / 1e12, dt, threads, n


def time_plan(b, sms, calls=200):
    """Host time of fi_plan for the batch (the planner runs on the CPU, off
    the GPU timeline, before every step of a serving loop): median over
    `calls` plans, with the work-item count it produced."""
    import numpy as np

    from paged_kv_attention_27_gb300 import binding as B
    from paged_kv_attention_27_gb300.device import plan_options

    decode = b.is_decode and not b.causal     # the mode DeviceBatch plans with
    mode = B.FI_MODE_DECODE if decode else B.FI_MODE_PREFILL
    args = (mode, b.batch, None if decode else b.qo_indptr.astype(np.int32),
            b.page_indptr.astype(np.int32), b.last_page_len.astype(np.int32),
            b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.causal,
            plan_options(b), sms)
    for _ in range(5):
        B.fi_plan(*args)
    ts = []
    for _ in range(calls):
        t0 = time.perf_counter()
        p = B.fi_plan(*args)
        ts.append(time.perf_counter() - t0)
    return {"median_us": float(np.median(ts)) * 1e6, "calls": calls,
            "items": B.fi_plan_get_info(p)["num_items"],
            "includes": "fi_plan through the Python binding, host only"}


def run_e2e(b, db, K, local_rank, unit):
    """The same metric for a serving step through the C ABI's host-buffer
    call: plan from the host page table, then fi_batch_attention_host, which
    copies q and the page table (and qo_indptr) from host memory, runs the
    kernels, copies out and lse back and synchronises. The KV cache stays
    resident in HBM (it is the cache); only the step's own inputs and outputs
    cross the host link."""
    import numpy as np
    import torch

    from paged_kv_attention_27_gb300 import binding as B
    from paged_kv_attention_27_gb300.device import num_sms, plan_options

    dev = f"cuda:{local_rank}"
    pin = lambda t: t.pin_memory()
    q_h = pin(db.q.cpu())
    indptr_h = b.page_indptr.astype(np.int32)
    indices_h = b.page_indices.astype(np.int32)
    last_h = b.last_page_len.astype(np.int32)
    qo_h = b.qo_indptr.astype(np.int32)
    # two output buffers: step t+1 is issued before step t's results are read
    outs = [(pin(torch.empty_like(db.out, device="cpu")),
             pin(torch.empty_like(db.lse, device="cpu"))) for _ in range(2)]
    out_h, lse_h = outs[0]
    sms = num_sms(dev)
    decode = db.mode == B.FI_MODE_DECODE
    ins = [q_h.numel() * q_h.element_size(), indptr_h.nbytes, indices_h.nbytes, last_h.nbytes]
    if not decode:
        ins.append(qo_h.nbytes)
    h2d = sum(ins)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    layout = B.LAYOUTS[b.layout]

    def plan():
        return B.fi_plan(db.mode, b.batch, None if decode else qo_h, indptr_h, last_h,
                         b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.causal,
                         plan_options(b), sms)

    info = B.fi_plan_get_info(plan())
    ws_bytes = info["workspace_bytes"] + info["host_io_bytes"]
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    # a serving loop keeps its host buffers and its stream from step to step:
    # their addresses are looked up once and passed as plain integers
    addr = lambda x: None if x is None else (x.data_ptr() if hasattr(x, "data_ptr")
                                             else x.ctypes.data)
    stream = torch.cuda.current_stream().cuda_stream
    args = [(addr(q_h), None if decode else addr(qo_h), addr(db.k), addr(db.v), layout, 0,
             b.num_pages, addr(indptr_h), addr(indices_h), addr(last_h), b.sm_scale, b.k_scale,
             b.v_scale, addr(o), addr(l), addr(ws), ws_bytes) for o, l in outs]
    heads = dict(k_head_scale=addr(db.k_head_scale), v_head_scale=addr(db.v_head_scale))

    def steps(n):
        # step i is planned, staged and enqueued while step i-1 runs; step
        # i-1's out and lse are then waited for (read back) before step i+1
        pending = 0
        for i in range(n):
            t = B.fi_batch_attention_host_async(plan(), *args[i % 2], stream=stream, **heads)
            B.fi_host_step_wait(pending)
            pending = t
        B.fi_host_step_wait(pending)

    steps(3)
    n = max(10, min(K, 200))
    t0 = time.perf_counter()
    steps(n)
    dt = (time.perf_counter() - t0) / n
    value = kv_bytes(b) / dt / 1e9 if unit == "GB/s" else attention_flops(b) / dt / 1e12
    return {"value": value, "unit": unit, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3, "steps": n,
            "includes": "per step: fi_plan on the host, fi_batch_attention_host_async (H2D of q "
                        "and the page table, kernels, D2H of out and lse) and fi_host_step_wait "
                        "on its results; two steps in flight (step t+1 is planned and enqueued "
                        "before step t's results are waited for), wall clock"}


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
