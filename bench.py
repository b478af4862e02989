#!/usr/bin/env python3
"""Benchmark of the paged-KV attention path on one GB300 (or N, one rank each).

Default workload: Llama-7B-shaped batch decode (64 requests, 32 q / 32 kv
heads, head_dim 128, page size 16, KV lengths uniform in [512, 4096], NHD,
shuffled page table), the configuration the headline metric is quoted on.
One step = one pass of the hot path over that batch through the C ABI: the
stream-ordered work-list upload, the decode kernel and, where the plan split
long requests, the merge kernel. The plan itself is host work done once per
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


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama7b_decode",
                    choices=["llama7b_decode", "llama70b_gqa_decode", "tiny_decode"])
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


def make_workload(name, batch=None):
    from paged_kv_attention_27_gb300 import synth
    fn = getattr(synth, name)
    return fn() if batch is None else fn(batch=batch)


def kv_bytes(b):
    """K+V bytes a pass reads: every request's kv_len rows of K and V for
    every kv head (bf16). Shared prefix pages are counted once."""
    seen = {}
    for r in range(b.batch):
        lo, hi = int(b.page_indptr[r]), int(b.page_indptr[r + 1])
        for j in range(lo, hi):
            used = b.page_size if j < hi - 1 else int(b.last_page_len[r])
            p = int(b.page_indices[j])
            seen[p] = max(seen.get(p, 0), used)
    return sum(seen.values()) * 2 * b.num_kv_heads * b.head_dim * 2


def io_bytes(b):
    """q + out (bf16) + lse (fp32) bytes of a pass."""
    rows = int(b.qo_lens.sum())
    return rows * b.num_qo_heads * (b.head_dim * 2 * 2 + 4)


KERNEL_SOURCES = {
    "decode_kernel": ["decode.cu", "ptx.cuh", "kernels.cuh", "fi_internal.h"],
}


def source_digest(kernel):
    """Hash of the sources a kernel is compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_attention_27_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, f), "rb").read())
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

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
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

    def stop(self):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        inside = [s for t, s in self.samples if self.t0 and self.t1 and self.t0 - 0.1 <= t <= self.t1 + 0.1]
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
                               b.page_size, b.sm_scale, b.causal, requests=[r])
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
    kvb = sum(int(b.kv_lens[r]) for r in done) * 2 * b.num_kv_heads * b.head_dim * 2
    return kvb / dt / 1e9, dt, threads, sorted(done)


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is a bounded sample."""
    if rank != 0:
        return
    b = make_workload(args.workload, args.batch)
    from paged_kv_attention_27_gb300 import synth
    threads = os.cpu_count() or 1
    sample = list(range(min(b.batch, threads)))
    sb = synth.sub_batch(b, sample)
    for _ in range(args.warmup):
        oracle_sample(sb, budget_s=0.0, threads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_sample(sb, budget_s=1e9, threads=threads)
        times.append(time.perf_counter() - t0)
    kvb = int(sb.kv_lens.sum()) * 2 * sb.num_kv_heads * sb.head_dim * 2
    step_s = sum(times) / len(times)
    value = kvb / step_s / 1e9
    desc = (f"fp64 oracle over requests {sample[0]}..{sample[-1]} of the batch "
            f"({int(sb.kv_lens.sum())} KV tokens per step), {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": b.name, "sample": desc},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    from paged_kv_attention_27_gb300 import binding as B
    from paged_kv_attention_27_gb300 import build as _build
    from paged_kv_attention_27_gb300.device import DeviceBatch, num_sms

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
    iob = io_bytes(b)
    launches_per_step = (1 if info["num_decode_items"] else 0) + \
                        (1 if info["num_prefill_items"] else 0) + \
                        (1 if info["num_split_requests"] else 0)

    # cpu baseline first (rank 0, N = 1 only), before the device is busy
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, thr, done = oracle_sample(b)
        cpu = {"value": v, "unit": "GB/s", "cores": thr, "kind": "oracle",
               "sample": f"fp64 oracle over {len(done)} of {b.batch} requests of the same batch "
                         f"(batch order, {thr} threads, {dt:.1f} s)"}

    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 1)):
        db.run()
    torch.cuda.synchronize()
    assert db.status() == B.FI_OK

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    ks = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    for ev in ks + ke:          # create the CUDA events (torch creates them on first record)
        ev.record(stream)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark_start()
    t_start.record(stream)
    for i in range(K):
        B.fi_profile_next_launch(ks[i], ke[i])
        db.run()
    t_end.record(stream)
    torch.cuda.synchronize()
    sampler.mark_end()
    if dist:
        dist.barrier()
    sampler.stop()
    st = db.status()
    assert st == B.FI_OK, B.status_string(st)
    ms_total = t_start.elapsed_time(t_end)
    kern_ms = sum(s.elapsed_time(e) for s, e in zip(ks, ke)) / K
    if dist:
        t = torch.tensor([ms_total], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_step = ms_total / K
    value = kvb * world / (ms_step / 1e3) / 1e9

    # end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(b, db, K, local_rank)

    hbm, bf16, src = peaks()
    achieved = kvb / (kern_ms / 1e3) / 1e9
    kernel_key = f"decode_kernel<{b.head_dim},{b.num_qo_heads // b.num_kv_heads}>"
    traffic = committed_traffic(args.workload, "decode_kernel")
    clocks = sampler.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Philox normals rounded to bf16, shuffled page table)",
        "config": {"workload": b.name, "batch": b.batch, "num_qo_heads": b.num_qo_heads,
                   "num_kv_heads": b.num_kv_heads, "head_dim": b.head_dim,
                   "page_size": b.page_size, "layout": b.layout,
                   "kv_tokens": int(b.kv_lens.sum()), "kv_bytes_per_step": kvb,
                   "io_bytes_per_step": iob,
                   "l2": f"inputs larger than L2 ({kvb / 1e9:.2f} GB of KV per step vs 129 MB "
                         "L2): no flush",
                   "plan": {k: info[k] for k in ("num_decode_items", "num_prefill_items",
                                                 "chunk_tokens", "num_split_requests")}},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "kernel": kernel_key, "kernel_ms": kern_ms,
                     "peak_source": f"{src} hbm_gbs (MEASURED_PEAKS.json)" if src == "measured"
                     else "fallback 6.8 TB/s"},
        "tokens_per_s": b.batch * world / (ms_step / 1e3),
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_e2e(b, db, K, local_rank):
    """KV GB/s of a serving step through the C ABI: plan from the host page
    table, copy q and the page table from pinned host memory, run, copy out
    and lse back, synchronise. The KV cache stays resident in HBM (it is the
    cache); only the step's own inputs and outputs cross the host link."""
    import numpy as np
    import torch

    from paged_kv_attention_27_gb300 import binding as B
    from paged_kv_attention_27_gb300.device import num_sms

    dev = f"cuda:{local_rank}"
    pin = lambda t: t.pin_memory()
    q_h = pin(db.q.cpu())
    indptr_h = pin(torch.from_numpy(b.page_indptr.astype(np.int32)))
    indices_h = pin(torch.from_numpy(b.page_indices.astype(np.int32)))
    last_h = pin(torch.from_numpy(b.last_page_len.astype(np.int32)))
    out_h = pin(torch.empty_like(db.out, device="cpu"))
    lse_h = pin(torch.empty_like(db.lse, device="cpu"))
    sms = num_sms(dev)
    h2d = sum(t.numel() * t.element_size() for t in (q_h, indptr_h, indices_h, last_h))
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    layout = B.LAYOUTS[b.layout]

    def step():
        plan = B.fi_plan(B.FI_MODE_DECODE, b.batch, None, indptr_h.numpy(), last_h.numpy(),
                         b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, 0, sms)
        assert plan.workspace_bytes <= db.workspace.numel()
        db.q.copy_(q_h, non_blocking=True)
        db.page_indptr.copy_(indptr_h, non_blocking=True)
        db.page_indices.copy_(indices_h, non_blocking=True)
        db.last_page_len.copy_(last_h, non_blocking=True)
        B.fi_batch_decode_paged(plan, db.q, db.k, db.v, layout, 0, b.num_pages, db.page_indptr,
                                db.page_indices, db.last_page_len, b.sm_scale, db.out, db.lse,
                                db.workspace)
        out_h.copy_(db.out, non_blocking=True)
        lse_h.copy_(db.lse, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        step()
    n = max(10, min(K, 200))
    t0 = time.perf_counter()
    for _ in range(n):
        step()
    dt = (time.perf_counter() - t0) / n
    return {"value": kv_bytes(b) / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3, "steps": n,
            "includes": "fi_plan on the host + H2D of q and page table + kernels + D2H of "
                        "out and lse, wall clock"}


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
