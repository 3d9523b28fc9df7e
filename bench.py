"""Benchmark: one decode step of paged attention over a block-tabled KV cache.

A step is the whole decode hot path on one batch: write each sequence's fresh
token K/V into its cache slot (pa_reshape_and_cache), then decode attention
(pa_decode: split-K pass + log-sum-exp reduce).  The default workload is the
long-context decode batch: 8 sequences with cached lengths uniform in
[16384, 32768], block size 32, 32 query / 8 kv heads, head dim 128, bf16 cache
(about 0.8 GB of K/V read per step, larger than L2; L2 is also flushed
between timed steps).

Prints ONE JSON line (rank 0).  ``value`` is achieved HBM GB/s of the step:
algorithmic bytes (every visible K/V element read once, q read, output and
fresh K/V written, block-table entries read) over the device time of the step.
``--impl reference`` times the fp64 CPU oracle on the same workload instead.
Multi-GPU (torchrun): every rank runs its own replica (weak scaling, no
data-path collective); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np
import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import workloads  # noqa: E402

METRIC = "paged-attn decode achieved HBM GB/s (% of GB300 peak) and seq-steps/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 8000.0


# ----------------------------------------------------------------------------- helpers

def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def decode_bytes(case) -> dict:
    """Algorithmic bytes of one decode step (each visible K/V element read once)."""
    eb = case.kv_elem_bytes()
    S, Hq, Hkv, D, bs = case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim, case.block_size
    ctx = case.context_lens.to(torch.int64)
    kv = int(ctx.sum()) * Hkv * D * eb * 2
    q = S * Hq * D * eb
    out = S * Hq * D * 4
    tables = int(((ctx + bs - 1) // bs).sum()) * 4 + S * 4
    fresh = case.new_key.numel() * eb * 2 * 2 + case.slot_mapping.numel() * 8  # read + write
    return {"kv": kv, "decode": kv + q + out + tables, "step": kv + q + out + tables + fresh}


def prefill_work(case) -> tuple[float, int]:
    """Causal-exact FLOPs (QK^T and PV) and algorithmic bytes of one prefill call."""
    eb = case.kv_elem_bytes()
    Hq, Hkv, D = case.num_heads, case.num_kv_heads, case.head_dim
    qsl = case.query_start_loc.tolist()
    pairs = 0
    for s in range(case.num_seqs):
        lq, c = qsl[s + 1] - qsl[s], int(case.context_lens[s])
        pairs += sum(c - lq + i + 1 for i in range(lq))
    flops = 4.0 * D * Hq * pairs
    byts = int(case.context_lens.sum()) * Hkv * D * eb * 2 + case.query.numel() * eb + case.query.numel() * 4
    return flops, byts


def _code_only(text: str) -> str:
    """Source text without comments and blank lines (comments do not change a kernel)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash(kind: str = "decode") -> str:
    """Hash of the code of the CUDA sources a kernel is built from, comments left out (ties
    ncu counters to a kernel version)."""
    csrc = ROOT / "paged_kv_attention_write_gb300" / "csrc"
    files = {"decode": ["decode_kernels.cuh", "decode.cu", "tma.cuh", "common.cuh"],
             "prefill": ["prefill.cu", "tma.cuh", "common.cuh"]}[kind]
    h = hashlib.sha256()
    for f in files:
        h.update(_code_only((csrc / f).read_text()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kind: str, workload: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary, if it was taken
    on the current kernel sources and this workload; else None."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    e = json.loads(p.read_text()).get(kind, {}).get(workload)
    if not e or e.get("source_sha256_16") != kernel_source_hash(kind):
        return None
    return e.get("dram_bytes_per_launch")


class L2Flush:
    """Between timed steps: write a buffer twice the L2 size, then read another one, so
    that L2 holds neither the step's inputs nor dirty lines that the timed kernels would
    have to write back.  Runs outside the CUDA-event pair of each step."""

    def __init__(self, device):
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n = max(2 * l2, 256 << 20)
        self.w = torch.empty(n, dtype=torch.uint8, device=device)
        self.r = torch.ones(n // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm

class DecodeStep:
    """Device-resident inputs of one decode step and the calls that run it."""

    def __init__(self, case, device):
        import paged_kv_attention_write_gb300 as pa
        self.pa = pa
        self.case = case
        self.dev = device
        self.kc = case.key_cache.to(device)
        self.vc = case.value_cache.to(device)
        self.bt = case.block_tables.to(device)
        self.cl = case.context_lens.to(device)
        self.q = case.query.to(device)
        self.nk = case.new_key.to(device)
        self.nv = case.new_value.to(device)
        self.slots = case.slot_mapping.to(device)
        self.out = torch.empty(tuple(case.query.shape), dtype=torch.float32, device=device)
        nbytes = pa.pa_decode_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                             case.head_dim,
                                             case.max_context_len)
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
        self.max_ctx = case.max_context_len
        # End-to-end staging: the step's inputs packed in one pinned host buffer and one
        # device buffer (256-byte aligned fields), one copy each way per step.
        names = ("q", "nk", "nv", "slots", "bt", "cl")
        offs, total = {}, 0
        for k in names:
            t = getattr(self, k)
            offs[k] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        self.h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.d_in = torch.empty(total, dtype=torch.uint8, device=device)
        self.e2e_views = {}
        for k in names:
            t = getattr(self, k)
            nb = t.numel() * t.element_size()
            self.h_in[offs[k]:offs[k] + nb].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
            self.e2e_views[k] = self.d_in[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
        self.h_out = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()

    def reshape(self):
        self.pa.pa_reshape_and_cache(self.nk, self.nv, self.kc, self.vc, self.slots)

    def decode(self):
        self.pa.pa_decode(self.out, self.q, self.kc, self.vc, self.bt, self.cl, self.max_ctx,
                          self.case.scale, workspace=self.ws)

    def step(self):
        """The decode step: every sequence's new token written to its slot and attended, in
        one call (pa_decode_write)."""
        self.pa.pa_decode_write(self.out, self.q, self.nk, self.nv, self.slots, self.kc, self.vc, self.bt,
                                self.cl, self.max_ctx, self.case.scale, workspace=self.ws)

    def step_separate(self):
        """The same step as two calls: pa_reshape_and_cache, then pa_decode."""
        self.reshape()
        self.decode()

    def e2e_step(self):
        """Host buffers in, host result out: one H2D copy of the packed step inputs, the
        step through the public API on the device copies, one D2H copy of the output."""
        self.d_in.copy_(self.h_in, non_blocking=True)
        v = self.e2e_views
        self.pa.pa_decode_write(self.out, v["q"], v["nk"], v["nv"], v["slots"], self.kc, self.vc, v["bt"],
                                v["cl"], self.max_ctx, self.case.scale, workspace=self.ws)
        self.h_out.copy_(self.out, non_blocking=True)

    def h2d_bytes(self):
        return self.h_in.numel()

    def d2h_bytes(self):
        return self.h_out.numel() * self.h_out.element_size()

    def launches_per_step(self):
        # pa_decode_write: split (with the cache write) + reduce, and a plan kernel first
        # when there are 2048 or more (kv-head group, sequence) segments
        c = self.case
        segments = max(1, c.num_kv_heads // 8) * c.num_seqs
        return 2 + (1 if segments >= 2048 else 0)


class PrefillStep:
    """Device-resident inputs of one chunked-prefill step: the chunk's K/V written to their
    slots, then prefill attention of the chunk over prefix + chunk."""

    def __init__(self, case, device):
        import paged_kv_attention_write_gb300 as pa
        self.pa = pa
        self.case = case
        self.kc = case.key_cache.to(device)
        self.vc = case.value_cache.to(device)
        self.bt = case.block_tables.to(device)
        self.cl = case.context_lens.to(device)
        self.q = case.query.to(device)
        self.qsl = case.query_start_loc.to(device)
        self.nk = case.new_key.to(device)
        self.nv = case.new_value.to(device)
        self.slots = case.slot_mapping.to(device)
        self.out = torch.empty(tuple(case.query.shape), dtype=torch.float32, device=device)
        self.mq = int((case.query_start_loc[1:] - case.query_start_loc[:-1]).max())
        names = ("q", "nk", "nv", "slots", "bt", "cl", "qsl")
        offs, total = {}, 0
        for k in names:
            t = getattr(self, k)
            offs[k] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        self.h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.d_in = torch.empty(total, dtype=torch.uint8, device=device)
        self.e2e_views = {}
        for k in names:
            t = getattr(self, k)
            nb = t.numel() * t.element_size()
            self.h_in[offs[k]:offs[k] + nb].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
            self.e2e_views[k] = self.d_in[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
        self.h_out = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()

    def prefill(self, v=None):
        v = v or {"q": self.q, "qsl": self.qsl, "bt": self.bt, "cl": self.cl}
        self.pa.pa_prefill_chunk(self.out, v["q"], v["qsl"], self.mq, self.kc, self.vc, v["bt"],
                                 v["cl"], self.case.max_context_len, self.case.scale)

    def step(self):
        self.pa.pa_reshape_and_cache(self.nk, self.nv, self.kc, self.vc, self.slots)
        self.prefill()

    def e2e_step(self):
        self.d_in.copy_(self.h_in, non_blocking=True)
        v = self.e2e_views
        self.pa.pa_reshape_and_cache(v["nk"], v["nv"], self.kc, self.vc, v["slots"])
        self.prefill(v)
        self.h_out.copy_(self.out, non_blocking=True)


def prefill_arm(args, case, device, rank, world, dist_on):
    """``--workload prefill_chunk``: the chunked-prefill row timed on its own."""
    hbm_peak, tc_peak, peak_kind = peaks()
    st = PrefillStep(case, device)
    flush = L2Flush(device)
    flops, byts = prefill_work(case)
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    pf_ms, _ = time_steps(st.prefill, args.steps, flush, dist_on)
    with ClockSampler(device.index) as clocks:
        step_ms, wall = time_steps(st.step, args.steps, flush, dist_on)
    e2e_ms, _ = time_steps(st.e2e_step, max(3, args.steps // 4), flush, dist_on)
    ms_step = _max_over_ranks(statistics.median(step_ms), dist_on)
    ms_pf = _max_over_ranks(statistics.median(pf_ms), dist_on)
    ms_e2e = _max_over_ranks(statistics.median(e2e_ms), dist_on)
    if rank != 0:
        return None
    tfs = flops / (ms_pf * 1e-3) / 1e12
    line = {
        "metric": "paged-attn chunked-prefill TFLOP/s (causal-exact FLOPs)",
        "value": round(world * flops / (ms_step * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, shuffled block pool)",
        "config": {"workload": case.name, "num_seqs": case.num_seqs,
                   "prefix_lens": case.meta.get("prefix_lens"), "chunk_lens": case.meta.get("chunk_lens"),
                   "block_size": case.block_size, "num_heads": case.num_heads,
                   "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
                   "flops_per_step": flops,
                   "l2": "L2 flushed before each timed step (256 MB write, then 256 MB read of another buffer, outside the timed events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tokens_per_s": round(world * int(case.query.shape[0]) / (ms_step * 1e-3), 1),
        "roofline": {"kernel": "pa_prefill_chunk", "bound": "tensor", "achieved": round(tfs, 1),
                     "peak": tc_peak, "unit": "TFLOP/s", "frac": round(tfs / tc_peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops, burst)",
                     "traffic": profiled_traffic("prefill", args.workload),
                     "algorithmic_bytes_per_launch": byts, "ms_per_launch": round(ms_pf, 5),
                     "hbm_frac": round(byts / (ms_pf * 1e-3) / 1e9 / hbm_peak, 4)},
        "e2e": {"value": round(world * flops / (ms_e2e * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(ms_e2e, 5), "h2d_bytes_per_step": st.h_in.numel(),
                "d2h_bytes_per_step": st.h_out.numel() * 4},
        "gpu_launches": args.steps * 2,
        "step_ms": {"step": step_stats(step_ms), "pa_prefill_chunk": step_stats(pf_ms), "e2e": step_stats(e2e_ms),
                    "statistic": "median of the per-step CUDA-event times (p10 / p90 / mean beside it)"},
        "clocks": clocks.summary(),
        "timed_region_s": round(wall, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = {**oracle_prefill_timing(), "kind": "oracle"}
    return line


def _barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()


def _max_over_ranks(x: float, dist_on: bool) -> float:
    """Slowest rank's time: a MAX all-reduce of one number (timing only, not the data path)."""
    if not dist_on:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def shard_of(num_units: int, rank: int, world: int) -> range:
    """Units of a sharded batch owned by ``rank`` (contiguous, sizes differ by at most 1).
    The bench runs whole replicas per rank (weak scaling); a caller that splits one batch
    of independent sequences over ranks takes this range of it, with no collective."""
    lo = num_units * rank // world
    hi = num_units * (rank + 1) // world
    return range(lo, hi)


def time_steps(fn, steps, flush, dist_on):
    """Per-step device time (ms) with CUDA events on the launching stream; L2 flushed before
    each step outside the event pair.  The region is bracketed by barrier + synchronize."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    _barrier(dist_on)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        flush()
        starts[i].record()
        fn()
        ends[i].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    _barrier(dist_on)
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return ms, wall


def step_stats(ms) -> dict:
    """Median and spread of per-step device times (ms): the median is the figure used."""
    q = np.percentile(np.asarray(ms, dtype=np.float64), [10, 50, 90])
    return {"median": round(float(q[1]), 5), "p10": round(float(q[0]), 5), "p90": round(float(q[2]), 5),
            "mean": round(float(np.mean(ms)), 5), "n": len(ms)}


def gpu_arm(args, rank, world, dist_on):
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(device)
    hbm_peak, tc_peak, peak_kind = peaks()
    case = workloads.WORKLOADS[args.workload]()
    if not case.is_decode:
        return prefill_arm(args, case, device, rank, world, dist_on)
    st = DecodeStep(case, device)
    flush = L2Flush(device)
    byts = decode_bytes(case)

    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()

    # decode kernel alone (the dominant launch: split-K pass + reduce), then the whole step
    dec_ms, _ = time_steps(st.decode, args.steps, flush, dist_on)
    with ClockSampler(device.index) as clocks:
        step_ms, wall = time_steps(st.step, args.steps, flush, dist_on)
    sep_ms, _ = time_steps(st.step_separate, max(3, args.steps // 4), flush, dist_on)
    for _ in range(3):
        st.e2e_step()
    torch.cuda.synchronize()
    e2e_ms, _ = time_steps(st.e2e_step, max(3, args.steps // 4), flush, dist_on)

    ms_step = _max_over_ranks(statistics.median(step_ms), dist_on)
    ms_sep = _max_over_ranks(statistics.median(sep_ms), dist_on)
    ms_dec = _max_over_ranks(statistics.median(dec_ms), dist_on)
    ms_e2e = _max_over_ranks(statistics.median(e2e_ms), dist_on)
    value = world * byts["step"] / (ms_step * 1e-3) / 1e9
    dec_gbs = byts["decode"] / (ms_dec * 1e-3) / 1e9
    e2e_gbs = world * byts["step"] / (ms_e2e * 1e-3) / 1e9

    secondary = {}
    if not args.no_secondary and rank == 0:
        secondary = secondary_measurements(device, flush, hbm_peak, tc_peak, peak_kind)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, byts)

    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, shuffled block pool)",
        "config": {
            "workload": case.name,
            "num_seqs": case.num_seqs,
            "context_lens": case.context_lens.tolist(),
            "block_size": case.block_size,
            "num_heads": case.num_heads,
            "num_kv_heads": case.num_kv_heads,
            "head_dim": case.head_dim,
            "kv_bytes_per_step": byts["kv"],
            "l2": "inputs larger than L2, and L2 flushed before each timed step (256 MB write, then 256 MB read of another buffer, outside the timed events)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "step": "pa_decode_write: every sequence's new token written to its cache slot and decode attention, one call",
        },
        "seq_steps_per_s": round(world * case.num_seqs / (ms_step * 1e-3), 1),
        "step_as_two_calls": {"ms": round(ms_sep, 5), "GB/s": round(world * byts["step"] / (ms_sep * 1e-3) / 1e9, 2),
                              "calls": "pa_reshape_and_cache, then pa_decode"},
        "pct_of_peak": {"measured_hbm": round(100 * value / world / hbm_peak, 1),
                        "nominal_8TBs": round(100 * value / world / NOMINAL_HBM_GBS, 1)},
        "roofline": {
            "kernel": "pa_decode (split-K pass + log-sum-exp reduce)",
            "bound": "hbm",
            "achieved": round(dec_gbs, 1),
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": round(dec_gbs / hbm_peak, 4),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
            "traffic": profiled_traffic("decode", args.workload),
            "algorithmic_bytes_per_launch": byts["decode"],
            "ms_per_launch": round(ms_dec, 5),
        },
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "ms_per_step": round(ms_e2e, 5),
                "h2d_bytes_per_step": st.h2d_bytes(), "d2h_bytes_per_step": st.d2h_bytes()},
        "gpu_launches": args.steps * st.launches_per_step(),
        "step_ms": {"step": step_stats(step_ms), "step_as_two_calls": step_stats(sep_ms),
                    "pa_decode": step_stats(dec_ms), "e2e": step_stats(e2e_ms),
                    "statistic": "median of the per-step CUDA-event times (p10 / p90 / mean beside it)"},
        "clocks": clocks.summary(),
        "timed_region_s": round(wall, 3),
    }
    if secondary:
        line["secondary"] = secondary
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def manager_stream(seed: int = 9, num_requests: int = 400):
    """A seeded serving-like stream of KV-cache manager calls: requests whose prompts start
    with one of four system prompts (64-1024 tokens) plus their own text (16-1024 tokens),
    at most 64 running at once; each running request takes one step per round (the next
    512-token prefill chunk of its prompt, else one decode token), ceil(prompt / 512) + 32
    steps, then it is freed.  Returns the calls: ("admit", id, tokens), ("step", id),
    ("free", id)."""
    rng = np.random.default_rng(seed)
    systems = [rng.integers(0, 32000, size=int(rng.integers(64, 1025))).tolist() for _ in range(4)]
    calls, running, nxt = [], {}, 0
    while nxt < num_requests or running:
        while nxt < num_requests and len(running) < 64:
            toks = systems[int(rng.integers(4))] + rng.integers(0, 32000, size=int(rng.integers(16, 1025))).tolist()
            calls.append(("admit", nxt, toks))
            running[nxt] = -(-len(toks) // 512) + 32
            nxt += 1
        for rid in list(running):
            calls.append(("step", rid))
            running[rid] -= 1
            if running[rid] == 0:
                calls.append(("free", rid))
                del running[rid]
    return calls


def replay_manager(mgr, calls, rng_seed: int = 1) -> int:
    """Run a call stream on a manager (library or reference): admit, then per step allocate
    the next prefill chunk (prompt tokens not yet computed, at most 512) or one decode token
    and register full blocks, then free.  Tokens live in int32 arrays (no per-call list
    conversion).  Returns the number of manager calls made."""
    rng = np.random.default_rng(rng_seed)
    state, n = {}, 0
    for c in calls:
        if c[0] == "admit":
            _, rid, toks = c
            buf = np.zeros(len(toks) + 64, dtype=np.int32)
            buf[:len(toks)] = toks
            state[rid] = [buf, mgr.admit(rid, buf[:len(toks)]), len(toks), len(toks)]
            n += 1
        elif c[0] == "step":
            buf, done, plen, ntok = state[c[1]]
            if done < plen:
                new = min(plen, done + 512)
            else:
                buf[ntok] = int(rng.integers(32000))
                ntok += 1
                new = ntok
            mgr.allocate_slots(c[1], new)
            mgr.cache_blocks(c[1], buf[:ntok], new)
            state[c[1]][1], state[c[1]][3] = new, ntok
            n += 2
        else:
            mgr.free(c[1])
            del state[c[1]]
            n += 1
    return n


MANAGER_STREAM = "400 requests, 4 shared system prompts, 512-token chunks, 32 decode tokens, <= 64 running, bs 16, 16384 blocks"


def manager_measurement():
    """Host KV-cache manager (the library's C++ code): calls per second on a seeded
    serving-like stream."""
    from paged_kv_attention_write_gb300.kv_manager import KVCacheManager
    calls = manager_stream()
    mgr = KVCacheManager(16384, 16)
    t0 = time.perf_counter()
    n = replay_manager(mgr, calls)
    dt = time.perf_counter() - t0
    return {"stream": MANAGER_STREAM, "calls": n, "s": round(dt, 4), "calls_per_s": round(n / dt, 1),
            "us_per_call": round(dt / n * 1e6, 3), "stats": mgr.stats(),
            "note": "host time through the Python binding (ctypes marshalling included)"}


SERVE_REPLAY = ("256 requests at once: 70 % start with one of 4 system prompts (128-1024 tokens), "
                "own text 64-1024 tokens, 32-256 generated tokens; 32 q / 8 kv heads, D 128, bs 16, bf16; "
                "budget 4096 tokens, 512-token chunks, <= 8 decode steps in a row; q/k/v gathered on the "
                "device from seeded random tables by (token, position); one device read of each step's output")


def _serve_replay(device, num_requests: int, seed: int):
    from paged_kv_attention_write_gb300.engine import PagedAttentionEngine
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, R = 32, 8, 128, 8192
    g = torch.Generator().manual_seed(seed)
    kt = torch.randn((R, Hkv, D), generator=g).to(torch.bfloat16).to(device)
    vt = torch.randn((R, Hkv, D), generator=g).to(torch.bfloat16).to(device)
    qt = torch.randn((R, Hq, D), generator=g).to(torch.bfloat16).to(device)
    systems = [rng.integers(0, 32000, size=int(rng.integers(128, 1025))).tolist() for _ in range(4)]
    eng = PagedAttentionEngine(40000, 16, Hq, Hkv, D, torch.bfloat16, device)
    for rid in range(num_requests):
        own = rng.integers(0, 32000, size=int(rng.integers(64, 1025))).tolist()
        prompt = (systems[int(rng.integers(4))] + own) if rng.random() < 0.7 else own
        eng.add_request(rid, prompt, int(rng.integers(32, 257)))
    gpu = []

    cb = [0.0]  # host seconds spent in the two callbacks (the stand-in model and sampler)

    def qkv(step):
        # the table row of each (token, position), from the step's device copy of both
        # (int32 arithmetic: token < 32000 and position < 8192 keep the sum below 2^31;
        # R is a power of two)
        c0 = time.perf_counter()
        tok, pos = eng.device_tokens(step)
        i = torch.add(tok * 7919, pos, alpha=104729).bitwise_and_(R - 1)
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        gpu.append([e, None])
        r = torch.index_select(qt, 0, i), torch.index_select(kt, 0, i), torch.index_select(vt, 0, i)
        cb[0] += time.perf_counter() - c0
        return r

    def sample(step, out):
        c0 = time.perf_counter()
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        gpu[-1][1] = e
        out[:, 0, 0].cpu()  # the step's result reaches the host (a sampler would need it)
        r = rng.integers(0, 32000, size=step["num_seqs"])
        cb[0] += time.perf_counter() - c0
        return r
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    steps = eng.run(qkv, sample)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    gpu_s = sum(a.elapsed_time(b) for a, b in gpu) / 1e3
    return eng, steps, wall, gpu_s, cb[0]


def serve_replay_measurement(device, num_requests: int = 256, seed: int = 11):
    """The scheduler-driven replay (mistral.rs-style alternating prefill / decode steps)
    through PagedAttentionEngine: host scheduling, one packed host-to-device copy, K/V write
    and attention per step, one device read per step (the sampled tokens of a real engine
    depend on it).  One untimed warm-up replay first; reports generated tokens per second
    (seq-steps/s) end to end and the share of the wall time the step's kernels took."""
    _serve_replay(device, num_requests, seed)          # warm-up (lazy loading, allocator)
    eng, steps, wall, gpu_s, cb_s = _serve_replay(device, num_requests, seed)
    st, ms = eng.sched.stats(), eng.sched.manager_stats()
    return {"workload": SERVE_REPLAY, "steps": steps, "s": round(wall, 3),
            "seq_steps_per_s": round(st["generated_tokens"] / wall, 1),
            "prompt_tokens_per_s": round(st["prefill_tokens"] / wall, 1),
            "ms_per_step": round(wall / max(1, steps) * 1e3, 4),
            "kernel_share_of_wall": round(gpu_s / wall, 3),
            "callbacks_ms_per_step": round(cb_s / max(1, steps) * 1e3, 4),
            "engine_host_ms_per_step": round((wall - cb_s) / max(1, steps) * 1e3, 4),
            "note": ("callbacks = the stand-in model and sampler (q/k/v gathers, the step's device read, "
                     "which waits for the step's kernels); engine_host = the rest of the wall: "
                     "scheduling, the packed copy and the attention call"),
            "scheduler": st, "kv_manager": ms, "warmup": "one untimed replay of the same workload"}


def rope_measurement(device, flush, hbm_peak):
    """The fused rotary-embedding entry points beside their plain counterparts on the same
    data: the chunked-prefill workload's 2048-token cache write, and decode on the
    decode-batch workload (its query rotated and scaled at each sequence's position)."""
    import paged_kv_attention_write_gb300 as pa
    res = {}
    freqs = torch.from_numpy(pa.pa_rope_yarn_freqs(128, 1e6, 8.0, 4096, 32.0, 1.0)).to(device)
    rope = pa.Rope(freqs, 128, 0.1, 4096)
    case = workloads.prefill_chunk()
    kc, vc = case.key_cache.to(device), case.value_cache.to(device)
    nk, nv, sl = case.new_key.to(device), case.new_value.to(device), case.slot_mapping.to(device)
    qsl = case.query_start_loc.tolist()
    pos = torch.tensor(sum((list(range(int(case.context_lens[s]) - (qsl[s + 1] - qsl[s]), int(case.context_lens[s])))
                            for s in range(case.num_seqs)), []), dtype=torch.int32, device=device)
    rb = nk.numel() * nk.element_size() * 4 + sl.numel() * 8 + pos.numel() * 4
    for name, fn in (("reshape_and_cache", lambda: pa.pa_reshape_and_cache(nk, nv, kc, vc, sl)),
                     ("reshape_and_cache_rope", lambda: pa.pa_reshape_and_cache_rope(nk, nv, kc, vc, sl, pos, rope))):
        for _ in range(3):
            fn()
        t = statistics.median(time_steps(fn, 50, flush, False)[0])
        res[name + "_2048_tokens"] = {"ms": round(t, 5), "GB/s": round(rb / (t * 1e-3) / 1e9, 1)}
    del kc, vc
    case = workloads.decode_batch()
    st = DecodeStep(case, device)
    st.reshape()
    b = decode_bytes(case)["decode"]
    for name, fn in (("decode", st.decode),
                     ("decode_rope", lambda: pa.pa_decode_rope(st.out, st.q, st.kc, st.vc, st.bt, st.cl, st.max_ctx,
                                                               case.scale, rope, workspace=st.ws))):
        for _ in range(3):
            fn()
        t = statistics.median(time_steps(fn, 50, flush, False)[0])
        res[name + "_decode_batch"] = {"ms": round(t, 5), "GB/s": round(b / t / 1e6, 1),
                                       "frac_hbm": round(b / t / 1e6 / hbm_peak, 4)}
    res["workloads"] = "cache write: prefill_chunk's 2048 tokens; decode: decode_batch (32 sequences)"
    return res


def mixed_batch_measurement(device, flush, hbm_peak, tc_peak):
    """The mixed decode + prefill step as one pa_prefill_chunk launch, against the same rows
    as two launches (pa_decode for the decode rows, pa_prefill_chunk for the chunks).  The
    roofline time is the larger of FLOPs at the tensor peak and bytes at the HBM peak."""
    import paged_kv_attention_write_gb300 as pa
    case = workloads.mixed_batch()
    nd = int(((case.query_start_loc[1:] - case.query_start_loc[:-1]) == 1).sum())
    kc, vc = case.key_cache.to(device), case.value_cache.to(device)
    pa.pa_reshape_and_cache(case.new_key.to(device), case.new_value.to(device), kc, vc,
                            case.slot_mapping.to(device))
    bt, cl = case.block_tables.to(device), case.context_lens.to(device)
    q, qsl = case.query.to(device), case.query_start_loc.to(device)
    out = torch.empty(tuple(q.shape), dtype=torch.float32, device=device)
    mq = int((case.query_start_loc[1:] - case.query_start_loc[:-1]).max())
    # the same rows split: decode rows (the first nd sequences) and the chunks
    q_d, bt_d, cl_d = q[:nd], bt[:nd].contiguous(), cl[:nd].contiguous()
    q_p, bt_p, cl_p = q[nd:], bt[nd:].contiguous(), cl[nd:].contiguous()
    qsl_p = (qsl[nd:] - nd).contiguous()
    out_d, out_p = torch.empty_like(out[:nd]), torch.empty_like(out[nd:])
    ws = torch.empty(max(1, pa.pa_decode_workspace_size(nd, case.num_heads, case.num_kv_heads,
                                                        case.head_dim, int(cl_d.max()))),
                     dtype=torch.uint8, device=device)

    def mixed():
        pa.pa_prefill_chunk(out, q, qsl, mq, kc, vc, bt, cl, case.max_context_len, case.scale)

    def split():
        pa.pa_decode(out_d, q_d, kc, vc, bt_d, cl_d, int(cl_d.max()), case.scale, workspace=ws)
        pa.pa_prefill_chunk(out_p, q_p, qsl_p, mq, kc, vc, bt_p, cl_p, case.max_context_len, case.scale)
    for _ in range(5):
        mixed()
        split()
    t_mix = statistics.median(time_steps(mixed, 50, flush, False)[0])
    t_split = statistics.median(time_steps(split, 50, flush, False)[0])
    flops, byts = prefill_work(case)
    t_roof = max(flops / (tc_peak * 1e12), byts / (hbm_peak * 1e9)) * 1e3
    return {"workload": case.name, "decode_rows": nd, "chunks": case.num_seqs - nd,
            "ms_one_launch": round(t_mix, 5), "ms_decode_plus_prefill_launches": round(t_split, 5),
            "tokens_per_s": round(int(q.shape[0]) / (t_mix * 1e-3), 1),
            "TFLOP/s": round(flops / (t_mix * 1e-3) / 1e12, 1), "GB/s": round(byts / (t_mix * 1e-3) / 1e9, 1),
            "roofline_ms": round(t_roof, 5), "frac_roofline": round(t_roof / t_mix, 4)}


def secondary_measurements(device, flush, hbm_peak, tc_peak, peak_kind):
    """Shorter timings of the other hot-path rows: decode batch, chunked prefill, cache write,
    RoPE variants, mixed batch, host manager and scheduler replay, block copy, and decode on
    the stress workload (block 16, bf16)."""
    import paged_kv_attention_write_gb300 as pa
    res = {}
    case = workloads.decode_batch()
    st = DecodeStep(case, device)
    for _ in range(5):
        st.step()
    ms, _ = time_steps(st.decode, 50, flush, False)
    b = decode_bytes(case)["decode"]
    t = statistics.median(ms)
    res["decode_batch"] = {"workload": case.name, "ms": round(t, 5),
                           "GB/s": round(b / t / 1e6, 1), "frac_hbm": round(b / t / 1e6 / hbm_peak, 4),
                           "seq_steps_per_s": round(case.num_seqs / t * 1e3, 1)}
    del st
    case = workloads.prefill_chunk()
    kc, vc = case.key_cache.to(device), case.value_cache.to(device)
    bt, cl = case.block_tables.to(device), case.context_lens.to(device)
    q, qsl = case.query.to(device), case.query_start_loc.to(device)
    nk, nv, sl = case.new_key.to(device), case.new_value.to(device), case.slot_mapping.to(device)
    out = torch.empty(tuple(q.shape), dtype=torch.float32, device=device)
    mq = int((case.query_start_loc[1:] - case.query_start_loc[:-1]).max())
    pa.pa_reshape_and_cache(nk, nv, kc, vc, sl)

    def prefill():
        pa.pa_prefill_chunk(out, q, qsl, mq, kc, vc, bt, cl, case.max_context_len, case.scale)
    for _ in range(5):
        prefill()
    ms, _ = time_steps(prefill, 50, flush, False)
    t = statistics.median(ms)
    flops, byts = prefill_work(case)
    tfs = flops / (t * 1e-3) / 1e12
    res["prefill_chunk"] = {"workload": case.name, "ms": round(t, 5), "TFLOP/s": round(tfs, 1),
                            "bound": "tensor", "peak_tflops": tc_peak,
                            "frac_tensor": round(tfs / tc_peak, 4),
                            "GB/s": round(byts / (t * 1e-3) / 1e9, 1),
                            "tokens_per_s": round(int(q.shape[0]) / (t * 1e-3), 1)}

    def reshape():
        pa.pa_reshape_and_cache(nk, nv, kc, vc, sl)
    ms, _ = time_steps(reshape, 50, flush, False)
    t = statistics.median(ms)
    rb = nk.numel() * nk.element_size() * 4 + sl.numel() * 8
    res["reshape_and_cache_2048_tokens"] = {"ms": round(t, 5), "GB/s": round(rb / (t * 1e-3) / 1e9, 1)}
    # the same call on 8 tokens: the floor of a launch timed this way (events around one call
    # after the L2 flush), next to which the 2048 tokens' 16.8 MB are measured
    ms, _ = time_steps(lambda: pa.pa_reshape_and_cache(nk[:8], nv[:8], kc, vc, sl[:8]), 50, flush, False)
    res["reshape_and_cache_8_tokens"] = {"ms": round(statistics.median(ms), 5),
                                         "note": "launch floor under the same timing"}
    del kc, vc
    res["rope"] = rope_measurement(device, flush, hbm_peak)
    res["mixed_batch"] = mixed_batch_measurement(device, flush, hbm_peak, tc_peak)
    res["kv_manager"] = manager_measurement()
    res["serve_replay"] = serve_replay_measurement(device)
    # block copy: 26 recipients' leading blocks of the stress workload (bs 16, bf16)
    stress16 = case = workloads.stress_decode(block_size=16, dtype=torch.bfloat16)
    kc, vc = case.key_cache.to(device), case.value_cache.to(device)
    bm = case.block_mapping.to(device)

    def copy():
        pa.pa_copy_blocks(kc, vc, bm)
    for _ in range(3):
        copy()
    ms, _ = time_steps(copy, 50, flush, False)
    t = statistics.median(ms)
    cb = int(bm.shape[0]) * case.block_size * case.num_kv_heads * case.head_dim * 2 * 2 * 2
    res["copy_blocks_stress"] = {"pairs": int(bm.shape[0]), "ms": round(t, 5),
                                 "GB/s": round(cb / (t * 1e-3) / 1e9, 1)}
    del kc, vc, bm
    # decode on the stress workload (256 sequences, log-uniform lengths, 20 % free blocks,
    # prefix copies) for every block size and cache dtype
    res["stress_decode"] = {}
    for bs in (8, 16, 32):
        for dt, tag in ((torch.float16, "fp16"), (torch.bfloat16, "bf16")):
            case = stress16 if (bs == 16 and dt == torch.bfloat16) else \
                workloads.stress_decode(block_size=bs, dtype=dt)
            st = DecodeStep(case, device)
            if case.block_mapping is not None:
                pa.pa_copy_blocks(st.kc, st.vc, case.block_mapping.to(device))
            st.reshape()
            for _ in range(3):
                st.decode()
            ms, _ = time_steps(st.decode, 30, flush, False)
            t = statistics.median(ms)
            b = decode_bytes(case)["decode"]
            res["stress_decode"][f"bs{bs}_{tag}"] = {
                "workload": case.name, "ms": round(t, 5), "GB/s": round(b / t / 1e6, 1),
                "frac_hbm": round(b / t / 1e6 / hbm_peak, 4),
                "seq_steps_per_s": round(case.num_seqs / t * 1e3, 1)}
            del st
            torch.cuda.empty_cache()
    res["decode_group_sizes"] = group_size_measurement(device, flush, hbm_peak)
    return res


def group_size_measurement(device, flush, hbm_peak):
    """pa_decode on one long-context cache (8 kv heads) with 1, 2, 4 and 8 query heads per kv
    head: the same K/V bytes, a fresh random query of each width."""
    import paged_kv_attention_write_gb300 as pa
    case = workloads.gqa_decode(8)
    st = DecodeStep(case, device)
    st.reshape()
    S, D = case.num_seqs, case.head_dim
    g = torch.Generator(device=device).manual_seed(8)
    res = {"workload": case.name, "note": "query heads = 8 x G; K/V bytes identical across G"}
    for G in (1, 2, 4, 8):
        q = torch.randn((S, 8 * G, D), generator=g, device=device).to(case.dtype)
        out = torch.empty((S, 8 * G, D), dtype=torch.float32, device=device)

        def dec():
            pa.pa_decode(out, q, st.kc, st.vc, st.bt, st.cl, st.max_ctx, case.scale, workspace=st.ws)
        for _ in range(3):
            dec()
        ms, _ = time_steps(dec, 30, flush, False)
        t = statistics.median(ms)
        b = decode_bytes(case)["kv"] + S * 8 * G * D * (2 + 4)
        res[f"G{G}"] = {"ms": round(t, 5), "GB/s": round(b / t / 1e6, 1), "frac_hbm": round(b / t / 1e6 / hbm_peak, 4)}
    del st
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- CPU oracle

def _oracle_step(oracle, case, kc, vc):
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, case.block_size)
    return oracle.paged_attention(case.query, case.query_start_loc, kc, vc, case.block_tables,
                                  case.context_lens, case.scale)


def cpu_baseline(case, byts, reps: int = 2):
    """The fp64 oracle, as it stands, on the host cores: whole steps of the same workload."""
    import oracle
    oracle.build()
    kc, vc = case.key_cache.clone(), case.value_cache.clone()
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        _oracle_step(oracle, case, kc, vc)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return {"value": round(byts["step"] / t / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds_per_step": round(t, 3),
            "sample": f"{reps} whole steps of the same workload ({case.num_seqs} sequences, all heads), median",
            "per_workload": {"decode_batch": oracle_decode_timing("decode_batch", reps),
                             "decode_batch_single_thread": oracle_single_thread("decode_batch", reps),
                             "prefill_chunk": oracle_prefill_timing()},
            "kv_manager_reference": reference_manager_measurement()}


def oracle_decode_timing(workload: str, reps: int = 2) -> dict:
    """The oracle on whole decode steps of a workload (cache write + attention), median."""
    import oracle
    oracle.build()
    case = workloads.WORKLOADS[workload]()
    kc, vc = case.key_cache.clone(), case.value_cache.clone()
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        _oracle_step(oracle, case, kc, vc)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    b = decode_bytes(case)["step"]
    return {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "seconds_per_step": round(t, 3), "seq_steps_per_s": round(case.num_seqs / t, 2),
            "sample": f"{reps} whole steps of {case.name}, median"}


def oracle_single_thread(workload: str, reps: int = 2) -> dict:
    """oracle_decode_timing with one thread: a child process started with OMP_NUM_THREADS=1
    (the oracle's thread count is fixed when its library loads)."""
    code = (f"import sys, json; sys.path.insert(0, {str(ROOT)!r}); import bench; "
            f"print(json.dumps(bench.oracle_decode_timing({workload!r}, {reps})))")
    env = {**os.environ, "OMP_NUM_THREADS": "1"}
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=900, cwd=str(ROOT))
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout).strip().splitlines()[-1:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_prefill_timing(budget_s: float = 8.0) -> dict:
    """The oracle on a bounded sample of the chunked-prefill workload: the last R rows of
    every sequence's chunk (all heads), R chosen so that one run takes about budget_s."""
    import oracle
    oracle.build()
    case = workloads.prefill_chunk()
    kc, vc = case.key_cache.clone(), case.value_cache.clone()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, case.block_size)
    qsl = case.query_start_loc.tolist()

    def sub_case(rows):
        sub = workloads.PagedCase(**{**case.__dict__})
        idx = torch.cat([torch.arange(qsl[s + 1] - min(rows, qsl[s + 1] - qsl[s]), qsl[s + 1])
                         for s in range(case.num_seqs)])
        sub.query = case.query[idx].contiguous()
        lens = [min(rows, qsl[s + 1] - qsl[s]) for s in range(case.num_seqs)]
        sub.query_start_loc = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
        return sub

    def run(sub):
        t0 = time.perf_counter()
        oracle.paged_attention(sub.query, sub.query_start_loc, kc, vc, sub.block_tables,
                               sub.context_lens, case.scale)
        return time.perf_counter() - t0

    probe = sub_case(2)
    per_row = run(probe) / 2
    lq = max(qsl[s + 1] - qsl[s] for s in range(case.num_seqs))
    rows = int(max(1, min(lq, budget_s / max(per_row, 1e-9))))
    sub = sub_case(rows)
    t = run(sub)
    flops, _ = prefill_work(sub)
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "seconds": round(t, 3),
            "sample": f"last {rows} chunk rows of each of the {case.num_seqs} sequences of {case.name}, all heads"}


def reference_manager_measurement():
    """The reference KV-cache manager (plain Python) on the library manager's stream."""
    from oracle.kv_manager import ReferenceKVManager
    calls = manager_stream()
    mgr = ReferenceKVManager(16384, 16)
    t0 = time.perf_counter()
    n = replay_manager(mgr, calls)
    dt = time.perf_counter() - t0
    return {"stream": MANAGER_STREAM, "calls": n, "s": round(dt, 4), "calls_per_s": round(n / dt, 1),
            "cores": 1, "kind": "oracle"}


def reference_arm(args, rank, world, budget_s: float = 150.0):
    """``--impl reference``: the fp64 CPU oracle timed on the host cores (rank 0 only).

    Each step is a bounded sample of the workload -- the first sequence, all heads, its
    context truncated to the first T tokens -- with T calibrated so that the whole
    ``--warmup W --steps K`` run takes about ``budget_s`` seconds."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    case = workloads.WORKLOADS[args.workload]()
    kc, vc = case.key_cache.clone(), case.value_cache.clone()

    def sample(tokens: int):
        sub = workloads.PagedCase(**{**case.__dict__})
        sub.query = case.query[:1]
        sub.query_start_loc = case.query_start_loc[:2]
        sub.block_tables = case.block_tables[:1]
        sub.context_lens = torch.tensor([tokens], dtype=torch.int32)
        sub.new_key, sub.new_value = case.new_key[:1], case.new_value[:1]
        sub.slot_mapping = case.slot_mapping[:1]
        return sub

    if not case.is_decode:
        return reference_prefill(args, case, world)
    full = int(case.context_lens[0])
    probe = sample(min(full, 2048))
    t0 = time.perf_counter()
    _oracle_step(oracle, probe, kc, vc)
    per_token = (time.perf_counter() - t0) / int(probe.context_lens[0])
    target = budget_s / (args.steps + args.warmup)
    tokens = int(max(64, min(full, target / max(per_token, 1e-9))))
    sub = sample(tokens)
    sb = decode_bytes(sub)
    for _ in range(args.warmup):
        _oracle_step(oracle, sub, kc, vc)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_step(oracle, sub, kc, vc)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    value = sb["step"] / t / 1e9
    desc = (f"first sequence of {case.num_seqs}, all {case.num_heads} heads, context truncated "
            f"to its first {tokens} of {full} tokens, per step")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/k/v, shuffled block pool)",
        "config": {"workload": case.name, "sample": desc},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle",
                         "cores": oracle.num_threads(), "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def reference_prefill(args, case, world, budget_s: float = 150.0):
    """Reference arm on the prefill workload: the oracle on the first sequence's chunk,
    its rows truncated so that the whole run takes about ``budget_s`` seconds."""
    import oracle
    kc, vc = case.key_cache.clone(), case.value_cache.clone()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, case.block_size)
    lq = int(case.query_start_loc[1] - case.query_start_loc[0])

    def sub_case(rows):
        sub = workloads.PagedCase(**{**case.__dict__})
        sub.query = case.query[lq - rows:lq].contiguous()  # the chunk's last rows
        sub.query_start_loc = torch.tensor([0, rows], dtype=torch.int32)
        sub.block_tables = case.block_tables[:1]
        sub.context_lens = case.context_lens[:1]
        return sub

    def run(sub):
        return oracle.paged_attention(sub.query, sub.query_start_loc, kc, vc, sub.block_tables,
                                      sub.context_lens, case.scale)

    probe = sub_case(min(lq, 8))
    t0 = time.perf_counter()
    run(probe)
    per_row = (time.perf_counter() - t0) / int(probe.query.shape[0])
    rows = int(max(1, min(lq, budget_s / (args.steps + args.warmup) / max(per_row, 1e-9))))
    sub = sub_case(rows)
    flops, _ = prefill_work(sub)
    for _ in range(args.warmup):
        run(sub)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run(sub)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    value = flops / t / 1e12
    desc = f"last {rows} of the first sequence's {lq} chunk rows, all heads, per step"
    return {
        "impl": "reference", "metric": "paged-attn chunked-prefill TFLOP/s (causal-exact FLOPs)",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/k/v, shuffled block pool)",
        "config": {"workload": case.name, "sample": desc},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "kind": "oracle",
                         "cores": oracle.num_threads(), "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_decode", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", 1))
    rank = int(os.environ.get("RANK", 0))
    dist_on = world > 1
    if args.impl == "reference":
        line = reference_arm(args, rank, world)
    else:
        if dist_on:
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            torch.distributed.init_process_group("nccl")
        line = gpu_arm(args, rank, world, dist_on)
        if dist_on:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
