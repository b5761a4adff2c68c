"""Benchmark of the FP8 paged KV-cache hot path on GB300.

A step is one pass of the whole path over one batch of seeded synthetic input:
kvfp8_reshape_and_cache of the batch's K/V rows into the paged FP8 cache, then
kvfp8_paged_decode_attention of one query per sequence over that cache.  The metric is
achieved HBM bandwidth: algorithmic bytes (each input byte read once, each output byte
written once) divided by device time, in GB/s.

Default workload: long_context, the largest configuration (64 q / 8 kv heads, head_dim 128,
block 16, 8 sequences of 32768-131072 tokens; the step writes all ~655k context rows and
decodes 8 queries).  In the same run (unless --per-config off), the other timed
configurations are measured the same way and reported under "per_config":
  llama3_8b      write 262144 context rows, then decode 64 queries
  prefill_write  write 32768 rows (padding rows skipped)
  mixed_serving  write 1 new token per sequence, then decode 256 queries

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                  [--variant fp8|rope|k_bf16|v_bf16|multi]

--variant swaps in one of the widened forms of the path (same workload, same metric):
  fp8     (default) reshape_and_cache + paged_decode_attention, both caches E4M3
  rope    rope on K fused into the cache write (rope_reshape_and_cache), then decode
  k_bf16  mixed cache dtypes, K cache bf16 and V E4M3 (reshape_and_cache_mixed +
          paged_decode_attention_mixed); v_bf16 the other way round
  multi   causal multi-query attention (paged_attention_multi) with 16 // G query
          tokens per sequence (G = n_q / n_kv), after the same cache write
  prefill chunked prefill: the context is in the cache before timing; a step writes the
          last 512 tokens of every sequence (16 on mixed_serving) and runs causal
          attention for them (paged_attention_multi on its tensor-core kernel)

Under torchrun (N > 1) every rank runs the same workload on its own GPU (replicas, weak
scaling, no collective on the data path); the time is the max over ranks.

Timing: W warm-up steps, a short untimed soak, then K steps bracketed by events on the
launching stream.  Just before the first timed step a GPU-side wait of a few milliseconds
is enqueued (outside the timed region), so the host has queued every timed launch before
the GPU reaches them: the steps run back to back and no host enqueue gap falls inside an
event interval.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = {
    "reshape_and_cache": ["fp8_paged_kv_reshape_gb300/csrc/reshape_and_cache.cu",
                          "fp8_paged_kv_reshape_gb300/csrc/kvfp8_device.cuh"],
    "paged_decode_attention": ["fp8_paged_kv_reshape_gb300/csrc/paged_decode_kernel.cuh",
                               "fp8_paged_kv_reshape_gb300/csrc/kvfp8_device.cuh"],
    # the multi-query calls whose long chunks run on the tensor-core kernels
    "prefill_attention": ["fp8_paged_kv_reshape_gb300/csrc/prefill_attention.cu",
                          "fp8_paged_kv_reshape_gb300/csrc/paged_decode_kernel.cuh",
                          "fp8_paged_kv_reshape_gb300/csrc/kvfp8_device.cuh"],
}
VARIANTS = ("fp8", "rope", "k_bf16", "v_bf16", "multi", "prefill")
# a CPU sample of the multi-query forms attends with at most this many oracle FLOPs: the
# last m of a sequence's new tokens (a 512-token chunk over a 128K context would otherwise
# take the double-precision oracle most of an hour)
SAMPLE_QUERY_FLOPS = 1 << 28
# a CPU sample takes at most this many tokens of a sequence (its first ones), so that one
# sample of a 128K-token context stays near a second of oracle time
SAMPLE_MAX_TOKENS = 8192
METRIC = "FP8 paged decode attn KV-read GB/s & cache-write GB/s, % of GB300 HBM peak"


# ----------------------------------------------------------------- byte accounting

def reshape_bytes(w: workloads.Workload, slot_mapping: np.ndarray, src_elem: int = 2,
                  k_elem: int = 1, v_elem: int = 1, positions: np.ndarray | None = None,
                  rot: int = 0) -> int:
    """Algorithmic bytes of one cache write: per valid row K+V read at src_elem bytes and
    written at k_elem / v_elem bytes (1 for E4M3, 2 for a bf16 side), plus the 8-byte slot of
    every row (padding rows read only it).  The rope-fused write also reads every row's
    8-byte position and, once, the float32 table row of every distinct position."""
    row = w.n_kv * w.head_dim
    ok = slot_mapping >= 0
    valid = int(np.count_nonzero(ok))
    n = valid * row * (2 * src_elem + k_elem + v_elem) + 8 * int(slot_mapping.size)
    if positions is not None:
        n += 8 * int(slot_mapping.size) + 4 * rot * int(np.unique(positions[ok]).size)
    return n


def decode_bytes(w: workloads.Workload, seq_lens: np.ndarray, k_elem: int = 1, v_elem: int = 1,
                 query_rows: int | None = None) -> int:
    """Algorithmic bytes of one attention call: every cached K and V byte of every sequence
    (k_elem / v_elem bytes per element), its block-table entries and length, the bf16 query
    rows in and the bf16 output rows out; the multi-query form (query_rows given) also reads
    the num_seqs + 1 query_start_loc entries."""
    L = seq_lens.astype(np.int64)
    row = w.n_kv * w.head_dim
    kv = int((L * row).sum()) * (k_elem + v_elem)
    tables = int((4 * np.ceil(L / w.block_size)).sum()) + 4 * L.size
    rows = L.size if query_rows is None else query_rows
    qo = 2 * 2 * rows * w.n_q * w.head_dim
    qsl = 0 if query_rows is None else 4 * (L.size + 1)
    return kv + tables + qo + qsl


def query_len(w: workloads.Workload, variant: str, seq_lens: np.ndarray | None = None) -> int:
    """Query tokens per sequence: 16 // G score columns' worth for the multi-query variant;
    for prefill a 512-token chunk, or the shortest context when that is shorter (16 on the
    serving mix)."""
    if variant == "multi":
        return max(1, 16 // (w.n_q // w.n_kv))
    if variant == "prefill":
        shortest = int(seq_lens.min()) if seq_lens is not None and seq_lens.size else 512
        return max(1, min(512, shortest))
    return 1


def attention_flops(w: workloads.Workload, seq_lens: np.ndarray, qlen: int) -> int:
    """Tensor FLOPs of causal attention for qlen new tokens per sequence: every (query head,
    visible key) pair costs 2*hd for q.k and 2*hd for p.v; token j of a sequence of length
    L sees L - qlen + j + 1 keys."""
    L = seq_lens.astype(np.int64)
    pairs = int((qlen * (L - qlen) + qlen * (qlen + 1) // 2).sum())
    return 4 * w.head_dim * w.n_q * pairs


def step_rows(w: workloads.Workload, lay: workloads.Layout, qlen: int, serving: bool = False):
    """(slots, positions) of the rows one step writes: every context row, or for a serving
    step the last qlen tokens of every sequence (sequence-major)."""
    if w.kind != "mixed" and not serving:
        return lay.slot_mapping, np.maximum(lay.row_pos, 0).astype(np.int64)
    L = lay.seq_lens.astype(np.int64)
    pos = (L[:, None] - qlen + np.arange(qlen)[None, :]).reshape(-1)
    seq = np.repeat(np.arange(lay.num_seqs), qlen)
    slots = lay.block_tables[seq, pos // w.block_size].astype(np.int64) * w.block_size + \
        pos % w.block_size
    return slots, pos


# ----------------------------------------------------------------- helpers

def max_over_ranks(x: float, world: int, device) -> float:
    """The maximum of x over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the bytes every rank processed over the slowest rank's time."""
    return world * bytes_per_step * steps / (max_ms * 1e-3) / 1e9


def source_sha(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense f16/bf16 tensor TFLOP/s: the measured sustained cuBLAS bf16 figure (the kernel
    runs inside a step repeated back to back; f16 and bf16 share one tensor rate)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured (bf16 sustained)"
    return 1700.0, "fallback (bf16 sustained)"


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(kernel, {}).get(workload)
    if not rec or rec.get("source_sha") != source_sha(KERNEL_SOURCES[kernel]):
        return None
    return int(rec["bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.t0 = time.time()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        self.samples = []

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append(dict(sm=float(parts[1]), sm_max=float(parts[2]),
                                         reasons=parts[4:9]))
            except ValueError:
                continue

    def summary(self):
        if not self.samples:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        active = set()
        for s in self.samples:
            for n, v in zip(names, s["reasons"][1:]):
                if v.lower() in ("active", "1"):
                    active.add(n)
        sm = [s["sm"] for s in self.samples]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(s["sm_max"] for s in self.samples),
                "reasons": sorted(active), "samples": len(sm)}


# ----------------------------------------------------------------- problem set-up

class Problem:
    """Device-resident inputs, caches and outputs of one workload in one variant."""

    def __init__(self, name: str, device, num_seqs: int | None = None, variant: str = "fp8"):
        import fp8_paged_kv_reshape_gb300 as kv

        self.kv = kv
        self.w = w = workloads.WORKLOADS[name]
        self.variant = variant
        if variant in ("multi", "prefill") and w.kind == "write":
            raise ValueError("the %s workload has no attention step" % name)
        self.lay = lay = workloads.make_layout(w, num_seqs=num_seqs)
        self.device = device
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.qlen = query_len(w, variant, lay.seq_lens)
        self.ksc = workloads.scale_tensor(w.k_scale, w.scale_dtype, device)
        self.vsc = workloads.scale_tensor(w.v_scale, w.scale_dtype, device)
        self.k_elem = 2 if variant == "k_bf16" else 1
        self.v_elem = 2 if variant == "v_bf16" else 1
        self.kc = self._new_cache(self.k_elem)
        self.vc = self._new_cache(self.v_elem)
        self.rot = w.head_dim
        self.table = None
        if variant == "rope":
            max_pos = max(1, int(lay.seq_lens.max()) if lay.num_seqs else 1)
            self.table = torch.from_numpy(workloads.rope_table(max_pos, self.rot)).to(device)
        self.serving = w.kind == "mixed" or variant == "prefill"
        slots, pos = step_rows(w, lay, self.qlen, self.serving)
        if self.serving:
            # the cache holds the context before the timed region; a step writes the last
            # qlen tokens of every sequence and attends
            ctx_k, ctx_v = workloads.make_kv(w, lay.slot_mapping.size, device)
            self._write(ctx_k, ctx_v, torch.from_numpy(lay.slot_mapping).to(device),
                        torch.from_numpy(lay.row_pos.astype(np.int64)).to(device))
            del ctx_k, ctx_v
            self.k, self.v = workloads.make_new_token_kv(w, lay.num_seqs * self.qlen, device)
        else:
            self.k, self.v = workloads.make_kv(w, lay.slot_mapping.size, device)
        self.slots_np, self.pos_np = slots, pos
        self.slots = torch.from_numpy(slots).to(device)
        self.pos = torch.from_numpy(pos).to(device) if variant == "rope" else None
        self.decode = w.kind != "write"
        if self.decode:
            rows = lay.num_seqs * self.qlen
            self.q = workloads.make_query(w, rows, device)
            self.bt = torch.from_numpy(lay.block_tables).to(device)
            self.sl = torch.from_numpy(lay.seq_lens).to(device)
            self.qsl = torch.arange(0, rows + 1, self.qlen, dtype=torch.int32, device=device) \
                if variant in ("multi", "prefill") else None
            self.out = torch.empty_like(self.q)
            if self.qsl is not None:
                need = kv.paged_attention_multi_workspace_size(lay.num_seqs, w.n_q, w.n_kv,
                                                                w.head_dim, self.qlen)
            else:
                need = kv.paged_decode_workspace_size(lay.num_seqs, w.n_q, w.head_dim)
            self.tensor_route = self.qsl is not None and need == 0
            self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        self.rs_bytes = reshape_bytes(w, slots, 2, self.k_elem, self.v_elem,
                                      pos if variant == "rope" else None, self.rot)
        self.dec_bytes = decode_bytes(w, lay.seq_lens, self.k_elem, self.v_elem,
                                      self.lay.num_seqs * self.qlen if self.qsl is not None else None) \
            if self.decode else 0
        self.attn_flops = attention_flops(w, lay.seq_lens, self.qlen) if self.decode else 0

    def _new_cache(self, elem: int) -> torch.Tensor:
        if elem == 1:
            return workloads.new_cache(self.lay.num_blocks, self.w, self.device)
        w = self.w
        return torch.zeros((self.lay.num_blocks, w.block_size, w.n_kv, w.head_dim),
                           dtype=torch.bfloat16, device=self.device)

    def _write(self, k, v, slots, pos):
        kv = self.kv
        if self.variant == "rope":
            kv.rope_reshape_and_cache(k, v, self.kc, self.vc, slots, pos, self.table, True,
                                      self.ksc, self.vsc, status=self.status)
        elif self.variant in ("k_bf16", "v_bf16"):
            kv.reshape_and_cache_mixed(k, v, self.kc, self.vc, slots, self.ksc, self.vsc,
                                       status=self.status)
        else:
            kv.reshape_and_cache(k, v, self.kc, self.vc, slots, self.ksc, self.vsc,
                                 status=self.status)

    def reshape(self):
        self._write(self.k, self.v, self.slots, self.pos)

    def attend(self):
        kv = self.kv
        if self.qsl is not None:
            kv.paged_attention_multi(self.q, self.qsl, self.qlen, self.kc, self.vc, self.bt,
                                     self.sl, self.ksc, self.vsc, out=self.out, workspace=self.ws,
                                     status=self.status)
        elif self.variant in ("k_bf16", "v_bf16"):
            kv.paged_decode_attention_mixed(self.q, self.kc, self.vc, self.bt, self.sl, self.ksc,
                                            self.vsc, out=self.out, workspace=self.ws,
                                            status=self.status)
        else:
            kv.paged_decode_attention(self.q, self.kc, self.vc, self.bt, self.sl, self.ksc,
                                      self.vsc, out=self.out, workspace=self.ws,
                                      status=self.status)

    def step_inputs(self):
        """The device tensors a step consumes that a caller supplies per step."""
        ins = [self.k, self.v, self.slots]
        if self.pos is not None:
            ins.append(self.pos)
        if self.decode:
            ins += [self.q, self.bt, self.sl]
            if self.qsl is not None:
                ins.append(self.qsl)
        return ins

    def set_step_inputs(self, ins):
        """Point the step at another set of input tensors (the order of step_inputs)."""
        it = iter(ins)
        self.k, self.v, self.slots = next(it), next(it), next(it)
        if self.pos is not None:
            self.pos = next(it)
        if self.decode:
            self.q, self.bt, self.sl = next(it), next(it), next(it)
            if self.qsl is not None:
                self.qsl = next(it)

    def attention_launches(self) -> int:
        # plan + split-KV attention + combine, or one tensor-core attention kernel
        return (1 if self.tensor_route else 3) if self.decode else 0

    def launches_per_step(self) -> int:
        return 1 + self.attention_launches()

    def describe(self) -> dict:
        w, lay = self.w, self.lay
        write = {"fp8": "reshape_and_cache", "multi": "reshape_and_cache",
                 "prefill": "reshape_and_cache",
                 "rope": "rope_reshape_and_cache", "k_bf16": "reshape_and_cache_mixed",
                 "v_bf16": "reshape_and_cache_mixed"}[self.variant]
        attn = {"multi": "paged_attention_multi", "prefill": "paged_attention_multi (tcgen05)",
                "k_bf16": "paged_decode_attention_mixed",
                "v_bf16": "paged_decode_attention_mixed"}.get(self.variant,
                                                              "paged_decode_attention")
        d = {"workload": w.name, "variant": self.variant, "n_q": w.n_q, "n_kv": w.n_kv,
             "head_dim": w.head_dim, "block_size": w.block_size, "num_seqs": lay.num_seqs,
             "context_tokens": int(lay.seq_lens.sum()),
             "rows_written_per_step": int(self.slots_np.size),
             "k_scale": w.k_scale, "v_scale": w.v_scale, "scale_dtype": w.scale_dtype,
             "k_cache": "bf16" if self.k_elem == 2 else "e4m3",
             "v_cache": "bf16" if self.v_elem == 2 else "e4m3"}
        if self.decode:
            d["query_tokens_per_seq"] = self.qlen
            d["step"] = "%s(%d rows) + %s(%d seqs x %d queries)" % (
                write, self.slots_np.size, attn, lay.num_seqs, self.qlen)
        else:
            d["step"] = "%s(%d rows)" % (write, self.slots_np.size)
        if self.variant == "rope":
            d["rope"] = {"rot_dim": self.rot, "neox": True, "theta": 500000.0,
                         "table": "float32 [%d, %d], resident" % tuple(self.table.shape)}
        per_step = self.rs_bytes + self.dec_bytes
        d["l2"] = ("inputs larger than L2 (%.2f GB of algorithmic traffic per step), no flush"
                   % (per_step / 1e9)) if per_step > L2_BYTES else \
            "L2 flushed between steps (a %d MB buffer written)" % (2 * L2_BYTES >> 20)
        return d


# ----------------------------------------------------------------- timed runs

TIMING_NOTE = ("value and ms_per_step: K steps back to back with no event between kernels; "
               "kernels[*].ms and the roofline: a second pass of K steps with an event around "
               "each kernel group (evented_ms_per_step: that pass's step time)")
NOMINAL_HBM_GBS = 8000.0  # the GB300's ~8 TB/s HBM3e figure, for context beside the measured peak
PER_CONFIG = ("llama3_8b", "prefill_write", "mixed_serving")
CLOCK_HZ = 2.07e9  # the GB300's maximum SM clock, for sizing the pre-timing GPU wait


def time_problem(p: "Problem", args, world, device) -> dict:
    """Time K steps of one problem (after W warm-up steps and a short soak) with CUDA events
    on the launching stream: the whole timed region, and each kernel group inside every step.
    Returns the slowest rank's total and this rank's per-kernel means."""
    per_step = p.rs_bytes + p.dec_bytes
    flush = None if per_step > L2_BYTES else torch.empty(2 * L2_BYTES, dtype=torch.uint8,
                                                         device=device)
    stream = torch.cuda.current_stream(device)

    def step(evs=None):
        if flush is not None:
            flush.fill_(1)
        if evs:
            evs[0].record(stream)
        p.reshape()
        if evs:
            evs[1].record(stream)
        if p.decode:
            p.attend()
        if evs:
            evs[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    assert int(p.status.item()) == 0, "device status set during warm-up"

    sampler = ClockSampler(device.index if device.index is not None else 0)
    # keep the GPU busy for ~0.5 s before timing so the sampler sees it under load; measure
    # the host's cost of enqueueing one step on the way
    host = []
    t_end = time.time() + 0.5
    while time.time() < t_end:
        h0 = time.perf_counter()
        step()
        host.append(time.perf_counter() - h0)
        torch.cuda.synchronize(device)
    host_s = statistics.median(host) if host else 1e-4

    def timed_pass(with_events: bool):
        """K steps back to back between two events; with_events adds an event around each
        kernel group (a timestamped event drains the GPU's pipeline between launches, which
        costs a few microseconds a step, so the value comes from a pass without them)."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
               for _ in range(args.steps)] if with_events else None
        t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        # a GPU-side wait, outside the timed region, long enough for the host to queue every
        # timed launch first: the timed steps then run back to back on the device
        wait_s = min(0.25, 2.0 * args.steps * (host_s + 20e-6) + 1e-3)
        torch.cuda._sleep(int(wait_s * CLOCK_HZ))
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i] if evs else None)
        t_stop.record(stream)
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()
        return t_start.elapsed_time(t_stop), evs

    # the value: K steps with nothing between the kernels; then K more steps with events
    # around each kernel group for the per-kernel durations (the roofline's)
    total_ms, _ = timed_pass(False)
    evented_ms, evs = timed_pass(True)
    sampler.stop()
    rs_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps if p.decode else 0.0
    assert int(p.status.item()) == 0, "device status set during the timed steps"
    total_ms = max_over_ranks(total_ms, world, device)
    return {"total_ms": total_ms, "rs_ms": rs_ms, "dec_ms": dec_ms,
            "evented_ms_per_step": evented_ms / args.steps,
            "host_enqueue_ms_per_step": host_s * 1e3, "clocks": sampler.summary()}


def kernel_report(p: "Problem", t: dict, workload: str, variant: str):
    """Per-kernel-group bytes, event-timed ms, GB/s and fractions (of the measured HBM peak
    and of the nominal 8 TB/s), and the dominant kernel's roofline object."""
    peak, peak_kind = measured_peaks()
    kernels = {"reshape_and_cache": {"bytes_per_launch": p.rs_bytes, "ms": t["rs_ms"],
                                     "gbs": p.rs_bytes / (t["rs_ms"] * 1e-3) / 1e9}}
    if p.decode:
        kernels["paged_decode_attention"] = {"bytes_per_launch": p.dec_bytes, "ms": t["dec_ms"],
                                             "gbs": p.dec_bytes / (t["dec_ms"] * 1e-3) / 1e9,
                                             "launches": p.attention_launches()}
    for k in kernels.values():
        k["frac"] = k["gbs"] / peak
        k["frac_of_nominal_8tbs"] = k["gbs"] / NOMINAL_HBM_GBS
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    # the attention group of the tensor-core route is recorded under its own kernel source
    rec_kernel = "prefill_attention" if dom == "paged_decode_attention" and p.decode and p.tensor_route else dom
    traffic = recorded_traffic(rec_kernel, workload if variant == "fp8" else "%s:%s" % (workload, variant))
    if p.decode and p.tensor_route:
        att = kernels["paged_decode_attention"]
        att["tflops"] = p.attn_flops / (att["ms"] * 1e-3) / 1e12
        att["flops_per_launch"] = p.attn_flops
    if dom == "paged_decode_attention" and p.tensor_route:
        tpeak, tkind = measured_tensor_peak()
        att = kernels[dom]
        roof = {"bound": "tensor", "kernel": dom, "achieved": att["tflops"], "peak": tpeak,
                "peak_kind": tkind, "unit": "TFLOP/s", "frac": att["tflops"] / tpeak,
                "traffic": traffic, "algorithmic_flops_per_launch": p.attn_flops,
                "algorithmic_bytes_per_launch": att["bytes_per_launch"]}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["gbs"], "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": kernels[dom]["gbs"] / peak,
                "frac_of_nominal_8tbs": kernels[dom]["gbs"] / NOMINAL_HBM_GBS,
                "traffic": traffic,
                "algorithmic_bytes_per_launch": kernels[dom]["bytes_per_launch"]}
    return kernels, roof


def run_per_config(args, world, device) -> dict:
    """The other timed configurations, each measured exactly as the main one (own warm-up,
    soak, clock samples and event timing); one problem on the device at a time."""
    res = {}
    for name in PER_CONFIG:
        if name == args.workload:
            continue
        p = Problem(name, device, None, "fp8")
        t = time_problem(p, args, world, device)
        kernels, roof = kernel_report(p, t, name, "fp8")
        per_step = p.rs_bytes + p.dec_bytes
        res[name] = {"value": whole_job_gbs(per_step, args.steps, world, t["total_ms"]),
                     "unit": "GB/s", "ms_per_step": t["total_ms"] / args.steps,
                     "config": p.describe(), "kernels": kernels, "roofline": roof,
                     "gpu_launches": p.launches_per_step() * args.steps,
                     "evented_ms_per_step": t["evented_ms_per_step"],
                     "host_enqueue_ms_per_step": t["host_enqueue_ms_per_step"],
                     "clocks": t["clocks"]}
        del p
        torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, device):
    import fp8_paged_kv_reshape_gb300 as kv  # noqa: F401  (fails loudly without the library)

    p = Problem(args.workload, device, args.num_seqs, args.variant)
    per_step = p.rs_bytes + p.dec_bytes
    t = time_problem(p, args, world, device)
    total_ms = t["total_ms"]
    e2e = run_e2e(args, p, device) if not args.no_e2e else None
    if e2e is not None:
        e2e["ms_per_step"] = max_over_ranks(e2e["ms_per_step"], world, device)
        e2e["value"] = whole_job_gbs(per_step, 1, world, e2e["ms_per_step"])
    kernels, roof = kernel_report(p, t, args.workload, args.variant)
    describe = p.describe()
    launches = p.launches_per_step() * args.steps
    del p
    torch.cuda.empty_cache()
    per_config = None
    want_per_config = args.per_config == "on" or (
        args.per_config == "auto" and args.workload == "long_context" and args.variant == "fp8"
        and args.num_seqs is None)
    if want_per_config:
        per_config = run_per_config(args, world, device)

    if rank != 0:
        return None
    value = whole_job_gbs(per_step, args.steps, world, total_ms)
    line = {
        "metric": METRIC,
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3",
        "compute": "f32 divide + E4M3 encode; fp16 (bf16 for a bf16 cache side) mma.sync "
                   "with f32 accumulate",
        "data": "synthetic (seeded; see workloads/)",
        "config": describe, "roofline": roof, "kernels": kernels,
        "gpu_launches": launches,
        "timing": TIMING_NOTE, "evented_ms_per_step": t["evented_ms_per_step"],
        "host_enqueue_ms_per_step": t["host_enqueue_ms_per_step"],
        "clocks": t["clocks"], "e2e": e2e,
    }
    if per_config is not None:
        line["per_config"] = per_config
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, target_s=args.cpu_seconds,
                                            variant=args.variant)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(
            args.workload, target_s=max(2.0, args.cpu_seconds / 3), variant=args.variant)
    return line


def gpu_local_cpus(device):
    """The host CPUs on the GPU's own NUMA node (from sysfs), or None where that is not
    available: pinned buffers allocated from one of them land in the memory next to the GPU's
    host link instead of behind the link between host sockets."""
    try:
        pr = torch.cuda.get_device_properties(device)
        bus = "%04x:%02x:%02x.0" % (getattr(pr, "pci_domain_id", 0), pr.pci_bus_id, pr.pci_device_id)
        with open("/sys/bus/pci/devices/%s/local_cpulist" % bus) as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            if "-" in part:
                lo, hi = part.split("-")
                cpus.update(range(int(lo), int(hi) + 1))
            elif part:
                cpus.add(int(part))
        avail = os.sched_getaffinity(0)
        cpus &= avail
        return cpus if cpus and cpus != avail else None
    except (OSError, ValueError, AttributeError):
        return None


def run_e2e(args, p: Problem, device):
    """The end-to-end leg, run with the process on the GPU's own host CPUs (where sysfs names
    them) so that its pinned buffers are allocated in the memory next to the GPU."""
    local = gpu_local_cpus(device)
    old = os.sched_getaffinity(0) if local else None
    if local:
        os.sched_setaffinity(0, local)
    try:
        r = run_e2e_pinned(args, p, device)
    finally:
        if old:
            os.sched_setaffinity(0, old)
    r["host_cpus"] = "GPU-local NUMA node (%d CPUs)" % len(local) if local else "unrestricted"
    return r


def run_e2e_pinned(args, p: Problem, device):
    """Same metric through the public API with host inputs: every step copies its inputs
    from pinned host memory and reads the output back, inside the timed region.  As a serving
    loop would, the copies go on a copy stream into two alternating device input sets, so
    step i+1's inputs cross the host link while step i computes."""
    import fp8_paged_kv_reshape_gb300 as kv  # noqa: F401  (the library the steps call)

    dev_a = p.step_inputs()
    host = [d.cpu().pin_memory() for d in dev_a]
    sets = [dev_a, [torch.empty_like(d) for d in dev_a]]
    if p.decode:
        hout = torch.empty(p.out.shape, dtype=p.out.dtype).pin_memory()
    stream = torch.cuda.current_stream(device)
    copy_stream = torch.cuda.Stream(device)
    h2d = sum(h.numel() * h.element_size() for h in host)
    d2h = hout.numel() * hout.element_size() if p.decode else 4
    hstat = torch.empty(1, dtype=torch.int32).pin_memory()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]
    used = [False, False]

    def step(i):
        b = i & 1
        with torch.cuda.stream(copy_stream):
            if used[b]:  # the set's previous step has finished with it
                copy_stream.wait_event(consumed[b])
            for h, d in zip(host, sets[b]):
                d.copy_(h, non_blocking=True)
            copied[b].record(copy_stream)
        stream.wait_event(copied[b])
        p.set_step_inputs(sets[b])
        p.reshape()
        if p.decode:
            p.attend()
            consumed[b].record(stream)
            hout.copy_(p.out, non_blocking=True)
        else:
            consumed[b].record(stream)
            hstat.copy_(p.status, non_blocking=True)
        used[b] = True

    for i in range(max(1, min(args.warmup, 3))):
        step(i)
    torch.cuda.synchronize(device)
    n = max(1, min(args.steps, 20))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    copy_stream.wait_event(a)
    for i in range(n):
        step(i)
    b.record(stream)
    torch.cuda.synchronize(device)
    p.set_step_inputs(dev_a)
    ms = a.elapsed_time(b) / n
    per_step = p.rs_bytes + p.dec_bytes
    return {"value": per_step / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "steps": n, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelining": "inputs copied on a second stream into two alternating device sets"}


# ----------------------------------------------------------------- CPU oracle legs

def sampled_queries(w: workloads.Workload, qlen: int, seq_len: int) -> int:
    """How many of a sequence's qlen new tokens (its last ones) a CPU sample attends with."""
    per_token = 4 * w.head_dim * w.n_q * max(1, seq_len)
    return int(min(qlen, max(1, SAMPLE_QUERY_FLOPS // per_token)))


def _oracle_sample(w: workloads.Workload, lay: workloads.Layout, seqs, k_all, v_all, q,
                   variant: str = "fp8", max_tokens: int | None = SAMPLE_MAX_TOKENS):
    """Run the CPU oracle on the given sequences of the workload in the given variant: write
    their rows into a cache, then attend with every head of them.  A sequence longer than
    max_tokens is sampled as its first max_tokens tokens (a shorter sequence of the same
    workload: written, then attended over whole).  The multi-query forms attend with the
    last m of each sequence's qlen new tokens (sampled_queries; token j of those m sees the
    same keys as in the full chunk) and are credited m/qlen of the sequences' attention
    bytes.  Returns (seconds, algorithmic bytes)."""
    import oracle

    ks = workloads.stored_scale(w.k_scale, w.scale_dtype)
    vs = workloads.stored_scale(w.v_scale, w.scale_dtype)
    rows = np.nonzero(np.isin(lay.row_seq, seqs))[0] if lay.row_seq.size else np.zeros(0, int)
    if max_tokens is not None:
        rows = rows[lay.row_pos[rows] < max_tokens]
    kh = k_all[torch.from_numpy(rows)].contiguous()
    vh = v_all[torch.from_numpy(rows)].contiguous()
    pos = np.maximum(lay.row_pos[rows], 0).astype(np.int64)
    # the sampled sequences' physical blocks, relabelled 0..n-1 into a pool of their own
    # (the store and the attention do not depend on which physical block holds a page)
    bt_full = lay.block_tables[seqs]
    if max_tokens is not None:
        bt_full = bt_full[:, :-(-max_tokens // w.block_size)]
    used = np.unique(bt_full[bt_full >= 0])
    relabel = np.full(lay.num_blocks, -1, np.int64)
    relabel[used] = np.arange(used.size)
    bs = w.block_size
    slots_full = lay.slot_mapping[rows]
    slots = np.where(slots_full >= 0, relabel[np.maximum(slots_full, 0) // bs] * bs + slots_full % bs, -1)
    bt = np.where(bt_full >= 0, relabel[np.maximum(bt_full, 0)], -1).astype(np.int32)
    shape = (max(1, used.size), bs, w.n_kv, w.head_dim)
    k_elem = 2 if variant == "k_bf16" else 1
    v_elem = 2 if variant == "v_bf16" else 1
    kc = np.full(shape, workloads.SENTINEL, np.uint8 if k_elem == 1 else np.uint16)
    vc = np.full(shape, workloads.SENTINEL, np.uint8 if v_elem == 1 else np.uint16)
    kinds = (oracle.E4M3 if k_elem == 1 else oracle.CACHE_BF16,
             oracle.E4M3 if v_elem == 1 else oracle.CACHE_BF16)
    decode = w.kind != "write"
    sub_lens = lay.seq_lens[seqs]
    if max_tokens is not None:
        sub_lens = np.minimum(sub_lens, max_tokens).astype(np.int32)
    qlen = query_len(w, variant, lay.seq_lens)
    m = sampled_queries(w, qlen, int(sub_lens.max())) if variant in ("multi", "prefill") else qlen
    seq_idx = np.asarray(seqs)
    table = workloads.rope_table(max(1, int(lay.seq_lens.max())), w.head_dim) \
        if variant == "rope" else None
    t0 = time.perf_counter()
    if variant == "rope":
        oracle.rope_reshape_and_cache(kh, vh, kc, vc, slots, pos, table, w.head_dim, True,
                                      w.block_size, ks, vs)
    elif variant in ("k_bf16", "v_bf16"):
        oracle.reshape_and_cache_mixed(kh, vh, kc, kinds[0], vc, kinds[1], slots, w.block_size,
                                       ks, vs)
    else:
        oracle.reshape_and_cache(kh, vh, kc, vc, slots, w.block_size, ks, vs)
    if decode:
        if variant in ("multi", "prefill"):
            qrows = (seq_idx[:, None] * qlen + (qlen - m) + np.arange(m)[None, :]).reshape(-1)
            qsl = np.arange(0, qrows.size + 1, m, dtype=np.int32)
            oracle.paged_attention_multi(q[torch.from_numpy(qrows)], qsl, kc, vc, bt, sub_lens,
                                         ks, vs)
        elif variant in ("k_bf16", "v_bf16"):
            oracle.paged_decode_attention_mixed(q[torch.from_numpy(seq_idx)], kc, kinds[0], vc,
                                                kinds[1], bt, sub_lens, ks, vs)
        else:
            oracle.paged_decode_attention(q[torch.from_numpy(seq_idx)], kc, vc, bt, sub_lens,
                                          ks, vs)
    dt = time.perf_counter() - t0
    nbytes = reshape_bytes(w, slots, 2, k_elem, v_elem, pos if variant == "rope" else None,
                           w.head_dim)
    if decode:
        if variant in ("multi", "prefill"):
            nbytes += decode_bytes(w, sub_lens, k_elem, v_elem, len(seqs) * qlen) * m // qlen
        else:
            nbytes += decode_bytes(w, sub_lens, k_elem, v_elem)
    return dt, nbytes


def _cap_note(lay: workloads.Layout) -> str:
    if int(lay.seq_lens.max()) <= SAMPLE_MAX_TOKENS:
        return ""
    return "; a sequence longer than %d tokens is sampled as its first %d" % (
        SAMPLE_MAX_TOKENS, SAMPLE_MAX_TOKENS)


def _query_note(w: workloads.Workload, lay: workloads.Layout, variant: str) -> str:
    if variant not in ("multi", "prefill"):
        return _cap_note(lay)
    qlen = query_len(w, variant, lay.seq_lens)
    lo = sampled_queries(w, qlen, min(int(lay.seq_lens.max()), SAMPLE_MAX_TOKENS))
    hi = sampled_queries(w, qlen, min(int(lay.seq_lens.min()), SAMPLE_MAX_TOKENS))
    return ("; attention for the last %s of each sampled sequence's %d new tokens (at most "
            "2^28 oracle FLOPs), credited that fraction of its attention bytes%s"
            % (str(lo) if lo == hi else "%d-%d" % (lo, hi), qlen, _cap_note(lay)))


@functools.lru_cache(maxsize=2)
def _cpu_inputs(name, variant="fp8"):
    w = workloads.WORKLOADS[name]
    lay = workloads.make_layout(w)
    k, v = workloads.make_kv(w, lay.slot_mapping.size, "cpu")
    q = workloads.make_query(w, lay.num_seqs * query_len(w, variant, lay.seq_lens), "cpu")
    return w, lay, k, v, q


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline_all_cores(name: str, target_s: float = 4.0, variant: str = "fp8") -> dict:
    """The same oracle samples run side by side on every host core, one independent sample
    per thread (the oracle's C calls release the interpreter lock), for about target_s of
    wall time: throughput = all samples' algorithmic bytes / wall time."""
    import concurrent.futures as cf
    import itertools
    import threading

    w, lay, k, v, q = _cpu_inputs(name, variant)
    order = np.random.Generator(np.random.PCG64(w.seed + 7)).permutation(lay.num_seqs)
    cores = host_cores()
    nxt = itertools.cycle(order.tolist())
    lock = threading.Lock()
    t_end = time.perf_counter() + target_s

    def worker():
        nb, n = 0, 0
        while time.perf_counter() < t_end:
            with lock:
                s = next(nxt)
            nb += _oracle_sample(w, lay, [int(s)], k, v, q, variant)[1]
            n += 1
        return nb, n

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        res = list(ex.map(lambda _: worker(), range(cores)))
    wall = time.perf_counter() - t0
    nb = sum(r[0] for r in res)
    n = sum(r[1] for r in res)
    return {"value": nb / wall / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d sequence samples of %s, variant %s, on %d threads (one sample "
                      "per thread at a time), %.1f s wall%s"
                      % (n, name, variant, cores, wall, _query_note(w, lay, variant))}


def cpu_baseline(name: str, target_s: float = 12.0, variant: str = "fp8") -> dict:
    """The oracle as it stands, single-threaded on the host, on a bounded sample of the same
    workload (sequences, at most their first SAMPLE_MAX_TOKENS tokens: their rows written,
    then every head attended)."""
    w, lay, k, v, q = _cpu_inputs(name, variant)
    order = np.random.Generator(np.random.PCG64(w.seed + 5)).permutation(lay.num_seqs)
    t, nb, used = 0.0, 0, []
    for s in order:
        dt, b = _oracle_sample(w, lay, [int(s)], k, v, q, variant)
        t += dt
        nb += b
        used.append(int(s))
        if t >= target_s:
            break
    return {"value": nb / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%d of %d sequences of %s (%d tokens), variant %s: oracle write of their "
                      "rows + attention for all %d heads, %.1f s single-threaded%s"
                      % (len(used), lay.num_seqs, name,
                         int(np.minimum(lay.seq_lens[used], SAMPLE_MAX_TOKENS).sum()), variant,
                         w.n_q, t, _query_note(w, lay, variant))}


def run_reference(args):
    """The CPU oracle timed on the host cores on this arm's workload and metric: each step
    is a bounded sample (one sequence, at most its first SAMPLE_MAX_TOKENS tokens, its rows
    written and all heads decoded)."""
    w, lay, k, v, q = _cpu_inputs(args.workload, args.variant)
    order = np.random.Generator(np.random.PCG64(w.seed + 6)).permutation(lay.num_seqs)
    for i in range(args.warmup):
        _oracle_sample(w, lay, [int(order[i % lay.num_seqs])], k, v, q, args.variant)
    t, nb = 0.0, 0
    for i in range(args.steps):
        dt, b = _oracle_sample(w, lay, [int(order[(args.warmup + i) % lay.num_seqs])], k, v, q,
                               args.variant)
        t += dt
        nb += b
    value = nb / t / 1e9
    sample = ("each step: 1 of %d sequences of %s, variant %s, oracle write of its rows + "
              "attention for all %d heads, single-threaded%s"
              % (lay.num_seqs, args.workload, args.variant, w.n_q,
                 _query_note(w, lay, args.variant)))
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded; see workloads/)",
        "config": {"workload": args.workload, "variant": args.variant, "n_q": w.n_q, "n_kv": w.n_kv,
                   "head_dim": w.head_dim, "block_size": w.block_size},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_context", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--variant", default="fp8", choices=VARIANTS)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-config", choices=["auto", "on", "off"], default="auto",
                    help="also time llama3_8b, prefill_write and mixed_serving (auto: with the "
                         "default long_context workload)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="fewer sequences than the workload names (small profiling cases)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    line = run_ours(args, rank, world, device)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
