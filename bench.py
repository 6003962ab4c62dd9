#!/usr/bin/env python3
"""Decode-step benchmark of paged attention on GB300.

One step = the whole hot path over one synthetic decode batch through
pagedkv_decode_step: the slot of each sequence's new token, its append into
the pool, and the paged attention (the per-partition decode kernel, with the
append fused in, plus the log-sum-exp merge of sequences that span several
partitions).  The same step as three calls (slot mapping, reshape_and_cache,
paged_attention_decode) is timed beside it.  The default workload is the
largest single-GPU one: long-context split-K decode (B 8, 32/8 heads, d 128,
16-token blocks, lengths U{32768..131072}, 2.4 GB of KV per step).  Every
other decode workload (tiny, Llama-3.1-8B-like, shared prefix, Llama-2-70B-like
INT8) is measured the same way under ``rows.configs``, and the FP8,
multi-token and copy-on-write rows beside them.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the same workload instead (the reference arm: a plain fp64 program, not a
target).  Timing: CUDA events on the launching stream, W warm-up steps, K
timed steps, barrier + synchronize on both sides, max over ranks.  The KV
read per step of every bandwidth-bound workload is larger than the 129 MB L2,
so no flush is needed (the tiny workload fits in L2 and is reported as a
launch-latency figure).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged decode attention: KV-read GB/s & % of GB300 HBM peak; µs per decode step"
UNIT = "GB/s"
DEFAULT_CONFIG = 3
ROW_CONFIGS = (1, 2, 3, 4, 5)                       # the decode workloads under rows.configs
STEADY_S = 0.5                                        # length of the steady timed region
FALLBACK_HBM_GBS = 6800.0
GRAPH_STEPS = 20
L2_BYTES = 129e6                                         # GB300 L2
CSRC = os.path.join(ROOT, "paged_kv_cache_97_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# sources whose hash a stored DRAM-traffic capture of each kernel must match
KERNEL_SOURCES = {
    "decode_kernel": ("pagedkv_decode.cu", "pagedkv_device.cuh", "pagedkv_common.cuh"),
    "multi_tc_kernel": ("pagedkv_multi_tc.cu", "pagedkv_device.cuh", "pagedkv_common.cuh"),
    "multi_m16_kernel": ("pagedkv_multi_m16.cu", "pagedkv_device.cuh", "pagedkv_common.cuh"),
}


def workload_config(wl, nbytes) -> dict:
    """The workload as both arms report it in `config`: shapes, the seeded
    length mix and the KV bytes one step reads."""
    s = wl.spec
    return {"workload": s.name, "batch": s.batch, "num_q_heads": s.num_q_heads,
            "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim,
            "block_size": s.block_size, "kv_dtype": s.kv_dtype,
            "seq_lens": f"seed {wl.seed}: min {int(wl.seq_lens.min())}, "
                        f"mean {float(wl.seq_lens.mean()):.0f}, max {int(wl.seq_lens.max())}",
            "kv_bytes_per_step": nbytes["kv_logical"],
            "l2": ("inputs larger than L2 (KV read per step > 129 MB), no flush"
                   if nbytes["kv_logical"] > L2_BYTES else
                   "inputs fit in L2 and are not flushed: an L2-resident, launch-latency figure")}


# ---------------------------------------------------------------------------
# Byte accounting (algorithmic bytes per step)
# ---------------------------------------------------------------------------

def algorithmic_bytes(wl) -> dict:
    """Bytes the step must move at minimum: K/V of every attended token (a
    shared prefix counted once: it is read once from HBM and then hits L2),
    8-bit scales, the block-table entries in use, q and out, and the append's
    reads and writes."""
    s = wl.spec
    elem = wl.kv_elem_bytes
    B, hq, hkv, d, bs = s.batch, s.num_q_heads, s.num_kv_heads, s.head_dim, s.block_size
    T = wl.num_tokens                                    # query tokens (= B for decode)
    L = wl.seq_lens.astype(np.int64)
    blocks = int(((L + bs - 1) // bs).sum())
    kv_unique = wl.kv_bytes_unique()
    scales = blocks * 2 * hkv * 4 if s.kv_dtype != "bf16" else 0
    qo = 2 * T * hq * d * 2
    table = blocks * 4 + B * 4
    append = T * hkv * d * 2 * 2 + T * hkv * d * elem * 2 + T * 8 * 2
    attn = kv_unique + scales + qo + table
    return {"kv_logical": wl.kv_bytes_logical(), "kv_unique": kv_unique, "attention": attn,
            "step": attn + append}


# ---------------------------------------------------------------------------
# Clocks during the timed region (NVML through ctypes; reading only)
# ---------------------------------------------------------------------------

REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
           0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
           0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
           0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, uuid: str, period_s: float = 0.02):
        self.samples, self.max_mhz, self.reasons = [], None, set()
        self.period, self._stop, self._t, self.error = period_s, threading.Event(), None, None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            assert self.nvml.nvmlInit_v2() == 0
            self.h = ctypes.c_void_p()
            u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            assert self.nvml.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.h)) == 0
            m = ctypes.c_uint()
            assert self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(m)) == 0
            self.max_mhz = m.value
        except Exception as e:  # noqa: BLE001 - clocks are reported, not required
            self.error = f"nvml unavailable: {e!r}"

    def _run(self):
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            if fn(self.h, ctypes.byref(r)) == 0:
                for bit, name in REASONS.items():
                    if r.value & bit and bit != 0x1:
                        self.reasons.add(name)
            time.sleep(self.period)

    def __enter__(self):
        if self.error is None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self._t:
            self._stop.set()
            self._t.join()

    def summary(self):
        if self.error:
            return {"error": self.error}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples)}


# ---------------------------------------------------------------------------
# Ranks (replicas: every rank runs its own batch; no collective on the data path)
# ---------------------------------------------------------------------------

def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(elapsed_s: float, units_per_rank: float, world: int, dist=None):
    """Max time over ranks; whole-job throughput = units all ranks processed
    / that time."""
    if world > 1:
        import torch
        t = torch.tensor([elapsed_s], dtype=torch.float64)
        if dist.get_backend() == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_s = float(t.item())
    return elapsed_s, units_per_rank * world / elapsed_s


# ---------------------------------------------------------------------------
# Oracle (CPU baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_pools(wl):
    """The oracle's own pools for the whole batch (setup, not timed)."""
    import oracle
    oracle.build()
    return oracle.workload_pools(wl)


def oracle_time(wl, pools, seqs, threads):
    """Time the oracle's attention over every query head of ``seqs``.
    Returns (seconds, KV bytes attended)."""
    import oracle
    kc, vc, ks, vs = pools
    rows = np.array([(b, h) for b in seqs for h in range(wl.spec.num_q_heads)], np.int32)
    t0 = time.perf_counter()
    _, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale,
                                   k_scale=ks, v_scale=vs, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    assert rc == 0
    s = wl.spec
    kv = int(wl.seq_lens[list(seqs)].astype(np.int64).sum()) * 2 * s.num_kv_heads * s.head_dim * wl.kv_elem_bytes
    return dt, kv


def oracle_sample(wl, threads, target_s=10.0, max_s=30.0, pools=None):
    """Time the oracle for about target_s of work (bounded by max_s): growing
    prefixes of the batch, and when the whole batch takes less than
    target_s, repeated passes over it.  Returns a cpu_baseline dict."""
    if pools is None:
        pools = oracle_pools(wl)
    n = 2
    while True:
        seqs = list(range(min(n, wl.spec.batch)))
        dt, kv = oracle_time(wl, pools, seqs, threads)
        if dt >= target_s or len(seqs) == wl.spec.batch or dt * 2 > max_s:
            break
        n = min(wl.spec.batch, max(n + 1, int(n * target_s / max(dt, 1e-3))))
    passes = 1
    while len(seqs) == wl.spec.batch and dt < target_s and dt * (passes + 1) / passes <= max_s:
        d2, k2 = oracle_time(wl, pools, seqs, threads)
        dt, kv, passes = dt + d2, kv + k2, passes + 1
    return {"value": round(kv / dt / 1e9, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{passes} pass(es) over {len(seqs)} of {wl.spec.batch} sequences, all "
                      f"{wl.spec.num_q_heads} query heads ({kv / 1e6:.1f} MB of KV in all), fp64 "
                      f"three-pass oracle, {dt:.2f} s"}


# ---------------------------------------------------------------------------
# GPU arm: helpers
# ---------------------------------------------------------------------------

def source_hash(files):
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_hash(kernel):
    return source_hash(KERNEL_SOURCES[kernel])


NOMINAL_HBM_GBS = 8000.0                              # GB300 HBM3e, nominal


def stored_capture(workload_name, kernel="decode_kernel"):
    """The committed ncu capture of `kernel` on this workload, if it was
    taken on the kernel's current sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            captures = json.load(f)["captures"]
    except (OSError, ValueError, KeyError):
        return None
    want = kernel_hash(kernel)
    for t in captures:
        if t.get("workload") == workload_name and t.get("kernel") == kernel and \
                t.get("source_sha256_16") == want:
            return t
    return None


def stored_traffic(workload_name, kernel="decode_kernel"):
    """DRAM bytes (read + write) per launch of `kernel` on this workload from
    a committed ncu capture of the current sources, else None."""
    t = stored_capture(workload_name, kernel)
    return None if t is None else t.get("dram_bytes_per_launch")


def ncu_bandwidth(workload_name, peak, kernel="decode_kernel"):
    """The kernel's DRAM read rate as ncu measured it (bytes read / its
    duration in that capture), against the measured copy peak and the
    nominal 8 TB/s; None without a capture of the current sources."""
    t = stored_capture(workload_name, kernel)
    if t is None or not t.get("gpu_time_us") or not t.get("dram_bytes_read_per_launch"):
        return None
    gbs = t["dram_bytes_read_per_launch"] / t["gpu_time_us"] / 1e3
    return {"kernel": kernel, "dram_read_gbs": round(gbs, 1), "us": t["gpu_time_us"],
            "frac_of_measured": round(gbs / peak, 4), "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}


def measured_peak_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, ValueError, KeyError):
        return 1900.0, "fallback"


class StepPlan:
    """How one workload's step runs through the public API: the call, a
    description of its kernels, the token partition and the launches of
    this library's kernels per step."""

    def __init__(self, wl, g, pkv, no_shared_prefix=False):
        s = wl.spec
        self.multi = bool((wl.query_lens != 1).any())      # several query tokens per sequence
        self.m16 = self.row = False
        self.traffic_kernel = "decode_kernel"               # the kernel the roofline's traffic is of
        self.prefix = s.shared_prefix_tokens > 0 and not no_shared_prefix and not self.multi
        if self.multi:
            self.fn = g.multi_step
            self.part = pkv.multi_partition_tokens(s.batch, wl.num_tokens,
                                                   max(int(wl.query_lens.max()), 1),
                                                   s.num_q_heads, s.num_kv_heads, g.max_seq_len)
            G = s.num_q_heads // s.num_kv_heads
            tpg = 8 // G if G <= 8 else 0
            col_max = 4 * tpg
            maxq = max(int(wl.query_lens.max()), 1)
            # the launches pagedkv_multi_step makes: the append (slot mapping
            # fused in); the decode kernel's column groups whenever G <= 8,
            # except beside the 16-column kernel on a batch whose sequences
            # all have max_query_len tokens; the tensor-core kernel when a
            # sequence may need row tiles, else on bf16 pools the 16-column
            # kernel once a sequence may hold more than one group's tokens;
            # the merge when a sequence may span several partitions
            self.row = maxq > col_max
            self.m16 = tpg > 0 and s.kv_dtype == "bf16" and maxq > tpg and not self.row
            if self.m16:
                self.traffic_kernel = "multi_m16_kernel"
            uniform = wl.num_tokens == s.batch * maxq
            self.launches = (1 + int(tpg > 0 and not (self.m16 and uniform)) + int(self.m16)
                             + int(self.row) + int(g.max_seq_len > self.part))
            self.kernels = ("append_tokens_kernel + decode_kernel column groups / multi_m16_kernel "
                            "(16-column tiles, bf16) / multi_tc_kernel (+ multi_merge_kernel), "
                            "one pagedkv_multi_step")
        else:
            skip = s.shared_prefix_tokens if self.prefix else 0
            self.fn = g.prefix_step if self.prefix else g.fused_step
            self.part = pkv.partition_tokens(s.batch, s.num_kv_heads, g.max_seq_len - skip,
                                             s.block_size)
            if self.prefix:
                self.launches = 3
                self.kernels = ("multi_tc_kernel (shared-prefix mode) + decode_kernel (append "
                                "fused) + merge_kernel, one pagedkv_decode_step_prefix")
            else:
                self.launches = 1 + int(g.max_seq_len > self.part)
                self.kernels = "decode_kernel (append fused) + merge_kernel, one pagedkv_decode_step"


def capture(step_fn, dev, warm=5):
    """GRAPH_STEPS consecutive steps captured once in a CUDA graph (the GPU
    work of the steps without Python's per-call overhead or a gap between
    launches), after `warm` eager steps, then replayed three times."""
    import torch
    for _ in range(warm):
        step_fn()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(GRAPH_STEPS):
            step_fn()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(dev)
    return graph


def time_replays(graph, stream, dev, replays):
    """Per-step ms of each of `replays` graph replays (CUDA events on the
    launching stream) and the ms from the first event to the last."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(replays)]
    torch.cuda.synchronize(dev)
    for a, b in ev:
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) / GRAPH_STEPS for a, b in ev], ev[0][0].elapsed_time(ev[-1][1])


def steady_region(graph, stream, dev, seconds=STEADY_S):
    """Replays for at least `seconds` with clocks sampled throughout: the
    spread of the per-replay step time and the clocks under load."""
    import torch
    probe, _ = time_replays(graph, stream, dev, 3)
    n = max(10, int(math.ceil(seconds * 1e3 / (statistics.fmean(probe) * GRAPH_STEPS))))
    sampler = ClockSampler(str(torch.cuda.get_device_properties(dev).uuid))
    with sampler:
        ms, total = time_replays(graph, stream, dev, n)
    us = sorted(x * 1e3 for x in ms)
    q = lambda f: us[min(len(us) - 1, int(f * len(us)))]  # noqa: E731
    return {"seconds": round(total / 1e3, 3), "replays": n, "steps": n * GRAPH_STEPS,
            "us_per_step": round(statistics.fmean(us), 2), "us_per_step_p10": round(q(0.1), 2),
            "us_per_step_p50": round(q(0.5), 2), "us_per_step_p90": round(q(0.9), 2),
            "spread_p90_p10": round((q(0.9) - q(0.1)) / q(0.5), 4), "clocks": sampler.summary()}


def roofline_of(wl, plan, us, peak, peak_kind):
    """Roofline object of one step: algorithmic bytes (SURVEY's per-token
    figure x the tokens one step attends, plus q/out, tables and the append)
    over the measured step time, against the measured copy peak."""
    nbytes = algorithmic_bytes(wl)
    achieved = nbytes["step"] / us / 1e3
    traffic = stored_traffic(wl.spec.name, plan.traffic_kernel)
    return {"bound": "hbm", "kernel": plan.kernels, "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
            "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "algorithmic_bytes_per_launch": nbytes["step"], "us_per_launch": round(us, 2),
            "traffic": traffic,
            "traffic_over_algorithmic": round(traffic / nbytes["step"], 4) if traffic else None,
            "traffic_kernel": plan.traffic_kernel,
            "ncu": ncu_bandwidth(wl.spec.name, peak, plan.traffic_kernel)}


def check_status(pkv):
    st, flags = pkv.get_status()
    assert st == 0 and flags == 0, f"device status 0x{flags:x}"


def eager_us(step_fn, stream, dev, n=50):
    """Per-step device time of `n` steps called from Python one by one."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(n):
        step_fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / n * 1e3


def measure_config(config, pkv, dev, stream, peak, peak_kind, replays=40, kv_dtype=None):
    """One decode workload's step (the fused decode step; the shared-prefix
    step where the workload has a shared prefix), timed like the headline:
    GRAPH_STEPS steps captured in one CUDA graph, replayed.  kv_dtype: the
    same workload on a pool of another type."""
    import torch
    from paged_kv_cache_97_gb300.batch import DecodeBatch
    wl = workloads.make(config, kv_dtype=kv_dtype)
    g = DecodeBatch(wl, dev=dev)
    plan = StepPlan(wl, g, pkv)
    graph = capture(plan.fn, dev)
    ms, _ = time_replays(graph, stream, dev, replays)
    check_status(pkv)
    us = statistics.fmean(ms) * 1e3
    nbytes = algorithmic_bytes(wl)
    row = {"workload": wl.spec.name, "kv_dtype": wl.spec.kv_dtype,
           "us_per_step": round(us, 2),
           "kv_read_gbs": round(nbytes["kv_logical"] / us / 1e3, 1),
           "unique_kv_gbs": round(nbytes["kv_unique"] / us / 1e3, 1),
           "partition_tokens": plan.part, "launches_per_step": plan.launches,
           "eager_us_per_step": round(eager_us(plan.fn, stream, dev), 2),
           "roofline": roofline_of(wl, plan, us, peak, peak_kind)}
    if nbytes["kv_logical"] <= L2_BYTES:
        row["note"] = ("launch-bound: the step reads %.2f MB of KV, which stays in L2; one "
                       "launch of a few microseconds, so no bandwidth fraction is reachable"
                       % (nbytes["kv_logical"] / 1e6))
    if plan.prefix:
        row["note"] = ("shared prefix counted once in the algorithmic bytes (read from HBM "
                       "once, then L2); kv_read_gbs counts it per sequence")
    del graph, g
    torch.cuda.empty_cache()
    return row


# ---------------------------------------------------------------------------
# The rows beyond the decode step: copy-on-write
# ---------------------------------------------------------------------------

def measure_cow(pkv, dev, stream, peak):
    """Copy-on-write (block copy + beam-search decode steps), timed with CUDA
    events on the launching stream."""
    import torch
    from paged_kv_cache_97_gb300.batch import to_dev_bf16

    # (1) pagedkv_copy_blocks: 2048 block pairs of the 8B-like geometry
    # (16 x 8 x 128 bf16 = 32 KB per block and pool); two disjoint pair sets
    # alternate so each launch reads and writes 256 MB that are not in L2.
    nb, bs, hkv, d, npairs = 8192, 16, 8, 128, 2048
    kc = torch.zeros((nb, bs, hkv, d), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(7)).to(torch.int32)
    sets = [torch.stack([perm[i * 2 * npairs: i * 2 * npairs + npairs],
                         perm[i * 2 * npairs + npairs: (i + 1) * 2 * npairs]], 1).contiguous().to(dev)
            for i in range(2)]
    for i in range(6):
        pkv.copy_blocks(kc, vc, sets[i % 2])
    reps = 40
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
    torch.cuda.synchronize(dev)
    for i in range(reps):
        ev[2 * i].record(stream)
        pkv.copy_blocks(kc, vc, sets[i % 2])
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize(dev)
    us = statistics.fmean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(reps)) * 1e3
    copy_bytes = npairs * 2 * bs * hkv * d * 2 * 2          # K and V, read + write
    del kc, vc
    copy_row = {"kernel": "copy_blocks_kernel", "pairs": npairs, "bytes_per_launch": copy_bytes,
                "us_per_launch": round(us, 2), "achieved_gbs": round(copy_bytes / us / 1e3, 1),
                "frac": round(copy_bytes / us / 1e3 / peak, 4)}

    # (2) beam search: 16 prompts x 4 beams; per step the pool's copy-on-write
    # bookkeeping (host), the block copies and the fused decode step
    w = workloads.beam_search_8b()
    pool = pkv.KVPool(w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.zeros((w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16,
                     device=dev)
    vc = torch.zeros_like(kc)
    tables = np.full((w.num_seqs, w.max_blocks_per_seq), -1, np.int32)
    for p, L in enumerate(w.parent_lens):
        L = int(L)
        ids = pool.alloc((L + w.block_size - 1) // w.block_size)
        tables[p * w.beams, :len(ids)] = ids
        slots = torch.empty(L, dtype=torch.int64, device=dev)
        pkv.token_slot_mapping(torch.from_numpy(tables[p * w.beams:p * w.beams + 1].copy()).to(dev),
                               torch.arange(L, dtype=torch.int32, device=dev), w.num_blocks,
                               w.block_size, slots, seq_idx=torch.zeros(L, dtype=torch.int32, device=dev))
        pkv.reshape_and_cache(to_dev_bf16(w.parent_k[p], dev), to_dev_bf16(w.parent_v[p], dev), kc, vc,
                              slots)
        for j in range(1, w.beams):
            pool.fork(ids)
            tables[p * w.beams + j] = tables[p * w.beams]
    q = to_dev_bf16(w.step_q, dev)
    nk, nv = to_dev_bf16(w.step_k, dev), to_dev_bf16(w.step_v, dev)
    n = w.num_seqs
    out = torch.empty((n, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
    max_len = int(w.seq_lens_at(w.steps - 1).max())
    ws = torch.empty(max(pkv.workspace_bytes(n, w.num_q_heads, w.head_dim, max_len, w.block_size), 16),
                     dtype=torch.uint8, device=dev)
    bt_dev = torch.empty(tables.shape, dtype=torch.int32, device=dev)
    sl_dev = torch.empty(n, dtype=torch.int32, device=dev)
    pairs_dev = torch.empty((n, 2), dtype=torch.int32, device=dev)
    h_bt = torch.empty(tables.shape, dtype=torch.int32).pin_memory()
    h_sl = torch.empty(n, dtype=torch.int32).pin_memory()
    h_pairs = torch.empty((n, 2), dtype=torch.int32).pin_memory()
    copies, kv_read = 0, 0
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for step in range(w.steps):
        lens = w.seq_lens_at(step)
        pairs = pool.prepare_append(tables, lens)
        copies += len(pairs)
        kv_read += int(lens.sum()) * 2 * w.num_kv_heads * w.head_dim * 2
        torch.cuda.current_stream(dev).synchronize()      # pinned staging is reused next step
        h_bt.numpy()[:] = tables
        h_sl.numpy()[:] = lens
        bt_dev.copy_(h_bt, non_blocking=True)
        sl_dev.copy_(h_sl, non_blocking=True)
        if len(pairs):
            h_pairs.numpy()[:len(pairs)] = pairs
            pairs_dev[:len(pairs)].copy_(h_pairs[:len(pairs)], non_blocking=True)
            pkv.copy_blocks(kc, vc, pairs_dev[:len(pairs)])
        pkv.decode_step(out, q[step], nk[step], nv[step], kc, vc, bt_dev, sl_dev, int(lens.max()),
                        w.scale, ws)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall_us = (time.perf_counter() - t0) / w.steps * 1e6
    gpu_us = e0.elapsed_time(e1) / w.steps * 1e3
    check_status(pkv)
    used, _ = pool.stats()
    unshared = sum((int(L) + w.block_size - 1) // w.block_size for L in w.seq_lens_at(w.steps - 1))
    beam_row = {"workload": f"beam search, 16 prompts U{{512..4096}} x 4 beams, 32/8 heads, d 128, "
                            f"bs 16, {w.steps} steps",
                "us_per_step": round(gpu_us, 2), "wall_us_per_step": round(wall_us, 2),
                "kv_read_gbs": round(kv_read / w.steps / gpu_us / 1e3, 1),
                "block_copies": copies,
                "blocks_used": used, "blocks_unshared": unshared,
                "memory_saved": round(1 - used / unshared, 4),
                "note": "per step: host copy-on-write bookkeeping, table/length upload, block "
                        "copies, fused decode step; synchronised once per step for the host tables"}
    del kc, vc
    torch.cuda.empty_cache()
    return {"copy_blocks": copy_row, "beam_search": beam_row}


def multi_flops(wl) -> int:
    """Multiply-adds x 2 of S = Q.K^T and O = P.V over the attended (causal)
    tokens: 4 * d per (query row, attended token), Hq rows per query token."""
    s = wl.spec
    total = 0
    for b in range(s.batch):
        L, n = int(wl.seq_lens[b]), int(wl.query_lens[b])
        # query i attends L - n + i + 1 tokens
        total += n * (L - n + 1) + n * (n - 1) // 2
    return 4 * s.head_dim * s.num_q_heads * total


def multi_step_bytes(wl) -> int:
    s = wl.spec
    T = wl.num_tokens
    return (wl.kv_bytes_logical() + 2 * T * s.num_q_heads * s.head_dim * 2
            + T * s.num_kv_heads * s.head_dim * 2 * 2 * 2
            + int(((wl.seq_lens + s.block_size - 1) // s.block_size).sum()) * 4)


def measure_multi(config, pkv, dev, stream, peak, replays=40, kv_dtype=None):
    """A multi-token workload's step (append of every query token through
    the general slot mapping + paged_attention_multi), timed like the
    headline: GRAPH_STEPS steps captured in one CUDA graph, replayed."""
    import torch
    from paged_kv_cache_97_gb300.batch import DecodeBatch
    wl = workloads.make(config, kv_dtype=kv_dtype)
    g = DecodeBatch(wl, dev=dev)
    plan = StepPlan(wl, g, pkv)
    graph = capture(plan.fn, dev)
    ms, _ = time_replays(graph, stream, dev, replays)
    check_status(pkv)
    us = statistics.fmean(ms) * 1e3
    s = wl.spec
    step_bytes = multi_step_bytes(wl)
    fl = multi_flops(wl)
    tpeak, _ = measured_peak_tflops()
    col_kernel = plan.traffic_kernel
    del graph, g
    torch.cuda.empty_cache()
    return {"workload": s.name, "kv_dtype": s.kv_dtype, "query_tokens": wl.num_tokens,
            "us_per_step": round(us, 2),
            "kv_read_gbs": round(wl.kv_bytes_logical() / us / 1e3, 1),
            "partition_tokens": plan.part, "launches_per_step": plan.launches,
            "roofline": {"bound": "hbm", "kernel": plan.kernels,
                         "achieved": round(step_bytes / us / 1e3, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(step_bytes / us / 1e3 / peak, 4),
                         "algorithmic_bytes_per_launch": step_bytes,
                         "traffic": stored_traffic(s.name, col_kernel),
                         "traffic_kernel": col_kernel},
            "tensor": {"achieved_tflops": round(fl / us / 1e6, 2), "peak_tflops": tpeak,
                       "frac": round(fl / us / 1e6 / tpeak, 4), "flops_per_step": fl,
                       "multi_tc_kernel_dram_bytes": stored_traffic(s.name, "multi_tc_kernel"),
                       "note": "long queries on tcgen05 (TMEM accumulators), few on mma.sync "
                               "m16n8k16; peak = measured cuBLAS bf16 (burst)"}}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def gpu_arm(args, rank, world, local_rank, dist):
    import torch

    import paged_kv_cache_97_gb300 as pkv
    from paged_kv_cache_97_gb300.batch import DecodeBatch
    pkv.load()

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = workloads.make(args.config)
    g = DecodeBatch(wl, dev=dev)
    s = wl.spec
    plan = StepPlan(wl, g, pkv, no_shared_prefix=args.no_shared_prefix)
    multi, step_fn = plan.multi, plan.fn
    stream = torch.cuda.current_stream(dev)
    nbytes = algorithmic_bytes(wl)
    peak, peak_kind = measured_peak_gbs()

    for _ in range(args.warmup):
        step_fn()
        if not multi:
            g.step()
    graph = capture(step_fn, dev, warm=args.warmup)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    st, flags = pkv.get_status()
    assert st == 0, f"device status 0x{flags:x}"

    # ---- device-resident timed region ---------------------------------
    K = args.steps
    R = max(1, K // GRAPH_STEPS)                        # graph replays in the timed region
    K = R * GRAPH_STEPS
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(R)]
    sampler = ClockSampler(str(torch.cuda.get_device_properties(dev).uuid))
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with sampler:
        for i in range(R):
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    total_ms = ev[0][0].elapsed_time(ev[-1][1])
    step_ms = [ev[i][0].elapsed_time(ev[i][1]) / GRAPH_STEPS for i in range(R)]
    ms_step = total_ms / K
    elapsed, agg_bytes_per_s = aggregate(total_ms / 1e3, nbytes["kv_logical"] * K, world, dist)
    value = agg_bytes_per_s / 1e9
    # a longer steady region of the same replays: run-to-run spread and clocks
    steady = steady_region(graph, stream, dev)
    check_status(pkv)

    # the same step through eager calls: the fused step, and the three calls
    # (slot mapping, append, attention)
    K3 = max(K // 4, 10)
    eager_ms = eager_us(step_fn, stream, dev, K3) / 1e3
    ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K3)]
    torch.cuda.synchronize(dev)
    for i in range(K3):
        ev3[i][0].record(stream)
        g.append_tokens() if multi else g.append()
        ev3[i][1].record(stream)
        g.attend_multi() if multi else g.attend()
        ev3[i][2].record(stream)
    torch.cuda.synchronize(dev)
    unfused_ms = ev3[0][0].elapsed_time(ev3[-1][2]) / K3
    attn_only_ms = statistics.fmean(ev3[i][1].elapsed_time(ev3[i][2]) for i in range(K3))
    append_only_ms = statistics.fmean(ev3[i][0].elapsed_time(ev3[i][1]) for i in range(K3))
    st, flags = pkv.get_status()
    assert st == 0, f"device status 0x{flags:x}"

    # ---- end to end through the public API, host buffers -----------------
    # Every step copies its inputs from pinned host memory and reads its
    # output back.  Two sets of device inputs/outputs alternate: step i's
    # inputs are copied on a copy stream while step i-1 computes, and step
    # i's output is read back on a third stream while step i+1 computes.
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    h_in = {"q": pin(wl.q.view(np.int16)).view(torch.bfloat16),
            "new_k": pin(wl.new_k.view(np.int16)).view(torch.bfloat16),
            "new_v": pin(wl.new_v.view(np.int16)).view(torch.bfloat16),
            "block_tables": pin(wl.block_tables), "seq_lens": pin(wl.seq_lens)}
    if multi:
        h_in["query_start"] = pin(wl.query_start)
    out_name = "out_multi" if multi else "out"
    sets = [{k: getattr(g, k) for k in list(h_in) + [out_name]}]
    sets.append({k: torch.empty_like(v) for k, v in sets[0].items()})
    h_out = [torch.empty(sets[0][out_name].shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = h_out[0].numel() * h_out[0].element_size()
    # One side stream carries both directions: while step i computes, it
    # reads back step i-1's output and then copies step i+1's inputs into the
    # same buffer set (so the compute stream waits on one event per step).
    io_s = torch.cuda.Stream(dev)
    K2 = max(args.steps // 4, 10)
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def copy_in(j):
        for k, h in h_in.items():
            sets[j % 2][k].copy_(h, non_blocking=True)
        copied[j % 2].record(io_s)

    def read_back(j):
        io_s.wait_event(done[j % 2])
        h_out[j % 2].copy_(sets[j % 2][out_name], non_blocking=True)

    torch.cuda.synchronize(dev)
    e0.record(stream)
    io_s.wait_event(e0)
    with torch.cuda.stream(io_s):
        copy_in(0)
    for i in range(K2):
        cur = sets[i % 2]
        stream.wait_event(copied[i % 2])              # its inputs landed (after step i-2's read-back)
        for k, v in cur.items():
            setattr(g, k, v)
        step_fn()
        done[i % 2].record(stream)
        with torch.cuda.stream(io_s):
            if i >= 1:
                read_back(i - 1)
            if i + 1 < K2:
                copy_in(i + 1)
    with torch.cuda.stream(io_s):
        read_back(K2 - 1)
    stream.wait_stream(io_s)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    for k, v in sets[0].items():
        setattr(g, k, v)
    e2e_ms = e0.elapsed_time(e1) / K2
    _, e2e_agg = aggregate(e2e_ms / 1e3, nbytes["kv_logical"], world, dist)
    assert np.isfinite(h_out[(K2 - 1) % 2].float().numpy()).all()

    step_mean_ms = statistics.fmean(step_ms)
    roofline = roofline_of(wl, plan, step_mean_ms * 1e3, peak, peak_kind)
    if plan.multi:
        roofline["algorithmic_bytes_per_launch"] = multi_step_bytes(wl)
        roofline["achieved"] = round(multi_step_bytes(wl) / (step_mean_ms * 1e3) / 1e3, 1)
        roofline["frac"] = round(roofline["achieved"] / peak, 4)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2),
        "pct_of_hbm_peak": round(100 * value / world / peak, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if s.kv_dtype == "bf16" else f"{s.kv_dtype} KV, bf16 q/out, fp32 accumulate",
        "data": "synthetic",
        "config": dict(workload_config(wl, nbytes), parallelism=f"replicas x{world}"),
        "partition_tokens": plan.part,
        "roofline": roofline,
        "timing": f"value and ms_per_step: {GRAPH_STEPS} steps captured in one CUDA graph, replayed",
        "steady": steady,
        "eager_us_per_step": round(eager_ms * 1e3, 2),
        "unfused": {"us_per_step": round(unfused_ms * 1e3, 2),
                    "append_us": round(append_only_ms * 1e3, 2),
                    "attention_us": round(attn_only_ms * 1e3, 2),
                    "note": ("token slot mapping + reshape_and_cache, then paged_attention_multi" if multi
                             else "slot mapping + reshape_and_cache (append_us), then "
                                  "paged_attention_decode (attention_us: decode + merge), as three calls")},
        "e2e": {"value": round(e2e_agg / 1e9, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                "note": "inputs of every step copied from pinned host memory and outputs read "
                        "back inside the timed region; two buffer sets alternate, and one side "
                        "stream reads back step i-1's output and copies step i+1's inputs while "
                        "step i computes"},
        "gpu_launches": plan.launches * K,
        "clocks": sampler.summary(),
    }
    del graph, g, sets
    torch.cuda.empty_cache()
    if not args.no_rows:
        configs = {}
        for c in ROW_CONFIGS:
            if c == args.config:
                configs[str(c)] = {"workload": s.name, "kv_dtype": s.kv_dtype,
                                   "us_per_step": line["us_per_step"],
                                   "kv_read_gbs": round(nbytes["kv_logical"] / (ms_step * 1e3) / 1e3, 1),
                                   "partition_tokens": plan.part, "launches_per_step": plan.launches,
                                   "eager_us_per_step": line["eager_us_per_step"],
                                   "roofline": roofline, "note": "the headline workload (above)"}
            else:
                configs[str(c)] = measure_config(c, pkv, dev, stream, peak, peak_kind)
        line["rows"] = {"configs": configs,
                        "fp8_kv": measure_config(6, pkv, dev, stream, peak, peak_kind),
                        "multi_token": {"speculative_verification": measure_multi(7, pkv, dev, stream, peak),
                                        "decode_maximal_batch": measure_multi(8, pkv, dev, stream, peak)},
                        # the tensor-core paths (shared prefix, long queries) on 8-bit pools
                        "kv8_tensor_core": {
                            "shared_prefix_int8": measure_config(4, pkv, dev, stream, peak, peak_kind,
                                                                 kv_dtype="int8"),
                            "shared_prefix_fp8": measure_config(4, pkv, dev, stream, peak, peak_kind,
                                                                kv_dtype="fp8"),
                            "decode_maximal_batch_int8": measure_multi(8, pkv, dev, stream, peak,
                                                                       kv_dtype="int8")},
                        "cow": measure_cow(pkv, dev, stream, peak)}
    return line, wl


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=sorted(workloads.CONFIGS),
                    help="workload (default 3: long-context split-K decode, the largest single-GPU one)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="for workloads with a shared prefix, time the plain step instead of "
                         "pagedkv_decode_step_prefix")
    ap.add_argument("--no-rows", action="store_true",
                    help="skip the other workloads and the copy-on-write rows reported under 'rows'")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = rank_info()

    if args.impl == "reference":
        if rank != 0:
            return 0
        wl = workloads.make(args.config)
        threads = os.cpu_count() or 1
        pools = oracle_pools(wl)
        per_step = []
        for i in range(args.warmup + args.steps):
            # each step is a bounded sample: one sequence (cycling), all its query heads
            dt, kv = oracle_time(wl, pools, [i % wl.spec.batch], threads)
            if i >= args.warmup:
                per_step.append((dt, kv))
        t = sum(d for d, _ in per_step)
        kv = sum(k for _, k in per_step)
        v = kv / t / 1e9
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict(workload_config(wl, algorithmic_bytes(wl)), parallelism=f"replicas x{world}"),
            "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "per step: one sequence of the batch (cycling), all query heads, "
                                       "fp64 three-pass oracle on the host cores (rank 0 only)"},
            "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return 0

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    line, wl = gpu_arm(args, rank, world, local_rank, dist)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pools = oracle_pools(wl)
        line["cpu_baseline"] = oracle_sample(wl, os.cpu_count() or 1, pools=pools)
        if args.config in (1, 2):
            # the same oracle on one core (a few seconds of work)
            one = oracle_sample(wl, 1, target_s=3.0, max_s=8.0, pools=pools)
            line["cpu_baseline"]["single_thread"] = {"value": one["value"], "unit": one["unit"],
                                                     "cores": 1, "sample": one["sample"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
