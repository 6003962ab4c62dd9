#!/usr/bin/env python3
"""Decode-step benchmark of paged attention on GB300.

One step = the whole hot path over one synthetic decode batch through
pagedkv_decode_step: the slot of each sequence's new token, its append into
the pool, and the paged attention (the per-partition decode kernel, with the
append fused in, plus the log-sum-exp merge of sequences that span several
partitions).  The same step as three calls (slot mapping, reshape_and_cache,
paged_attention_decode) is timed beside it.  The default workload is the
Llama-3.1-8B-like decode layer (B 64, 32/8 heads, d 128, 16-token blocks,
lengths U{512..4096}).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the same workload instead (the reference arm: a plain fp64 program, not a
target).  Timing: CUDA events on the launching stream, W warm-up steps, K
timed steps, barrier + synchronize on both sides, max over ranks.  The KV
read per step (~600 MB) is larger than the 129 MB L2, so no flush is needed.
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
DEFAULT_CONFIG = 2
FALLBACK_HBM_GBS = 6800.0
GRAPH_STEPS = 20
L2_BYTES = 129e6                                         # GB300 L2
DECODE_SOURCE = os.path.join(ROOT, "paged_kv_cache_97_gb300", "csrc", "pagedkv_decode.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")


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
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from oracle_helpers import oracle_pool
    oracle.build()
    return oracle_pool(wl)


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
# GPU arm
# ---------------------------------------------------------------------------

def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def stored_traffic(workload_name):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current decode kernel source and this workload; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_sha256_16") != source_hash(DECODE_SOURCE) or t.get("workload") != workload_name:
        return None
    return t.get("dram_bytes_per_launch")


def measured_peak_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# The rows beyond the decode step: copy-on-write
# ---------------------------------------------------------------------------

def measure_cow(pkv, dev, stream, peak):
    """Copy-on-write (block copy + beam-search decode steps), timed with CUDA
    events on the launching stream."""
    import torch
    from gpu_helpers import to_dev_bf16

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
    st, flags = pkv.get_status()
    assert st == 0 and flags == 0, f"device status 0x{flags:x}"
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
    return {"copy_blocks": copy_row, "beam_search": beam_row}


def measure_config_step(config, pkv, dev, stream, peak, replays=40):
    """One workload's fused decode step (pagedkv_decode_step), timed like the
    headline: GRAPH_STEPS steps captured in one CUDA graph, replayed."""
    import torch
    from gpu_helpers import GpuStep
    wl = workloads.make(config)
    g = GpuStep(wl, dev=dev)
    for _ in range(5):
        g.fused_step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(GRAPH_STEPS):
            g.fused_step()
    for _ in range(3):
        graph.replay()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * replays)]
    torch.cuda.synchronize(dev)
    for i in range(replays):
        ev[2 * i].record(stream)
        graph.replay()
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize(dev)
    st, flags = pkv.get_status()
    assert st == 0 and flags == 0, f"device status 0x{flags:x}"
    us = statistics.fmean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(replays)) * 1e3 / GRAPH_STEPS
    nbytes = algorithmic_bytes(wl)
    achieved = nbytes["step"] / us / 1e3
    return {"workload": wl.spec.name, "us_per_step": round(us, 2),
            "kv_read_gbs": round(nbytes["kv_logical"] / us / 1e3, 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "algorithmic_bytes_per_step": nbytes["step"]}}


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


def measure_multi(config, pkv, dev, stream, peak, replays=40):
    """A multi-token workload's step (append of every query token through
    the general slot mapping + paged_attention_multi), timed like the
    headline: GRAPH_STEPS steps captured in one CUDA graph, replayed."""
    import torch
    from gpu_helpers import GpuStep
    wl = workloads.make(config)
    g = GpuStep(wl, dev=dev)
    for _ in range(5):
        g.multi_step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(GRAPH_STEPS):
            g.multi_step()
    for _ in range(3):
        graph.replay()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * replays)]
    torch.cuda.synchronize(dev)
    for i in range(replays):
        ev[2 * i].record(stream)
        graph.replay()
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize(dev)
    st, flags = pkv.get_status()
    assert st == 0 and flags == 0, f"device status 0x{flags:x}"
    us = statistics.fmean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(replays)) * 1e3 / GRAPH_STEPS
    s = wl.spec
    T = wl.num_tokens
    kv = wl.kv_bytes_logical()
    step_bytes = (kv + 2 * T * s.num_q_heads * s.head_dim * 2 + T * s.num_kv_heads * s.head_dim * 2 * 2 * 2
                  + int(((wl.seq_lens + s.block_size - 1) // s.block_size).sum()) * 4)
    fl = multi_flops(wl)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpeak = float(json.load(f)["bf16_tflops"])
    except (OSError, ValueError, KeyError):
        tpeak = 1900.0
    return {"workload": s.name, "query_tokens": T, "us_per_step": round(us, 2),
            "kv_read_gbs": round(kv / us / 1e3, 1),
            "roofline": {"bound": "hbm", "achieved": round(step_bytes / us / 1e3, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(step_bytes / us / 1e3 / peak, 4),
                         "algorithmic_bytes_per_step": step_bytes},
            "tensor": {"achieved_tflops": round(fl / us / 1e6, 2), "peak_tflops": tpeak,
                       "frac": round(fl / us / 1e6 / tpeak, 4), "flops_per_step": fl,
                       "note": "long queries on tcgen05 (TMEM accumulators), few on mma.sync "
                               "m16n8k16; peak = measured cuBLAS bf16 (burst)"}}


def gpu_arm(args, rank, world, local_rank, dist):
    import torch

    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import paged_kv_cache_97_gb300 as pkv
    from gpu_helpers import GpuStep
    pkv.load()

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = workloads.make(args.config)
    g = GpuStep(wl, dev=dev)
    s = wl.spec
    multi = bool((wl.query_lens != 1).any())             # several query tokens per sequence
    use_prefix = s.shared_prefix_tokens > 0 and not args.no_shared_prefix and not multi
    step_fn = g.multi_step if multi else (g.prefix_step if use_prefix else g.fused_step)
    stream = torch.cuda.current_stream(dev)
    nbytes = algorithmic_bytes(wl)
    # token partition of the decode kernel, or of the multi-token call
    if multi:
        part = pkv.multi_partition_tokens(s.batch, wl.num_tokens, max(int(wl.query_lens.max()), 1),
                                          s.num_q_heads, s.num_kv_heads, g.max_seq_len)
    else:
        part = pkv.partition_tokens(s.batch, s.num_kv_heads,
                                    g.max_seq_len - s.shared_prefix_tokens * use_prefix, s.block_size)
    # decode (append fused) + merge, + the prefix kernel on the shared-prefix
    # path; multi-token: slot mapping + append + the column groups (sequences
    # with few queries) and/or the tensor-core kernel (long ones) + the merge
    # when a sequence spans several partitions
    if multi:
        G = s.num_q_heads // s.num_kv_heads
        col_max = (8 // G) * 4 if G <= 8 else 0
        launches_per_step = (2 + int(G <= 8)              # the column groups' launch
                             + int(bool((wl.query_lens > col_max).any()))
                             + int(g.max_seq_len > part))
    else:
        launches_per_step = 3 if use_prefix else 1 + (1 if g.max_seq_len > part else 0)

    for _ in range(args.warmup):
        step_fn()
        if not multi:
            g.step()
    torch.cuda.synchronize(dev)
    # GRAPH_STEPS consecutive steps captured once in a CUDA graph (each a
    # decode + merge pair), the graph replayed: the GPU work of the steps
    # without Python's per-call overhead or a gap between graph launches.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(GRAPH_STEPS):
            step_fn()
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
    sampler = ClockSampler(torch.cuda.get_device_properties(dev).uuid.__str__())
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

    # the same step through eager calls: the fused step, and the three calls
    # (slot mapping, append, attention)
    K3 = max(K // 4, 10)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(K3):
        step_fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    eager_ms = e0.elapsed_time(e1) / K3
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
    elapsed, agg_bytes_per_s = aggregate(total_ms / 1e3, nbytes["kv_logical"] * K, world, dist)
    value = agg_bytes_per_s / 1e9
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
    copy_s, back_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    K2 = max(args.steps // 4, 10)
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    copy_s.wait_event(e0)
    back_s.wait_event(e0)
    for i in range(K2):
        cur = sets[i % 2]
        with torch.cuda.stream(copy_s):
            if i >= 2:
                copy_s.wait_event(done[i % 2])        # step i-2 is done with this set
            for k, h in h_in.items():
                cur[k].copy_(h, non_blocking=True)
            copied[i % 2].record(copy_s)
        stream.wait_event(copied[i % 2])
        if i >= 2:
            stream.wait_event(read[i % 2])            # step i-2's output has been read
        for k, v in cur.items():
            setattr(g, k, v)
        step_fn()
        done[i % 2].record(stream)
        with torch.cuda.stream(back_s):
            back_s.wait_event(done[i % 2])
            h_out[i % 2].copy_(cur[out_name], non_blocking=True)
            read[i % 2].record(back_s)
    stream.wait_stream(back_s)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    for k, v in sets[0].items():
        setattr(g, k, v)
    e2e_ms = e0.elapsed_time(e1) / K2
    _, e2e_agg = aggregate(e2e_ms / 1e3, nbytes["kv_logical"], world, dist)
    assert np.isfinite(h_out[(K2 - 1) % 2].float().numpy()).all()

    peak, peak_kind = measured_peak_gbs()
    step_mean_ms = statistics.fmean(step_ms)
    achieved = nbytes["step"] / (step_mean_ms / 1e3) / 1e9
    traffic = stored_traffic(s.name)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2),
        "pct_of_hbm_peak": round(100 * value / world / peak, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if s.kv_dtype == "bf16" else f"{s.kv_dtype} KV, bf16 q/out, fp32 accumulate",
        "data": "synthetic",
        "config": dict(workload_config(wl, nbytes), partition_tokens=part,
                       parallelism=f"replicas x{world}"),
        "roofline": {"bound": "hbm",
                     "kernel": ("token slot mapping + append + decode_kernel column groups / "
                                "multi_tc_kernel (+ multi_merge_kernel), "
                                "paged_attention_multi" if multi else
                                "multi_tc_kernel (shared-prefix mode) + decode_kernel (append fused) + merge_kernel, one "
                                "pagedkv_decode_step_prefix" if use_prefix else
                                "decode_kernel (append fused) + merge_kernel, one pagedkv_decode_step"),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": nbytes["step"],
                     "us_per_launch": round(step_mean_ms * 1e3, 2), "traffic": traffic},
        "timing": f"value and ms_per_step: {GRAPH_STEPS} steps captured in one CUDA graph, replayed",
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
                        "back inside the timed region; two buffer sets alternate so step i's "
                        "copies overlap step i-1's compute"},
        "gpu_launches": launches_per_step * K,
        "clocks": sampler.summary(),
    }
    if not args.no_rows:
        line["rows"] = {"cow": measure_cow(pkv, dev, stream, peak),
                        "fp8_kv": measure_config_step(6, pkv, dev, stream, peak),
                        "multi_token": {"speculative_verification": measure_multi(7, pkv, dev, stream, peak),
                                        "decode_maximal_batch": measure_multi(8, pkv, dev, stream, peak)}}
    return line, wl


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=sorted(workloads.CONFIGS),
                    help="workload (default 2: the Llama-3.1-8B-like decode layer)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="for workloads with a shared prefix, time the plain step instead of "
                         "pagedkv_decode_step_prefix")
    ap.add_argument("--no-rows", action="store_true",
                    help="skip the extra measurements (copy-on-write) reported under 'rows'")
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
            "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(workload_config(wl, algorithmic_bytes(wl)), parallelism="oracle on host cores"),
            "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "per step: one sequence of the batch (cycling), all query heads, "
                                       "fp64 three-pass oracle"},
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
