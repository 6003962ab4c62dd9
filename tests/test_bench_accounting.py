"""The bench's byte accounting, recounted from the block tables.

The roofline the bench reports is algorithmic bytes / measured time, so the
byte count is checked here against an independent count on the workloads'
own tables: every (physical block, row) that some sequence attends is read
once (a shared prefix block by every sequence, but from HBM once), every
table entry in use is read once per sequence, and the 8-bit scales once per
block in use.  Per row of a block: K and V for every KV head, d elements each
(the block layout [num_blocks, block_size, Hkv, d] of “LLM 推理引擎深度解析”,
§2.1; the per-token KV size of “让 Agent 跑得快：LLM 推理服务”, §一).
"""
import json

import numpy as np
import pytest

import bench
import workloads


def attended_rows(wl):
    """Set of (physical block, row) pairs the step's attention reads."""
    bs = wl.spec.block_size
    pairs = set()
    for b, L in enumerate(wl.seq_lens.astype(np.int64)):
        for t in range(int(L)):
            pairs.add((int(wl.block_tables[b, t // bs]), t % bs))
    return pairs


@pytest.mark.parametrize("config", [1, 2, 4, 5, 7, 8])
def test_kv_bytes_match_a_recount_of_the_tables(config):
    wl = workloads.make(config)
    s = wl.spec
    row_bytes = 2 * s.num_kv_heads * s.head_dim * wl.kv_elem_bytes
    pairs = attended_rows(wl)
    nb = bench.algorithmic_bytes(wl)
    assert nb["kv_unique"] == len(pairs) * row_bytes
    assert nb["kv_logical"] == int(wl.seq_lens.astype(np.int64).sum()) * row_bytes
    if s.shared_prefix_tokens:
        assert nb["kv_unique"] < nb["kv_logical"]
    else:
        assert nb["kv_unique"] == nb["kv_logical"]


@pytest.mark.parametrize("config", [2, 5])
def test_step_bytes_add_up(config):
    wl = workloads.make(config)
    s = wl.spec
    bs, hkv, d, hq = s.block_size, s.num_kv_heads, s.head_dim, s.num_q_heads
    elem = wl.kv_elem_bytes
    T = wl.num_tokens
    pairs = attended_rows(wl)
    blocks_in_use = {p for p, _ in pairs}
    table_entries = sum(-(-int(L) // bs) for L in wl.seq_lens)
    kv = len(pairs) * 2 * hkv * d * elem
    scales = len(blocks_in_use) * 2 * hkv * 4 if elem == 1 else 0
    q_and_out = 2 * T * hq * d * 2
    lengths_and_table = 4 * s.batch + 4 * table_entries
    new_kv_in = T * hkv * d * 2 * 2                      # bf16 k and v of the new tokens
    new_kv_out = T * hkv * d * elem * 2                  # their rows written into the pool
    slots = T * 8 * 2
    want = kv + scales + q_and_out + lengths_and_table + new_kv_in + new_kv_out + slots
    assert bench.algorithmic_bytes(wl)["step"] == want


def test_default_workload_is_larger_than_l2():
    # the timed region relies on inputs larger than L2 instead of a flush
    nb = bench.algorithmic_bytes(workloads.make(bench.DEFAULT_CONFIG))
    assert nb["kv_unique"] > bench.L2_BYTES


def test_stored_traffic_needs_the_current_kernel_source(tmp_path, monkeypatch):
    # a capture counts only for its workload, its kernel and the hash of the
    # kernel's current sources
    name = workloads.make(2).spec.name
    cur = bench.kernel_hash("decode_kernel")
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"captures": [
        {"workload": name, "kernel": "decode_kernel", "source_sha256_16": "0" * 16,
         "dram_bytes_per_launch": 1},
        {"workload": name, "kernel": "decode_kernel", "source_sha256_16": cur,
         "dram_bytes_per_launch": 2, "dram_bytes_read_per_launch": 8000, "gpu_time_us": 2.0}]}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.stored_traffic(name, "decode_kernel") == 2
    assert bench.stored_traffic(name, "multi_tc_kernel") is None
    assert bench.stored_traffic("another workload", "decode_kernel") is None
    # the ncu read rate: 8000 B in 2 us = 4 GB/s, against a 5 GB/s peak and 8 TB/s nominal
    bw = bench.ncu_bandwidth(name, 5.0)
    assert bw["dram_read_gbs"] == 4.0 and bw["frac_of_measured"] == 0.8
    assert bw["frac_of_nominal_8tbs"] == 0.0005
    assert bench.ncu_bandwidth("another workload", 5.0) is None
