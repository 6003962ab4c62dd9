"""Pins of the oracle's size formulas and block-pool rules against the pages'
printed examples (tests/golden/kv_sizes.json, tests/golden/pool_fifo.json)."""
import json
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _call(spec):
    return getattr(oracle, spec["fn"])(**spec["args"])


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _load("kv_sizes.json")["cases"], ids=lambda c: c["citation"][:60])
def test_printed_kv_sizes(case):
    got = _call(case)
    assert got == pytest.approx(case["printed"], rel=case["rtol"], abs=0), case["citation"]


@pytest.mark.parametrize("case", _load("kv_sizes.json")["ratios"], ids=lambda c: c["citation"][:60])
def test_printed_ratios(case):
    assert _call(case["numerator"]) / _call(case["denominator"]) == case["printed"]


def test_block_memory_is_block_size_tokens_of_one_layer():
    # Two formulas from two pages: one block of one layer holds block_size
    # tokens' worth of the per-token KV of a single layer.
    for bs in (1, 16, 32):
        for h in (1, 2, 8, 32):
            for d in (64, 128):
                for dt in (1, 2, 4):
                    assert oracle.block_memory_bytes(bs, h, d, dt) == bs * oracle.kv_bytes_per_token(1, h, d, dt)


def test_waste_bound_in_last_block_only():
    w = _load("kv_sizes.json")["waste"]
    bs = w["block_size"]
    seen = set()
    for L in range(1, 4 * bs * 10):
        n = oracle.blocks_needed(L, bs)
        waste = oracle.internal_waste_tokens(L, bs)
        assert (n - 1) * bs < L <= n * bs          # the last block holds >= 1 token
        assert 0 <= waste <= w["max_waste"]
        seen.add(waste)
    assert seen == set(range(bs))                   # every waste value occurs, 15 included


def measured_waste(wl):
    """Unused token rows of the blocks a workload's tables hold (each physical
    block counted once), and all rows of those blocks."""
    import numpy as np
    bs = wl.spec.block_size
    rows = {}
    for b, L in enumerate(wl.seq_lens.astype(np.int64)):
        for t in range(int(L)):
            rows.setdefault(int(wl.block_tables[b, t // bs]), set()).add(t % bs)
    used = sum(len(r) for r in rows.values())
    return len(rows) * bs - used, len(rows) * bs


def test_measured_waste_depends_on_the_lengths():
    # The pages claim under 4 % KV waste with paging (“让 Agent 跑得快”, §二;
    # “LLM 推理引擎深度解析”, §2.1): only each sequence's last block is partly
    # empty (“让 Agent 跑得快”, §五), so the fraction is at most
    # (block_size - 1) / block_size per sequence and shrinks with length.
    import workloads
    for config in (1, 2, 4, 5):
        wl = workloads.make(config)
        bs = wl.spec.block_size
        waste, rows = measured_waste(wl)
        if not wl.spec.shared_prefix_tokens:
            assert waste == sum(oracle.internal_waste_tokens(int(L), bs) for L in wl.seq_lens)
        assert waste <= wl.spec.batch * (bs - 1)
        frac = waste / rows
        if config == 1:
            assert frac > 0.04          # 4 short sequences (L <= 200): about 7.6 %
        else:
            assert frac < 0.04          # hundreds to thousands of tokens: 0.3-1.1 %


def test_pool_trace():
    g = _load("pool_fifo.json")
    pool = oracle.BlockPoolModel(g["num_blocks"])
    for st in g["steps"]:
        if st["op"] == "alloc_seq":
            if st["expect"] == "MemoryError":
                before = pool.stats()
                with pytest.raises(MemoryError):
                    pool.alloc_sequence(st["seq_len"], g["block_size"])
                assert pool.stats() == before      # all or nothing
            else:
                assert pool.alloc_sequence(st["seq_len"], g["block_size"]) == st["expect"]
        elif st["op"] == "free":
            if st.get("expect") == "ValueError":
                with pytest.raises(ValueError):
                    pool.free(st["ids"])
            else:
                pool.free(st["ids"])
        elif st["op"] == "stats":
            assert list(pool.stats()) == st["expect"]
