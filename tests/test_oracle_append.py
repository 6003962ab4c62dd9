"""Pins of the oracle's slot mapping and append.

* bf16 append is a bit copy into the token's slot and touches nothing else
  (“让 Agent 跑得快”, §五 共享前缀: only the current decode token writes);
* the int8 code is clamp(round_half_even(x / s), -127, 127) decided in IEEE
  fp32 (checked against numpy's fp32 divide and rint, including cases where
  an fp64 quotient would round differently);
* with s = max|x| / 127 the largest element of a block stores +-127 and every
  element round-trips within s / 2 (The engineering behind LLM inference,
  §3.2: INT8 KV halves memory at a small loss);
* the slots of a sequence's positions cover its table's blocks row by row.
"""
import numpy as np
import pytest

import oracle
import workloads
from oracle_helpers import oracle_pool
from workloads import bf16_bits_to_f32, to_bf16_bits


def test_bf16_append_is_a_bit_copy(oracle_mod):
    wl = workloads.custom(batch=3, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                          seq_lens=[5, 17, 40], seed=6)
    kc, vc = wl.poisoned_pool(), wl.poisoned_pool()
    slots, rc = oracle.token_slots(wl.block_tables, wl.seq_lens - 1, 16, wl.num_blocks)
    assert rc == 0
    before_k = kc.copy()
    assert oracle.append_bf16(wl.new_k, wl.new_v, kc, vc, slots) == 0
    flat_k = kc.reshape(-1, 2, 64)
    flat_v = vc.reshape(-1, 2, 64)
    np.testing.assert_array_equal(flat_k[slots], wl.new_k)
    np.testing.assert_array_equal(flat_v[slots], wl.new_v)
    mask = np.ones(flat_k.shape[0], bool)
    mask[slots] = False
    np.testing.assert_array_equal(flat_k[mask], before_k.reshape(-1, 2, 64)[mask])


def test_negative_slot_skips_and_bad_slot_reports(oracle_mod):
    k = to_bf16_bits(np.ones((2, 1, 64), np.float32))
    kc = np.zeros((4, 16, 1, 64), np.uint16)
    vc = np.zeros_like(kc)
    assert oracle.append_bf16(k, k, kc, vc, np.array([-1, 64])) == oracle.INDEX
    assert not kc.any()


def test_slots_walk_the_table_row_by_row(oracle_mod):
    wl = workloads.make(1)
    bs = wl.spec.block_size
    for b in range(wl.spec.batch):
        L = int(wl.seq_lens[b])
        slots, rc = oracle.token_slots(wl.block_tables, np.arange(L), bs, wl.num_blocks,
                                       seq_idx=np.full(L, b))
        assert rc == 0
        assert len(set(slots.tolist())) == L                      # distinct slots
        blocks = slots[::bs] // bs                                # block of each logical block's row 0
        np.testing.assert_array_equal(blocks, wl.block_tables[b, :len(blocks)])
        first = slots[(np.arange(L) // bs) * bs]
        np.testing.assert_array_equal(slots - first, np.arange(L) % bs)   # rows in order


def check_rounding(quant):
    cases = [(0.5, 1.0, 0), (1.5, 1.0, 2), (2.5, 1.0, 2), (-0.5, 1.0, 0), (-1.5, 1.0, -2),
             (-2.5, 1.0, -2), (126.5, 1.0, 126), (127.5, 1.0, 127), (200.0, 1.0, 127),
             (-300.0, 1.0, -127), (float("nan"), 1.0, 0), (3.4, 0.0, 3), (-3.6, 0.0, -4),
             (float("inf"), 1.0, 127), (1e-30, 1.0, 0)]
    for x, s, want in cases:
        assert quant(x, s) == want, (x, s)


def check_fp32_decision(quant):
    rng = np.random.default_rng(5)
    x = bf16_bits_to_f32(to_bf16_bits(rng.standard_normal(400000).astype(np.float32) * 3))
    s = (np.abs(rng.standard_normal(400000)).astype(np.float32) * 0.05 + 1e-3).astype(np.float32)
    q32 = np.rint(x / s)                               # IEEE fp32 divide, ties to even
    q64 = np.rint(x.astype(np.float64) / s.astype(np.float64))
    differ = np.nonzero((q32 != q64) & (np.abs(q32) <= 127))[0]
    assert differ.size > 0, "no fp32/fp64 disagreement found to test"
    for i in differ[:50]:
        assert quant(float(x[i]), float(s[i])) == int(q32[i])
    for i in range(0, 400000, 4001):
        want = int(np.clip(q32[i], -127, 127))
        assert quant(float(x[i]), float(s[i])) == want


def test_int8_rounding_rules(oracle_mod):
    check_rounding(oracle.quantize_int8)


def test_int8_decision_is_fp32(oracle_mod):
    check_fp32_decision(oracle.quantize_int8)


def test_int8_block_max_stores_127_and_round_trips(oracle_mod):
    wl = workloads.custom(batch=4, num_q_heads=16, num_kv_heads=2, head_dim=128, block_size=32,
                          seq_lens=[1, 31, 64, 200], kv_dtype="int8", seed=12)
    kc, vc, ks, vs = oracle_pool(wl)
    for b in range(4):
        L = int(wl.seq_lens[b])
        pos, k, v = wl.own_tokens(b)
        xs = np.concatenate([bf16_bits_to_f32(k), bf16_bits_to_f32(wl.new_k[b:b + 1])])
        t = np.arange(L)
        blk = wl.block_tables[b, t // 32]
        codes = kc[blk, t % 32].astype(np.float64)                 # [L, H, d]
        sc = ks[blk].astype(np.float64)[:, :, None]
        # within half a step, plus the fp32 rounding of the quotient x / s
        assert (np.abs(codes * sc - xs) <= sc * (0.5 + 127 * 2.0 ** -23)).all()
        for j in range((L + 31) // 32):
            sel = (t // 32) == j
            for h in range(2):
                assert np.abs(codes[sel, h]).max() == 127


def test_int8_pool_is_deterministic_per_sequence(oracle_mod):
    """Filling only some sequences gives the same codes in their blocks."""
    wl = workloads.custom(batch=3, num_q_heads=8, num_kv_heads=1, head_dim=64, block_size=32,
                          seq_lens=[40, 70, 9], kv_dtype="int8", seed=19)
    full = oracle_pool(wl)
    part = oracle_pool(wl, seqs=[1])
    blocks = wl.block_tables[1, :3]
    np.testing.assert_array_equal(full[0][blocks], part[0][blocks])
    np.testing.assert_array_equal(full[2][blocks], part[2][blocks])
