"""Test-side helpers that build the oracle's view of a workload.

Every pool here is filled by the oracle itself (its slot mapping and its
append) from the generator's token values; nothing comes from the CUDA path.
"""
import numpy as np

import oracle
from workloads import bf16_bits_to_f32


def oracle_pool(wl, seqs=None, with_new_token=True):
    """Oracle K/V pools for workload ``wl`` (optionally only sequences
    ``seqs``): poisoned pools, the cached tokens appended through the oracle's
    slot mapping, then (by default) the decode step's new token appended at
    position L_b - 1.  Returns (k_cache, v_cache, k_scale, v_scale)."""
    s = wl.spec
    kc, vc = wl.poisoned_pool(), wl.poisoned_pool()
    int8 = s.kv_dtype == "int8"
    ks = vs = None
    if int8:
        ks, vs = wl.scales(seqs)
    for ch in wl.fill_chunks(seqs):
        slots, rc = oracle.token_slots(wl.block_tables, ch.positions, s.block_size,
                                       wl.num_blocks, seq_idx=ch.seq_idx)
        assert rc == 0
        if int8:
            rc = oracle.append_int8(ch.k, ch.v, kc, vc, ks, vs, slots)
        else:
            rc = oracle.append_bf16(ch.k, ch.v, kc, vc, slots)
        assert rc == 0
    if with_new_token:
        b_all = np.arange(s.batch) if seqs is None else np.asarray(list(seqs))
        slots, rc = decode_slots(wl)
        assert rc == 0
        sel = np.full(s.batch, -1, np.int64)
        sel[b_all] = slots[b_all]
        if int8:
            rc = oracle.append_int8(wl.new_k, wl.new_v, kc, vc, ks, vs, sel)
        else:
            rc = oracle.append_bf16(wl.new_k, wl.new_v, kc, vc, sel)
        assert rc == 0
    return kc, vc, ks, vs


def decode_slots(wl):
    """Oracle slots of each sequence's new token (position L_b - 1)."""
    pos = (wl.seq_lens.astype(np.int64) - 1).astype(np.int32)
    return oracle.token_slots(wl.block_tables, pos, wl.spec.block_size, wl.num_blocks)


def contiguous_kv(wl, b):
    """fp64 K, V [L_b, Hkv, d] of sequence b in logical order, straight from
    the generator's values (no pool, no block table): the un-paged layout."""
    s = wl.spec
    P = s.shared_prefix_tokens
    parts_k, parts_v = [], []
    if P:
        pk, pv = wl._prefix_kv()
        parts_k.append(bf16_bits_to_f32(pk))
        parts_v.append(bf16_bits_to_f32(pv))
    _, k, v = wl.own_tokens(b)
    parts_k += [bf16_bits_to_f32(k), bf16_bits_to_f32(wl.new_k[b:b + 1])]
    parts_v += [bf16_bits_to_f32(v), bf16_bits_to_f32(wl.new_v[b:b + 1])]
    return (np.concatenate(parts_k).astype(np.float64),
            np.concatenate(parts_v).astype(np.float64))
