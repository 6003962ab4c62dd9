"""Test-side helpers that build the oracle's view of a workload.

Every pool here is filled by the oracle itself (its slot mapping and its
append) from the generator's token values; nothing comes from the CUDA path.
"""
import numpy as np

import oracle
from workloads import bf16_bits_to_f32


def oracle_pool(wl, seqs=None, with_new_token=True):
    """Oracle K/V pools for workload ``wl``: ``oracle.workload_pools``."""
    return oracle.workload_pools(wl, seqs, with_new_token)


append_any = oracle.append_any


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
    nk, nv = wl.new_kv_of(b)
    parts_k += [bf16_bits_to_f32(k), bf16_bits_to_f32(nk)]
    parts_v += [bf16_bits_to_f32(v), bf16_bits_to_f32(nv)]
    return (np.concatenate(parts_k).astype(np.float64),
            np.concatenate(parts_v).astype(np.float64))


class OracleBeamRun:
    """A beam-search decode run driven entirely by the oracle: the block pool
    model decides sharing, copies and new blocks; ``oracle.copy_blocks``
    copies; the oracle's slot mapping and append write each step's tokens;
    ``oracle.paged_attention`` attends.  ``pool`` may be any object with the
    model's alloc / fork / prepare_append methods (a mutant in the tests)."""

    def __init__(self, w, pool=None):
        self.w = w
        self.pool = pool if pool is not None else oracle.BlockPoolModel(w.num_blocks)
        self.q8 = w.kv_dtype != "bf16"
        self.kc, self.vc = w.poisoned_pool(), w.poisoned_pool()
        self.ks = w.k_scale.copy() if self.q8 else None
        self.vs = w.v_scale.copy() if self.q8 else None
        MB, bs = w.max_blocks_per_seq, w.block_size
        self.tables = []
        for p, L in enumerate(w.parent_lens):
            ids = self.pool.alloc_sequence(int(L), bs)
            row = np.full(MB, -1, np.int32)
            row[:len(ids)] = ids
            pos = np.arange(L, dtype=np.int32)
            slots, rc = oracle.token_slots(row[None], pos, bs, w.num_blocks,
                                           seq_idx=np.zeros(int(L), np.int32))
            assert rc == 0
            self._append(w.parent_k[p], w.parent_v[p], slots)
            for j in range(w.beams):
                if j:
                    self.pool.fork(ids)
                self.tables.append(row.copy())
        self.step = -1

    def _append(self, k, v, slots):
        assert append_any(k, v, self.kc, self.vc, self.ks, self.vs, slots) == 0

    def table_array(self):
        return np.stack(self.tables).astype(np.int32)

    def advance(self):
        """One decode step: make the targets writable, copy, append.  Returns
        the (src, dst) copies."""
        w = self.w
        self.step += 1
        lens = w.seq_lens_at(self.step)
        rows = [list(t) for t in self.tables]
        copies = self.pool.prepare_append(rows, lens, w.block_size)
        self.tables = [np.asarray(r, np.int32) for r in rows]
        oracle.copy_blocks(self.kc, self.vc, copies, self.ks, self.vs)
        pos = (lens - 1).astype(np.int32)
        slots, rc = oracle.token_slots(self.table_array(), pos, w.block_size, w.num_blocks)
        assert rc == 0
        self._append(w.step_k[self.step], w.step_v[self.step], slots)
        return copies

    def attend(self, rows=None):
        w = self.w
        return oracle.paged_attention(w.step_q[self.step], self.kc, self.vc, self.table_array(),
                                      w.seq_lens_at(self.step), w.scale, k_scale=self.ks,
                                      v_scale=self.vs, rows=rows)
