"""Seeded synthetic decode batches for paged attention (inputs only).

This module draws inputs and nothing else: sequence lengths, the random
physical placement of each sequence's blocks, q, the K/V values of every
cached token, the new token's k/v and (for int8 pools) the per-(block, KV
head) scales.  It holds none of the method's arithmetic: it never computes a
slot, never writes a pool, never quantises and never attends.  Each side of a
parity check (the CUDA path, the CPU oracle) fills its own pool from the
``fill_chunks`` this module yields, with its own slot mapping and append.

Workloads follow the shapes of the pages' examples (Llama-3.1-8B-like GQA with
32 query / 8 KV heads and head_dim 128; a Llama-2-70B-like 64 / 8 layout; a
shared 800-token system prompt; 16-token blocks, 32 for the int8 case):

  1 tiny           B 4,   8/2 heads,  d 64,  bs 16, L ~ U{1..200}, pool 64 blocks
  2 8B-like        B 64,  32/8 heads, d 128, bs 16, L ~ U{512..4096}
  3 long split-K   B 8,   32/8 heads, d 128, bs 16, L ~ U{32768..131072}
  4 shared prefix  B 256, 32/8 heads, d 128, bs 16, L = 800 + clip(round(
                   lognormal(6, 1)), 16, 2048); blocks 0..49 shared by all
  5 70B-like INT8  B 128, 64/8 heads, d 128, bs 32, L ~ U{1024..8192},
                   int8 pool, scale = max|x| / 127 per (block, KV head)
  6 70B-like FP8   as 5 with an FP8 E4M3 pool, scale = max|x| / 448
  7 spec. verify   as 2, the last 5 tokens of each sequence are queries
                   (the gamma = 5 draft tokens scored in one pass)
  8 decode-max     as 2, sequence 0's last 512 tokens are a prefill chunk,
                   the other 63 sequences decode one token

Recipe: ``numpy.random.Generator(PCG64)`` streams spawned from
``SeedSequence(20260000 + config)``: stream 0 draws lengths then placement,
stream 1 draws q, stream 2 the new tokens' k and v, stream 3 a shared prefix,
and stream 4 + b the cached tokens of sequence b (so one sequence can be
regenerated alone).  Values are N(0, 1) in fp32 rounded to the nearest-even
bf16.  The pool holds ceil(1.25 x needed blocks) unless the config fixes it;
placement is a seeded random permutation of the pool, each sequence taking
the next ``ceil(L_b / bs)`` entries.  With query_len n_b > 1 the last n_b
tokens of sequence b are this step's queries and appended tokens (q and the
new k, v have one row per query token, sequences in order); its cached
tokens are positions ``0 .. L_b - n_b - 1``.  Unused pool memory starts poisoned
(bf16 NaN, int8 127, E4M3 NaN 0x7F) and table padding is -1.  ``L_b`` counts the token
appended in this step; cached tokens are positions ``0 .. L_b - 2``.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from typing import Callable, Iterable, Iterator, Optional, Sequence

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
INT8_POISON = np.int8(127)
FP8_NAN = np.uint8(0x7F)            # the E4M3 NaN pattern
# largest code magnitude of each 8-bit KV format: scale = max |x| / this
CODE_MAX = {"int8": 127.0, "fp8": 448.0}
SEED_BASE = 20260000


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to the nearest-even bf16 and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    t = np.right_shift(u, np.uint32(16))
    np.bitwise_and(t, np.uint32(1), out=t)             # the kept part's lowest bit
    np.add(t, np.uint32(0x7FFF), out=t)
    np.add(t, u, out=t)
    np.right_shift(t, np.uint32(16), out=t)
    return t.astype(np.uint16)


def default_workers() -> int:
    """Threads for drawing per-sequence token values (numpy's generators and
    ufuncs release the GIL on large arrays)."""
    return max(1, min(16, os.cpu_count() or 1))


def ordered_map(fn: Callable, items: Iterable, workers: int) -> Iterator:
    """fn over items, results in input order, at most 2 x workers computed
    ahead (so a long batch never holds all its values at once)."""
    items = list(items)
    if workers <= 1 or len(items) <= 1:
        for it in items:
            yield fn(it)
        return
    with ThreadPoolExecutor(max_workers=workers) as ex:
        ahead = 2 * workers
        futs = [ex.submit(fn, it) for it in items[:ahead]]
        nxt = len(futs)
        for i in range(len(items)):
            res = futs[i].result()
            futs[i] = None
            if nxt < len(items):
                futs.append(ex.submit(fn, items[nxt]))
                nxt += 1
            yield res


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Spec:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str                      # "bf16" | "int8" | "fp8" (E4M3)
    lens: tuple                        # ("uniform", lo, hi) | ("prefix_lognormal", ...) | ("fixed", [..])
    num_blocks: Optional[int] = None   # None: ceil(1.25 * needed)
    max_blocks_per_seq: Optional[int] = None
    shared_prefix_tokens: int = 0
    query_len: object = 1              # query tokens per sequence: an int, or
                                       # ("chunk_first", n): sequence 0 has n, the rest 1

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


CONFIGS = {
    1: Spec("tiny paged decode (B4, 8/2 heads, d64, bs16, L 1..200, 64 blocks)",
            4, 8, 2, 64, 16, "bf16", ("uniform", 1, 200), num_blocks=64,
            max_blocks_per_seq=13),
    2: Spec("Llama-3.1-8B-like decode layer (B64, 32/8 heads, d128, bs16, L 512..4096)",
            64, 32, 8, 128, 16, "bf16", ("uniform", 512, 4096),
            max_blocks_per_seq=256),
    3: Spec("long-context split-K (B8, 32/8 heads, d128, bs16, L 32768..131072)",
            8, 32, 8, 128, 16, "bf16", ("uniform", 32768, 131072),
            max_blocks_per_seq=8192),
    4: Spec("shared-prefix mixed batch (B256, 32/8 heads, d128, bs16, 800-token shared prefix)",
            256, 32, 8, 128, 16, "bf16", ("prefix_lognormal", 6.0, 1.0, 16, 2048),
            max_blocks_per_seq=(800 + 2048 + 15) // 16, shared_prefix_tokens=800),
    5: Spec("Llama-2-70B-like INT8 KV (B128, 64/8 heads, d128, bs32, L 1024..8192)",
            128, 64, 8, 128, 32, "int8", ("uniform", 1024, 8192),
            max_blocks_per_seq=256),
    6: Spec("Llama-2-70B-like FP8 E4M3 KV (B128, 64/8 heads, d128, bs32, L 1024..8192)",
            128, 64, 8, 128, 32, "fp8", ("uniform", 1024, 8192),
            max_blocks_per_seq=256),
    7: Spec("speculative verification, 5 draft tokens per sequence (B64, 32/8 heads, d128, "
            "bs16, L 512..4096)",
            64, 32, 8, 128, 16, "bf16", ("uniform", 512, 4096),
            max_blocks_per_seq=256, query_len=5),
    8: Spec("decode-maximal batch: one 512-token prefill chunk + 63 decodes (B64, 32/8 heads, "
            "d128, bs16, L 512..4096)",
            64, 32, 8, 128, 16, "bf16", ("uniform", 512, 4096),
            max_blocks_per_seq=256, query_len=("chunk_first", 512)),
}


@dataclass
class FillChunk:
    """Cached tokens to append before the decode step: token i belongs to
    sequence ``seq_idx[i]`` at position ``positions[i]``."""
    seq_idx: np.ndarray    # int32 [n]
    positions: np.ndarray  # int32 [n]
    k: np.ndarray          # bf16 bits [n, Hkv, d]
    v: np.ndarray


class Workload:
    """One synthetic decode step."""

    def __init__(self, spec: Spec, seed: int, seq_lens: Optional[Sequence[int]] = None,
                 query_lens: Optional[Sequence[int]] = None):
        self.spec = spec
        self.seed = seed
        ss = np.random.SeedSequence(seed)
        self._children = ss.spawn(4)
        self._seq_root = self._children[3]
        s0 = np.random.Generator(np.random.PCG64(self._children[0]))
        B, bs = spec.batch, spec.block_size
        P = spec.shared_prefix_tokens
        if seq_lens is not None:
            lens = np.asarray(seq_lens, np.int64)
            assert lens.shape == (B,)
        elif spec.lens[0] == "uniform":
            lens = s0.integers(spec.lens[1], spec.lens[2], size=B, endpoint=True)
        elif spec.lens[0] == "prefix_lognormal":
            _, mu, sigma, lo, hi = spec.lens
            suffix = np.clip(np.rint(s0.lognormal(mu, sigma, size=B)), lo, hi)
            lens = P + suffix.astype(np.int64)
        else:
            raise ValueError(spec.lens)
        self.seq_lens = lens.astype(np.int32)
        nblk = [(int(L) + bs - 1) // bs for L in self.seq_lens]
        shared = P // bs
        needed = sum(nblk) - shared * max(B - 1, 0) if shared else sum(nblk)
        NB = spec.num_blocks or int(math.ceil(1.25 * needed))
        self.num_blocks = NB
        MB = spec.max_blocks_per_seq or max(max(nblk), 1)
        assert max(nblk) <= MB, "a sequence needs more blocks than the table holds"
        self.max_blocks_per_seq = MB
        perm = s0.permutation(NB).astype(np.int32)
        bt = np.full((B, MB), -1, np.int32)
        nxt = shared
        for b in range(B):
            bt[b, :shared] = perm[:shared]
            own = nblk[b] - shared
            bt[b, shared:nblk[b]] = perm[nxt:nxt + own]
            nxt += own
        assert nxt <= NB
        self.block_tables = bt
        # query tokens: the last n_b tokens of sequence b (n_b = 1: decode)
        if query_lens is not None:
            n = np.asarray(query_lens, np.int64)
        elif isinstance(spec.query_len, tuple):
            assert spec.query_len[0] == "chunk_first"
            n = np.ones(B, np.int64)
            n[0] = spec.query_len[1]
        else:
            n = np.full(B, spec.query_len, np.int64)
        assert n.shape == (B,) and (n >= 0).all() and (n <= self.seq_lens).all()
        self.query_lens = n.astype(np.int32)
        self.query_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        T = int(self.query_start[-1])
        s1 = np.random.Generator(np.random.PCG64(self._children[1]))
        self.q = to_bf16_bits(s1.standard_normal((T, spec.num_q_heads, spec.head_dim), np.float32))
        s2 = np.random.Generator(np.random.PCG64(self._children[2]))
        shp = (T, spec.num_kv_heads, spec.head_dim)
        self.new_k = to_bf16_bits(s2.standard_normal(shp, np.float32))
        self.new_v = to_bf16_bits(s2.standard_normal(shp, np.float32))
        self._prefix = None
        self._scales = None

    # -- shapes ----------------------------------------------------------
    @property
    def pool_shape(self):
        s = self.spec
        return (self.num_blocks, s.block_size, s.num_kv_heads, s.head_dim)

    @property
    def kv_elem_bytes(self) -> int:
        return 2 if self.spec.kv_dtype == "bf16" else 1

    def poisoned_pool(self) -> np.ndarray:
        if self.spec.kv_dtype == "int8":
            return np.full(self.pool_shape, INT8_POISON, np.int8)
        if self.spec.kv_dtype == "fp8":
            return np.full(self.pool_shape, FP8_NAN, np.uint8)
        return np.full(self.pool_shape, BF16_NAN, np.uint16)

    # -- cached token values ---------------------------------------------
    def _stream(self, which: int) -> np.random.Generator:
        child = np.random.SeedSequence(self.seed, spawn_key=(3, which))
        return np.random.Generator(np.random.PCG64(child))

    def _prefix_kv(self):
        if self._prefix is None:
            P, s = self.spec.shared_prefix_tokens, self.spec
            g = self._stream(0)
            shp = (P, s.num_kv_heads, s.head_dim)
            self._prefix = (to_bf16_bits(g.standard_normal(shp, np.float32)),
                            to_bf16_bits(g.standard_normal(shp, np.float32)))
        return self._prefix

    @property
    def num_tokens(self) -> int:
        """Query tokens of the step (= batch for one-token decode)."""
        return int(self.query_start[-1])

    def new_kv_of(self, b: int):
        """bf16 bits of the K, V rows sequence b appends this step."""
        a, e = int(self.query_start[b]), int(self.query_start[b + 1])
        return self.new_k[a:e], self.new_v[a:e]

    def new_positions(self):
        """(sequence, position) int32 [T] of every token appended this step:
        the last n_b positions of sequence b."""
        seq = np.repeat(np.arange(self.spec.batch, dtype=np.int32), self.query_lens)
        first = np.repeat(self.seq_lens - self.query_lens, self.query_lens)
        off = np.arange(self.num_tokens, dtype=np.int32) - np.repeat(self.query_start[:-1], self.query_lens)
        return seq, (first + off).astype(np.int32)

    def own_tokens(self, b: int):
        """Cached tokens that sequence b alone owns: (positions, k, v)."""
        s = self.spec
        P = s.shared_prefix_tokens
        L = int(self.seq_lens[b])
        hi = L - int(self.query_lens[b])
        lo = min(P, hi)
        n = max(hi - lo, 0)
        g = self._stream(1 + b)
        shp = (n, s.num_kv_heads, s.head_dim)
        k = to_bf16_bits(g.standard_normal(shp, np.float32))
        v = to_bf16_bits(g.standard_normal(shp, np.float32))
        return np.arange(lo, hi, dtype=np.int32), k, v

    def fill_chunks(self, seqs: Optional[Sequence[int]] = None,
                    workers: Optional[int] = None) -> Iterator[FillChunk]:
        """Chunks of cached tokens to append before the step (the shared
        prefix once, through sequence 0's table, then each sequence's own).
        Sequences are drawn on ``workers`` threads (default: the host's cores,
        at most 16); each has its own stream, so the values do not depend on
        the thread count."""
        s = self.spec
        seqs = range(s.batch) if seqs is None else seqs
        P = s.shared_prefix_tokens
        if P:
            pk, pv = self._prefix_kv()
            first = 0 if seqs is None else min(seqs)
            yield FillChunk(np.full(P, first, np.int32), np.arange(P, dtype=np.int32), pk, pv)
        nw = default_workers() if workers is None else workers
        for b, (pos, k, v) in zip(seqs, ordered_map(self.own_tokens, seqs, nw)):
            if pos.size:
                yield FillChunk(np.full(pos.size, b, np.int32), pos, k, v)

    # -- 8-bit scales ------------------------------------------------------
    def scales(self, seqs: Optional[Sequence[int]] = None):
        """fp32 k_scale, v_scale [NB, Hkv]: max |x| / 127 (int8) or / 448
        (E4M3) over the bf16 values (cached plus new) that land in each
        (block, KV head), the shared prefix's blocks included; 1.0 elsewhere."""
        s = self.spec
        NB, H, bs = self.num_blocks, s.num_kv_heads, s.block_size
        ks = np.ones((NB, H), np.float32)
        vs = np.ones((NB, H), np.float32)
        seqs = range(s.batch) if seqs is None else seqs
        P = s.shared_prefix_tokens
        assert P % bs == 0, "a shared prefix fills whole blocks"
        top = np.float32(CODE_MAX[s.kv_dtype])

        def put(rows_k, rows_v, phys):
            # rows [n, H, d] fp32 of whole blocks phys (zero-padded at the end)
            n = len(phys) * bs
            pad = ((0, n - rows_k.shape[0]), (0, 0), (0, 0))
            kmax = np.abs(np.pad(rows_k, pad)).reshape(len(phys), bs, H, -1).max(axis=(1, 3))
            vmax = np.abs(np.pad(rows_v, pad)).reshape(len(phys), bs, H, -1).max(axis=(1, 3))
            ks[phys] = np.where(kmax > 0, kmax / top, np.float32(1.0))
            vs[phys] = np.where(vmax > 0, vmax / top, np.float32(1.0))

        if P:
            pk, pv = self._prefix_kv()
            first = min(seqs) if len(seqs) else 0
            put(bf16_bits_to_f32(pk), bf16_bits_to_f32(pv), self.block_tables[first, :P // bs])
        for b, (pos, k, v) in zip(seqs, ordered_map(self.own_tokens, seqs, default_workers())):
            L = int(self.seq_lens[b])
            nk, nv = self.new_kv_of(b)
            kf = np.concatenate([bf16_bits_to_f32(k), bf16_bits_to_f32(nk)])
            vf = np.concatenate([bf16_bits_to_f32(v), bf16_bits_to_f32(nv)])
            nblk = (L + bs - 1) // bs
            put(kf, vf, self.block_tables[b, P // bs:nblk])
        return ks, vs

    # -- byte accounting -----------------------------------------------------
    def kv_bytes_logical(self) -> int:
        """K and V bytes the step reads, counting shared blocks per reader."""
        s = self.spec
        return int(self.seq_lens.astype(np.int64).sum()) * 2 * s.num_kv_heads * s.head_dim * self.kv_elem_bytes

    def kv_bytes_unique(self) -> int:
        """K and V bytes of distinct cached tokens (a shared prefix once)."""
        s = self.spec
        P = s.shared_prefix_tokens
        toks = int(self.seq_lens.astype(np.int64).sum()) - P * max(s.batch - 1, 0)
        return toks * 2 * s.num_kv_heads * s.head_dim * self.kv_elem_bytes


def make(config: int, seed: Optional[int] = None, seq_lens=None,
         kv_dtype: Optional[str] = None) -> Workload:
    """Workload `config`; with kv_dtype, the same shapes, lengths and values
    on a pool of that type ("bf16", "int8" or "fp8")."""
    spec = CONFIGS[config]
    if kv_dtype is not None and kv_dtype != spec.kv_dtype:
        spec = replace(spec, kv_dtype=kv_dtype, name=f"{spec.name}, {kv_dtype} KV")
    return Workload(spec, SEED_BASE + config if seed is None else seed, seq_lens)


def custom(*, batch, num_q_heads, num_kv_heads, head_dim, block_size, seq_lens,
           kv_dtype="bf16", num_blocks=None, max_blocks_per_seq=None,
           shared_prefix_tokens=0, seed=1234, query_lens=None) -> Workload:
    """A small workload with explicit lengths (tests: edge cases); with
    query_lens, each sequence's last query_lens[b] tokens are its queries."""
    spec = Spec("custom", batch, num_q_heads, num_kv_heads, head_dim, block_size,
                kv_dtype, ("fixed",), num_blocks=num_blocks,
                max_blocks_per_seq=max_blocks_per_seq,
                shared_prefix_tokens=shared_prefix_tokens)
    return Workload(spec, seed, seq_lens=seq_lens, query_lens=query_lens)


class BeamWorkload:
    """Seeded inputs of a beam-search (parallel-sampling) decode run over a
    shared pool: ``num_parents`` prompts of ``parent_lens`` tokens, each
    forked into ``beams`` sequences (beam 0 is the parent itself) that then
    decode ``steps`` tokens each, every beam its own k, v and q per step.

    Inputs only, like ``Workload``: which blocks are shared, copied or taken
    is decided by the pool under test.  Recipe: ``SeedSequence(seed)`` spawns
    stream 0 (the prompts' k and v), stream 1 (per-step q), stream 2 (per-step
    k and v) and stream 3 (8-bit scales of every physical block: U(3.5, 4.5) /
    127 (int8) or / 448 (E4M3) per (block, KV head), fixed up front because a block's scale outlives
    the sequence that first fills it).  Values are N(0, 1) rounded to bf16.
    Sequence ``p * beams + j`` is beam j of parent p."""

    def __init__(self, *, num_parents, beams, parent_lens, steps, num_q_heads, num_kv_heads,
                 head_dim, block_size, num_blocks, max_blocks_per_seq, kv_dtype="bf16",
                 seed=SEED_BASE + 97):
        self.num_parents, self.beams, self.steps = num_parents, beams, steps
        self.parent_lens = np.asarray(parent_lens, np.int32)
        assert self.parent_lens.shape == (num_parents,)
        self.num_q_heads, self.num_kv_heads, self.head_dim = num_q_heads, num_kv_heads, head_dim
        self.block_size, self.num_blocks = block_size, num_blocks
        self.max_blocks_per_seq, self.kv_dtype = max_blocks_per_seq, kv_dtype
        self.scale = 1.0 / math.sqrt(head_dim)
        st = [np.random.Generator(np.random.PCG64(c)) for c in np.random.SeedSequence(seed).spawn(4)]
        kv = (num_kv_heads, head_dim)
        self.parent_k = [to_bf16_bits(st[0].standard_normal((int(L),) + kv, np.float32))
                         for L in self.parent_lens]
        self.parent_v = [to_bf16_bits(st[0].standard_normal((int(L),) + kv, np.float32))
                         for L in self.parent_lens]
        n = num_parents * beams
        self.step_q = to_bf16_bits(st[1].standard_normal((steps, n, num_q_heads, head_dim),
                                                         np.float32))
        self.step_k = to_bf16_bits(st[2].standard_normal((steps, n) + kv, np.float32))
        self.step_v = to_bf16_bits(st[2].standard_normal((steps, n) + kv, np.float32))
        sc = st[3].uniform(3.5, 4.5, size=(2, num_blocks, num_kv_heads)).astype(np.float32)
        top = np.float32(CODE_MAX.get(kv_dtype, 127.0))
        self.k_scale, self.v_scale = sc[0] / top, sc[1] / top

    @property
    def num_seqs(self) -> int:
        return self.num_parents * self.beams

    def seq_lens_at(self, step: int) -> np.ndarray:
        """Lengths of every sequence in decode step ``step`` (counting the
        token that step appends)."""
        return np.repeat(self.parent_lens, self.beams).astype(np.int32) + np.int32(step + 1)

    def poisoned_pool(self) -> np.ndarray:
        shape = (self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim)
        if self.kv_dtype == "int8":
            return np.full(shape, INT8_POISON, np.int8)
        if self.kv_dtype == "fp8":
            return np.full(shape, FP8_NAN, np.uint8)
        return np.full(shape, BF16_NAN, np.uint16)

    def dense_tokens(self, seq: int, step: int):
        """bf16 bits of K, V [L, Hkv, d] of sequence ``seq`` after decode step
        ``step`` in logical order: the parent's prompt, then the beam's own
        step tokens (the un-paged, unshared view)."""
        p = seq // self.beams
        k = np.concatenate([self.parent_k[p], self.step_k[:step + 1, seq]])
        v = np.concatenate([self.parent_v[p], self.step_v[:step + 1, seq]])
        return k, v


def beam_search_8b(seed: int = SEED_BASE + 98, steps: int = 64) -> BeamWorkload:
    """Beam search over the Llama-3.1-8B-like decode layer: 16 prompts of
    U{512..4096} tokens, 4 beams each (B 64, 32/8 heads, d 128, 16-token
    blocks); the pool holds ceil(1.25 x) the blocks the prompts and every
    beam's own decoded tokens (plus one copied block per beam) need."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(5)[4]))
    parents, beams, bs = 16, 4, 16
    lens = g.integers(512, 4096, size=parents, endpoint=True)
    need = sum((int(L) + bs - 1) // bs for L in lens) + parents * beams * ((steps + bs - 1) // bs + 1)
    mb = (int(lens.max()) + steps + bs - 1) // bs
    return BeamWorkload(num_parents=parents, beams=beams, parent_lens=lens, steps=steps,
                        num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=bs,
                        num_blocks=int(math.ceil(1.25 * need)), max_blocks_per_seq=mb, seed=seed)
