"""Plain CPU oracle for decode-phase paged attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product (``paged_kv_cache_97_gb300``)
never imports it, and it imports nothing from the product.

Contents, each citing the passage it follows (page titles as printed):

* size formulas -- ``block_memory_bytes`` (“让 Agent 跑得快：LLM 推理服务”, §二
  PagedAttention, the block_memory formula), ``kv_bytes_per_token`` (same page,
  §一 “KV Cache”), ``kv_cache_bytes`` (“LLM 推理优化技术全景”, KV Cache 大小公式),
  ``blocks_needed`` / ``internal_waste_tokens`` (“LLM 推理引擎深度解析”, §2.1
  PagedKVCache.allocate; “让 Agent 跑得快”, §五: waste only in the last block);
* ``BlockPoolModel`` -- the block pool's allocation rules (“LLM 推理引擎深度解析”,
  §2.1: FIFO free list, all-or-nothing allocation that fails when short,
  free returns every block) and its sharing rules (“让 Agent 跑得快”, §二
  Copy-on-Write: reference counts, copy before writing a shared block);
* ``copy_blocks`` -- the block copy of copy-on-write (plain numpy);
* ``fnv1a64``, ``block_hash`` -- the prefix cache's block hash chain
  (“让 Agent 跑得快”, §七; FNV-1a from its published definition);
* ``workload_pools`` -- the oracle's own pools for a seeded workload (its
  slot mapping and append over the generator's token values);
* ``token_slots``, ``append_bf16``, ``append_int8``, ``quantize_int8``,
  ``append_fp8``, ``quantize_fp8``, ``fp8_value``, ``paged_attention_multi``
  (multi-token causal queries),
  ``paged_attention`` (three-pass or online), ``attention_partials``,
  ``lse_merge`` -- thin ctypes wrappers over ``pagedkv_oracle.c`` (plain C,
  fp64), whose header cites the passages it follows.

Parity pins: every function here is pinned by tests under ``tests/`` that run
without a GPU (``-m "not gpu"``) against values the pages print, closed forms,
brute force and a library routine; none is "parity unpinned".
"""
from __future__ import annotations

import copy
import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle_pagedkv.so")
_lib = None

OK, INVALID, INDEX = 0, 1, 4


# --------------------------------------------------------------------------
# Build / load
# --------------------------------------------------------------------------

def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", "-D_GNU_SOURCE",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _bind(lib):
    """Declare the C signatures on a loaded copy of the oracle library."""
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_token_slots.argtypes = [P, I, P, P, I, I, I, P]
    lib.oracle_append_bf16.argtypes = [P, P, P, P, P, I, I, I, I, I]
    lib.oracle_append_int8.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I]
    lib.oracle_quantize_int8.argtypes = [ctypes.c_float, ctypes.c_float]
    lib.oracle_append_fp8.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I]
    lib.oracle_quantize_fp8.argtypes = [ctypes.c_float, ctypes.c_float]
    lib.oracle_fp8_value.argtypes = [I]
    lib.oracle_fp8_value.restype = D
    lib.oracle_paged_attention.argtypes = [P, P, P, P, P, P, I, P, I, P, I, I,
                                           I, I, I, I, D, P, I, I, I]
    lib.oracle_attention_partials.argtypes = [P, P, P, P, P, P, P, I, P, I, P,
                                              I, I, I, I, I, I, D, I, I, I]
    lib.oracle_paged_attention_multi.argtypes = [P, P, P, P, P, P, I, P, I, P, P, I, I, I, I,
                                                 I, I, I, D, I, I]
    lib.oracle_lse_merge.argtypes = [P, P, I, I, P]
    lib.oracle_lse_merge.restype = None
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# Size formulas
# --------------------------------------------------------------------------

def block_memory_bytes(block_size: int, num_kv_heads: int, head_size: int,
                       dtype_size: int) -> int:
    """Bytes of one physical block holding K and V.

    “让 Agent 跑得快：LLM 推理服务”, §二 PagedAttention: block_memory =
    2 × block_size × num_kv_heads × head_size × dtype_size, the 2 counting
    K and V.
    """
    return 2 * block_size * num_kv_heads * head_size * dtype_size


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int,
                       dtype_size: int) -> int:
    """KV bytes one token occupies over all layers.

    “让 Agent 跑得快：LLM 推理服务”, §一 KV Cache: 2 × L × H × head_dim ×
    dtype_size (H = KV heads).
    """
    return 2 * num_layers * num_kv_heads * head_dim * dtype_size


def kv_cache_bytes(num_layers: int, num_kv_heads: int, head_dim: int,
                   seq_len: int, batch: int, dtype_size: int) -> int:
    """Whole KV cache of a batch.

    “LLM 推理优化技术全景”, KV Cache 大小公式: 2 × n_layers × n_kv_heads ×
    d_head × seq_len × batch × dtype_bytes.
    """
    return 2 * num_layers * num_kv_heads * head_dim * seq_len * batch * dtype_size


def blocks_needed(seq_len: int, block_size: int) -> int:
    """ceil(seq_len / block_size) (“LLM 推理引擎深度解析”, §2.1 allocate)."""
    return (seq_len + block_size - 1) // block_size


def internal_waste_tokens(seq_len: int, block_size: int) -> int:
    """Unused token slots, all in the last block (“让 Agent 跑得快”, §五)."""
    return blocks_needed(seq_len, block_size) * block_size - seq_len


# --------------------------------------------------------------------------
# Block pool model
# --------------------------------------------------------------------------

@dataclass
class BlockPoolModel:
    """Allocation, sharing and copy-on-write rules of the physical block pool.

    “LLM 推理引擎深度解析”, §2.1 (PagedKVCache): the pool starts with every
    block id free in ascending order; allocation takes ids from the front of
    the free list, all or none, and fails when too few are free; freeing
    appends the ids to the back.

    “让 Agent 跑得快：LLM 推理服务”, §二 (Copy-on-Write：Beam Search 的内存优化):
    sequences forked from one prefix map the same physical blocks, each
    holding a reference; a sequence that must write a token into a block
    held more than once first copies the block and points its table at the
    copy; a block whose count reaches zero goes back to the pool.  §五 (共享
    前缀): only the current decode token writes, and a new block is taken each
    time a sequence fills its last one.

    Readings of this library where the pages are silent: freeing drops one
    reference per listed id (an id listed more often than it is held, or not
    held at all, is an error and nothing changes); blocks whose count reaches
    zero join the free list in the order listed; ``prepare_append`` handles
    the sequences of a step in order, each copy or new block taking the front
    of the free list, and changes nothing when the list runs short.

    Prefix cache, “让 Agent 跑得快”, §七 (前缀缓存): a full block's hash
    chains its parent's hash, its tokens and extra keys (``block_hash``); a
    request looks its prompt's full blocks up in order, stopping at the first
    miss, and takes a reference on every hit (a cached free block leaves the
    free list); a finished request's blocks stay findable in the free list
    until allocation takes them again, which evicts them.  Readings: a hit
    also requires the stored tokens, parent hash and key to match; a block
    whose content is already registered elsewhere is not registered again.
    """
    num_blocks: int
    free_list: list = field(default_factory=list)
    refs: dict = field(default_factory=dict)      # block id -> references (> 0)
    cache: dict = field(default_factory=dict)     # block id -> (hash, parent, key, tokens)
    by_hash: dict = field(default_factory=dict)   # hash -> block id

    def __post_init__(self):
        self.free_list = list(range(self.num_blocks))

    def alloc(self, n: int) -> list:
        if n < 0:
            raise ValueError("negative block count")
        if len(self.free_list) < n:
            raise MemoryError("block pool exhausted")
        ids, self.free_list = self.free_list[:n], self.free_list[n:]
        for i in ids:
            self.refs[i] = 1
            if i in self.cache:                       # reused: its cached content goes
                del self.by_hash[self.cache.pop(i)[0]]
        return ids

    def match_prefix(self, tokens, block_size, extra_key=0) -> list:
        hits, parent = [], 0
        for j in range(len(tokens) // block_size):
            blk = tuple(int(x) for x in tokens[j * block_size:(j + 1) * block_size])
            h = block_hash(parent, blk, extra_key)
            i = self.by_hash.get(h)
            if i is None or self.cache[i] != (h, parent, extra_key, blk):
                break
            if i not in self.refs:                    # cached but free
                self.free_list.remove(i)
                self.refs[i] = 0
            self.refs[i] += 1
            hits.append(i)
            parent = h
        return hits

    def register_prefix(self, ids, tokens, block_size, extra_key=0) -> None:
        n = len(tokens) // block_size
        ids = list(ids)[:n]
        if any(i not in self.refs for i in ids):
            raise ValueError("registering a block that is not allocated")
        parent, plan = 0, []
        for j, i in enumerate(ids):
            blk = tuple(int(x) for x in tokens[j * block_size:(j + 1) * block_size])
            h = block_hash(parent, blk, extra_key)
            if i in self.cache and self.cache[i][0] != h:
                raise ValueError("block already holds another prefix")
            plan.append((i, (h, parent, extra_key, blk)))
            parent = h
        for i, entry in plan:
            if i not in self.cache and entry[0] not in self.by_hash:
                self.cache[i] = entry
                self.by_hash[entry[0]] = i

    def cached_blocks(self) -> int:
        return len(self.by_hash)

    def alloc_sequence(self, seq_len: int, block_size: int) -> list:
        return self.alloc(blocks_needed(seq_len, block_size))

    def fork(self, ids) -> None:
        ids = list(ids)
        if any(i not in self.refs for i in ids):
            raise ValueError("forking a block that is not allocated")
        for i in ids:
            self.refs[i] += 1

    def free(self, ids) -> None:
        ids = list(ids)
        for i in set(ids):
            if ids.count(i) > self.refs.get(i, 0):
                raise ValueError("freeing a block that is not allocated")
        for i in ids:
            self.refs[i] -= 1
            if self.refs[i] == 0:
                del self.refs[i]
                self.free_list.append(i)

    def refcount(self, i: int) -> int:
        return self.refs.get(i, 0) if 0 <= i < self.num_blocks else -1

    def stats(self):
        return len(self.refs), len(self.free_list)

    def prepare_append(self, tables, seq_lens, block_size):
        """Make each sequence's append target writable; ``tables`` is a list
        of per-sequence block-id lists (updated in place, grown when the token
        opens a block).  Returns the (src, dst) block copies in order."""
        trial = copy.deepcopy(self)
        new_tables = [list(t) for t in tables]
        copies = []
        for t, L in zip(new_tables, seq_lens):
            if L <= 0:
                raise ValueError("sequence length must be positive")
            j, row = (L - 1) // block_size, (L - 1) % block_size
            if row == 0:                                  # the token opens a block
                new = trial.alloc(1)[0]
                if j < len(t):
                    t[j] = new
                else:
                    t.extend([-1] * (j - len(t)) + [new])
                continue
            if j >= len(t) or t[j] not in trial.refs:
                raise ValueError("writing into a block that is not allocated")
            old = t[j]
            if trial.refs[old] > 1:                       # shared: copy, then write
                new = trial.alloc(1)[0]
                trial.free([old])
                t[j] = new
                copies.append((old, new))
        self.__dict__.update(trial.__dict__)
        for t, nt in zip(tables, new_tables):
            t[:] = nt
        return copies


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64-bit: start at the offset basis 0xcbf29ce484222325; for
    every byte, xor it in, then multiply by the prime 0x100000001b3 mod 2^64."""
    h = 0xcbf29ce484222325
    for byte in data:
        h ^= byte
        h = (h * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return h


def block_hash(parent: int, tokens, extra_key: int = 0) -> int:
    """Hash of one full block (“让 Agent 跑得快”, §七: parent block's hash +
    the block's tokens + extra keys): FNV-1a 64 over the parent hash and the
    key (8 bytes each) and the token ids (4 bytes each, two's complement),
    little-endian."""
    data = parent.to_bytes(8, "little") + extra_key.to_bytes(8, "little")
    data += b"".join(int(t).to_bytes(4, "little", signed=True) for t in tokens)
    return fnv1a64(data)


def copy_blocks(k_cache, v_cache, pairs, k_scale=None, v_scale=None) -> None:
    """Block copy of copy-on-write (“让 Agent 跑得快”, §二): for each (src, dst)
    in order, block dst of both pools (and its scale rows) becomes block src."""
    for src, dst in pairs:
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]
        if k_scale is not None:
            k_scale[dst] = k_scale[src]
            v_scale[dst] = v_scale[src]


# --------------------------------------------------------------------------
# Slot mapping and append
# --------------------------------------------------------------------------

def token_slots(block_tables, positions, block_size, num_blocks, seq_idx=None):
    """slot = block_tables[s][p // bs] * bs + p % bs; -1 for p < 0 or a bad
    index.  Returns (slots int64, status)."""
    lib = _load()
    bt = _c(block_tables, np.int32)
    pos = _c(positions, np.int32)
    si = None if seq_idx is None else _c(seq_idx, np.int32)
    out = np.empty(pos.shape[0], np.int64)
    rc = lib.oracle_token_slots(_ptr(bt), bt.shape[1], _ptr(si), _ptr(pos),
                                pos.shape[0], block_size, num_blocks, _ptr(out))
    return out, rc


def append_bf16(k, v, k_cache, v_cache, slots):
    """Copy bf16 bits of k, v [n, Hkv, d] into the pools (in place)."""
    lib = _load()
    k, v, s = _c(k, np.uint16), _c(v, np.uint16), _c(slots, np.int64)
    nb, bs, hkv, d = k_cache.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    return lib.oracle_append_bf16(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(s), k.shape[0], nb, bs, hkv, d)


def append_int8(k, v, k_cache, v_cache, k_scale, v_scale, slots):
    """Store int8 codes of bf16 k, v under the slot's block scales."""
    lib = _load()
    k, v, s = _c(k, np.uint16), _c(v, np.uint16), _c(slots, np.int64)
    ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
    nb, bs, hkv, d = k_cache.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    return lib.oracle_append_int8(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(ks), _ptr(vs), _ptr(s), k.shape[0], nb,
                                  bs, hkv, d)


def quantize_int8(x: float, s: float) -> int:
    """fp32 clamp(round_half_even(x / s), -127, 127); NaN -> 0; s = 0 -> 1."""
    return _load().oracle_quantize_int8(float(x), float(s))


def append_fp8(k, v, k_cache, v_cache, k_scale, v_scale, slots):
    """Store E4M3 codes (uint8 pools) of bf16 k, v under the slot's block
    scales."""
    lib = _load()
    k, v, s = _c(k, np.uint16), _c(v, np.uint16), _c(slots, np.int64)
    ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
    nb, bs, hkv, d = k_cache.shape
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    return lib.oracle_append_fp8(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(ks), _ptr(vs), _ptr(s), k.shape[0], nb,
                                 bs, hkv, d)


def quantize_fp8(x: float, s: float) -> int:
    """E4M3 code of the fp32 quotient x / s: nearest finite value, ties to
    the even code, |.| > 448 -> 448, NaN -> 0x7F, s = 0 -> 1."""
    return _load().oracle_quantize_fp8(float(x), float(s))


def fp8_value(code: int) -> float:
    """Value of an E4M3 code (NaN for 0x7F / 0xFF)."""
    return _load().oracle_fp8_value(int(code))


def append_any(k, v, k_cache, v_cache, k_scale, v_scale, slots):
    """The append for the pool's dtype (uint16 bf16 bits, int8 codes, uint8
    E4M3 codes)."""
    if k_cache.dtype == np.int8:
        return append_int8(k, v, k_cache, v_cache, k_scale, v_scale, slots)
    if k_cache.dtype == np.uint8:
        return append_fp8(k, v, k_cache, v_cache, k_scale, v_scale, slots)
    return append_bf16(k, v, k_cache, v_cache, slots)


def workload_pools(wl, seqs=None, with_new_token=True):
    """The oracle's own K/V pools for a seeded workload ``wl`` (optionally
    only sequences ``seqs``): poisoned pools, the cached tokens appended
    through this module's slot mapping and append, then (by default) the
    step's new tokens at their positions.  Nothing comes from the CUDA path.
    Returns (k_cache, v_cache, k_scale, v_scale)."""
    s = wl.spec
    kc, vc = wl.poisoned_pool(), wl.poisoned_pool()
    ks = vs = None
    if s.kv_dtype != "bf16":
        ks, vs = wl.scales(seqs)
    for ch in wl.fill_chunks(seqs):
        slots, rc = token_slots(wl.block_tables, ch.positions, s.block_size, wl.num_blocks,
                                seq_idx=ch.seq_idx)
        assert rc == 0
        assert append_any(ch.k, ch.v, kc, vc, ks, vs, slots) == 0
    if with_new_token:
        seq, pos = wl.new_positions()
        slots, rc = token_slots(wl.block_tables, pos, s.block_size, wl.num_blocks, seq_idx=seq)
        assert rc == 0
        if seqs is not None:
            slots[~np.isin(seq, np.asarray(list(seqs)))] = -1
        assert append_any(wl.new_k, wl.new_v, kc, vc, ks, vs, slots) == 0
    return kc, vc, ks, vs


def _kv_kind(k_cache):
    """0 bf16 bits (uint16), 1 int8 codes, 2 E4M3 codes (uint8)."""
    kinds = {np.dtype(np.uint16): 0, np.dtype(np.int8): 1, np.dtype(np.uint8): 2}
    assert k_cache.dtype in kinds, k_cache.dtype
    return kinds[k_cache.dtype]


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, scale, *,
                    num_kv_heads=None, k_scale=None, v_scale=None, rows=None,
                    mode="three_pass", threads=1):
    """fp64 decode attention through the block table.

    q: bf16 bits [B, Hq, d]; k_cache / v_cache: bf16 bits (uint16), int8 or
    E4M3 codes (uint8) [NB, bs, Hkv, d]; block_tables int32 [B, MB]; seq_lens
    int32 [B].
    rows: optional int array [n, 2] of (b, h) to compute; default all, in
    b-major order.  Returns (out fp64 [n, d] or [B, Hq, d], status).
    """
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape
    kind = _kv_kind(k_cache)
    if kind:
        k_scale, v_scale = _c(k_scale, np.float32), _c(v_scale, np.float32)
    kc, vc = np.ascontiguousarray(k_cache), np.ascontiguousarray(v_cache)
    bt, sl = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    r = None if rows is None else _c(rows, np.int32).reshape(-1, 2)
    n = B * Hq if r is None else r.shape[0]
    out = np.zeros((n, d), np.float64)
    m = {"three_pass": 0, "online": 1}[mode]
    rc = lib.oracle_paged_attention(
        _ptr(out), _ptr(q), _ptr(kc), _ptr(vc),
        _ptr(k_scale) if kind else None, _ptr(v_scale) if kind else None,
        kind, _ptr(bt), bt.shape[1], _ptr(sl), B, Hq, hkv, d, nb, bs,
        float(scale), _ptr(r), n, m, int(threads))
    if r is None:
        out = out.reshape(B, Hq, d)
    return out, rc


def paged_attention_multi(q, k_cache, v_cache, block_tables, seq_lens, query_start, scale, *,
                          k_scale=None, v_scale=None, mode="three_pass", threads=1):
    """fp64 attention of multi-token queries: q bf16 bits [T, Hq, d], the
    query tokens of sequence b being rows query_start[b] .. query_start[b+1]-1,
    the last of its seq_lens[b] tokens, each attending causally up to its own
    position.  Returns (out fp64 [T, Hq, d], status)."""
    lib = _load()
    q = _c(q, np.uint16)
    T, Hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape
    kind = _kv_kind(k_cache)
    if kind:
        k_scale, v_scale = _c(k_scale, np.float32), _c(v_scale, np.float32)
    kc, vc = np.ascontiguousarray(k_cache), np.ascontiguousarray(v_cache)
    bt, sl = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    qs = _c(query_start, np.int32)
    B = sl.shape[0]
    assert qs.shape == (B + 1,)
    out = np.zeros((T, Hq, d), np.float64)
    m = {"three_pass": 0, "online": 1}[mode]
    rc = lib.oracle_paged_attention_multi(
        _ptr(out), _ptr(q), _ptr(kc), _ptr(vc),
        _ptr(k_scale) if kind else None, _ptr(v_scale) if kind else None,
        kind, _ptr(bt), bt.shape[1], _ptr(sl), _ptr(qs), B, T, Hq, hkv, d, nb, bs,
        float(scale), m, int(threads))
    return out, rc


def attention_partials(q, k_cache, v_cache, block_tables, seq_lens, scale, b, h,
                       part, *, k_scale=None, v_scale=None):
    """Per-partition (m_i, l_i) [np, 2] and unnormalised acc_i [np, d] of query
    row (b, h), partitions of ``part`` consecutive logical tokens."""
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    kind = _kv_kind(k_cache)
    if kind:
        k_scale, v_scale = _c(k_scale, np.float32), _c(v_scale, np.float32)
    kc, vc = np.ascontiguousarray(k_cache), np.ascontiguousarray(v_cache)
    bt, sl = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    npart = (int(sl[b]) + part - 1) // part
    ml = np.zeros((max(npart, 1), 2), np.float64)
    acc = np.zeros((max(npart, 1), d), np.float64)
    rc = lib.oracle_attention_partials(
        _ptr(ml), _ptr(acc), _ptr(q), _ptr(kc), _ptr(vc),
        _ptr(k_scale) if kind else None, _ptr(v_scale) if kind else None,
        kind, _ptr(bt), bt.shape[1], _ptr(sl), B, Hq, hkv, d, nb, bs,
        float(scale), int(b), int(h), int(part))
    if rc < 0:
        raise ValueError(f"oracle_attention_partials failed ({-rc})")
    return ml[:rc], acc[:rc]


def lse_merge(ml, acc):
    """o = sum_i exp(m_i - M) acc_i / sum_i exp(m_i - M) l_i, M = max m_i."""
    lib = _load()
    ml, acc = _c(ml, np.float64), _c(acc, np.float64)
    out = np.zeros(acc.shape[1], np.float64)
    lib.oracle_lse_merge(_ptr(ml), _ptr(acc), ml.shape[0], acc.shape[1], _ptr(out))
    return out


def bf16_bits_to_float(a) -> np.ndarray:
    """Widen bf16 bits (uint16) to float32 exactly."""
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)
