"""Prefix-cache (APC) pins, without a GPU (“让 Agent 跑得快：LLM 推理服务”, §七
前缀缓存: chained block hashes over parent hash + block tokens + extra keys;
hits take references; freed blocks stay matchable in the free queue).

* FNV-1a 64 (the hash this library chooses; the pages name none) against the
  test vectors its authors publish with the algorithm.
* The library's block hash equals the oracle's on random blocks and keys.
* The oracle's pool model and the C pool replay the hand-derived trace
  tests/golden/pool_apc.json.
* The C pool equals the model on long random traffic mixing prefix matches,
  registrations, forks, decode appends and frees.
* Planted mistakes in the model are caught.
"""
import inspect
import json
import os

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "pool_apc.json")))

# FNV-1a 64 test vectors published with the algorithm by its authors
# (Fowler, Noll, Vo): input bytes -> hash.
FNV_VECTORS = [(b"", 0xcbf29ce484222325), (b"a", 0xaf63dc4c8601ec8c),
               (b"ab", 0x089c4407b545986a), (b"abc", 0xe71fa2190541574b)]


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_97_gb300 as pkv
    from paged_kv_cache_97_gb300 import _build
    _build.build()
    pkv.load()
    return pkv


def test_fnv1a64_published_vectors():
    for data, want in FNV_VECTORS:
        assert oracle.fnv1a64(data) == want, data


def test_block_hash_equals_the_oracles(pkv):
    rng = np.random.default_rng(4)
    for _ in range(300):
        bs = int(rng.choice([1, 2, 16, 32]))
        toks = rng.integers(-2 ** 31, 2 ** 31, size=bs, dtype=np.int64).astype(np.int32)
        parent = int(rng.integers(0, 2 ** 63)) * 2 + int(rng.integers(0, 2))
        key = int(rng.integers(0, 2 ** 63))
        assert pkv.block_hash(parent, toks, key) == oracle.block_hash(parent, toks, key)


def replay(ops, nb, bs):
    for i, st in enumerate(GOLDEN["steps"]):
        op, want = st["op"], st.get("expect")
        got = ops(op, st)
        assert want is None or got == want, (i, op, got, want)


def model_ops(m, bs):
    def ops(op, st):
        if op == "match":
            return m.match_prefix(st["tokens"], bs, st["key"])
        if op == "alloc":
            return m.alloc(st["n"])
        if op == "register":
            m.register_prefix(st["ids"], st["tokens"], bs, st["key"])
        elif op == "cached":
            return m.cached_blocks()
        elif op == "stats":
            return list(m.stats())
        elif op == "refcounts":
            return [m.refcount(i) for i in range(m.num_blocks)]
        elif op == "free":
            m.free(st["ids"])
        return None
    return ops


def c_ops(p, nb):
    def ops(op, st):
        if op == "match":
            return p.match_prefix(st["tokens"], st["key"])
        if op == "alloc":
            return p.alloc(st["n"])
        if op == "register":
            p.register_prefix(st["ids"], st["tokens"], st["key"])
        elif op == "cached":
            return p.cached_blocks()
        elif op == "stats":
            return list(p.stats())
        elif op == "refcounts":
            return [p.refcount(i) for i in range(nb)]
        elif op == "free":
            p.free(st["ids"])
        return None
    return ops


def test_model_follows_apc_trace():
    nb, bs = GOLDEN["num_blocks"], GOLDEN["block_size"]
    replay(model_ops(oracle.BlockPoolModel(nb), bs), nb, bs)


def test_c_pool_follows_apc_trace(pkv):
    nb, bs = GOLDEN["num_blocks"], GOLDEN["block_size"]
    replay(c_ops(pkv.KVPool(nb, bs, 2, 64), nb), nb, bs)


def test_register_rejects_free_and_reassigned_blocks(pkv):
    p = pkv.KVPool(6, 2, 2, 64)
    ids = p.alloc(2)
    p.register_prefix(ids, [1, 2, 3, 4])
    with pytest.raises(pkv.KVError):
        p.register_prefix([ids[0], 5], [7, 7, 8, 8])          # 5 is free; nothing registered
    with pytest.raises(pkv.KVError):
        p.register_prefix([ids[1]], [5, 6])                    # holds [3, 4] under another chain
    assert p.cached_blocks() == 2


def test_c_pool_matches_model_on_random_cache_traffic(pkv):
    """Prompts drawn from a few shared system prompts plus private suffixes;
    each request matches, allocates the rest, registers, decodes a few
    tokens (prepare_append), may fork, and finishes."""
    rng = np.random.default_rng(11)
    nb, bs, MB = 96, 4, 24
    model = oracle.BlockPoolModel(nb)
    pool = pkv.KVPool(nb, bs, 2, 64)
    systems = [list(rng.integers(0, 50, size=int(rng.integers(4, 30)))) for _ in range(4)]
    live = []                                          # [tokens, table row]
    for it in range(1500):
        r = rng.random()
        if r < 0.35 or not live:
            toks = systems[int(rng.integers(len(systems)))] + \
                list(rng.integers(0, 50, size=int(rng.integers(1, 12))))
            key = int(rng.integers(0, 2))
            toks = toks[:MB * bs - 8]
            hit_m = model.match_prefix(toks, bs, key)
            hit_c = pool.match_prefix(toks, key)
            assert hit_c == hit_m, it
            need = oracle.blocks_needed(len(toks), bs) - len(hit_m)
            try:
                new_m = model.alloc(need)
            except MemoryError:
                with pytest.raises(pkv.KVError):
                    pool.alloc(need)
                model.free(hit_m)
                pool.free(hit_c)
                continue
            assert pool.alloc(need) == new_m
            ids = hit_m + new_m
            model.register_prefix(ids, toks, bs, key)
            pool.register_prefix(ids, toks, key)
            row = np.full(MB, -1, np.int32)
            row[:len(ids)] = ids
            live.append([toks, row, key])
        elif r < 0.5:                                  # a parallel sample forks
            toks, row, key = live[int(rng.integers(len(live)))]
            ids = [int(x) for x in row[:oracle.blocks_needed(len(toks), bs)]]
            model.fork(ids)
            pool.fork(ids)
            live.append([list(toks), row.copy(), key])
        elif r < 0.75:                                 # one decode step of a subset
            pick = [i for i in range(len(live)) if len(live[i][0]) < MB * bs and rng.random() < 0.5]
            if not pick:
                continue
            tables = np.stack([live[i][1] for i in pick])
            lens = np.asarray([len(live[i][0]) + 1 for i in pick], np.int32)
            t_m, t_c = tables.copy(), tables.copy()
            rows = [list(x) for x in t_m]
            try:
                cm = model.prepare_append(rows, lens, bs)
            except MemoryError:
                with pytest.raises(pkv.KVError):
                    pool.prepare_append(t_c, lens)
                continue
            cc = pool.prepare_append(t_c, lens)
            assert cc.tolist() == [list(c) for c in cm]
            assert (t_c == np.asarray(rows, np.int32)).all()
            for k, i in enumerate(pick):
                live[i][0] = live[i][0] + [int(rng.integers(0, 50))]
                live[i][1] = t_c[k].copy()
        else:                                          # a request finishes
            toks, row, key = live.pop(int(rng.integers(len(live))))
            ids = [int(x) for x in row[:oracle.blocks_needed(len(toks), bs)]]
            model.free(ids)
            pool.free(ids)
        assert pool.stats() == model.stats(), it
        assert pool.cached_blocks() == model.cached_blocks(), it
    assert [pool.refcount(i) for i in range(nb)] == [model.refcount(i) for i in range(nb)]


def _mutant_model(old, new):
    src = inspect.getsource(oracle.BlockPoolModel)
    assert src.count(old) == 1, "mutation site not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns["BlockPoolModel"]


MUTANTS = {
    "hash_without_parent": ("            h = block_hash(parent, blk, extra_key)\n            i = self.by_hash",
                            "            h = block_hash(0, blk, extra_key)\n            i = self.by_hash"),
    "no_eviction_on_reuse": ("                del self.by_hash[self.cache.pop(i)[0]]", "                pass"),
    "revive_stays_in_queue": ("                self.free_list.remove(i)\n", ""),
    "continue_after_miss": ("            if i is None or self.cache[i] != (h, parent, extra_key, blk):\n                break",
                            "            if i is None or self.cache[i] != (h, parent, extra_key, blk):\n                continue"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_model_mistake_is_caught(name):
    cls = _mutant_model(*MUTANTS[name])
    nb, bs = GOLDEN["num_blocks"], GOLDEN["block_size"]
    with pytest.raises((AssertionError, ValueError, KeyError)):
        replay(model_ops(cls(nb), bs), nb, bs)
