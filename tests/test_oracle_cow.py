"""Copy-on-write pins, without a GPU (“让 Agent 跑得快：LLM 推理服务”, §二
Copy-on-Write：Beam Search 的内存优化; §五 共享前缀).

* The oracle's pool model and the library's C pool both replay the
  hand-derived trace tests/golden/pool_cow.json.
* The C pool equals the model on long random fork / append / free traffic.
* Beam pin: after forks, copies and appends chosen by the model, every
  sequence read back through its block table holds exactly its own tokens
  (parent prompt + its own decode tokens), and the oracle's paged attention
  over the shared pool is bit-identical to attention over a private, unshared
  copy of each sequence.  This ties the model's sharing decisions and the
  block copy to the plain un-paged definition.
* Planted mistakes in the model and the copy are caught by these pins.
"""
import inspect
import json
import os

import numpy as np
import pytest

import oracle
import workloads
from oracle_helpers import OracleBeamRun

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "pool_cow.json")))


# --------------------------------------------------------------------------
# Trace replay, for the model and for the C pool
# --------------------------------------------------------------------------

class _ModelAdapter:
    """The model behind the C pool's call shapes (fixed-width tables)."""

    out_of_blocks, invalid = MemoryError, ValueError

    def __init__(self, model_cls, nb, bs):
        self.m, self.bs = model_cls(nb), bs

    def alloc(self, n):
        return self.m.alloc(n)

    def fork(self, ids):
        self.m.fork(ids)

    def free(self, ids):
        self.m.free(ids)

    def stats(self):
        return self.m.stats()

    def refcount(self, i):
        return self.m.refcount(i)

    def prepare_append(self, tables, lens):
        rows = [list(r) for r in tables]
        copies = self.m.prepare_append(rows, list(lens), self.bs)
        tables[:] = np.asarray(rows, np.int32)
        return np.asarray(copies, np.int32).reshape(-1, 2)


class _CAdapter:
    def __init__(self, pkv, nb, bs):
        self.pkv, self.p = pkv, pkv.KVPool(nb, bs, 2, 64)
        self.out_of_blocks = self.invalid = pkv.KVError

    def __getattr__(self, name):
        return getattr(self.p, name)


def replay(pool, g, expect_status=None):
    nb, bs = g["num_blocks"], g["block_size"]
    for i, st in enumerate(g["steps"]):
        op, want = st["op"], st.get("expect")
        where = f"step {i} ({op})"
        if op == "alloc_seq":
            assert pool.alloc(oracle.blocks_needed(st["seq_len"], bs)) == want, where
        elif op == "fork":
            pool.fork(st["ids"])
        elif op == "free":
            if want == "ValueError":
                before = pool.stats(), [pool.refcount(j) for j in range(nb)]
                with pytest.raises(pool.invalid) as e:
                    pool.free(st["ids"])
                if expect_status:
                    assert e.value.status == expect_status["invalid"], where
                assert (pool.stats(), [pool.refcount(j) for j in range(nb)]) == before, where
            else:
                pool.free(st["ids"])
        elif op == "stats":
            assert list(pool.stats()) == want, where
        elif op == "refcounts":
            assert [pool.refcount(j) for j in range(nb)] == want, where
        elif op == "prepare_append":
            tables = np.asarray(st["tables"], np.int32)
            if want == "MemoryError":
                before = pool.stats(), [pool.refcount(j) for j in range(nb)]
                t0 = tables.copy()
                with pytest.raises(pool.out_of_blocks) as e:
                    pool.prepare_append(tables, st["seq_lens"])
                if expect_status:
                    assert e.value.status == expect_status["oob"], where
                assert (pool.stats(), [pool.refcount(j) for j in range(nb)]) == before, where
                assert (tables == t0).all(), where
            else:
                copies = pool.prepare_append(tables, st["seq_lens"])
                assert np.asarray(copies).reshape(-1, 2).tolist() == want["copies"], where
                assert tables.tolist() == want["tables"], where
        else:
            raise AssertionError(op)


def test_model_follows_cow_trace():
    replay(_ModelAdapter(oracle.BlockPoolModel, GOLDEN["num_blocks"], GOLDEN["block_size"]), GOLDEN)


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_97_gb300 as pkv
    from paged_kv_cache_97_gb300 import _build
    _build.build()
    pkv.load()
    return pkv


def test_c_pool_follows_cow_trace(pkv):
    replay(_CAdapter(pkv, GOLDEN["num_blocks"], GOLDEN["block_size"]), GOLDEN,
           expect_status={"invalid": pkv.KV_ERR_INVALID_ARG, "oob": pkv.KV_ERR_OUT_OF_BLOCKS})


def test_c_pool_rejects_bad_appends_without_change(pkv):
    p = pkv.KVPool(8, 4, 2, 64)
    ids = p.alloc(2)
    before = p.stats()
    for tables, lens in (([[ids[0], ids[1], -1]], [0]),            # empty sequence
                         ([[ids[0], ids[1], -1]], [13]),           # past the table
                         ([[ids[0], 5, -1]], [7])):                # block 5 is free
        t = np.asarray(tables, np.int32)
        t0 = t.copy()
        with pytest.raises(pkv.KVError) as e:
            p.prepare_append(t, lens)
        assert e.value.status == pkv.KV_ERR_INVALID_ARG
        assert (t == t0).all() and p.stats() == before
    with pytest.raises(pkv.KVError):
        p.fork([ids[0], 7])                                        # 7 is free: nothing changes
    assert p.refcount(ids[0]) == 1 and p.refcount(-1) == -1 and p.refcount(8) == -1


def test_c_pool_matches_model_on_random_fork_traffic(pkv):
    rng = np.random.default_rng(97)
    nb, bs, MB = 61, 4, 12
    model = _ModelAdapter(oracle.BlockPoolModel, nb, bs)
    pool = _CAdapter(pkv, nb, bs)
    seqs = []                                   # [table row (np int32 [MB]), length]
    for it in range(4000):
        r = rng.random()
        if r < 0.15 or not seqs:                # a new prompt
            L = int(rng.integers(1, 4 * bs))
            n = oracle.blocks_needed(L, bs)
            try:
                want = model.alloc(n)
            except MemoryError:
                with pytest.raises(pkv.KVError):
                    pool.alloc(n)
                continue
            assert pool.alloc(n) == want
            row = np.full(MB, -1, np.int32)
            row[:n] = want
            seqs.append([row, L])
        elif r < 0.30:                          # fork a sequence
            row, L = seqs[int(rng.integers(len(seqs)))]
            ids = [int(x) for x in row[:oracle.blocks_needed(L, bs)]]
            model.fork(ids)
            pool.fork(ids)
            seqs.append([row.copy(), L])
        elif r < 0.45:                          # a sequence finishes
            row, L = seqs.pop(int(rng.integers(len(seqs))))
            ids = [int(x) for x in row[:oracle.blocks_needed(L, bs)]]
            model.free(ids)
            pool.free(ids)
        else:                                   # a decode step of a random subset
            pick = [i for i in range(len(seqs)) if seqs[i][1] < MB * bs and rng.random() < 0.5]
            if not pick:
                continue
            tables = np.stack([seqs[i][0] for i in pick])
            lens = np.asarray([seqs[i][1] + 1 for i in pick], np.int32)
            t_model, t_c = tables.copy(), tables.copy()
            try:
                want = model.prepare_append(t_model, lens)
            except MemoryError:
                with pytest.raises(pkv.KVError) as e:
                    pool.prepare_append(t_c, lens)
                assert e.value.status == pkv.KV_ERR_OUT_OF_BLOCKS
                assert (t_c == tables).all()
                continue
            got = pool.prepare_append(t_c, lens)
            assert got.tolist() == want.tolist(), it
            assert (t_c == t_model).all(), it
            for k, i in enumerate(pick):
                seqs[i] = [t_c[k].copy(), int(lens[k])]
        assert pool.stats() == model.stats(), it
        if it % 50 == 0:
            assert [pool.refcount(j) for j in range(nb)] == [model.refcount(j) for j in range(nb)]
    # every reference the live sequences hold is counted exactly once
    held = np.zeros(nb, int)
    for row, L in seqs:
        for x in row[:oracle.blocks_needed(L, bs)]:
            held[x] += 1
    assert held.tolist() == [model.refcount(j) for j in range(nb)]


# --------------------------------------------------------------------------
# Beam pin: shared pool == private copies
# --------------------------------------------------------------------------

def beam_workload(kv="bf16", seed=workloads.SEED_BASE + 97):
    return workloads.BeamWorkload(num_parents=3, beams=4, parent_lens=[37, 16, 50], steps=21,
                                  num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                                  num_blocks=64, max_blocks_per_seq=6, kv_dtype=kv, seed=seed)


def private_attention(w, step):
    """Oracle attention with every sequence in private blocks of its own,
    filled with its dense tokens (nothing shared, nothing copied)."""
    n, MB, bs = w.num_seqs, w.max_blocks_per_seq, w.block_size
    shape = (n * MB, bs, w.num_kv_heads, w.head_dim)
    kc, vc = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    bt = np.arange(n * MB, dtype=np.int32).reshape(n, MB)
    for s in range(n):
        k, v = w.dense_tokens(s, step)
        slots, rc = oracle.token_slots(bt[s:s + 1], np.arange(len(k), dtype=np.int32), bs, n * MB,
                                       seq_idx=np.zeros(len(k), np.int32))
        assert rc == 0
        assert oracle.append_bf16(k, v, kc, vc, slots) == 0
    return oracle.paged_attention(w.step_q[step], kc, vc, bt, w.seq_lens_at(step), w.scale)


def check_beam_pin(run):
    w = run.w
    saw_copy = False
    for step in range(w.steps):
        copies = run.advance()
        saw_copy |= bool(copies)
        lens = w.seq_lens_at(step)
        for s in range(w.num_seqs):                     # read back through the table
            L, t = int(lens[s]), run.tables[s]
            k, v = w.dense_tokens(s, step)
            pos = np.arange(L)
            blk = t[pos // w.block_size]
            assert (run.kc[blk, pos % w.block_size] == k).all(), (step, s, "K")
            assert (run.vc[blk, pos % w.block_size] == v).all(), (step, s, "V")
        got, rc = run.attend()
        assert rc == 0
        want, rc = private_attention(w, step)
        assert rc == 0
        assert np.array_equal(got, want), step
    assert saw_copy


def test_beam_run_equals_private_copies():
    w = beam_workload()
    run = OracleBeamRun(w)
    check_beam_pin(run)
    # sharing saves memory: the pool holds fewer blocks than private copies would
    private = sum(oracle.blocks_needed(int(L), w.block_size) for L in w.seq_lens_at(w.steps - 1))
    used, _ = run.pool.stats()
    assert used < private


def test_int8_copy_carries_the_scales():
    """An int8 beam's copied block keeps its source's scales: a sequence's
    dequantised tokens after a copy equal the parent's before it."""
    w = beam_workload("int8")
    run = OracleBeamRun(w)
    bs = w.block_size
    before = {}
    for s in range(0, w.num_seqs, w.beams):            # parents' dequantised prompts
        L, t = int(w.parent_lens[s // w.beams]), run.tables[s]
        pos = np.arange(L)
        blk = t[pos // bs]
        before[s] = (run.kc[blk, pos % bs] * run.ks[blk][:, :, None].astype(np.float64),
                     run.vc[blk, pos % bs] * run.vs[blk][:, :, None].astype(np.float64))
    copies = run.advance()
    assert copies
    for s in range(w.num_seqs):
        p0 = (s // w.beams) * w.beams
        L, t = int(w.parent_lens[s // w.beams]), run.tables[s]
        pos = np.arange(L)
        blk = t[pos // bs]
        dk = run.kc[blk, pos % bs] * run.ks[blk][:, :, None].astype(np.float64)
        dv = run.vc[blk, pos % bs] * run.vs[blk][:, :, None].astype(np.float64)
        assert np.array_equal(dk, before[p0][0]) and np.array_equal(dv, before[p0][1]), s


# --------------------------------------------------------------------------
# Planted mistakes (in the oracle, on the CPU)
# --------------------------------------------------------------------------

def _mutant_model(old, new):
    src = inspect.getsource(oracle.BlockPoolModel)
    assert src.count(old) == 1, "mutation site not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns["BlockPoolModel"]


MODEL_MUTANTS = {
    "copies_private_blocks": ("if trial.refs[old] > 1:", "if trial.refs[old] >= 1:"),
    "never_copies": ("if trial.refs[old] > 1:", "if trial.refs[old] > 10 ** 6:"),
    "keeps_old_reference": ("                trial.free([old])\n", ""),
    "fork_without_reference": ("        for i in ids:\n            self.refs[i] += 1\n",
                               "        for i in ids:\n            pass\n"),
    "free_returns_shared_block": ("            if self.refs[i] == 0:", "            if self.refs[i] <= 1:"),
}


def _trace_rejects(model_cls):
    try:
        replay(_ModelAdapter(model_cls, GOLDEN["num_blocks"], GOLDEN["block_size"]), GOLDEN)
    except (AssertionError, ValueError, MemoryError, KeyError, pytest.fail.Exception):
        return True
    return False


def _beam_rejects(model_cls=None, copy_fn=None):
    w = beam_workload()
    saved = oracle.copy_blocks
    try:
        if copy_fn is not None:
            oracle.copy_blocks = copy_fn
        run = OracleBeamRun(w, None if model_cls is None else model_cls(w.num_blocks))
        check_beam_pin(run)
    except (AssertionError, ValueError, MemoryError, KeyError):
        return True
    finally:
        oracle.copy_blocks = saved
    return False


@pytest.mark.parametrize("name", sorted(MODEL_MUTANTS))
def test_planted_model_mistake_is_caught(name):
    cls = _mutant_model(*MODEL_MUTANTS[name])
    assert _trace_rejects(cls) or _beam_rejects(cls), name


def _copy_k_only(kc, vc, pairs, ks=None, vs=None):
    for src, dst in pairs:
        kc[dst] = kc[src]


def _copy_reversed(kc, vc, pairs, ks=None, vs=None):
    for src, dst in pairs:
        kc[src], vc[src] = kc[dst], vc[dst]


@pytest.mark.parametrize("fn", [_copy_k_only, _copy_reversed])
def test_planted_copy_mistake_is_caught(fn):
    assert _beam_rejects(copy_fn=fn)
