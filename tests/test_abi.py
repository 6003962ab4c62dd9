"""The C ABI without a GPU: the library builds, loads and exports every
function include/pagedkv.h declares; the host-only calls (block pool, sizes,
argument checks) behave as the oracle's model says."""
import json
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_97_gb300 as pkv
    from paged_kv_cache_97_gb300 import _build
    _build.build()
    pkv.load()
    return pkv


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)) - {"defined"})


def test_every_declared_symbol_is_exported_and_bound(pkv):
    names = declared_functions()
    assert len(names) >= 14, names
    lib = pkv.load()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pagedkv.h but not exported"
    assert sorted(pkv.SIGNATURES) == names, "binding and header disagree"


def test_pool_follows_golden_trace(pkv):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "pool_fifo.json")))
    pool = pkv.KVPool(g["num_blocks"], g["block_size"], 2, 64)
    for st in g["steps"]:
        if st["op"] == "alloc_seq":
            n = oracle.blocks_needed(st["seq_len"], g["block_size"])
            if st["expect"] == "MemoryError":
                before = pool.stats()
                with pytest.raises(pkv.KVError) as e:
                    pool.alloc(n)
                assert e.value.status == pkv.KV_ERR_OUT_OF_BLOCKS
                assert pool.stats() == before
            else:
                assert pool.alloc(n) == st["expect"]
        elif st["op"] == "free":
            if st.get("expect") == "ValueError":
                with pytest.raises(pkv.KVError) as e:
                    pool.free(st["ids"])
                assert e.value.status == pkv.KV_ERR_INVALID_ARG
            else:
                pool.free(st["ids"])
        elif st["op"] == "stats":
            assert list(pool.stats()) == st["expect"]


def test_pool_matches_model_on_random_traffic(pkv):
    rng = np.random.default_rng(3)
    model = oracle.BlockPoolModel(97)
    pool = pkv.KVPool(97, 16, 8, 128)
    live = []
    for _ in range(3000):
        if live and rng.random() < 0.45:
            ids = live.pop(int(rng.integers(len(live))))
            model.free(ids)
            pool.free(ids)
        else:
            n = int(rng.integers(0, 9))
            try:
                want = model.alloc(n)
            except MemoryError:
                with pytest.raises(pkv.KVError):
                    pool.alloc(n)
                continue
            assert pool.alloc(n) == want
            live.append(want)
        assert pool.stats() == model.stats()


@pytest.mark.parametrize("bs,h,d,dt", [(16, 8, 128, 0), (32, 8, 128, 1), (16, 2, 64, 0), (32, 1, 64, 1)])
def test_block_bytes_follow_the_formula(pkv, bs, h, d, dt):
    pool = pkv.KVPool(10, bs, h, d, dt)
    elem = 1 if dt == pkv.DTYPE_INT8 else 2
    assert pool.block_bytes() == oracle.block_memory_bytes(bs, h, d, elem)
    assert pkv.pool_tensor_bytes(10, bs, h, d, dt) * 2 == 10 * oracle.block_memory_bytes(bs, h, d, elem)


def test_workspace_bound_covers_the_smallest_partition(pkv):
    lib = pkv.load()
    assert lib.pagedkv_workspace_bytes(4, 8, 64, 200, 16) == 0          # one partition always
    assert lib.pagedkv_workspace_bytes(8, 32, 128, 131072, 16) == 8 * 32 * 512 * 130 * 4


def test_host_checks_fail_before_touching_the_gpu(pkv):
    lib = pkv.load()
    P = 16  # any non-null, 16-byte aligned fake address: nothing is dereferenced
    st = lib.paged_attention_decode(P, P, P, P, None, None, P, 4, P, 2, 8, 2, 96, 10, 16, 100,
                                    0.1, 0, None, 0, None)
    assert st == pkv.KV_ERR_INVALID_ARG and b"head_dim" in lib.pagedkv_last_error()
    st = lib.paged_attention_decode(P, P, P, P, None, None, P, 4, P, 2, 8, 3, 64, 10, 16, 100,
                                    0.1, 0, None, 0, None)
    assert st == pkv.KV_ERR_INVALID_ARG
    st = lib.paged_attention_decode(P, P, P, P, None, None, P, 4, P, 2, 24, 2, 64, 10, 16, 100,
                                    0.1, 0, None, 0, None)
    assert st == pkv.KV_ERR_INVALID_ARG and b"at most 8" in lib.pagedkv_last_error()
    st = lib.pagedkv_decode_step(P, P, None, None, P, P, None, None, P, 4, P, 2, 8, 2, 64, 10, 16,
                                 100, 0.1, 0, P, 1 << 20, None)
    assert st == pkv.KV_ERR_INVALID_ARG and b"NULL k or v" in lib.pagedkv_last_error()
    st = lib.paged_attention_decode(P, P, P, P, P, P, P, 4, P, 2, 8, 2, 64, 10, 16, 100,
                                    0.1, 0, None, 0, None)
    assert st == pkv.KV_ERR_INVALID_ARG and b"NULL" in lib.pagedkv_last_error()   # bf16 + scales
    # the multi-token step: new rows are required, aligned, and checked first
    st = lib.pagedkv_multi_step(P, P, None, P, P, P, None, None, P, 4, P, P, 2, 6, 3, 8, 2, 64,
                                10, 16, 100, 0.1, 0, P, 1 << 20, None)
    assert st == pkv.KV_ERR_INVALID_ARG and b"NULL" in lib.pagedkv_last_error()
    st = lib.pagedkv_multi_step(P, P, P + 8, P, P, P, None, None, P, 4, P, P, 2, 6, 3, 8, 2, 64,
                                10, 16, 100, 0.1, 0, P, 1 << 20, None)
    assert st == pkv.KV_ERR_INVALID_ARG and b"aligned" in lib.pagedkv_last_error()
    st = lib.pagedkv_multi_step(P, P, P, P, P, P, None, None, P, 4, P, P, 2, 6, 3, 8, 2, 96,
                                10, 16, 100, 0.1, 0, P, 1 << 20, None)
    assert st == pkv.KV_ERR_INVALID_ARG and b"head_dim" in lib.pagedkv_last_error()
    st = lib.reshape_and_cache(P, P, P, P, None, None, P, 3, 10, 16, 2, 80, 0, None)
    assert st == pkv.KV_ERR_INVALID_ARG
    st = lib.reshape_and_cache(P + 8, P, P, P, None, None, P, 3, 10, 16, 2, 64, 0, None)
    assert st == pkv.KV_ERR_INVALID_ARG and b"aligned" in lib.pagedkv_last_error()
    assert lib.reshape_and_cache(None, None, None, None, None, None, None, 0, 10, 16, 2, 64, 0, None) == 0


def test_empty_inputs_return_ok_without_a_device(pkv):
    # Zero sequences, tokens or block pairs: every entry point checks its
    # sizes, then returns KV_OK with no launch.  This runs on a machine with
    # no GPU, where any CUDA call would fail, so it also shows that nothing
    # reaches the device.
    lib = pkv.load()
    assert lib.pagedkv_slot_mapping(None, 4, None, 0, 16, 10, None, None) == pkv.KV_OK
    assert lib.pagedkv_token_slot_mapping(None, 4, None, None, 0, 16, 10, None, None) == pkv.KV_OK
    assert lib.reshape_and_cache(None, None, None, None, None, None, None, 0, 10, 16, 2, 64, 0,
                                 None) == pkv.KV_OK
    assert lib.paged_attention_decode(None, None, None, None, None, None, None, 4, None, 0, 8, 2,
                                      64, 10, 16, 64, 0.125, 0, None, 0, None) == pkv.KV_OK
    assert lib.paged_attention_decode_noalloc(None, None, None, None, None, None, None, 4, None,
                                              0, 8, 2, 64, 10, 16, 64, 0.125, 0, None) == pkv.KV_OK
    assert lib.pagedkv_decode_step(None, None, None, None, None, None, None, None, None, 4, None,
                                   0, 8, 2, 64, 10, 16, 64, 0.125, 0, None, 0, None) == pkv.KV_OK
    assert lib.pagedkv_decode_step_prefix(None, None, None, None, None, None, None, None, None, 4,
                                          None, 0, 8, 2, 64, 10, 16, 64, 0.125, 0, None, 0, None,
                                          0, None) == pkv.KV_OK
    assert lib.paged_attention_multi(None, None, None, None, None, None, None, 4, None, None, 0, 0,
                                     1, 8, 2, 64, 10, 16, 64, 0.125, 0, None, 0, None) == pkv.KV_OK
    assert lib.pagedkv_multi_step(None, None, None, None, None, None, None, None, None, 4, None,
                                  None, 0, 0, 1, 8, 2, 64, 10, 16, 64, 0.125, 0, None, 0,
                                  None) == pkv.KV_OK
    assert lib.pagedkv_copy_blocks(None, None, None, None, None, 0, 10, 16, 2, 64, 0,
                                   None) == pkv.KV_OK
    assert lib.pagedkv_workspace_bytes(0, 8, 64, 64, 16) == 0
    assert lib.pagedkv_multi_workspace_bytes(0, 8, 64, 64, 16) == 0
    assert lib.pagedkv_prefix_workspace_bytes(0, 8, 64, 64, 16, 2) == 0
    # an empty batch still gets its sizes checked
    assert lib.paged_attention_decode_noalloc(None, None, None, None, None, None, None, 4, None,
                                              0, 8, 3, 64, 10, 16, 64, 0.125, 0,
                                              None) == pkv.KV_ERR_INVALID_ARG
    assert lib.paged_attention_decode_noalloc(None, None, None, None, None, None, None, 4, None,
                                              -1, 8, 2, 64, 10, 16, 64, 0.125, 0,
                                              None) == pkv.KV_ERR_INVALID_ARG


def test_noalloc_scratch_size_matches_the_header(pkv):
    text = open(HEADER).read()
    m = re.search(r"#define PAGEDKV_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m, "PAGEDKV_NOALLOC_SCRATCH_BYTES not found in the header"
    assert pkv.noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_noalloc_leaves_bad_shapes_to_the_decode_checks(pkv):
    # a shape paged_attention_decode rejects gets its message (before any
    # device call), not a scratch-size one
    lib = pkv.load()
    P = 256
    st = lib.paged_attention_decode_noalloc(P, P, P, P, None, None, P, 64, P, 4, 30, 8, 128,
                                            1000, 16, 1024, 0.1, 0, None)
    assert st == pkv.KV_ERR_INVALID_ARG
    assert "bad sizes" in lib.pagedkv_last_error().decode()
    st = lib.paged_attention_decode_noalloc(P, P, P, P, None, None, P, 64, P, 4, 32, 8, 96,
                                            1000, 16, 1024, 0.1, 0, None)
    assert st == pkv.KV_ERR_INVALID_ARG
    assert "head_dim" in lib.pagedkv_last_error().decode()


@pytest.mark.parametrize("pairs,ok", [
    ([], True),
    ([[3, 7], [4, 8], [3, 9]], True),              # one source copied twice: fine
    ([[5, 5], [1, 2]], True),                      # src == dst is a no-op
    ([[3, 7], [4, 7]], False),                     # a destination twice
    ([[3, 7], [7, 8]], False),                     # a destination is another pair's source
    ([[3, 7], [2, 3]], False),                     # (the other order)
    ([[3, 16]], False),                            # id past the pool
    ([[-1, 2]], False),
])
def test_block_pair_check(pkv, pairs, ok):
    if ok:
        pkv.check_block_pairs(np.array(pairs, np.int32).reshape(-1, 2), 16)
    else:
        with pytest.raises(pkv.KVError) as e:
            pkv.check_block_pairs(np.array(pairs, np.int32).reshape(-1, 2), 16)
        assert e.value.status == pkv.KV_ERR_INVALID_ARG


def test_prepare_append_copies_are_a_valid_batch(pkv):
    # forks of several sequences, then one step where every shared block is
    # written: the copy list passes the check (distinct fresh destinations)
    pool = pkv.KVPool(64, 16, 2, 64)
    ids = pool.alloc(3)
    tables = np.full((4, 8), -1, np.int32)
    for b in range(4):
        if b:
            pool.fork(ids)
        tables[b, :3] = ids
    lens = np.array([40, 40, 40, 40], np.int32)             # all write into block 2 (shared by 4)
    pairs = pool.prepare_append(tables, lens)
    assert len(pairs) == 3
    pkv.check_block_pairs(pairs, 64)
