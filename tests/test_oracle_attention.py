"""Pins of the oracle's attention (and, through it, its slot mapping, append
and block-table gather) against what the pages and mathematics fix:

* a library routine: torch's scaled_dot_product_attention in fp64 on the
  un-paged, contiguous K/V straight from the generator (GQA heads repeated);
* closed forms: one token gives o = v exactly; two tokens give the logistic
  form; q = 0 or identical keys give mean(V);
* brute force at 40 digits (mpmath) for 1..3 tokens, with no max subtraction;
* the online recurrence and a log-sum-exp merge of partition partials equal
  the three-pass softmax (“LLM 推理优化技术全景”, 在线 Softmax: the result is
  exact);
* placement freedom (“让 Agent 跑得快”, §五: any free block serves any
  request): permuting physical placement leaves the output bit-identical;
* shared prefix (same page, 共享前缀): shared blocks give the same bits as
  private copies;
* masked rows and table padding are never read.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from oracle_helpers import contiguous_kv, decode_slots, oracle_pool
from workloads import bf16_bits_to_f32


def small(lens, hq=8, hkv=2, d=64, bs=16, kv="bf16", nb=None, seed=7, prefix=0, mb=None):
    return workloads.custom(batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                            block_size=bs, seq_lens=lens, kv_dtype=kv, num_blocks=nb,
                            max_blocks_per_seq=mb, shared_prefix_tokens=prefix, seed=seed)


def run(wl, pools=None, **kw):
    kc, vc, ks, vs = pools or oracle_pool(wl)
    out, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale,
                                     k_scale=ks, v_scale=vs, **kw)
    return out, rc


# ---------------------------------------------------------------------------
# Library routine
# ---------------------------------------------------------------------------

def check_against_sdpa(wl, atol=1e-12):
    """Oracle on the paged pool vs torch SDPA (CPU, fp64) on contiguous K/V."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    out, rc = run(wl)
    assert rc == 0
    G = wl.spec.num_q_heads // wl.spec.num_kv_heads
    q = torch.from_numpy(bf16_bits_to_f32(wl.q).astype(np.float64))
    for b in range(wl.spec.batch):
        K, V = contiguous_kv(wl, b)
        assert K.shape[0] == wl.seq_lens[b]
        Kx = torch.from_numpy(K).repeat_interleave(G, dim=1).transpose(0, 1)  # [Hq, L, d]
        Vx = torch.from_numpy(V).repeat_interleave(G, dim=1).transpose(0, 1)
        ref = F.scaled_dot_product_attention(q[b][:, None, :], Kx, Vx, scale=wl.spec.scale)[:, 0, :]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=0, atol=atol)


@pytest.mark.parametrize("geom", [dict(hq=8, hkv=2, d=64, bs=16), dict(hq=32, hkv=8, d=128, bs=16),
                                  dict(hq=64, hkv=8, d=128, bs=32), dict(hq=4, hkv=4, d=64, bs=32)],
                         ids=["g4d64", "g4d128", "g8bs32", "mha"])
def test_oracle_matches_sdpa_on_contiguous_layout(oracle_mod, geom):
    lens = [1, 2, 3, 15, 16, 17, 31, 33, 100, 250]
    check_against_sdpa(small(lens, seed=11, **geom))


def test_oracle_matches_sdpa_shared_prefix(oracle_mod):
    check_against_sdpa(small([33, 40, 64, 65, 100], prefix=32, seed=5))


def check_int8_against_sdpa(wl):
    """int8 pools: the oracle equals SDPA on code * scale (gathered in numpy)."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    kc, vc, ks, vs = oracle_pool(wl)
    out, rc = run(wl, (kc, vc, ks, vs))
    assert rc == 0
    bs, G = wl.spec.block_size, wl.spec.num_q_heads // wl.spec.num_kv_heads
    q = torch.from_numpy(bf16_bits_to_f32(wl.q).astype(np.float64))
    for b in range(wl.spec.batch):
        t = np.arange(wl.seq_lens[b])
        blk = wl.block_tables[b, t // bs]
        K = kc[blk, t % bs].astype(np.float64) * ks[blk][:, :, None].astype(np.float64)
        V = vc[blk, t % bs].astype(np.float64) * vs[blk][:, :, None].astype(np.float64)
        Kx = torch.from_numpy(K).repeat_interleave(G, dim=1).transpose(0, 1)
        Vx = torch.from_numpy(V).repeat_interleave(G, dim=1).transpose(0, 1)
        ref = F.scaled_dot_product_attention(q[b][:, None, :], Kx, Vx, scale=wl.spec.scale)[:, 0, :]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=0, atol=1e-12)


def test_oracle_matches_sdpa_int8_dequantised(oracle_mod):
    check_int8_against_sdpa(small([1, 5, 32, 33, 70, 200], hq=16, hkv=2, d=128, bs=32, kv="int8", seed=3))


# ---------------------------------------------------------------------------
# Closed forms and brute force
# ---------------------------------------------------------------------------

def test_single_token_returns_v_exactly(oracle_mod):
    wl = small([1, 1, 1], hq=8, hkv=2, d=64)
    out, rc = run(wl)
    assert rc == 0
    v = bf16_bits_to_f32(wl.new_v).astype(np.float64)          # [B, Hkv, d]
    np.testing.assert_array_equal(out, np.repeat(v, 4, axis=1))


def test_two_tokens_logistic_form(oracle_mod):
    wl = small([2, 2], hq=4, hkv=1, d=64, seed=21)
    out, rc = run(wl)
    assert rc == 0
    q = bf16_bits_to_f32(wl.q).astype(np.float64)
    for b in range(2):
        K, V = contiguous_kv(wl, b)
        for h in range(4):
            s1, s2 = (wl.spec.scale * float(q[b, h] @ K[t, 0]) for t in (0, 1))
            w1 = 1.0 / (1.0 + math.exp(s2 - s1))
            w2 = 1.0 / (1.0 + math.exp(s1 - s2))
            np.testing.assert_allclose(out[b, h], w1 * V[0, 0] + w2 * V[1, 0], rtol=0, atol=1e-14)


def test_brute_force_high_precision(oracle_mod):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    wl = small([1, 2, 3, 3], hq=4, hkv=2, d=64, seed=99)
    out, rc = run(wl)
    assert rc == 0
    q = bf16_bits_to_f32(wl.q).astype(np.float64)
    for b in range(wl.spec.batch):
        K, V = contiguous_kv(wl, b)
        for h in range(4):
            hk = h // 2
            e = [mpmath.exp(mpmath.mpf(wl.spec.scale) * mpmath.fsum(mpmath.mpf(float(x)) * mpmath.mpf(float(y))
                                                                     for x, y in zip(q[b, h], K[t, hk])))
                 for t in range(K.shape[0])]
            Z = mpmath.fsum(e)
            ref = [float(mpmath.fsum(e[t] * mpmath.mpf(float(V[t, hk, i])) for t in range(K.shape[0])) / Z)
                   for i in range(64)]
            np.testing.assert_allclose(out[b, h], ref, rtol=0, atol=1e-14)


def test_zero_query_gives_mean_of_v(oracle_mod):
    wl = small([1, 7, 16, 45], hq=8, hkv=2, d=64, seed=4)
    wl.q[:] = 0
    out, rc = run(wl)
    assert rc == 0
    for b in range(wl.spec.batch):
        _, V = contiguous_kv(wl, b)
        np.testing.assert_allclose(out[b], np.repeat(V.mean(axis=0), 4, axis=0), rtol=0, atol=1e-14)


def test_identical_keys_give_mean_of_v(oracle_mod):
    wl = small([9, 40], hq=8, hkv=2, d=64, seed=8)
    kc, vc, ks, vs = oracle_pool(wl)
    for b in range(wl.spec.batch):
        for t in range(wl.seq_lens[b]):
            blk = wl.block_tables[b, t // 16]
            kc[blk, t % 16] = kc[wl.block_tables[0, 0], 0]
    out, rc = run(wl, (kc, vc, ks, vs))
    assert rc == 0
    for b in range(wl.spec.batch):
        _, V = contiguous_kv(wl, b)
        np.testing.assert_allclose(out[b], np.repeat(V.mean(axis=0), 4, axis=0), rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# Online recurrence and split-K merge
# ---------------------------------------------------------------------------

def check_online(bs):
    wl = small([1, 16, 17, 100, 333, 1000], hq=8, hkv=2, d=64, bs=bs, seed=13)
    ref, rc = run(wl)
    got, rc2 = run(wl, mode="online")
    assert rc == rc2 == 0
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("bs", [16, 32])
def test_online_equals_three_pass(oracle_mod, bs):
    check_online(bs)


def check_partials_merge(part):
    wl = small([1, 17, 100, 700], hq=8, hkv=2, d=64, seed=17)
    kc, vc, ks, vs = oracle_pool(wl)
    ref, _ = run(wl, (kc, vc, ks, vs))
    for b in range(wl.spec.batch):
        for h in (0, 5):
            ml, acc = oracle.attention_partials(wl.q, kc, vc, wl.block_tables, wl.seq_lens,
                                                wl.spec.scale, b, h, part)
            assert ml.shape[0] == -(-int(wl.seq_lens[b]) // part)
            np.testing.assert_allclose(oracle.lse_merge(ml, acc), ref[b, h], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("part", [16, 48, 64, 512, 4096])
def test_partials_merge_equals_full(oracle_mod, part):
    check_partials_merge(part)


# ---------------------------------------------------------------------------
# Placement, sharing, masking
# ---------------------------------------------------------------------------

def test_permuted_placement_is_bit_identical(oracle_mod):
    wl = small([5, 16, 60, 123], hq=8, hkv=2, d=64, seed=23, nb=40)
    kc, vc, ks, vs = oracle_pool(wl)
    ref, _ = run(wl, (kc, vc, ks, vs))
    perm = np.random.default_rng(0).permutation(wl.num_blocks)   # old id -> new id
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt = wl.block_tables.copy()
    used = bt >= 0
    bt[used] = perm[bt[used]]
    wl.block_tables = bt
    got, rc = run(wl, (kc2, vc2, ks, vs))
    assert rc == 0
    np.testing.assert_array_equal(got, ref)


def test_shared_prefix_equals_private_copies(oracle_mod):
    wl = small([33, 48, 90], hq=8, hkv=2, d=64, prefix=32, seed=31)
    kc, vc, ks, vs = oracle_pool(wl)
    ref, _ = run(wl, (kc, vc, ks, vs))
    # give every sequence past the first a private copy of the 2 prefix blocks
    extra = 2 * (wl.spec.batch - 1)
    kc2 = np.concatenate([kc, np.zeros((extra,) + kc.shape[1:], kc.dtype)])
    vc2 = np.concatenate([vc, np.zeros((extra,) + vc.shape[1:], vc.dtype)])
    bt = wl.block_tables.copy()
    nxt = wl.num_blocks
    for b in range(1, wl.spec.batch):
        for j in range(2):
            kc2[nxt], vc2[nxt] = kc[bt[b, j]], vc[bt[b, j]]
            bt[b, j] = nxt
            nxt += 1
    wl.block_tables, wl.num_blocks = bt, nxt
    got, rc = run(wl, (kc2, vc2, ks, vs))
    assert rc == 0
    np.testing.assert_array_equal(got, ref)


def test_poisoned_rows_and_padding_are_never_read(oracle_mod):
    wl = small([1, 17, 31, 64], hq=8, hkv=2, d=64, seed=41, nb=30, mb=8)
    kc, vc, ks, vs = oracle_pool(wl)       # unused rows / blocks hold NaN
    ref, rc = run(wl, (kc, vc, ks, vs))
    assert rc == 0 and np.isfinite(ref).all()
    clean_k = np.where(np.isnan(bf16_bits_to_f32(kc)), np.uint16(0), kc)
    clean_v = np.where(np.isnan(bf16_bits_to_f32(vc)), np.uint16(0), vc)
    got, _ = run(wl, (clean_k, clean_v, ks, vs))
    np.testing.assert_array_equal(got, ref)
    bt = wl.block_tables.copy()
    pad = bt < 0
    bt[pad] = np.random.default_rng(1).integers(-1000, 1000, size=int(pad.sum()))
    wl.block_tables = bt
    got2, rc2 = run(wl, (kc, vc, ks, vs))
    assert rc2 == 0
    np.testing.assert_array_equal(got2, ref)


def test_bad_indices_zero_the_row_and_report(oracle_mod):
    wl = small([10, 20, 30], hq=4, hkv=2, d=64, seed=2)
    kc, vc, ks, vs = oracle_pool(wl)
    ref, _ = run(wl, (kc, vc, ks, vs))
    wl.block_tables[1, 0] = wl.num_blocks          # out of range
    wl.seq_lens[2] = 0                              # empty
    out, rc = run(wl, (kc, vc, ks, vs))
    assert rc == oracle.INDEX
    assert not out[1].any() and not out[2].any()
    np.testing.assert_array_equal(out[0], ref[0])


def test_row_subset_matches_full(oracle_mod):
    wl = small([3, 70, 129], hq=8, hkv=2, d=64, seed=9)
    kc, vc, ks, vs = oracle_pool(wl)
    full, _ = run(wl, (kc, vc, ks, vs), threads=3)
    rows = np.array([[2, 7], [0, 0], [1, 3]], np.int32)
    sub, rc = run(wl, (kc, vc, ks, vs), rows=rows)
    assert rc == 0
    np.testing.assert_array_equal(sub, full[rows[:, 0], rows[:, 1]])
