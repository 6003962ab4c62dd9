"""Multi-token query pins for the oracle, without a GPU (“让 Agent 跑得快：LLM
推理服务”, §六 投机解码: the target model scores the draft tokens in one
parallel pass; “LLM 推理优化技术全景”, SARATHI: 512-token prefill chunks
batched with decodes).

* Library routine: for every sequence, the oracle equals torch SDPA (CPU,
  fp64) on the contiguous K/V with the causal mask of the last n_b positions
  (query i sees positions 0 .. L_b - n_b + i).
* Invariant: query token i equals a one-token decode over the sequence cut
  at its position (bit-identical: the same fp64 arithmetic on the same
  gathered tokens).
* The online recurrence equals the three-pass form; bad offsets are flagged
  and their rows zeroed.
"""
import numpy as np
import pytest

import oracle
import workloads
from oracle_helpers import contiguous_kv, oracle_pool
from workloads import bf16_bits_to_f32

torch = pytest.importorskip("torch")


def multi(lens, qlens, hq=8, hkv=2, d=64, bs=16, kv="bf16", seed=21, prefix=0):
    return workloads.custom(batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                            block_size=bs, seq_lens=lens, kv_dtype=kv, seed=seed,
                            query_lens=qlens, shared_prefix_tokens=prefix)


def run_multi(wl, pools=None, **kw):
    kc, vc, ks, vs = pools or oracle_pool(wl)
    return oracle.paged_attention_multi(wl.q, kc, vc, wl.block_tables, wl.seq_lens,
                                        wl.query_start, wl.spec.scale, k_scale=ks, v_scale=vs, **kw)


def check_multi_against_sdpa(wl):
    import torch.nn.functional as F
    out, rc = run_multi(wl)
    assert rc == 0
    G = wl.spec.num_q_heads // wl.spec.num_kv_heads
    q = torch.from_numpy(bf16_bits_to_f32(wl.q).astype(np.float64))
    for b in range(wl.spec.batch):
        K, V = contiguous_kv(wl, b)
        L, n = int(wl.seq_lens[b]), int(wl.query_lens[b])
        a = int(wl.query_start[b])
        Kx = torch.from_numpy(K).repeat_interleave(G, dim=1).transpose(0, 1)      # [Hq, L, d]
        Vx = torch.from_numpy(V).repeat_interleave(G, dim=1).transpose(0, 1)
        pos = torch.arange(L - n, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos                                   # [n, L]
        ref = F.scaled_dot_product_attention(q[a:a + n].transpose(0, 1), Kx, Vx, attn_mask=mask,
                                             scale=wl.spec.scale)                # [Hq, n, d]
        np.testing.assert_allclose(out[a:a + n], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("geom", [dict(hq=8, hkv=2, d=64, bs=16), dict(hq=32, hkv=8, d=128, bs=16),
                                  dict(hq=16, hkv=2, d=128, bs=32), dict(hq=4, hkv=4, d=64, bs=32)],
                         ids=["g4d64", "g4d128", "g8bs32", "mha"])
def test_multi_matches_causal_sdpa(oracle_mod, geom):
    check_multi_against_sdpa(multi([1, 5, 17, 40, 100, 250], [1, 5, 3, 40, 7, 64], **geom))


def test_multi_with_shared_prefix_matches_causal_sdpa(oracle_mod):
    check_multi_against_sdpa(multi([40, 50, 70], [4, 18, 6], prefix=32, seed=4))


def test_multi_row_equals_decode_over_the_cut_sequence(oracle_mod):
    wl = multi([9, 33, 120, 300], [9, 5, 17, 2], hq=8, hkv=2, d=64, bs=16, seed=5)
    pools = oracle_pool(wl)
    got, rc = run_multi(wl, pools)
    assert rc == 0
    seq, pos = wl.new_positions()
    kc, vc, ks, vs = pools
    # one decode "sequence" per query token: same table, length pos + 1
    want, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables[seq], pos + 1, wl.spec.scale)
    assert rc == 0
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kv", ["int8", "fp8"])
def test_multi_8bit_row_equals_decode_over_the_cut_sequence(oracle_mod, kv):
    wl = multi([40, 70], [6, 33], hq=16, hkv=2, d=128, bs=32, kv=kv, seed=6)
    kc, vc, ks, vs = pools = oracle_pool(wl)
    got, rc = run_multi(wl, pools)
    assert rc == 0
    seq, pos = wl.new_positions()
    want, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables[seq], pos + 1, wl.spec.scale,
                                      k_scale=ks, v_scale=vs)
    assert rc == 0 and np.array_equal(got, want)


def test_multi_online_equals_three_pass(oracle_mod):
    wl = multi([64, 200], [20, 64], seed=7)
    pools = oracle_pool(wl)
    a, rc = run_multi(wl, pools)
    b, rc2 = run_multi(wl, pools, mode="online")
    assert rc == rc2 == 0
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-14)


def test_multi_bad_offsets_are_flagged_and_zeroed(oracle_mod):
    wl = multi([30, 40], [3, 4], seed=8)
    kc, vc, ks, vs = oracle_pool(wl)
    for qs in ([0, 3, 6], [1, 3, 7], [0, 5, 4]):           # wrong total, wrong start, decreasing
        out, rc = oracle.paged_attention_multi(wl.q, kc, vc, wl.block_tables, wl.seq_lens,
                                               np.asarray(qs, np.int32), wl.spec.scale)
        assert rc == oracle.INDEX
    too_many = np.array([0, 3, 7], np.int32)
    lens = wl.seq_lens.copy()
    lens[0] = 2                                            # 3 query tokens in a 2-token sequence
    out, rc = oracle.paged_attention_multi(wl.q, kc, vc, wl.block_tables, lens, too_many, wl.spec.scale)
    assert rc == oracle.INDEX and not out[:3].any() and out[3:].any()
