"""Multi-token queries on the GPU (paged_attention_multi through the C ABI)
against the oracle (“让 Agent 跑得快：LLM 推理服务”, §六 投机解码; “LLM 推理
优化技术全景”, SARATHI chunked prefill).

The step's tokens are appended with the general slot mapping and
reshape_and_cache (pools compared bit for bit with the oracle's), then
attended causally; outputs within max-abs 1e-2 / mean-abs 1e-3 of the fp64
oracle (3e-2 / 1e-3 for 8-bit pools), on small cases covering the three kernels
(decode-kernel column groups for one group's query tokens, 16-column CTAs
for a few groups' on bf16 pools, the tcgen05 tensor-core kernel for many),
the one-partition path and the split path with its merge, and on
sampled sequences of the full-size workloads.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_97_gb300 as pkv
import workloads
from gpu_helpers import GpuStep, bits_of, out_f64
from oracle_helpers import oracle_pool

pytestmark = pytest.mark.gpu
TOL = {"bf16": (1e-2, 1e-3), "int8": (3e-2, 1e-3), "fp8": (3e-2, 1e-3)}


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_97_gb300 import _build
    _build.build()
    oracle.build()
    torch.cuda.set_device(0)
    pkv.get_status()


def multi(lens, qlens, hq=8, hkv=2, d=64, bs=16, seed=31, prefix=0, kv="bf16"):
    return workloads.custom(batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                            block_size=bs, seq_lens=lens, seed=seed, query_lens=qlens,
                            shared_prefix_tokens=prefix, kv_dtype=kv)


def check(got, ref, what, kv="bf16"):
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    assert err.max() <= TOL[kv][0] and err.mean() <= TOL[kv][1], (what, err.max(), err.mean())


CASES = {
    "g4_d64_mixed": lambda: multi([1, 5, 17, 40, 100, 250], [1, 5, 3, 40, 7, 64]),
    "g4_d128_spec": lambda: multi([300, 777, 1024, 2050], [5, 5, 5, 5], hq=32, hkv=8, d=128, seed=32),
    "g8_d128_bs32": lambda: multi([33, 640, 1500], [9, 130, 1], hq=64, hkv=8, d=128, bs=32, seed=33),
    "mha_d64_bs32": lambda: multi([70, 600], [70, 16], hq=4, hkv=4, d=64, bs=32, seed=34),
    "g2_prefill_chunk": lambda: multi([3000, 40, 2000], [512, 1, 1], hq=4, hkv=2, d=64, seed=35),
    "zero_query_seq": lambda: multi([50, 60, 70], [4, 0, 2], seed=36),
    "shared_prefix": lambda: multi([48, 64, 100], [8, 16, 4], hq=32, hkv=8, d=128, prefix=32, seed=37),
    # few query tokens: decode-kernel column groups (<= 4 groups of 8 / G tokens)
    "col_g4_mixed": lambda: multi([1, 5, 17, 40, 100, 2500], [1, 2, 8, 3, 7, 5], hq=32, hkv=8, d=128,
                                  seed=41),
    "col_g8_bs32": lambda: multi([33, 640, 1500], [4, 1, 3], hq=64, hkv=8, d=128, bs=32, seed=42),
    "col_mha_d64": lambda: multi([70, 600], [32, 9], hq=4, hkv=4, d=64, seed=43),
    "col_g2_bs32_d64": lambda: multi([300, 16, 1000], [16, 16, 5], hq=4, hkv=2, d=64, bs=32, seed=44),
    "col_int8_g8": lambda: multi([33, 700, 2049], [4, 2, 3], hq=64, hkv=8, d=128, bs=32, kv="int8",
                                 seed=45),
    "col_fp8_g4": lambda: multi([20, 900, 1600], [8, 5, 1], hq=32, hkv=8, d=128, bs=16, kv="fp8",
                                seed=46),
    # column groups only, one sequence past 8192 tokens: two of the longest
    # (8192-token) partitions and their merge
    "col_long_g4": lambda: multi([9000, 300, 2], [5, 3, 1], hq=32, hkv=8, d=128, seed=49),
    # one query head, 43 tokens: with 3 partitions the (m, l) region holds 258
    # floats, so the acc region is 16-byte aligned only by its rounding
    "odd_rows_mha": lambda: multi([300, 700, 37], [41, 1, 1], hq=1, hkv=1, d=64, seed=48),
    # long queries on 8-bit pools: the tensor-core kernel widens the codes to fp16
    "row_int8_g4_d64": lambda: multi([20, 300, 1500], [2, 9, 200], hq=8, hkv=2, d=64, kv="int8",
                                     seed=50),
    "row_fp8_g8_d128_bs32": lambda: multi([33, 700, 2600], [9, 130, 1], hq=64, hkv=8, d=128, bs=32,
                                          kv="fp8", seed=51),
    "row_int8_g4_prefill_chunk": lambda: multi([3000, 40, 2000], [512, 1, 1], hq=32, hkv=8, d=128,
                                               kv="int8", seed=52),
    "row_fp8_mha_d64_bs32": lambda: multi([70, 600], [70, 16], hq=4, hkv=4, d=64, bs=32, kv="fp8",
                                          seed=53),
    "row_int8_g2_d128_bs32": lambda: multi([129, 1000, 5], [129, 40, 5], hq=4, hkv=2, d=128, bs=32,
                                           kv="int8", seed=54),
    # tile-pair edges of the tensor-core kernel (rows = query tokens x G = 4):
    # exactly one tile (128 rows), one row into the second tile (132), exactly
    # one pair (256), one row into the next pair (260)
    "pair_edges_g4": lambda: multi([700, 900, 1100, 1300], [32, 33, 64, 65], hq=32, hkv=8, d=128,
                                   seed=55),
    "pair_edges_fp8_bs32": lambda: multi([300, 257, 400, 2200], [32, 33, 64, 65], hq=32, hkv=8,
                                         d=128, bs=32, kv="fp8", seed=56),
    # 16-column CTAs (bf16, more than one 8-column group's tokens): G = 3
    # leaves column 15 as padding (5 tokens x 3 heads); G = 6 puts 2 tokens in
    # a CTA and a sequence whose every token is a query (L = n = 2: the first
    # query sees key 0 alone); at G = 4, n = 8 fills two CTAs exactly, n = 9
    # is the first length for the tensor-core kernel, and L = 8 = n
    "m16_g3_d64": lambda: multi([7, 300, 1000, 33], [3, 8, 5, 6], hq=6, hkv=2, d=64, seed=57),
    "m16_g6_bs32": lambda: multi([2, 100, 2049], [2, 4, 3], hq=12, hkv=2, d=128, bs=32, seed=58),
    "m16_edges_g4": lambda: multi([8, 9, 513, 4100], [8, 9, 8, 3], hq=32, hkv=8, d=128, seed=59),
    # every sequence within 16 columns: one m-tile per CTA (Q in registers)
    "m16_one_tile_g4": lambda: multi([700, 33, 1500], [3, 4, 4], hq=32, hkv=8, d=128, seed=61),
    "m16_one_tile_g2_bs32": lambda: multi([300, 1000, 77], [5, 8, 6], hq=4, hkv=2, d=64, bs=32,
                                          seed=62),
    # uniform batches (every sequence max_query_len tokens: the decode
    # kernel's launch is left out); with 256-token partitions the new rows of
    # the first two sequences straddle a partition boundary
    "m16_uniform_cross": lambda: multi([258, 515, 40, 1030], [5, 5, 5, 5], hq=32, hkv=8, d=128,
                                       seed=64),
    "m16_uniform_one_tile": lambda: multi([130, 257, 600], [4, 4, 4], hq=32, hkv=8, d=128,
                                          seed=65),
    # more sequences than the in-kernel ranking takes (128): grid order
    "m16_unranked_130": lambda: multi([20 + (37 * i) % 181 for i in range(130)], [5] * 130,
                                      hq=8, hkv=2, d=64, seed=66),
    # few-query batches are taken longest first: equal lengths tie-break by index
    "m16_equal_lens": lambda: multi([300, 300, 40, 300, 40], [5, 3, 5, 4, 8], hq=32, hkv=8, d=128,
                                    seed=60),
}


@pytest.mark.parametrize("part", ["", "256", "2048", "8192"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_multi_matches_oracle(monkeypatch, case, part):
    if part:
        monkeypatch.setenv("PAGEDKV_PARTITION_TOKENS", part)
    wl = CASES[case]()
    g = GpuStep(wl)
    got = out_f64(g.multi_step())
    torch.cuda.synchronize()
    st, flags = pkv.get_status()
    assert flags == 0, hex(flags)
    kc, vc, ks, vs = oracle_pool(wl)
    np.testing.assert_array_equal(bits_of(g.k_cache), kc)      # the appended tokens, bit for bit
    np.testing.assert_array_equal(bits_of(g.v_cache), vc)
    ref, rc = oracle.paged_attention_multi(wl.q, kc, vc, wl.block_tables, wl.seq_lens,
                                           wl.query_start, wl.spec.scale, k_scale=ks, v_scale=vs,
                                           threads=os.cpu_count())
    assert rc == 0
    check(got, ref, case, wl.spec.kv_dtype)


@pytest.mark.parametrize("part", ["", "256"])
@pytest.mark.parametrize("case", ["g4_d128_spec", "m16_uniform_cross", "m16_uniform_one_tile",
                                  "col_g4_mixed", "g4_d64_mixed", "zero_query_seq",
                                  "m16_one_tile_g4", "col_int8_g8", "col_fp8_g4",
                                  "row_int8_g4_d64", "g2_prefill_chunk"])
def test_fused_multi_step_equals_three_calls(monkeypatch, case, part):
    """pagedkv_multi_step (the append, then the attention) leaves the pools
    and the output bit-identical to token slot mapping + reshape_and_cache +
    paged_attention_multi, on every kernel of the path (uniform few-query
    batches, whose decode launch is left out, and mixed ones) and on 8-bit
    pools."""
    if part:
        monkeypatch.setenv("PAGEDKV_PARTITION_TOKENS", part)
    wl = CASES[case]()
    fused, three = GpuStep(wl), GpuStep(wl)
    out_f = fused.multi_step().clone()
    out_u = three.multi_step_unfused().clone()
    torch.cuda.synchronize()
    st, flags = pkv.get_status()
    assert flags == 0, hex(flags)
    np.testing.assert_array_equal(bits_of(fused.k_cache), bits_of(three.k_cache))
    np.testing.assert_array_equal(bits_of(fused.v_cache), bits_of(three.v_cache))
    assert torch.equal(out_f.view(torch.int16), out_u.view(torch.int16))


def test_fused_multi_step_skips_a_sequence_with_bad_offsets():
    """A sequence with more queries than tokens appends nothing, is flagged
    and zeroed; the other sequences' rows and outputs are the unfused path's."""
    wl = multi([30, 40, 50], [3, 4, 5], seed=63)
    fused, three = GpuStep(wl), GpuStep(wl)
    lens = wl.seq_lens.copy()
    lens[1] = 3                                                   # 4 queries in 3 tokens
    for g in (fused, three):
        g.seq_lens = torch.from_numpy(lens).cuda()
    k_before = bits_of(fused.k_cache).copy()
    out_f = bits_of(fused.multi_step()).copy()
    torch.cuda.synchronize()
    st, flags = pkv.get_status()
    assert flags & pkv.FLAG_BAD_SEQ_LEN
    e0, e1 = int(wl.query_start[1]), int(wl.query_start[2])
    assert not out_f[e0:e1].any() and out_f[:e0].any() and out_f[e1:].any()
    # sequence 1's block rows are untouched; sequences 0 and 2 as three calls
    three.multi_step_unfused()
    torch.cuda.synchronize()
    pkv.get_status()
    kf, ku = bits_of(fused.k_cache), bits_of(three.k_cache)
    for b in (0, 2):
        for blk in wl.block_tables[b][: -(-int(lens[b]) // wl.spec.block_size)]:
            np.testing.assert_array_equal(kf[blk], ku[blk])
    for blk in wl.block_tables[1][: -(-int(wl.seq_lens[1]) // wl.spec.block_size)]:
        np.testing.assert_array_equal(kf[blk], k_before[blk])


def test_one_query_per_sequence_matches_decode():
    """n_b = 1 everywhere: the multi-token kernel and the decode kernel agree
    with the oracle on the same step."""
    wl = multi([1, 90, 300, 1290], [1, 1, 1, 1], hq=32, hkv=8, d=128, seed=38)
    g = GpuStep(wl)
    got_multi = out_f64(g.multi_step())
    got_dec = out_f64(g.attend())
    kc, vc, _, _ = oracle_pool(wl)
    ref, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale)
    assert rc == 0
    check(got_multi, ref, "multi")
    check(got_dec, ref, "decode")


@pytest.mark.parametrize("qlens", [[3, 4, 5], [3, 4, 40]], ids=["column_groups", "row_tiles"])
def test_bad_sequence_is_flagged_and_zeroed(qlens):
    wl = multi([30, 40, 50], qlens, seed=39)
    e = int(wl.query_start[2])
    g = GpuStep(wl)
    g.multi_step()
    torch.cuda.synchronize()
    pkv.get_status()
    lens = wl.seq_lens.copy()
    lens[1] = 3                                                   # 4 queries in 3 tokens
    g.seq_lens = torch.from_numpy(lens).cuda()
    out = bits_of(g.attend_multi()).copy()
    st, flags = pkv.get_status()
    assert flags & pkv.FLAG_BAD_SEQ_LEN
    assert not out[3:7].any() and out[:3].any() and out[e:].any()
    bt = wl.block_tables.copy()
    bt[2, 1] = wl.num_blocks + 7                                  # a block past the pool
    g.seq_lens = torch.from_numpy(wl.seq_lens).cuda()
    g.block_tables = torch.from_numpy(bt).cuda()
    out = bits_of(g.attend_multi()).copy()
    st, flags = pkv.get_status()
    assert flags == pkv.FLAG_BAD_BLOCK
    assert not out[e:].any() and out[:e].any()


def sub_problem(wl, seqs):
    """The oracle inputs restricted to sequences `seqs` (tables, lengths,
    their q rows and offsets); the pool keeps its physical ids."""
    seqs = list(seqs)
    rows = np.concatenate([np.arange(wl.query_start[b], wl.query_start[b + 1]) for b in seqs])
    qs = np.concatenate([[0], np.cumsum(wl.query_lens[seqs])]).astype(np.int32)
    return rows, wl.q[rows], wl.block_tables[seqs], wl.seq_lens[seqs], qs


@pytest.mark.parametrize("cfg,kv", [(7, "bf16"), (8, "bf16"), (8, "int8"), (8, "fp8")])
def test_full_size_multi_workload_sampled_sequences(cfg, kv):
    wl = workloads.make(cfg, kv_dtype=kv)
    g = GpuStep(wl)
    got = out_f64(g.multi_step())
    torch.cuda.synchronize()
    st, flags = pkv.get_status()
    assert flags == 0, hex(flags)
    L = wl.seq_lens
    rng = np.random.default_rng(cfg)
    seqs = sorted({0, int(np.argmax(L)), int(np.argmin(L)), int(rng.integers(len(L)))})
    kc, vc, ks, vs = oracle_pool(wl, seqs=seqs)
    rows, q, bt, sl, qs = sub_problem(wl, seqs)
    ref, rc = oracle.paged_attention_multi(q, kc, vc, bt, sl, qs, wl.spec.scale, k_scale=ks,
                                           v_scale=vs, threads=os.cpu_count())
    assert rc == 0
    check(got[rows], ref, f"workload {cfg}, {kv} pools", kv)


@pytest.mark.parametrize("scale", [-0.125, 0.0, 1.0], ids=["negative", "zero", "sharp"])
def test_multi_softmax_scale_values(scale):
    """Scales other than 1/sqrt(d), on both kernels (sequence 0 takes the
    tensor-core kernel, the others the column groups): a negative scale, a zero
    scale (equal weights over the visible keys) and a sharp one whose running
    maximum moves by more than 2^8 mid-row, so that O is rescaled in TMEM.
    Near-one-hot rows put outputs near a single V row (|v| up to about 4.5),
    where rounding P and the output to bf16 each cost up to 2^-9 relative: the
    bound is 1e-2 + 2^-8 |ref| there."""
    wl = multi([3000, 40, 700], [300, 1, 5], hq=8, hkv=2, d=64, seed=47)
    g = GpuStep(wl)
    g.multi_step()
    out = torch.empty_like(g.out_multi)
    pkv.paged_attention_multi(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens,
                              g.query_start, g.max_seq_len, int(wl.query_lens.max()), scale,
                              g.ws_multi)
    torch.cuda.synchronize()
    st, flags = pkv.get_status()
    assert flags == 0, hex(flags)
    got = out_f64(out)
    kc, vc, _, _ = oracle_pool(wl)
    ref, rc = oracle.paged_attention_multi(wl.q, kc, vc, wl.block_tables, wl.seq_lens,
                                           wl.query_start, scale, threads=os.cpu_count())
    assert rc == 0
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert (err <= 1e-2 + 2.0 ** -8 * np.abs(ref)).all(), (scale, err.max())
    assert err.mean() <= 1e-3, (scale, err.mean())


def test_partition_choice_follows_the_kernels_in_the_call(monkeypatch):
    """Column groups alone may take one partition of up to 8192 tokens (no
    merge launch); with a long query in the call the tensor-core kernel caps
    it at 2048; the override is honoured within those limits only."""
    monkeypatch.delenv("PAGEDKV_PARTITION_TOKENS", raising=False)
    # 64 sequences x 5 draft tokens, 32/8 heads, up to 4096 tokens: column groups only
    assert pkv.multi_partition_tokens(64, 320, 5, 32, 8, 4096) == 8192
    # the same batch with one 512-token prefill chunk: the tensor-core kernel joins
    assert pkv.multi_partition_tokens(64, 575, 512, 32, 8, 4096) == 2048
    monkeypatch.setenv("PAGEDKV_PARTITION_TOKENS", "4096")
    assert pkv.multi_partition_tokens(64, 320, 5, 32, 8, 4096) == 4096
    assert pkv.multi_partition_tokens(64, 575, 512, 32, 8, 4096) == 2048    # beyond its limit: ignored
    monkeypatch.setenv("PAGEDKV_PARTITION_TOKENS", "512")
    assert pkv.multi_partition_tokens(64, 575, 512, 32, 8, 4096) == 512
    assert pkv.multi_partition_tokens(0, 0, 5, 32, 8, 4096) == 0             # nothing to size
