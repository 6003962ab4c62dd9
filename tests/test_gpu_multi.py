"""Multi-token queries on the GPU (paged_attention_multi through the C ABI)
against the oracle (“让 Agent 跑得快：LLM 推理服务”, §六 投机解码; “LLM 推理
优化技术全景”, SARATHI chunked prefill).

The step's tokens are appended with the general slot mapping and
reshape_and_cache (pools compared bit for bit with the oracle's), then
attended causally; outputs within max-abs 1e-2 / mean-abs 1e-3 of the fp64
oracle, on small cases covering both the one-partition path and the split
path with its merge, and on sampled sequences of the full-size workloads.
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
TOL = (1e-2, 1e-3)


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_97_gb300 import _build
    _build.build()
    oracle.build()
    torch.cuda.set_device(0)
    pkv.get_status()


def multi(lens, qlens, hq=8, hkv=2, d=64, bs=16, seed=31, prefix=0):
    return workloads.custom(batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                            block_size=bs, seq_lens=lens, seed=seed, query_lens=qlens,
                            shared_prefix_tokens=prefix)


def check(got, ref, what):
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    assert err.max() <= TOL[0] and err.mean() <= TOL[1], (what, err.max(), err.mean())


CASES = {
    "g4_d64_mixed": lambda: multi([1, 5, 17, 40, 100, 250], [1, 5, 3, 40, 7, 64]),
    "g4_d128_spec": lambda: multi([300, 777, 1024, 2050], [5, 5, 5, 5], hq=32, hkv=8, d=128, seed=32),
    "g8_d128_bs32": lambda: multi([33, 640, 1500], [9, 130, 1], hq=64, hkv=8, d=128, bs=32, seed=33),
    "mha_d64_bs32": lambda: multi([70, 600], [70, 16], hq=4, hkv=4, d=64, bs=32, seed=34),
    "g2_prefill_chunk": lambda: multi([3000, 40, 2000], [512, 1, 1], hq=4, hkv=2, d=64, seed=35),
    "zero_query_seq": lambda: multi([50, 60, 70], [4, 0, 2], seed=36),
    "shared_prefix": lambda: multi([48, 64, 100], [8, 16, 4], hq=32, hkv=8, d=128, prefix=32, seed=37),
}


@pytest.mark.parametrize("part", ["", "256", "2048"])
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
                                           wl.query_start, wl.spec.scale, threads=os.cpu_count())
    assert rc == 0
    check(got, ref, case)


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


def test_bad_sequence_is_flagged_and_zeroed():
    wl = multi([30, 40, 50], [3, 4, 5], seed=39)
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
    assert not out[3:7].any() and out[:3].any() and out[7:].any()
    bt = wl.block_tables.copy()
    bt[2, 1] = wl.num_blocks + 7                                  # a block past the pool
    g.seq_lens = torch.from_numpy(wl.seq_lens).cuda()
    g.block_tables = torch.from_numpy(bt).cuda()
    out = bits_of(g.attend_multi()).copy()
    st, flags = pkv.get_status()
    assert flags == pkv.FLAG_BAD_BLOCK
    assert not out[7:].any() and out[:7].any()


def test_multi_rejects_8bit_pools():
    wl = workloads.custom(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                          seq_lens=[20, 30], kv_dtype="int8", seed=40, query_lens=[2, 3])
    g = GpuStep(wl)
    with pytest.raises(pkv.KVError) as e:
        g.attend_multi()
    assert e.value.status == pkv.KV_ERR_NOT_IMPLEMENTED


def sub_problem(wl, seqs):
    """The oracle inputs restricted to sequences `seqs` (tables, lengths,
    their q rows and offsets); the pool keeps its physical ids."""
    seqs = list(seqs)
    rows = np.concatenate([np.arange(wl.query_start[b], wl.query_start[b + 1]) for b in seqs])
    qs = np.concatenate([[0], np.cumsum(wl.query_lens[seqs])]).astype(np.int32)
    return rows, wl.q[rows], wl.block_tables[seqs], wl.seq_lens[seqs], qs


@pytest.mark.parametrize("cfg", [7, 8])
def test_full_size_multi_workload_sampled_sequences(cfg):
    wl = workloads.make(cfg)
    g = GpuStep(wl)
    got = out_f64(g.multi_step())
    torch.cuda.synchronize()
    st, flags = pkv.get_status()
    assert flags == 0, hex(flags)
    L = wl.seq_lens
    rng = np.random.default_rng(cfg)
    seqs = sorted({0, int(np.argmax(L)), int(np.argmin(L)), int(rng.integers(len(L)))})
    kc, vc, _, _ = oracle_pool(wl, seqs=seqs)
    rows, q, bt, sl, qs = sub_problem(wl, seqs)
    ref, rc = oracle.paged_attention_multi(q, kc, vc, bt, sl, qs, wl.spec.scale, threads=os.cpu_count())
    assert rc == 0
    check(got[rows], ref, f"workload {cfg}")
