"""paged_attention_decode_noalloc: the decode entry point for callers that
cannot allocate device memory (a C host program with no device allocator of
its own, or an engine that reserves all of HBM up front).  Its split-K
partials live in a fixed 32 MiB scratch array inside the library instead of
a caller workspace.

Both entry points run the same kernels with the same partition choice on the
same inputs, so the output must be bit-identical to paged_attention_decode's
on each of two calls in a row (different batches and dtypes, so stale
scratch from the first call cannot pass for the second's); any difference is
a scratch bug.  Each output is also compared element by element with the
fp64 oracle at the attention tolerances (bf16 1e-2 / 1e-3, int8 3e-2 / 1e-3).
A shape whose partials exceed the scratch must be refused with a clear
message.  This file is named to be collected last; it builds and loads the
library itself so that it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_97_gb300 as pkv
import workloads
from gpu_helpers import GpuStep, out_f64
from oracle_helpers import oracle_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_97_gb300 import _build
    _build.build()
    pkv.load()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    pkv.get_status()


def batch(seed, lens, kv="bf16", hq=32, hkv=8, bs=16):
    return workloads.custom(batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                            block_size=bs, seq_lens=lens, kv_dtype=kv, seed=seed)


def test_noalloc_is_bit_identical_to_the_workspace_entry_point_on_two_calls():
    cases = [batch(101, [3, 257, 1000, 3001, 4096, 64]),                       # several partitions
             batch(202, [2048, 17, 900, 2600], kv="int8", hq=64, bs=32)]
    for wl in cases:
        g = GpuStep(wl)
        g.append()
        ref = g.attend().clone()
        assert pkv.partition_tokens(wl.spec.batch, wl.spec.num_kv_heads, g.max_seq_len,
                                    wl.spec.block_size) < g.max_seq_len, "case must use the scratch"
        out = torch.full_like(g.out, float("nan"))
        pkv.paged_attention_decode_noalloc(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.seq_lens,
                                           g.max_seq_len, wl.spec.scale, k_scale=g.k_scale,
                                           v_scale=g.v_scale)
        torch.cuda.synchronize()
        st, flags = pkv.get_status()
        assert st == pkv.KV_OK and flags == 0
        # same kernels, same partitions, same inputs: every bit equal
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        # and the answer is the oracle's
        kc, vc, ks, vs = oracle_pool(wl)
        want, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale,
                                          k_scale=ks, v_scale=vs)
        assert rc == 0
        err = np.abs(out_f64(out) - want)
        max_tol = 3e-2 if wl.spec.kv_dtype == "int8" else 1e-2
        assert err.max() <= max_tol and err.mean() <= 1e-3, (err.max(), err.mean())


def test_noalloc_rejects_shapes_beyond_the_scratch():
    # 128 sequences x 64 query heads x 128K tokens split into partitions need
    # more than 32 MiB of partials; the call must refuse before launching.
    lib = pkv.load()
    B, hq, hkv, d, L = 128, 64, 8, 128, 131072
    part = pkv.partition_tokens(B, hkv, L, 16)
    need = B * hq * (-(-L // part)) * (d + 2) * 4
    assert need > pkv.noalloc_scratch_bytes()
    P = 256  # never dereferenced: the size check comes first
    st = lib.paged_attention_decode_noalloc(P, P, P, P, None, None, P, L // 16, P, B, hq, hkv, d,
                                            1000, 16, L, 0.1, 0, None)
    assert st == pkv.KV_ERR_INVALID_ARG
    msg = lib.pagedkv_last_error().decode()
    assert "scratch" in msg and str(need) in msg

