"""Copy-on-write on the GPU, through the C ABI (“让 Agent 跑得快：LLM 推理服务”,
§二 Copy-on-Write：Beam Search 的内存优化).

* pagedkv_copy_blocks is bit-exact against the oracle's block copy (bf16 and
  int8 pools with their scales); a bad id is skipped and flagged.
* A beam-search run: the library's pool decides sharing, copies and new
  blocks, the CUDA path copies, appends and attends (fused decode step); the
  oracle runs the same inputs with its own pool model, copy, append and
  attention.  Pools are compared bit for bit after every step, outputs within
  the attention tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_97_gb300 as pkv
import workloads
from gpu_helpers import bits_of, out_f64, to_dev_bf16
from oracle_helpers import OracleBeamRun

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-3), "int8": (3e-2, 3e-3)}


def _dev_pool(host):
    if host.dtype == np.int8:
        return torch.from_numpy(host.copy()).cuda()
    return to_dev_bf16(host)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("hkv,d,bs", [(8, 128, 16), (2, 64, 32)])
def test_copy_blocks_bit_exact(kv, hkv, d, bs):
    rng = np.random.default_rng(5)
    nb = 200
    shape = (nb, bs, hkv, d)
    if kv == "int8":
        kc = rng.integers(-127, 128, size=shape, dtype=np.int8)
        vc = rng.integers(-127, 128, size=shape, dtype=np.int8)
        ks = rng.random((nb, hkv), dtype=np.float32)
        vs = rng.random((nb, hkv), dtype=np.float32)
    else:
        kc = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
        vc = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
        ks = vs = None
    perm = rng.permutation(nb)
    pairs = [(int(perm[i]), int(perm[100 + i])) for i in range(60)]   # dsts never sources
    pairs.append((int(perm[70]), int(perm[70])))                      # src == dst: no-op
    bad = [(nb, int(perm[199])), (int(perm[198]), -1)]                # skipped and flagged
    dk, dv = _dev_pool(kc), _dev_pool(vc)
    dks = None if ks is None else torch.from_numpy(ks).cuda()
    dvs = None if vs is None else torch.from_numpy(vs).cuda()
    dp = torch.tensor(pairs + bad, dtype=torch.int32).cuda()
    pkv.get_status()
    pkv.copy_blocks(dk, dv, dp, dks, dvs)
    torch.cuda.synchronize()
    st, flags = pkv.get_status()
    assert flags == pkv.FLAG_BAD_BLOCK
    oracle.copy_blocks(kc, vc, pairs, ks, vs)
    assert (bits_of(dk) == kc).all() and (bits_of(dv) == vc).all()
    if ks is not None:
        assert np.array_equal(dks.cpu().numpy(), ks) and np.array_equal(dvs.cpu().numpy(), vs)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_beam_search_matches_oracle(kv):
    bs = 16 if kv == "bf16" else 32
    w = workloads.BeamWorkload(num_parents=4, beams=4, parent_lens=[37, 16, 300, 1100], steps=40,
                               num_q_heads=8, num_kv_heads=2, head_dim=128 if kv == "int8" else 64,
                               block_size=bs, num_blocks=400, max_blocks_per_seq=80, kv_dtype=kv)
    ref = OracleBeamRun(w)
    # GPU side: its own pool, tables and device pools
    pool = pkv.KVPool(w.num_blocks, bs, w.num_kv_heads, w.head_dim,
                      pkv.DTYPE_INT8 if kv == "int8" else pkv.DTYPE_BF16)
    kc, vc = _dev_pool(w.poisoned_pool()), _dev_pool(w.poisoned_pool())
    ks = torch.from_numpy(w.k_scale.copy()).cuda() if kv == "int8" else None
    vs = torch.from_numpy(w.v_scale.copy()).cuda() if kv == "int8" else None
    MB = w.max_blocks_per_seq
    tables = np.full((w.num_seqs, MB), -1, np.int32)
    for p, L in enumerate(w.parent_lens):
        ids = pool.alloc(oracle.blocks_needed(int(L), bs))
        tables[p * w.beams, :len(ids)] = ids
        bt = torch.from_numpy(tables[p * w.beams:p * w.beams + 1].copy()).cuda()
        pos = torch.arange(int(L), dtype=torch.int32).cuda()
        slots = torch.empty(int(L), dtype=torch.int64).cuda()
        pkv.token_slot_mapping(bt, pos, w.num_blocks, bs, slots,
                               seq_idx=torch.zeros(int(L), dtype=torch.int32).cuda())
        pkv.reshape_and_cache(to_dev_bf16(w.parent_k[p]), to_dev_bf16(w.parent_v[p]), kc, vc, slots,
                              ks, vs)
        for j in range(1, w.beams):
            pool.fork(ids)
            tables[p * w.beams + j] = tables[p * w.beams]
    n = w.num_seqs
    out = torch.empty((n, w.num_q_heads, w.head_dim), dtype=torch.bfloat16).cuda()
    max_len = int(w.seq_lens_at(w.steps - 1).max())
    ws = torch.empty(max(pkv.workspace_bytes(n, w.num_q_heads, w.head_dim, max_len, bs), 16),
                     dtype=torch.uint8).cuda()
    tol_max, tol_mean = TOL[kv]
    copies_seen = 0
    pkv.get_status()
    for step in range(w.steps):
        lens = w.seq_lens_at(step)
        pairs = pool.prepare_append(tables, lens)
        want_pairs = ref.advance()
        assert pairs.tolist() == [list(p) for p in want_pairs], step
        copies_seen += len(pairs)
        if len(pairs):
            pkv.copy_blocks(kc, vc, torch.from_numpy(pairs).cuda(), ks, vs)
        pkv.decode_step(out, to_dev_bf16(w.step_q[step]), to_dev_bf16(w.step_k[step]),
                        to_dev_bf16(w.step_v[step]), kc, vc, torch.from_numpy(tables.copy()).cuda(),
                        torch.from_numpy(lens).cuda(), int(lens.max()), w.scale, ws,
                        k_scale=ks, v_scale=vs)
        got = out_f64(out)
        st, flags = pkv.get_status()
        assert flags == 0, step
        assert (tables == ref.table_array()).all(), step
        assert (bits_of(kc) == ref.kc).all() and (bits_of(vc) == ref.vc).all(), step
        if kv == "int8":
            assert np.array_equal(ks.cpu().numpy(), ref.ks) and np.array_equal(vs.cpu().numpy(), ref.vs)
        want, rc = ref.attend()
        assert rc == 0
        err = np.abs(got - want)
        assert err.max() <= tol_max and err.mean() <= tol_mean, (step, err.max(), err.mean())
    assert copies_seen >= (w.beams - 1) * 3            # every parent with a partial block forked
