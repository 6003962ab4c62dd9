"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars: slot mapping and appends bit-exact (whole pools compared bit for bit,
poison included); attention max-abs <= 1e-2 and mean-abs <= 1e-3 for bf16
pools, max-abs <= 3e-2 and mean-abs <= 1e-3 for int8 and FP8 E4M3 pools (the
oracle runs on the dequantised stored codes, so quantisation error is not
counted).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_97_gb300 as pkv
import workloads
from gpu_helpers import GpuStep, bits_of, out_f64
from oracle_helpers import decode_slots, oracle_pool

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-3), "int8": (3e-2, 1e-3), "fp8": (3e-2, 1e-3)}


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_97_gb300 import _build
    _build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    pkv.get_status()


def check_status(expect_flags=0):
    st, flags = pkv.get_status()
    assert flags == expect_flags, f"device status flags 0x{flags:x}, expected 0x{expect_flags:x}"


def assert_close(got, ref, kv_dtype, what=""):
    max_tol, mean_tol = TOL[kv_dtype]
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert err.max() <= max_tol, f"{what}: max-abs {err.max():.3e} > {max_tol}"
    assert err.mean() <= mean_tol, f"{what}: mean-abs {err.mean():.3e} > {mean_tol}"
    return err.max(), err.mean()


def small(lens, hq=8, hkv=2, d=64, bs=16, kv="bf16", nb=None, seed=7, prefix=0, mb=None):
    return workloads.custom(batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                            block_size=bs, seq_lens=lens, kv_dtype=kv, num_blocks=nb,
                            max_blocks_per_seq=mb, shared_prefix_tokens=prefix, seed=seed)


CASES = {
    "tiny_b4_g4_d64": lambda: workloads.make(1),
    "ragged_g4_d128": lambda: small([1, 2, 15, 16, 17, 255, 256, 257, 1000, 3001], hq=32, hkv=8, d=128, seed=1),
    "g8_int8_bs32": lambda: small([1, 31, 32, 33, 511, 700, 2049], hq=64, hkv=8, d=128, bs=32, kv="int8", seed=2),
    "g1_mha_d64": lambda: small([5, 77, 300, 1290], hq=4, hkv=4, d=64, seed=3),
    "g2_bs32_d64": lambda: small([3, 64, 500, 999], hq=4, hkv=2, d=64, bs=32, seed=4),
    "g8_bf16_d128": lambda: small([17, 600, 1500], hq=16, hkv=2, d=128, seed=5),
    "int8_d64_bs16": lambda: small([1, 90, 300, 777], hq=8, hkv=2, d=64, bs=16, kv="int8", seed=6),
    "shared_prefix": lambda: small([33, 48, 300, 700], hq=32, hkv=8, d=128, prefix=32, seed=8),
    "g8_fp8_bs32": lambda: small([1, 31, 32, 33, 511, 700, 2049], hq=64, hkv=8, d=128, bs=32, kv="fp8", seed=12),
    "fp8_d64_bs16": lambda: small([1, 90, 300, 777], hq=8, hkv=2, d=64, bs=16, kv="fp8", seed=13),
    "fp8_g4_d128_bs16": lambda: small([2, 17, 1000, 2500], hq=32, hkv=8, d=128, bs=16, kv="fp8", seed=14),
}


# ---------------------------------------------------------------------------
# Slot mapping and append: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", ["tiny_b4_g4_d64", "g8_int8_bs32", "int8_d64_bs16", "shared_prefix", "g2_bs32_d64",
                                  "g8_fp8_bs32", "fp8_d64_bs16"])
def test_append_and_slots_bit_exact(case):
    wl = CASES[case]()
    g = GpuStep(wl)
    g.append()
    torch.cuda.synchronize()
    check_status()
    want_slots, rc = decode_slots(wl)
    assert rc == 0
    np.testing.assert_array_equal(g.slots.cpu().numpy(), want_slots)
    kc, vc, _, _ = oracle_pool(wl)
    np.testing.assert_array_equal(bits_of(g.k_cache), kc)
    np.testing.assert_array_equal(bits_of(g.v_cache), vc)


def test_int8_append_rounding_is_the_oracles():
    """Values at and near rounding ties: device codes equal the oracle's."""
    rng = np.random.default_rng(0)
    n, H, d, bs, NB = 64, 2, 128, 32, 4
    scale = np.float32(0.0234375)
    ties = (np.arange(-128, 128) + 0.5).astype(np.float32) * scale  # exact ties in fp32
    x = np.concatenate([ties, rng.standard_normal(n * H * d - ties.size).astype(np.float32) * 3])
    bits = workloads.to_bf16_bits(x).reshape(n, H, d)
    ks = np.full((NB, H), scale, np.float32)
    ks[1, 0] = 0.0                                                    # zero scale reads as 1
    slots = rng.permutation(NB * bs)[:n].astype(np.int64)
    kc = np.zeros((NB, bs, H, d), np.int8)
    vc = np.zeros_like(kc)
    assert oracle.append_int8(bits, bits, kc, vc, ks, ks, slots) == 0
    from gpu_helpers import to_dev_bf16
    dk = torch.zeros((NB, bs, H, d), dtype=torch.int8, device="cuda")
    dv = torch.zeros_like(dk)
    t = to_dev_bf16(bits)
    s = torch.from_numpy(ks).cuda()
    pkv.reshape_and_cache(t, t, dk, dv, torch.from_numpy(slots).cuda(), s, s)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dk.cpu().numpy(), kc)
    np.testing.assert_array_equal(dv.cpu().numpy(), vc)


def test_fp8_append_rounding_is_the_oracles():
    """E4M3 codes at and near every rounding tie, in the subnormal range and
    past the saturation point: device codes equal the oracle's; NaN inputs
    give the NaN pattern on both sides."""
    rng = np.random.default_rng(1)
    n, H, d, bs, NB = 64, 2, 128, 32, 4
    scale = np.float32(2.0 ** -5)                                     # x / scale exact
    vals = np.array([oracle.fp8_value(c) for c in range(0x7F)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)            # ties, bf16-exact
    special = np.array([448.0, 460.0, 464.0, 500.0, 1e4, 2.0 ** -10, 3 * 2.0 ** -11, 0.0],
                       np.float32)
    x = np.concatenate([mids, -mids, special, -special]) * scale
    x = np.concatenate([x, rng.standard_normal(n * H * d - x.size - 2).astype(np.float32) * 0.1,
                        np.array([np.nan, -np.nan], np.float32)])
    bits = workloads.to_bf16_bits(x).reshape(n, H, d)
    ks = np.full((NB, H), scale, np.float32)
    ks[1, 0] = 0.0                                                    # zero scale reads as 1
    slots = rng.permutation(NB * bs)[:n].astype(np.int64)
    kc = np.zeros((NB, bs, H, d), np.uint8)
    vc = np.zeros_like(kc)
    assert oracle.append_fp8(bits, bits, kc, vc, ks, ks, slots) == 0
    from gpu_helpers import dev_pool, to_dev_bf16
    dk, dv = dev_pool(np.zeros_like(kc)), dev_pool(np.zeros_like(kc))
    t = to_dev_bf16(bits)
    s = torch.from_numpy(ks).cuda()
    pkv.reshape_and_cache(t, t, dk, dv, torch.from_numpy(slots).cuda(), s, s)
    torch.cuda.synchronize()
    got_k, got_v = bits_of(dk), bits_of(dv)
    nan = (kc & 0x7F) == 0x7F
    assert nan.sum() == 2 and ((got_k[nan] & 0x7F) == 0x7F).all()
    np.testing.assert_array_equal(got_k[~nan], kc[~nan])
    np.testing.assert_array_equal(got_v[~nan], vc[~nan])


# ---------------------------------------------------------------------------
# Attention against the oracle (small, every row)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", sorted(CASES))
def test_attention_matches_oracle(case):
    wl = CASES[case]()
    g = GpuStep(wl)
    got = out_f64(g.step())
    torch.cuda.synchronize()
    check_status()
    kc, vc, ks, vs = oracle_pool(wl)
    ref, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale,
                                     k_scale=ks, v_scale=vs, threads=os.cpu_count())
    assert rc == 0
    assert_close(got, ref, wl.spec.kv_dtype, case)


def test_repeated_steps_are_deterministic():
    wl = CASES["ragged_g4_d128"]()
    g = GpuStep(wl)
    a = bits_of(g.step()).copy()
    b = bits_of(g.step())
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("part", ["256", "512", "2048"])
def test_partition_size_does_not_change_the_answer(monkeypatch, part):
    wl = CASES["ragged_g4_d128"]()
    kc, vc, ks, vs = oracle_pool(wl)
    ref, _ = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale,
                                    threads=os.cpu_count())
    monkeypatch.setenv("PAGEDKV_PARTITION_TOKENS", part)
    g = GpuStep(wl)
    assert pkv.partition_tokens(wl.spec.batch, wl.spec.num_kv_heads, g.max_seq_len, 16) == int(part)
    assert_close(out_f64(g.step()), ref, "bf16", f"partition {part}")
    assert_close(out_f64(g.fused_step()), ref, "bf16", f"partition {part}, fused")
    check_status()


def test_odd_partial_count_keeps_the_workspace_aligned(monkeypatch):
    """3 sequences x 1 query head x 3 partitions: 18 floats of (m, l), so the
    acc region after it is 16-byte aligned only because the (m, l) region is
    rounded up; the merge reads it with 16-byte loads."""
    wl = small([300, 700, 37], hq=1, hkv=1, d=64, seed=15)
    monkeypatch.setenv("PAGEDKV_PARTITION_TOKENS", "256")
    g = GpuStep(wl)
    got = out_f64(g.step())
    torch.cuda.synchronize()
    check_status()
    kc, vc, _, _ = oracle_pool(wl)
    ref, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale,
                                     threads=os.cpu_count())
    assert rc == 0
    assert_close(got, ref, "bf16", "odd partial count")


@pytest.mark.parametrize("case", ["tiny_b4_g4_d64", "ragged_g4_d128", "g8_int8_bs32", "shared_prefix", "int8_d64_bs16",
                                  "g8_fp8_bs32"])
def test_fused_step_equals_separate_calls(case):
    """pagedkv_decode_step (append inside the attention kernel) leaves the same
    pools, bit for bit, and the same output as slot mapping + append +
    attention as three calls."""
    wl = CASES[case]()
    a = GpuStep(wl)
    out_a = bits_of(a.step()).copy()
    b = GpuStep(wl)
    out_b = bits_of(b.fused_step())
    check_status()
    np.testing.assert_array_equal(bits_of(b.k_cache), bits_of(a.k_cache))
    np.testing.assert_array_equal(bits_of(b.v_cache), bits_of(a.v_cache))
    np.testing.assert_array_equal(out_b, out_a)


@pytest.mark.parametrize("case", ["tiny_b4_g4_d64", "ragged_g4_d128", "g8_int8_bs32", "fp8_d64_bs16"])
def test_decode_step_replays_from_a_cuda_graph(case):
    """The fused step captured once in a CUDA graph (decode + PDL merge) and
    replayed gives the eager step's output bit for bit; replaying re-appends
    the same token, so the pools stay bit-identical too."""
    wl = CASES[case]()
    eager = GpuStep(wl)
    want = bits_of(eager.fused_step()).copy()
    g = GpuStep(wl)
    g.fused_step()                       # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    g.out.zero_()
    with torch.cuda.graph(graph):
        g.fused_step()
    for _ in range(2):
        g.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits_of(g.out), want)
    np.testing.assert_array_equal(bits_of(g.k_cache), bits_of(eager.k_cache))
    np.testing.assert_array_equal(bits_of(g.v_cache), bits_of(eager.v_cache))
    check_status()


# ---------------------------------------------------------------------------
# Shared prefix (one dense pass per KV head over the shared blocks)
# ---------------------------------------------------------------------------

PREFIX_CASES = {
    "g4_d128_bs16": lambda: small([33, 48, 49, 300, 1000, 2100], hq=32, hkv=8, d=128, prefix=32, seed=31),
    "g8_d128_bs32": lambda: small([65, 90, 700, 1500], hq=64, hkv=8, d=128, bs=32, prefix=64, seed=32),
    "g4_d64_bs16_long_prefix": lambda: small([600, 601, 640, 1200, 700, 900, 650, 3000, 610, 800,
                                              999, 1001, 608, 2048, 1800, 777, 650],
                                             hq=8, hkv=2, d=64, prefix=592, seed=33),
    "g1_d128": lambda: small([17, 40, 333], hq=4, hkv=4, d=128, prefix=16, seed=34),
    # prefixes past one 2048-token prefix partial: three partials of 1408
    # tokens (and a 16-row tile: three of four softmax warps hold padding)
    "g4_d128_bs16_prefix_4224": lambda: small([4225, 4300, 5000, 6500], hq=32, hkv=8, d=128,
                                              prefix=4224, seed=35),
    # two partials of 1152 tokens over 65 blocks of 32, G = 8
    "g8_d64_bs32_prefix_2080": lambda: small([2081, 2100, 3000], hq=16, hkv=2, d=64, bs=32,
                                             prefix=2080, seed=36),
    # 8-bit pools: the prefix product widens the codes to fp16
    "int8_g4_d128_bs16": lambda: small([33, 48, 49, 300, 1000, 2100], hq=32, hkv=8, d=128, prefix=32,
                                       kv="int8", seed=37),
    "fp8_g4_d128_bs16": lambda: small([33, 48, 49, 300, 1000, 2100], hq=32, hkv=8, d=128, prefix=32,
                                      kv="fp8", seed=38),
    "int8_g8_d64_bs32_prefix_2080": lambda: small([2081, 2100, 3000], hq=16, hkv=2, d=64, bs=32,
                                                  prefix=2080, kv="int8", seed=39),
    "fp8_g2_d64_bs16_long_prefix": lambda: small([600, 601, 640, 1200, 3000, 610], hq=4, hkv=2, d=64,
                                                 prefix=592, kv="fp8", seed=40),
    "fp8_g1_d128_bs32": lambda: small([33, 40, 333], hq=4, hkv=4, d=128, bs=32, prefix=32, kv="fp8",
                                      seed=41),
    # prefix rows = batch x G at the tensor-core kernel's tile-pair edges:
    # 32 x 4 = 128 (one tile), 33 x 4 = 132 (one row into the second), 65 x 4 = 260
    "pair_edge_128_rows": lambda: small([40 + 9 * i for i in range(32)], hq=32, hkv=8, d=128,
                                        prefix=32, seed=42),
    "pair_edge_132_rows": lambda: small([40 + 9 * i for i in range(33)], hq=32, hkv=8, d=128,
                                        prefix=32, seed=43),
    "pair_edge_260_rows_int8": lambda: small([70 + 5 * i for i in range(65)], hq=16, hkv=4, d=64,
                                             bs=32, prefix=64, kv="int8", seed=44),
}


@pytest.mark.parametrize("case", sorted(PREFIX_CASES))
def test_prefix_step_matches_oracle(case):
    wl = PREFIX_CASES[case]()
    g = GpuStep(wl)
    got = out_f64(g.prefix_step())
    torch.cuda.synchronize()
    check_status()
    kc, vc, ks, vs = oracle_pool(wl)
    np.testing.assert_array_equal(bits_of(g.k_cache), kc)          # the append, bit for bit
    np.testing.assert_array_equal(bits_of(g.v_cache), vc)
    ref, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale,
                                     k_scale=ks, v_scale=vs, threads=os.cpu_count())
    assert rc == 0
    assert_close(got, ref, wl.spec.kv_dtype, case)
    plain = out_f64(GpuStep(wl).fused_step())
    assert_close(got, plain, wl.spec.kv_dtype, case + " vs plain step")


def test_prefix_attend_only_and_repeat():
    wl = PREFIX_CASES["g4_d128_bs16"]()
    g = GpuStep(wl)
    first = bits_of(g.prefix_step()).copy()
    again = bits_of(g.prefix_step(append=False))        # token already appended: same answer
    np.testing.assert_array_equal(first, again)


def test_prefix_mismatch_is_flagged_and_zeroed():
    wl = PREFIX_CASES["g4_d128_bs16"]()
    g = GpuStep(wl)
    g.prefix_step()
    bt = wl.block_tables.copy()
    bt[2, 1] = bt[2, 5] if bt[2, 5] >= 0 else wl.num_blocks - 1   # sequence 2 leaves the prefix
    g.block_tables = torch.from_numpy(bt).cuda()
    out = bits_of(g.prefix_step(append=False))
    st, flags = pkv.get_status()
    assert flags == pkv.FLAG_BAD_BLOCK
    assert not out[2].any() and out[0].any() and out[3].any()


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
def test_full_size_shared_prefix_workload_sampled_rows(kv):
    """256 sequences behind an 800-token shared prefix on bf16, int8 and E4M3
    pools, through the shared-prefix path."""
    wl = workloads.make(4, kv_dtype=kv)
    g = GpuStep(wl)
    got = out_f64(g.prefix_step())
    torch.cuda.synchronize()
    check_status()
    seqs, rows = sample_rows(wl)
    kc, vc, ks, vs = oracle_pool(wl, seqs=seqs)
    ref, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale,
                                     k_scale=ks, v_scale=vs, rows=rows, threads=os.cpu_count())
    assert rc == 0
    assert_close(got[rows[:, 0], rows[:, 1]], ref, kv,
                 f"256 sequences behind an 800-token prefix, {kv} pools, shared-prefix path")


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

def test_single_token_returns_v_bit_exact():
    for kv in ("bf16",):
        wl = small([1] * 6, hq=32, hkv=8, d=128, kv=kv, seed=10)
        g = GpuStep(wl)
        out = bits_of(g.step())
        want = np.repeat(wl.new_v, 4, axis=1)
        np.testing.assert_array_equal(out, want)


def test_permuted_placement_is_bit_identical():
    wl = small([40, 257, 1000, 2222], hq=32, hkv=8, d=128, seed=12)
    a = bits_of(GpuStep(wl).step()).copy()
    perm = np.random.default_rng(1).permutation(wl.num_blocks).astype(np.int32)
    bt = wl.block_tables.copy()
    used = bt >= 0
    bt[used] = perm[bt[used]]
    wl.block_tables = bt
    b = bits_of(GpuStep(wl).step())
    np.testing.assert_array_equal(a, b)


def test_shared_prefix_equals_private_copies_bit_exact():
    wl = small([40, 64, 300, 1000], hq=32, hkv=8, d=128, prefix=32, seed=13)
    a = bits_of(GpuStep(wl).step()).copy()
    g = GpuStep(wl)
    # private copies of the 2 prefix blocks for every sequence but the first
    extra = 2 * (wl.spec.batch - 1)
    nb = wl.num_blocks
    k2 = torch.cat([g.k_cache, g.k_cache[:extra].clone()])
    v2 = torch.cat([g.v_cache, g.v_cache[:extra].clone()])
    bt = wl.block_tables.copy()
    nxt = nb
    for b in range(1, wl.spec.batch):
        for j in range(2):
            k2[nxt], v2[nxt] = g.k_cache[bt[b, j]], g.v_cache[bt[b, j]]
            bt[b, j] = nxt
            nxt += 1
    wl.block_tables, wl.num_blocks = bt, nxt
    g.k_cache, g.v_cache = k2.contiguous(), v2.contiguous()
    g.block_tables = torch.from_numpy(bt).cuda()
    b2 = bits_of(g.step())
    np.testing.assert_array_equal(a, b2)


def test_table_padding_and_poison_are_never_read():
    wl = small([1, 17, 300, 900], hq=32, hkv=8, d=128, seed=14, mb=64)
    g = GpuStep(wl)
    a = bits_of(g.step()).copy()
    bt = wl.block_tables.copy()
    pad = bt < 0
    bt[pad] = np.random.default_rng(2).integers(-5000, 5000, size=int(pad.sum()))
    g.block_tables = torch.from_numpy(bt).cuda()
    b = bits_of(g.attend())
    np.testing.assert_array_equal(a, b)
    check_status()


# ---------------------------------------------------------------------------
# Device-side index faults: flagged, zeroed, never a GPU fault
# ---------------------------------------------------------------------------

def test_bad_block_id_and_length_zero_the_row_and_flag():
    wl = small([100, 600, 700, 50], hq=8, hkv=2, d=64, seed=15)
    g = GpuStep(wl)
    good = bits_of(g.step()).copy()
    bt = wl.block_tables.copy()
    bt[1, 3] = wl.num_blocks + 7            # inside sequence 1's range
    sl = wl.seq_lens.copy()
    sl[2] = 0
    g.block_tables = torch.from_numpy(bt).cuda()
    g.seq_lens = torch.from_numpy(sl).cuda()
    out = bits_of(g.attend(max_seq_len=700))
    st, flags = pkv.get_status()
    assert st == pkv.KV_ERR_DEVICE_INDEX
    assert flags == pkv.FLAG_BAD_BLOCK | pkv.FLAG_BAD_SEQ_LEN
    assert not out[1].any() and not out[2].any()
    # Other rows keep their values; not their exact bits, since a changed
    # batch moves the balanced split between workers (and so the order in
    # which a sequence's partials combine).
    from workloads import bf16_bits_to_f32
    for b in (0, 3):
        np.testing.assert_allclose(bf16_bits_to_f32(out[b]), bf16_bits_to_f32(good[b]), rtol=0, atol=1e-2)


def test_length_past_the_hint_is_flagged():
    wl = small([100, 600], hq=8, hkv=2, d=64, seed=16)
    g = GpuStep(wl)
    g.step()
    out = bits_of(g.attend(max_seq_len=300))
    st, flags = pkv.get_status()
    assert flags == pkv.FLAG_BAD_SEQ_LEN and not out[1].any()


def test_bad_slot_is_flagged_and_skipped():
    wl = small([10, 20], hq=8, hkv=2, d=64, seed=17)
    g = GpuStep(wl)
    before = bits_of(g.k_cache).copy()
    bad = torch.tensor([wl.num_blocks * 16, -1], dtype=torch.int64, device="cuda")
    pkv.reshape_and_cache(g.new_k, g.new_v, g.k_cache, g.v_cache, bad)
    st, flags = pkv.get_status()
    assert flags == pkv.FLAG_BAD_SLOT
    np.testing.assert_array_equal(bits_of(g.k_cache), before)


# ---------------------------------------------------------------------------
# Full-size workloads: sampled rows against the oracle
# ---------------------------------------------------------------------------

def sample_rows(wl, n_seqs=3, rng_seed=0):
    """The longest and shortest sequences plus a random one; all query heads
    of each (covers every KV head and both ends of the length range)."""
    L = wl.seq_lens
    rng = np.random.default_rng(rng_seed)
    seqs = sorted({int(np.argmax(L)), int(np.argmin(L)), int(rng.integers(len(L)))})[:n_seqs]
    rows = np.array([(b, h) for b in seqs for h in range(wl.spec.num_q_heads)], np.int32)
    return seqs, rows


@pytest.mark.parametrize("cfg", [2, 3, 4, 5, 6])
def test_full_size_config_sampled_rows(cfg):
    wl = workloads.make(cfg)
    g = GpuStep(wl)
    got = out_f64(g.step())
    torch.cuda.synchronize()
    check_status()
    assert np.isfinite(got).all()
    seqs, rows = sample_rows(wl)
    kc, vc, ks, vs = oracle_pool(wl, seqs=seqs)
    ref, rc = oracle.paged_attention(wl.q, kc, vc, wl.block_tables, wl.seq_lens, wl.spec.scale,
                                     k_scale=ks, v_scale=vs, rows=rows, threads=os.cpu_count())
    assert rc == 0
    assert_close(got[rows[:, 0], rows[:, 1]], ref, wl.spec.kv_dtype, f"config {cfg}")
    # the appended rows of the sampled sequences are the oracle's, bit for bit
    slots, _ = decode_slots(wl)
    for b in seqs:
        blk, row = divmod(int(slots[b]), wl.spec.block_size)
        np.testing.assert_array_equal(bits_of(g.k_cache[blk, row]), kc[blk, row])
        np.testing.assert_array_equal(bits_of(g.v_cache[blk, row]), vc[blk, row])


@pytest.mark.parametrize("case", ["ragged_g4_d128", "g8_int8_bs32", "fp8_d64_bs16"])
def test_decode_step_plan_equals_decode_step(case):
    """A prepared DecodeStepPlan (arguments checked and marshalled once) runs
    the same step as decode_step: outputs and pools bit-identical."""
    wl = CASES[case]()
    a, b = GpuStep(wl), GpuStep(wl)
    out_plan = bits_of(a.fused_step()).copy()
    pkv.decode_step(b.out, b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                    b.max_seq_len, wl.spec.scale, b.workspace, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    check_status()
    np.testing.assert_array_equal(bits_of(b.out), out_plan)
    np.testing.assert_array_equal(bits_of(a.k_cache), bits_of(b.k_cache))
    np.testing.assert_array_equal(bits_of(a.v_cache), bits_of(b.v_cache))
