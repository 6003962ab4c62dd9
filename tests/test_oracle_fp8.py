"""FP8 E4M3 pins for the oracle, without a GPU (“让 Agent 跑得快：LLM 推理服务”,
§四 FP8 量化: a 1-byte FP8 KV cache; “LLM 推理优化技术全景”, Flash Attention
v3: E4M3 with block-wise scales).

* Every code's value equals torch's float8_e4m3fn -> float conversion (a
  library routine written independently of this oracle).
* Encoding equals torch's float -> float8_e4m3fn cast (round to nearest,
  ties to even) on every code value, every midpoint between neighbouring
  codes (the ties), the subnormal range and random values below the
  overflow threshold 464; above it torch gives NaN while this library
  saturates to 448 (its reading, as int8 clamps to 127), checked apart.
* The quotient is decided in fp32 (as for int8).
* Attention over an E4M3 pool equals SDPA on the codes decoded by torch
  times their block scales.
"""
import numpy as np
import pytest

import oracle
import workloads
from oracle_helpers import oracle_pool
from test_oracle_attention import run, small
from workloads import bf16_bits_to_f32, to_bf16_bits

torch = pytest.importorskip("torch")


def torch_value(codes):
    """float64 values of uint8 E4M3 codes through torch's float8_e4m3fn."""
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_code(x32):
    """uint8 codes of fp32 values through torch's float8_e4m3fn cast."""
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def check_decode(value):
    want = torch_value(np.arange(256))
    got = np.array([value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))          # -0 for 0x80


def encode_cases():
    """fp32 values: every finite code value, every midpoint of neighbouring
    positive codes (exact in fp32), values just around each midpoint, the
    region below the smallest subnormal, random values; both signs."""
    vals = torch_value(np.arange(0x7F))                                     # 0 .. 448
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(8)
    xs = [vals, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
          np.nextafter(mids.astype(np.float32), np.float32(1000)),
          np.array([2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11, 1e-30, 448.0, 463.99, 460.0]),
          np.abs(rng.standard_normal(20000)) * rng.choice([1e-3, 0.1, 1.0, 30.0, 300.0], 20000)]
    x = np.concatenate([a.astype(np.float32) for a in xs])
    x = x[np.abs(x) < 464.0]
    return np.concatenate([x, -x]).astype(np.float32)


def check_encode(quant):
    x = encode_cases()
    want = torch_code(x)
    got = np.array([quant(float(v), 1.0) for v in x], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(want[i])) for i in bad[:5]]


def check_saturation(quant):
    assert quant(449.0, 1.0) == 0x7E and quant(1000.0, 1.0) == 0x7E and quant(1e30, 1.0) == 0x7E
    assert quant(-1000.0, 1.0) == 0xFE and quant(float("inf"), 1.0) == 0x7E
    assert quant(float("-inf"), 1.0) == 0xFE
    assert quant(float("nan"), 1.0) == 0x7F
    assert quant(3.3, 0.0) == quant(3.3, 1.0)                 # scale 0 is read as 1
    assert quant(-0.0, 1.0) == 0x80 and quant(0.0, 1.0) == 0x00


def check_fp32_quotient(quant):
    """The code is taken from the fp32 quotient x / s, as for int8."""
    rng = np.random.default_rng(6)
    x = bf16_bits_to_f32(to_bf16_bits(rng.standard_normal(300000).astype(np.float32) * 3))
    s = (np.abs(rng.standard_normal(300000)).astype(np.float32) * 0.02 + 1e-3).astype(np.float32)
    q32 = (x / s).astype(np.float32)
    c32 = torch_code(q32)
    c64 = torch_code((x.astype(np.float64) / s.astype(np.float64)).astype(np.float32))
    keep = np.abs(q32) < 448
    differ = np.nonzero((c32 != c64) & keep)[0]
    for i in differ[:50]:
        assert quant(float(x[i]), float(s[i])) == int(c32[i])
    for i in range(0, 300000, 3001):
        if keep[i]:
            assert quant(float(x[i]), float(s[i])) == int(c32[i])


def test_fp8_decode_matches_torch(oracle_mod):
    check_decode(oracle.fp8_value)


def test_fp8_closed_forms(oracle_mod):
    v = oracle.fp8_value
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0 and v(0x38) == 1.0 and v(0x40) == 2.0
    assert v(0x08) == 2.0 ** -6 and v(0x07) == 7 * 2.0 ** -9 and v(0x01) == 2.0 ** -9
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))


def test_fp8_encode_matches_torch(oracle_mod):
    check_encode(oracle.quantize_fp8)


def test_fp8_saturation_and_special_values(oracle_mod):
    check_saturation(oracle.quantize_fp8)


def test_fp8_decision_is_fp32(oracle_mod):
    check_fp32_quotient(oracle.quantize_fp8)


def test_fp8_append_stores_the_block_max_at_448(oracle_mod):
    """With scale = max|x| / 448 the block's largest element stores +-448,
    and every stored value is within half an E4M3 step of x."""
    wl = small([1, 31, 64, 200], hq=16, hkv=2, d=128, bs=32, kv="fp8", seed=12)
    kc, vc, ks, vs = oracle_pool(wl)
    bs = wl.spec.block_size
    for b in range(4):
        L = int(wl.seq_lens[b])
        pos, k, v = wl.own_tokens(b)
        xs = np.concatenate([bf16_bits_to_f32(k), bf16_bits_to_f32(wl.new_k[b:b + 1])])
        t = np.arange(L)
        blk = wl.block_tables[b, t // bs]
        codes = kc[blk, t % bs]
        vals = torch_value(codes) * ks[blk][:, :, None].astype(np.float64)
        # a relative step of E4M3 is at most 2^-3 (normals); subnormals step 2^-9 * scale
        err = np.abs(vals - xs)
        bound = np.maximum(np.abs(xs) * 2.0 ** -4, ks[blk][:, :, None] * 2.0 ** -10) * (1 + 1e-6)
        assert (err <= bound).all()
        for j in range(-(-L // bs)):
            sel = (t // bs) == j
            for h in range(wl.spec.num_kv_heads):
                c = codes[sel, h]
                assert (np.abs(torch_value(c)) == 448.0).any()


def check_fp8_against_sdpa(wl):
    """E4M3 pools: the oracle equals SDPA on torch-decoded codes * scale."""
    import torch.nn.functional as F
    kc, vc, ks, vs = oracle_pool(wl)
    out, rc = run(wl, (kc, vc, ks, vs))
    assert rc == 0
    bs, G = wl.spec.block_size, wl.spec.num_q_heads // wl.spec.num_kv_heads
    q = torch.from_numpy(bf16_bits_to_f32(wl.q).astype(np.float64))
    for b in range(wl.spec.batch):
        t = np.arange(wl.seq_lens[b])
        blk = wl.block_tables[b, t // bs]
        K = torch_value(kc[blk, t % bs]) * ks[blk][:, :, None].astype(np.float64)
        V = torch_value(vc[blk, t % bs]) * vs[blk][:, :, None].astype(np.float64)
        Kx = torch.from_numpy(K).repeat_interleave(G, dim=1).transpose(0, 1)
        Vx = torch.from_numpy(V).repeat_interleave(G, dim=1).transpose(0, 1)
        ref = F.scaled_dot_product_attention(q[b][:, None, :], Kx, Vx, scale=wl.spec.scale)[:, 0, :]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=0, atol=1e-12)


def test_oracle_matches_sdpa_fp8_dequantised(oracle_mod):
    check_fp8_against_sdpa(small([1, 5, 32, 33, 70, 200], hq=16, hkv=2, d=128, bs=32, kv="fp8", seed=3))
