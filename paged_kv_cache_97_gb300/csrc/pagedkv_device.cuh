// pagedkv_device.cuh -- device helpers shared by the library's kernels:
// the K/V block geometry in shared memory and thin PTX wrappers (mbarrier,
// TMA tensor loads, ldmatrix, mma.sync, byte permutes).  Internal only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pagedkv {
namespace dev {

#ifndef PAGEDKV_STAGE_BUDGET
#define PAGEDKV_STAGE_BUDGET (48 * 1024)
#endif
#ifndef PAGEDKV_CONSUMERS
#define PAGEDKV_CONSUMERS 3
#endif
// Stage memory and consumer warps per decode CTA: 48 KB and 3 consumers
// (about 4 CTAs per SM) measured best across the bench workloads on GB300
// against 64-128 KB with 4 consumers and 32-48 KB with 2.
constexpr int kConsumers = PAGEDKV_CONSUMERS;        // consumer warps per decode CTA
constexpr int kMaxStages = 8;
constexpr int kStageBudget = PAGEDKV_STAGE_BUDGET;    // shared memory for decode stages
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

template <int D, int BS, bool kQ8>
struct Geo {
  static constexpr int kElem = kQ8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;                          // 256, 128, 64
  static constexpr int kBoxRow = kRowBytes > 128 ? 128 : kRowBytes;    // bytes per box row
  static constexpr int kBoxes = kRowBytes / kBoxRow;                   // 2 for bf16 d128
  static constexpr int kBoxElems = kBoxRow / kElem;
  static constexpr bool kSwizzle = kBoxRow == 128;                     // SWIZZLE_128B
  static constexpr int kBoxBytes = BS * kBoxRow;
  static constexpr int kTensorBytes = kBoxes * kBoxBytes;              // K (or V) of a block
  static constexpr int kBlockBytes = 2 * kTensorBytes;                 // K + V
  static constexpr int kStageBytes = kConsumers * kBlockBytes;
  static constexpr int kStages0 = kStageBudget / kStageBytes;
  static constexpr int kStages = kStages0 < 2 ? 2 : (kStages0 > kMaxStages ? kMaxStages : kStages0);
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;      // + alignment slack
  static constexpr int kTiles = BS / 16;                               // 16-token MMA tiles
  static constexpr int kKSteps = D / 16;                               // MMA k-steps over d
  static constexpr int kMTiles = D / 16;                               // O^T m-tiles over d
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of the phase of `bar` with the given parity.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase of `bar` with the given parity, giving up after
// kWaitLimitNs; returns false on time-out (the caller reports it).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// D += A . B for one m16n8k16 tile, fp32 accumulate; A, B bf16 or fp16.
template <bool kF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (kF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Two fp32 -> packed pair, lower index in the low half.
template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (kF16)
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// XOR applied to each 32-bit word of codes before codes_to_f16x2: int8
// codes are biased by 128 (below); E4M3 codes are converted as they are.
template <bool kFp8>
constexpr uint32_t kCodeBias = kFp8 ? 0u : 0x80808080u;

// Two 8-bit codes of w as an fp16 pair (low half = the lower byte), exact
// either way; sel 0x4140 takes bytes 0,1 and 0x4342 bytes 2,3.
//   int8: w already XORed with kCodeBias, so each byte is c + 128; the
//         bytes are placed under 0x64 (fp16 1024 + byte) and 1152 is
//         subtracted: c.  kBiased leaves c + 1152 (the caller removes the
//         1152 from its sums).
//   E4M3: the hardware conversion of an e4m3 pair to f16x2 (every E4M3
//         value, subnormals included, is an fp16 value).
template <bool kFp8, bool kBiased = false>
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t w, uint32_t sel) {
  if constexpr (kFp8) {
    const unsigned short pair = sel == 0x4140u ? (unsigned short)(w & 0xffffu)
                                               : (unsigned short)(w >> 16);
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(pair));
    return h;
  } else {
    const uint32_t h = prmt(w, 0x64646464u, sel);
    if constexpr (kBiased) return h;
    __half2 x = *reinterpret_cast<const __half2*>(&h);
    x = __hsub2(x, __half2half2(__ushort_as_half((unsigned short)0x6480)));  // 1152.0
    return *reinterpret_cast<const uint32_t*>(&x);
  }
}

__device__ __forceinline__ int8_t quantize(float x, float s) {
  // clamp(round_half_even(x / s), -127, 127) with an IEEE fp32 divide.
  if (s == 0.0f) s = 1.0f;
  int c = __float2int_rn(__fdiv_rn(x, s));
  c = c > 127 ? 127 : (c < -127 ? -127 : c);
  return (int8_t)c;
}

// E4M3 code of x / s (IEEE fp32 divide; s == 0 -> 1): round to nearest even,
// magnitudes above 448 saturate to 448, NaN gives the NaN pattern.  The
// conversion packs its first operand in the upper byte, its second in the
// lower one.
__device__ __forceinline__ uint8_t quantize_e4m3(float x, float s) {
  if (s == 0.0f) s = 1.0f;
  const float r = __fdiv_rn(x, s);
  unsigned short h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(r));
  return (uint8_t)(h & 0xffu);
}

// The byte an 8-bit pool stores for x under scale s.
template <bool kFp8>
__device__ __forceinline__ uint8_t code8(float x, float s) {
  if constexpr (kFp8) return quantize_e4m3(x, s);
  else return (uint8_t)quantize(x, s);
}

// Byte offset of 16-byte chunk `c` of row `r` inside one K or V block of a
// stage.  Rows of a box are kBoxRow bytes; with SWIZZLE_128B the chunk index
// inside each 128-byte row is XORed with (row mod 8), the pattern TMA writes
// (box starts are 1024-byte aligned).
template <class G>
__device__ __forceinline__ uint32_t chunk_off(int r, int c) {
  constexpr int kChunksPerBox = G::kBoxRow / 16;
  const int box = c / kChunksPerBox, cc = c % kChunksPerBox;
  const int phys = G::kSwizzle ? (cc ^ (r & 7)) : cc;
  return box * G::kBoxBytes + r * G::kBoxRow + phys * 16;
}


}  // namespace dev
}  // namespace pagedkv
