// pagedkv_multi_tc.cu -- attention of long multi-token queries (prefill
// chunks: “LLM 推理优化技术全景”, SARATHI -- 512-token chunks batched with
// decodes) on the fifth-generation tensor cores, accumulators in TMEM.
//
// Sequence b's query token i (of n_b, its last tokens) at position
// L_b - n_b + i attends positions 0 .. L_b - n_b + i.  A CTA takes two tiles
// of 128 rows (query token, grouped head) of one sequence and KV head -- each
// tile the MMA's M -- and one token partition, in chunks of 128 keys that
// both tiles share:
//
//   * warps 9 and 10 (one lane issues): TMA tensor loads of each chunk's K
//     (warp 9) and V (warp 10) blocks (ids staged in shared memory) into one
//     of two stages each, laid out as 128 contiguous 128-byte-swizzled rows
//     per 64-element column band, so one descriptor covers the chunk; a
//     stage is refilled once both tiles' MMAs of the chunk two back have
//     read it;
//   * warp 8 (one lane issues), per tile g:
//       S_g[128 x 128] = Q_g[128 x d] . K^T          (A and B from smem)
//       O_g[128 x d]  += P_g[128 x 128] . V[128 x d] (A = P_g from TMEM)
//     in ping-pong order -- P . V_0(c), S_0(c+1), P . V_1(c), S_1(c+1) -- so
//     the tensor core works on one tile while the other tile's softmax runs
//     (an N = 64 MMA takes as long to issue as an N = 128 one, so wide chunks
//     halve S's issue time);
//   * warps 0-3 (tile 0) and 4-7 (tile 1), one row per thread: read S from
//     TMEM, apply the causal mask (only in chunks that cross a row's last
//     key) and the scale, update the row's running maximum and sum (“LLM
//     推理优化技术全景”, 在线 Softmax; “Flash Attention v2 的改进”: deferred
//     normalisation), write P back over its S in TMEM, and at the end
//     normalise O.  The maximum used for P moves only when a row's scores
//     pass it by more than 2^8 (then O is rescaled in TMEM): P <= 2^8 stays
//     exact in the sums, and O and l always share the same reference, so the
//     result is the softmax's.  A negative scale flips Q's signs instead
//     (exact), so maxima are taken on raw scores.
//
// TMEM: O_0, O_1 (d columns each) and two 128-column S/P buffers, all 512
// columns, so one CTA per SM (its shared memory is sized to keep it so).  The
// CTAs are persistent: each takes units (KV head fastest, then partition,
// then tile pair) gridDim apart, over the real tiles only, with TMEM held
// throughout and the barriers invalidated and set up again per unit; the
// host launches one per SM (beside the decode kernel's column groups, on a
// side stream, or alone).  V rows past the sequence end are zeroed in shared
// memory before P . V (p is 0 there but the pool may hold NaN).  Every wait
// is bounded; a CTA that gives up flags PAGEDKV_FLAG_WAIT_TIMEOUT, drains its
// copies and tensor-core work, frees its TMEM and marks its rows bad.  A warp
// whose 32 rows are all padding only keeps the barrier phases; a pair whose
// second tile holds no rows runs the first alone.  bf16, int8 and E4M3 pools
// (the 8-bit kinds in fp16, described at the kernel).
//
// Shared-prefix mode (kPrefix): when every sequence's first blocks are the
// same physical blocks (“让 Agent 跑得快”, §五 共享前缀), the prefix part of
// attention is one dense, unmasked product per KV head; the batch's query
// tokens (one per sequence) form the query block, every row sees every prefix
// token, the block ids come from the prefix list, and each row's partial goes
// to its slots after the decode partitions for the merge.  The host runs it
// on few CTAs ahead of the decode kernel, which it releases at once.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv_common.cuh"
#include "pagedkv_device.cuh"

namespace pagedkv {
namespace {

using namespace dev;

constexpr int kTRows = 128;               // query rows per tile (the MMA's M)
constexpr int kTiles = 2;                 // row tiles per CTA, computed in ping-pong
constexpr int kChunk = 128;               // keys per chunk (the S MMA's N)
constexpr int kKStages = 2;               // K chunk stages
constexpr int kVStages = 3;               // V chunk stages (V is released later than K)
constexpr int kTcStages = kVStages;    // barrier slots per operand
constexpr int kSoftmaxWarps = 4 * kTiles; // warps 0-3: tile 0, 4-7: tile 1 (one row per thread)
constexpr int kMmaWarp = kSoftmaxWarps;   // one lane issues the MMAs
constexpr int kKWarp = kMmaWarp + 1;      // K loads (and 8-bit widening)
constexpr int kVWarp = kMmaWarp + 2;      // V loads (and 8-bit widening)
constexpr int kTThreads = (kSoftmaxWarps + 3) * 32;
constexpr int kTmemCols = 512;            // the whole TMEM: one CTA per SM
constexpr float kRescaleLog2 = 8.0f;      // move the reference max past 2^8

template <int D>
struct TcGeo {
  static constexpr int kAtoms = D / 64;                  // 64-element (128-byte) column bands
  static constexpr int kQBytes = kTRows * D * 2;         // Q image of one tile
  static constexpr int kKBytes = kChunk * D * 2;         // K (or V) of a chunk
  // Q of both tiles, the K and V stages (+ alignment); at least 120 KB so
  // that two CTAs never share an SM (each takes the whole TMEM)
  static constexpr int kUsed = kTiles * kQBytes + (kKStages + kVStages) * kKBytes + 1024;
  static constexpr int kSmemBytes = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
  // TMEM: O of tile g in columns [g D, g D + D), S (and P over it) of tile g
  // in [2 D + 128 g, 2 D + 128 g + 128)
  __host__ __device__ static constexpr uint32_t ocol(int g) { return (uint32_t)(g * D); }
  __host__ __device__ static constexpr uint32_t scol(int g) { return (uint32_t)(2 * D + 128 * g); }
};

// 128-byte-swizzled K-major / MN-major shared-memory matrix descriptor.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;                                // descriptor version
  d |= (uint64_t)2 << 61;                                // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: fp32 D, A and B both bf16 (or both
// fp16: kF16), A K-major, B K- or MN-major, N, M.
template <bool kF16>
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, int b_mn_major) {
  return (1u << 4) | (kF16 ? 0u : (1u << 7) | (1u << 10)) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
               ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
               ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mbar_inval(uint32_t bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes (one row per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),
        "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15])
      : "memory");
}

// A bounded mbarrier wait whose outcome the whole warp agrees on (the
// warp's later tcgen05 loads and stores are collective).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled
// band (the pattern TMA writes; bands start 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32: relative error
// about 2^-22, results below 2^-126 flushed to 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Scores of 32 consecutive keys of a chunk row times per-key factors: the
// first 16 keys by f[0], the next 16 by f[1] (8-bit pools: each key's block
// K scale with the score scale; blocks hold 16 or 32 keys).
__device__ __forceinline__ void scale_keys(uint32_t (&raw)[32], const float (&f)[2]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) raw[j] = __float_as_uint(__uint_as_float(raw[j]) * f[j >> 4]);
}

// Largest score of a chunk row (keys past `lim` left out when kMask), four
// independent partial maxima.
template <bool kMask, int kH>
__device__ __forceinline__ float chunk_max(const uint32_t (&raw)[kH][32], int first_tok, int lim) {
  float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int h = 0; h < kH; ++h)
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float v = __uint_as_float(raw[h][j]);
      if (kMask && first_tok + 32 * h + j > lim) v = -INFINITY;
      mr[j & 3] = fmaxf(mr[j & 3], v);
    }
  return fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3]));
}

// p = 2^(s * sl2 - ref) of a chunk row (0 for keys past `lim` when kMask).
// P goes out as bf16 pairs and the returned fp32 sum adds those bf16 values,
// so that O and the row sum weigh every key alike (a row whose weight sits
// on one key returns that key's V exactly); or (kF16) P goes out as fp16
// pairs of p times the key's factor vr[h][j >> 4] (8-bit pools: the block's
// V scale relative to the partition's largest) and the sum adds p.
template <bool kMask, bool kF16, int kH>
__device__ __forceinline__ float chunk_exp(const uint32_t (&raw)[kH][32], uint32_t (&pw)[kH][16],
                                           int first_tok, int lim, float sl2, float ref,
                                           const float (&vr)[kH][2]) {
  float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int h = 0; h < kH; ++h)
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float p0 = ex2(fmaf(__uint_as_float(raw[h][2 * j]), sl2, -ref));
      float p1 = ex2(fmaf(__uint_as_float(raw[h][2 * j + 1]), sl2, -ref));
      if (kMask) {
        const int tok = first_tok + 32 * h + 2 * j;
        p0 = tok <= lim ? p0 : 0.0f;
        p1 = tok + 1 <= lim ? p1 : 0.0f;
      }
      if constexpr (kF16) {
        ls[(2 * j) & 3] += p0;
        ls[(2 * j + 1) & 3] += p1;
        const float f = vr[h][j >> 3];
        pw[h][j] = pack2<true>(p0 * f, p1 * f);
      } else {
        const uint32_t w = pack2<false>(p0, p1);
        pw[h][j] = w;
        ls[(2 * j) & 3] += __uint_as_float(w << 16);
        ls[(2 * j + 1) & 3] += __uint_as_float(w & 0xffff0000u);
      }
    }
  return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// A packed pair of P values (bf16, or fp16 when kF16) times a power of two.
template <bool kF16>
__device__ __forceinline__ uint32_t scale_pair(uint32_t w, float f) {
  if constexpr (kF16) {
    __half2 h = *reinterpret_cast<const __half2*>(&w);
    const float2 x = __half22float2(h);
    return pack2<true>(x.x * f, x.y * f);
  } else {
    return pack2<false>(__uint_as_float(w << 16) * f, __uint_as_float(w & 0xffff0000u) * f);
  }
}

// Sixteen 8-bit codes as sixteen exact fp16 values (zeros when `zero`).
template <bool kFp8>
__device__ __forceinline__ void widen16(uint4 w, bool zero, uint4& lo, uint4& hi) {
  const uint32_t x[4] = {w.x ^ kCodeBias<kFp8>, w.y ^ kCodeBias<kFp8>, w.z ^ kCodeBias<kFp8>,
                         w.w ^ kCodeBias<kFp8>};
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[2 * i] = zero ? 0u : codes_to_f16x2<kFp8>(x[i], 0x4140u);
    h[2 * i + 1] = zero ? 0u : codes_to_f16x2<kFp8>(x[i], 0x4342u);
  }
  lo = make_uint4(h[0], h[1], h[2], h[3]);
  hi = make_uint4(h[4], h[5], h[6], h[7]);
}

// 8-bit pools: the codes of chunk rows [0, nrows), landed by TMA in the
// second half of the chunk's operand image (D bytes per row; 128-byte
// swizzled rows when D = 128), widened exactly to fp16 in the image's own
// layout (128 contiguous 128-byte-swizzled rows per 64-element band), rows
// at or past `zero_from` written as zeros (the pool's rows past a sequence's
// end may hold NaN patterns).  One warp; lane i takes rows i, i + 32, ...
//   D = 128: a row's staged codes sit exactly under its fp16 row in band 1;
//     taking its 16-code chunks in order, each fp16 write lands on codes
//     already read (chunk c >= 4 writes band-1 chunks 2c - 8 and 2c - 7).
//   D = 64: fp16 rows 64.. overwrite the staged codes of rows 2r - 128 and
//     2r - 127, which other lanes of the same round may still need, so each
//     round reads all its codes before any lane writes.
template <int D, bool kFp8>
__device__ __forceinline__ void widen_chunk(unsigned char* img, int nrows, int zero_from, int lane) {
  const unsigned char* stg = img + D * kChunk;           // second half of the D * 2 * kChunk image
  auto put = [&](int r, int e8, uint4 v) {               // 8-element chunk e8 of fp16 row r
    const int band = e8 >> 3, cc = e8 & 7;
    *reinterpret_cast<uint4*>(img + band * (kChunk * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
  };
#pragma unroll 1
  for (int r0 = 0; r0 < nrows; r0 += 32) {
    const int r = r0 + lane;
    const bool live = r < nrows, zero = r >= zero_from;
    if constexpr (D == 128) {
      if (live) {
#pragma unroll 2
        for (int c = 0; c < 8; ++c) {
          const uint4 w = *reinterpret_cast<const uint4*>(stg + r * 128 + ((c ^ (r & 7)) << 4));
          uint4 lo, hi;
          widen16<kFp8>(w, zero, lo, hi);
          put(r, 2 * c, lo);
          put(r, 2 * c + 1, hi);
        }
      }
    } else {
      uint4 w[4];
      if (live) {
#pragma unroll
        for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint4*>(stg + r * 64 + c * 16);
      }
      __syncwarp();
      if (live) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint4 lo, hi;
          widen16<kFp8>(w[c], zero, lo, hi);
          put(r, 2 * c, lo);
          put(r, 2 * c + 1, hi);
        }
      }
      __syncwarp();
    }
  }
}

// Pairs of 128-row tiles of a sequence with n query tokens served here
// (n > col_max_n); in shared-prefix mode n is the batch (col_max_n = 0).
__host__ __device__ __forceinline__ int tc_pairs(int n, int GQ, int col_max_n) {
  return n > col_max_n ? (n * GQ + kTiles * kTRows - 1) / (kTiles * kTRows) : 0;
}

// kKind: the pool's dtype (KV_DTYPE_BF16, KV_DTYPE_INT8, KV_DTYPE_FP8_E4M3).
// 8-bit pools run the MMAs in fp16: Q is converted (scaled by a power of two
// when its magnitude needs it, folded back into the score scale), the codes
// are widened exactly by the load warp after each chunk lands, each key's
// block K scale multiplies its score and each block's V scale, relative to
// the partition's largest, multiplies P (the output takes that largest back).
template <int D, int BS, bool kPrefix, int kKind>
__global__ void __launch_bounds__(kTThreads, 1)
    multi_tc_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
  constexpr bool kQ8 = kKind != KV_DTYPE_BF16, kFp8 = kKind == KV_DTYPE_FP8_E4M3;
  using T = TcGeo<D>;
  using Gm = Geo<D, BS, kQ8>;                            // TMA box geometry of one block
  constexpr int kBlocksPerChunk = kChunk / BS;
  constexpr int kMaxPartBlocks = kMaxPartTokens / 16;
  extern __shared__ unsigned char smem_raw[];
  // per K (V) stage: landed, widened (8-bit), free again; per tile: S done,
  // P written, P . V done
  __shared__ uint64_t k_full[kTcStages], k_ready[kTcStages], k_empty[kTcStages];
  __shared__ uint64_t v_full[kTcStages], v_ready[kTcStages], v_empty[kTcStages];
  __shared__ uint64_t s_full[kTiles], p_full[kTiles], o_done[kTiles], drain_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int scan[32];
  __shared__ int sh_b, sh_pr, sh_bad, sh_fail;
  __shared__ int32_t blk_ids[kMaxPartBlocks];            // this partition's physical blocks
  __shared__ float blk_ks[kQ8 ? kMaxPartBlocks : 1];     // 8-bit: their K scales
  __shared__ float blk_vs[kQ8 ? kMaxPartBlocks : 1];     //        and V scales
  __shared__ float sh_vmax;                              //        the largest |V scale|

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads, GQ = Hq / Hkv;
  const int B = a.batch;
  const int32_t* qs = a.query_start;
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - smem_addr(smem_raw));
  auto q_img = [&](int g) { return base + (uint32_t)(g * T::kQBytes); };
  auto k_img = [&](int s) { return base + (uint32_t)(kTiles * T::kQBytes + s * T::kKBytes); };
  auto v_img = [&](int s) { return base + (uint32_t)(kTiles * T::kQBytes + (kKStages + s) * T::kKBytes); };

  // ---- work units: (KV head, partition, pair of 128-row tiles).  Multi-token
  // mode: tile pairs per sequence (sequences past the column groups' limit,
  // in order), prefix-summed once by warp 0: scan[lane] ends the pairs of
  // sequences lane*per .. lane*per + per - 1.  Shared-prefix mode: the
  // batch's query tokens form one query block over the prefix blocks.
  const int per = (B + 31) / 32;
  int mine = 0;
  int64_t units;
  if constexpr (kPrefix) {
    // the decode kernel queued behind this one reads nothing it writes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    units = (int64_t)tc_pairs(B, GQ, 0) * Hkv * a.prefix_chunks;
  } else {
    if (warp == 0) {
      for (int i = 0; i < per; ++i) {
        const int b = lane * per + i;
        if (b < B) mine += tc_pairs(qs[b + 1] - qs[b], GQ, a.col_max_n);
      }
      int incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      scan[lane] = incl;
    }
    __syncthreads();
    units = (int64_t)scan[31] * Hkv * a.max_parts;
  }
  const int nparts = kPrefix ? a.prefix_chunks : a.max_parts;
  const int ptok = kPrefix ? a.prefix_part_tokens : a.part_tokens;
  bool tm_held = false;                                  // TMEM allocated (CTA-uniform)
  uint32_t tm = 0;

  // ---- persistent loop over units, KV head fastest
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
  const int hk = (int)(u % Hkv), part = (int)((u / Hkv) % nparts);
  const int x = (int)(u / ((int64_t)Hkv * nparts));      // tile pair over all sequences
  __syncthreads();                                       // the last unit's readers are done
  if (tid == 0) {
    sh_b = -1;
    sh_bad = 0;
    sh_fail = 0;
    sh_vmax = 0.0f;
  }
  __syncthreads();
  if (!kPrefix && warp == 0 && x >= scan[lane] - mine && x < scan[lane]) {
    int acc = scan[lane] - mine;
    for (int i = 0; i < per; ++i) {
      const int b = lane * per + i;
      if (b >= B) break;
      const int pl = tc_pairs(qs[b + 1] - qs[b], GQ, a.col_max_n);
      if (x < acc + pl) {
        sh_b = b;
        sh_pr = x - acc;
        break;
      }
      acc += pl;
    }
  }
  __syncthreads();
  // Shared-prefix mode: row r is sequence r / GQ's one query token, which
  // sees every prefix token.
  const int b = kPrefix ? 0 : sh_b, pr = kPrefix ? x : sh_pr;   // x < the pair count: found
  const int q0 = kPrefix ? 0 : qs[b], n = kPrefix ? B : qs[b + 1] - q0;
  const int L = kPrefix ? a.num_prefix_blocks * BS : a.seq_lens[b];
  const int t0 = part * ptok;
  if (t0 >= L && L > 0) continue;                        // no such partition (CTA-uniform)
  const bool rows_ok = kPrefix || (q0 >= 0 && q0 + n <= a.num_tokens);
  const bool len_ok = kPrefix || (rows_ok && L > 0 && n <= L && n <= a.max_query_len &&
                                  L <= a.max_seq_len && (int64_t)L <= (int64_t)a.max_blocks_per_seq * BS);
  const int rows_b = n * GQ;
  const int row0 = pr * (kTiles * kTRows);               // first row of tile 0
  const bool live1 = row0 + kTRows < rows_b;             // tile 1 holds rows
  const int last_row = min(row0 + kTiles * kTRows, rows_b) - 1;
  const int pos_max = kPrefix ? L - 1 : L - n + last_row / GQ;
  const int t_end = min(min(t0 + ptok, L), pos_max + 1);
  const int nch = (len_ok && t_end > t0) ? (t_end - t0 + kChunk - 1) / kChunk : 0;
  const int first_blk = t0 / BS;
  const int last_blk = nch > 0 ? (t_end - 1) / BS : first_blk - 1;
  const int32_t* bt = kPrefix ? a.prefix_blocks : a.block_tables + (int64_t)b * a.max_blocks_per_seq;
  // the partition's block ids, checked and kept in shared memory (the host
  // holds partitions to kMaxPartTokens tokens)
  for (int j = first_blk + tid; j <= last_blk; j += kTThreads) {
    const int32_t p = bt[j];
    const bool ok = p >= 0 && p < a.num_blocks;
    if (!ok) sh_bad = 1;
    blk_ids[j - first_blk] = p;
    if constexpr (kQ8) {
      if (ok) {
        blk_ks[j - first_blk] = a.k_scale[(int64_t)p * Hkv + hk];
        const float vs = a.v_scale[(int64_t)p * Hkv + hk];
        blk_vs[j - first_blk] = vs;
        atomicMax(reinterpret_cast<int*>(&sh_vmax), __float_as_int(fabsf(vs)));
      }
    }
  }
  // This thread's row (softmax warps 0-7): tile g = warp / 4, row i of it
  const int tile = warp >> 2, ri = tid & (kTRows - 1);
  const int r = row0 + tile * kTRows + ri;               // meaningful for warp < 8
  const bool row_valid = warp < kSoftmaxWarps && len_ok && r < rows_b;
  const int pos = row_valid ? (kPrefix ? L - 1 : L - n + r / GQ) : -1;
  const int64_t qrow = row_valid ? (int64_t)(q0 + r / GQ) * Hq + (int64_t)hk * GQ + r % GQ : 0;
  // Q row into its tile's swizzled bands (zeros for rows past the sequence's
  // queries).  A negative scale flips Q's signs instead (exact), so that the
  // softmax below scales S by |scale| and may take maxima of raw scores.
  float sl2 = fabsf(a.scale_log2);
  if (warp < kSoftmaxWarps) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + qrow * D);
    const uint32_t flip = a.scale_log2 < 0.0f ? 0x80008000u : 0u;
    // the whole row in registers first, so its loads are in flight together
    uint4 qv[D / 8];
#pragma unroll
    for (int c = 0; c < D / 8; ++c) qv[c] = row_valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    float qscale = 1.0f;
    if constexpr (kQ8) {
      // fp16 holds |q| < 65504: rows with a larger entry are scaled by a
      // power of two, undone in the score scale (exact either way)
      float amax = 0.0f;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint32_t w4[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w4[i] << 16)),
                                   fabsf(__uint_as_float(w4[i] & 0xffff0000u))));
      }
      int e = 0;
      if (amax >= 16384.0f) {
        frexpf(amax, &e);
        e -= 14;
      }
      qscale = ldexpf(1.0f, -e);
      sl2 = sl2 / qscale;
    }
    unsigned char* qdst = gbase + (q_img(tile) - base);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      uint4 v = qv[c];
      if constexpr (kQ8) {
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t o4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          o4[i] = pack2<true>(__uint_as_float(w4[i] << 16) * qscale,
                              __uint_as_float(w4[i] & 0xffff0000u) * qscale);
        v = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      v.x ^= flip;
      v.y ^= flip;
      v.z ^= flip;
      v.w ^= flip;
      *reinterpret_cast<uint4*>(qdst + (c / 8) * (kTRows * 128) + sw128(ri, c % 8)) = v;
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(smem_addr(&k_full[s]), 1);
      mbar_init(smem_addr(&k_ready[s]), 1);
      mbar_init(smem_addr(&k_empty[s]), 1);
      mbar_init(smem_addr(&v_full[s]), 1);
      mbar_init(smem_addr(&v_ready[s]), 1);
      mbar_init(smem_addr(&v_empty[s]), 1);
    }
    for (int g = 0; g < kTiles; ++g) {
      mbar_init(smem_addr(&s_full[g]), 1);
      mbar_init(smem_addr(&p_full[g]), kTRows);
      mbar_init(smem_addr(&o_done[g]), 1);
    }
    mbar_init(smem_addr(&drain_bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const bool work = nch > 0;
  const bool alloc_now = work && !tm_held;
  if (alloc_now && warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(&tmem_base)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // Q images -> tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (alloc_now) {
    tm_held = true;
    tm = tmem_base;
  }
  const bool bad = sh_bad != 0;
  float m_ref = -INFINITY, l = 0.0f;

  if (work && !bad) {
    if (warp == kMmaWarp) {
      // ======================= tensor-core issue ===========================
      // One lane.  Ping-pong over the two tiles: while one tile's softmax
      // runs, the tensor core computes the other tile's P . V and next S.
      // Per chunk c:  P . V_0(c), S_0(c+1), P . V_1(c), [V stage free],
      // S_1(c+1), [K stage free].  (S_g(c+1) overwrites the S/P columns
      // P . V_g(c) reads; the MMAs of one issuing thread run in issue order.)
      if (lane == 0) {
        bool ok = true;
        const uint32_t id_s = mma_idesc<kQ8>(kTRows, kChunk, 0);
        const uint32_t id_o = mma_idesc<kQ8>(kTRows, D, 1);
        auto issue_s = [&](int g, int c) {
          const uint32_t kb = k_img(c % kKStages);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t ad = smem_desc(q_img(g) + (ks / 4) * (kTRows * 128) + (ks % 4) * 32, 16, 1024);
            const uint64_t bd = smem_desc(kb + (ks / 4) * (kChunk * 128) + (ks % 4) * 32, 16, 1024);
            mma_ss(tm + T::scol(g), ad, bd, id_s, ks > 0);
          }
          mma_commit(smem_addr(&s_full[g]));
        };
        auto issue_pv = [&](int g, int c, int nsub) {
          const uint32_t vb = v_img(c % kVStages);
          for (int kk = 0; kk < nsub; ++kk) {
            const uint64_t bd = smem_desc(vb + kk * (16 * 128), kChunk * 128, 1024);
            mma_ts(tm + T::ocol(g), tm + T::scol(g) + kk * 8, bd, id_o, (c > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(smem_addr(&o_done[g]));
        };
        if (mbar_wait(smem_addr(&k_ready[0]), 0)) {
          tc_fence_after();
          issue_s(0, 0);
          if (live1) issue_s(1, 0);
          mma_commit(smem_addr(&k_empty[0]));
        } else {
          ok = false;
        }
        for (int c = 0; c < nch && ok; ++c) {
          const int vs = c % kVStages;
          if (!mbar_wait(smem_addr(&v_ready[vs]), (c / kVStages) & 1)) { ok = false; break; }
          const int cstart = t0 + c * kChunk;
          const int nsub = (min(t_end, cstart + kChunk) - cstart + 15) / 16;
          const bool next = c + 1 < nch;
          const int ks1 = (c + 1) % kKStages;
          if (!mbar_wait(smem_addr(&p_full[0]), c & 1)) { ok = false; break; }
          if (next && !mbar_wait(smem_addr(&k_ready[ks1]), ((c + 1) / kKStages) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, c, nsub);
          if (next) issue_s(0, c + 1);
          if (live1) {
            if (!mbar_wait(smem_addr(&p_full[1]), c & 1)) { ok = false; break; }
            tc_fence_after();
            issue_pv(1, c, nsub);
          }
          mma_commit(smem_addr(&v_empty[vs]));
          if (next) {
            if (live1) issue_s(1, c + 1);
            mma_commit(smem_addr(&k_empty[ks1]));
          }
        }
        if (!ok) sh_fail = 1;
      }
      __syncwarp();
    } else if (warp == kKWarp || warp == kVWarp) {
      // ======================= loads (TMA) ==================================
      // One warp per operand: chunk c goes to stage c % stages once the chunk
      // that used the stage before has been consumed there.  Once it lands,
      // 8-bit codes are widened to fp16 and bf16 V rows past the sequence end
      // are zeroed (p is 0 there but the pool may hold NaN); then the stage
      // is ready.
      const bool is_k = warp == kKWarp;
      const int nst = is_k ? kKStages : kVStages;
      const CUtensorMap* map = is_k ? &k_map : &v_map;
      uint64_t* ready = is_k ? k_ready : v_ready;
      uint64_t* empty = is_k ? k_empty : v_empty;
      // bf16 K needs no work after landing: its loads complete on the ready
      // barrier itself
      uint64_t* full = (is_k && !kQ8) ? k_ready : (is_k ? k_full : v_full);
      bool ok = true;
      auto issue = [&](int c) {                          // lane 0: chunk c into stage c % nst
        const int st = c % nst;
        const uint32_t img = is_k ? k_img(st) : v_img(st);
        const int blk0 = first_blk + c * kBlocksPerChunk;
        const int nb = min(kBlocksPerChunk, last_blk - blk0 + 1);
        const uint32_t bar = smem_addr(&full[st]);
        mbar_expect_tx(bar, (uint32_t)(nb * Gm::kTensorBytes));
        for (int j = 0; j < nb; ++j) {
          const int p = blk_ids[blk0 - first_blk + j];
          if constexpr (kQ8) {
            // codes of rows j*BS .. j*BS + BS - 1 into the image's second half
            tma_load_4d(img + D * kChunk + j * (BS * D), map, bar, 0, hk, 0, p);
          } else {
#pragma unroll
            for (int xx = 0; xx < Gm::kBoxes; ++xx)
              // band xx of the chunk image, rows j*BS .. j*BS + BS - 1
              tma_load_4d(img + xx * (kChunk * 128) + j * (BS * 128), map, bar, xx * Gm::kBoxElems, hk, 0, p);
          }
        }
      };
      // Every stage is filled up front.  Then two kinds of events, taken as
      // they come (polled, so neither waits behind the other): a landed
      // chunk is made ready in order (8-bit: widened; bf16 V: its rows past
      // the sequence end zeroed), and a stage the MMAs have finished with is
      // refilled with the chunk nst ahead.  bf16 K needs no work: its loads
      // complete on the ready barrier.
      const bool process = kQ8 || !is_k;
      int issued = min(nst, nch);
      if (lane == 0)
        for (int c = 0; c < issued; ++c) issue(c);
      __syncwarp();
      int nproc = process ? 0 : nch;                     // next chunk to make ready
      int nref = 0;                                      // next chunk whose stage to refill
      unsigned long long idle_since = global_ns();
      while (nproc < nch || nref + nst < nch) {
        bool did = false;
        if (nproc < nch &&
            __shfl_sync(0xffffffffu, mbar_test(smem_addr(&full[nproc % nst]), (nproc / nst) & 1), 0)) {
          const int c = nproc, st = c % nst;
          const uint32_t img = is_k ? k_img(st) : v_img(st);
          const int cstart = t0 + c * kChunk;
          if constexpr (kQ8) {
            const int blk0 = first_blk + c * kBlocksPerChunk;
            const int nb = min(kBlocksPerChunk, last_blk - blk0 + 1);
            widen_chunk<D, kFp8>(gbase + (img - base), nb * BS, is_k ? kChunk : L - cstart, lane);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // fp16 -> tensor core
          } else if (L < cstart + kChunk && L > cstart && (L % BS) != 0) {
            const int row_lo = L - cstart, row_hi = min(kChunk, ((L + BS - 1) / BS) * BS - cstart);
            const int nrow = row_hi - row_lo;
            unsigned char* vdst = gbase + (img - base);
            for (int i = lane; i < nrow * 8 * T::kAtoms; i += 32) {
              const int rr = row_lo + i / (8 * T::kAtoms), rest = i % (8 * T::kAtoms);
              const int band = rest / 8, cc = rest % 8;
              *reinterpret_cast<uint4*>(vdst + band * (kChunk * 128) + sw128(rr, cc)) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&ready[st]));
          ++nproc;
          did = true;
        } else if (nref + nst < nch && nref < nproc &&
                   __shfl_sync(0xffffffffu, mbar_test(smem_addr(&empty[nref % nst]), (nref / nst) & 1), 0)) {
          if (lane == 0) issue(nref + nst);
          issued = nref + nst + 1;
          ++nref;
          __syncwarp();
          did = true;
        }
        if (did) {
          idle_since = global_ns();
        } else if (global_ns() - idle_since > kWaitLimitNs) {
          ok = false;
          break;
        }
      }
      if (!ok && lane == 0) sh_fail = 1;
      // every load issued has landed before the CTA moves on (bounded;
      // normally already complete)
      if (lane == 0) {
        for (int st = 0; st < nst && st < issued; ++st) {
          const int last = st + nst * ((issued - 1 - st) / nst);
          mbar_wait(smem_addr(&full[st]), (last / nst) & 1);
        }
      }
    } else if (warp < kSoftmaxWarps && (tile == 0 || live1)) {
      // ======================= softmax: one row per thread (warps 0-7) ======
      // A chunk row's 128 scores in two halves of 64, each read from TMEM
      // once: its maximum is tested against the row's reference, then P is
      // formed and written back.  P of keys [64h, 64h + 64) lands in packed
      // columns [32h, 32h + 32), which that half has already read.  When a
      // half passes the reference by more than 2^8, the reference moves up
      // by a whole number of octaves (so the rescale factor is a power of two
      // and every rescale is exact): O is rescaled once P . V of the chunk
      // before has finished, and a first half of P already written is
      // rescaled in place.
      const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
      const uint32_t s_tmem = tm + lane_base + T::scol(tile);
      const uint32_t o_tmem = tm + lane_base + T::ocol(tile);
      constexpr int kH = 2;                              // 32-key groups per half
      constexpr int kPasses = kChunk / (32 * kH);
      bool ok = true;
      // A warp whose 32 rows are all padding (a tile's last rows) has nothing
      // to compute: its P rows feed only O rows that are never written out,
      // so it just keeps the barrier phases (S(c) done, then P(c) "written").
      const bool warp_live = __any_sync(0xffffffffu, row_valid);
      const float sl2c = kQ8 ? 1.0f : sl2;               // (8-bit: applied per key)
      for (int c = 0; c < nch; ++c) {
        if (__shfl_sync(0xffffffffu, sh_fail, 0)) { ok = false; break; }
        if (!warp_wait(smem_addr(&s_full[tile]), c & 1)) { ok = false; break; }
        tc_fence_after();
        if (!warp_live) {
          tc_fence_before();
          mbar_arrive(smem_addr(&p_full[tile]));
          continue;
        }
        const int cstart = t0 + c * kChunk;
        const int lim = min(pos, t_end - 1);             // last key this row may see
        // only chunks that cross some row's last visible key need the mask
        const bool masked = __any_sync(0xffffffffu, cstart + kChunk - 1 > lim);
        // 8-bit pools: per-key factors of each 32-key group of a half, the K
        // scale of the key's block times the score scale (scores then leave
        // in log2 units) and its relative V scale
        auto key_factors = [&](int ps, float (&kf)[kH][2], float (&vf)[kH][2]) {
          const float inv_vmax = sh_vmax > 0.0f ? 1.0f / sh_vmax : 1.0f;
#pragma unroll
          for (int h = 0; h < kH; ++h)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int jb = (c * kChunk + 64 * ps + 32 * h + 16 * half) / BS;   // < kMaxPartBlocks
              kf[h][half] = blk_ks[jb] * sl2;
              vf[h][half] = blk_vs[jb] * inv_vmax;
            }
        };
        float lsum = 0.0f;
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
          uint32_t raw[kH][32];
#pragma unroll
          for (int h = 0; h < kH; ++h) tmem_ld32(s_tmem + 64 * ps + 32 * h, raw[h]);
          tmem_wait_ld();
          float kf[kH][2], vf[kH][2] = {};
          if constexpr (kQ8) {
            key_factors(ps, kf, vf);
#pragma unroll
            for (int h = 0; h < kH; ++h) scale_keys(raw[h], kf[h]);
          }
          const int first = cstart + 64 * ps;
          const float mx_raw = masked ? chunk_max<true>(raw, first, lim) : chunk_max<false>(raw, first, lim);
          const float mx = mx_raw == -INFINITY ? -INFINITY : mx_raw * sl2c;
          const bool need = m_ref == -INFINITY ? mx > -INFINITY : mx > m_ref + kRescaleLog2;
          if (__any_sync(0xffffffffu, need)) {
            // a whole number k of octaves: the factor is exactly 2^-k
            const float k = (need && m_ref != -INFINITY) ? ceilf(mx - m_ref) : 0.0f;
            const float m_new = !need ? m_ref : (m_ref == -INFINITY ? mx : m_ref + k);
            const float alpha = need ? (m_ref == -INFINITY ? 0.0f : ldexpf(1.0f, -(int)k)) : 1.0f;
            if (c > 0) {
              // O holds earlier chunks: rescale it once P . V(c - 1) is done
              if (!warp_wait(smem_addr(&o_done[tile]), (c - 1) & 1)) {
                ok = false;
                break;
              }
              tc_fence_after();
#pragma unroll 1
              for (int c0 = 0; c0 < D; c0 += 16) {
                uint32_t ov[16];
                tmem_ld16(o_tmem + c0, ov);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
                tmem_st16(o_tmem + c0, ov);
              }
            }
            if (ps > 0) {
              // this chunk's first half of P went out under the old reference
              tmem_wait_st();
#pragma unroll 1
              for (int c0 = 0; c0 < 32; c0 += 16) {
                uint32_t pv[16];
                tmem_ld16(s_tmem + c0, pv);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) pv[j] = scale_pair<kQ8>(pv[j], alpha);
                tmem_st16(s_tmem + c0, pv);
              }
              lsum *= alpha;
            }
            tmem_wait_st();
            l *= alpha;
            m_ref = m_new;
          }
          const float zero_ref = m_ref == -INFINITY ? 0.0f : m_ref;
          uint32_t pw[kH][16];
          lsum += masked ? chunk_exp<true, kQ8>(raw, pw, first, lim, sl2c, zero_ref, vf)
                         : chunk_exp<false, kQ8>(raw, pw, first, lim, sl2c, zero_ref, vf);
          // P (16-bit pairs) of these 64 keys: packed columns [32 ps, 32 ps + 32)
#pragma unroll
          for (int h = 0; h < kH; ++h) tmem_st16(s_tmem + 32 * ps + 16 * h, pw[h]);
        }
        if (!ok) break;
        tmem_wait_st();
        l += lsum;
        tc_fence_before();
        mbar_arrive(smem_addr(&p_full[tile]));
      }
      if (ok && nch > 0 && !warp_wait(smem_addr(&o_done[tile]), (nch - 1) & 1)) ok = false;
      if (!ok) sh_fail = 1;
      tc_fence_after();
    }
  }
  __syncthreads();
  const bool failed = bad || sh_fail != 0 || !len_ok;
  if (work && !bad && warp == kMmaWarp && lane == 0) {
    // all tensor-core work of this CTA completes before TMEM is read or freed
    tc_fence_after();
    mma_commit(smem_addr(&drain_bar));
    if (!mbar_wait(smem_addr(&drain_bar), 0)) sh_fail = 1;
  }
  __syncthreads();
  if (bad && tid == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_BLOCK);
  if (sh_fail && tid == 0) atomicOr(a.flags, PAGEDKV_FLAG_WAIT_TIMEOUT);
  if (!len_ok && tid == 0 && pr == 0 && hk == 0 && part == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_SEQ_LEN);

  // ---- epilogue: this thread's row (TMEM read by whole warps)
  if (warp < kSoftmaxWarps && (tile == 0 || live1) && rows_ok) {
    const bool mine_row = r < rows_b;
    const int64_t orow = mine_row ? (int64_t)(q0 + r / GQ) * Hq + (int64_t)hk * GQ + r % GQ : 0;
    const bool split = kPrefix || a.max_parts > 1;
    const uint32_t o_tmem = tm + ((uint32_t)(32 * (warp & 3)) << 16) + T::ocol(tile);
    const bool have = work && !failed;                   // CTA-uniform
    // 8-bit pools: P carried V scales relative to the partition's largest
    const float oscale = kQ8 ? (sh_vmax > 0.0f ? sh_vmax : 1.0f) : 1.0f;
    const float inv = (have && l > 0.0f) ? oscale / l : 0.0f;
    // prefix partials sit after the row's max_parts decode partitions
    const int64_t slot = kPrefix ? orow * a.slots + a.max_parts + part : orow * a.max_parts + part;
    if (split && mine_row) {
      a.ws_ml[2 * slot] = m_ref;
      a.ws_ml[2 * slot + 1] = failed ? -1.0f : (have ? l : 0.0f);
    }
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t ov[32];
      if (have) {
        tmem_ld32(o_tmem + c0, ov);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] = 0u;
      }
      if (!mine_row) continue;
      if (!split) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + orow * D + c0;
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(ov[j + 2 * e]) * inv,
                                                     __uint_as_float(ov[j + 2 * e + 1]) * inv);
            w[e] = *reinterpret_cast<uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(out + j) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        float* acc = a.ws_acc + slot * D + c0;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(acc + j) =
              make_float4(__uint_as_float(ov[j]) * oscale, __uint_as_float(ov[j + 1]) * oscale,
                          __uint_as_float(ov[j + 2]) * oscale, __uint_as_float(ov[j + 3]) * oscale);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every copy, MMA and arrival of this unit is done: the barriers start over
  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_inval(smem_addr(&k_full[s]));
      mbar_inval(smem_addr(&k_ready[s]));
      mbar_inval(smem_addr(&k_empty[s]));
      mbar_inval(smem_addr(&v_full[s]));
      mbar_inval(smem_addr(&v_ready[s]));
      mbar_inval(smem_addr(&v_empty[s]));
    }
    for (int g = 0; g < kTiles; ++g) {
      mbar_inval(smem_addr(&s_full[g]));
      mbar_inval(smem_addr(&p_full[g]));
      mbar_inval(smem_addr(&o_done[g]));
    }
    mbar_inval(smem_addr(&drain_bar));
  }
  }  // units
  tc_fence_before();
  __syncthreads();
  if (tm_held && warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(kTmemCols)
                 : "memory");
}


template <int D, int BS, bool kPrefix, int kKind>
kv_status launch_tc(const DecodeArgs& a, int ctas, cudaStream_t s) {
  using T = TcGeo<D>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  kv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != KV_OK) return st;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
      st = cuda_check(cudaFuncSetAttribute(multi_tc_kernel<D, BS, kPrefix, kKind>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes),
                      "cudaFuncSetAttribute(multi_tc_kernel)");
      if (st != KV_OK) return st;
      attr_set[dev] = true;
    }
  }
  CUtensorMap km, vm;
  if ((st = make_kv_maps(a, &km, &vm)) != KV_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = T::kSmemBytes;
  cfg.stream = s;
  return cuda_check(cudaLaunchKernelEx(&cfg, multi_tc_kernel<D, BS, kPrefix, kKind>, km, vm, a),
                    "multi_tc_kernel launch");
}

template <bool kPrefix, int kKind>
kv_status launch_tc_geo(const DecodeArgs& a, int ctas, cudaStream_t s) {
  if (a.head_dim == 128)
    return a.block_size == 32 ? launch_tc<128, 32, kPrefix, kKind>(a, ctas, s)
                              : launch_tc<128, 16, kPrefix, kKind>(a, ctas, s);
  return a.block_size == 32 ? launch_tc<64, 32, kPrefix, kKind>(a, ctas, s)
                            : launch_tc<64, 16, kPrefix, kKind>(a, ctas, s);
}

template <bool kPrefix>
kv_status launch_tc_kind(const DecodeArgs& a, int ctas, cudaStream_t s) {
  if (a.dtype == KV_DTYPE_INT8) return launch_tc_geo<kPrefix, KV_DTYPE_INT8>(a, ctas, s);
  if (a.dtype == KV_DTYPE_FP8_E4M3) return launch_tc_geo<kPrefix, KV_DTYPE_FP8_E4M3>(a, ctas, s);
  return launch_tc_geo<kPrefix, KV_DTYPE_BF16>(a, ctas, s);
}

}  // namespace

kv_status launch_multi_tc(const DecodeArgs& a, int ctas, cudaStream_t s) {
  if (a.part_tokens > kMaxPartTokens || a.part_tokens % kChunk || ctas <= 0)
    return fail(KV_ERR_INVALID_ARG, "paged_attention_multi: bad tensor-core launch");
  return launch_tc_kind<false>(a, ctas, s);
}

kv_status launch_prefix_tc(const DecodeArgs& a, int ctas, cudaStream_t s) {
  if (a.prefix_part_tokens <= 0 || a.prefix_part_tokens > kMaxPartTokens ||
      a.prefix_part_tokens % kChunk || a.prefix_chunks < 1 ||
      (int64_t)a.prefix_chunks * a.prefix_part_tokens < (int64_t)a.num_prefix_blocks * a.block_size ||
      (int64_t)(a.prefix_chunks - 1) * a.prefix_part_tokens >= (int64_t)a.num_prefix_blocks * a.block_size ||
      ctas <= 0)
    return fail(KV_ERR_INVALID_ARG, "shared prefix: bad tensor-core launch");
  return launch_tc_kind<true>(a, ctas, s);
}

}  // namespace pagedkv
