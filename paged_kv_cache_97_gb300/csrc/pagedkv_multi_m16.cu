// pagedkv_multi_m16.cu -- few-token multi-token queries with the (query
// token, grouped head) columns on the MMA's M side, 16 per m-tile (speculative
// verification, “让 Agent 跑得快：LLM 推理服务”, §六 投机解码: the target model
// scores the draft tokens in one parallel pass).
//
// Sequence b's query token i (of n_b, its last tokens) sits at position
// L_b - n_b + i and attends positions 0 .. L_b - n_b + i.  This kernel takes
// the sequences whose n_b is too large for one 8-column group of the decode
// kernel's multi-token mode (8 / G tokens) but small enough for its column
// path (at most 4 x 8 / G tokens).  An m-tile holds 16 / G query tokens times
// the G heads; a CTA serves one (KV head, sequence, token partition) and MT
// m-tiles: MT = 1 when every sequence fits 16 columns, else MT = 2, which
// covers every sequence of the path in one CTA.  With the columns on M
// (mma.sync m16n8k16, bf16, fp32 accumulate):
//   S[16 cols x 16 keys] = Q[16 x d] . K^T   (B = K rows by ldmatrix)
//   O[16 cols x d]      += P[16 x 16] . V    (B = V rows by ldmatrix.trans)
// P is packed straight from the S accumulators (the fragment of S for keys
// 0-7 and 8-15 is the A fragment of P), so no shuffles move it, and every K
// and V fragment read from shared memory serves 16 columns instead of 8.
// Each column keeps its own causal limit; the online softmax (“LLM 推理优化
// 技术全景”, 在线 Softmax; “Flash Attention v2 的改进”: deferred
// normalisation) runs per column in base 2.  Lane 4g + t holds columns g and
// g + 8 (its S and O rows), so the softmax state of a column lives in the
// four lanes that hold its scores.
//
// The pipeline is the decode kernel's: a producer warp walks the partition's
// blocks and issues TMA tensor loads of K and V into an mbarrier ring; each
// block of a stage is taken by one consumer warp per m-tile (so a block is
// loaded once for all the sequence's columns), and the warps then combine
// through shared memory and write the output (one partition) or (m, l, acc)
// partials that the multi-token merge combines.  Every wait is bounded.
// bf16 pools.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv_common.cuh"
#include "pagedkv_device.cuh"

namespace pagedkv {
namespace {

using namespace dev;

constexpr int kCols = 16;                                // query columns per m-tile (the MMA's M)
constexpr int kMaxBlocks = kMaxColumnPartTokens / 16;    // blocks per partition (max)
// Threads of a CTA with MT m-tiles: kConsumers warps per m-tile + one
// producer warp.
template <int MT>
constexpr int kThreadsOf = (kConsumers * MT + 1) * 32;
// Batches of up to this many sequences may be taken longest first.
constexpr int kRankMax = 128;

// One TMA request for a whole d128 K or V block of one head: a 5-D map
// (d mod 64, row, d / 64, head, block) whose box holds both 64-element halves
// of every row, laid out as two [bs][128 B] swizzled halves (the layout of
// two 4-D boxes).  Each request carries a fixed cost in the SM's TMA unit,
// which 2 KB boxes (two requests per K or V block) made the loads' limit.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %2, %2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(c3), "r"(c4), "r"(bar)
      : "memory");
}

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared memory of a CTA.  MT = 1: a stage ring of up to 72 KB (three
// stages of three bf16 d128 16-row blocks), Q in registers: three CTAs fit
// an SM's 228 KB, and with two stages in flight per CTA the loads cover the
// time the consumers take per stage.  MT = 2: up to 100 KB of ring and the
// Q tile (rows padded by 16 bytes, so ldmatrix reads it without bank
// conflicts): two CTAs per SM, their registers freed of Q.
template <int D, int BS, int MT>
struct Ring {
  using G = Geo<D, BS, false>;
  static constexpr int kStages0 = (MT == 1 ? 72 * 1024 : 100 * 1024) / G::kStageBytes;
  static constexpr int kStages = kStages0 < 2 ? 2 : (kStages0 > kMaxStages ? kMaxStages : kStages0);
  static constexpr int kRingBytes = kStages * G::kStageBytes;
  static constexpr int kQRow = (D + 8) * 2;                             // bytes per Q row
  static constexpr int kQBytes = MT == 1 ? 0 : MT * kCols * kQRow;
  static constexpr int kSmemBytes = kRingBytes + kQBytes + 1024;       // + alignment slack
  // CTAs per SM that shared memory admits (1 KB reserved per CTA and a
  // little static memory): the register budget's divisor
  static constexpr int kWant = MT == 1 ? 3 : 2;
  static constexpr int kMinCtas = kWant * (kSmemBytes + 2048) <= 228 * 1024 ? kWant : kWant - 1;
  // the combine buffers reuse the ring
  static_assert((2 * kConsumers * MT * kCols + kConsumers * MT * kCols * D) * 4 <= kRingBytes,
                "combine buffers exceed the stage ring");
};

template <int D, int BS, int MT>
__global__ void __launch_bounds__(kThreadsOf<MT>, Ring<D, BS, MT>::kMinCtas)
    multi_m16_kernel(const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap v_map, const DecodeArgs a, int n_lo,
                     int vgroups, int rank) {
  using G = Geo<D, BS, false>;
  using R = Ring<D, BS, MT>;
  constexpr int S = R::kStages;
  constexpr int kThreads = kThreadsOf<MT>;
  constexpr int kWarpsC = kConsumers * MT;                // consumer warps
  constexpr int kColsC = kCols * MT;                      // columns of the CTA
  constexpr int kSpec = (kMaxBlocks + kThreads - 1) / kThreads;
  constexpr int kKSteps = D / 16;                         // k-steps of S over d
  constexpr int kDBlocks = D / 8;                         // 8-wide d blocks of O
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ int cta_bad, cta_timeout;
  __shared__ int rank_len[kRankMax];
  __shared__ int rank_seq;

  const int hk = blockIdx.x;
  const int part = a.reverse_parts ? (int)(gridDim.z - 1 - blockIdx.z) : (int)blockIdx.z;
  const int vg = (int)(blockIdx.y % vgroups);
  int b = (int)(blockIdx.y / vgroups);
  if (rank) {
    // Longest sequences first: CTA row r takes the sequence of rank r by
    // (length descending, index ascending), so that the last wave holds the
    // short ones (with one partition per sequence, CTA lengths differ
    // several-fold).  The ranks are a permutation: every sequence is taken
    // exactly once.
    const int r = b;
    for (int i = threadIdx.x; i < a.batch; i += kThreads) rank_len[i] = a.seq_lens[i];
    __syncthreads();
    for (int i = threadIdx.x; i < a.batch; i += kThreads) {
      const int li = rank_len[i];
      int ri = 0;
      for (int k = 0; k < a.batch; ++k) {
        const int lk = rank_len[k];
        ri += (lk > li || (lk == li && k < i)) ? 1 : 0;
      }
      if (ri == r) rank_seq = i;
    }
    __syncthreads();
    b = rank_seq;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  const int GQ = Hq / Hkv;                               // grouped query heads (1..8)
  const int TPG = kCols / GQ;                            // query tokens per m-tile
  const int tok0 = vg * MT * TPG;                        // the CTA's first query token
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);

  // This kernel's sequences: n > n_lo (the decode kernel takes the shorter
  // ones; it runs only in calls without long queries, so a sequence above
  // col_max_n is above max_query_len too, and flagged below).
  const int q0 = a.query_start[b];
  const int nq = a.query_start[b + 1] - q0;
  if (nq <= n_lo) return;
  const bool rows_ok = q0 >= 0 && nq >= 0 && q0 + nq <= a.num_tokens;
  // Row of the q / out tensors that column c (m-tile c / 16) serves (-1:
  // padding): token tok0 + (c / 16) TPG + (c % 16) / GQ of the sequence, head
  // (c % 16) % GQ of the group.
  auto col_row = [&](int c) -> int64_t {
    const int cc = c % kCols;
    const int i = tok0 + (c / kCols) * TPG + cc / GQ;
    return (rows_ok && cc < TPG * GQ && i < nq) ? (int64_t)(q0 + i) * Hq + (int64_t)hk * GQ + cc % GQ
                                                  : -1;
  };

  // Block ids of the partition and the consumers' Q fragments are loaded
  // before the sequence length arrives (neither depends on it).
  const int t0 = part * a.part_tokens;
  const int first_blk = t0 / BS;
  const int spec_blk = min(a.part_tokens / BS, a.max_blocks_per_seq - first_blk);
  const int32_t* bt = a.block_tables + (int64_t)b * a.max_blocks_per_seq + first_blk;
  int32_t spec_id[kSpec];
#pragma unroll
  for (int r = 0; r < kSpec; ++r) {
    const int j = threadIdx.x + r * kThreads;
    spec_id[r] = j < spec_blk ? bt[j] : -1;
  }
  // Q: A fragments (rows = columns g and g + 8, k = d): a0 = (g, 2t..2t+1),
  // a1 = (g + 8, 2t..), a2 = (g, 2t + 8..), a3 = (g + 8, 2t + 8..) of each
  // 16-wide k-step; padding columns are zero.  MT = 1: in registers; MT = 2:
  // 16-byte pieces of the Q rows, stored to the shared Q tile after the
  // checks and read by ldmatrix per k-step.
  const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q);
  constexpr int kQPieces = kColsC * D / 8;                // 16-byte pieces of the Q tile
  constexpr int kQPer = MT == 1 ? 1 : (kQPieces + kThreads - 1) / kThreads;
  uint32_t qa[MT == 1 ? kKSteps : 1][4];
  uint4 qpiece[kQPer];
  if constexpr (MT == 1) {
    if (warp < kWarpsC) {
      const int64_t r0 = col_row(g), r1 = col_row(g + 8);
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks) {
        const int d0 = 16 * ks + 2 * t;
        qa[ks][0] = r0 >= 0 ? *reinterpret_cast<const uint32_t*>(qb + r0 * D + d0) : 0u;
        qa[ks][1] = r1 >= 0 ? *reinterpret_cast<const uint32_t*>(qb + r1 * D + d0) : 0u;
        qa[ks][2] = r0 >= 0 ? *reinterpret_cast<const uint32_t*>(qb + r0 * D + d0 + 8) : 0u;
        qa[ks][3] = r1 >= 0 ? *reinterpret_cast<const uint32_t*>(qb + r1 * D + d0 + 8) : 0u;
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < kQPer; ++r) {
      const int i = threadIdx.x + r * kThreads;
      const int64_t row = i < kQPieces ? col_row(i / (D / 8)) : -1;
      qpiece[r] = row >= 0 ? *reinterpret_cast<const uint4*>(qb + row * D + (i % (D / 8)) * 8)
                           : make_uint4(0u, 0u, 0u, 0u);
    }
  }

  // ---- sequence checks (uniform over the CTA) -----------------------------
  const int L = a.seq_lens[b];
  const int64_t table_tokens = (int64_t)a.max_blocks_per_seq * BS;
  const bool len_bad = L <= 0 || L > a.max_seq_len || L > table_tokens || !rows_ok || nq > L ||
                       nq > a.max_query_len;
  if (len_bad) {
    if (part == 0) {
      if (threadIdx.x == 0 && vg == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_SEQ_LEN);
      // (with several partitions, the multi-token merge zeroes these rows)
      if (a.max_parts == 1)
        for (int i = threadIdx.x; i < kColsC * D; i += blockDim.x) {
          const int64_t r = col_row(i / D);
          if (r >= 0) out[r * D + i % D] = __float2bfloat16_rn(0.0f);
        }
    }
    return;
  }
  if (tok0 >= nq) return;                                // a group with no queries
  if (t0 >= L) return;
  // keys up to the CTA's last query position
  int t1 = min(t0 + a.part_tokens, L);
  t1 = min(t1, L - nq + min(nq - 1, tok0 + MT * TPG - 1) + 1);
  const bool direct = a.max_parts == 1;
  if (t1 <= t0) {
    // every query of this CTA precedes the partition: empty partials
    for (int i = threadIdx.x; i < kColsC * D; i += blockDim.x) {
      const int64_t r = col_row(i / D);
      if (r < 0) continue;
      const int64_t sl = r * a.slots + part;
      a.ws_acc[sl * D + i % D] = 0.0f;
      if (i % D == 0) {
        a.ws_ml[2 * sl] = -INFINITY;
        a.ws_ml[2 * sl + 1] = 0.0f;
      }
    }
    return;
  }
  const int nblk = (t1 - 1) / BS - first_blk + 1;        // >= 1, <= spec_blk
  const uint32_t stages = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t qtile = stages + R::kRingBytes;           // MT = 2: [MT x 16][kQRow]
  if constexpr (MT > 1) {
#pragma unroll
    for (int r = 0; r < kQPer; ++r) {
      const int i = threadIdx.x + r * kThreads;
      if (i < kQPieces) {
        const uint32_t dst = qtile + (uint32_t)((i / (D / 8)) * R::kQRow + (i % (D / 8)) * 16);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(qpiece[r].x),
                     "r"(qpiece[r].y), "r"(qpiece[r].z), "r"(qpiece[r].w)
                     : "memory");
      }
    }
  }

  // ---- set-up: barriers, and a check of the partition's block ids ---------
  if (threadIdx.x == 0) {
    cta_bad = 0;
    cta_timeout = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kWarpsC);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kSpec; ++r) {
    const int j = threadIdx.x + r * kThreads;
    if (j >= nblk) continue;
    const int32_t p = spec_id[r];
    if (p < 0 || p >= a.num_blocks) cta_bad = 1;
  }
  __syncthreads();
  const bool bad = cta_bad != 0;
  const int n_iter = (nblk + kConsumers - 1) / kConsumers;

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};   // columns g, g + 8
  float o[kDBlocks][4];
#pragma unroll
  for (int i = 0; i < kDBlocks; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;

  if (!bad && warp == kWarpsC) {
    // ======================= producer =======================================
    // Block ids 32 at a time, lane l holding block 32 k + l of chunk k (the
    // ids were checked above; the table is read again here, from L2, with
    // the next chunk always in flight).
    auto chunk_id = [&](int k) -> int32_t {
      const int j = 32 * k + lane;
      return j < nblk ? bt[j] : 0;
    };
    int32_t id_cur = chunk_id(0), id_nxt = chunk_id(1);
    int k_cur = 0;
    int issued = 0;
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % S;
      if (it >= S && !mbar_wait(smem_addr(&empty_bar[s]), ((it / S) - 1) & 1)) {
        ok = false;
        break;
      }
      const int j0 = it * kConsumers;
      const int cnt = min(kConsumers, nblk - j0);
      const uint32_t fb = smem_addr(&full_bar[s]);
      if (lane == 0) mbar_expect_tx(fb, (uint32_t)(cnt * G::kBlockBytes));
      for (int c = 0; c < cnt; ++c) {
        const int j = j0 + c;
        if ((j >> 5) != k_cur) {                           // next chunk (warp-uniform)
          id_cur = id_nxt;
          ++k_cur;
          id_nxt = chunk_id(k_cur + 1);
        }
        int32_t p = __shfl_sync(0xffffffffu, id_cur, j & 31);
        p = (p >= 0 && p < a.num_blocks) ? p : 0;
        if (lane == 0) {
          const uint32_t kdst = stages + (uint32_t)((s * kConsumers + c) * G::kBlockBytes);
          const uint32_t vdst = kdst + G::kTensorBytes;
          if constexpr (D == 128) {
            tma_load_5d(kdst, &k_map, fb, hk, p);
            tma_load_5d(vdst, &v_map, fb, hk, p);
          } else {
            tma_load_4d(kdst, &k_map, fb, 0, hk, 0, p);
            tma_load_4d(vdst, &v_map, fb, 0, hk, 0, p);
          }
        }
      }
      __syncwarp();
      issued = it + 1;
    }
    // every fill issued lands before the CTA may reuse or release the stages
    for (int s = 0; s < S && s < issued; ++s) {
      const int last = s + S * ((issued - 1 - s) / S);
      if (!mbar_wait(smem_addr(&full_bar[s]), (last / S) & 1)) ok = false;
    }
    if (!ok && lane == 0) cta_timeout = 1;
  } else if (!bad) {
    // ======================= consumers =====================================
    // warp = mt * kConsumers + w: block w of every stage, columns of m-tile mt
    const int w = warp % kConsumers, mt = warp / kConsumers;
    const float kfac = a.scale_log2;
    // causal limits of this lane's columns g and g + 8 (padding: no limit),
    // and the m-tile's first query position: a block whose last key is at or
    // before it is visible to every column
    const int pos_lo = L - nq + tok0 + mt * TPG;
    const int cpos0 = g < TPG * GQ ? pos_lo + g / GQ : 0x7fffffff;
    const int cpos1 = g + 8 < TPG * GQ ? pos_lo + (g + 8) / GQ : 0x7fffffff;
    // ldmatrix row addresses inside a block (the same for K and V): matrix
    // q = lane / 8 covers keys 8 (q & 1) .. + 7 and 16-byte chunk
    // 2 ks + (q >> 1); the next 16-key tile is 16 rows further on
    uint32_t off[kKSteps];
    {
      const int row = ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks) off[ks] = chunk_off<G>(row, 2 * ks + (lane >> 4));
    }
    // MT = 2: this lane's ldmatrix row of the m-tile's Q (matrix q = lane / 8
    // covers columns 8 (q & 1) .. + 7 and d 8 (q >> 1) .. + 7 of a k-step)
    const uint32_t qrow = qtile + (uint32_t)((mt * kCols + ((lane >> 3) & 1) * 8 + (lane & 7)) * R::kQRow +
                                             (lane >> 4) * 16);
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % S;
      if (!mbar_wait(smem_addr(&full_bar[s]), (it / S) & 1)) {
        ok = false;
        break;
      }
      const int j = it * kConsumers + w;
      if (j < nblk) {
        const uint32_t kb = stages + (uint32_t)((s * kConsumers + w) * G::kBlockBytes);
        const uint32_t vb = kb + G::kTensorBytes;
        const int key0 = (first_blk + j) * BS;             // position of the block's first row
        const int valid = min(BS, L - key0);
        // interior block: every row written and visible to every column
        const bool plain = valid == BS && key0 + BS - 1 <= pos_lo;

        // ---- S for every 16-key tile: sc[tile][nb][...] for keys 8 nb + 2t, +1
        // (r0 / r2 = keys 0-7, d low / high: B of n-block 0; r1 / r3 = keys
        // 8-15: B of n-block 1; with one tile per block, even and odd k-steps
        // accumulate apart, which halves the dependent MMA chains)
        constexpr int kSplit = G::kTiles == 1 ? 2 : 1;
        float sc[G::kTiles][2][4];
#pragma unroll
        for (int tile = 0; tile < G::kTiles; ++tile) {
          float c[2 * kSplit][4] = {};
#pragma unroll
          for (int ks = 0; ks < kKSteps; ++ks) {
            uint32_t r[4];
            ldsm_x4(r, kb + off[ks] + tile * 16 * G::kBoxRow);
            if constexpr (MT == 1) {
              mma16816<false>(c[ks % kSplit], qa[ks], r[0], r[2]);
              mma16816<false>(c[kSplit + ks % kSplit], qa[ks], r[1], r[3]);
            } else {
              uint32_t qf[4];
              ldsm_x4(qf, qrow + ks * 32);
              mma16816<false>(c[ks % kSplit], qf, r[0], r[2]);
              mma16816<false>(c[kSplit + ks % kSplit], qf, r[1], r[3]);
            }
          }
#pragma unroll
          for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float x = c[kSplit * nb][e];
              if constexpr (kSplit == 2) x += c[kSplit * nb + 1][e];
              sc[tile][nb][e] = x * kfac;
            }
          if (!plain) {
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
              const int k0 = tile * 16 + 8 * nb + 2 * t;   // key row in the block
              const bool v0 = k0 < valid, v1 = k0 + 1 < valid;
              if (!(v0 && key0 + k0 <= cpos0)) sc[tile][nb][0] = -INFINITY;
              if (!(v1 && key0 + k0 + 1 <= cpos0)) sc[tile][nb][1] = -INFINITY;
              if (!(v0 && key0 + k0 <= cpos1)) sc[tile][nb][2] = -INFINITY;
              if (!(v1 && key0 + k0 + 1 <= cpos1)) sc[tile][nb][3] = -INFINITY;
            }
          }
        }

        // ---- online softmax update of columns g (index 0) and g + 8 (1) ----
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int tile = 0; tile < G::kTiles; ++tile)
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            mx0 = fmaxf(mx0, fmaxf(sc[tile][nb][0], sc[tile][nb][1]));
            mx1 = fmaxf(mx1, fmaxf(sc[tile][nb][2], sc[tile][nb][3]));
          }
#pragma unroll
        for (int o2 = 1; o2 < 4; o2 <<= 1) {              // the quad holding the column
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
        }
        const float mx0n = fmaxf(m_run[0], mx0), mx1n = fmaxf(m_run[1], mx1);
        // a column with no key yet keeps m = -inf: subtract 0 then
        const float mn0 = mx0n == -INFINITY ? 0.0f : mx0n;
        const float mn1 = mx1n == -INFINITY ? 0.0f : mx1n;
        // O is rescaled only when some column's maximum moved (warp-uniform)
        if (__any_sync(0xffffffffu, mx0n != m_run[0] || mx1n != m_run[1])) {
          const float al0 = ex2(m_run[0] - mn0), al1 = ex2(m_run[1] - mn1);
          l_run[0] *= al0;
          l_run[1] *= al1;
#pragma unroll
          for (int i = 0; i < kDBlocks; ++i) {
            o[i][0] *= al0;
            o[i][1] *= al0;
            o[i][2] *= al1;
            o[i][3] *= al1;
          }
        }
        m_run[0] = mx0n;
        m_run[1] = mx1n;

#pragma unroll
        for (int tile = 0; tile < G::kTiles; ++tile) {
          if (tile * 16 >= valid) break;                  // whole tile masked
          float p[2][4];
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            p[nb][0] = ex2(sc[tile][nb][0] - mn0);
            p[nb][1] = ex2(sc[tile][nb][1] - mn0);
            p[nb][2] = ex2(sc[tile][nb][2] - mn1);
            p[nb][3] = ex2(sc[tile][nb][3] - mn1);
            l_run[0] += p[nb][0] + p[nb][1];
            l_run[1] += p[nb][2] + p[nb][3];
          }
          // A fragment of P: (g, keys 2t..), (g + 8, 2t..), (g, 2t + 8..), (g + 8, 2t + 8..)
          const uint32_t pa[4] = {pack2<false>(p[0][0], p[0][1]), pack2<false>(p[0][2], p[0][3]),
                                  pack2<false>(p[1][0], p[1][1]), pack2<false>(p[1][2], p[1][3])};
          // ldmatrix.x4.trans over the same rows: r0 / r1 = b0 / b1 of
          // d-block 2 jj, r2 / r3 of d-block 2 jj + 1
          if (valid == BS) {
#pragma unroll
            for (int jj = 0; jj < kDBlocks / 2; ++jj) {
              uint32_t r[4];
              ldsm_x4_t(r, vb + off[jj] + tile * 16 * G::kBoxRow);
              mma16816<false>(o[2 * jj], pa, r[0], r[1]);
              mma16816<false>(o[2 * jj + 1], pa, r[2], r[3]);
            }
          } else {
            // V rows past `valid` are zeroed in the B fragments (keys 2t,
            // 2t+1 in b0, 2t+8, 2t+9 in b1): p is 0 there, but the pool may
            // hold NaN
            const int k0 = tile * 16 + 2 * t;
            const uint32_t mlo = (k0 < valid ? 0x0000ffffu : 0u) | (k0 + 1 < valid ? 0xffff0000u : 0u);
            const uint32_t mhi = (k0 + 8 < valid ? 0x0000ffffu : 0u) | (k0 + 9 < valid ? 0xffff0000u : 0u);
#pragma unroll
            for (int jj = 0; jj < kDBlocks / 2; ++jj) {
              uint32_t r[4];
              ldsm_x4_t(r, vb + off[jj] + tile * 16 * G::kBoxRow);
              mma16816<false>(o[2 * jj], pa, r[0] & mlo, r[1] & mhi);
              mma16816<false>(o[2 * jj + 1], pa, r[2] & mlo, r[3] & mhi);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
    }
    if (!ok) cta_timeout = 1;
  }

  // ---- combine the consumer warps -----------------------------------------
  __syncthreads();  // all fills landed and all stage reads done
  const bool failed = bad || cta_timeout != 0;
  float* red = reinterpret_cast<float*>(smem_raw + (stages - smem_addr(smem_raw)));
  float* red_m = red;                              // [kWarpsC][kCols]
  float* red_l = red + kWarpsC * kCols;            // [kWarpsC][kCols]
  float* red_acc = red + 2 * kWarpsC * kCols;      // [kWarpsC][kCols][D]
  if (!failed && warp < kWarpsC) {
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
      l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
    }
    if (t == 0) {
      red_m[warp * kCols + g] = m_run[0];
      red_m[warp * kCols + g + 8] = m_run[1];
      red_l[warp * kCols + g] = l_run[0];
      red_l[warp * kCols + g + 8] = l_run[1];
    }
    float* acc = red_acc + warp * kCols * D;
#pragma unroll
    for (int i = 0; i < kDBlocks; ++i) {
      const int d0 = 8 * i + 2 * t;
      acc[g * D + d0] = o[i][0];
      acc[g * D + d0 + 1] = o[i][1];
      acc[(g + 8) * D + d0] = o[i][2];
      acc[(g + 8) * D + d0 + 1] = o[i][3];
    }
  }
  __syncthreads();

  if (failed) {
    if (threadIdx.x == 0)
      atomicOr(a.flags, bad ? PAGEDKV_FLAG_BAD_BLOCK : PAGEDKV_FLAG_WAIT_TIMEOUT);
    for (int i = threadIdx.x; i < kColsC * D; i += blockDim.x) {
      const int c = i / D, e = i % D;
      const int64_t row = col_row(c);
      if (row < 0) continue;
      if (direct) {
        out[row * D + e] = __float2bfloat16_rn(0.0f);
      } else {
        const int64_t r = row * a.slots + part;
        a.ws_acc[r * D + e] = 0.0f;
        if (e == 0) {
          a.ws_ml[2 * r] = 0.0f;
          a.ws_ml[2 * r + 1] = -1.0f;  // marks the row bad for the merge
        }
      }
    }
    return;
  }

  for (int i = threadIdx.x; i < kColsC * D; i += blockDim.x) {
    const int c = i / D, e = i % D;
    const int64_t row = col_row(c);
    if (row < 0) continue;
    // the m-tile's warps mt * kConsumers .. + kConsumers - 1, its column cc
    const int w0 = (c / kCols) * kConsumers, cc = c % kCols;
    float M = -INFINITY;
#pragma unroll
    for (int w = w0; w < w0 + kConsumers; ++w) M = fmaxf(M, red_m[w * kCols + cc]);
    const float Mz = M == -INFINITY ? 0.0f : M;    // a column with no key here
    float num = 0.0f, den = 0.0f;
#pragma unroll
    for (int w = w0; w < w0 + kConsumers; ++w) {
      const float f = exp2f(red_m[w * kCols + cc] - Mz);  // 0 for a warp that saw no key
      num = fmaf(f, red_acc[(w * kCols + cc) * D + e], num);
      den = fmaf(f, red_l[w * kCols + cc], den);
    }
    if (direct) {
      out[row * D + e] = __float2bfloat16_rn(num / den);
    } else {
      const int64_t r = row * a.slots + part;
      a.ws_acc[r * D + e] = num;
      if (e == 0) {
        a.ws_ml[2 * r] = M;
        a.ws_ml[2 * r + 1] = den;
      }
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The 5-D map of tma_load_5d over a bf16 d128 pool [NB, bs, Hkv, 128]:
// dims (64, bs, 2, Hkv, NB) with byte strides (row, 128, head, block).
kv_status make_map5(CUtensorMap* map, const void* pool, const DecodeArgs& a) {
  auto fn = encode_fn();
  if (!fn) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  const cuuint64_t head_bytes = 128 * 2, row_bytes = (cuuint64_t)a.num_kv_heads * head_bytes;
  const cuuint64_t dims[5] = {64, (cuuint64_t)a.block_size, 2, (cuuint64_t)a.num_kv_heads,
                              (cuuint64_t)a.num_blocks};
  const cuuint64_t strides[4] = {row_bytes, 128, head_bytes, row_bytes * a.block_size};
  const cuuint32_t box[5] = {64, (cuuint32_t)a.block_size, 2, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(pool), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled (5-D) failed (%d)", (int)r);
  return KV_OK;
}

// Maps of this kernel: 5-D for d128, the shared 4-D maps for d64 (one
// 128-byte box per row already).  The 5-D maps are encoded once per (device,
// pools, geometry) and then served from a small cache.
kv_status m16_maps(const DecodeArgs& a, CUtensorMap* km, CUtensorMap* vm) {
  if (a.head_dim != 128) return make_kv_maps(a, km, vm);
  struct Entry {
    const void *k = nullptr, *v = nullptr;
    int device = -1, block_size = 0, num_kv_heads = 0, num_blocks = 0;
    CUtensorMap km, vm;
  };
  static std::mutex mu;
  static Entry cache[8];
  static int next = 0;
  int dev = 0;
  kv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != KV_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.device == dev && e.k == a.k_cache && e.v == a.v_cache && e.block_size == a.block_size &&
        e.num_kv_heads == a.num_kv_heads && e.num_blocks == a.num_blocks) {
      *km = e.km;
      *vm = e.vm;
      return KV_OK;
    }
  Entry& e = cache[next];
  e.device = -1;
  if ((st = make_map5(&e.km, a.k_cache, a)) != KV_OK || (st = make_map5(&e.vm, a.v_cache, a)) != KV_OK)
    return st;
  e.device = dev;
  e.k = a.k_cache;
  e.v = a.v_cache;
  e.block_size = a.block_size;
  e.num_kv_heads = a.num_kv_heads;
  e.num_blocks = a.num_blocks;
  next = (next + 1) % 8;
  *km = e.km;
  *vm = e.vm;
  return KV_OK;
}

template <int D, int BS, int MT>
kv_status launch_t(const DecodeArgs& a, int n_lo, int groups, int rank, cudaStream_t s) {
  using R = Ring<D, BS, MT>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  kv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != KV_OK) return st;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
      st = cuda_check(cudaFuncSetAttribute(multi_m16_kernel<D, BS, MT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           R::kSmemBytes),
                      "cudaFuncSetAttribute(multi_m16_kernel)");
      if (st != KV_OK) return st;
      attr_set[dev] = true;
    }
  }
  CUtensorMap km, vm;
  if ((st = m16_maps(a, &km, &vm)) != KV_OK) return st;
  const dim3 grid(a.num_kv_heads, a.batch * groups, a.max_parts);
  multi_m16_kernel<D, BS, MT><<<grid, kThreadsOf<MT>, R::kSmemBytes, s>>>(km, vm, a, n_lo, groups, rank);
  return cuda_check(cudaGetLastError(), "multi_m16_kernel launch");
}

// One m-tile per CTA when every sequence fits 16 columns (vgroups == 1),
// else two, which cover every sequence of the path (at most 4 x 8 / G
// tokens = 32 columns) in one CTA.
template <int D, int BS>
kv_status launch_mt(const DecodeArgs& a, int n_lo, int vgroups, int rank, cudaStream_t s) {
  if (vgroups == 1) return launch_t<D, BS, 1>(a, n_lo, 1, rank, s);
  return launch_t<D, BS, 2>(a, n_lo, (vgroups + 1) / 2, rank, s);
}

}  // namespace

// Few-token multi-token queries with n_lo < n_b <= a.col_max_n on 16-column
// m-tiles (bf16 pools); `vgroups` m-tiles per sequence at most; `rank`: take
// the sequences longest first (batches of up to kRankMax sequences).
kv_status launch_multi_m16(const DecodeArgs& a, int n_lo, int vgroups, bool rank, cudaStream_t s) {
  if (a.dtype != KV_DTYPE_BF16 || vgroups <= 0)
    return fail(KV_ERR_INVALID_ARG, "paged_attention_multi: bad 16-column launch");
  if ((int64_t)a.batch * vgroups > 65535 || a.max_parts > 65535)
    return fail(KV_ERR_INVALID_ARG, "batch x groups and the partition count must be at most 65535");
  if (a.part_tokens / a.block_size > kMaxBlocks || a.part_tokens % a.block_size)
    return fail(KV_ERR_INVALID_ARG, "partition must be a multiple of block_size, at most %d blocks",
                kMaxBlocks);
  const int rk = rank && a.batch <= kRankMax ? 1 : 0;
  if (a.head_dim == 128)
    return a.block_size == 32 ? launch_mt<128, 32>(a, n_lo, vgroups, rk, s)
                              : launch_mt<128, 16>(a, n_lo, vgroups, rk, s);
  return a.block_size == 32 ? launch_mt<64, 32>(a, n_lo, vgroups, rk, s)
                            : launch_mt<64, 16>(a, n_lo, vgroups, rk, s);
}

}  // namespace pagedkv
