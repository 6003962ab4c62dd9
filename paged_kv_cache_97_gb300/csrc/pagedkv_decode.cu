// pagedkv_decode.cu -- per-partition decode attention over a paged KV pool.
//
// One CTA serves one (token partition, KV head, sequence) and all G <= 8 query
// heads grouped on that KV head, so every K/V byte of the step is read from
// HBM once.  The CTA is a small producer/consumer pipeline:
//
//   * warp 4 (producer): one lane walks the partition's blocks in logical
//     order and issues TMA tensor loads (cp.async.bulk.tensor) of each block's
//     K and V rows for this KV head into a ring of shared-memory stages,
//     completing on per-stage mbarriers;
//   * warps 0..3 (consumers): consumer w takes block w of every stage and
//     runs the online-softmax recurrence (“LLM 推理优化技术全景”, 在线 Softmax:
//     m' = max(m, max S), l' = l e^(m-m') + sum e^(S-m'), O rescaled) on
//     tensor cores, in base 2 and with the division deferred to the end
//     (“Flash Attention v2 的改进”);
//   * finally the four consumers' (m, l, acc) are combined through shared
//     memory and the CTA writes either the normalised output (the sequence
//     has one partition) or its partial for the log-sum-exp merge kernel.
//
// Tensor-core formulation (mma.sync m16n8k16, fp32 accumulate), per 16-token
// tile of a block:
//   S^T[16 tokens x 8 heads] = K[16 x d] . Q^T[d x 8]      (A = K from smem)
//   O^T[d x 8 heads]        += V^T[d x 16] . P^T[16 x 8]   (A = V^T from smem)
// Heads sit on the N = 8 side, so G <= 8 grouped query heads cost one MMA
// column block; the padded heads carry q = 0 and are never written out.
// Lane l = 4g + t of a warp holds S^T rows (tokens) g, g+8 and columns
// (heads) 2t, 2t+1 -- the same heads as its O^T accumulator columns -- so the
// softmax state (m, l) of heads 2t and 2t+1 lives in the lane that rescales
// their accumulators.
//
// Multi-token queries (kMulti, paged_attention_multi with few query tokens
// per sequence: speculative verification, “让 Agent 跑得快”, §六): the 8 MMA
// columns of a CTA become (query token, grouped head) pairs -- 8 / G tokens
// of one sequence times its G heads, a "column group" -- each with its own
// causal limit (query i of n sits at position L - n + i and sees positions up
// to it).  The column groups of one (sequence, KV head, partition) are
// neighbouring CTAs, so their reads of the same blocks meet in L2.
//
// bf16 pools: K and V tiles come straight from the swizzled stage with
// ldmatrix (V transposed by ldmatrix.trans).  int8 pools: codes are read with
// 16-byte shared loads and widened to fp16 exactly (c + 128 placed in the
// mantissa of 1024.0, minus 1152); q is fp16 (scaled by a power of two when
// its magnitude needs it), the block's K scale multiplies the fp32 score and
// its V scale (relative to the CTA's largest) multiplies p.  Every pairing
// of d (or token) indices between the two MMA operands is the same on both
// sides, so each dot product sums the same terms as the plain definition.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv_common.cuh"
#include "pagedkv_device.cuh"

namespace pagedkv {
namespace {

using namespace dev;

constexpr int kThreads = (kConsumers + 1) * 32;      // + one producer warp
constexpr int kMaxBlocks = 8192 / 16;                // blocks per partition (max)
constexpr int kSpec = (kMaxBlocks + kThreads - 1) / kThreads;  // table entries per thread

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// kQ8: the pools hold 8-bit codes under per-(block, KV head) scales, int8
// or (kFp8) E4M3; otherwise bf16.
// 8-bit and multi-token instances may be held to 128 registers (4 CTAs of
// 4 warps per SM, the residency their shared memory allows).
#ifndef PAGEDKV_Q8_MIN_BLOCKS
#define PAGEDKV_Q8_MIN_BLOCKS 4
#endif
template <int D, int BS, bool kQ8, bool kFp8, bool kMulti>
__global__ void __launch_bounds__(kThreads, (kQ8 || kMulti) ? PAGEDKV_Q8_MIN_BLOCKS : 1)
    decode_kernel(const __grid_constant__ CUtensorMap k_map,
                  const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
  using G = Geo<D, BS, kQ8>;
  constexpr int S = G::kStages;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ int32_t blk_id[kMaxBlocks];
  __shared__ float blk_ks[kQ8 ? kMaxBlocks : 1], blk_vr[kQ8 ? kMaxBlocks : 1];
  __shared__ int cta_bad, cta_timeout;
  __shared__ float v_max_scale;

  // Grid (KV head, sequence, partition), partition slowest: every sequence's
  // first partitions launch first and the short last partitions of long
  // sequences launch last, which trims the tail; neighbouring heads of one
  // block run side by side.
  // (kMulti: blockIdx.y = sequence * vgroups + column group.)
  const int hk = blockIdx.x, part = a.reverse_parts ? (int)(gridDim.z - 1 - blockIdx.z) : (int)blockIdx.z;
  const int b = kMulti ? (int)(blockIdx.y / a.vgroups) : (int)blockIdx.y;
  const int vg = kMulti ? (int)(blockIdx.y % a.vgroups) : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;                 // MMA fragment coordinates
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
  const int GQ = Hq / Hkv;                               // grouped query heads (1..8)
  const int64_t head0 = (int64_t)b * Hq + (int64_t)hk * GQ;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  // Multi-token queries: the sequence's q rows [q0, q0 + nq), TPG tokens per
  // column group.
  int q0 = 0, nq = 1;
  if constexpr (kMulti) {
    q0 = a.query_start[b];
    nq = a.query_start[b + 1] - q0;
  }
  const int TPG = kMulti ? kMaxGroup / GQ : 1;
  if (kMulti && nq > a.col_max_n) return;                // a long query: the tensor-core kernel's
  const bool rows_ok = !kMulti || (q0 >= 0 && nq >= 0 && q0 + nq <= a.num_tokens);
  // Row of the q / out tensors that column c serves (-1: a padding column):
  // head c of the group, or (kMulti) token vg * TPG + c / GQ, head c % GQ.
  auto col_row = [&](int c) -> int64_t {
    if constexpr (kMulti) {
      const int i = vg * TPG + c / GQ;
      return (rows_ok && c < TPG * GQ && i < nq) ? (int64_t)(q0 + i) * Hq + (int64_t)hk * GQ + c % GQ
                                                   : -1;
    } else {
      return c < GQ ? head0 + c : -1;
    }
  };
  const int ncols = kMulti ? kMaxGroup : GQ;             // columns that may be written

  // This partition's block-table entries and the consumers' q fragments are
  // loaded before the sequence length arrives (neither depends on it), so
  // the start-up costs one round trip to memory instead of two.
  const int skip = a.skip_tokens;
  const int t0 = skip + part * a.part_tokens;
  const int first_blk = t0 / BS;
  const int spec_blk = min(a.part_tokens / BS, a.max_blocks_per_seq - first_blk);
  const int32_t* bt = a.block_tables + (int64_t)b * a.max_blocks_per_seq + first_blk;
  int32_t spec_id[kSpec];
#pragma unroll
  for (int r = 0; r < kSpec; ++r) {
    const int j = threadIdx.x + r * kThreads;
    spec_id[r] = j < spec_blk ? bt[j] : -1;
  }
  // Q^T fragments (B operand of S^T = K . Q^T): b0 = (k = 2t, 2t+1; n = g),
  // b1 = (k = 2t+8, 2t+9; n = g).  k indexes d: for bf16 the natural order
  // 16ks + k; for int8 the order in which each lane reads its own 16-byte
  // chunks of a K row (see the int8 K loads below).
  uint32_t qraw[G::kKSteps][2];
  if (warp < kConsumers) {
    const int64_t qrow = col_row(g);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + (qrow < 0 ? 0 : qrow) * D;
#pragma unroll
    for (int ks = 0; ks < G::kKSteps; ++ks) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        int d0;
        if constexpr (kQ8) {
          // lane t reads chunks t*NC .. t*NC+NC-1 (16 d each, NC = D/64)
          // of a row; k-step ks uses 4 consecutive d of chunk ks/4.
          constexpr int NC = D / 64;
          d0 = 16 * (t * NC + ks / 4) + 4 * (ks % 4) + 2 * r;
        } else {
          d0 = 16 * ks + 2 * t + 8 * r;
        }
        qraw[ks][r] = qrow >= 0 ? *reinterpret_cast<const uint32_t*>(q + d0) : 0u;
      }
    }
  }

  // ---- sequence checks (uniform over the CTA) -----------------------------
  const int L = a.seq_lens[b];
  const int64_t table_tokens = (int64_t)a.max_blocks_per_seq * BS;
  const bool len_bad = L <= a.skip_tokens || L > a.max_seq_len || L > table_tokens ||
                       (kMulti && (!rows_ok || nq > L || nq > a.max_query_len));
  if (len_bad) {
    if (part == 0) {
      if (threadIdx.x == 0 && vg == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_SEQ_LEN);
      // (with several partitions, the multi-token merge zeroes these rows)
      if (!kMulti || a.max_parts == 1)
        for (int i = threadIdx.x; i < ncols * D; i += blockDim.x) {
          const int64_t r = col_row(i / D);
          if (r >= 0) out[r * D + i % D] = __float2bfloat16_rn(0.0f);
        }
    }
    return;
  }
  if (kMulti && vg * TPG >= nq) return;                  // a column group with no queries
  // Tokens [skip, L) are split into partitions here; a shared prefix
  // (skip > 0) is attended by the prefix kernel and merged afterwards, so
  // with one every row writes a partial.  A column group of multi-token
  // queries needs keys only up to its last query's position.
  if (t0 >= L) return;
  int t1 = min(t0 + a.part_tokens, L);
  if constexpr (kMulti) t1 = min(t1, L - nq + min(nq - 1, vg * TPG + TPG - 1) + 1);
  const int nparts = (L - skip + a.part_tokens - 1) / a.part_tokens + (skip > 0 ? a.prefix_chunks : 0);
  // direct output (one partial per row) or a partial for the merge
  const bool direct = kMulti ? a.max_parts == 1 : nparts == 1;
  if (kMulti && t1 <= t0) {
    // every query of this group precedes the partition: empty partials
    for (int i = threadIdx.x; i < ncols * D; i += blockDim.x) {
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

  // ---- set-up: barriers, the partition's block ids (and int8 scales) ------
  if (threadIdx.x == 0) {
    cta_bad = 0;
    cta_timeout = 0;
    v_max_scale = 0.0f;
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();  // barriers and flags initialised
  if (part == 0 && a.prefix_blocks != nullptr) {
    // The sequence's first blocks must be the shared prefix blocks.
    const int32_t* bt0 = a.block_tables + (int64_t)b * a.max_blocks_per_seq;
    for (int j = threadIdx.x; j < a.num_prefix_blocks; j += blockDim.x)
      if (bt0[j] != a.prefix_blocks[j]) cta_bad = 1;
  }
#pragma unroll
  for (int r = 0; r < kSpec; ++r) {
    const int j = threadIdx.x + r * kThreads;
    if (j >= nblk) continue;
    const int32_t p = spec_id[r];
    const bool ok = p >= 0 && p < a.num_blocks;
    blk_id[j] = ok ? p : 0;
    if (!ok) cta_bad = 1;
    if constexpr (kQ8) {
      if (ok) {
        blk_ks[j] = a.k_scale[(int64_t)p * Hkv + hk];
        const float vs = a.v_scale[(int64_t)p * Hkv + hk];
        blk_vr[j] = vs;
        atomicMax(reinterpret_cast<int*>(&v_max_scale), __float_as_int(fabsf(vs)));
      }
    }
  }
  __syncthreads();
  if constexpr (kQ8) {
    // p is multiplied by (V scale / the CTA's largest V scale) so that it stays
    // in fp16 range; the output is multiplied back by the largest scale.
    const float vmax = v_max_scale > 0.0f ? v_max_scale : 1.0f;
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) blk_vr[j] = blk_vr[j] / vmax;
    __syncthreads();
  }

  const bool bad = cta_bad != 0;
  const int n_iter = (nblk + kConsumers - 1) / kConsumers;

  // Per-consumer softmax state for heads 2t, 2t+1 and the O^T accumulator.
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
  float o[G::kMTiles][4];
#pragma unroll
  for (int i = 0; i < G::kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  // int8 V enters P . V as c + 1152 (no subtraction per code pair); vb holds
  // sum_t p_t per column (an all-ones A fragment times P^T, one MMA per tile)
  // and O loses 1152 vsum before the warps combine.
  float vsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};

  if (!bad && warp == kConsumers) {
    // ======================= producer =======================================
    // The whole warp walks the stages (lane 0 issues the loads).  When this
    // partition ends the sequence and a new token is given, the warp first
    // writes that token's K/V row into the last block and orders the write
    // before the TMA read of the block (the append, fused into this launch).
    const bool append = a.new_k != nullptr && t1 == L;
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
      if (append && j0 + cnt == nblk) {
        constexpr int kChunks = D / 8;                 // 8 elements per lane
        const int p = blk_id[nblk - 1];
        const int row = (L - 1) % BS;
        const int64_t dst = (((int64_t)p * BS + row) * Hkv + hk) * D;
        const int64_t src = ((int64_t)b * Hkv + hk) * D;
        if (lane < 2 * kChunks) {
          const bool is_v = lane >= kChunks;
          const int e0 = (is_v ? lane - kChunks : lane) * 8;
          const uint4 x = *reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(is_v ? a.new_v : a.new_k) + src + e0);
          void* pool = const_cast<void*>(is_v ? a.v_cache : a.k_cache);
          if constexpr (kQ8) {
            const float sc = is_v ? a.v_scale[(int64_t)p * Hkv + hk] : blk_ks[nblk - 1];
            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
            uint32_t o2[2] = {0u, 0u};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t lo = code8<kFp8>(__uint_as_float(w4[i] << 16), sc);
              const uint32_t hi = code8<kFp8>(__uint_as_float(w4[i] & 0xffff0000u), sc);
              o2[i / 2] |= (lo | (hi << 8)) << (16 * (i % 2));
            }
            *reinterpret_cast<uint2*>(static_cast<int8_t*>(pool) + dst + e0) = make_uint2(o2[0], o2[1]);
          } else {
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(pool) + dst + e0) = x;
          }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t fb = smem_addr(&full_bar[s]);
        mbar_expect_tx(fb, (uint32_t)(cnt * G::kBlockBytes));
        for (int c = 0; c < cnt; ++c) {
          const int p = blk_id[j0 + c];
          const uint32_t kdst = stages + (uint32_t)((s * kConsumers + c) * G::kBlockBytes);
          const uint32_t vdst = kdst + G::kTensorBytes;
#pragma unroll
          for (int x = 0; x < G::kBoxes; ++x) {
            tma_load_4d(kdst + x * G::kBoxBytes, &k_map, fb, x * G::kBoxElems, hk, 0, p);
            tma_load_4d(vdst + x * G::kBoxBytes, &v_map, fb, x * G::kBoxElems, hk, 0, p);
          }
        }
      }
      __syncwarp();
      issued = it + 1;
    }
    // Wait for every fill this warp issued before the CTA may reuse or
    // release the stages (bounded; normally already complete).
    for (int s = 0; s < S && s < issued; ++s) {
      const int last = s + S * ((issued - 1 - s) / S);
      if (!mbar_wait(smem_addr(&full_bar[s]), (last / S) & 1)) ok = false;
    }
    if (!ok && lane == 0) cta_timeout = 1;
  } else if (!bad) {
    // ======================= consumers =====================================
    const int w = warp;
    constexpr bool kF16 = kQ8;
    uint32_t qf[G::kKSteps][2];
    float qscale = 1.0f;
    {
      float qv[G::kKSteps][4];
      float amax = 0.0f;
#pragma unroll
      for (int ks = 0; ks < G::kKSteps; ++ks) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float x0 = __uint_as_float(qraw[ks][r] << 16);
          const float x1 = __uint_as_float(qraw[ks][r] & 0xffff0000u);
          qv[ks][2 * r] = x0;
          qv[ks][2 * r + 1] = x1;
          amax = fmaxf(amax, fmaxf(fabsf(x0), fabsf(x1)));
        }
      }
      if constexpr (kQ8) {
        // fp16 holds |q| < 65504; scale by a power of two when needed and
        // fold the inverse into the score scale (exact either way).
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        int e = 0;
        if (amax >= 16384.0f) {
          frexpf(amax, &e);
          e -= 14;
        }
        qscale = ldexpf(1.0f, -e);
      }
#pragma unroll
      for (int ks = 0; ks < G::kKSteps; ++ks) {
        qf[ks][0] = pack2<kF16>(qv[ks][0] * qscale, qv[ks][1] * qscale);
        qf[ks][1] = pack2<kF16>(qv[ks][2] * qscale, qv[ks][3] * qscale);
      }
    }
    const float score_scale = a.scale_log2 / qscale;
    // int8 K enters the MMA as fp16 w = c + 1152 (one byte permute per code
    // pair, no subtraction): S = sum_d q_d w_d - 1152 sum_d q_d, so each
    // score column (heads 2t, 2t+1 of this lane) subtracts 1152 times the
    // sum of its fp16 q -- summed here from the B fragments lane (g, t)
    // holds for head g (exact products; the cancellation costs about 2^-24
    // of the biased sum, some 1e-6 of a score).
    float kb0 = 0.0f, kb1 = 0.0f;
    if constexpr (kQ8 && !kFp8) {
      float sq = 0.0f;
#pragma unroll
      for (int ks = 0; ks < G::kKSteps; ++ks) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const __half2 h = *reinterpret_cast<const __half2*>(&qf[ks][r]);
          sq += __low2float(h) + __high2float(h);
        }
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sq += __shfl_xor_sync(0xffffffffu, sq, 2);        // sum over head g (lanes 4g..4g+3)
      kb0 = -1152.0f * __shfl_sync(0xffffffffu, sq, (2 * t) * 4);
      kb1 = -1152.0f * __shfl_sync(0xffffffffu, sq, (2 * t + 1) * 4);
    }
    // causal limits of this lane's columns 2t and 2t+1 (multi-token queries)
    int cpos0 = 0x7fffffff, cpos1 = 0x7fffffff;
    if constexpr (kMulti) {
      if (2 * t < TPG * GQ) cpos0 = L - nq + vg * TPG + (2 * t) / GQ;
      if (2 * t + 1 < TPG * GQ) cpos1 = L - nq + vg * TPG + (2 * t + 1) / GQ;
    }
    // P^T transpose sources: token 2t (and 2t+8) of head g sits in lane
    // (2t)*4 + g/2, token 2t+1 (2t+9) in the lane 4 higher.
    const int src_a = (2 * t) * 4 + (g >> 1), src_b = src_a + 4;
    const uint32_t half_sel = (g & 1) ? 0x7632u : 0x5410u;

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
        const int valid = min(BS, L - (first_blk + j) * BS);
        const float kfac = kQ8 ? score_scale * blk_ks[j] : score_scale;

        // ---- scores S^T for every 16-token tile ---------------------------
        float sc[G::kTiles][4];
#pragma unroll
        for (int tile = 0; tile < G::kTiles; ++tile) {
          float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (!kQ8) {
            // ldmatrix.x4: matrix q = lane/8 covers rows (tokens) 8*(q&1)..+7
            // and d-chunk 2ks + (q>>1): registers = A fragment a0..a3.
            const int row = tile * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
            for (int ks = 0; ks < G::kKSteps; ++ks) {
              uint32_t fa[4];
              ldsm_x4(fa, kb + chunk_off<G>(row, 2 * ks + (lane >> 4)));
              if (ks & 1) mma16816<false>(c1, fa, qf[ks][0], qf[ks][1]);
              else        mma16816<false>(c0, fa, qf[ks][0], qf[ks][1]);
            }
          } else {
            // Rows g and g+8 of the tile; lane t reads its NC chunks of each.
            constexpr int NC = D / 64;
            uint32_t kw[2][NC][4];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int row = tile * 16 + g + 8 * rr;
#pragma unroll
              for (int ci = 0; ci < NC; ++ci) {
                const uint4 v = lds128(kb + chunk_off<G>(row, t * NC + ci));
                kw[rr][ci][0] = v.x ^ kCodeBias<kFp8>;
                kw[rr][ci][1] = v.y ^ kCodeBias<kFp8>;
                kw[rr][ci][2] = v.z ^ kCodeBias<kFp8>;
                kw[rr][ci][3] = v.w ^ kCodeBias<kFp8>;
              }
            }
#pragma unroll
            for (int ks = 0; ks < G::kKSteps; ++ks) {
              const uint32_t w0 = kw[0][ks / 4][ks % 4], w1 = kw[1][ks / 4][ks % 4];
              const uint32_t fa[4] = {codes_to_f16x2<kFp8, true>(w0, 0x4140u), codes_to_f16x2<kFp8, true>(w1, 0x4140u),
                                      codes_to_f16x2<kFp8, true>(w0, 0x4342u), codes_to_f16x2<kFp8, true>(w1, 0x4342u)};
              if (ks & 1) mma16816<true>(c1, fa, qf[ks][0], qf[ks][1]);
              else        mma16816<true>(c0, fa, qf[ks][0], qf[ks][1]);
            }
          }
          // rows (tokens) g and g+8 of this tile; masked rows -> -inf (and,
          // for multi-token queries, tokens past a column's position)
          const int tok_lo = tile * 16 + g, tok_hi = tok_lo + 8;
          if constexpr (kMulti) {
            const int abs_lo = (first_blk + j) * BS + tok_lo, abs_hi = abs_lo + 8;
            sc[tile][0] = (tok_lo < valid && abs_lo <= cpos0) ? (c0[0] + c1[0] + kb0) * kfac : -INFINITY;
            sc[tile][1] = (tok_lo < valid && abs_lo <= cpos1) ? (c0[1] + c1[1] + kb1) * kfac : -INFINITY;
            sc[tile][2] = (tok_hi < valid && abs_hi <= cpos0) ? (c0[2] + c1[2] + kb0) * kfac : -INFINITY;
            sc[tile][3] = (tok_hi < valid && abs_hi <= cpos1) ? (c0[3] + c1[3] + kb1) * kfac : -INFINITY;
          } else {
            sc[tile][0] = tok_lo < valid ? (c0[0] + c1[0] + kb0) * kfac : -INFINITY;
            sc[tile][1] = tok_lo < valid ? (c0[1] + c1[1] + kb1) * kfac : -INFINITY;
            sc[tile][2] = tok_hi < valid ? (c0[2] + c1[2] + kb0) * kfac : -INFINITY;
            sc[tile][3] = tok_hi < valid ? (c0[3] + c1[3] + kb1) * kfac : -INFINITY;
          }
        }

        // ---- online softmax update for heads 2t (index 0) and 2t+1 (1) ----
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int tile = 0; tile < G::kTiles; ++tile) {
          mx0 = fmaxf(mx0, fmaxf(sc[tile][0], sc[tile][2]));
          mx1 = fmaxf(mx1, fmaxf(sc[tile][1], sc[tile][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mx0n = fmaxf(m_run[0], mx0), mx1n = fmaxf(m_run[1], mx1);
        // a column with no key yet keeps m = -inf: subtract 0 then (multi-
        // token queries; a decode column always has a key)
        const float mn0 = (kMulti && mx0n == -INFINITY) ? 0.0f : mx0n;
        const float mn1 = (kMulti && mx1n == -INFINITY) ? 0.0f : mx1n;
        const float al0 = exp2f(m_run[0] - mn0), al1 = exp2f(m_run[1] - mn1);
        m_run[0] = mx0n;
        m_run[1] = mx1n;
        l_run[0] *= al0;
        l_run[1] *= al1;
#pragma unroll
        for (int i = 0; i < G::kMTiles; ++i) {
          o[i][0] *= al0;
          o[i][1] *= al1;
          o[i][2] *= al0;
          o[i][3] *= al1;
        }
        if constexpr (kQ8 && !kFp8) {
          vsum[0] *= al0;
          vsum[1] *= al1;
          vsum[2] *= al0;
          vsum[3] *= al1;
        }
        const float vr = kQ8 ? blk_vr[j] : 1.0f;

#pragma unroll
        for (int tile = 0; tile < G::kTiles; ++tile) {
          if (tile * 16 >= valid) break;                    // whole tile masked
          const float p0 = exp2f(sc[tile][0] - mn0), p1 = exp2f(sc[tile][1] - mn1);
          const float p2 = exp2f(sc[tile][2] - mn0), p3 = exp2f(sc[tile][3] - mn1);
          l_run[0] += p0 + p2;
          l_run[1] += p1 + p3;
          // P^T as the B operand: b0 = (tokens 2t, 2t+1; head g),
          // b1 = (tokens 2t+8, 2t+9; head g), gathered from the lanes that
          // hold those tokens' scores.
          const uint32_t r0 = pack2<kF16>(p0 * vr, p1 * vr), r1 = pack2<kF16>(p2 * vr, p3 * vr);
          const uint32_t x0 = __shfl_sync(0xffffffffu, r0, src_a);
          const uint32_t x1 = __shfl_sync(0xffffffffu, r0, src_b);
          const uint32_t y0 = __shfl_sync(0xffffffffu, r1, src_a);
          const uint32_t y1 = __shfl_sync(0xffffffffu, r1, src_b);
          const uint32_t pb0 = prmt(x0, x1, half_sel), pb1 = prmt(y0, y1, half_sel);

          // V rows past `valid` are zeroed in the A fragments (tokens 2t, 2t+1
          // in fa[0..1], 2t+8, 2t+9 in fa[2..3]): p is 0 there, but the pool
          // may hold NaN (bf16 or E4M3 patterns) and 0 * NaN is NaN.  int8
          // codes are always finite and skip it.
          uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
          if ((!kQ8 || kFp8) && valid < BS) {
            const int k0 = tile * 16 + 2 * t;
            mlo = (k0 < valid ? 0x0000ffffu : 0u) | (k0 + 1 < valid ? 0xffff0000u : 0u);
            mhi = (k0 + 8 < valid ? 0x0000ffffu : 0u) | (k0 + 9 < valid ? 0xffff0000u : 0u);
          }
          if constexpr (!kQ8) {
            // V^T tiles by ldmatrix.trans: matrix q = lane/8 covers tokens
            // 8*(q>>1)..+7 of the tile and d-chunk 2i + (q&1).
            const int row = tile * 16 + (lane >> 4) * 8 + (lane & 7);
#pragma unroll
            for (int i = 0; i < G::kMTiles; ++i) {
              uint32_t fa[4];
              ldsm_x4_t(fa, vb + chunk_off<G>(row, 2 * i + ((lane >> 3) & 1)));
              fa[0] &= mlo;
              fa[1] &= mlo;
              fa[2] &= mhi;
              fa[3] &= mhi;
              mma16816<false>(o[i], fa, pb0, pb1);
            }
          } else {
            // Lane (g, t) reads tokens 2t, 2t+1, 2t+8, 2t+9 of the tile, the
            // D/8 bytes of d in [g*D/8, (g+1)*D/8); m-tile i pairs d rows
            // g <-> g*D/8 + 2i and g+8 <-> g*D/8 + 2i + 1.
            constexpr int NB = D / 8;                 // bytes per lane per token
            constexpr int NW = NB / 4;
            uint32_t vw[4][NW];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int row = tile * 16 + 2 * t + (rr & 1) + 8 * (rr >> 1);
              if constexpr (NB == 16) {
                const uint4 v = lds128(vb + chunk_off<G>(row, g));
                vw[rr][0] = v.x ^ kCodeBias<kFp8>;
                vw[rr][1] = v.y ^ kCodeBias<kFp8>;
                vw[rr][2] = v.z ^ kCodeBias<kFp8>;
                vw[rr][3] = v.w ^ kCodeBias<kFp8>;
              } else {
                const uint2 v = lds64(vb + chunk_off<G>(row, g / 2) + (g & 1) * 8);
                vw[rr][0] = v.x ^ kCodeBias<kFp8>;
                vw[rr][1] = v.y ^ kCodeBias<kFp8>;
              }
            }
            if constexpr (!kFp8) {
              const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};
              mma16816<true>(vsum, ones, pb0, pb1);
            }
#pragma unroll
            for (int i = 0; i < G::kMTiles; ++i) {
              const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;  // bytes 2,3 or 0,1
              const uint32_t ulo = prmt(vw[0][i / 2], vw[1][i / 2], sel);  // tokens 2t, 2t+1
              const uint32_t uhi = prmt(vw[2][i / 2], vw[3][i / 2], sel);  // tokens 2t+8, 2t+9
              uint32_t fa[4] = {codes_to_f16x2<kFp8, true>(ulo, 0x4140u), codes_to_f16x2<kFp8, true>(ulo, 0x4342u),
                                codes_to_f16x2<kFp8, true>(uhi, 0x4140u), codes_to_f16x2<kFp8, true>(uhi, 0x4342u)};
              if constexpr (kFp8) {
                fa[0] &= mlo;
                fa[1] &= mlo;
                fa[2] &= mhi;
                fa[3] &= mhi;
              }
              mma16816<true>(o[i], fa, pb0, pb1);
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
  float* red_m = red;                              // [kConsumers][8]
  float* red_l = red + kConsumers * 8;             // [kConsumers][8]
  float* red_acc = red + 2 * kConsumers * 8;       // [kConsumers][8][D]
  if (!failed && warp < kConsumers) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
      l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
    }
    if (g == 0) {
      red_m[warp * 8 + 2 * t] = m_run[0];
      red_m[warp * 8 + 2 * t + 1] = m_run[1];
      red_l[warp * 8 + 2 * t] = l_run[0];
      red_l[warp * 8 + 2 * t + 1] = l_run[1];
    }
    if constexpr (kQ8 && !kFp8) {
#pragma unroll
      for (int i = 0; i < G::kMTiles; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[i][k] = fmaf(-1152.0f, vsum[k], o[i][k]);
    }
    float* acc = red_acc + warp * 8 * D;
#pragma unroll
    for (int i = 0; i < G::kMTiles; ++i) {
      int d_lo, d_hi;                              // d rows g and g+8 of m-tile i
      if constexpr (kQ8) {
        d_lo = g * (D / 8) + 2 * i;
        d_hi = d_lo + 1;
      } else {
        d_lo = 16 * i + g;
        d_hi = d_lo + 8;
      }
      acc[(2 * t) * D + d_lo] = o[i][0];
      acc[(2 * t + 1) * D + d_lo] = o[i][1];
      acc[(2 * t) * D + d_hi] = o[i][2];
      acc[(2 * t + 1) * D + d_hi] = o[i][3];
    }
  }
  __syncthreads();

  if (failed) {
    if (threadIdx.x == 0)
      atomicOr(a.flags, bad ? PAGEDKV_FLAG_BAD_BLOCK : PAGEDKV_FLAG_WAIT_TIMEOUT);
    for (int i = threadIdx.x; i < ncols * D; i += blockDim.x) {
      const int hh = i / D, e = i % D;
      const int64_t row = col_row(hh);
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

  const float out_scale = kQ8 ? (v_max_scale > 0.0f ? v_max_scale : 1.0f) : 1.0f;
  for (int i = threadIdx.x; i < ncols * D; i += blockDim.x) {
    const int hh = i / D, e = i % D;
    const int64_t row = col_row(hh);
    if (row < 0) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, red_m[w * 8 + hh]);
    const float Mz = (kMulti && M == -INFINITY) ? 0.0f : M;  // a column with no key here
    float num = 0.0f, den = 0.0f;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) {
      const float c = exp2f(red_m[w * 8 + hh] - Mz);  // 0 for a warp that saw no token
      num = fmaf(c, red_acc[(w * 8 + hh) * D + e], num);
      den = fmaf(c, red_l[w * 8 + hh], den);
    }
    num *= out_scale;
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
  // this CTA's partials are written: the merge launched behind this grid
  // (programmatic dependent; it waits for the whole grid) may be scheduled
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------

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

// 4-D map over a pool [NB, bs, Hkv, d] (innermost first: d, head, row, block)
// whose box is one block's rows of one head: [1, bs, 1, box elements].
template <int D, int BS, bool kQ8>
kv_status make_map(CUtensorMap* map, const void* pool, const DecodeArgs& a) {
  using G = Geo<D, BS, kQ8>;
  auto fn = encode_fn();
  if (!fn) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.num_kv_heads, (cuuint64_t)BS,
                              (cuuint64_t)a.num_blocks};
  const cuuint64_t strides[3] = {(cuuint64_t)D * G::kElem,
                                 (cuuint64_t)a.num_kv_heads * D * G::kElem,
                                 (cuuint64_t)BS * a.num_kv_heads * D * G::kElem};
  const cuuint32_t box[4] = {(cuuint32_t)G::kBoxElems, 1, (cuuint32_t)BS, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, kQ8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        4, const_cast<void*>(pool), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        G::kSwizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        G::kRowBytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                            : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return KV_OK;
}

template <int D, int BS, bool kQ8, bool kFp8, bool kMulti>
kv_status launch_t(const DecodeArgs& a, cudaStream_t s) {
  using G = Geo<D, BS, kQ8>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  kv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != KV_OK) return st;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
      st = cuda_check(cudaFuncSetAttribute(decode_kernel<D, BS, kQ8, kFp8, kMulti>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           G::kSmemBytes),
                      "cudaFuncSetAttribute(decode_kernel)");
      if (st != KV_OK) return st;
      attr_set[dev] = true;
    }
  }
  alignas(64) CUtensorMap km, vm;
  if ((st = make_kv_maps(a, &km, &vm)) != KV_OK) return st;
  const dim3 grid(a.num_kv_heads, kMulti ? a.batch * a.vgroups : a.batch, a.max_parts);
  if (a.prefix_chunks == 0) {
    decode_kernel<D, BS, kQ8, kFp8, kMulti><<<grid, kThreads, G::kSmemBytes, s>>>(km, vm, a);
    return cuda_check(cudaGetLastError(), "decode_kernel launch");
  }
  // Behind the prefix kernel: launched as its programmatic dependent so the
  // two run side by side (this kernel never reads the prefix results; the
  // merge, a plain launch, waits for both).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = G::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, decode_kernel<D, BS, kQ8, kFp8, kMulti>, km, vm, a),
                    "decode_kernel launch");
}

template <int D, bool kQ8, bool kFp8>
kv_status launch_bs(const DecodeArgs& a, cudaStream_t s) {
  if (a.query_start != nullptr)
    return a.block_size == 32 ? launch_t<D, 32, kQ8, kFp8, true>(a, s) : launch_t<D, 16, kQ8, kFp8, true>(a, s);
  return a.block_size == 32 ? launch_t<D, 32, kQ8, kFp8, false>(a, s) : launch_t<D, 16, kQ8, kFp8, false>(a, s);
}

template <int D, int BS, bool kQ8>
kv_status maps_t(const DecodeArgs& a, CUtensorMap* km, CUtensorMap* vm) {
  kv_status st = make_map<D, BS, kQ8>(km, a.k_cache, a);
  return st != KV_OK ? st : make_map<D, BS, kQ8>(vm, a.v_cache, a);
}

kv_status encode_kv_maps(const DecodeArgs& a, CUtensorMap* km, CUtensorMap* vm) {
  const bool q8 = a.dtype != KV_DTYPE_BF16, b32 = a.block_size == 32;
  if (a.head_dim == 128) {
    if (q8) return b32 ? maps_t<128, 32, true>(a, km, vm) : maps_t<128, 16, true>(a, km, vm);
    return b32 ? maps_t<128, 32, false>(a, km, vm) : maps_t<128, 16, false>(a, km, vm);
  }
  if (q8) return b32 ? maps_t<64, 32, true>(a, km, vm) : maps_t<64, 16, true>(a, km, vm);
  return b32 ? maps_t<64, 32, false>(a, km, vm) : maps_t<64, 16, false>(a, km, vm);
}

// The K and V tensor maps of recently used pools.  A map holds only the
// pool's address and geometry, so an entry whose key matches is the map
// that encoding would produce again (a pool freed and re-allocated at the
// same address with the same geometry gets the same map).  Looking one up
// costs a mutex and a short scan instead of two driver encodings per call.
struct MapEntry {
  const void* k = nullptr;
  const void* v = nullptr;
  int64_t num_blocks = 0;
  int device = -1, kv8 = 0, head_dim = 0, block_size = 0, num_kv_heads = 0;
  CUtensorMap km, vm;                 // (CUtensorMap carries its own alignment)
};
constexpr int kMapCache = 16;

}  // namespace

kv_status make_kv_maps(const DecodeArgs& a, CUtensorMap* km, CUtensorMap* vm) {
  static std::mutex mu;
  static MapEntry cache[kMapCache];
  static int next = 0;
  int dev = 0;
  kv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != KV_OK) return st;
  const int kv8 = a.dtype != KV_DTYPE_BF16;
  std::lock_guard<std::mutex> lock(mu);
  for (const MapEntry& e : cache) {
    if (e.device == dev && e.k == a.k_cache && e.v == a.v_cache && e.kv8 == kv8 &&
        e.head_dim == a.head_dim && e.block_size == a.block_size &&
        e.num_kv_heads == a.num_kv_heads && e.num_blocks == a.num_blocks) {
      *km = e.km;
      *vm = e.vm;
      return KV_OK;
    }
  }
  MapEntry& e = cache[next];
  if ((st = encode_kv_maps(a, &e.km, &e.vm)) != KV_OK) {
    e.device = -1;
    return st;
  }
  e.device = dev;
  e.k = a.k_cache;
  e.v = a.v_cache;
  e.kv8 = kv8;
  e.head_dim = a.head_dim;
  e.block_size = a.block_size;
  e.num_kv_heads = a.num_kv_heads;
  e.num_blocks = a.num_blocks;
  next = (next + 1) % kMapCache;
  *km = e.km;
  *vm = e.vm;
  return KV_OK;
}

kv_status launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const int64_t rows = (int64_t)a.batch * (a.query_start ? a.vgroups : 1);
  if (rows > 65535 || a.max_parts > 65535)
    return fail(KV_ERR_INVALID_ARG, "batch (x column groups) and the partition count must be at most 65535");
  if (a.num_q_heads / a.num_kv_heads > 8)
    return fail(KV_ERR_INVALID_ARG, "at most 8 query heads per KV head");
  if (a.part_tokens / a.block_size > kMaxBlocks || a.part_tokens % a.block_size)
    return fail(KV_ERR_INVALID_ARG, "partition must be a multiple of block_size, at most %d blocks",
                kMaxBlocks);
  if (a.head_dim == 128) {
    if (a.dtype == KV_DTYPE_FP8_E4M3) return launch_bs<128, true, true>(a, s);
    return a.dtype == KV_DTYPE_INT8 ? launch_bs<128, true, false>(a, s)
                                    : launch_bs<128, false, false>(a, s);
  }
  if (a.dtype == KV_DTYPE_FP8_E4M3) return launch_bs<64, true, true>(a, s);
  return a.dtype == KV_DTYPE_INT8 ? launch_bs<64, true, false>(a, s) : launch_bs<64, false, false>(a, s);
}

}  // namespace pagedkv
