// pagedkv_multi.cu -- attention of multi-token queries over the paged pool:
// speculative verification (“让 Agent 跑得快：LLM 推理服务”, §六 投机解码: the
// target model scores the gamma draft tokens in one parallel pass) and
// chunked prefill batched with decodes (“LLM 推理优化技术全景”, SARATHI: a
// 512-token prefill chunk plus as many decodes as fit).
//
// Sequence b has n_b query tokens, already appended: its last n_b tokens,
// q rows query_start[b] .. query_start[b + 1] - 1.  Query token i sits at
// position L_b - n_b + i and attends positions 0 .. L_b - n_b + i (causal).
//
// Tiling (rows on the MMA's M, as in Flash Attention v2): rows of one
// (sequence, KV head) are (query token, grouped head) pairs, token-major; a
// CTA of 4 warps takes up to 64 of them and one token partition of the
// sequence, and streams that range's blocks through a 4-stage ring of TMA
// tensor loads, stopping at the tile's last query position.  The tile's
// 16-row groups (1, 2 or 4) share the warps: with fewer than four groups,
// the warps of a group take alternate blocks and combine their (m, l, O)
// through shared memory at the end (speculative verification has 5 tokens x
// 4 heads = 20 rows).  Per 16-token tile a warp computes S = Q . K^T, masks
// tokens past each row's position, updates the online softmax, and reuses
// the S accumulators as the A operand of O += P . V.  One partition writes
// the output; several write per-row (m, l, acc) partials that a merge kernel
// combines (“LLM 推理优化技术全景”, 在线 Softmax; “Flash Attention v2 的改进”).
// bf16 pools.  Sequences with few query tokens (at most 4 x 8 / G) go to the
// decode kernel instead, whose 8 MMA columns per CTA then hold (token, head)
// pairs (pagedkv_decode.cu); both paths share the per-row merge below.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv_common.cuh"
#include "pagedkv_device.cuh"

namespace pagedkv {
namespace {

using namespace dev;

constexpr int kMWarps = 4;
constexpr int kMThreads = kMWarps * 32;
constexpr int kMRows = kMWarps * 16;     // query rows per CTA
// Shared memory for the ring of stages (one block of K and V each): as many
// stages as fit, 4 to 8, so that several blocks per CTA are in flight.
#ifndef PAGEDKV_MULTI_STAGE_BUDGET
#define PAGEDKV_MULTI_STAGE_BUDGET (32 * 1024)
#endif
template <class G>
__host__ __device__ constexpr int multi_stages() {
  return PAGEDKV_MULTI_STAGE_BUDGET / G::kBlockBytes > 8 ? 8
         : PAGEDKV_MULTI_STAGE_BUDGET / G::kBlockBytes < 4 ? 4
         : PAGEDKV_MULTI_STAGE_BUDGET / G::kBlockBytes;
}

// Column groups the decode kernel may serve per sequence (8 columns each):
// beyond this, the row-tiled kernel below takes the queries.
constexpr int kMaxVGroups = 4;

// Row tiles of a sequence with n query tokens and GQ grouped heads (none for
// a sequence the decode kernel's column groups serve: n <= col_max_n).
__device__ __forceinline__ int row_tiles(int n, int GQ, int col_max_n) {
  return n > col_max_n ? (n * GQ + kMRows - 1) / kMRows : 0;
}

#ifndef PAGEDKV_MULTI_MIN_BLOCKS
#define PAGEDKV_MULTI_MIN_BLOCKS 3
#endif
template <int D, int BS>
__global__ void __launch_bounds__(kMThreads, PAGEDKV_MULTI_MIN_BLOCKS)
    multi_kernel(const __grid_constant__ CUtensorMap k_map,
                 const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
  using G = Geo<D, BS, false>;
  constexpr int S = multi_stages<G>();
  // the warps' combine parks up to 3 x (O[16][D], m[16], l[16]) in the stages
  static_assert(3 * (16 * D + 32) * 4 <= S * G::kBlockBytes, "stage memory too small to combine");
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full_bar[S], empty_bar[S];
  __shared__ int scan[kMThreads];
  __shared__ int sh_b, sh_rt, sh_bad, sh_fail;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads, GQ = Hq / Hkv;
  const int hk = blockIdx.y, part = blockIdx.z;
  const int B = a.batch;
  const int32_t* qs = a.query_start;
  const uint32_t stages = (smem_addr(smem_raw) + 1023u) & ~1023u;

  if (tid == 0) {
    sh_b = -1;
    sh_bad = 0;
    sh_fail = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kMWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // ---- which (sequence, row tile) CTA x serves: the x-th tile, sequences in
  // order.  Thread i counts the tiles of sequences [i*per, (i+1)*per); an
  // inclusive scan over threads locates x.
  const int per = (B + kMThreads - 1) / kMThreads;
  int mine = 0;
  for (int i = 0; i < per; ++i) {
    const int b = tid * per + i;
    if (b < B) {
      const int n = qs[b + 1] - qs[b];
      if (n < 0 && blockIdx.x == 0 && hk == 0 && part == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_SEQ_LEN);
      mine += row_tiles(n, GQ, a.col_max_n);
    }
  }
  scan[tid] = mine;
  __syncthreads();
  for (int off = 1; off < kMThreads; off <<= 1) {
    const int v = tid >= off ? scan[tid - off] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  const int x = blockIdx.x;
  if (x >= scan[tid] - mine && x < scan[tid]) {
    int acc = scan[tid] - mine;
    for (int i = 0; i < per; ++i) {
      const int b = tid * per + i;
      if (b >= B) break;
      const int tl = row_tiles(qs[b + 1] - qs[b], GQ, a.col_max_n);
      if (x < acc + tl) {
        sh_b = b;
        sh_rt = x - acc;
        break;
      }
      acc += tl;
    }
  }
  __syncthreads();
  if (sh_b < 0) return;                                    // past the last tile
  const int b = sh_b, rt = sh_rt;
  const int q0 = qs[b], n = qs[b + 1] - q0;
  const int L = a.seq_lens[b];
  const int rows_b = n * GQ;
  const bool split = a.max_parts > 1;
  const int t0 = part * a.part_tokens;
  if (t0 >= L && L > 0) return;                            // no such partition for this sequence
  const bool rows_ok = q0 >= 0 && q0 + n <= a.num_tokens;
  const bool len_ok = rows_ok && L > 0 && n <= L && n <= a.max_query_len && L <= a.max_seq_len &&
                      (int64_t)L <= (int64_t)a.max_blocks_per_seq * BS;

  // The tile's 16-row groups (RG of them, 1, 2 or 4) and the warps per
  // group (W = 4 / RG), which take the blocks k with k % W == lane_i.  This
  // warp's rows ra = r0 + g and rb = ra + 8 of the sequence's rows.
  const int groups = (min(kMRows, rows_b - rt * kMRows) + 15) / 16;
  const int RG = groups <= 1 ? 1 : (groups <= 2 ? 2 : 4);
  const int W = kMWarps / RG;
  const int grp = warp % RG, lane_i = warp / RG;
  const int r0 = rt * kMRows + grp * 16;
  const int ra = r0 + g, rb = ra + 8;
  const bool va = len_ok && ra < rows_b, vb = len_ok && rb < rows_b;
  const int64_t qrow_a = va ? (int64_t)(q0 + ra / GQ) * Hq + hk * GQ + ra % GQ : 0;
  const int64_t qrow_b = vb ? (int64_t)(q0 + rb / GQ) * Hq + hk * GQ + rb % GQ : 0;
  const int pos_a = va ? L - n + ra / GQ : -1, pos_b = vb ? L - n + rb / GQ : -1;
  const int last_row = min(rt * kMRows + kMRows, rows_b) - 1;
  const int pos_max = L - n + last_row / GQ;               // the tile's last position
  const int t_end = min(min(t0 + a.part_tokens, L), pos_max + 1);
  const int first_blk = t0 / BS;
  const int nblk = (len_ok && t_end > t0) ? (t_end - 1) / BS - first_blk + 1 : 0;
  const bool warp_live = r0 < rows_b;
  const int wpos_min = L - n + r0 / GQ;                    // the warp's first row's position

  uint32_t qa[G::kKSteps][4];
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
    for (int ks = 0; ks < G::kKSteps; ++ks) {
      const int d0 = 16 * ks + 2 * t;
      qa[ks][0] = va ? *reinterpret_cast<const uint32_t*>(q + qrow_a * D + d0) : 0u;
      qa[ks][1] = vb ? *reinterpret_cast<const uint32_t*>(q + qrow_b * D + d0) : 0u;
      qa[ks][2] = va ? *reinterpret_cast<const uint32_t*>(q + qrow_a * D + d0 + 8) : 0u;
      qa[ks][3] = vb ? *reinterpret_cast<const uint32_t*>(q + qrow_b * D + d0 + 8) : 0u;
    }
  }
  const int32_t* bt = a.block_tables + (int64_t)b * a.max_blocks_per_seq + first_blk;
  for (int j = tid; j < nblk; j += kMThreads) {
    const int32_t p = bt[j];
    if (p < 0 || p >= a.num_blocks) sh_bad = 1;
  }
  __syncthreads();
  const bool bad = sh_bad != 0;

  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  bool ok = true;

  auto issue = [&](int k) {                               // thread 0 only
    const int s = k % S;
    if (k >= S && !mbar_wait(smem_addr(&empty_bar[s]), ((k / S) - 1) & 1)) return false;
    const int p = bt[k];
    const uint32_t fb = smem_addr(&full_bar[s]);
    mbar_expect_tx(fb, (uint32_t)G::kBlockBytes);
    const uint32_t kdst = stages + (uint32_t)(s * G::kBlockBytes);
    const uint32_t vdst = kdst + G::kTensorBytes;
#pragma unroll
    for (int xx = 0; xx < G::kBoxes; ++xx) {
      tma_load_4d(kdst + xx * G::kBoxBytes, &k_map, fb, xx * G::kBoxElems, hk, 0, p);
      tma_load_4d(vdst + xx * G::kBoxBytes, &v_map, fb, xx * G::kBoxElems, hk, 0, p);
    }
    return true;
  };

  int issued = 0;
  if (!bad && nblk > 0) {
    if (tid == 0)
      for (int k = 0; k < S - 1 && k < nblk; ++k) ok = ok && issue(k);
    issued = min(S - 1, nblk);
    for (int k = 0; k < nblk; ++k) {
      if (tid == 0 && k + S - 1 < nblk) ok = ok && issue(k + S - 1);
      issued = min(nblk, k + S);
      const int s = k % S;
      if (!mbar_wait(smem_addr(&full_bar[s]), (k / S) & 1)) {
        ok = false;
        break;
      }
      const uint32_t kb = stages + (uint32_t)(s * G::kBlockBytes), vb_ = kb + G::kTensorBytes;
      const int tb = (first_blk + k) * BS;                  // the block's first token
      const int valid = L - tb;                             // rows holding tokens (may exceed BS)
      if (warp_live && k % W == lane_i) {
#pragma unroll
        for (int tile = 0; tile < G::kTiles; ++tile) {
          const int tt = tb + tile * 16;
          if (tt >= t_end) break;                           // CTA-uniform
          // ---- S = Q . K^T for 16 tokens (n-tiles of tokens 0-7, 8-15)
          float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          const int krow = tile * 16 + (lane >> 4) * 8 + (lane & 7);
#pragma unroll
          for (int ks = 0; ks < G::kKSteps; ++ks) {
            uint32_t fb4[4];
            ldsm_x4(fb4, kb + chunk_off<G>(krow, 2 * ks + ((lane >> 3) & 1)));
            mma16816<false>(c[0], qa[ks], fb4[0], fb4[1]);
            mma16816<false>(c[1], qa[ks], fb4[2], fb4[3]);
          }
          // ---- causal mask and scale: token tt + 8nt + 2t + (e&1), row a
          // for e < 2 and row b for e >= 2.  A tile wholly at or before the
          // warp's first position and before t_end needs no mask (rows past
          // the sequence's queries are never written, whatever they hold).
          if (tt + 15 <= wpos_min && tt + 16 <= t_end) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) c[nt][e] *= a.scale_log2;
          } else {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int tok = tt + 8 * nt + 2 * t + (e & 1);
                const int pos = e < 2 ? pos_a : pos_b;
                c[nt][e] = (tok <= pos && tok < t_end) ? c[nt][e] * a.scale_log2 : -INFINITY;
              }
          }
          float mx_a = fmaxf(fmaxf(c[0][0], c[0][1]), fmaxf(c[1][0], c[1][1]));
          float mx_b = fmaxf(fmaxf(c[0][2], c[0][3]), fmaxf(c[1][2], c[1][3]));
#pragma unroll
          for (int off = 1; off < 4; off <<= 1) {
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
          }
          // a row that has seen no token yet keeps m = -inf: subtract 0 then
          // (its p and the rescale of its empty state are all 0)
          const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
          const float base_a = mn_a == -INFINITY ? 0.0f : mn_a;
          const float base_b = mn_b == -INFINITY ? 0.0f : mn_b;
          const float al_a = exp2f(m_a - base_a), al_b = exp2f(m_b - base_b);
          m_a = mn_a;
          m_b = mn_b;
          float p[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            p[nt][0] = exp2f(c[nt][0] - base_a);
            p[nt][1] = exp2f(c[nt][1] - base_a);
            p[nt][2] = exp2f(c[nt][2] - base_b);
            p[nt][3] = exp2f(c[nt][3] - base_b);
          }
          l_a = l_a * al_a + p[0][0] + p[0][1] + p[1][0] + p[1][1];
          l_b = l_b * al_b + p[0][2] + p[0][3] + p[1][2] + p[1][3];
          // the accumulator is rescaled only when some row's maximum moved
          // (the factor is exactly 1 otherwise)
          if (__any_sync(0xffffffffu, al_a != 1.0f || al_b != 1.0f)) {
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
              o[i][0] *= al_a;
              o[i][1] *= al_a;
              o[i][2] *= al_b;
              o[i][3] *= al_b;
            }
          }
          // ---- O += P . V.  Rows at or past L in the sequence's last block
          // are zeroed in the V fragments (tokens 2t, 2t+1 of each half in
          // b0, 2t+8, 2t+9 in b1): p is 0 there but the pool may hold NaN.
          const uint32_t pa[4] = {pack2<false>(p[0][0], p[0][1]), pack2<false>(p[0][2], p[0][3]),
                                  pack2<false>(p[1][0], p[1][1]), pack2<false>(p[1][2], p[1][3])};
          uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
          if (valid < BS) {
            const int k0 = tile * 16 + 2 * t;
            mlo = (k0 < valid ? 0x0000ffffu : 0u) | (k0 + 1 < valid ? 0xffff0000u : 0u);
            mhi = (k0 + 8 < valid ? 0x0000ffffu : 0u) | (k0 + 9 < valid ? 0xffff0000u : 0u);
          }
          const int vrow = tile * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
          for (int jj = 0; jj < D / 16; ++jj) {
            uint32_t fb4[4];
            ldsm_x4_t(fb4, vb_ + chunk_off<G>(vrow, 2 * jj + (lane >> 4)));
            fb4[0] &= mlo;
            fb4[2] &= mlo;
            fb4[1] &= mhi;
            fb4[3] &= mhi;
            mma16816<false>(o[2 * jj], pa, fb4[0], fb4[1]);
            mma16816<false>(o[2 * jj + 1], pa, fb4[2], fb4[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
    }
    if (tid == 0) {
      // let every issued fill land before the CTA may exit (bounded)
      for (int s = 0; s < S && s < issued; ++s) {
        const int last = s + S * ((issued - 1 - s) / S);
        if (!mbar_wait(smem_addr(&full_bar[s]), (last / S) & 1)) ok = false;
      }
    }
  }
  if (!ok) {
    atomicOr(a.flags, PAGEDKV_FLAG_WAIT_TIMEOUT);
    sh_fail = 1;
  }
  if (bad && tid == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_BLOCK);
  if (!len_ok && tid == 0 && rt == 0 && hk == 0 && part == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_SEQ_LEN);
  if (!rows_ok) return;                                    // no rows to write (CTA-uniform)

#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  // ---- the warps of a row group combine: lane_i > 0 park (m, l, O) in the
  // stage memory (every fill has landed and every warp is past its reads),
  // lane_i == 0 folds them in and writes the rows.
  __syncthreads();
  const bool failed = bad || sh_fail != 0 || !len_ok;
  if (W > 1) {
    float* park = reinterpret_cast<float*>(smem_raw + (stages - smem_addr(smem_raw)));
    constexpr int kSlot = 16 * D + 32;                     // O[16][D], m[16], l[16]
    if (lane_i > 0) {
      float* base = park + ((lane_i - 1) * RG + grp) * kSlot;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        *reinterpret_cast<float2*>(base + g * D + 8 * i + 2 * t) = make_float2(o[i][0], o[i][1]);
        *reinterpret_cast<float2*>(base + (g + 8) * D + 8 * i + 2 * t) = make_float2(o[i][2], o[i][3]);
      }
      if (t == 0) {
        base[16 * D + g] = m_a;
        base[16 * D + g + 8] = m_b;
        base[16 * D + 16 + g] = l_a;
        base[16 * D + 16 + g + 8] = l_b;
      }
    }
    __syncthreads();
    if (lane_i > 0) return;
    for (int w2 = 1; w2 < W; ++w2) {
      const float* base = park + ((w2 - 1) * RG + grp) * kSlot;
      const float m2a = base[16 * D + g], m2b = base[16 * D + g + 8];
      const float l2a = base[16 * D + 16 + g], l2b = base[16 * D + 16 + g + 8];
      const float mna = fmaxf(m_a, m2a), mnb = fmaxf(m_b, m2b);
      const float za = mna == -INFINITY ? 0.0f : mna, zb = mnb == -INFINITY ? 0.0f : mnb;
      const float sa = exp2f(m_a - za), s2a = exp2f(m2a - za);
      const float sb = exp2f(m_b - zb), s2b = exp2f(m2b - zb);
      l_a = l_a * sa + l2a * s2a;
      l_b = l_b * sb + l2b * s2b;
      m_a = mna;
      m_b = mnb;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const float2 xa = *reinterpret_cast<const float2*>(base + g * D + 8 * i + 2 * t);
        const float2 xb = *reinterpret_cast<const float2*>(base + (g + 8) * D + 8 * i + 2 * t);
        o[i][0] = o[i][0] * sa + xa.x * s2a;
        o[i][1] = o[i][1] * sa + xa.y * s2a;
        o[i][2] = o[i][2] * sb + xb.x * s2b;
        o[i][3] = o[i][3] * sb + xb.y * s2b;
      }
    }
  }

  // ---- epilogue: rows of this tile (invalid sequences: zeros)
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rb : ra;
    if (r >= rows_b) continue;
    const int64_t qrow = (int64_t)(q0 + r / GQ) * Hq + hk * GQ + r % GQ;
    if (!split) {
      const float l = half ? l_b : l_a;
      const float inv = (failed || !(l > 0.0f)) ? 0.0f : 1.0f / l;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + qrow * D;
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<__nv_bfloat162*>(out + 8 * i + 2 * t) =
            __floats2bfloat162_rn(o[i][2 * half] * inv, o[i][2 * half + 1] * inv);
    } else {
      const int64_t slot = qrow * a.max_parts + part;
      if (t == 0) {
        a.ws_ml[2 * slot] = half ? m_b : m_a;
        a.ws_ml[2 * slot + 1] = failed ? -1.0f : (half ? l_b : l_a);
      }
      float* acc = a.ws_acc + slot * D;
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<float2*>(acc + 8 * i + 2 * t) =
            make_float2(o[i][2 * half], o[i][2 * half + 1]);
    }
  }
}

// Log-sum-exp merge of the partition partials of every (query token, head)
// row: one warp per row.  Partials of partitions wholly past a row's position
// hold l = 0 and are skipped; a partial marked l < 0 (bad sequence or a wait
// that gave up) zeroes the row.
template <int D>
__global__ void __launch_bounds__(128) multi_merge_kernel(const DecodeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x, h = blockIdx.y * 4 + warp;
  if (h >= a.num_q_heads) return;
  const int32_t* qs = a.query_start;
  // sequence of token j: the last b with query_start[b] <= j (offsets checked
  // by the attention kernel; a row it did not serve is left untouched)
  int lo = 0, hi = a.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qs[mid] <= j) lo = mid;
    else hi = mid - 1;
  }
  const int b = lo;
  if (j < qs[b] || j >= qs[b + 1]) return;
  const int L = a.seq_lens[b], n = qs[b + 1] - qs[b];
  // the sequence checks of the attention kernel: a bad sequence's rows are 0
  const bool seq_ok = qs[b] >= 0 && qs[b + 1] <= a.num_tokens && L > 0 && n <= L &&
                      n <= a.max_query_len &&
                      L <= a.max_seq_len &&
                      (int64_t)L <= (int64_t)a.max_blocks_per_seq * a.block_size;
  const int np = seq_ok ? min((L + a.part_tokens - 1) / a.part_tokens, a.max_parts) : 0;
  const int64_t row = (int64_t)j * a.num_q_heads + h;
  const float* ml = a.ws_ml + row * a.max_parts * 2;
  float M = -INFINITY;
  bool bad = np == 0;
  for (int i = 0; i < np; ++i) {
    const float l = ml[2 * i + 1];
    if (l < 0.0f) bad = true;
    if (l > 0.0f) M = fmaxf(M, ml[2 * i]);
  }
  constexpr int E = D / 32;                                // elements per lane
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;
  float den = 0.0f;
  if (!bad) {
    for (int i = 0; i < np; ++i) {
      const float l = ml[2 * i + 1];
      if (!(l > 0.0f)) continue;
      const float w = exp2f(ml[2 * i] - M);
      den += w * l;
      const float* src = a.ws_acc + (row * a.max_parts + i) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += w * src[e];
    }
  }
  const float inv = (bad || !(den > 0.0f)) ? 0.0f : 1.0f / den;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + row * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(out + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
}

template <int D, int BS>
kv_status launch_m(const DecodeArgs& a, int tiles, cudaStream_t s) {
  using G = Geo<D, BS, false>;
  constexpr int kSmem = multi_stages<G>() * G::kBlockBytes + 1024;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  kv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != KV_OK) return st;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
      st = cuda_check(cudaFuncSetAttribute(multi_kernel<D, BS>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem),
                      "cudaFuncSetAttribute(multi_kernel)");
      if (st != KV_OK) return st;
      attr_set[dev] = true;
    }
  }
  alignas(64) CUtensorMap km, vm;
  if ((st = make_kv_maps(a, &km, &vm)) != KV_OK) return st;
  const dim3 grid((unsigned)tiles, (unsigned)a.num_kv_heads, (unsigned)a.max_parts);
  if (a.col_max_n == 0) {
    multi_kernel<D, BS><<<grid, kMThreads, kSmem, s>>>(km, vm, a);
    return cuda_check(cudaGetLastError(), "multi_kernel launch");
  }
  // behind the decode kernel's column groups (it needs nothing from them):
  // a programmatic dependent, so it starts during their tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kMThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, multi_kernel<D, BS>, km, vm, a), "multi_kernel launch");
}

kv_status launch_multi_merge(const DecodeArgs& a, cudaStream_t s) {
  if (a.max_parts == 1) return KV_OK;
  const dim3 mgrid((unsigned)a.num_tokens, (unsigned)((a.num_q_heads + 3) / 4));
  if (a.head_dim == 128) multi_merge_kernel<128><<<mgrid, 128, 0, s>>>(a);
  else multi_merge_kernel<64><<<mgrid, 128, 0, s>>>(a);
  return cuda_check(cudaGetLastError(), "multi_merge_kernel launch");
}

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

namespace {

size_t multi_need(int num_tokens, int num_q_heads, int head_dim, int parts) {
  return parts > 1 ? (size_t)num_tokens * num_q_heads * parts * (head_dim + 2) * sizeof(float) : 0;
}

}  // namespace

extern "C" {

size_t pagedkv_multi_workspace_bytes(int num_tokens, int num_q_heads, int head_dim,
                                     int max_seq_len, int block_size) {
  (void)block_size;
  if (num_tokens <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len <= 0) return 0;
  return multi_need(num_tokens, num_q_heads, head_dim, (max_seq_len + 255) / 256);
}

kv_status paged_attention_multi(void* out, const void* q, const void* k_cache,
                                const void* v_cache, const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* seq_lens, const int32_t* query_start, int batch,
                                int num_tokens, int max_query_len, int num_q_heads,
                                int num_kv_heads, int head_dim, int num_blocks, int block_size,
                                int max_seq_len, float scale, kv_dtype dtype, void* workspace,
                                size_t workspace_bytes, void* stream) {
  const char* who = "paged_attention_multi";
  if (batch < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
      max_seq_len <= 0 || max_query_len <= 0 || !valid_dtype(dtype))
    return fail(KV_ERR_INVALID_ARG, "%s: bad sizes", who);
  if (head_dim != 64 && head_dim != 128)
    return fail(KV_ERR_INVALID_ARG, "%s: head_dim must be 64 or 128", who);
  if (block_size != 16 && block_size != 32)
    return fail(KV_ERR_INVALID_ARG, "%s: block_size must be 16 or 32", who);
  const bool q8 = dtype != KV_DTYPE_BF16;
  if (q8 != (k_scale != nullptr) || q8 != (v_scale != nullptr))
    return fail(KV_ERR_INVALID_ARG, "%s: 8-bit pools need k_scale and v_scale; bf16 pools take NULL", who);
  const int GQ = num_q_heads / num_kv_heads;
  // Sequences with few query tokens (at most 4 x 8 / G): the decode
  // kernel's 8 columns per CTA hold (token, head) pairs, 8 / G tokens per
  // column group.  Longer queries: the row-tiled kernel (bf16 pools), in the
  // same call when both kinds occur.
  const int tpg = GQ <= kMaxGroup ? kMaxGroup / GQ : 0;
  const int col_max_n = tpg * kMaxVGroups;               // 0 when G > 8
  const int vgroups = tpg > 0 ? (min(max_query_len, col_max_n) + tpg - 1) / tpg : 0;
  const bool column_path = tpg > 0;                       // some sequences may use it
  const bool row_path = max_query_len > col_max_n;        // some sequences may need it
  if (row_path && q8)
    return fail(KV_ERR_NOT_IMPLEMENTED,
                "%s: 8-bit pools support up to %d query tokens per sequence here", who,
                tpg * kMaxVGroups);
  if (batch == 0 || num_tokens == 0) return KV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start)
    return fail(KV_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(KV_ERR_INVALID_ARG, "%s: out, q and the pools must be 16-byte aligned", who);
  if (num_kv_heads > 65535) return fail(KV_ERR_INVALID_ARG, "%s: too many KV heads", who);
  DeviceInfo di;
  kv_status st = device_info(&di);
  if (st != KV_OK) return st;
  // Upper bound of the row tiles over all sequences: sum ceil(n_b GQ / 64)
  // <= T GQ / 64 + batch (tiles past the real count exit at once).
  const int64_t tiles = ((int64_t)num_tokens * GQ + kMRows - 1) / kMRows + batch;
  if (tiles > 0x7fffffffLL) return fail(KV_ERR_INVALID_ARG, "%s: too many query tokens", who);

  DecodeArgs a = {};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.query_start = query_start;
  a.num_tokens = num_tokens;
  a.max_query_len = max_query_len;
  a.vgroups = column_path ? vgroups : 1;
  a.col_max_n = col_max_n;
  a.flags = di.flags;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.max_seq_len = max_seq_len;
  a.part_tokens = choose_part_tokens((column_path ? batch * vgroups : 0) + (row_path ? (int)tiles : 0),
                                     num_kv_heads, max_seq_len, di.num_sms);
  a.max_parts = (max_seq_len + a.part_tokens - 1) / a.part_tokens;
  if (a.max_parts > 65535) return fail(KV_ERR_INVALID_ARG, "%s: too many partitions", who);
  a.slots = a.max_parts;
  a.scale_log2 = scale * kLog2e;
  a.dtype = dtype;
  const size_t need = multi_need(num_tokens, num_q_heads, head_dim, a.max_parts);
  if (need > 0) {
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
      return fail(KV_ERR_INVALID_ARG,
                  "%s: workspace must be 16-byte aligned and hold %zu bytes "
                  "(pagedkv_multi_workspace_bytes gives a safe size)", who, need);
    a.ws_ml = static_cast<float*>(workspace);
    a.ws_acc = a.ws_ml + (size_t)num_tokens * num_q_heads * a.max_parts * 2;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (column_path && (st = launch_decode(a, s)) != KV_OK) return st;
  if (row_path &&
      (st = launch_multi_tc(a, multi_tc_tiles_upper(num_tokens, num_q_heads, num_kv_heads, batch), s)) !=
          KV_OK)
    return st;
  return launch_multi_merge(a, s);
}

}  // extern "C"
