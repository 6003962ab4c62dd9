// pagedkv_decode.cu -- per-partition decode attention over a paged KV pool.
//
// One CTA serves one (token partition, KV head, sequence) and all G query
// heads grouped on that KV head.  It walks the partition's logical tokens
// through the block table, keeps the online-softmax state (m, l) and an
// unnormalised accumulator per query head, and either writes the normalised
// output (one partition) or its partial (m, l, acc) for the merge kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pagedkv_common.cuh"

namespace pagedkv {
namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Elements [lane * E, lane * E + E) of one K or V row, widened to fp32 and,
// for int8 pools, multiplied by the block's scale.
template <int E, bool kInt8>
__device__ __forceinline__ void load_row(const void* base, int64_t row, int lane, float scale,
                                         float (&x)[E]) {
  if constexpr (kInt8) {
    const int8_t* p = static_cast<const int8_t*>(base) + row + lane * E;
    if constexpr (E == 4) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = (float)(int8_t)(w >> (8 * i)) * scale;
    } else {
      const uint16_t w = *reinterpret_cast<const uint16_t*>(p);
      x[0] = (float)(int8_t)(w & 0xff) * scale;
      x[1] = (float)(int8_t)(w >> 8) * scale;
    }
  } else {
    const uint16_t* p = static_cast<const uint16_t*>(base) + row + lane * E;
    if constexpr (E == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      x[0] = bf16_lo(w.x);
      x[1] = bf16_hi(w.x);
      x[2] = bf16_lo(w.y);
      x[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      x[0] = bf16_lo(w);
      x[1] = bf16_hi(w);
    }
  }
}

template <int D, int G, bool kInt8>
__global__ void __launch_bounds__(kWarps * 32) decode_kernel(DecodeArgs a) {
  constexpr int E = D / 32;  // elements per lane
  const int part = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int Hq = a.num_q_heads, Hkv = a.num_kv_heads, bs = a.block_size;
  const int64_t head0 = (int64_t)b * Hq + (int64_t)hk * G;  // first query row of the group
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);

  const int L = a.seq_lens[b];
  const int64_t table_tokens = (int64_t)a.max_blocks_per_seq * bs;
  if (L <= 0 || L > a.max_seq_len || L > table_tokens) {
    if (part == 0) {
      if (threadIdx.x == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_SEQ_LEN);
      for (int i = threadIdx.x; i < G * D; i += blockDim.x)
        out[head0 * D + i] = __float2bfloat16_rn(0.0f);
    }
    return;
  }
  const int t0 = part * a.part_tokens;
  if (t0 >= L) return;
  const int t1 = min(t0 + a.part_tokens, L);
  const int nparts = (L + a.part_tokens - 1) / a.part_tokens;

  __shared__ float qs[G][D];
  __shared__ float red_m[kWarps][G], red_l[kWarps][G];
  __shared__ float red_acc[kWarps][G][D];
  __shared__ int bad;

  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + head0 * D;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x)
    qs[i / D][i % D] = __bfloat162float(q[i]) * a.scale_log2;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();

  const int32_t* bt = a.block_tables + (int64_t)b * a.max_blocks_per_seq;
  for (int j = t0 / bs + threadIdx.x; j <= (t1 - 1) / bs; j += blockDim.x) {
    const int32_t p = bt[j];
    if (p < 0 || p >= a.num_blocks) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) atomicOr(a.flags, PAGEDKV_FLAG_BAD_BLOCK);
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
      const int g = i / D, e = i % D;
      if (nparts == 1) {
        out[head0 * D + i] = __float2bfloat16_rn(0.0f);
      } else {
        const int64_t r = (head0 + g) * a.max_parts + part;
        a.ws_acc[r * D + e] = 0.0f;
        if (e == 0) {
          a.ws_ml[2 * r] = 0.0f;
          a.ws_ml[2 * r + 1] = -1.0f;  // marks the row bad for the merge
        }
      }
    }
    return;
  }

  float qr[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < E; ++i) qr[g][i] = qs[g][lane * E + i];

  float m[G], l[G], acc[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.0f;
#pragma unroll
    for (int i = 0; i < E; ++i) acc[g][i] = 0.0f;
  }

  for (int t = t0 + warp; t < t1; t += kWarps) {
    const int32_t blk = bt[t / bs];
    const int64_t row = (((int64_t)blk * bs + t % bs) * Hkv + hk) * D;
    const float ks = kInt8 ? a.k_scale[(int64_t)blk * Hkv + hk] : 1.0f;
    const float vs = kInt8 ? a.v_scale[(int64_t)blk * Hkv + hk] : 1.0f;
    float k[E], v[E];
    load_row<E, kInt8>(a.k_cache, row, lane, ks, k);
    load_row<E, kInt8>(a.v_cache, row, lane, vs, v);
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x = 0.0f;
#pragma unroll
      for (int i = 0; i < E; ++i) x = fmaf(qr[g][i], k[i], x);
      s[g] = x;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] += __shfl_xor_sync(0xffffffffu, s[g], off);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m_new = fmaxf(m[g], s[g]);
      const float alpha = exp2f(m[g] - m_new);
      const float p = exp2f(s[g] - m_new);
      l[g] = l[g] * alpha + p;
#pragma unroll
      for (int i = 0; i < E; ++i) acc[g][i] = fmaf(p, v[i], acc[g][i] * alpha);
      m[g] = m_new;
    }
  }

#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      red_m[warp][g] = m[g];
      red_l[warp][g] = l[g];
    }
#pragma unroll
    for (int i = 0; i < E; ++i) red_acc[warp][g][lane * E + i] = acc[g][i];
  }
  __syncthreads();

  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int g = i / D, e = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][g]);
    float num = 0.0f, den = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float c = exp2f(red_m[w][g] - M);  // 0 for a warp that saw no token
      num = fmaf(c, red_acc[w][g][e], num);
      den = fmaf(c, red_l[w][g], den);
    }
    if (nparts == 1) {
      out[head0 * D + i] = __float2bfloat16_rn(num / den);
    } else {
      const int64_t r = (head0 + g) * a.max_parts + part;
      a.ws_acc[r * D + e] = num;
      if (e == 0) {
        a.ws_ml[2 * r] = M;
        a.ws_ml[2 * r + 1] = den;
      }
    }
  }
}

template <int D, bool kInt8>
kv_status launch_d(const DecodeArgs& a, dim3 grid, cudaStream_t s) {
  const int G = a.num_q_heads / a.num_kv_heads;
  switch (G) {
    case 1: decode_kernel<D, 1, kInt8><<<grid, kWarps * 32, 0, s>>>(a); break;
    case 2: decode_kernel<D, 2, kInt8><<<grid, kWarps * 32, 0, s>>>(a); break;
    case 4: decode_kernel<D, 4, kInt8><<<grid, kWarps * 32, 0, s>>>(a); break;
    case 8: decode_kernel<D, 8, kInt8><<<grid, kWarps * 32, 0, s>>>(a); break;
    default: return fail(KV_ERR_INVALID_ARG, "unsupported query group %d", G);
  }
  return cuda_check(cudaGetLastError(), "decode_kernel launch");
}

}  // namespace

kv_status launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.batch > 65535 || a.num_kv_heads > 65535)
    return fail(KV_ERR_INVALID_ARG, "batch and num_kv_heads must be at most 65535");
  const dim3 grid(a.max_parts, a.num_kv_heads, a.batch);
  const bool int8 = a.dtype == KV_DTYPE_INT8;
  if (a.head_dim == 128) return int8 ? launch_d<128, true>(a, grid, s) : launch_d<128, false>(a, grid, s);
  return int8 ? launch_d<64, true>(a, grid, s) : launch_d<64, false>(a, grid, s);
}

}  // namespace pagedkv
