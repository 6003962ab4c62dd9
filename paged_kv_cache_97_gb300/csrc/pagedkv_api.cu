// pagedkv_api.cu -- the C ABI of libpagedkv: argument checks, slot mapping
// and append kernels, the split-K merge kernel, and the device status word.
// The block pool is in pagedkv_pool.cu, the decode kernel in
// pagedkv_decode.cu, the tensor-core kernel for long multi-token queries and
// the shared prefix in pagedkv_multi_tc.cu.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <mutex>
#include <vector>

#include "pagedkv_common.cuh"
#include "pagedkv_device.cuh"

namespace pagedkv {

static thread_local char g_last_error[512] = "";

kv_status fail(kv_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

kv_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return KV_OK;
  return fail(KV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// One status word per device; kernels atomicOr PAGEDKV_FLAG_* bits into it.
__device__ unsigned int g_status_word;

kv_status device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  kv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != KV_OK) return st;
  if (dev < 0 || dev >= 64) return fail(KV_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = cache[dev];
  if (d.device != dev) {
    int sms = 0;
    st = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                    "cudaDeviceGetAttribute(MultiProcessorCount)");
    if (st != KV_OK) return st;
    void* p = nullptr;
    st = cuda_check(cudaGetSymbolAddress(&p, g_status_word), "cudaGetSymbolAddress(status word)");
    if (st != KV_OK) return st;
    d.num_sms = sms;
    d.flags = static_cast<unsigned int*>(p);
    d.device = dev;
  }
  *out = d;
  return KV_OK;
}

// ---------------------------------------------------------------------------
// Slot mapping
// ---------------------------------------------------------------------------

// Slot of position p of sequence s: block_tables[s][p / bs] * bs + p % bs.
__device__ __forceinline__ int64_t slot_of(const int32_t* __restrict__ block_tables,
                                           int max_blocks, int s, int p, int bs,
                                           int num_blocks, unsigned int* flags) {
  int logical = p / bs;
  if (logical >= max_blocks) {
    atomicOr(flags, PAGEDKV_FLAG_BAD_SEQ_LEN);
    return -1;
  }
  int32_t phys = block_tables[(int64_t)s * max_blocks + logical];
  if (phys < 0 || phys >= num_blocks) {
    atomicOr(flags, PAGEDKV_FLAG_BAD_BLOCK);
    return -1;
  }
  return (int64_t)phys * bs + (p % bs);
}

__global__ void decode_slots_kernel(const int32_t* __restrict__ block_tables, int max_blocks,
                                    const int32_t* __restrict__ seq_lens, int batch, int bs,
                                    int num_blocks, int64_t* __restrict__ slots,
                                    unsigned int* flags) {
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  int L = seq_lens[b];
  if (L <= 0) {
    atomicOr(flags, PAGEDKV_FLAG_BAD_SEQ_LEN);
    slots[b] = -1;
    return;
  }
  slots[b] = slot_of(block_tables, max_blocks, b, L - 1, bs, num_blocks, flags);
}

__global__ void token_slots_kernel(const int32_t* __restrict__ block_tables, int max_blocks,
                                   const int32_t* __restrict__ seq_idx,
                                   const int32_t* __restrict__ positions, int n, int bs,
                                   int num_blocks, int64_t* __restrict__ slots,
                                   unsigned int* flags) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  int p = positions[i];
  int s = seq_idx ? seq_idx[i] : i;
  slots[i] = p < 0 ? -1 : slot_of(block_tables, max_blocks, s, p, bs, num_blocks, flags);
}

// ---------------------------------------------------------------------------
// Append: one thread moves 8 elements (16 bytes of bf16 input).
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Eight bf16 values as eight 8-bit codes (int8, or E4M3 when kFp8).
template <bool kFp8>
__device__ __forceinline__ uint2 quantize8(uint4 x, float s) {
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t o[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo = dev::code8<kFp8>(bf16_lo(w[i]), s);
    uint32_t hi = dev::code8<kFp8>(bf16_hi(w[i]), s);
    o[i / 2] |= (lo | (hi << 8)) << (16 * (i % 2));
  }
  return make_uint2(o[0], o[1]);
}

// kKind: the pool dtype (KV_DTYPE_BF16, KV_DTYPE_INT8, KV_DTYPE_FP8_E4M3).
template <int kKind>
__global__ void append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                              void* __restrict__ k_cache, void* __restrict__ v_cache,
                              const float* __restrict__ k_scale,
                              const float* __restrict__ v_scale,
                              const int64_t* __restrict__ slots, int num_tokens,
                              int num_blocks, int bs, int num_kv_heads, int head_dim,
                              unsigned int* flags) {
  const int chunks_per_head = head_dim / 8;
  const int chunks_per_token = num_kv_heads * chunks_per_head;
  int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)num_tokens * chunks_per_token) return;
  int token = (int)(idx / chunks_per_token);
  int c = (int)(idx % chunks_per_token);
  int h = c / chunks_per_head;
  int64_t slot = slots[token];
  if (slot < 0) return;
  if (slot >= (int64_t)num_blocks * bs) {
    atomicOr(flags, PAGEDKV_FLAG_BAD_SLOT);
    return;
  }
  // Destination chunk: element ((slot * Hkv + h) * D + e0) of the pool.
  int64_t dst = (slot * num_kv_heads + h) * chunks_per_head + (c % chunks_per_head);
  uint4 kx = k[idx], vx = v[idx];
  if (kKind != KV_DTYPE_BF16) {
    int64_t sidx = (slot / bs) * num_kv_heads + h;
    constexpr bool kFp8 = kKind == KV_DTYPE_FP8_E4M3;
    reinterpret_cast<uint2*>(k_cache)[dst] = quantize8<kFp8>(kx, k_scale[sidx]);
    reinterpret_cast<uint2*>(v_cache)[dst] = quantize8<kFp8>(vx, v_scale[sidx]);
  } else {
    reinterpret_cast<uint4*>(k_cache)[dst] = kx;
    reinterpret_cast<uint4*>(v_cache)[dst] = vx;
  }
}

// Append of a multi-token step: the slot mapping and reshape_and_cache in
// one pass.  Sequence b's n_b new tokens are rows query_start[b] ..
// query_start[b] + n_b - 1 of new_k / new_v ([T, Hkv, D] bf16) and go to
// positions L_b - n_b .. L_b - 1 (its last tokens: seq_lens already counts
// them).  One thread per 16-byte piece of a row; a row's sequence is the last
// b with query_start[b] <= row.  A sequence whose offsets do
// not fit (rows outside [0, T), n_b > L_b or n_b > max_query_len) writes
// nothing and sets PAGEDKV_FLAG_BAD_SEQ_LEN; a position past the table or an
// entry outside the pool sets the flag slot_of sets and skips the write.
template <int kKind>
__global__ void append_tokens_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                     void* __restrict__ k_cache, void* __restrict__ v_cache,
                                     const float* __restrict__ k_scale,
                                     const float* __restrict__ v_scale,
                                     const int32_t* __restrict__ block_tables, int max_blocks,
                                     const int32_t* __restrict__ seq_lens,
                                     const int32_t* __restrict__ query_start, int batch,
                                     int num_tokens, int max_query_len, int num_blocks, int bs,
                                     int num_kv_heads, int head_dim, unsigned int* flags) {
  const int chunks_per_head = head_dim / 8;
  const int chunks_per_token = num_kv_heads * chunks_per_head;
  // The sequence of the CTA's first row, found by the whole CTA in rounds of
  // blockDim.x samples of query_start (one round for up to 256 sequences);
  // each thread then walks on to its own row's sequence (a CTA spans few
  // rows).
  const int64_t idx0 = (int64_t)blockIdx.x * blockDim.x;
  const int t0 = (int)(idx0 / chunks_per_token);
  int lo = 0, hi = batch;                                // b in [lo, hi)
  while (hi - lo > 1) {
    const int step = (hi - lo + (int)blockDim.x - 1) / (int)blockDim.x;
    const int j = lo + (int)threadIdx.x * step;
    const int cnt = __syncthreads_count(j < hi && query_start[j] <= t0);
    if (cnt == 0) break;                                 // before every sequence: start at lo
    lo += (cnt - 1) * step;
    hi = min(lo + step, hi);
  }
  const int64_t idx = idx0 + threadIdx.x;
  if (idx >= (int64_t)num_tokens * chunks_per_token) return;
  const int t = (int)(idx / chunks_per_token);           // row of new_k / new_v
  const int c = (int)(idx % chunks_per_token);
  int b = lo;
  while (b + 1 < batch && query_start[b + 1] <= t) ++b;
  const int q0 = query_start[b], n = query_start[b + 1] - q0;
  if (t < q0 || t - q0 >= n) return;                     // a row of no sequence
  const int L = seq_lens[b];
  if (q0 < 0 || q0 > num_tokens - n || n > L || n > max_query_len) {
    if (t == q0 && c == 0) atomicOr(flags, PAGEDKV_FLAG_BAD_SEQ_LEN);
    return;
  }
  const int i = t - q0;
  const int64_t slot = slot_of(block_tables, max_blocks, b, L - n + i, bs, num_blocks, flags);
  if (slot < 0) return;
  const int h = c / chunks_per_head;
  const int64_t dst = (slot * num_kv_heads + h) * chunks_per_head + (c % chunks_per_head);
  const uint4 kx = k[idx], vx = v[idx];
  if (kKind != KV_DTYPE_BF16) {
    const int64_t sidx = (slot / bs) * num_kv_heads + h;
    constexpr bool kFp8 = kKind == KV_DTYPE_FP8_E4M3;
    reinterpret_cast<uint2*>(k_cache)[dst] = quantize8<kFp8>(kx, k_scale[sidx]);
    reinterpret_cast<uint2*>(v_cache)[dst] = quantize8<kFp8>(vx, v_scale[sidx]);
  } else {
    reinterpret_cast<uint4*>(k_cache)[dst] = kx;
    reinterpret_cast<uint4*>(v_cache)[dst] = vx;
  }
}

// Launches append_tokens_kernel (arguments checked by the caller).
kv_status launch_append_tokens(const void* new_k, const void* new_v, void* k_cache, void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, int max_blocks,
                               const int32_t* seq_lens, const int32_t* query_start, int batch,
                               int num_tokens, int max_query_len, int num_blocks, int block_size,
                               int num_kv_heads, int head_dim, kv_dtype dtype, unsigned int* flags,
                               cudaStream_t s) {
  const int64_t threads = (int64_t)num_tokens * num_kv_heads * (head_dim / 8);
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return fail(KV_ERR_INVALID_ARG, "multi-token append: too many tokens");
  const uint4 *k = static_cast<const uint4*>(new_k), *v = static_cast<const uint4*>(new_v);
  if (dtype == KV_DTYPE_INT8)
    append_tokens_kernel<KV_DTYPE_INT8><<<(unsigned)grid, block, 0, s>>>(
        k, v, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks, seq_lens, query_start,
        batch, num_tokens, max_query_len, num_blocks, block_size, num_kv_heads, head_dim, flags);
  else if (dtype == KV_DTYPE_FP8_E4M3)
    append_tokens_kernel<KV_DTYPE_FP8_E4M3><<<(unsigned)grid, block, 0, s>>>(
        k, v, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks, seq_lens, query_start,
        batch, num_tokens, max_query_len, num_blocks, block_size, num_kv_heads, head_dim, flags);
  else
    append_tokens_kernel<KV_DTYPE_BF16><<<(unsigned)grid, block, 0, s>>>(
        k, v, k_cache, v_cache, nullptr, nullptr, block_tables, max_blocks, seq_lens, query_start,
        batch, num_tokens, max_query_len, num_blocks, block_size, num_kv_heads, head_dim, flags);
  return cuda_check(cudaGetLastError(), "append_tokens_kernel launch");
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge.  One CTA per (sequence, KV head), `wpr` warps per query
// head; a row's partials are its partitions of tokens [skip, L) (slots
// 0 .. np-1) and, with a shared prefix, the prefix kernel's chunks (slots
// max_parts .. slots-1):
//   M = max_i m_i, w_i = 2^(m_i - M), out = sum_i w_i acc_i / sum_i w_i l_i
// The warps of a row take its partials in turn (a long context has dozens:
// one warp walking them alone waits on memory once per few partials) and add
// their sums through shared memory.  A partial whose l is negative marks a
// bad block: the row becomes zeros.  Launched as a programmatic dependent of
// the kernel before it: the wait returns once that grid has completed and
// its partials are visible.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(1024)
    merge_kernel(__nv_bfloat16* __restrict__ out, const float* __restrict__ ws_ml,
                 const float* __restrict__ ws_acc, const int32_t* __restrict__ seq_lens,
                 int num_q_heads, int num_kv_heads, int head_dim, int part_tokens, int max_parts,
                 int slots, int skip, int prefix_chunks, int max_len, int wpr) {
  extern __shared__ float red[];                   // [G][wpr][32][5] when wpr > 1
  const int b = blockIdx.x / num_kv_heads, hk = blockIdx.x % num_kv_heads;
  const int G = num_q_heads / num_kv_heads;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = w / wpr, sub = w % wpr;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int L = seq_lens[b];
  // (CTA-uniform exits, before the barrier below)
  if (L <= skip || L > max_len) return;             // invalid rows were zeroed by the decode kernel
  const int np = (L - skip + part_tokens - 1) / part_tokens;
  const int total = np + (skip > 0 ? prefix_chunks : 0);
  if (total <= 1) return;                           // written whole by the decode kernel
  const int64_t row = (int64_t)b * num_q_heads + (int64_t)hk * G + g;
  const float* ml = ws_ml + row * slots * 2;
  const float* acc = ws_acc + row * slots * head_dim;
  // pass 1: the largest m and any bad partial (every warp of the row)
  float M = -INFINITY;
  bool bad = false;
  for (int i = lane; i < total; i += 32) {
    const int s = i < np ? i : max_parts + (i - np);
    M = fmaxf(M, ml[2 * s]);
    bad |= ml[2 * s + 1] < 0.0f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  bad = __any_sync(0xffffffffu, bad);
  // pass 2: this warp's partials sub, sub + wpr, ...; each lane owns 4
  // consecutive elements
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.0f;
  const int e0 = lane * 4;
  if (!bad) {
#pragma unroll 8
    for (int i = sub; i < total; i += wpr) {
      const int s = i < np ? i : max_parts + (i - np);
      const float wgt = exp2f(ml[2 * s] - M);
      den = fmaf(wgt, ml[2 * s + 1], den);
      if (e0 < head_dim) {
        const float4 x = *reinterpret_cast<const float4*>(acc + (int64_t)s * head_dim + e0);
        num.x = fmaf(wgt, x.x, num.x);
        num.y = fmaf(wgt, x.y, num.y);
        num.z = fmaf(wgt, x.z, num.z);
        num.w = fmaf(wgt, x.w, num.w);
      }
    }
  }
  if (wpr > 1) {
    float* r = red + ((g * wpr + sub) * 32 + lane) * 5;
    r[0] = num.x;
    r[1] = num.y;
    r[2] = num.z;
    r[3] = num.w;
    r[4] = den;
    __syncthreads();
    if (sub == 0) {
      for (int k = 1; k < wpr; ++k) {
        const float* o = red + ((g * wpr + k) * 32 + lane) * 5;
        num.x += o[0];
        num.y += o[1];
        num.z += o[2];
        num.w += o[3];
        den += o[4];
      }
    }
  }
  if (sub == 0 && e0 < head_dim) {
    const float r = bad ? 0.0f : 1.0f / den;
    __nv_bfloat162 lo = __floats2bfloat162_rn(bad ? 0.0f : num.x * r, bad ? 0.0f : num.y * r);
    __nv_bfloat162 hi = __floats2bfloat162_rn(bad ? 0.0f : num.z * r, bad ? 0.0f : num.w * r);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + row * head_dim + e0) = v;
  }
}

size_t decode_workspace_need(int batch, int num_q_heads, int head_dim, int slots) {
  if (slots <= 1) return 0;
  const size_t rows = (size_t)batch * num_q_heads;
  return (ml_region_floats(rows, slots) + rows * slots * head_dim) * sizeof(float);
}

// Longest valid sequence: bounded by the host hint and by the table.
static int valid_len_limit(const DecodeArgs& a) {
  const int64_t table = (int64_t)a.max_blocks_per_seq * a.block_size;
  return (int)(table < a.max_seq_len ? table : a.max_seq_len);
}

kv_status launch_merge(const DecodeArgs& a, cudaStream_t stream) {
  if (a.max_parts <= 1 && a.skip_tokens == 0) return KV_OK;
  // With a shared prefix the partials come from two kernels: a plain launch
  // waits for both; otherwise launch behind the decode kernel (PDL).
  const int G = a.num_q_heads / a.num_kv_heads;
  // warps per row: about 8 partials each, at most 1024 threads per CTA
  const int most = a.max_parts + a.prefix_chunks;
  int wpr = (most + 7) / 8;
  if (wpr > 32 / G) wpr = 32 / G;
  if (wpr < 1) wpr = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.batch * a.num_kv_heads));
  cfg.blockDim = dim3((unsigned)(32 * G * wpr));
  cfg.dynamicSmemBytes = wpr > 1 ? (size_t)G * wpr * 32 * 5 * sizeof(float) : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.prefix_chunks > 0 ? 0 : 1;
  return cuda_check(cudaLaunchKernelEx(&cfg, merge_kernel, static_cast<__nv_bfloat16*>(a.out),
                                       (const float*)a.ws_ml, (const float*)a.ws_acc, a.seq_lens,
                                       a.num_q_heads, a.num_kv_heads, a.head_dim, a.part_tokens,
                                       a.max_parts, a.slots, a.skip_tokens, a.prefix_chunks,
                                       valid_len_limit(a), wpr),
                    "merge_kernel launch");
}

// ---------------------------------------------------------------------------
// Partition size
// ---------------------------------------------------------------------------

// Largest power-of-two partition in [256, 2048] that still gives at least
// 8 CTAs per SM over (sequence, KV head, partition) and, with split_longest,
// splits a sequence of the longest length in two.  Longer partitions measured
// slower on GB300 for one-token decode (fewer, longer CTAs leave a longer
// tail; with lengths spread as widely as the lognormal suffixes of a
// shared-prefix batch, the CTAs of the longest sequences alone set the step
// time), but not for multi-token queries, whose column groups re-read each
// block and whose partials cost more to merge.  The environment variable
// PAGEDKV_PARTITION_TOKENS (a multiple of 256, read on every call) overrides it.
int choose_part_tokens(int batch, int num_kv_heads, int max_seq_len, int num_sms,
                       bool split_longest, int max_tokens) {
  const char* s = getenv("PAGEDKV_PARTITION_TOKENS");
  const int env = s ? atoi(s) : 0;
  if (env >= kMinPartTokens && env <= max_tokens && env % kMinPartTokens == 0) return env;
  const int64_t target = 8LL * num_sms;
  int pt = max_tokens;
  while (pt > kMinPartTokens &&
         ((int64_t)batch * num_kv_heads * ((max_seq_len + pt - 1) / pt) < target ||
          (split_longest && 2 * pt > max_seq_len)))
    pt /= 2;
  return pt;
}

}  // namespace pagedkv

using namespace pagedkv;

// ===========================================================================
// C ABI
// ===========================================================================

extern "C" {

const char* pagedkv_last_error(void) { return g_last_error; }

kv_status pagedkv_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* seq_lens, int batch, int block_size,
                               int num_blocks, int64_t* slot_mapping, void* stream) {
  if (batch < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0)
    return fail(KV_ERR_INVALID_ARG, "pagedkv_slot_mapping: bad sizes");
  if (batch == 0) return KV_OK;
  if (!block_tables || !seq_lens || !slot_mapping)
    return fail(KV_ERR_INVALID_ARG, "pagedkv_slot_mapping: NULL pointer");
  DeviceInfo di;
  kv_status st = device_info(&di);
  if (st != KV_OK) return st;
  decode_slots_kernel<<<(batch + 255) / 256, 256, 0, (cudaStream_t)stream>>>(
      block_tables, max_blocks_per_seq, seq_lens, batch, block_size, num_blocks, slot_mapping,
      di.flags);
  return cuda_check(cudaGetLastError(), "decode_slots_kernel launch");
}

kv_status pagedkv_token_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* seq_idx, const int32_t* positions,
                                     int num_tokens, int block_size, int num_blocks,
                                     int64_t* slot_mapping, void* stream) {
  if (num_tokens < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0)
    return fail(KV_ERR_INVALID_ARG, "pagedkv_token_slot_mapping: bad sizes");
  if (num_tokens == 0) return KV_OK;
  if (!block_tables || !positions || !slot_mapping)
    return fail(KV_ERR_INVALID_ARG, "pagedkv_token_slot_mapping: NULL pointer");
  DeviceInfo di;
  kv_status st = device_info(&di);
  if (st != KV_OK) return st;
  token_slots_kernel<<<(num_tokens + 255) / 256, 256, 0, (cudaStream_t)stream>>>(
      block_tables, max_blocks_per_seq, seq_idx, positions, num_tokens, block_size, num_blocks,
      slot_mapping, di.flags);
  return cuda_check(cudaGetLastError(), "token_slots_kernel launch");
}

kv_status reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                            const float* k_scale, const float* v_scale,
                            const int64_t* slot_mapping, int num_tokens, int num_blocks,
                            int block_size, int num_kv_heads, int head_dim, kv_dtype dtype,
                            void* stream) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
      (head_dim != 64 && head_dim != 128) || !valid_dtype(dtype))
    return fail(KV_ERR_INVALID_ARG,
                "reshape_and_cache: bad geometry (head_dim must be 64 or 128, sizes positive)");
  if (num_tokens == 0) return KV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping)
    return fail(KV_ERR_INVALID_ARG, "reshape_and_cache: NULL pointer");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(KV_ERR_INVALID_ARG, "reshape_and_cache: k, v and the pools must be 16-byte aligned");
  const bool q8 = dtype != KV_DTYPE_BF16;
  if (q8 != (k_scale != nullptr) || q8 != (v_scale != nullptr))
    return fail(KV_ERR_INVALID_ARG,
                "reshape_and_cache: 8-bit pools need k_scale and v_scale; bf16 pools take NULL");
  DeviceInfo di;
  kv_status st = device_info(&di);
  if (st != KV_OK) return st;
  const int64_t threads = (int64_t)num_tokens * num_kv_heads * (head_dim / 8);
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return fail(KV_ERR_INVALID_ARG, "reshape_and_cache: too many tokens");
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == KV_DTYPE_INT8)
    append_kernel<KV_DTYPE_INT8><<<(unsigned)grid, block, 0, s>>>(
        (const uint4*)k, (const uint4*)v, k_cache, v_cache, k_scale, v_scale, slot_mapping,
        num_tokens, num_blocks, block_size, num_kv_heads, head_dim, di.flags);
  else if (dtype == KV_DTYPE_FP8_E4M3)
    append_kernel<KV_DTYPE_FP8_E4M3><<<(unsigned)grid, block, 0, s>>>(
        (const uint4*)k, (const uint4*)v, k_cache, v_cache, k_scale, v_scale, slot_mapping,
        num_tokens, num_blocks, block_size, num_kv_heads, head_dim, di.flags);
  else
    append_kernel<KV_DTYPE_BF16><<<(unsigned)grid, block, 0, s>>>(
        (const uint4*)k, (const uint4*)v, k_cache, v_cache, nullptr, nullptr, slot_mapping,
        num_tokens, num_blocks, block_size, num_kv_heads, head_dim, di.flags);
  return cuda_check(cudaGetLastError(), "append_kernel launch");
}

size_t pagedkv_workspace_bytes(int batch, int num_q_heads, int head_dim, int max_seq_len,
                               int block_size) {
  (void)block_size;
  if (batch <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len <= 0) return 0;
  const int parts = (max_seq_len + kMinPartTokens - 1) / kMinPartTokens;
  return decode_workspace_need(batch, num_q_heads, head_dim, parts);
}

int pagedkv_partition_tokens(int batch, int num_kv_heads, int max_seq_len, int block_size) {
  (void)block_size;
  DeviceInfo di;
  if (batch <= 0 || num_kv_heads <= 0 || max_seq_len <= 0 || device_info(&di) != KV_OK) return 0;
  return choose_part_tokens(batch, num_kv_heads, max_seq_len, di.num_sms, true);
}

// Prefix partials per row.  The tensor-core prefix kernel takes units of
// (128-row tile, KV head, prefix partial); a partial covers a multiple of 128
// prefix tokens and at most kMaxPartTokens.  The product runs beside the
// decode kernel and only has to finish before it, so rows get as few partials
// as that allows: ceil(T / kMaxPartTokens) for T prefix tokens (fewer partials
// to write and merge; 256 sequences behind an 800-token shared prefix: one
// 896-token partial 119.3 us per step, two 122.0, three 123.9).  pagedkv_prefix_workspace_bytes sizes for this.
static int prefix_chunk_count(int prefix_tokens) {
  return (prefix_tokens + kMaxPartTokens - 1) / kMaxPartTokens;
}

static void choose_prefix_parts(int prefix_tokens, int* part_tokens, int* chunks) {
  const int nc = prefix_chunk_count(prefix_tokens);
  const int per = (prefix_tokens + nc - 1) / nc;
  *part_tokens = (per + 127) / 128 * 128;
  *chunks = (prefix_tokens + *part_tokens - 1) / *part_tokens;   // <= nc
}

// Shared body of paged_attention_decode, pagedkv_decode_step and
// pagedkv_decode_step_prefix.
static kv_status decode_common(void* out, const void* q, const void* new_k, const void* new_v,
                               const void* k_cache, const void* v_cache, const float* k_scale,
                               const float* v_scale, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                               int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                               int block_size, int max_seq_len, float scale, kv_dtype dtype,
                               const int32_t* prefix_blocks, int num_prefix_blocks,
                               void* workspace, size_t workspace_bytes, void* stream,
                               const char* who) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
      max_blocks_per_seq <= 0 || num_blocks <= 0 || max_seq_len <= 0 || !valid_dtype(dtype))
    return fail(KV_ERR_INVALID_ARG, "%s: bad sizes", who);
  const int G = num_q_heads / num_kv_heads;
  if (G > 8)
    return fail(KV_ERR_INVALID_ARG, "%s: at most 8 query heads per KV head (got %d)", who, G);
  if (head_dim != 64 && head_dim != 128)
    return fail(KV_ERR_INVALID_ARG, "%s: head_dim must be 64 or 128", who);
  if (block_size != 16 && block_size != 32)
    return fail(KV_ERR_INVALID_ARG, "%s: block_size must be 16 or 32", who);
  if (batch == 0) return KV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens)
    return fail(KV_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(new_k) || !aligned16(new_v))
    return fail(KV_ERR_INVALID_ARG, "%s: out, q, k, v and the pools must be 16-byte aligned", who);
  const bool q8 = dtype != KV_DTYPE_BF16;
  if (q8 != (k_scale != nullptr) || q8 != (v_scale != nullptr))
    return fail(KV_ERR_INVALID_ARG,
                "%s: 8-bit pools need k_scale and v_scale; bf16 pools take NULL", who);
  const int skip = num_prefix_blocks * block_size;
  if (num_prefix_blocks < 0 || (num_prefix_blocks > 0 && !prefix_blocks) ||
      num_prefix_blocks > max_blocks_per_seq || (num_prefix_blocks > 0 && max_seq_len <= skip))
    return fail(KV_ERR_INVALID_ARG,
                "%s: the shared prefix needs 1..max_blocks_per_seq block ids and sequences "
                "longer than it", who);
  DeviceInfo di;
  kv_status st = device_info(&di);
  if (st != KV_OK) return st;

  DecodeArgs a = {};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.new_k = new_k;
  a.new_v = new_v;
  a.flags = di.flags;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.max_seq_len = max_seq_len;
  a.part_tokens = choose_part_tokens(batch, num_kv_heads, max_seq_len - skip, di.num_sms, true);
  a.max_parts = (max_seq_len - skip + a.part_tokens - 1) / a.part_tokens;
  // Few partitions per sequence: the last ones hold the ragged remainders of
  // the sequences long enough to have them; dispatching those first leaves
  // full partitions for the last wave (measured 4 % faster on B64 sequences
  // of 512..4096 tokens, 2 % slower with 64 partitions per sequence).
  a.reverse_parts = a.max_parts <= 8;
  a.skip_tokens = skip;
  a.num_prefix_blocks = num_prefix_blocks;
  a.prefix_chunks = 0;
  a.prefix_part_tokens = 0;
  if (num_prefix_blocks > 0)
    choose_prefix_parts(skip, &a.prefix_part_tokens, &a.prefix_chunks);
  a.slots = a.max_parts + a.prefix_chunks;
  a.prefix_blocks = prefix_blocks;
  a.scale_log2 = scale * kLog2e;
  a.dtype = dtype;
  a.ws_ml = nullptr;
  a.ws_acc = nullptr;
  const size_t need = decode_workspace_need(batch, num_q_heads, head_dim, a.slots);
  if (need > 0) {
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
      return fail(KV_ERR_INVALID_ARG,
                  "%s: workspace must be 16-byte aligned and hold %zu bytes "
                  "(pagedkv_workspace_bytes gives a safe size)", who, need);
    a.ws_ml = static_cast<float*>(workspace);
    a.ws_acc = a.ws_ml + ml_region_floats((size_t)batch * num_q_heads, a.slots);
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (num_prefix_blocks > 0) {
    // The prefix product is small beside the decode's KV stream and only has
    // to finish before it: about 16 chunks of 128 keys per CTA but no fewer
    // than a quarter of the SMs (each of those SMs still holds two decode
    // CTAs, enough loads in flight to keep its share of HBM bandwidth).
    // Workload of 256 sequences behind an 800-token prefix: 38 CTAs 123.4 us
    // per step, 76 CTAs 123.8, 152 CTAs 128.5, 304 CTAs 130.3 (three partials).
    // (units: pairs of 128-row tiles x KV heads x prefix partials; one CTA per SM)
    const int G = num_q_heads / num_kv_heads;
    const int64_t units = (int64_t)((batch * G + 255) / 256) * num_kv_heads * a.prefix_chunks;
    const int64_t chunks = units * 2 * (a.prefix_part_tokens / 128);
    int64_t ctas = (chunks + 15) / 16;
    const int64_t quarter = di.num_sms / 4 > 0 ? di.num_sms / 4 : 1;
    if (ctas < quarter) ctas = quarter;
    if (ctas > di.num_sms) ctas = di.num_sms;
    if (ctas > units) ctas = units;
    if ((st = launch_prefix_tc(a, (int)ctas, s)) != KV_OK) return st;
  }
  st = launch_decode(a, s);
  if (st != KV_OK) return st;
  return launch_merge(a, s);
}

kv_status paged_attention_decode(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const float* k_scale, const float* v_scale,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* seq_lens, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, int num_blocks, int block_size,
                                 int max_seq_len, float scale, kv_dtype dtype, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return decode_common(out, q, nullptr, nullptr, k_cache, v_cache, k_scale, v_scale,
                       block_tables, max_blocks_per_seq, seq_lens, batch, num_q_heads,
                       num_kv_heads, head_dim, num_blocks, block_size, max_seq_len, scale, dtype,
                       nullptr, 0, workspace, workspace_bytes, stream, "paged_attention_decode");
}

kv_status pagedkv_decode_step(void* out, const void* q, const void* k, const void* v,
                              void* k_cache, void* v_cache, const float* k_scale,
                              const float* v_scale, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                              int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                              int block_size, int max_seq_len, float scale, kv_dtype dtype,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (batch > 0 && (!k || !v))
    return fail(KV_ERR_INVALID_ARG, "pagedkv_decode_step: NULL k or v");
  return decode_common(out, q, k, v, k_cache, v_cache, k_scale, v_scale, block_tables,
                       max_blocks_per_seq, seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                       num_blocks, block_size, max_seq_len, scale, dtype, nullptr, 0, workspace,
                       workspace_bytes, stream, "pagedkv_decode_step");
}

kv_status pagedkv_decode_step_prefix(void* out, const void* q, const void* k, const void* v,
                                     void* k_cache, void* v_cache, const float* k_scale,
                                     const float* v_scale, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                                     int num_q_heads, int num_kv_heads, int head_dim,
                                     int num_blocks, int block_size, int max_seq_len,
                                     float scale, kv_dtype dtype, const int32_t* prefix_blocks,
                                     int num_prefix_blocks, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (batch > 0 && ((k == nullptr) != (v == nullptr)))
    return fail(KV_ERR_INVALID_ARG, "pagedkv_decode_step_prefix: give both k and v, or neither");
  if (batch > 0 && num_prefix_blocks <= 0)
    return fail(KV_ERR_INVALID_ARG, "pagedkv_decode_step_prefix: num_prefix_blocks must be >= 1");
  return decode_common(out, q, k, v, k_cache, v_cache, k_scale, v_scale, block_tables,
                       max_blocks_per_seq, seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                       num_blocks, block_size, max_seq_len, scale, dtype, prefix_blocks,
                       num_prefix_blocks, workspace, workspace_bytes, stream,
                       "pagedkv_decode_step_prefix");
}

size_t pagedkv_prefix_workspace_bytes(int batch, int num_q_heads, int head_dim, int max_seq_len,
                                      int block_size, int num_prefix_blocks) {
  if (batch <= 0 || num_q_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_prefix_blocks <= 0)
    return 0;
  const int rest = max_seq_len - num_prefix_blocks * block_size;
  if (rest <= 0) return 0;
  const int parts = (rest + kMinPartTokens - 1) / kMinPartTokens;
  return decode_workspace_need(batch, num_q_heads, head_dim,
                               parts + prefix_chunk_count(num_prefix_blocks * block_size));
}

kv_status pagedkv_get_status(void* stream, unsigned int* device_flags) {
  DeviceInfo di;
  kv_status st = device_info(&di);
  if (st != KV_OK) return st;
  unsigned int h = 0;
  cudaStream_t s = (cudaStream_t)stream;
  st = cuda_check(cudaMemcpyAsync(&h, di.flags, sizeof h, cudaMemcpyDeviceToHost, s),
                  "pagedkv_get_status: read");
  if (st == KV_OK) st = cuda_check(cudaStreamSynchronize(s), "pagedkv_get_status: sync");
  if (st == KV_OK && h)
    st = cuda_check(cudaMemsetAsync(di.flags, 0, sizeof h, s), "pagedkv_get_status: clear");
  if (st == KV_OK) st = cuda_check(cudaStreamSynchronize(s), "pagedkv_get_status: sync");
  if (device_flags) *device_flags = h;
  if (st != KV_OK) return st;
  if (h) return fail(KV_ERR_DEVICE_INDEX, "device status word 0x%x", h);
  return KV_OK;
}

}  // extern "C"
