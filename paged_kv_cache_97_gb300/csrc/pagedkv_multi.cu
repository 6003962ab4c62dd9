// pagedkv_multi.cu -- attention of multi-token queries over the paged pool:
// speculative verification (“让 Agent 跑得快：LLM 推理服务”, §六 投机解码: the
// target model scores the gamma draft tokens in one parallel pass) and
// chunked prefill batched with decodes (“LLM 推理优化技术全景”, SARATHI: a
// 512-token prefill chunk plus as many decodes as fit).
//
// Sequence b has n_b query tokens, its last n_b tokens (appended before the
// attention: by the caller, or by pagedkv_multi_step's append launch), q rows
// query_start[b] .. query_start[b + 1] - 1.  Query token i sits at
// position L_b - n_b + i and attends positions 0 .. L_b - n_b + i (causal).
//
// Each sequence goes to one of three kernels in the same call:
//   * one column group (n_b <= 8 / G): the decode kernel, whose 8 MMA
//     columns per CTA then hold (token, head) pairs (pagedkv_decode.cu);
//   * a few column groups (8 / G < n_b <= 4 x 8 / G): in calls without
//     long queries on bf16 pools the 16-column kernel (pagedkv_multi_m16.cu):
//     16 / G tokens per m-tile, every such sequence in one CTA, so each block
//     is read once per (sequence, KV head); otherwise the decode kernel's
//     column groups;
//   * longer queries: the tensor-core kernel with TMEM accumulators
//     (pagedkv_multi_tc.cu), 128 rows per CTA.
// All write the normalised output (one partition) or per-row (m, l, acc)
// partials that the log-sum-exp merge below combines (“LLM 推理优化技术全景”,
// 在线 Softmax; “Flash Attention v2 的改进”).
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cuda_runtime.h>

#include "pagedkv_common.cuh"
#include "pagedkv_device.cuh"

namespace pagedkv {

// pagedkv_api.cu: slot mapping + append of a multi-token step's new rows.
kv_status launch_append_tokens(const void* new_k, const void* new_v, void* k_cache, void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, int max_blocks,
                               const int32_t* seq_lens, const int32_t* query_start, int batch,
                               int num_tokens, int max_query_len, int num_blocks, int block_size,
                               int num_kv_heads, int head_dim, kv_dtype dtype, unsigned int* flags,
                               cudaStream_t s);

// pagedkv_multi_m16.cu: sequences with more than n_lo query tokens,
// `vgroups` 16-column m-tiles per sequence at most (bf16 pools), longest
// sequences first when `rank` is set.
kv_status launch_multi_m16(const DecodeArgs& a, int n_lo, int vgroups, bool rank, cudaStream_t s);

namespace {

// Column groups the decode kernel may serve per sequence (8 columns each):
// longer queries go to the tensor-core kernel.
constexpr int kMaxVGroups = 4;
// Columns of one m-tile of the 16-column kernel.
constexpr int kM16Cols = 16;

// Log-sum-exp merge of the partition partials of every (query token, head)
// row: one warp per row, four heads per CTA.  Partials of partitions wholly
// past a row's position hold l = 0 and are skipped (their acc is never read
// into the sum); a partial marked l < 0 (bad sequence or a wait that gave up)
// zeroes the row.
template <int D>
__global__ void __launch_bounds__(128) multi_merge_kernel(const DecodeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x, h = blockIdx.y * 4 + warp;
  const int32_t* qs = a.query_start;
  // sequence of token j: the last b with query_start[b] <= j, found by the
  // whole CTA in rounds of 128 samples of query_start (one round for up to
  // 128 sequences).  Offsets are checked by the attention kernels; a row they
  // did not serve is left untouched.
  int lo = 0, hi = a.batch;                              // b in [lo, hi)
  while (hi - lo > 1) {
    const int step = (hi - lo + 127) / 128;
    const int idx = lo + (int)threadIdx.x * step;
    const int cnt = __syncthreads_count(idx < hi && qs[idx] <= j);
    if (cnt == 0) return;                                // before every sequence (CTA-uniform)
    lo += (cnt - 1) * step;
    hi = min(lo + step, hi);
  }
  const int b = lo;
  if (h >= a.num_q_heads || j < qs[b] || j >= qs[b + 1]) return;
  const int L = a.seq_lens[b], n = qs[b + 1] - qs[b];
  // the sequence checks of the attention kernels: a bad sequence's rows are 0
  const bool seq_ok = qs[b] >= 0 && qs[b + 1] <= a.num_tokens && L > 0 && n <= L &&
                      n <= a.max_query_len && L <= a.max_seq_len &&
                      (int64_t)L <= (int64_t)a.max_blocks_per_seq * a.block_size;
  const int np = seq_ok ? min((L + a.part_tokens - 1) / a.part_tokens, a.max_parts) : 0;
  const int64_t row = (int64_t)j * a.num_q_heads + h;
  const float* ml = a.ws_ml + row * a.max_parts * 2;
  // pass 1 (32 partials per round): the largest m among l > 0, any bad partial
  float M = -INFINITY;
  bool bad = np == 0;
  for (int i = lane; i < np; i += 32) {
    const float l = ml[2 * i + 1];
    bad |= l < 0.0f;
    if (l > 0.0f) M = fmaxf(M, ml[2 * i]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  bad = __any_sync(0xffffffffu, bad);
  // pass 2: each lane owns D / 32 consecutive elements
  constexpr int E = D / 32;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;
  float den = 0.0f;
  if (!bad) {
#pragma unroll 4
    for (int i = 0; i < np; ++i) {
      const float m = ml[2 * i], l = ml[2 * i + 1];
      const float* src = a.ws_acc + (row * a.max_parts + i) * D + lane * E;
      float x[E];
      if constexpr (E == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        x[0] = v.x;
        x[1] = v.y;
      }
      if (l > 0.0f) {
        const float w = exp2f(m - M);
        den = fmaf(w, l, den);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(w, x[e], acc[e]);
      }
    }
  }
  const float inv = (bad || !(den > 0.0f)) ? 0.0f : 1.0f / den;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + row * D + lane * E;
  uint32_t w2[E / 2];
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    __nv_bfloat162 v = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
    w2[e / 2] = *reinterpret_cast<uint32_t*>(&v);
  }
  if constexpr (E == 4) *reinterpret_cast<uint2*>(out) = make_uint2(w2[0], w2[1]);
  else *reinterpret_cast<uint32_t*>(out) = w2[0];
}

kv_status launch_multi_merge(const DecodeArgs& a, cudaStream_t s) {
  if (a.max_parts == 1) return KV_OK;
  const dim3 mgrid((unsigned)a.num_tokens, (unsigned)((a.num_q_heads + 3) / 4));
  if (a.head_dim == 128) multi_merge_kernel<128><<<mgrid, 128, 0, s>>>(a);
  else multi_merge_kernel<64><<<mgrid, 128, 0, s>>>(a);
  return cuda_check(cudaGetLastError(), "multi_merge_kernel launch");
}

// A side stream and two events per (host thread, device): the tensor-core
// kernel runs there, concurrently with the decode kernel's column groups on
// the caller's stream (fork from it, join before the merge; the same pattern
// records as two parallel branches under graph capture).  Thread-local, so
// callers on different host threads never share an event.
struct SideLane {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  ~SideLane() {
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
    if (stream) cudaStreamDestroy(stream);
  }
};

kv_status side_lane(int dev, SideLane** out) {
  static thread_local SideLane lanes[64];
  SideLane& l = lanes[dev];
  if (!l.stream) {
    kv_status st;
    if ((st = cuda_check(cudaEventCreateWithFlags(&l.fork, cudaEventDisableTiming), "cudaEventCreate")) != KV_OK ||
        (st = cuda_check(cudaEventCreateWithFlags(&l.join, cudaEventDisableTiming), "cudaEventCreate")) != KV_OK ||
        (st = cuda_check(cudaStreamCreateWithFlags(&l.stream, cudaStreamNonBlocking), "cudaStreamCreate")) != KV_OK)
      return st;
  }
  *out = &l;
  return KV_OK;
}


}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

namespace {

size_t multi_need(int num_tokens, int num_q_heads, int head_dim, int parts) {
  if (parts <= 1) return 0;
  const size_t rows = (size_t)num_tokens * num_q_heads;
  return (ml_region_floats(rows, parts) + rows * parts * head_dim) * sizeof(float);
}

}  // namespace

extern "C" {

size_t pagedkv_multi_workspace_bytes(int num_tokens, int num_q_heads, int head_dim,
                                     int max_seq_len, int block_size) {
  (void)block_size;
  if (num_tokens <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len <= 0) return 0;
  return multi_need(num_tokens, num_q_heads, head_dim, (max_seq_len + 255) / 256);
}

// Token partition of a multi-token call (the same choice for both kernels
// of one call).  Column groups alone take partitions up to 8192 tokens:
// their per-CTA start and the merge cost more than the tail of fewer, longer
// CTAs (speculative verification, 64 sequences of 512..4096 tokens with 5
// queries each: 512-token partitions 215.5 us per step, 1024 182.1, 2048
// 166.1, one 8192-token partition 159.6).  With the tensor-core kernel in
// the call, at most the 2048 tokens its block-id table holds.
static int multi_part_tokens(int batch, int num_tokens, int max_query_len, int num_q_heads,
                             int num_kv_heads, int max_seq_len, int num_sms) {
  const int GQ = num_q_heads / num_kv_heads;
  const int tpg = GQ <= kMaxGroup ? kMaxGroup / GQ : 0;
  const int col_max_n = tpg * kMaxVGroups;
  const int vgroups = tpg > 0 ? (min(max_query_len, col_max_n) + tpg - 1) / tpg : 0;
  const bool column_path = tpg > 0;
  const bool row_path = max_query_len > col_max_n;
  const int64_t tiles = ((int64_t)num_tokens * GQ + 127) / 128 + batch;
  return choose_part_tokens((column_path ? batch * vgroups : 0) + (row_path ? (int)tiles : 0),
                            num_kv_heads, max_seq_len, num_sms, false,
                            row_path ? kMaxPartTokens : kMaxColumnPartTokens);
}

int pagedkv_multi_partition_tokens(int batch, int num_tokens, int max_query_len, int num_q_heads,
                                   int num_kv_heads, int max_seq_len) {
  DeviceInfo di;
  if (batch <= 0 || num_tokens <= 0 || max_query_len <= 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || num_q_heads % num_kv_heads || max_seq_len <= 0 ||
      ((int64_t)num_tokens * (num_q_heads / num_kv_heads) + 127) / 128 + batch > 0x7fffffffLL ||
      device_info(&di) != KV_OK)
    return 0;
  return multi_part_tokens(batch, num_tokens, max_query_len, num_q_heads, num_kv_heads,
                           max_seq_len, di.num_sms);
}

}  // extern "C"

// paged_attention_multi, and with new_k / new_v set the append of the step's
// tokens before it on the same stream (pagedkv_multi_step): every argument
// is checked before the first launch.
static kv_status multi_impl(const char* who, bool append, void* out, const void* q, const void* new_k,
                            const void* new_v, const void* k_cache, const void* v_cache,
                            const float* k_scale, const float* v_scale,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* seq_lens, const int32_t* query_start, int batch,
                            int num_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                            int head_dim, int num_blocks, int block_size, int max_seq_len,
                            float scale, kv_dtype dtype, void* workspace, size_t workspace_bytes,
                            void* stream) {
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
  // column group; in calls of few-query sequences alone on bf16 pools,
  // those with more than one group's tokens go to the 16-column kernel
  // instead (16 / G tokens per CTA).  Longer queries: the tensor-core kernel,
  // in the same call when both kinds occur.
  const int tpg = GQ <= kMaxGroup ? kMaxGroup / GQ : 0;
  const int col_max_n = tpg * kMaxVGroups;               // 0 when G > 8
  const int vgroups = tpg > 0 ? (min(max_query_len, col_max_n) + tpg - 1) / tpg : 0;
  const bool column_path = tpg > 0;                       // some sequences may use it
  const bool row_path = max_query_len > col_max_n;        // some sequences may need it
  // (batches that also hold long queries keep the column groups for all
  // few-query sequences: the tensor-core kernel shares the GPU with them)
  const bool m16_path = column_path && !row_path && dtype == KV_DTYPE_BF16 && max_query_len > tpg;
  const int tpg16 = column_path ? kM16Cols / GQ : 0;
  const int vgroups16 = m16_path ? (min(max_query_len, col_max_n) + tpg16 - 1) / tpg16 : 0;
  if (batch == 0 || num_tokens == 0) return KV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start ||
      (append && (!new_k || !new_v)))
    return fail(KV_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(new_k) || !aligned16(new_v))
    return fail(KV_ERR_INVALID_ARG, "%s: out, q, the new rows and the pools must be 16-byte aligned",
                who);
  if (num_kv_heads > 65535) return fail(KV_ERR_INVALID_ARG, "%s: too many KV heads", who);
  DeviceInfo di;
  kv_status st = device_info(&di);
  if (st != KV_OK) return st;
  // Upper bound of the tensor-core kernel's 128-row tiles over all sequences
  // (it sizes the persistent grid; the kernel counts the real tiles).
  const int64_t tiles = ((int64_t)num_tokens * GQ + 127) / 128 + batch;
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
  a.part_tokens = multi_part_tokens(batch, num_tokens, max_query_len, num_q_heads, num_kv_heads,
                                    max_seq_len, di.num_sms);
  a.max_parts = (max_seq_len + a.part_tokens - 1) / a.part_tokens;
  if (a.max_parts > 65535) return fail(KV_ERR_INVALID_ARG, "%s: too many partitions", who);
  if (row_path && tiles * num_kv_heads * a.max_parts > 0x7fffffffLL)
    return fail(KV_ERR_INVALID_ARG, "%s: too many query tokens", who);
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
    a.ws_acc = a.ws_ml + ml_region_floats((size_t)num_tokens * num_q_heads, a.max_parts);
  }
  cudaStream_t s = (cudaStream_t)stream;
  // Persistent tensor-core CTAs, one per SM (each takes the whole TMEM),
  // never more than the units (pairs of row tiles <= tiles).
  auto tc_ctas = [&](int per_sm) {
    return (int)std::min<int64_t>(tiles * num_kv_heads * a.max_parts, (int64_t)di.num_sms * per_sm);
  };
  if (append &&
      (st = launch_append_tokens(new_k, new_v, const_cast<void*>(k_cache),
                                 const_cast<void*>(v_cache), k_scale, v_scale, block_tables,
                                 max_blocks_per_seq, seq_lens, query_start, batch, num_tokens,
                                 max_query_len, num_blocks, block_size, num_kv_heads, head_dim,
                                 dtype, di.flags, s)) != KV_OK)
    return st;
  if (m16_path) {
    // the decode kernel's column groups for sequences of one group's tokens,
    // then the 16-column CTAs, longest sequences first.  When every sequence
    // has max_query_len tokens (T = batch x max_query_len, none above the
    // bound: a longer one is flagged by the 16-column kernel) none has one
    // group's tokens, and the decode launch is left out.
    const bool uniform = (int64_t)num_tokens == (int64_t)batch * max_query_len;
    DecodeArgs one = a;
    one.col_max_n = tpg;
    one.vgroups = 1;
    if ((!uniform && (st = launch_decode(one, s)) != KV_OK) ||
        (st = launch_multi_m16(a, tpg, vgroups16, true, s)) != KV_OK)
      return st;
  } else if (row_path && column_path) {
    // the tensor-core kernel (tensor-bound) beside the column groups (HBM-bound)
    SideLane* lane = nullptr;
    if ((st = side_lane(di.device, &lane)) != KV_OK ||
        (st = cuda_check(cudaEventRecord(lane->fork, s), "cudaEventRecord")) != KV_OK ||
        (st = cuda_check(cudaStreamWaitEvent(lane->stream, lane->fork, 0), "cudaStreamWaitEvent")) != KV_OK ||
        (st = launch_multi_tc(a, tc_ctas(1), lane->stream)) != KV_OK ||
        (st = cuda_check(cudaEventRecord(lane->join, lane->stream), "cudaEventRecord")) != KV_OK)
      return st;
    st = launch_decode(a, s);
    const kv_status sj = cuda_check(cudaStreamWaitEvent(s, lane->join, 0), "cudaStreamWaitEvent");
    if (st != KV_OK) return st;
    if (sj != KV_OK) return sj;
  } else if (column_path) {
    if ((st = launch_decode(a, s)) != KV_OK) return st;
  } else if (row_path) {
    if ((st = launch_multi_tc(a, tc_ctas(1), s)) != KV_OK) return st;
  }
  return launch_multi_merge(a, s);
}

extern "C" {

kv_status paged_attention_multi(void* out, const void* q, const void* k_cache,
                                const void* v_cache, const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* seq_lens, const int32_t* query_start, int batch,
                                int num_tokens, int max_query_len, int num_q_heads,
                                int num_kv_heads, int head_dim, int num_blocks, int block_size,
                                int max_seq_len, float scale, kv_dtype dtype, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return multi_impl("paged_attention_multi", false, out, q, nullptr, nullptr, k_cache, v_cache, k_scale,
                    v_scale, block_tables, max_blocks_per_seq, seq_lens, query_start, batch,
                    num_tokens, max_query_len, num_q_heads, num_kv_heads, head_dim, num_blocks,
                    block_size, max_seq_len, scale, dtype, workspace, workspace_bytes, stream);
}

kv_status pagedkv_multi_step(void* out, const void* q, const void* new_k, const void* new_v,
                             void* k_cache, void* v_cache, const float* k_scale,
                             const float* v_scale, const int32_t* block_tables,
                             int max_blocks_per_seq, const int32_t* seq_lens,
                             const int32_t* query_start, int batch, int num_tokens,
                             int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
                             int num_blocks, int block_size, int max_seq_len, float scale,
                             kv_dtype dtype, void* workspace, size_t workspace_bytes,
                             void* stream) {
  return multi_impl("pagedkv_multi_step", true, out, q, new_k, new_v, k_cache, v_cache, k_scale,
                    v_scale, block_tables, max_blocks_per_seq, seq_lens, query_start, batch,
                    num_tokens, max_query_len, num_q_heads, num_kv_heads, head_dim, num_blocks,
                    block_size, max_seq_len, scale, dtype, workspace, workspace_bytes, stream);
}

}  // extern "C"
