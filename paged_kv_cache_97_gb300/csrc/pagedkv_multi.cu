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
// Each sequence goes to one of two kernels in the same call:
//   * few query tokens (n_b <= 4 x 8 / G): the decode kernel, whose 8 MMA
//     columns per CTA then hold (token, head) pairs (pagedkv_decode.cu);
//   * longer queries: the tensor-core kernel with TMEM accumulators
//     (pagedkv_multi_tc.cu), 128 rows per CTA.
// Both write the normalised output (one partition) or per-row (m, l, acc)
// partials that the log-sum-exp merge below combines (“LLM 推理优化技术全景”,
// 在线 Softmax; “Flash Attention v2 的改进”).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pagedkv_common.cuh"
#include "pagedkv_device.cuh"

namespace pagedkv {
namespace {

// Column groups the decode kernel may serve per sequence (8 columns each):
// longer queries go to the tensor-core kernel.
constexpr int kMaxVGroups = 4;

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
  // column group.  Longer queries: the tensor-core kernel (bf16 pools), in the
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
  // Upper bound of the tensor-core kernel's 128-row tiles over all sequences
  // (tiles past the real count exit at once).
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
  a.part_tokens = choose_part_tokens((column_path ? batch * vgroups : 0) + (row_path ? (int)tiles : 0),
                                     num_kv_heads, max_seq_len, di.num_sms);
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
    a.ws_acc = a.ws_ml + (size_t)num_tokens * num_q_heads * a.max_parts * 2;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (column_path && (st = launch_decode(a, s)) != KV_OK) return st;
  if (row_path && (st = launch_multi_tc(a, (int)tiles, s)) != KV_OK) return st;
  return launch_multi_merge(a, s);
}

}  // extern "C"
