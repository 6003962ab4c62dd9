// pagedkv_common.cuh -- internal declarations shared by the library's CUDA
// translation units (never installed, never seen by callers).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pagedkv {

// Records a message for pagedkv_last_error() (thread-local) and returns `st`.
kv_status fail(kv_status st, const char* fmt, ...);
// Checks a CUDA runtime result; on failure records it and returns KV_ERR_CUDA.
kv_status cuda_check(cudaError_t e, const char* what);

// Per-device facts the launchers need (cached once per device).
struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  unsigned int* flags = nullptr;  // device address of this device's status word
};
kv_status device_info(DeviceInfo* out);

// Bytes of one stored K/V element.
inline int dtype_size(kv_dtype t) { return t == KV_DTYPE_BF16 ? 2 : 1; }
inline bool valid_dtype(kv_dtype t) {
  return t == KV_DTYPE_BF16 || t == KV_DTYPE_INT8 || t == KV_DTYPE_FP8_E4M3;
}
// 16-byte alignment (NULL passes).
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Query heads per KV head the kernels serve (the MMA's N = 8 columns).
constexpr int kMaxGroup = 8;

// Token partitions of the split-K path: powers of two in [256, 2048].
constexpr int kMinPartTokens = 256;
constexpr int kMaxPartTokens = 2048;
// Longest partition the decode kernel's column groups take (its block-id
// table holds 512 blocks: 8192 tokens of 16-token blocks).
constexpr int kMaxColumnPartTokens = 8192;

// log2(e): scores are kept in the base-2 domain so exp() becomes exp2().
constexpr float kLog2e = 1.4426950408889634f;

// Arguments of one decode launch, as resolved on the host.
struct DecodeArgs {
  void* out;                   // bf16 [B, Hq, D]
  const void* q;               // bf16 [B, Hq, D]
  const void* k_cache;         // [NB, bs, Hkv, D]
  const void* v_cache;
  const float* k_scale;        // [NB, Hkv] (int8 only)
  const float* v_scale;
  const int32_t* block_tables; // [B, MB]
  const int32_t* seq_lens;     // [B]
  const void* new_k;           // bf16 [B, Hkv, D] appended in the same launch, or null
  const void* new_v;
  const int32_t* prefix_blocks; // [num_prefix_blocks] shared first blocks of every sequence, or null
  float* ws_ml;                // [B, Hq, slots, 2]   (m, l) per partial
  float* ws_acc;               // [B, Hq, slots, D]   unnormalised acc
  unsigned int* flags;
  int max_blocks_per_seq, batch, num_q_heads, num_kv_heads, head_dim;
  int num_blocks, block_size, max_seq_len;
  int part_tokens, max_parts;  // partitions of tokens [skip_tokens, L)
  int skip_tokens;             // leading tokens attended elsewhere (the shared prefix)
  int num_prefix_blocks;       // = skip_tokens / block_size
  int prefix_chunks;           // prefix partials per row, in slots [max_parts, slots)
  int prefix_part_tokens;      // tokens per prefix partial (a multiple of 128)
  int slots;                   // max_parts + prefix_chunks
  int reverse_parts;           // decode grid: partition max_parts-1-blockIdx.z (else blockIdx.z)
  float scale_log2;            // scale * log2(e)
  kv_dtype dtype;
  // multi-token queries: sequence b's query tokens are q rows
  // query_start[b] .. query_start[b + 1] - 1 (its last tokens); null otherwise
  const int32_t* query_start;  // [batch + 1]
  int num_tokens;
  int max_query_len;           // host bound on query tokens per sequence
  int vgroups;                 // column groups per sequence (decode kernel, multi-token)
  int col_max_n;               // sequences with at most this many queries use the
                               // decode kernel's column groups, longer ones the row tiles
};

// Workspace of one decode call: (m, l) and acc of `slots` partials per query
// row, or nothing when every row has a single partial.
size_t decode_workspace_need(int batch, int num_q_heads, int head_dim, int slots);

// Floats of the (m, l) region of a workspace holding `rows` x `slots`
// partials, rounded up to 16 bytes so that the acc region after it takes
// 16-byte vector loads and stores.
inline size_t ml_region_floats(size_t rows, int slots) {
  return (rows * (size_t)slots * 2 + 3) & ~(size_t)3;
}

// Tensor maps over the K and V pools for this launch's geometry: 4-D
// [NB, bs, Hkv, d], box = one block's rows of one head (128-byte swizzle).
// Encoded once per (device, pool addresses, geometry) and then served from
// a small cache.
kv_status make_kv_maps(const DecodeArgs& a, CUtensorMap* k_map, CUtensorMap* v_map);

// Launches the per-partition decode kernel (with the append fused in when
// new_k is set).
kv_status launch_decode(const DecodeArgs& a, cudaStream_t stream);
// Launches the log-sum-exp merge of the partials (when any row can have more
// than one), as a programmatic dependent of the kernel before it.
kv_status launch_merge(const DecodeArgs& a, cudaStream_t stream);

// Long multi-token queries on the tensor cores with TMEM accumulators
// (pagedkv_multi_tc.cu): `ctas` persistent CTAs over all (KV head,
// partition, 128-row tile) units.
kv_status launch_multi_tc(const DecodeArgs& a, int ctas, cudaStream_t stream);
// The same kernel in shared-prefix mode: every sequence's query rows against
// the prefix blocks, one partial per row and prefix_part_tokens of prefix
// (slots max_parts .. slots-1); releases the kernel queued behind it at once.
kv_status launch_prefix_tc(const DecodeArgs& a, int ctas, cudaStream_t stream);

// Token partition length for `work` independent (row group, KV head) units
// over sequences of up to max_seq_len tokens (power of two in [256,
// max_tokens]).  With split_longest, also at most half of max_seq_len
// (one-token decode).
int choose_part_tokens(int work, int num_kv_heads, int max_seq_len, int num_sms,
                       bool split_longest, int max_tokens = kMaxPartTokens);

}  // namespace pagedkv
