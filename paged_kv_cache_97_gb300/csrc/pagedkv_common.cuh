// pagedkv_common.cuh -- internal declarations shared by the library's CUDA
// translation units (never installed, never seen by callers).
#pragma once

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
  float* ws_ml;                // [B, Hq, max_parts, 2]   (m, l) per partition
  float* ws_acc;               // [B, Hq, max_parts, D]   unnormalised acc
  unsigned int* flags;
  int max_blocks_per_seq, batch, num_q_heads, num_kv_heads, head_dim;
  int num_blocks, block_size, max_seq_len;
  int part_tokens, max_parts;
  float scale_log2;            // scale * log2(e)
  kv_dtype dtype;
};

// Launches the per-partition decode kernel (with the append fused in when
// new_k is set).
kv_status launch_decode(const DecodeArgs& a, cudaStream_t stream);
// Launches the log-sum-exp merge of the partitions (only when max_parts > 1),
// as a programmatic dependent of the decode kernel.
kv_status launch_merge(const DecodeArgs& a, cudaStream_t stream);

}  // namespace pagedkv
