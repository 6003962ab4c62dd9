// pagedkv_noalloc.cu -- paged_attention_decode for callers that cannot hand
// the library any scratch memory.
//
// paged_attention_decode needs a caller-provided workspace when a sequence is
// split into several token partitions (the per-partition (m, l, acc) partials
// live there until the merge kernel combines them).  Some callers cannot
// provide one: a plain C host program that links only this library and the
// CUDA runtime may have no device allocator of its own, and a serving engine
// that reserves all of HBM for its KV pool at start-up forbids allocation
// afterwards (a later cudaMalloc would fail or fragment its arena).  This
// entry point serves them from a fixed scratch array that is part of the
// library's device image: the library never calls cudaMalloc, cudaFree or any
// allocating routine here.
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv_common.cuh"

namespace pagedkv {
namespace {

// The scratch: PAGEDKV_NOALLOC_SCRATCH_BYTES of device memory, resident on
// every GPU that loads the library, from load until process exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PAGEDKV_NOALLOC_SCRATCH_BYTES];

// Device address of this device's copy of the scratch, looked up once per
// device with that device current.  (In host code the array's name is only a
// host-side stand-in; the kernels must get this address instead.)
kv_status scratch_address(void** out) {
  static std::mutex mu;
  static void* cache[64] = {};
  int dev = 0;
  kv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != KV_OK) return st;
  if (dev < 0 || dev >= 64) return fail(KV_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    st = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch),
                    "cudaGetSymbolAddress(no-alloc scratch)");
    if (st != KV_OK) return st;
    cache[dev] = p;
  }
  *out = cache[dev];
  return KV_OK;
}

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" size_t pagedkv_noalloc_scratch_bytes(void) { return PAGEDKV_NOALLOC_SCRATCH_BYTES; }

extern "C" kv_status paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
    int num_blocks, int block_size, int max_seq_len, float scale, kv_dtype dtype, void* stream) {
  // An empty batch and every shape paged_attention_decode rejects are left to
  // its own argument checks (they return before it touches a device or reads
  // the workspace), so those callers get its messages.
  const bool shape_ok = batch > 0 && num_q_heads > 0 && num_kv_heads > 0 &&
                        num_q_heads % num_kv_heads == 0 && num_q_heads / num_kv_heads <= kMaxGroup &&
                        (head_dim == 64 || head_dim == 128) && (block_size == 16 || block_size == 32) &&
                        max_blocks_per_seq > 0 && num_blocks > 0 && max_seq_len > 0 &&
                        valid_dtype(dtype);
  if (!shape_ok)
    return paged_attention_decode(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                  max_blocks_per_seq, seq_lens, batch, num_q_heads,
                                  num_kv_heads, head_dim, num_blocks, block_size, max_seq_len,
                                  scale, dtype, nullptr, 0, stream);
  // Scratch this call needs: the partials of every (sequence, query head,
  // partition) when a sequence spans several partitions, with the partition
  // paged_attention_decode will choose on this device.
  DeviceInfo di;
  kv_status st = device_info(&di);
  if (st != KV_OK) return st;
  const int part = choose_part_tokens(batch, num_kv_heads, max_seq_len, di.num_sms, true);
  const int parts = (max_seq_len + part - 1) / part;
  const size_t need = decode_workspace_need(batch, num_q_heads, head_dim, parts);
  if (need > PAGEDKV_NOALLOC_SCRATCH_BYTES)
    return fail(KV_ERR_INVALID_ARG,
                "paged_attention_decode_noalloc: this shape needs %zu bytes of scratch, more "
                "than the fixed %u bytes; use paged_attention_decode with a workspace",
                need, (unsigned)PAGEDKV_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != KV_OK) return st;
  // Nothing in the scratch needs clearing: every partial the merge kernel
  // reads is written earlier in the same call.
  return paged_attention_decode(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                max_blocks_per_seq, seq_lens, batch, num_q_heads, num_kv_heads,
                                head_dim, num_blocks, block_size, max_seq_len, scale, dtype,
                                scratch, PAGEDKV_NOALLOC_SCRATCH_BYTES, stream);
}
