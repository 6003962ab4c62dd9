// pagedkv_pool.cu -- the physical block pool (host bookkeeping: FIFO free
// list, reference counts, copy-on-write before a decode append) and the
// device kernel that copies whole blocks for copy-on-write.
//
// “LLM 推理引擎深度解析”, §2.1 (PagedKVCache): the free list starts as every
// block id in order, allocation takes ids from its front (all or none) and
// finished sequences return theirs to its back.
// “让 Agent 跑得快”, §七 (前缀缓存): a full block's hash chains its parent
// block's hash, its tokens and optional extra keys; a new request looks its
// prompt's blocks up in order and takes a reference on every hit (prefill
// resumes at the first miss); freed blocks stay findable in the free queue
// until allocation reuses them (least recently freed first).
// “让 Agent 跑得快：LLM 推理服务”, §二 (Copy-on-Write：Beam Search 的内存优化):
// candidate sequences forked from one prefix map the same physical blocks,
// each holding a reference; a sequence about to write a token into a block
// whose count is above one first copies it and repoints its table entry; a
// block whose count drops to zero goes back to the pool.  §五 (共享前缀): only
// the current decode token writes, so that write is the only trigger.
#include <cuda_runtime.h>

#include <unordered_map>
#include <vector>

#include "pagedkv_common.cuh"

using namespace pagedkv;

namespace {

// The free blocks in queue order, as an intrusive doubly linked list so that
// a cached block can leave from the middle in O(1) when a request hits it.
struct FreeQueue {
  std::vector<int32_t> prev, next;  // -1 = none
  int32_t head = -1, tail = -1;
  size_t count = 0;

  void init(int n) {
    prev.assign(n, -1);
    next.assign(n, -1);
    for (int i = 0; i < n; ++i) push_back(i);
  }
  size_t size() const { return count; }
  void push_back(int32_t id) {
    prev[id] = tail;
    next[id] = -1;
    if (tail >= 0) next[tail] = id;
    else head = id;
    tail = id;
    ++count;
  }
  void remove(int32_t id) {
    if (prev[id] >= 0) next[prev[id]] = next[id];
    else head = next[id];
    if (next[id] >= 0) prev[next[id]] = prev[id];
    else tail = prev[id];
    prev[id] = next[id] = -1;
    --count;
  }
  int32_t pop_front() {
    const int32_t id = head;
    remove(id);
    return id;
  }
};

// What the prefix cache knows of a registered full block.
struct CachedBlock {
  bool registered = false;
  uint64_t hash = 0, parent = 0, extra_key = 0;
  std::vector<int32_t> tokens;
};

// FNV-1a, 64-bit (offset basis 0xcbf29ce484222325, prime 0x100000001b3):
// for every input byte, h ^= byte, then h *= prime (mod 2^64).
constexpr uint64_t kFnvBasis = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

inline uint64_t fnv_bytes(uint64_t h, uint64_t v, int nbytes) {
  for (int i = 0; i < nbytes; ++i) {
    h ^= (v >> (8 * i)) & 0xffu;
    h *= kFnvPrime;
  }
  return h;
}

// Hash of one full block: FNV-1a over the parent hash (8 bytes), the extra
// key (8 bytes) and the block's token ids (4 bytes each), little-endian.
uint64_t block_hash(uint64_t parent, const int32_t* tokens, int bs, uint64_t extra_key) {
  uint64_t h = kFnvBasis;
  h = fnv_bytes(h, parent, 8);
  h = fnv_bytes(h, extra_key, 8);
  for (int i = 0; i < bs; ++i) h = fnv_bytes(h, (uint32_t)tokens[i], 4);
  return h;
}

}  // namespace

struct kv_pool {
  int num_blocks, block_size, num_kv_heads, head_dim;
  kv_dtype dtype;
  FreeQueue free_list;            // front = next to hand out
  std::vector<int32_t> refs;      // references per block; 0 = free
  int used = 0;                   // blocks with refs > 0
  std::vector<CachedBlock> cache;                    // per block
  std::unordered_map<uint64_t, int32_t> by_hash;     // registered blocks
};

namespace {

// Drops a block's prefix-cache entry (its contents are about to change).
void evict(kv_pool* p, int32_t id) {
  CachedBlock& c = p->cache[id];
  if (!c.registered) return;
  auto it = p->by_hash.find(c.hash);
  if (it != p->by_hash.end() && it->second == id) p->by_hash.erase(it);
  c = CachedBlock();
}

// Takes the front of the free list with one reference (evicting whatever
// the prefix cache still kept in that block).
int32_t take_block(kv_pool* p) {
  const int32_t id = p->free_list.pop_front();
  evict(p, id);
  p->refs[id] = 1;
  ++p->used;
  return id;
}

// Drops one reference; a block left with none goes to the back of the list
// (a registered block stays findable there until it is taken again).
void drop_ref(kv_pool* p, int32_t id) {
  if (--p->refs[id] == 0) {
    p->free_list.push_back(id);
    --p->used;
  }
}

// One copy-on-write copy: bytes [chunk * kChunk, +kChunk) of block src of one
// pool tensor to block dst.  Each thread issues kCopyUnroll 16-byte loads
// before its stores, so several loads per thread are in flight (source and
// destination share a base pointer, so the compiler cannot reorder a plain
// copy loop by itself).
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int kChunk = kCopyThreads * kCopyUnroll * 16;   // 16 KB

__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   float* __restrict__ k_scale, float* __restrict__ v_scale,
                   const int32_t* __restrict__ pairs, int num_blocks, int block_bytes,
                   int num_kv_heads, unsigned int* flags) {
  const int pair = blockIdx.y;
  const int src = pairs[2 * pair], dst = pairs[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0)
      atomicOr(flags, PAGEDKV_FLAG_BAD_BLOCK);
    return;
  }
  if (src == dst) return;
  uint4* pool = blockIdx.z == 0 ? k_cache : v_cache;
  const int64_t words = block_bytes / 16;
  const uint4* from = pool + (int64_t)src * words;
  uint4* to = pool + (int64_t)dst * words;
  const int64_t w0 = (int64_t)blockIdx.x * (kChunk / 16) + threadIdx.x;
  uint4 r[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t w = w0 + u * kCopyThreads;
    if (w < words) r[u] = __ldcs(from + w);              // read once: streaming
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t w = w0 + u * kCopyThreads;
    if (w < words) to[w] = r[u];
  }
  if (blockIdx.x == 0) {  // the block's scales ([num_blocks, num_kv_heads] fp32)
    float* sc = blockIdx.z == 0 ? k_scale : v_scale;
    if (sc != nullptr)
      for (int h = threadIdx.x; h < num_kv_heads; h += kCopyThreads)
        sc[(int64_t)dst * num_kv_heads + h] = sc[(int64_t)src * num_kv_heads + h];
  }
}

}  // namespace

extern "C" {

kv_status kv_pool_create(int num_blocks, int block_size, int num_kv_heads, int head_dim,
                         kv_dtype dtype, kv_pool** out) {
  if (!out) return fail(KV_ERR_INVALID_ARG, "kv_pool_create: out is NULL");
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      !valid_dtype(dtype))
    return fail(KV_ERR_INVALID_ARG, "kv_pool_create: sizes must be positive and dtype valid");
  kv_pool* p = new kv_pool;
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->num_kv_heads = num_kv_heads;
  p->head_dim = head_dim;
  p->dtype = dtype;
  p->free_list.init(num_blocks);
  p->refs.assign(num_blocks, 0);
  p->cache.assign(num_blocks, CachedBlock());
  *out = p;
  return KV_OK;
}

void kv_pool_destroy(kv_pool* pool) { delete pool; }

size_t kv_pool_block_bytes(const kv_pool* p) {
  if (!p) return 0;
  return 2ull * p->block_size * p->num_kv_heads * p->head_dim * dtype_size(p->dtype);
}

kv_status kv_pool_alloc(kv_pool* p, int n, int32_t* out_ids) {
  if (!p || n < 0 || (n > 0 && !out_ids))
    return fail(KV_ERR_INVALID_ARG, "kv_pool_alloc: bad arguments");
  if ((size_t)n > p->free_list.size())
    return fail(KV_ERR_OUT_OF_BLOCKS, "kv_pool_alloc: %d blocks requested, %zu free", n,
                p->free_list.size());
  for (int i = 0; i < n; ++i) out_ids[i] = take_block(p);
  return KV_OK;
}

kv_status kv_pool_fork(kv_pool* p, const int32_t* ids, int n) {
  if (!p || n < 0 || (n > 0 && !ids)) return fail(KV_ERR_INVALID_ARG, "kv_pool_fork: bad arguments");
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= p->num_blocks || p->refs[ids[i]] == 0)
      return fail(KV_ERR_INVALID_ARG, "kv_pool_fork: block %d is not allocated", ids[i]);
  for (int i = 0; i < n; ++i) ++p->refs[ids[i]];
  return KV_OK;
}

kv_status kv_pool_free(kv_pool* p, const int32_t* ids, int n) {
  if (!p || n < 0 || (n > 0 && !ids)) return fail(KV_ERR_INVALID_ARG, "kv_pool_free: bad arguments");
  std::vector<int32_t> drops(p->num_blocks, 0);
  for (int i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= p->num_blocks || ++drops[id] > p->refs[id])
      return fail(KV_ERR_INVALID_ARG,
                  "kv_pool_free: block %d is not allocated (or freed more often than it is held)",
                  id);
  }
  for (int i = 0; i < n; ++i) drop_ref(p, ids[i]);
  return KV_OK;
}

int kv_pool_refcount(const kv_pool* p, int32_t id) {
  if (!p || id < 0 || id >= p->num_blocks) return -1;
  return p->refs[id];
}

kv_status kv_pool_stats(const kv_pool* p, int* used, int* free_blocks) {
  if (!p) return fail(KV_ERR_INVALID_ARG, "kv_pool_stats: pool is NULL");
  if (used) *used = p->used;
  if (free_blocks) *free_blocks = (int)p->free_list.size();
  return KV_OK;
}

kv_status kv_pool_prepare_append(kv_pool* p, int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* seq_lens, int batch, int32_t* copy_pairs,
                                 int* num_copies) {
  if (!p || batch < 0 || max_blocks_per_seq <= 0 ||
      (batch > 0 && (!block_tables || !seq_lens || !copy_pairs)) || !num_copies)
    return fail(KV_ERR_INVALID_ARG, "kv_pool_prepare_append: bad arguments");
  *num_copies = 0;
  const int bs = p->block_size;
  // Pass 1: check every sequence and count the blocks the step takes, with
  // the references that earlier copies in this batch drop (a block shared by
  // k sequences of the batch is copied k - 1 times; the last writer keeps it).
  std::vector<int32_t> dropped(p->num_blocks, 0);
  size_t need = 0;
  for (int b = 0; b < batch; ++b) {
    const int L = seq_lens[b];
    if (L <= 0 || (L - 1) / bs >= max_blocks_per_seq)
      return fail(KV_ERR_INVALID_ARG,
                  "kv_pool_prepare_append: sequence %d: length %d outside (0, %d]", b, L,
                  max_blocks_per_seq * bs);
    const int j = (L - 1) / bs;
    if ((L - 1) % bs == 0) {  // the token opens a block
      ++need;
      continue;
    }
    const int32_t id = block_tables[(int64_t)b * max_blocks_per_seq + j];
    if (id < 0 || id >= p->num_blocks || p->refs[id] == 0)
      return fail(KV_ERR_INVALID_ARG,
                  "kv_pool_prepare_append: sequence %d writes into block %d, which is not "
                  "allocated", b, id);
    if (p->refs[id] - dropped[id] > 1) {
      ++need;
      ++dropped[id];
    }
  }
  if (need > p->free_list.size())
    return fail(KV_ERR_OUT_OF_BLOCKS, "kv_pool_prepare_append: %zu blocks needed, %zu free", need,
                p->free_list.size());
  // Pass 2: apply, sequences in order, blocks from the front of the list.
  int n = 0;
  for (int b = 0; b < batch; ++b) {
    const int L = seq_lens[b], j = (L - 1) / bs;
    int32_t& entry = block_tables[(int64_t)b * max_blocks_per_seq + j];
    if ((L - 1) % bs == 0) {
      entry = take_block(p);
      continue;
    }
    const int32_t id = entry;
    if (p->refs[id] > 1) {
      const int32_t fresh = take_block(p);
      drop_ref(p, id);
      entry = fresh;
      copy_pairs[2 * n] = id;
      copy_pairs[2 * n + 1] = fresh;
      ++n;
    }
  }
  *num_copies = n;
  // (fresh blocks come from the free list, shared sources are in use: the
  // list is a valid batch for pagedkv_copy_blocks by construction)
  return pagedkv_check_block_pairs(copy_pairs, n, p->num_blocks);
}

kv_status pagedkv_check_block_pairs(const int32_t* block_pairs, int num_pairs, int num_blocks) {
  if (num_pairs < 0 || num_blocks <= 0 || (num_pairs > 0 && !block_pairs))
    return fail(KV_ERR_INVALID_ARG, "pagedkv_check_block_pairs: bad arguments");
  std::vector<uint8_t> role(num_blocks, 0);          // bit 0: a source, bit 1: a destination
  for (int i = 0; i < num_pairs; ++i) {
    const int32_t src = block_pairs[2 * i], dst = block_pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
      return fail(KV_ERR_INVALID_ARG, "block pair %d (%d, %d): id outside [0, %d)", i, src, dst,
                  num_blocks);
    if (src != dst) role[src] |= 1;
  }
  for (int i = 0; i < num_pairs; ++i) {
    const int32_t src = block_pairs[2 * i], dst = block_pairs[2 * i + 1];
    if (src == dst) continue;
    if (role[dst] & 2)
      return fail(KV_ERR_INVALID_ARG, "block pair %d (%d, %d): destination %d appears twice", i,
                  src, dst, dst);
    if (role[dst] & 1)
      return fail(KV_ERR_INVALID_ARG, "block pair %d (%d, %d): destination %d is also a source", i,
                  src, dst, dst);
    role[dst] |= 2;
  }
  return KV_OK;
}

uint64_t pagedkv_block_hash(uint64_t parent_hash, const int32_t* tokens, int block_size,
                            uint64_t extra_key) {
  if (!tokens || block_size <= 0) return 0;
  return block_hash(parent_hash, tokens, block_size, extra_key);
}

kv_status kv_pool_match_prefix(kv_pool* p, const int32_t* tokens, int num_tokens,
                               uint64_t extra_key, int32_t* out_ids, int* num_hit) {
  if (!p || num_tokens < 0 || (num_tokens > 0 && (!tokens || !out_ids)) || !num_hit)
    return fail(KV_ERR_INVALID_ARG, "kv_pool_match_prefix: bad arguments");
  const int bs = p->block_size;
  int n = 0;
  uint64_t parent = 0;
  for (int j = 0; j < num_tokens / bs; ++j) {
    const int32_t* tk = tokens + (int64_t)j * bs;
    const uint64_t h = block_hash(parent, tk, bs, extra_key);
    auto it = p->by_hash.find(h);
    if (it == p->by_hash.end()) break;
    const int32_t id = it->second;
    const CachedBlock& c = p->cache[id];
    // the stored block must really hold this content (a hash collision is a miss)
    bool same = c.registered && c.hash == h && c.parent == parent && c.extra_key == extra_key;
    for (int i = 0; same && i < bs; ++i) same = c.tokens[i] == tk[i];
    if (!same) break;
    if (p->refs[id] == 0) {          // cached but free: leave the free queue
      p->free_list.remove(id);
      ++p->used;
    }
    ++p->refs[id];
    out_ids[n++] = id;
    parent = h;
  }
  *num_hit = n;
  return KV_OK;
}

kv_status kv_pool_register_prefix(kv_pool* p, const int32_t* block_ids, const int32_t* tokens,
                                  int num_tokens, uint64_t extra_key) {
  if (!p || num_tokens < 0 || (num_tokens > 0 && (!tokens || !block_ids)))
    return fail(KV_ERR_INVALID_ARG, "kv_pool_register_prefix: bad arguments");
  const int bs = p->block_size, nfull = num_tokens / bs;
  for (int j = 0; j < nfull; ++j) {
    const int32_t id = block_ids[j];
    if (id < 0 || id >= p->num_blocks || p->refs[id] == 0)
      return fail(KV_ERR_INVALID_ARG, "kv_pool_register_prefix: block %d is not allocated", id);
  }
  uint64_t parent = 0;
  for (int j = 0; j < nfull; ++j) {
    const int32_t id = block_ids[j];
    const int32_t* tk = tokens + (int64_t)j * bs;
    const uint64_t h = block_hash(parent, tk, bs, extra_key);
    CachedBlock& c = p->cache[id];
    if (c.registered) {
      if (c.hash != h)
        return fail(KV_ERR_INVALID_ARG,
                    "kv_pool_register_prefix: block %d already holds another prefix", id);
    } else if (p->by_hash.find(h) == p->by_hash.end()) {
      // first block with this content: it becomes the cached copy (a later
      // duplicate keeps its contents but is not registered)
      c.registered = true;
      c.hash = h;
      c.parent = parent;
      c.extra_key = extra_key;
      c.tokens.assign(tk, tk + bs);
      p->by_hash.emplace(h, id);
    }
    parent = h;
  }
  return KV_OK;
}

int kv_pool_cached_blocks(const kv_pool* p) { return p ? (int)p->by_hash.size() : -1; }

size_t pagedkv_pool_tensor_bytes(int num_blocks, int block_size, int num_kv_heads, int head_dim,
                                 kv_dtype dtype) {
  if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      !valid_dtype(dtype))
    return 0;
  return (size_t)num_blocks * block_size * num_kv_heads * head_dim * dtype_size(dtype);
}

kv_status pagedkv_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                              const int32_t* block_pairs, int num_pairs, int num_blocks,
                              int block_size, int num_kv_heads, int head_dim, kv_dtype dtype,
                              void* stream) {
  if (num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
      (head_dim != 64 && head_dim != 128) || !valid_dtype(dtype))
    return fail(KV_ERR_INVALID_ARG, "pagedkv_copy_blocks: bad sizes or dtype");
  if (num_pairs == 0) return KV_OK;
  if (!k_cache || !v_cache || !block_pairs || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(KV_ERR_INVALID_ARG, "pagedkv_copy_blocks: pools must be non-NULL and 16-byte aligned");
  const bool scaled = dtype != KV_DTYPE_BF16;
  if (scaled != (k_scale != nullptr) || scaled != (v_scale != nullptr))
    return fail(KV_ERR_INVALID_ARG, "pagedkv_copy_blocks: scales are required for 8-bit pools only");
  if (num_pairs > 65535) return fail(KV_ERR_INVALID_ARG, "pagedkv_copy_blocks: at most 65535 pairs");
  DeviceInfo di;
  kv_status st = device_info(&di);
  if (st != KV_OK) return st;
  const int64_t block_bytes = (int64_t)block_size * num_kv_heads * head_dim * dtype_size(dtype);
  if (block_bytes > (1ll << 30)) return fail(KV_ERR_INVALID_ARG, "pagedkv_copy_blocks: block too large");
  const dim3 grid((unsigned)((block_bytes + kChunk - 1) / kChunk), (unsigned)num_pairs, 2);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, (cudaStream_t)stream>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), k_scale, v_scale, block_pairs,
      num_blocks, (int)block_bytes, num_kv_heads, di.flags);
  return cuda_check(cudaGetLastError(), "copy_blocks_kernel launch");
}

}  // extern "C"
