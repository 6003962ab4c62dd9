/*
 * pagedkv.h -- C ABI of libpagedkv: decode-phase paged attention on one GPU.
 *
 * The cache of every sequence lives in fixed-size blocks of a shared physical
 * pool, and a per-sequence block table maps its logical blocks to physical
 * ones (“让 Agent 跑得快：LLM 推理服务”, §二 and §五 “Block 级管理的优雅性”;
 * “LLM 推理优化技术全景”, PagedAttention).  Each decode step appends the new
 * token's K/V through a slot mapping and then attends with one query token per
 * sequence under GQA, using the online (m, l) softmax recurrence (“LLM 推理优化
 * 技术全景”, 在线 Softmax) so the score row is never materialised.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pool tensors (K and V, separate): [num_blocks, block_size, num_kv_heads,
 *    head_dim], row-major, elements bf16, int8 or FP8 E4M3 (“LLM 推理引擎深度解析”,
 *    §2.1: key_cache / value_cache of that shape).  The base of each pool must
 *    be 16-byte aligned.
 *  - 8-bit pools (int8, E4M3; see kv_dtype) carry fp32 scales [num_blocks,
 *    num_kv_heads] for K and for V; the stored value of element x is
 *    code * scale.
 *  - Token slot: slot = physical_block * block_size + row.
 *  - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  - seq_lens[b] counts every cached token of sequence b INCLUDING the one
 *    appended this step; the step appends first and then attends.
 *  - Supported geometry: head_dim in {64, 128}; block_size in {16, 32};
 *    num_q_heads a multiple of num_kv_heads with a group of at most 8 query
 *    heads per KV head.
 *  - Pointers named "device" are CUDA device pointers of the current device;
 *    "host" pointers are CPU memory.  The caller owns every buffer; the
 *    library allocates no device memory.
 *  - Calls that launch work are asynchronous on `stream` (a cudaStream_t
 *    passed as void*; NULL = the legacy default stream) and return as soon as
 *    the work is queued.
 *
 * Errors
 * ------
 *  - Problems visible on the host (null pointers, unsupported geometry, a
 *    workspace that is too small) return a kv_status != KV_OK at once and
 *    launch nothing; pagedkv_last_error() then describes it.
 *  - Index problems only visible on the device (a slot past the pool, a block
 *    id outside [0, num_blocks), a sequence length <= 0 or past the table or
 *    past max_seq_len) never fault: the kernel skips the element, writes zeros
 *    for that sequence's output rows and sets a bit in a per-device status
 *    word, read with pagedkv_get_status().
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1,    /* bad pointer, size or geometry           */
    KV_ERR_OUT_OF_BLOCKS = 2,  /* the pool has too few free blocks        */
    KV_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed       */
    KV_ERR_DEVICE_INDEX = 4,   /* device status word reported an index    */
    KV_ERR_NOT_IMPLEMENTED = 5
} kv_status;

/* Element type of the K/V pools.  The two 8-bit types store codes under an
 * fp32 scale per (block, KV head), k_scale / v_scale [num_blocks,
 * num_kv_heads]: the value of a code c is c * scale.
 *   KV_DTYPE_INT8       c = clamp(round_half_even(fp32(x) / scale), -127, 127)
 *                       (“The engineering behind LLM inference” notes, §3.2:
 *                       INT8 KV halves the cache)
 *   KV_DTYPE_FP8_E4M3   c = the E4M3 value nearest fp32(x) / scale, ties to
 *                       the even code, magnitudes above 448 saturating to
 *                       448 (“让 Agent 跑得快”, §四 FP8 量化: a 1-byte FP8 KV
 *                       cache; “LLM 推理优化技术全景”, Flash Attention v3:
 *                       E4M3 with block-wise scales).  E4M3: sign, 4
 *                       exponent bits (bias 7), 3 mantissa bits, no
 *                       infinities, 0x7F / 0xFF NaN. */
typedef enum { KV_DTYPE_BF16 = 0, KV_DTYPE_INT8 = 1, KV_DTYPE_FP8_E4M3 = 2 } kv_dtype;

/* Bits of the device status word (pagedkv_get_status). */
#define PAGEDKV_FLAG_BAD_SLOT 0x1u     /* slot >= num_blocks * block_size     */
#define PAGEDKV_FLAG_BAD_BLOCK 0x2u    /* block id outside [0, num_blocks)    */
#define PAGEDKV_FLAG_BAD_SEQ_LEN 0x4u  /* seq_len <= 0 or beyond table/hint   */
#define PAGEDKV_FLAG_WAIT_TIMEOUT 0x8u /* a bounded in-kernel wait gave up    */

/* ------------------------------------------------------------------------ */
/* Block pool (host bookkeeping)                                            */
/* ------------------------------------------------------------------------ */

/* Opaque host object: pool geometry, the free list and a reference count per
 * block.  It owns no device memory: the caller allocates the K/V pool tensors
 * (pagedkv_pool_tensor_bytes each) and the scales.  Not thread-safe: one
 * scheduler thread owns a pool. */
typedef struct kv_pool kv_pool;

/* Create a pool of num_blocks blocks.  Every id is free, in ascending order
 * (“LLM 推理引擎深度解析”, §2.1: the free list starts as every block id).
 * Returns KV_ERR_INVALID_ARG for non-positive sizes or a null `out`. */
kv_status kv_pool_create(int num_blocks, int block_size, int num_kv_heads,
                         int head_dim, kv_dtype dtype, kv_pool **out);

/* Free the host object (NULL is allowed). */
void kv_pool_destroy(kv_pool *pool);

/* Bytes of one block holding K and V, scales excluded:
 * 2 * block_size * num_kv_heads * head_dim * dtype_size
 * (“让 Agent 跑得快：LLM 推理服务”, §二, the block_memory formula). */
size_t kv_pool_block_bytes(const kv_pool *pool);

/* Allocate n blocks, all or none, from the front of the free list, writing
 * their ids to host array out_ids[n]; each starts with one reference
 * (“LLM 推理引擎深度解析”, §2.1: allocation takes ids in free-list order and
 * fails when too few are free).  KV_ERR_OUT_OF_BLOCKS leaves the pool
 * unchanged. */
kv_status kv_pool_alloc(kv_pool *pool, int n, int32_t *out_ids);

/* Add one reference to each of n allocated blocks (host array): a forked
 * sequence (a beam, a parallel sample) now maps them too (“让 Agent 跑得快：
 * LLM 推理服务”, §二 Copy-on-Write: candidates forked from one prefix share
 * its physical blocks, reference count above one).  An id that is not
 * allocated fails the whole call with KV_ERR_INVALID_ARG, changing nothing. */
kv_status kv_pool_fork(kv_pool *pool, const int32_t *ids, int n);

/* Drop one reference from each of n block ids (host array); a block left
 * with none goes to the back of the free list, in the order of `ids` (same
 * §二: a block whose count reaches zero returns to the pool; “LLM 推理引擎
 * 深度解析”, §2.1: finishing a request returns its blocks).  An id that is
 * not allocated, or listed more often than it is referenced, fails the whole
 * call with KV_ERR_INVALID_ARG and changes nothing. */
kv_status kv_pool_free(kv_pool *pool, const int32_t *ids, int n);

/* References held on block `id`: 0 when free, -1 for an id outside the
 * pool or a NULL pool. */
int kv_pool_refcount(const kv_pool *pool, int32_t id);

/* Number of allocated and free blocks (either pointer may be NULL). */
kv_status kv_pool_stats(const kv_pool *pool, int *used, int *free_blocks);

/* Makes every sequence's decode append target writable before the step
 * (host arrays; sequences in order b = 0..batch-1):
 *   - the new token sits at position p = seq_lens[b] - 1 (seq_lens counts
 *     it), in logical block j = p / block_size;
 *   - p % block_size == 0 (the token opens a block): a block is taken from
 *     the free list and written to block_tables[b][j], whose old value is
 *     ignored (“让 Agent 跑得快”, §五: a new block every block_size tokens);
 *   - otherwise, when block_tables[b][j] is shared (reference count above
 *     one), a free block d is taken, the old block loses one reference,
 *     block_tables[b][j] becomes d and the pair (old, d) is appended to
 *     copy_pairs (§二 Copy-on-Write: copy the block and repoint the table
 *     before writing).  A block shared by k sequences of the batch is copied
 *     for the first k - 1 and written in place by the last.
 * The caller copies the pairs with pagedkv_copy_blocks and uploads the
 * tables before the append.
 *   block_tables  host int32 [batch, max_blocks_per_seq], updated in place
 *   seq_lens      host int32 [batch]
 *   copy_pairs    host int32 [batch][2] (output: src, dst)
 *   num_copies    output: pairs written
 * All or nothing: KV_ERR_OUT_OF_BLOCKS when the free list is too short,
 * KV_ERR_INVALID_ARG for a length outside (0, max_blocks_per_seq *
 * block_size] or a write into a block that is not allocated; either leaves
 * the pool and the tables unchanged. */
kv_status kv_pool_prepare_append(kv_pool *pool, int32_t *block_tables,
                                 int max_blocks_per_seq, const int32_t *seq_lens,
                                 int batch, int32_t *copy_pairs, int *num_copies);

/* Prefix cache (“让 Agent 跑得快”, §七 前缀缓存: each full block is hashed from
 * its parent block's hash, its tokens and optional extra keys such as a LoRA
 * id or a cache salt; a new request looks its prompt's blocks up in order,
 * takes a reference on each hit and prefills from the first miss; blocks a
 * finished request frees stay findable in the free queue until reused).
 *
 * Hash of one full block: FNV-1a 64 (offset basis 0xcbf29ce484222325, prime
 * 0x100000001b3; per byte h ^= byte, h *= prime) over parent_hash (8 bytes),
 * extra_key (8 bytes) and the block_size token ids (4 bytes each, two's
 * complement), all little-endian.  The first block's parent hash is 0. */
uint64_t pagedkv_block_hash(uint64_t parent_hash, const int32_t *tokens,
                            int block_size, uint64_t extra_key);

/* Looks the full blocks of a prompt (host int32 tokens[num_tokens]) up in
 * the cache, in order, stopping at the first block whose hash chain has no
 * registered block with exactly these tokens, parent and key (so a hit
 * implies every earlier block hit too).  Every hit block gains a reference
 * (a cached block waiting in the free queue leaves it); their ids go to
 * out_ids[0 .. *num_hit) (capacity num_tokens / block_size).  The caller
 * allocates the rest and prefills from token *num_hit * block_size. */
kv_status kv_pool_match_prefix(kv_pool *pool, const int32_t *tokens,
                               int num_tokens, uint64_t extra_key,
                               int32_t *out_ids, int *num_hit);

/* Registers the full blocks of a sequence whose K/V are now in the pool:
 * block_ids[j] holds tokens [j * block_size, (j + 1) * block_size) of
 * tokens[num_tokens] (a partial last block is not registered).  A block
 * whose content is already registered under another id stays unregistered.
 * Registered blocks leave the cache when allocation takes them again.
 * KV_ERR_INVALID_ARG (nothing registered) for an id that is not allocated
 * or one already registered with a different content. */
kv_status kv_pool_register_prefix(kv_pool *pool, const int32_t *block_ids,
                                  const int32_t *tokens, int num_tokens,
                                  uint64_t extra_key);

/* Number of blocks the prefix cache holds (in use or free); -1 for NULL. */
int kv_pool_cached_blocks(const kv_pool *pool);

/* Bytes of one pool tensor (K or V): num_blocks * block_size * num_kv_heads
 * * head_dim * dtype_size. */
size_t pagedkv_pool_tensor_bytes(int num_blocks, int block_size,
                                 int num_kv_heads, int head_dim, kv_dtype dtype);

/* Copies whole physical blocks of both pools, bit for bit: for every pair i,
 * block block_pairs[i][1] of k_cache and v_cache (and its row of k_scale and
 * v_scale for 8-bit pools) becomes a copy of block block_pairs[i][0] (“让
 * Agent 跑得快”, §二 Copy-on-Write: the block is copied before a shared
 * sequence writes into it).
 *   k_cache, v_cache  device [num_blocks, block_size, num_kv_heads, head_dim],
 *                     16-byte aligned
 *   k_scale, v_scale  device fp32 [num_blocks, num_kv_heads] for 8-bit pools,
 *                     NULL for BF16
 *   block_pairs       device int32 [num_pairs][2] (src, dst)
 * The pairs of one call run at the same time, so every destination must be
 * distinct and no destination may be the source of any pair of the call
 * (pagedkv_check_block_pairs tests this on the host; kv_pool_prepare_append
 * checks its own output with it).  A pair with
 * an id outside [0, num_blocks) is skipped and sets PAGEDKV_FLAG_BAD_BLOCK;
 * src == dst is a no-op.  At most 65535 pairs per call.  Asynchronous on
 * `stream`. */
kv_status pagedkv_copy_blocks(void *k_cache, void *v_cache, float *k_scale,
                              float *v_scale, const int32_t *block_pairs,
                              int num_pairs, int num_blocks, int block_size,
                              int num_kv_heads, int head_dim, kv_dtype dtype,
                              void *stream);

/* Host check of a copy list for pagedkv_copy_blocks: KV_OK when every id is in
 * [0, num_blocks), every destination is distinct and no destination is the
 * source of any pair; else KV_ERR_INVALID_ARG naming the first offending
 * pair.  block_pairs is host int32 [num_pairs][2] (src, dst); pairs with
 * src == dst are no-ops and are ignored.  Reads only its arguments. */
kv_status pagedkv_check_block_pairs(const int32_t *block_pairs, int num_pairs,
                                    int num_blocks);

/* ------------------------------------------------------------------------ */
/* Slot mapping                                                             */
/* ------------------------------------------------------------------------ */

/* Decode-step slots: for every sequence b, the slot of position
 * seq_lens[b] - 1, i.e. block_tables[b][(L-1) / bs] * bs + (L-1) % bs
 * (“让 Agent 跑得快”, §五: a new block is taken every block_size tokens and the
 * block table maps logical to physical blocks).
 *   block_tables  device int32 [batch, max_blocks_per_seq]
 *   seq_lens      device int32 [batch]
 *   slot_mapping  device int64 [batch] (output)
 * A length <= 0 or past the table, or a table entry outside
 * [0, num_blocks), gives slot -1 and sets a status bit. */
kv_status pagedkv_slot_mapping(const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *seq_lens,
                               int batch, int block_size, int num_blocks,
                               int64_t *slot_mapping, void *stream);

/* General slots for a token list: token i of sequence seq_idx[i] (or i when
 * seq_idx is NULL) at 0-based position positions[i] (e.g. a prefill).
 *   seq_idx, positions  device int32 [num_tokens]
 *   slot_mapping        device int64 [num_tokens] (output)
 * Negative positions give slot -1 silently; bad indices as above. */
kv_status pagedkv_token_slot_mapping(const int32_t *block_tables,
                                     int max_blocks_per_seq,
                                     const int32_t *seq_idx,
                                     const int32_t *positions, int num_tokens,
                                     int block_size, int num_blocks,
                                     int64_t *slot_mapping, void *stream);

/* ------------------------------------------------------------------------ */
/* Append                                                                   */
/* ------------------------------------------------------------------------ */

/* Write each token's new K/V into its slot (“让 Agent 跑得快”, §一 KV Cache:
 * decode appends the new token's K/V; §五 “共享前缀”: only the current token
 * writes).
 *   k, v          device bf16 [num_tokens, num_kv_heads, head_dim]
 *   k_cache, v_cache  device pool tensors (bf16, int8 or E4M3, see above)
 *   k_scale, v_scale  device fp32 [num_blocks, num_kv_heads] for 8-bit pools;
 *                     must be NULL for bf16 pools
 *   slot_mapping  device int64 [num_tokens]; slot < 0 skips the token
 * bf16 pools receive the bits unchanged.  int8 pools receive
 * clamp(round_half_even(fp32(x) / scale), -127, 127) computed with an IEEE
 * fp32 divide (scale 0 is read as 1, NaN gives 0), with the scale of the
 * slot's block and head.  E4M3 pools receive the E4M3 code of the same fp32
 * quotient (nearest, ties to even, saturating at 448; NaN gives 0x7F).  A slot >= num_blocks * block_size is skipped and
 * sets PAGEDKV_FLAG_BAD_SLOT. */
kv_status reshape_and_cache(const void *k, const void *v, void *k_cache,
                            void *v_cache, const float *k_scale,
                            const float *v_scale, const int64_t *slot_mapping,
                            int num_tokens, int num_blocks, int block_size,
                            int num_kv_heads, int head_dim, kv_dtype dtype,
                            void *stream);

/* ------------------------------------------------------------------------ */
/* Attention                                                                */
/* ------------------------------------------------------------------------ */

/* Workspace bytes paged_attention_decode / pagedkv_decode_step may need for
 * the split-K partials of this shape (an upper bound over every partition
 * size the library picks; 0 when every sequence fits one partition). */
size_t pagedkv_workspace_bytes(int batch, int num_q_heads, int head_dim,
                               int max_seq_len, int block_size);

/* out[b, h, :] = softmax(scale * q[b, h, :] . K_t) . V_t over the
 * t < seq_lens[b] tokens of sequence b (“LLM 推理优化技术全景”: 在线 Softmax,
 * computed with the recurrence m' = max(m, max s), l' = l e^(m-m') + sum
 * e^(s-m'), and the rescale deferred to the end as in “Flash Attention v2 的
 * 改进”).  Each (sequence, KV head) is cut into token partitions; one CTA
 * serves a partition for all query heads of the KV head, and a sequence with
 * several partitions has their partials (m, l, unnormalised acc) merged by
 * log-sum-exp in a second kernel launched behind the first.
 *   out           device bf16 [batch, num_q_heads, head_dim] (output)
 *   q             device bf16 [batch, num_q_heads, head_dim]
 *   k_cache, v_cache, k_scale, v_scale   as for reshape_and_cache
 *   block_tables  device int32 [batch, max_blocks_per_seq]; entries past
 *                 ceil(seq_lens[b] / block_size) are never read
 *   seq_lens      device int32 [batch]
 *   max_seq_len   host bound on every seq_lens[b] (sizes the partitions)
 *   scale         softmax scale (1/sqrt(head_dim) for the usual attention)
 *   workspace     device memory of at least pagedkv_workspace_bytes(...)
 *                 bytes, 16-byte aligned; may be NULL when that size is 0.
 *                 Calls that overlap on the GPU need separate workspaces.
 * Rows past seq_lens[b] inside the last block and blocks not in the table
 * are never used, whatever they hold. */
kv_status paged_attention_decode(void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const float *k_scale,
                                 const float *v_scale,
                                 const int32_t *block_tables,
                                 int max_blocks_per_seq,
                                 const int32_t *seq_lens, int batch,
                                 int num_q_heads, int num_kv_heads,
                                 int head_dim, int num_blocks, int block_size,
                                 int max_seq_len, float scale, kv_dtype dtype,
                                 void *workspace, size_t workspace_bytes,
                                 void *stream);

/* One decode step in two launches: append each sequence's new token (k[b],
 * v[b] at position seq_lens[b] - 1, exactly as pagedkv_slot_mapping +
 * reshape_and_cache would) and then attend as paged_attention_decode.  The
 * append runs inside the attention kernel: the CTA that streams a (b, h)'s
 * last block writes the new row first and orders that write before its own
 * read of the block (“让 Agent 跑得快”, §五 共享前缀: only the current token
 * writes, so no other reader of the step can see the row).
 *   k, v  device bf16 [batch, num_kv_heads, head_dim]
 * Other arguments as paged_attention_decode (the pools are written).  The new
 * token's block must not be read by another sequence in the same step (shared
 * prefix blocks are full, so appends land in private blocks). */
kv_status pagedkv_decode_step(void *out, const void *q, const void *k,
                              const void *v, void *k_cache, void *v_cache,
                              const float *k_scale, const float *v_scale,
                              const int32_t *block_tables,
                              int max_blocks_per_seq, const int32_t *seq_lens,
                              int batch, int num_q_heads, int num_kv_heads,
                              int head_dim, int num_blocks, int block_size,
                              int max_seq_len, float scale, kv_dtype dtype,
                              void *workspace, size_t workspace_bytes,
                              void *stream);

/* pagedkv_decode_step for a batch whose sequences all begin with the same
 * num_prefix_blocks physical blocks (a shared system prompt: “让 Agent
 * 跑得快”, §五 共享前缀 -- several block tables map to the same read-only
 * blocks).  The prefix part of attention is computed once per KV head for
 * every query row of the batch (a dense product on tensor cores) instead of
 * once per sequence; tokens past the prefix go through the decode kernel and
 * the two are merged by log-sum-exp.  Results equal pagedkv_decode_step up
 * to rounding.
 *   prefix_blocks      device int32 [num_prefix_blocks]: the shared physical
 *                      blocks, which must also be entries 0..P-1 of every
 *                      row of block_tables (a mismatch zeroes that sequence's
 *                      rows and sets PAGEDKV_FLAG_BAD_BLOCK)
 *   num_prefix_blocks  P >= 1; every seq_lens[b] must exceed P * block_size
 *                      (shorter sequences are flagged and zeroed)
 *   k, v               as pagedkv_decode_step, or both NULL to attend
 *                      without appending
 *   workspace          at least pagedkv_prefix_workspace_bytes(...) bytes
 * bf16, int8 and E4M3 pools (for 8-bit pools the prefix product widens the
 * codes exactly to fp16 and runs in fp16; k_scale and v_scale as for
 * paged_attention_decode). */
kv_status pagedkv_decode_step_prefix(void *out, const void *q, const void *k,
                                     const void *v, void *k_cache,
                                     void *v_cache, const float *k_scale,
                                     const float *v_scale,
                                     const int32_t *block_tables,
                                     int max_blocks_per_seq,
                                     const int32_t *seq_lens, int batch,
                                     int num_q_heads, int num_kv_heads,
                                     int head_dim, int num_blocks,
                                     int block_size, int max_seq_len,
                                     float scale, kv_dtype dtype,
                                     const int32_t *prefix_blocks,
                                     int num_prefix_blocks, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* Workspace bytes pagedkv_decode_step_prefix may need for this shape. */
size_t pagedkv_prefix_workspace_bytes(int batch, int num_q_heads, int head_dim,
                                      int max_seq_len, int block_size,
                                      int num_prefix_blocks);

/* Size of the fixed device scratch paged_attention_decode_noalloc uses. */
#define PAGEDKV_NOALLOC_SCRATCH_BYTES (32u << 20)

/* paged_attention_decode without a workspace argument, for callers that
 * cannot allocate device memory: a plain C host program that links only this
 * library and the CUDA runtime and has no device allocator of its own, or a
 * serving engine that reserves all of HBM for its KV pool at start-up and
 * forbids allocation afterwards.  The pages describe no such entry point; it
 * is this library's own addition.
 *
 * Arguments, layouts, results and errors are those of paged_attention_decode
 * (minus workspace / workspace_bytes).  The split-K partials go to a scratch
 * array of PAGEDKV_NOALLOC_SCRATCH_BYTES (32 MiB) compiled into the library:
 * every GPU that loads the library holds it until the process exits, and the
 * call itself allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).  A shape whose partials need more than that returns
 * KV_ERR_INVALID_ARG with a message naming both sizes.
 *
 * The first call on each device looks up that device's scratch address
 * (cudaGetSymbolAddress) with the device current; make that first call before
 * any stream capture.  All calls on a device share the one scratch array,
 * which keeps the last call's contents; nothing in it needs clearing, since
 * each call writes every partial it later reads.  Calls whose work overlaps
 * on the GPU (different streams, or several host threads) race on the
 * scratch: serialise them, or use paged_attention_decode with one workspace
 * per stream. */
kv_status paged_attention_decode_noalloc(void *out, const void *q,
                                         const void *k_cache,
                                         const void *v_cache,
                                         const float *k_scale,
                                         const float *v_scale,
                                         const int32_t *block_tables,
                                         int max_blocks_per_seq,
                                         const int32_t *seq_lens, int batch,
                                         int num_q_heads, int num_kv_heads,
                                         int head_dim, int num_blocks,
                                         int block_size, int max_seq_len,
                                         float scale, kv_dtype dtype,
                                         void *stream);

/* PAGEDKV_NOALLOC_SCRATCH_BYTES as compiled into this library: the largest
 * split-K scratch paged_attention_decode_noalloc serves (a binding can read
 * the limit here instead of repeating the macro). */
size_t pagedkv_noalloc_scratch_bytes(void);

/* ------------------------------------------------------------------------ */
/* Multi-token queries                                                      */
/* ------------------------------------------------------------------------ */

/* Workspace bytes paged_attention_multi may need (an upper bound over every
 * partition size the library picks; 0 when every query fits one). */
size_t pagedkv_multi_workspace_bytes(int num_tokens, int num_q_heads,
                                     int head_dim, int max_seq_len,
                                     int block_size);

/* Attention of several query tokens per sequence over the paged pool, causal
 * within each sequence: speculative verification (“让 Agent 跑得快”, §六 投机
 * 解码: the target model scores the gamma draft tokens in one parallel pass)
 * and chunked prefill batched with decodes (“LLM 推理优化技术全景”, SARATHI:
 * 512-token prefill chunks plus decodes in one batch).  Sequence b has n_b =
 * query_start[b + 1] - query_start[b] query tokens, q rows query_start[b] ..
 * query_start[b + 1] - 1, which are its LAST n_b tokens and are already in
 * the pool (append them first with pagedkv_token_slot_mapping +
 * reshape_and_cache).  Query token i of sequence b sits at position
 * seq_lens[b] - n_b + i and attends positions 0 .. seq_lens[b] - n_b + i:
 *   out[j, h, :] = softmax_t(scale * q[j, h, :] . K_t) . V_t.
 *   out           device bf16 [num_tokens, num_q_heads, head_dim]
 *   q             device bf16 [num_tokens, num_q_heads, head_dim]
 *   k_cache, v_cache, k_scale, v_scale   as for paged_attention_decode
 *                 (bf16, int8 and E4M3 pools; with 8-bit pools the long-query
 *                 kernel widens the codes exactly to fp16 and runs its
 *                 products in fp16)
 *   block_tables, max_blocks_per_seq, seq_lens, batch  as for
 *                 paged_attention_decode (seq_lens counts the query tokens)
 *   query_start   device int32 [batch + 1], non-decreasing from 0 to
 *                 num_tokens (n_b = 0 is allowed: no queries)
 *   max_query_len host bound on every n_b (sizes the launch)
 *   max_seq_len   host bound on every seq_lens[b]
 *   workspace     at least pagedkv_multi_workspace_bytes(...) bytes,
 *                 16-byte aligned (may be NULL when that size is 0)
 * A sequence with a bad length (n_b > seq_lens[b] or > max_query_len, beyond
 * the table or the hint) or a bad table entry has its rows zeroed and sets
 * PAGEDKV_FLAG_BAD_SEQ_LEN or PAGEDKV_FLAG_BAD_BLOCK; offsets outside
 * [0, num_tokens] leave that sequence's rows unwritten and set
 * PAGEDKV_FLAG_BAD_SEQ_LEN (rows past max_query_len are not written).
 * Asynchronous on `stream`: the attention launches, plus a log-sum-exp
 * merge launch when the keys are split into partitions.  Sequences with at
 * most 8 / G query tokens go to the decode kernel (8 (token, head) columns
 * per CTA); with at most 4 * (8 / G), in calls without longer queries on
 * bf16 pools, to a kernel with 16 columns per MMA tile (up to 32 per CTA,
 * the decode kernel's launch left out when every sequence has max_query_len
 * tokens), else to the decode kernel's column groups; longer queries go to
 * a tensor-core kernel with TMEM accumulators (128 query rows per CTA). */
kv_status paged_attention_multi(void *out, const void *q, const void *k_cache,
                                const void *v_cache, const float *k_scale,
                                const float *v_scale, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *seq_lens,
                                const int32_t *query_start, int batch,
                                int num_tokens, int max_query_len,
                                int num_q_heads, int num_kv_heads,
                                int head_dim, int num_blocks, int block_size,
                                int max_seq_len, float scale, kv_dtype dtype,
                                void *workspace, size_t workspace_bytes,
                                void *stream);

/* One multi-token step: the step's new K/V rows appended to the pool, then
 * paged_attention_multi over its query tokens, on `stream` in that order
 * (the multi-token counterpart of pagedkv_decode_step; the append as in
 * reshape_and_cache, “让 Agent 跑得快”, §一 KV Cache, the attention as in the
 * passages cited for paged_attention_multi).  Results are identical to
 * pagedkv_token_slot_mapping + reshape_and_cache + paged_attention_multi.
 *   new_k, new_v  device bf16 [num_tokens, num_kv_heads, head_dim]: row
 *                 query_start[b] + i is the K/V of sequence b's token at
 *                 position seq_lens[b] - n_b + i (quantised on 8-bit pools
 *                 under k_scale / v_scale of its block, as reshape_and_cache)
 *   every other argument as for paged_attention_multi (seq_lens already
 *   counts the new tokens).
 * The append is one launch: each 16-byte piece of a new row finds its
 * sequence (the last b with query_start[b] <= row) and its slot from the
 * block table (block_tables[b][pos / block_size] * block_size +
 * pos % block_size) and is written there.  A sequence whose offsets do not
 * fit (rows outside [0, num_tokens], n_b > seq_lens[b] or > max_query_len)
 * appends nothing and sets PAGEDKV_FLAG_BAD_SEQ_LEN; a position past the
 * table sets PAGEDKV_FLAG_BAD_SEQ_LEN and an entry outside the pool
 * PAGEDKV_FLAG_BAD_BLOCK, and that row is skipped.  The attention then
 * flags and zeroes as paged_attention_multi (offsets that decrease are
 * flagged there).  Arguments are checked before the first launch;
 * KV_ERR_INVALID_ARG on a bad one (new_k and new_v must be non-NULL and
 * 16-byte aligned). */
kv_status pagedkv_multi_step(void *out, const void *q, const void *new_k,
                             const void *new_v, void *k_cache, void *v_cache,
                             const float *k_scale, const float *v_scale,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *seq_lens, const int32_t *query_start,
                             int batch, int num_tokens, int max_query_len,
                             int num_q_heads, int num_kv_heads, int head_dim,
                             int num_blocks, int block_size, int max_seq_len,
                             float scale, kv_dtype dtype, void *workspace,
                             size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* Status                                                                   */
/* ------------------------------------------------------------------------ */

/* Wait for `stream`, then read and clear the current device's status word
 * into *device_flags (PAGEDKV_FLAG_* bits).  Returns KV_ERR_DEVICE_INDEX
 * when any bit was set, KV_ERR_CUDA when a CUDA call failed, else KV_OK. */
kv_status pagedkv_get_status(void *stream, unsigned int *device_flags);

/* Message for the last error of the calling thread ("" if none). */
const char *pagedkv_last_error(void);

/* Token partition size paged_attention_decode would use for this shape on
 * the current device (0 on error).  The partitions split each sequence's
 * tokens among CTAs, the parallelism along the sequence of “LLM 推理优化技术
 * 全景”, Flash Attention v2 的改进.  The largest power of two in [256, 2048]
 * that still gives at least 8 CTAs per SM and is at most half of max_seq_len
 * (256 when nothing larger qualifies).  Sequences longer than one
 * partition go through the merge kernel.  The environment variable
 * PAGEDKV_PARTITION_TOKENS (a multiple of 256) overrides it. */
int pagedkv_partition_tokens(int batch, int num_kv_heads, int max_seq_len,
                             int block_size);

/* Token partition size paged_attention_multi would use for this call on the
 * current device (0 on error); arguments as for paged_attention_multi.  The
 * same split along the sequence (“LLM 推理优化技术全景”, Flash Attention v2
 * 的改进) as for paged_attention_decode.  A
 * power of two from 256 up to 8192 when every sequence's queries go to the
 * decode kernel's column groups (max_query_len <= 4 * (8 / G)), up to 2048
 * when the tensor-core kernel is in the call; the largest that still gives
 * at least 8 CTAs per SM.  Sequences longer than one partition go through
 * the merge kernel, which is launched only when max_seq_len exceeds it.
 * PAGEDKV_PARTITION_TOKENS (a multiple of 256, within the same limits)
 * overrides it. */
int pagedkv_multi_partition_tokens(int batch, int num_tokens, int max_query_len,
                                   int num_q_heads, int num_kv_heads,
                                   int max_seq_len);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
