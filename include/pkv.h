/*
 * pkv.h -- C ABI of libpkv: attention for one decode step (and for a causal
 * query chunk) over a paged BF16 KV cache, on one GB300 (sm_103a).
 *
 * Source of the operations. All section/figure references are to the web
 * textbook page "Chapter 8: Inference Optimization" (clxhxhhr.top/posts/4341):
 *   - §8.1.1 "Execution resources and request lifecycle": in decode, each step
 *     feeds the newly generated token, reads the request's context KV and
 *     stores the new token's K and V.
 *   - §8.1.2 "Storage of weights, KV and runtime buffers": K and V per token
 *     per layer are 8 KV heads x 128 dims x BF16; blocks hold 16 tokens.
 *   - §8.3.1 "Reservation, fragmentation and paged allocation", Fig. 8-10: KV
 *     lives in fixed-size physical blocks; a per-request block table maps
 *     logical block j to a physical block, and attention locates each token's
 *     KV through that table, so blocks may be scattered.
 *   - §8.3.1 worked example and Fig. 8-13: blocks of a common prefix are
 *     stored once and referenced from several block tables.
 *   - §8.2.3 "Interference of long prefill with generation and chunking",
 *     Fig. 8-8/8-9: in a chunk of c new tokens after h cached ones, new token j
 *     (1-based) attends to h + j tokens (causal inside the chunk).
 *   - §8.5.2: verifying several draft positions reads the same KV as one
 *     decode step; it is the same chunked attention with a short chunk.
 *
 * Conventions shared by every entry point:
 *   - All tensors are caller-owned device memory; the library never allocates,
 *     frees or synchronises (pkv_decode_graph_create/_destroy aside: they
 *     build and free CUDA graphs), and every call only enqueues work on `stream`
 *     (a cudaStream_t passed as void*; NULL is the legacy default stream).
 *   - BF16 values are passed as raw 16-bit patterns (void*).
 *   - Cache layout, per tensor (K and V are separate buffers of identical
 *     shape):  [num_blocks][num_kv_heads][block_size][head_dim] BF16, so one
 *     (physical block, kv head) tile of 16 x 128 BF16 = 4 KiB is contiguous.
 *     Slot s of the pool is token (s % block_size) of physical block
 *     (s / block_size).
 *   - Supported shapes: block_size 16, head_dim 128, num_kv_heads >= 1,
 *     num_q_heads = 4 * num_kv_heads (GQA groups of 4 query heads; query head
 *     h reads KV head h / 4).  Other shapes return PKV_ERR_UNSUPPORTED.
 *   - Argument errors detectable on the host return a non-zero status and
 *     enqueue nothing.  Errors that depend on device data (a block id outside
 *     the pool, a slot outside the pool, a context longer than the block
 *     table) never fault: the kernels clamp the access into the pool and set
 *     a device error word, read with pkv_get_device_error().
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_NULL = 1,        /* a required pointer is NULL                       */
  PKV_ERR_SHAPE = 2,       /* a size is negative or inconsistent               */
  PKV_ERR_UNSUPPORTED = 3, /* a shape the library has no kernel for           */
  PKV_ERR_WORKSPACE = 4,   /* split-KV workspace missing or too small          */
  PKV_ERR_CUDA = 5,        /* a CUDA runtime call failed (launch, attribute)   */
  PKV_ERR_EXHAUSTED = 6    /* a block pool has too few free blocks             */
} pkv_status;

/* Bits of the device error word (pkv_get_device_error). */
#define PKV_DEVERR_BLOCK_ID 1u   /* block table entry outside [0, num_blocks) */
#define PKV_DEVERR_SLOT 2u       /* slot_mapping entry >= num_blocks*16       */
#define PKV_DEVERR_CONTEXT 4u    /* context_lens[r] > max_blocks_per_seq*16   */
#define PKV_DEVERR_TIMEOUT 8u    /* a pipeline wait gave up (never expected)  */

/* Geometry of one layer's paged cache (both K and V use it). */
typedef struct pkv_cache_desc {
  int32_t num_blocks;   /* physical blocks in the pool                     */
  int32_t block_size;   /* tokens per block; must be 16                    */
  int32_t num_kv_heads; /* KV heads; query heads = 4 * num_kv_heads        */
  int32_t head_dim;     /* must be 128                                     */
} pkv_cache_desc;

/*
 * pkv_kv_append -- store each new token's K and V in its slot (§8.1.1: the
 * step stores the K and V of the token it processes; §8.3.1: the slot is
 * physical block * block_size + offset, found through the block table).
 *
 *   k_cache, v_cache : device, cache layout above, modified in place.
 *   cache            : host pointer to the pool geometry.
 *   slot_mapping     : device int64 [num_tokens]; slot of token t, or < 0 to
 *                      skip token t (padding).  Slots must be distinct; a
 *                      slot >= num_blocks*block_size is skipped and sets
 *                      PKV_DEVERR_SLOT.
 *   k_new, v_new     : device BF16 [num_tokens][num_kv_heads][head_dim].
 *   num_tokens       : >= 0; 0 enqueues nothing and returns PKV_OK.
 * The copy is bit-exact.
 */
pkv_status pkv_kv_append(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                         const int64_t* slot_mapping, const void* k_new, const void* v_new,
                         int32_t num_tokens, void* stream);

/*
 * pkv_choose_kv_blocks_per_split -- the split-KV heuristic used when
 * pkv_paged_attention is given kv_blocks_per_split = 0.  Long contexts are cut
 * into contiguous ranges of this many logical blocks, each reduced by its own
 * CTA, so that num_seqs x num_kv_heads x splits fills the GPU's SMs.  Returns
 * >= max_blocks_per_seq when no split is needed.  Pure host arithmetic.
 *   sm_count : SMs of the target GPU (<= 0: ask the current CUDA device).
 */
int32_t pkv_choose_kv_blocks_per_split(int32_t num_seqs, int32_t num_kv_heads, int32_t q_len,
                                       int32_t max_blocks_per_seq, int32_t sm_count);

/*
 * pkv_workspace_size -- bytes of device workspace pkv_paged_attention needs
 * for these sizes and this (already resolved, > 0) kv_blocks_per_split.  With
 * num_splits = ceil(max_blocks_per_seq / kv_blocks_per_split): 0 when
 * num_splits <= 8 (one split, or splits merged on chip inside a thread-block
 * cluster); otherwise partial_o FP32 [num_seqs][q_len][num_q_heads]
 * [num_splits][head_dim], then partial_lse FP32 [num_seqs][q_len][num_q_heads]
 * [num_splits], each part 256-byte aligned.
 */
size_t pkv_workspace_size(int32_t num_seqs, int32_t q_len, int32_t num_q_heads, int32_t head_dim,
                          int32_t max_blocks_per_seq, int32_t kv_blocks_per_split);

/*
 * pkv_paged_attention -- softmax(q K^T * scale) V for every request, query
 * position and query head, reading K/V through the block tables.
 *
 *   out          : device BF16 [num_seqs][q_len][num_q_heads][head_dim].
 *   q            : device BF16, same shape as out.
 *   k_cache, v_cache, cache : as for pkv_kv_append (read only).
 *   block_tables : device int32 [num_seqs][max_blocks_per_seq]; entry j of row
 *                  r is the physical block holding logical block j of request
 *                  r (tokens 16j .. 16j+15).  Rows may share entries (common
 *                  prefixes).  Entries past ceil(ctx/16) are never read.
 *   context_lens : device int32 [num_seqs]; ctx_r = number of tokens of
 *                  request r in the cache, INCLUDING the q_len tokens of this
 *                  step (append first, then attend).  Query i (0-based) of
 *                  request r sits at position ctx_r - q_len + i and attends to
 *                  the keys at positions 0 .. ctx_r - q_len + i.  ctx_r = 0 is a
 *                  padding row: its outputs are zero.  A query with no visible
 *                  key (ctx_r < q_len) also outputs zeros.
 *   q_len        : query tokens per request (1 = plain decode; >= 2 = causal
 *                  chunk).  q_len >= 16 runs on the tensor-core kernel.
 *   num_q_heads  : 4 * cache->num_kv_heads.
 *   scale        : logit scale (1/sqrt(head_dim) for standard attention).
 *   kv_blocks_per_split : 0 = choose with pkv_choose_kv_blocks_per_split;
 *                  >= max_blocks_per_seq = one pass per (request, kv head);
 *                  otherwise each request's blocks are reduced in ranges of
 *                  this many blocks and the ranges merged: on chip (one
 *                  thread-block cluster per row) for up to 8 ranges, else
 *                  through the workspace and the combine kernel.
 *   workspace, workspace_bytes : device scratch of at least
 *                  pkv_workspace_size(...) bytes for the resolved split (may be
 *                  NULL/0 when that size is 0).  Its contents are
 *                  overwritten; calls that share it must be stream-ordered.
 * The result does not depend on where blocks sit in the pool; with a fixed
 * split it is bitwise reproducible.  The split changes rounding only.
 */
pkv_status pkv_paged_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const pkv_cache_desc* cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               int32_t num_seqs, int32_t q_len, int32_t num_q_heads, float scale,
                               int32_t kv_blocks_per_split, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Cascade decode: requests whose block tables begin with the same physical
 * blocks (a common prefix stored once, §8.3.1 worked example and Fig. 8-13;
 * §8.3.2's shared-prefix batch) read that prefix together.  For each group of
 * up to 16 sharers, one tensor-core pass contracts the 16 x 4 query rows of
 * a KV head against the prefix tiles once; each request's private suffix goes
 * through the decode kernel; the partial results are merged by the
 * log-sum-exp identity.  The result equals pkv_paged_attention's (q_len 1).
 *
 *   group_seqs        : device int32 [num_groups][16]: member request indices,
 *                       -1 for unused places (member 0 must be valid).
 *   group_blocks      : device int32 [num_groups]: P_g, the number of leading
 *                       logical blocks every member of group g maps to the
 *                       same physical blocks (read through member 0's row).
 *   seq_prefix_blocks : device int32 [num_seqs]: P_g of the group holding
 *                       request r, 0 for a request in no group.  A request
 *                       belongs to at most one group.
 *   num_groups        : >= 0 (0: every request is a plain decode).
 *   max_prefix_blocks : host upper bound of every P_g (sizes the prefix split).
 *   max_suffix_blocks : host upper bound, over all requests, of the blocks
 *                       left after the request's prefix (ceil(ctx/16) - P_g,
 *                       or ceil(ctx/16) outside every group); 0 means
 *                       max_blocks_per_seq.  Sizes the suffix split grid.
 *   prefix_blocks_per_split, suffix_blocks_per_split : 0 = pkv_cascade_plan.
 *   workspace         : >= pkv_cascade_workspace_size(...) bytes, 256-aligned.
 * Every other argument is as for pkv_paged_attention with q_len = 1.  A member
 * whose context is shorter than P_g*16 tokens still gets the exact result (its
 * prefix rows are masked at its own context), it only saves nothing.
 */
void pkv_cascade_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t num_groups, int32_t max_prefix_blocks,
                      int32_t max_suffix_blocks, int32_t sm_count, int32_t* prefix_blocks_per_split,
                      int32_t* suffix_blocks_per_split);

size_t pkv_cascade_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t max_prefix_blocks,
                                  int32_t max_suffix_blocks, int32_t prefix_blocks_per_split,
                                  int32_t suffix_blocks_per_split);

pkv_status pkv_paged_attention_cascade(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const pkv_cache_desc* cache, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t num_seqs, int32_t num_q_heads, float scale,
                                       const int32_t* group_seqs, const int32_t* group_blocks,
                                       const int32_t* seq_prefix_blocks, int32_t num_groups,
                                       int32_t max_prefix_blocks, int32_t max_suffix_blocks,
                                       int32_t prefix_blocks_per_split, int32_t suffix_blocks_per_split,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * pkv_paged_attention_append -- pkv_kv_append followed by pkv_paged_attention,
 * in one call: the step's new tokens are stored (slot_mapping, k_new, v_new,
 * num_tokens as for pkv_kv_append), then attention runs over the pools that
 * hold them (every other argument as for pkv_paged_attention).  Ch8 §8.1.1:
 * a decode step stores the new token's K and V and reads the context KV,
 * the new token included.
 *
 * When q_len is 1, num_tokens == num_seqs and the decode runs on the
 * CTA-per-row kernel (pkv_paged_attention's choice), both happen in one
 * launch: the kernel block that reads the block holding request r's position
 * context_lens[r] - 1 stores token r's K/V row there and uses it in place of
 * the row it read.  That requires token r to be request r's new token and
 * slot_mapping[r] to be the slot the block table gives that position (or
 * negative: not stored); any other slot is stored as pkv_kv_append would but
 * sets PKV_DEVERR_SLOT, and the attention result is then undefined.  A token
 * is stored only when its row has a position context_lens[r] - 1 inside the
 * block table: a slot >= 0 for a row with context_lens[r] <= 0 is a caller
 * error (the token is not stored; PKV_DEVERR_SLOT), and a context longer than
 * the table (PKV_DEVERR_CONTEXT) leaves its token unstored too.  Other
 * shapes issue the append, then the attention.  For inputs that set no device
 * error, results equal the two calls' bit for bit.  Host-detectable errors of
 * either call return before anything is enqueued.
 */
pkv_status pkv_paged_attention_append(void* out, const void* q, void* k_cache, void* v_cache,
                                      const pkv_cache_desc* cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                      int32_t q_len, int32_t num_q_heads, float scale, int32_t kv_blocks_per_split,
                                      void* workspace, size_t workspace_bytes, const int64_t* slot_mapping,
                                      const void* k_new, const void* v_new, int32_t num_tokens, void* stream);

/*
 * pkv_paged_attention_cascade_append -- pkv_kv_append followed by
 * pkv_paged_attention_cascade, in one call (arguments as for the two).  When
 * num_tokens == num_seqs (token r is request r's new token) the suffix pass
 * stores the tokens and uses them as pkv_paged_attention_append's single
 * launch does; other counts issue the append, then the cascade.  A new token
 * must lie past its request's shared prefix (never append into a block
 * another table references); one inside it is not stored and sets
 * PKV_DEVERR_SLOT, as does a slot >= 0 for a row with context_lens[r] <= 0.
 * Results equal the two calls' bit for bit otherwise.
 */
pkv_status pkv_paged_attention_cascade_append(
    void* out, const void* q, void* k_cache, void* v_cache, const pkv_cache_desc* cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, float scale,
    const int32_t* group_seqs, const int32_t* group_blocks, const int32_t* seq_prefix_blocks, int32_t num_groups,
    int32_t max_prefix_blocks, int32_t max_suffix_blocks, int32_t prefix_blocks_per_split,
    int32_t suffix_blocks_per_split, void* workspace, size_t workspace_bytes, const int64_t* slot_mapping,
    const void* k_new, const void* v_new, int32_t num_tokens, void* stream);

/* Bytes of the scratch array compiled into libpkv for
 * pkv_paged_attention_static_workspace (held on every GPU that loads the
 * library, until the process exits). */
#define PKV_STATIC_WORKSPACE_BYTES (16u << 20)

/*
 * pkv_paged_attention_static_workspace -- pkv_paged_attention for callers
 * that cannot allocate device memory.  The pages have no counterpart to this
 * entry point; it exists for callers that may not enter a device allocator:
 * code running inside a memory manager or an allocation hook, under a
 * framework that forbids allocation on its hot path, or plain C callers that
 * hold no CUDA allocator.
 *
 * Arguments and results are those of pkv_paged_attention, minus the
 * workspace: split-KV partials go to one scratch array of
 * PKV_STATIC_WORKSPACE_BYTES inside the library, on the current device.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     routine.  The caller still provides inputs and outputs.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture.  Host threads may make first calls concurrently (the
 *     lookup is serialised).  cudaDeviceReset on a device invalidates the
 *     cached address: do not call this entry point on that device again in
 *     the same process.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents.  Nothing in it must start at zero.  Calls that can overlap on
 *     the GPU (unordered streams) race on it: order them.
 *   - Returns PKV_ERR_WORKSPACE, enqueuing nothing, when the resolved split
 *     needs more than PKV_STATIC_WORKSPACE_BYTES (pkv_workspace_size tells
 *     the need); a larger kv_blocks_per_split needs less.
 */
pkv_status pkv_paged_attention_static_workspace(void* out, const void* q, const void* k_cache,
                                                const void* v_cache, const pkv_cache_desc* cache,
                                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                const int32_t* context_lens, int32_t num_seqs,
                                                int32_t q_len, int32_t num_q_heads, float scale,
                                                int32_t kv_blocks_per_split, void* stream);

/*
 * pkv_attn_combine -- merge split-KV partial results (the log-sum-exp
 * identity of blockwise softmax: a softmax over the union of key ranges is
 * the lse-weighted mix of the per-range softmaxes).
 *
 *   out         : device BF16 [num_rows][head_dim], num_rows = num_seqs*q_len*
 *                 num_q_heads.
 *   partial_o   : device FP32 [num_rows][num_splits][head_dim]; split s holds
 *                 its own normalised softmax(q K_s^T) V_s.
 *   partial_lse : device FP32 [num_rows][num_splits]; natural-log
 *                 log-sum-exp of split s's scaled logits, -inf for an empty
 *                 split (its partial_o is then ignored).
 *   out_lse     : optional device FP32 [num_rows] (NULL to skip): the merged
 *                 log-sum-exp.
 * out = sum_s exp(lse_s - lse) * O_s with lse = log sum_s exp(lse_s); a row
 * whose splits are all empty gets zeros (and out_lse = -inf).
 */
pkv_status pkv_attn_combine(void* out, float* out_lse, const float* partial_o,
                            const float* partial_lse, int32_t num_rows, int32_t head_dim,
                            int32_t num_splits, void* stream);

/*
 * pkv_get_device_error -- copy the device error word (PKV_DEVERR_* bits,
 * accumulated over all calls on the current device since the last reset) to
 * *host_word; when reset != 0, clear it.  Synchronises the device.
 */
pkv_status pkv_get_device_error(uint32_t* host_word, int32_t reset);

/*
 * pkv_selftest_bounded_wait -- exercise the fail-fast path of the kernels'
 * pipeline waits.  Every wait in libpkv gives up after a wall-time limit and
 * sets PKV_DEVERR_TIMEOUT rather than hang (the PhyAI deployment page
 * "Parallel serving", failure handling: fail fast, a step that cannot finish
 * within its timeout is reported, not waited on).  Healthy calls never reach
 * the limit, so this entry point launches a
 * one-CTA kernel whose consumer waits, with the same bounded wait, on a ring
 * stage 0 that its producer arms and a stage 1 that it arms only when
 * arm_all != 0.
 *   wait_limit_us : 1 .. 1,000,000 (else PKV_ERR_SHAPE): the limit of each
 *                   wait, in microseconds of GPU wall time.
 *   arm_all       : 0 = stage 1 is never armed: its wait runs out and the
 *                   error word gets PKV_DEVERR_TIMEOUT; != 0 = both waits
 *                   complete and nothing is reported.
 * The kernel issues no memory copy and returns normally either way; the
 * stream and context stay usable.  Stream-ordered, allocates nothing.
 */
pkv_status pkv_selftest_bounded_wait(uint32_t wait_limit_us, int32_t arm_all, void* stream);

/*
 * Block pool and copy-on-write -- the host-side bookkeeping of §8.3.1/§8.3.2
 * ("Chapter 8: Inference Optimization"): blocks come from a free pool; each
 * block-table entry pointing at a block is a reference (Fig. 8-14: a block
 * returns to the pool when its last reference is released); before a request
 * writes into a shared, partly filled tail block it takes a private copy
 * (Fig. 8-15), while full shared blocks stay shared.
 *
 * The pool is host memory only and is not thread-safe.  It tracks counts; it
 * does not know when device work using a block has finished, so release a
 * block only after the work that reads it has completed (§8.3.2: a block is
 * reused only when no reference holds it and the accelerator no longer reads
 * it).  block_size is the pool's tokens per block (the kernels use 16).
 */
typedef struct pkv_block_pool pkv_block_pool;

pkv_status pkv_block_pool_create(int32_t num_blocks, int32_t block_size, pkv_block_pool** pool);
void pkv_block_pool_destroy(pkv_block_pool* pool);
/* Free blocks, or -1 for a NULL pool. */
int32_t pkv_block_pool_num_free(const pkv_block_pool* pool);
/* References held on `block`, or -1 if it is not a block of the pool. */
int32_t pkv_block_pool_refcount(const pkv_block_pool* pool, int32_t block);
/* n fresh blocks (one reference each) into blocks[0..n); all or nothing
 * (PKV_ERR_EXHAUSTED, nothing taken). */
pkv_status pkv_block_pool_alloc(pkv_block_pool* pool, int32_t n, int32_t* blocks);
/* One more reference on each listed block (a second table now points at it). */
pkv_status pkv_block_pool_share(pkv_block_pool* pool, const int32_t* blocks, int32_t n);
/* Drop one reference per listed block; blocks reaching 0 return to the pool.
 * Rejects (PKV_ERR_SHAPE, nothing changed) a release of a block without a
 * reference to drop. */
pkv_status pkv_block_pool_release(pkv_block_pool* pool, const int32_t* blocks, int32_t n);
/*
 * Make token positions ctx_before .. ctx_before+num_new-1 of one request
 * writable: append fresh blocks to its table row (row_blocks grows, up to
 * max_blocks) and give it a private copy of every shared block among those it
 * already holds that the new tokens fall into.  Each copy is reported as
 * (copy_src[i] -> copy_dst[i]), i < *num_copies (capacity: ceil(num_new /
 * block_size) + 1 entries); the table row already points at copy_dst, so the
 * caller runs pkv_copy_blocks on them before appending.  All or nothing.
 */
pkv_status pkv_block_pool_reserve(pkv_block_pool* pool, int32_t* table_row, int32_t* row_blocks,
                                  int32_t max_blocks, int32_t ctx_before, int32_t num_new,
                                  int32_t* copy_src, int32_t* copy_dst, int32_t* num_copies);

/*
 * pkv_copy_blocks -- copy whole physical blocks (all KV heads, K and V) from
 * src_blocks[i] to dst_blocks[i], bit for bit: the copy half of copy-on-write.
 * src_blocks, dst_blocks: device int32 [num_pairs]; destinations distinct and
 * no destination also a source.  An id outside the pool skips that pair and
 * sets PKV_DEVERR_BLOCK_ID.
 */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                           const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                           void* stream);

/*
 * ---------------------------------------------------------------------------
 * q8_0 KV cache (§8.4.2 "KV compression and read cost", Fig. 8-23): every 32
 * consecutive values of a token's head vector share one 2-byte scale and keep
 * 8-bit codes, 34 bytes instead of 64.  The page fixes the storage; this
 * library quantises with the plain symmetric rule, in FP32 with IEEE
 * rounding at every step:  d = max|x| / 127,  code = round-half-away-from-
 * zero(x * (1/d))  (0 when d = 0),  scale = FP16(d) (round to nearest even),
 * value = scale * code.  Inputs must be finite.
 *
 * Pool layout, per tensor: uint8 [num_blocks][num_kv_heads][PKV_Q8_TILE_BYTES];
 * one (block, kv head) tile is int8 codes [16 tokens][128 dims] (token-major)
 * followed by FP16 scales [16 tokens][4 groups] (group g = dims 32g..32g+31).
 * `cache` describes the geometry exactly as for BF16 pools.
 * ---------------------------------------------------------------------------
 */
#define PKV_Q8_TILE_BYTES 2176u

/*
 * pkv_kv_append_q8_0 -- pkv_kv_append for q8_0 pools: quantise each new
 * token's K and V (BF16 [num_tokens][num_kv_heads][128], 16-byte aligned) and
 * store codes and scales in its slot.  Same slot rules and errors as
 * pkv_kv_append.  Deterministic: the same bits as any IEEE FP32 evaluation of
 * the rule above.
 */
pkv_status pkv_kv_append_q8_0(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                              const int64_t* slot_mapping, const void* k_new, const void* v_new, int32_t num_tokens,
                              void* stream);

/*
 * pkv_choose_kv_blocks_per_split_q8_0 -- blocks per split for
 * pkv_paged_attention_q8_0: its kernel keeps one persistent CTA per SM, so
 * the split count is the one that best balances (request, KV head, split)
 * units over sm_count CTAs (0 = current device), in whole 8-block tiles.
 */
int32_t pkv_choose_kv_blocks_per_split_q8_0(int32_t num_seqs, int32_t num_kv_heads, int32_t max_blocks_per_seq,
                                            int32_t sm_count);

/* Workspace bytes pkv_paged_attention_q8_0 (and the FP8 call) needs (0 when there is one split). */
size_t pkv_workspace_size_q8_0(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                               int32_t kv_blocks_per_split);

/*
 * pkv_paged_attention_q8_0 -- pkv_paged_attention for one decode step
 * (q_len 1) over q8_0 pools: out = softmax(scale * q . K^T) V with K and V
 * the dequantised values (scale * code).  q, out: BF16 [num_seqs][num_q_heads]
 * [128].  kv_blocks_per_split 0 = pkv_choose_kv_blocks_per_split_q8_0; with
 * more than one split, partials go to `workspace` (256-byte aligned,
 * pkv_workspace_size_q8_0 bytes) and are merged by the combine kernel on the
 * same stream.  Queries are scaled by a power of two into FP16 range, so any
 * finite BF16 query is accepted.  Errors as pkv_paged_attention.
 */
pkv_status pkv_paged_attention_q8_0(void* out, const void* q, const void* k_cache, const void* v_cache,
                                    const pkv_cache_desc* cache, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                    int32_t num_q_heads, float scale, int32_t kv_blocks_per_split, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * pkv_paged_attention_q8_0_append -- pkv_kv_append_q8_0 followed by
 * pkv_paged_attention_q8_0, in one call (arguments as for the two).  Ch8
 * §8.1.1: a decode step stores the new token's K and V and reads the context
 * KV, the new token included; §8.4.2 / Fig. 8-23: the stored form is q8_0.
 * When num_tokens == num_seqs (token r is request r's new token, at position
 * context_lens[r] - 1) the decode kernel quantises and stores the tokens
 * itself, exactly as pkv_kv_append_q8_0 does, and uses them in place of the
 * rows it read; other counts issue the append, then the attention.  A slot
 * other than the one the block table gives that position is stored as the
 * append would but sets PKV_DEVERR_SLOT (the result is then undefined); rows
 * with context_lens[r] <= 0 (PKV_DEVERR_SLOT for a slot >= 0) or longer than
 * the table store nothing.  Results equal the two calls' bit for bit
 * otherwise.  Every host check runs before anything is enqueued.
 */
pkv_status pkv_paged_attention_q8_0_append(void* out, const void* q, void* k_cache, void* v_cache,
                                           const pkv_cache_desc* cache, const int32_t* block_tables,
                                           int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                           int32_t num_q_heads, float scale, int32_t kv_blocks_per_split,
                                           void* workspace, size_t workspace_bytes, const int64_t* slot_mapping,
                                           const void* k_new, const void* v_new, int32_t num_tokens, void* stream);

/* pkv_copy_blocks for q8_0 pools (num_kv_heads * PKV_Q8_TILE_BYTES per block). */
pkv_status pkv_copy_blocks_q8_0(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                                void* stream);

/*
 * ---------------------------------------------------------------------------
 * FP8 KV cache (§8.4.4 "Capacity and speed under a quality constraint": K and
 * V stored in FP8 while the query stays BF16).  The page does not fix the FP8
 * variant; this library uses OCP E4M3 (4 exponent bits, bias 7, 3 mantissa
 * bits, subnormals, no infinities, |x| <= 448), rounding each BF16 value to
 * the nearest E4M3 value (ties to even) and saturating finite values beyond
 * 448 to +-448; there is no scale.  Inputs must be finite.
 *
 * Pool layout, per tensor: uint8 [num_blocks][num_kv_heads][16][128] E4M3
 * codes (PKV_FP8_TILE_BYTES per (block, kv head)); `cache` as for BF16 pools.
 * ---------------------------------------------------------------------------
 */
#define PKV_FP8_TILE_BYTES 2048u

/* pkv_kv_append_fp8_e4m3 -- pkv_kv_append for E4M3 pools (rounding as above). */
pkv_status pkv_kv_append_fp8_e4m3(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                  const int64_t* slot_mapping, const void* k_new, const void* v_new,
                                  int32_t num_tokens, void* stream);

/*
 * pkv_choose_kv_blocks_per_split_fp8_e4m3 -- blocks per split for
 * pkv_paged_attention_fp8_e4m3: as pkv_choose_kv_blocks_per_split_q8_0 (one
 * persistent CTA per SM), in whole 16-block tiles, the unit its kernel reads.
 */
int32_t pkv_choose_kv_blocks_per_split_fp8_e4m3(int32_t num_seqs, int32_t num_kv_heads,
                                                int32_t max_blocks_per_seq, int32_t sm_count);

/*
 * pkv_paged_attention_fp8_e4m3 -- one decode step over E4M3 pools with the
 * query in BF16: out = softmax(scale * q . K^T) V on the stored values
 * (Ch8 §8.4.4: K and V in FP8, the query in BF16).  Arguments, workspace
 * (pkv_workspace_size_q8_0) and errors exactly as pkv_paged_attention_q8_0;
 * kv_blocks_per_split 0 = pkv_choose_kv_blocks_per_split_fp8_e4m3.
 */
pkv_status pkv_paged_attention_fp8_e4m3(void* out, const void* q, const void* k_cache, const void* v_cache,
                                        const pkv_cache_desc* cache, const int32_t* block_tables,
                                        int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                        int32_t num_q_heads, float scale, int32_t kv_blocks_per_split,
                                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * pkv_paged_attention_fp8_e4m3_append -- pkv_kv_append_fp8_e4m3 followed by
 * pkv_paged_attention_fp8_e4m3, in one call (arguments as for the two).  When
 * num_tokens == num_seqs (token r is request r's new token, at position
 * context_lens[r] - 1) the decode kernel rounds and stores the tokens itself
 * and uses them in place of the rows it read, as pkv_paged_attention_append
 * does; other counts issue the append, then the attention.  A slot other than
 * the one the block table gives that position is stored as the append would
 * but sets PKV_DEVERR_SLOT (the result is then undefined); rows with
 * context_lens[r] <= 0 or longer than the table store nothing, as for
 * pkv_paged_attention_append.  Results equal the two calls' bit for bit
 * otherwise.
 */
pkv_status pkv_paged_attention_fp8_e4m3_append(void* out, const void* q, void* k_cache, void* v_cache,
                                               const pkv_cache_desc* cache, const int32_t* block_tables,
                                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                                               int32_t num_seqs, int32_t num_q_heads, float scale,
                                               int32_t kv_blocks_per_split, void* workspace, size_t workspace_bytes,
                                               const int64_t* slot_mapping, const void* k_new, const void* v_new,
                                               int32_t num_tokens, void* stream);

/* pkv_copy_blocks for E4M3 pools (num_kv_heads * PKV_FP8_TILE_BYTES per block). */
pkv_status pkv_copy_blocks_fp8_e4m3(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                    const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                                    void* stream);

/* Human-readable name of a status code (static string). */
const char* pkv_status_string(pkv_status status);

/*
 * Decode step as one CUDA graph, with two fixed buffer sets.
 *
 * Ch8 §8.6.3 measures decode rounds with CUDA graphs off and traces the
 * roughly fixed time above the read bound (about 17.6 ms at batch 1) to
 * submitting kernels one by one from the host, which a CUDA graph removes.
 * The page "Popping the GPU bubble" (Photon, §3 "ping-pong slots") keeps a
 * decode step's buffers at fixed addresses, allocated once, so the step can
 * be captured as a graph, and alternates two such buffer sets so that the
 * host prepares one step while the GPU runs the other.  A step of L layers
 * issues L appends and L attention calls; pkv_decode_graph_create captures
 * that step -- for layer l: the append of the step's new tokens into layer
 * l's pools, then the attention over them -- once for each of two buffer
 * sets and instantiates the two graphs; pkv_decode_graph_launch replays one
 * with a single launch.  While the graph of buffer set s runs, the caller
 * fills set 1 - s (the next step's queries, new K/V, slots, tables and
 * lengths), so uploads overlap compute.
 *
 * Per buffer set (all device memory, caller-owned, fixed for the graph's
 * life; the graph reads and writes them at every launch):
 *   q, out        : BF16 [num_layers][num_seqs][q_len][num_q_heads][128]
 *   k_new, v_new  : BF16 [num_layers][num_tokens][num_kv_heads][128]
 *   slot_mapping  : int64 [num_tokens], shared by the layers (<0 = skip)
 *   block_tables  : int32 [num_seqs][max_blocks_per_seq], shared by the layers
 *   context_lens  : int32 [num_seqs], shared by the layers
 *   cascade only  : group_seqs [num_groups][16], group_blocks [num_groups],
 *                   seq_prefix_blocks [num_seqs] (as pkv_paged_attention_cascade)
 * Shared by both sets:
 *   k_caches, v_caches : host arrays of num_layers device pointers, the
 *                        layers' pools (format kv_format, geometry `cache`)
 *   workspace          : the attention call's workspace (the graphs run in
 *                        stream order, so one serves both), sized by
 *                        pkv_workspace_size / _q8_0 / pkv_cascade_workspace_size
 * kv_format: PKV_KV_BF16 (pkv_paged_attention_append, or
 * pkv_paged_attention_cascade_append when num_groups > 0), PKV_KV_FP8_E4M3
 * (pkv_paged_attention_fp8_e4m3_append) -- the append fused into the
 * attention where they can -- or PKV_KV_Q8_0 (its append and decode calls);
 * quantised pools: q_len 1, no groups.
 * Split sizes as for the direct calls (0 = the library's heuristic).
 *
 * Ownership and errors: create validates every call of the step with the
 * same rules as the direct calls, returning the first failing status and no
 * graph; it allocates host memory and two CUDA graph executables (the only
 * entry point that does) and enqueues nothing.  launch enqueues one graph on
 * `stream` and allocates nothing; buffer_set must be 0 or 1.  destroy frees
 * both graphs; the caller must not destroy a graph while a launch of it may
 * still run.  The device error word behaves as for the direct calls.
 */
typedef enum pkv_kv_format { PKV_KV_BF16 = 0, PKV_KV_Q8_0 = 1, PKV_KV_FP8_E4M3 = 2 } pkv_kv_format;

typedef struct pkv_decode_graph_buffers {
  const void* q;
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  const int32_t* group_seqs;
  const int32_t* group_blocks;
  const int32_t* seq_prefix_blocks;
} pkv_decode_graph_buffers;

typedef struct pkv_decode_graph_desc {
  int32_t num_layers;
  int32_t kv_format;             /* pkv_kv_format */
  pkv_cache_desc cache;
  void* const* k_caches;         /* [num_layers] */
  void* const* v_caches;         /* [num_layers] */
  int32_t num_seqs;
  int32_t q_len;
  int32_t num_q_heads;
  int32_t max_blocks_per_seq;
  int32_t num_tokens;            /* new tokens appended per layer */
  float scale;
  int32_t kv_blocks_per_split;   /* non-cascade calls; 0 = heuristic */
  int32_t num_groups;            /* BF16 decode only: > 0 = cascade */
  int32_t max_prefix_blocks;
  int32_t max_suffix_blocks;
  int32_t prefix_blocks_per_split;
  int32_t suffix_blocks_per_split;
  void* workspace;
  size_t workspace_bytes;
  pkv_decode_graph_buffers set[2];
} pkv_decode_graph_desc;

typedef struct pkv_decode_graph pkv_decode_graph; /* opaque */

pkv_status pkv_decode_graph_create(const pkv_decode_graph_desc* desc, pkv_decode_graph** graph);
pkv_status pkv_decode_graph_launch(pkv_decode_graph* graph, int32_t buffer_set, void* stream);
void pkv_decode_graph_destroy(pkv_decode_graph* graph);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
