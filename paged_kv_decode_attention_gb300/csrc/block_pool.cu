// block_pool.cu -- host-side block manager and the copy-on-write block copy.
//
// "Chapter 8: Inference Optimization" (clxhxhhr.top/posts/4341):
//   §8.3.1: KV is allocated in fixed-size physical blocks from a free pool;
//           a request's block table maps its logical blocks to them.
//   §8.3.2 / Fig. 8-14: every block-table entry pointing at a block is a
//           reference; the block returns to the pool only when its last
//           reference is released.
//   §8.3.2 / Fig. 8-15: before writing into a shared, partly filled tail
//           block, the writer takes a private copy (copy-on-write); blocks
//           already full stay shared.
// The pool is plain host code (no CUDA call); only pkv_copy_blocks launches
// work.  A pool is not thread-safe: callers serialise access to one pool.
#include <cstdint>
#include <new>
#include <vector>

#include "pkv.h"
#include "pkv_common.cuh"
#include "pkv_kernels.h"

struct pkv_block_pool {
  int32_t block_size = 16;
  std::vector<int32_t> refs;  // references per block; 0 = free
  std::vector<int32_t> free_list;
};

namespace pkv {
namespace {

bool valid_block(const pkv_block_pool* p, int32_t b) {
  return b >= 0 && b < static_cast<int32_t>(p->refs.size());
}

// One thread moves 16 bytes; a CTA moves one block of one tensor (K or V),
// i.e. all KV heads of that block, contiguous (BF16 or q8_0 tiles alike).
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                          int32_t num_blocks, int32_t chunks_per_block,
                                                          const int32_t* __restrict__ src,
                                                          const int32_t* __restrict__ dst, unsigned int* err) {
  pdl_wait();
  pdl_trigger();
  const int pair = blockIdx.x >> 1;
  uint4* cache = (blockIdx.x & 1) ? v_cache : k_cache;
  const int32_t s = src[pair];
  const int32_t d = dst[pair];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0) report(err, PKV_DEVERR_BLOCK_ID);
    return;
  }
  const uint4* from = cache + static_cast<int64_t>(s) * chunks_per_block;
  uint4* to = cache + static_cast<int64_t>(d) * chunks_per_block;
  for (int i = threadIdx.x; i < chunks_per_block; i += blockDim.x) to[i] = from[i];
}

}  // namespace

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, int32_t num_blocks, int64_t block_bytes,
                               const int32_t* src, const int32_t* dst, int32_t num_pairs, unsigned int* err,
                               cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int32_t chunks = static_cast<int32_t>(block_bytes / 16);
  return launch_pdl(copy_blocks_kernel, dim3(static_cast<unsigned>(num_pairs) * 2), dim3(256), 0, stream, 1,
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_blocks, chunks, src, dst, err);
}

}  // namespace pkv

using namespace pkv;

extern "C" {

pkv_status pkv_block_pool_create(int32_t num_blocks, int32_t block_size, pkv_block_pool** pool) {
  if (pool == nullptr) return PKV_ERR_NULL;
  *pool = nullptr;
  if (num_blocks < 0 || block_size < 1) return PKV_ERR_SHAPE;
  pkv_block_pool* p = new (std::nothrow) pkv_block_pool;
  if (p == nullptr) return PKV_ERR_EXHAUSTED;
  p->block_size = block_size;
  p->refs.assign(static_cast<size_t>(num_blocks), 0);
  p->free_list.reserve(static_cast<size_t>(num_blocks));
  for (int32_t b = num_blocks - 1; b >= 0; --b) p->free_list.push_back(b);  // hand out 0, 1, 2, ... first
  *pool = p;
  return PKV_OK;
}

void pkv_block_pool_destroy(pkv_block_pool* pool) { delete pool; }

int32_t pkv_block_pool_num_free(const pkv_block_pool* pool) {
  return pool ? static_cast<int32_t>(pool->free_list.size()) : -1;
}

int32_t pkv_block_pool_refcount(const pkv_block_pool* pool, int32_t block) {
  if (pool == nullptr || !valid_block(pool, block)) return -1;
  return pool->refs[static_cast<size_t>(block)];
}

pkv_status pkv_block_pool_alloc(pkv_block_pool* pool, int32_t n, int32_t* blocks) {
  if (pool == nullptr || (n > 0 && blocks == nullptr)) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_SHAPE;
  if (static_cast<size_t>(n) > pool->free_list.size()) return PKV_ERR_EXHAUSTED;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = pool->free_list.back();
    pool->free_list.pop_back();
    pool->refs[static_cast<size_t>(b)] = 1;
    blocks[i] = b;
  }
  return PKV_OK;
}

pkv_status pkv_block_pool_share(pkv_block_pool* pool, const int32_t* blocks, int32_t n) {
  if (pool == nullptr || (n > 0 && blocks == nullptr)) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_SHAPE;
  for (int32_t i = 0; i < n; ++i)
    if (!valid_block(pool, blocks[i]) || pool->refs[static_cast<size_t>(blocks[i])] == 0) return PKV_ERR_SHAPE;
  for (int32_t i = 0; i < n; ++i) ++pool->refs[static_cast<size_t>(blocks[i])];
  return PKV_OK;
}

pkv_status pkv_block_pool_release(pkv_block_pool* pool, const int32_t* blocks, int32_t n) {
  if (pool == nullptr || (n > 0 && blocks == nullptr)) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_SHAPE;
  // validate against the counts this call would leave (a block may repeat)
  std::vector<int32_t> seen;
  for (int32_t i = 0; i < n; ++i) {
    if (!valid_block(pool, blocks[i])) return PKV_ERR_SHAPE;
    int32_t k = 0;
    for (int32_t b : seen) k += (b == blocks[i]);
    if (k >= pool->refs[static_cast<size_t>(blocks[i])]) return PKV_ERR_SHAPE;
    seen.push_back(blocks[i]);
  }
  for (int32_t i = 0; i < n; ++i) {
    int32_t& r = pool->refs[static_cast<size_t>(blocks[i])];
    if (--r == 0) pool->free_list.push_back(blocks[i]);
  }
  return PKV_OK;
}

pkv_status pkv_block_pool_reserve(pkv_block_pool* pool, int32_t* table_row, int32_t* row_blocks,
                                  int32_t max_blocks, int32_t ctx_before, int32_t num_new, int32_t* copy_src,
                                  int32_t* copy_dst, int32_t* num_copies) {
  if (pool == nullptr || table_row == nullptr || row_blocks == nullptr || num_copies == nullptr) return PKV_ERR_NULL;
  *num_copies = 0;
  if (num_new < 0 || ctx_before < 0 || max_blocks < 0 || *row_blocks < 0 || *row_blocks > max_blocks)
    return PKV_ERR_SHAPE;
  if (num_new == 0) return PKV_OK;
  const int32_t p = pool->block_size;
  const int32_t have = *row_blocks;
  if (ctx_before > have * p) return PKV_ERR_SHAPE;  // the row must already hold every earlier token
  const int32_t need = (ctx_before + num_new + p - 1) / p;
  if (need > max_blocks) return PKV_ERR_SHAPE;
  // blocks already in the row that the new tokens write into: only a partly
  // filled tail can be both shared and written
  const int32_t first = ctx_before / p;
  int32_t cow = 0;
  for (int32_t j = first; j < have && j < need; ++j) {
    if (!valid_block(pool, table_row[j])) return PKV_ERR_SHAPE;
    if (pool->refs[static_cast<size_t>(table_row[j])] > 1) ++cow;
  }
  if (cow > 0 && (copy_src == nullptr || copy_dst == nullptr)) return PKV_ERR_NULL;
  const int32_t fresh = need > have ? need - have : 0;
  if (static_cast<size_t>(cow + fresh) > pool->free_list.size()) return PKV_ERR_EXHAUSTED;
  int32_t nc = 0;
  for (int32_t j = first; j < have && j < need; ++j) {
    const int32_t src = table_row[j];
    if (pool->refs[static_cast<size_t>(src)] <= 1) continue;
    int32_t dst = 0;
    pkv_block_pool_alloc(pool, 1, &dst);
    --pool->refs[static_cast<size_t>(src)];  // this row no longer references the shared block
    table_row[j] = dst;
    copy_src[nc] = src;
    copy_dst[nc] = dst;
    ++nc;
  }
  if (fresh > 0) pkv_block_pool_alloc(pool, fresh, table_row + have);
  *row_blocks = need > have ? need : have;
  *num_copies = nc;
  return PKV_OK;
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* cache, const int32_t* src_blocks,
                           const int32_t* dst_blocks, int32_t num_pairs, void* stream) {
  if (cache == nullptr) return PKV_ERR_NULL;
  if (cache->num_blocks < 0 || cache->num_kv_heads <= 0 || num_pairs < 0) return PKV_ERR_SHAPE;
  if (cache->block_size != kBlockSize || cache->head_dim != kHeadDim) return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_blocks || !dst_blocks) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15) return PKV_ERR_UNSUPPORTED;
  if (num_pairs > (1 << 30)) return PKV_ERR_UNSUPPORTED;
  return launch_copy_blocks(k_cache, v_cache, cache->num_blocks,
                            static_cast<int64_t>(cache->num_kv_heads) * kTileBytes, src_blocks, dst_blocks, num_pairs,
                            device_error_word(), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

static pkv_status copy_blocks_bytes(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                    const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                                    int32_t tile_bytes, void* stream) {
  if (cache == nullptr) return PKV_ERR_NULL;
  if (cache->num_blocks < 0 || cache->num_kv_heads <= 0 || num_pairs < 0) return PKV_ERR_SHAPE;
  if (cache->block_size != kBlockSize || cache->head_dim != kHeadDim) return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_blocks || !dst_blocks) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15) return PKV_ERR_UNSUPPORTED;
  if (num_pairs > (1 << 30)) return PKV_ERR_UNSUPPORTED;
  return launch_copy_blocks(k_cache, v_cache, cache->num_blocks, static_cast<int64_t>(cache->num_kv_heads) * tile_bytes,
                            src_blocks, dst_blocks, num_pairs, device_error_word(),
                            static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks_fp8_e4m3(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                    const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                                    void* stream) {
  return copy_blocks_bytes(k_cache, v_cache, cache, src_blocks, dst_blocks, num_pairs, kFp8TileBytes, stream);
}

pkv_status pkv_copy_blocks_q8_0(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                                void* stream) {
  if (cache == nullptr) return PKV_ERR_NULL;
  if (cache->num_blocks < 0 || cache->num_kv_heads <= 0 || num_pairs < 0) return PKV_ERR_SHAPE;
  if (cache->block_size != kBlockSize || cache->head_dim != kHeadDim) return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_blocks || !dst_blocks) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15) return PKV_ERR_UNSUPPORTED;
  if (num_pairs > (1 << 30)) return PKV_ERR_UNSUPPORTED;
  return launch_copy_blocks(k_cache, v_cache, cache->num_blocks,
                            static_cast<int64_t>(cache->num_kv_heads) * kQ8TileBytes, src_blocks, dst_blocks,
                            num_pairs, device_error_word(), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

}  // extern "C"
