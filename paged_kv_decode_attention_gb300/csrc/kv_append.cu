// kv_append.cu -- store each new token's K and V in its cache slot.
//
// "Chapter 8: Inference Optimization" (clxhxhhr.top/posts/4341), §8.1.1: a
// step stores the K and V of the token it processes; §8.3.1: token slot s
// lives in physical block s / 16 at offset s % 16.
//
// One thread moves 16 bytes; consecutive threads cover consecutive 16-byte
// chunks of one (token, kv head) row of 256 bytes, so both the read of
// k_new/v_new and the write into the 4 KiB cache tile are coalesced.  The
// copy is a bit copy.
#include "pkv_common.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

constexpr int kChunksPerRow = kHeadDim * 2 / 16;  // 16 x 16 B per (token, head) row

__global__ void __launch_bounds__(256) kv_append_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                        int64_t pool_slots, int32_t num_kv_heads,
                                                        const int64_t* __restrict__ slot_mapping,
                                                        const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new, int64_t total,
                                                        unsigned int* err) {
  pdl_wait();  // new K/V and slots may come from the previous grid
  pdl_trigger();
  // item = ((t * 2 + which) * Hkv + h) * 16 + chunk
  for (int64_t item = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; item < total;
       item += (int64_t)gridDim.x * blockDim.x) {
    const int chunk = static_cast<int>(item % kChunksPerRow);
    int64_t rest = item / kChunksPerRow;
    const int h = static_cast<int>(rest % num_kv_heads);
    rest /= num_kv_heads;
    const int which = static_cast<int>(rest & 1);
    const int64_t t = rest >> 1;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= pool_slots) {
      if (chunk == 0 && h == 0 && which == 0) report(err, PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = slot / kBlockSize;
    const int off = static_cast<int>(slot % kBlockSize);
    const int64_t src = (t * num_kv_heads + h) * kChunksPerRow + chunk;
    const int64_t dst = ((blk * num_kv_heads + h) * kBlockSize + off) * kChunksPerRow + chunk;
    if (which == 0)
      k_cache[dst] = k_new[src];
    else
      v_cache[dst] = v_new[src];
  }
}

}  // namespace

cudaError_t launch_kv_append(void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                             const int64_t* slot_mapping, const void* k_new, const void* v_new,
                             int32_t num_tokens, unsigned int* err, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(num_tokens) * 2 * num_kv_heads * kChunksPerRow;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 65536) blocks = 65536;
  return launch_pdl(kv_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, 1,
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                    static_cast<int64_t>(num_blocks) * kBlockSize, num_kv_heads, slot_mapping,
                    static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), total, err);
}

}  // namespace pkv
