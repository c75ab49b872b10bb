// kv_append.cu -- store each new token's K and V in its cache slot.
//
// "Chapter 8: Inference Optimization" (clxhxhhr.top/posts/4341), §8.1.1: a
// step stores the K and V of the token it processes; §8.3.1: token slot s
// lives in physical block s / 16 at offset s % 16.
//
// One thread moves 16 bytes; consecutive threads cover consecutive 16-byte
// chunks of one (token, kv head) row of 256 bytes, so both the read of
// k_new/v_new and the write into the 4 KiB cache tile are coalesced.  The
// copy is a bit copy.  The q8_0 variant quantises each 32-value group on
// the way in; the FP8 variant rounds each value to E4M3.
#include <cuda_fp16.h>

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

// q8_0 append ("Chapter 8: Inference Optimization" §8.4.2, Fig. 8-23): one
// warp per (token, kv head, K|V) row of 128 values; lane l holds values
// 4l..4l+3, so lanes 8g..8g+7 hold group g.  Per group: d = max|x| / 127,
// code = round-half-away(x * (1/d)), scale stored as FP16 (round to nearest
// even).  Every step is one IEEE-rounded FP32 operation, so the codes and
// scales are the same bits a CPU computes with the same operations.
__global__ void __launch_bounds__(256) kv_append_q8_kernel(uint8_t* __restrict__ k_cache,
                                                           uint8_t* __restrict__ v_cache, int64_t pool_slots,
                                                           int32_t num_kv_heads,
                                                           const int64_t* __restrict__ slot_mapping,
                                                           const uint2* __restrict__ k_new,
                                                           const uint2* __restrict__ v_new, int64_t rows,
                                                           unsigned int* err) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t item = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; item < rows;
       item += warps) {
    // item = (t * 2 + which) * Hkv + h
    const int h = static_cast<int>(item % num_kv_heads);
    const int64_t rest = item / num_kv_heads;
    const int which = static_cast<int>(rest & 1);
    const int64_t t = rest >> 1;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= pool_slots) {
      if (lane == 0 && h == 0 && which == 0) report(err, PKV_DEVERR_SLOT);
      continue;
    }
    const uint2 w = (which ? v_new : k_new)[(t * num_kv_heads + h) * (kHeadDim / 4) + lane];
    float d;
    const uint32_t codes = q8_0_quantize_lane(w, d);
    const int64_t blk = slot / kBlockSize;
    const int off = static_cast<int>(slot % kBlockSize);
    uint8_t* tile = (which ? v_cache : k_cache) + (blk * num_kv_heads + h) * kQ8TileBytes;
    *reinterpret_cast<uint32_t*>(tile + off * kHeadDim + lane * 4) = codes;
    if ((lane & 7) == 0)
      *reinterpret_cast<__half*>(tile + kQ8CodeBytes + (off * 4 + (lane >> 3)) * 2) = __float2half_rn(d);
  }
}

// FP8 append (§8.4.4): one thread converts 8 BF16 values of a (token, kv
// head) row to E4M3 (hardware round to nearest even, saturating at +-448)
// and stores 8 bytes; consecutive threads cover consecutive 8-value chunks.
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
                                                            int64_t pool_slots, int32_t num_kv_heads,
                                                            const int64_t* __restrict__ slot_mapping,
                                                            const uint4* __restrict__ k_new,
                                                            const uint4* __restrict__ v_new, int64_t total,
                                                            unsigned int* err) {
  pdl_wait();
  pdl_trigger();
  for (int64_t item = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; item < total;
       item += (int64_t)gridDim.x * blockDim.x) {
    const int chunk = static_cast<int>(item % kChunksPerRow);  // 8 values each
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
    const uint4 w = (which ? v_new : k_new)[(t * num_kv_heads + h) * kChunksPerRow + chunk];
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t pairs[4];  // E4M3 pairs, element 2e in the low byte
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint16_t p2;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(p2) : "f"(bf16_hi(in[e])), "f"(bf16_lo(in[e])));
      pairs[e] = p2;
    }
    const int64_t blk = slot / kBlockSize;
    const int off = static_cast<int>(slot % kBlockSize);
    const int64_t dst = ((blk * num_kv_heads + h) * kBlockSize + off) * kChunksPerRow + chunk;
    (which ? v_cache : k_cache)[dst] = make_uint2(pairs[0] | (pairs[1] << 16), pairs[2] | (pairs[3] << 16));
  }
}

}  // namespace

cudaError_t launch_kv_append_fp8(void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                                 const int64_t* slot_mapping, const void* k_new, const void* v_new,
                                 int32_t num_tokens, unsigned int* err, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(num_tokens) * 2 * num_kv_heads * kChunksPerRow;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  return launch_pdl(kv_append_fp8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1,
                    static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache),
                    static_cast<int64_t>(num_blocks) * kBlockSize, num_kv_heads, slot_mapping,
                    static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), total, err);
}

cudaError_t launch_kv_append_q8(void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                                const int64_t* slot_mapping, const void* k_new, const void* v_new,
                                int32_t num_tokens, unsigned int* err, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(num_tokens) * 2 * num_kv_heads;
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;  // 8 warps per CTA
  if (blocks > 65536) blocks = 65536;
  return launch_pdl(kv_append_q8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1,
                    static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache),
                    static_cast<int64_t>(num_blocks) * kBlockSize, num_kv_heads, slot_mapping,
                    static_cast<const uint2*>(k_new), static_cast<const uint2*>(v_new), rows, err);
}

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
