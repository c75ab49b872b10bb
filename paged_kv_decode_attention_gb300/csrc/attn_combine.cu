// attn_combine.cu -- merge split-KV partial attention results.
//
// A softmax over the union of disjoint key ranges equals the mix of the
// per-range softmaxes weighted by exp(lse_s - lse), lse = log sum_s exp(lse_s):
// the same identity the blockwise (FlashAttention-style) evaluation named in
// "Chapter 8: Inference Optimization" §8.3.1 applies inside one CTA, applied
// here across CTAs.  One warp per output row; lane l owns dims 4l..4l+3.
// Splits with lse = -inf (no keys) are skipped without reading their output.
#include <cmath>

#include "pkv_common.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRowsPerCta = 4;

__global__ void __launch_bounds__(kRowsPerCta * 32) attn_combine_kernel(uint16_t* __restrict__ out,
                                                                         float* __restrict__ out_lse,
                                                                         const float* __restrict__ part_o,
                                                                         const float* __restrict__ part_lse,
                                                                         int32_t num_rows, int32_t num_splits) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= num_rows) return;
  const float* lse = part_lse + row * num_splits;

  float mx = -INFINITY;
  for (int s = lane; s < num_splits; s += 32) mx = fmaxf(mx, lse[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

  float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f, sum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < num_splits; ++s) {
      const float l = lse[s];
      if (l == -INFINITY) continue;
      const float w = exp2_approx((l - mx) * kLog2e);
      sum += w;
      const float4 v = *reinterpret_cast<const float4*>(part_o + (row * num_splits + s) * kHeadDim + lane * 4);
      o0 = fmaf(w, v.x, o0);
      o1 = fmaf(w, v.y, o1);
      o2 = fmaf(w, v.z, o2);
      o3 = fmaf(w, v.w, o3);
    }
    const float inv = 1.f / sum;
    o0 *= inv;
    o1 *= inv;
    o2 *= inv;
    o3 *= inv;
  }
  uint2 packed;
  packed.x = pack_bf16x2(o0, o1);
  packed.y = pack_bf16x2(o2, o3);
  *reinterpret_cast<uint2*>(out + row * kHeadDim + lane * 4) = packed;
  if (out_lse != nullptr && lane == 0) out_lse[row] = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
}

}  // namespace

cudaError_t launch_attn_combine(void* out, float* out_lse, const float* part_o, const float* part_lse,
                                int32_t num_rows, int32_t num_splits, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((num_rows + kRowsPerCta - 1) / kRowsPerCta);
  attn_combine_kernel<<<blocks, kRowsPerCta * 32, 0, stream>>>(static_cast<uint16_t*>(out), out_lse, part_o,
                                                                 part_lse, num_rows, num_splits);
  return cudaGetLastError();
}

}  // namespace pkv
