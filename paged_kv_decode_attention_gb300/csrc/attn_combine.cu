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
constexpr int kThreadsCombine = 128;

// One row per warp (kWarpsPerRow = 1) or one row per CTA with the 4 warps
// taking every 4th split (kWarpsPerRow = 4, for many splits and few rows).
// Lane l owns dims 4l..4l+3.  The lse of 32 splits at a time sit one per
// lane; their weights are broadcast by shuffles, so the partial-output loads
// of consecutive splits are independent and overlap.
template <int kWarpsPerRow>
__global__ void __launch_bounds__(kThreadsCombine) attn_combine_kernel(uint16_t* __restrict__ out,
                                                                       float* __restrict__ out_lse,
                                                                       const float* __restrict__ part_o,
                                                                       const float* __restrict__ part_lse,
                                                                       int32_t num_rows, int32_t num_splits) {
  pdl_wait();  // the partials come from the previous grid
  pdl_trigger();
  constexpr int kRowsPerCta = 4 / kWarpsPerRow;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + warp / kWarpsPerRow;
  const int sub = warp % kWarpsPerRow;  // this warp's share of the splits
  __shared__ float red[4][4 * 32 + 1];  // partial sums when several warps share a row
  const bool live = row < num_rows;
  const float* lse = part_lse + (live ? row : 0) * num_splits;

  float mx = -INFINITY;
  if (live)
    for (int s = lane; s < num_splits; s += 32) mx = fmaxf(mx, lse[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

  float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f, sum = 0.f;
  if (live && mx != -INFINITY) {
    const float* po = part_o + (row * num_splits) * kHeadDim + lane * 4;
    for (int base = 0; base < num_splits; base += 32) {
      const int s_l = base + lane;
      const float l_l = s_l < num_splits ? lse[s_l] : -INFINITY;
      const float w_l = (l_l == -INFINITY) ? 0.f : exp2_approx((l_l - mx) * kLog2e);
      const int cnt = min(32, num_splits - base);
#pragma unroll 4
      for (int u = sub; u < cnt; u += kWarpsPerRow) {
        const float w = __shfl_sync(0xffffffffu, w_l, u);
        if (w == 0.f) continue;  // empty split: its output is never read
        const float4 v = *reinterpret_cast<const float4*>(po + static_cast<int64_t>(base + u) * kHeadDim);
        sum += w;
        o0 = fmaf(w, v.x, o0);
        o1 = fmaf(w, v.y, o1);
        o2 = fmaf(w, v.z, o2);
        o3 = fmaf(w, v.w, o3);
      }
    }
  }
  if constexpr (kWarpsPerRow > 1) {
    red[warp][lane * 4 + 0] = o0;
    red[warp][lane * 4 + 1] = o1;
    red[warp][lane * 4 + 2] = o2;
    red[warp][lane * 4 + 3] = o3;
    if (lane == 0) red[warp][128] = sum;
    __syncthreads();
    if (warp != 0) return;
    for (int w2 = 1; w2 < kWarpsPerRow; ++w2) {
      o0 += red[w2][lane * 4 + 0];
      o1 += red[w2][lane * 4 + 1];
      o2 += red[w2][lane * 4 + 2];
      o3 += red[w2][lane * 4 + 3];
      sum += red[w2][128];
    }
  }
  if (!live) return;
  const float inv = (mx != -INFINITY && sum > 0.f) ? 1.f / sum : 0.f;
  uint2 packed;
  packed.x = pack_bf16x2(o0 * inv, o1 * inv);
  packed.y = pack_bf16x2(o2 * inv, o3 * inv);
  *reinterpret_cast<uint2*>(out + row * kHeadDim + lane * 4) = packed;
  if (out_lse != nullptr && lane == 0) out_lse[row] = (mx == -INFINITY || sum <= 0.f) ? -INFINITY : mx + logf(sum);
}

}  // namespace

cudaError_t launch_attn_combine(void* out, float* out_lse, const float* part_o, const float* part_lse,
                                int32_t num_rows, int32_t num_splits, cudaStream_t stream) {
  if (num_rows == 0) return cudaSuccess;
  uint16_t* o = static_cast<uint16_t*>(out);
  // four warps per row only when the rows are too few to fill the GPU: with
  // many rows, one warp per row keeps more rows' loads in flight
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (num_splits >= 8 && num_rows < 16 * sms)
    return launch_pdl(attn_combine_kernel<4>, dim3(static_cast<unsigned>(num_rows)), dim3(kThreadsCombine), 0,
                      stream, 1, o, out_lse, part_o, part_lse, num_rows, num_splits);
  return launch_pdl(attn_combine_kernel<1>, dim3(static_cast<unsigned>((num_rows + 3) / 4)), dim3(kThreadsCombine), 0,
                    stream, 1, o, out_lse, part_o, part_lse, num_rows, num_splits);
}

}  // namespace pkv
