// paged_decode.cu -- attention of one query token per (request, KV head)
// over a paged BF16 KV cache, optionally over one range ("split") of the
// request's blocks.
//
// What it computes ("Chapter 8: Inference Optimization",
// clxhxhhr.top/posts/4341): §8.1.1 -- the decode step reads the request's
// context KV; §8.3.1 / Fig. 8-10 -- logical block j of the request is found
// through its block table; §8.3.2 / Fig. 8-13 -- shared prefix blocks are
// ordinary table entries; §8.2.3 -- query i of a q_len-token chunk sees the
// first ctx - q_len + 1 + i tokens (each query row is run as its own decode
// over that prefix).  Softmax is evaluated blockwise with a running maximum
// and sum (online softmax), the way FlashAttention organises attention inside
// the kernel (§8.3.1 names it), so no score vector reaches memory.
//
// Work decomposition: one CTA per (query row, split, KV head).  Consecutive
// CTAs take consecutive requests of the same split and KV head, so requests
// that share prefix blocks read them close together in time (L2 reuse).
//
// CTA = 4 consumer warps + 1 producer warp.
//   producer : lane 0 streams each (block, kv head) K tile and V tile (4 KiB
//              each, contiguous in the cache layout) into a ring of kStages
//              shared-memory stages with cp.async.bulk, completion counted on
//              a per-stage "full" mbarrier; block ids are fetched 32 at a time
//              by the whole warp.  A stage is refilled once all 4 consumer
//              warps have arrived on its "empty" mbarrier.
//   consumers: warp w owns tokens 4w..4w+3 of every block and keeps its own
//              running max / sum / accumulator for all 4 query heads of the
//              GQA group, so each KV tile is read from HBM once per group.
//   QK^T     : lanes (g = lane/8, j = lane%8): token 4w+g, dims 8j..8j+7 and
//              64+8j..64+8j+7 (two conflict-free 16-byte shared loads).  Each
//              lane holds the matching query slices of all 4 heads (FP32,
//              pre-scaled by scale*log2 e) in a lane-dependent head order, so
//              that the 4 partial dot products reduce-scatter over the 8
//              lanes in 4 shuffles with no selects; lane (g, j) ends with the
//              score of head j/2.
//   softmax  : base-2, FP32; block maximum per head by 2 shuffles; the
//              accumulators are rescaled only when some running max moved.
//   PV       : lanes (hf = lane/16, c = lane%16): tokens 4w+hf and 4w+hf+2,
//              dims 8c..8c+7, FP32 accumulators for the 4 heads; the weights
//              come from a tiny per-warp shared buffer (broadcast reads).
//   epilogue : the 4 warps' (max, sum, acc) are merged through shared memory;
//              with one split the BF16 result is written, otherwise the
//              split's normalised FP32 output and its natural-log lse.
#include <cmath>

#include "pkv_common.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageBytes = 2 * kTileBytes;  // K tile, then V tile
constexpr int kRowBytes = kHeadDim * 2;      // one token of one head: 256 B
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kFull = 0xffffffffu;

template <int NS>
struct DecodeSmem {
  static constexpr int kBarOffset = NS * kStageBytes;
  static constexpr int kPOffset = kBarOffset + 2 * NS * 8;            // float [2][4 warps][4 tok][4 heads]
  static constexpr int kMOffset = kPOffset + 2 * kConsumerWarps * 16 * 4;  // float [4 warps][4 heads]
  static constexpr int kLOffset = kMOffset + kConsumerWarps * 4 * 4;
  static constexpr int kBytes = kLOffset + kConsumerWarps * 4 * 4;
  static_assert(NS * kStageBytes >= kConsumerWarps * kGroup * kHeadDim * 4, "epilogue scratch");
};

__device__ __forceinline__ void unpack8(const uint4 v, float* f) {
  f[0] = bf16_lo(v.x);
  f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y);
  f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z);
  f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w);
  f[7] = bf16_hi(v.w);
}

template <int NS>
__global__ void __launch_bounds__(kThreads, 2) paged_decode_kernel(const DecodeArgs a) {
  using L = DecodeSmem<NS>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty_bar = full_bar + NS;
  float* p_s = reinterpret_cast<float*>(smem + L::kPOffset);
  float* m_s = reinterpret_cast<float*>(smem + L::kMOffset);
  float* l_s = reinterpret_cast<float*>(smem + L::kLOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int vrow = blockIdx.x;  // r * q_len + i
  const int split = blockIdx.y;
  const int kvh = blockIdx.z;
  const int r = vrow / a.q_len;
  const int i = vrow - r * a.q_len;
  const int hq = a.num_kv_heads * kGroup;

  const int ctx = a.context_lens[r];
  int n_vis = ctx - a.q_len + 1 + i;  // keys visible to query i
  if (n_vis > a.max_blocks * kBlockSize) {
    if (threadIdx.x == 0 && split == 0 && kvh == 0) report(a.err, PKV_DEVERR_CONTEXT);
    n_vis = a.max_blocks * kBlockSize;
  }
  if (ctx <= 0 || n_vis < 0) n_vis = 0;
  const int nb = (n_vis + kBlockSize - 1) / kBlockSize;
  const int b0 = split * a.blocks_per_split;
  const int b1 = min(nb, b0 + a.blocks_per_split);
  const int64_t qrow0 = static_cast<int64_t>(vrow) * hq + kvh * kGroup;  // (r, i, first head of group)

  if (b0 >= b1) {  // nothing to read: padding row, query without keys, or a split past the context
    if (a.num_splits == 1) {
      if (threadIdx.x < kGroup * kRowBytes / 16)
        reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + qrow0 * kHeadDim)[threadIdx.x] =
            make_uint4(0, 0, 0, 0);
    } else if (threadIdx.x < kGroup) {
      a.part_lse[(qrow0 + threadIdx.x) * a.num_splits + split] = -INFINITY;
    }
    return;
  }
  const int n_iter = b1 - b0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    const uint64_t policy = l2_policy_evict_first();
    const int32_t* table = a.block_tables + static_cast<int64_t>(r) * a.max_blocks + b0;
    const uint8_t* kbase = static_cast<const uint8_t*>(a.k_cache);
    const uint8_t* vbase = static_cast<const uint8_t*>(a.v_cache);
    bool ok = true;
    int issued = 0;
    for (int base = 0; base < n_iter && ok; base += 32) {
      int blk = 0;
      if (base + lane < n_iter) {
        blk = table[base + lane];
        if (blk < 0 || blk >= a.num_blocks) {
          report(a.err, PKV_DEVERR_BLOCK_ID);
          blk = 0;
        }
      }
      const int cnt = min(32, n_iter - base);
      for (int u = 0; u < cnt; ++u) {
        const int pb = __shfl_sync(kFull, blk, u);
        const int it = base + u;
        const int st = it % NS;
        if (lane == 0) {
          if (it >= NS) ok = mbar_wait(&empty_bar[st], ((it / NS) & 1) ^ 1);
          if (ok) {
            mbar_arrive_expect_tx(&full_bar[st], kStageBytes);
            const size_t off = (static_cast<size_t>(pb) * a.num_kv_heads + kvh) * kTileBytes;
            bulk_copy_g2s(stages + st * kStageBytes, kbase + off, kTileBytes, &full_bar[st], policy);
            bulk_copy_g2s(stages + st * kStageBytes + kTileBytes, vbase + off, kTileBytes, &full_bar[st],
                          policy);
            ++issued;
          }
        }
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0) {
      if (!ok) report(a.err, PKV_DEVERR_TIMEOUT);
      // every issued copy must land before the CTA's shared memory is released
      for (int it = max(0, issued - NS); it < issued; ++it) mbar_wait(&full_bar[it % NS], (it / NS) & 1);
    }
    return;
  }

  // ------------------------------ consumers ------------------------------
  const int g = lane >> 3;   // QK: token within the warp's 4
  const int j = lane & 7;    // QK: dim slice
  const int jj = j >> 1;     // QK: head whose score this lane ends with
  const int hf = lane >> 4;  // PV: token parity
  const int c = lane & 15;   // PV: dim slice

  // Query slices, slot hs = head (hs ^ jj), dims 8j..8j+7 then 64+8j..64+8j+7.
  float qf[4][16];
  {
    const uint16_t* qb = static_cast<const uint16_t*>(a.q) + qrow0 * kHeadDim;
#pragma unroll
    for (int hs = 0; hs < 4; ++hs) {
      const int h = hs ^ jj;
      const uint4 lo = *reinterpret_cast<const uint4*>(qb + h * kHeadDim + 8 * j);
      const uint4 hi = *reinterpret_cast<const uint4*>(qb + h * kHeadDim + 64 + 8 * j);
      unpack8(lo, &qf[hs][0]);
      unpack8(hi, &qf[hs][8]);
#pragma unroll
      for (int e = 0; e < 16; ++e) qf[hs][e] *= a.scale_log2;
    }
  }

  float acc[4][8];
#pragma unroll
  for (int h = 0; h < 4; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
  float m_run = -INFINITY;  // running max (base-2 logits) of head jj over this warp's tokens
  float l_run = 0.f;        // running sum of this lane's token's weights for head jj

  const int tq = warp * 4 + g;   // QK token in block
  const int t1 = warp * 4 + hf;  // PV tokens in block
  const int t2 = t1 + 2;
  bool ok = true;

  for (int it = 0; it < n_iter; ++it) {
    const int st = it % NS;
    if (!mbar_wait(&full_bar[st], (it / NS) & 1)) {
      ok = false;
      break;
    }
    const uint8_t* ks = stages + st * kStageBytes;
    const uint8_t* vs = ks + kTileBytes;
    const int tok0 = (b0 + it) * kBlockSize;

    // ---- scores: 4 heads x this lane's 16 dims of token tq ----
    float kf[16];
    unpack8(*reinterpret_cast<const uint4*>(ks + tq * kRowBytes + j * 16), &kf[0]);
    unpack8(*reinterpret_cast<const uint4*>(ks + tq * kRowBytes + 128 + j * 16), &kf[8]);
    float pd[4];
#pragma unroll
    for (int hs = 0; hs < 4; ++hs) {
      float x0 = 0.f, x1 = 0.f;
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        x0 = fmaf(qf[hs][e], kf[e], x0);
        x1 = fmaf(qf[hs][e + 1], kf[e + 1], x1);
      }
      pd[hs] = x0 + x1;
    }
    float s0 = pd[0] + __shfl_xor_sync(kFull, pd[2], 4);
    const float s1 = pd[1] + __shfl_xor_sync(kFull, pd[3], 4);
    s0 += __shfl_xor_sync(kFull, s1, 2);
    s0 += __shfl_xor_sync(kFull, s0, 1);
    const float s = (tok0 + tq < n_vis) ? s0 : -INFINITY;

    // ---- online softmax (per head jj, over the warp's 4 tokens) ----
    float mb = fmaxf(s, __shfl_xor_sync(kFull, s, 8));
    mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 16));
    const float m_new = fmaxf(m_run, mb);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float p = exp2_approx(s - m_use);
    const float alpha = exp2_approx(m_run - m_use);
    l_run = fmaf(l_run, alpha, p);
    m_run = m_new;
    float* pbuf = p_s + (it & 1) * (kConsumerWarps * 16) + warp * 16;
    if ((j & 1) == 0) pbuf[g * 4 + jj] = p;
    if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float al = __shfl_sync(kFull, alpha, 2 * h);  // lane 2h holds head h
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] *= al;
      }
    }
    __syncwarp();

    // ---- weighted values ----
    const float4 pa = *reinterpret_cast<const float4*>(pbuf + hf * 4);
    const float4 pb = *reinterpret_cast<const float4*>(pbuf + (hf + 2) * 4);
    uint4 va = *reinterpret_cast<const uint4*>(vs + t1 * kRowBytes + c * 16);
    uint4 vb = *reinterpret_cast<const uint4*>(vs + t2 * kRowBytes + c * 16);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[st]);  // this warp is done with the stage
    // slots past the context may hold anything (even NaN patterns): never let them in
    if (tok0 + t1 >= n_vis) va = make_uint4(0, 0, 0, 0);
    if (tok0 + t2 >= n_vis) vb = make_uint4(0, 0, 0, 0);
    float fa[8], fb[8];
    unpack8(va, fa);
    unpack8(vb, fb);
    const float wa[4] = {pa.x, pa.y, pa.z, pa.w};
    const float wb[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(wb[h], fb[e], fmaf(wa[h], fa[e], acc[h][e]));
  }
  if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);

  // ---- merge: lanes, then warps ----
  float l_tot = l_run + __shfl_xor_sync(kFull, l_run, 8);
  l_tot += __shfl_xor_sync(kFull, l_tot, 16);
#pragma unroll
  for (int h = 0; h < 4; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(kFull, acc[h][e], 16);

  named_barrier_sync(1, kConsumerWarps * 32);  // all consumer warps are done with the stages
  float* acc_s = reinterpret_cast<float*>(stages);  // [4 warps][4 heads][128]
  if (hf == 0) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float4* dst = reinterpret_cast<float4*>(acc_s + (warp * 4 + h) * kHeadDim + 8 * c);
      dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
    }
  }
  if (g == 0 && (j & 1) == 0) {
    m_s[warp * 4 + jj] = m_run;
    l_s[warp * 4 + jj] = l_tot;
  }
  named_barrier_sync(1, kConsumerWarps * 32);

  const int h = threadIdx.x >> 5;  // 0..3
  const int d0 = lane * 4;
  float mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, m_s[w * 4 + h]);
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  float sum = 0.f;
  if (mx != -INFINITY) {
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float sc = exp2_approx(m_s[w * 4 + h] - mx);
      sum = fmaf(l_s[w * 4 + h], sc, sum);
      const float4 v = *reinterpret_cast<const float4*>(acc_s + (w * 4 + h) * kHeadDim + d0);
      o[0] = fmaf(v.x, sc, o[0]);
      o[1] = fmaf(v.y, sc, o[1]);
      o[2] = fmaf(v.z, sc, o[2]);
      o[3] = fmaf(v.w, sc, o[3]);
    }
    const float inv = 1.f / sum;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] *= inv;
  }
  const int64_t orow = qrow0 + h;
  if (a.num_splits == 1) {
    uint2 packed;
    packed.x = pack_bf16x2(o[0], o[1]);
    packed.y = pack_bf16x2(o[2], o[3]);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + orow * kHeadDim + d0) = packed;
  } else {
    *reinterpret_cast<float4*>(a.part_o + (orow * a.num_splits + split) * kHeadDim + d0) =
        make_float4(o[0], o[1], o[2], o[3]);
    if (lane == 0)
      a.part_lse[orow * a.num_splits + split] = (mx == -INFINITY) ? -INFINITY : (mx + log2f(sum)) * kLn2;
  }
}

constexpr int kStages = 4;

}  // namespace

cudaError_t launch_paged_decode(const DecodeArgs& a, cudaStream_t stream) {
  using L = DecodeSmem<kStages>;
  const dim3 grid(static_cast<unsigned>(a.num_seqs * a.q_len), static_cast<unsigned>(a.num_splits),
                  static_cast<unsigned>(a.num_kv_heads));
  if (grid.x == 0) return cudaSuccess;
  static_assert(L::kBytes <= 48 * 1024, "raise the dynamic shared memory limit first");
  paged_decode_kernel<kStages><<<grid, kThreads, L::kBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv
