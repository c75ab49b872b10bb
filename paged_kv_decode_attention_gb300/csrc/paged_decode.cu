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
//              each, contiguous in the cache layout) into a ring of NS
//              shared-memory stages with cp.async.bulk, completion counted on
//              a per-stage "full" mbarrier; block ids are fetched 32 at a time
//              by the whole warp.  A stage is refilled once its consumer warp
//              has arrived on its "empty" mbarrier.
//   consumers: warp w reduces whole blocks w, w+4, w+8, ... and keeps its own
//              running max / sum / accumulator for all 4 query heads of the
//              GQA group, so each KV tile is read from HBM once per group and
//              the per-block fixed costs (wait, reductions, exp, weight
//              exchange) are paid once per 16 tokens.
//   QK^T     : lanes (g = lane/8, j = lane%8) take tokens g, g+4, g+8, g+12
//              and dims 8j..8j+7, 64+8j..64+8j+7 (conflict-free 16-byte shared
//              loads), with the matching query slices of all 4 heads in
//              registers (FP32, pre-scaled by scale*log2 e); products use
//              packed FP32x2 FMAs.  The 16 partial dot products per lane
//              reduce-scatter over the 8 lanes in 14 shuffles; lane-dependent
//              head and token orders make every step select-free, and lane
//              (g, j) ends with head j/2's scores for two tokens.
//   softmax  : base-2, FP32; block maximum per head by 3 shuffles; the
//              accumulators are rescaled only when some running max moved.
//   PV       : lanes (hf = lane/16, c = lane%16) take tokens hf, hf+2, ...,
//              hf+14 and dims 8c..8c+7, FP32x2 accumulators for the 4 heads;
//              the weights go through a per-warp shared buffer (broadcast).
//   merge    : the 4 warps' (max, sum, acc) are merged through shared memory.
// Split modes (chosen on the host):
//   kDirect    one split: write BF16 directly;
//   kCluster   2..8 splits launched as one thread-block cluster per
//              (row, KV head): every CTA leaves its (max, sum, acc) in its
//              shared memory and CTA 0 of the cluster merges them through
//              distributed shared memory and writes BF16 -- no workspace, no
//              second kernel;
//   kWorkspace more splits: each writes its normalised FP32 output and
//              natural-log lse to the workspace for the combine kernel.
#include <climits>
#include <cmath>

#include "pkv_common.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

// Pipeline depth (8 KiB per stage) and the CTAs per SM the register budget
// targets; compile-time knobs so the depth can be swept.
#ifndef PKV_DECODE_STAGES
#define PKV_DECODE_STAGES 12
#endif
#ifndef PKV_DECODE_MIN_CTAS
#define PKV_DECODE_MIN_CTAS 2
#endif

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageBytes = 2 * kTileBytes;  // K tile, then V tile
constexpr int kRowBytes = kHeadDim * 2;      // one token of one head: 256 B
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kFull = 0xffffffffu;

enum class SplitMode { kDirect, kCluster, kWorkspace };

template <int NS>
struct DecodeSmem {
  // Every use of a stage must go to the same consumer warp (stage st belongs
  // to warp st % 4): with another stage count a fast warp could wait for a
  // stage's phase k+2 while phase k+1 is still in flight, and a parity wait
  // cannot tell those phases apart.
  static_assert(NS % kConsumerWarps == 0, "stage count must be a multiple of the consumer warps");
  static constexpr int kBarOffset = NS * kStageBytes;
  static constexpr int kPOffset = kBarOffset + 2 * NS * 8;                 // float [4 warps][16 tok][4 heads]
  static constexpr int kMOffset = kPOffset + kConsumerWarps * 64 * 4;      // float [4 warps][4 heads]
  static constexpr int kLOffset = kMOffset + kConsumerWarps * 4 * 4;
  static constexpr int kCtaOOffset = kLOffset + kConsumerWarps * 4 * 4;    // float [4 heads][128]
  static constexpr int kCtaMOffset = kCtaOOffset + kGroup * kHeadDim * 4;  // float [4]
  static constexpr int kCtaLOffset = kCtaMOffset + kGroup * 4;             // float [4]
  static constexpr int kBytes = kCtaLOffset + kGroup * 4;
  static_assert(NS * kStageBytes >= kConsumerWarps * kGroup * kHeadDim * 4, "epilogue scratch");
};

__device__ __forceinline__ void unpack8x2(const uint4 v, float2* f) {
  f[0] = bf16x2_to_float2(v.x);
  f[1] = bf16x2_to_float2(v.y);
  f[2] = bf16x2_to_float2(v.z);
  f[3] = bf16x2_to_float2(v.w);
}

constexpr float kLog2eF = 1.4426950408889634f;

// The cascade prefix pass's partials of one output row, folded into a
// running (max in base-2 logits, weight sum, un-normalised dims d0..d0+3).  A
// partial (normalised O_s, natural-log lse_s) is a block of total weight 1 at
// the base-2 logit lse_s * log2 e.  The slots are read kPrefixChunk at a time
// with every load issued before the first is used.
constexpr int kPrefixChunk = 8;

__device__ __forceinline__ void load_prefix_chunk(const DecodeArgs& a, int64_t orow, int d0, int s0, float* ls,
                                                  float4* v) {
  const int ns = a.prefix_slots;
  const float* lse = a.prefix_lse + orow * ns;
  const float* po = a.prefix_o + orow * ns * kHeadDim + d0;
#pragma unroll
  for (int k = 0; k < kPrefixChunk; ++k) {
    const int sl = s0 + k;
    ls[k] = sl < ns ? lse[sl] * kLog2eF : -INFINITY;
    v[k] = sl < ns ? *reinterpret_cast<const float4*>(po + sl * kHeadDim) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__device__ __forceinline__ void fold_prefix_chunk(const float* ls, const float4* v, float& mx, float& sum,
                                                  float* o) {
  float m2 = mx;
#pragma unroll
  for (int k = 0; k < kPrefixChunk; ++k) m2 = fmaxf(m2, ls[k]);
  if (m2 == -INFINITY) return;
  const float sc_old = exp2_approx(mx - m2);  // 0 when nothing was accumulated yet
  sum *= sc_old;
#pragma unroll
  for (int e = 0; e < 4; ++e) o[e] *= sc_old;
#pragma unroll
  for (int k = 0; k < kPrefixChunk; ++k) {
    if (ls[k] == -INFINITY) continue;  // an empty prefix split: its output is never used
    const float w = exp2_approx(ls[k] - m2);
    sum += w;
    o[0] = fmaf(w, v[k].x, o[0]);
    o[1] = fmaf(w, v[k].y, o[1]);
    o[2] = fmaf(w, v[k].z, o[2]);
    o[3] = fmaf(w, v[k].w, o[3]);
  }
  mx = m2;
}

// Slots s_first.. of the row (all of them by default).
__device__ __forceinline__ void fold_prefix(const DecodeArgs& a, int64_t orow, int d0, float& mx, float& sum,
                                            float* o, int s_first = 0) {
  for (int s0 = s_first; s0 < a.prefix_slots; s0 += kPrefixChunk) {
    float ls[kPrefixChunk];
    float4 v[kPrefixChunk];
    load_prefix_chunk(a, orow, d0, s0, ls, v);
    fold_prefix_chunk(ls, v, mx, sum, o);
  }
}

template <int NS, SplitMode kMode>
__device__ __forceinline__ void paged_decode_body(const DecodeArgs& a) {
  using L = DecodeSmem<NS>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty_bar = full_bar + NS;
  float* p_s = reinterpret_cast<float*>(smem + L::kPOffset);
  float* m_s = reinterpret_cast<float*>(smem + L::kMOffset);
  float* l_s = reinterpret_cast<float*>(smem + L::kLOffset);
  float* cta_o = reinterpret_cast<float*>(smem + L::kCtaOOffset);
  float* cta_m = reinterpret_cast<float*>(smem + L::kCtaMOffset);
  float* cta_l = reinterpret_cast<float*>(smem + L::kCtaLOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int vrow = blockIdx.x;  // r * q_len + i
  const int split = blockIdx.y;
  const int kvh = blockIdx.z;
  const int r = vrow / a.q_len;
  const int i = vrow - r * a.q_len;
  const int hq = a.num_kv_heads * kGroup;

  const int start = a.seq_start_block ? a.seq_start_block[r] : 0;  // blocks before it are reduced elsewhere
  // The producer's first 32 block ids, loaded before the context length is
  // known (the load stays inside the table row; ids past the range are dropped
  // below), so the first copies do not wait for two dependent loads.
  int first_ids = 0;
  if (warp == kConsumerWarps)
    first_ids = a.block_tables[static_cast<int64_t>(r) * a.max_blocks +
                               max(0, min(start + split * a.blocks_per_split + lane, a.max_blocks - 1))];
  const int ctx = a.context_lens[r];
  int n_vis = ctx - a.q_len + 1 + i;  // keys visible to query i
  if (n_vis > a.max_blocks * kBlockSize) {
    if (threadIdx.x == 0 && split == 0 && kvh == 0) report(a.err, PKV_DEVERR_CONTEXT);
    n_vis = a.max_blocks * kBlockSize;
  }
  if (ctx <= 0 || n_vis < 0) n_vis = 0;
  const int nb = (n_vis + kBlockSize - 1) / kBlockSize;
  const int b0 = start + split * a.blocks_per_split;
  const int b1 = min(nb, b0 + a.blocks_per_split);
  const int64_t qrow0 = static_cast<int64_t>(vrow) * hq + kvh * kGroup;  // (r, i, first head of group)
  const bool empty = b0 >= b1;
  // Fused append (q_len 1): the iteration of this CTA whose block holds the
  // new token (position ctx - 1), or -1 when another CTA holds it or the
  // token is not stored.
  int new_it = -1;
  int64_t new_slot = -1;
  if (a.k_new != nullptr && ctx > 0 && ctx <= a.max_blocks * kBlockSize) {
    const int nbl = (ctx - 1) / kBlockSize;
    if (nbl >= b0 && nbl < b1) {
      new_slot = a.slot_mapping[r];
      if (new_slot >= 0) new_it = nbl - b0;
    } else if (nbl < start && split == 0 && kvh == 0 && threadIdx.x == 0 && a.slot_mapping[r] >= 0) {
      // a new token inside a shared prefix (cascade): appending into a block
      // other requests read is not allowed; it is not stored
      report(a.err, PKV_DEVERR_SLOT);
    }
  } else if (a.k_new != nullptr && ctx <= 0 && split == 0 && kvh == 0 && threadIdx.x == 0 &&
             a.slot_mapping[r] >= 0) {
    // a stored token needs a position ctx - 1 >= 0: a slot for an empty row is
    // a caller error and the token is not stored (a context beyond the table
    // is reported above as PKV_DEVERR_CONTEXT and its token not stored either)
    report(a.err, PKV_DEVERR_SLOT);
  }

  const bool has_prefix = a.prefix_o != nullptr && start > 0;
  if (empty) {  // nothing to read: padding row, query without keys, or a split past the context
    if constexpr (kMode == SplitMode::kDirect) {
      if (has_prefix) {
        // the whole context lies in the shared prefix: the result is the prefix pass's
        if (threadIdx.x < kGroup * 32) {
          const int hh = threadIdx.x >> 5, dd = (threadIdx.x & 31) * 4;
          float mx = -INFINITY, sum = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
          pdl_wait();
          fold_prefix(a, qrow0 + hh, dd, mx, sum, o);
          const float inv = sum > 0.f ? 1.f / sum : 0.f;
          uint2 packed;
          packed.x = pack_bf16x2(o[0] * inv, o[1] * inv);
          packed.y = pack_bf16x2(o[2] * inv, o[3] * inv);
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + (qrow0 + hh) * kHeadDim + dd) = packed;
        }
        return;
      }
      if (threadIdx.x < kGroup * kRowBytes / 16)
        reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + qrow0 * kHeadDim)[threadIdx.x] =
            make_uint4(0, 0, 0, 0);
      return;
    } else if constexpr (kMode == SplitMode::kWorkspace) {
      if (threadIdx.x < kGroup) {
        a.part_lse[(qrow0 + threadIdx.x) * a.part_slots + a.part_slot0 + split] = -INFINITY;
        if (split == 0 && start == 0)
          for (int sl = 0; sl < a.part_slot0; ++sl) a.part_lse[(qrow0 + threadIdx.x) * a.part_slots + sl] = -INFINITY;
      }
      return;
    } else {
      // cluster mode: an empty partial still takes part in the cluster merge
      if (threadIdx.x < kGroup) {
        cta_m[threadIdx.x] = -INFINITY;
        cta_l[threadIdx.x] = 0.f;
      }
    }
  } else {
    const int n_iter = b1 - b0;
    if (threadIdx.x == 0) {
      for (int s = 0; s < NS; ++s) {
        mbar_init(&full_bar[s], 1);
        mbar_init(&empty_bar[s], 1);
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
      // block ids of a 32-block chunk, one per lane (INT_MIN past the range);
      // validated only when the chunk is used (a bad id reads block 0), so the
      // load of the next chunk stays in flight while this one streams
      auto chunk = [&](int base) -> int { return base + lane < n_iter ? table[base + lane] : INT_MIN; };
      auto checked = [&](int b) -> int {
        if (b != INT_MIN && (b < 0 || b >= a.num_blocks)) {
          report(a.err, PKV_DEVERR_BLOCK_ID);
          b = 0;
        }
        return b;
      };
      int blk_next = lane < n_iter ? first_ids : INT_MIN;  // chunk(0), loaded at the top
      for (int base = 0; base < n_iter && ok; base += 32) {
        const int blk = checked(blk_next);
        blk_next = chunk(base + 32);  // the next chunk's ids, read while this one streams
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
      // Cascade: with every copy issued, this warp waits for the prefix pass
      // and pulls the row's prefix partials into L1, so that the merge at the
      // end (in the CTA that merges) finds them there instead of in L2.
      if (has_prefix && (kMode == SplitMode::kDirect || (kMode == SplitMode::kCluster && cluster_cta_rank() == 0))) {
        pdl_wait();
        const char* po = reinterpret_cast<const char*>(a.prefix_o + qrow0 * a.prefix_slots * kHeadDim);
        const int bytes = kGroup * a.prefix_slots * kHeadDim * static_cast<int>(sizeof(float));
        for (int off = lane * 128; off < bytes; off += 32 * 128) prefetch_l1(po + off);
        if (lane == 0) prefetch_l1(a.prefix_lse + qrow0 * a.prefix_slots);
      }
      if (lane == 0) {
        if (!ok) report(a.err, PKV_DEVERR_TIMEOUT);
        // every issued copy must land before the CTA's shared memory is released
        for (int it = max(0, issued - NS); it < issued; ++it) mbar_wait(&full_bar[it % NS], (it / NS) & 1);
      }
    } else {
      // ------------------------------ consumers ------------------------------
      // Warp w reduces blocks w, w+4, w+8, ... of the range (stage it % NS).
      const int g = lane >> 3;   // QK: token group (tokens g, g+4, g+8, g+12)
      const int j = lane & 7;    // QK: dim slice
      const int jj = j >> 1;     // QK: head whose scores this lane ends with
      const int tb = j & 1;      // QK: which token pair this lane ends with
      const int hf = lane >> 4;  // PV: token parity (tokens hf, hf+2, ..., hf+14)
      const int c = lane & 15;   // PV: dim slice

      // Query slices as FP32 pairs: slot hs = head (hs ^ jj), dims 8j..8j+7 then 64+8j..64+8j+7.
      float2 qf[4][8];
      {
        const uint16_t* qb = static_cast<const uint16_t*>(a.q) + qrow0 * kHeadDim;
        const float2 sc = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll
        for (int hs = 0; hs < 4; ++hs) {
          const int h = hs ^ jj;
          unpack8x2(*reinterpret_cast<const uint4*>(qb + h * kHeadDim + 8 * j), &qf[hs][0]);
          unpack8x2(*reinterpret_cast<const uint4*>(qb + h * kHeadDim + 64 + 8 * j), &qf[hs][4]);
#pragma unroll
          for (int e = 0; e < 8; ++e) qf[hs][e] = __fmul2_rn(qf[hs][e], sc);
        }
      }

      float2 acc[4][4];  // head h, dims 8c+2e, 8c+2e+1
#pragma unroll
      for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = make_float2(0.f, 0.f);
      float m_run = -INFINITY;  // running max (base-2 logits) of head jj over this warp's blocks
      float l_run = 0.f;        // running sum of the weights of this lane's tokens for head jj
      float* pbuf = p_s + warp * (kBlockSize * 4);  // this warp's weights [16 tokens][4 heads]
      // tokens whose final scores this lane holds after the reduction
      const int tk0 = g + 8 * tb;
      const int tk1 = tk0 + 4;
      bool ok = true;

      // Fused append: the warp that reduces the new token's block stores the
      // token's K/V row (8 bytes per lane) into the pools, where the append
      // would, and patches it into the block's tile once that has landed --
      // the copy may have read the slot before or after the store.
      bool patch = false;
      int new_off = 0;
      uint2 kn8 = make_uint2(0, 0), vn8 = make_uint2(0, 0);
      if (new_it >= 0 && new_it % kConsumerWarps == warp) {
        new_off = (ctx - 1) % kBlockSize;
        const int pb = a.block_tables[static_cast<int64_t>(r) * a.max_blocks + b0 + new_it];
        const int64_t row = static_cast<int64_t>(r) * a.num_kv_heads + kvh;  // token r, KV head kvh
        kn8 = reinterpret_cast<const uint2*>(a.k_new)[row * (kRowBytes / 8) + lane];
        vn8 = reinterpret_cast<const uint2*>(a.v_new)[row * (kRowBytes / 8) + lane];
        const int64_t pool_slots = static_cast<int64_t>(a.num_blocks) * kBlockSize;
        if (new_slot < pool_slots) {
          const size_t off = (static_cast<size_t>(new_slot / kBlockSize) * a.num_kv_heads + kvh) * kTileBytes +
                             static_cast<size_t>(new_slot % kBlockSize) * kRowBytes + lane * 8;
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(const_cast<void*>(a.k_cache)) + off) = kn8;
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(const_cast<void*>(a.v_cache)) + off) = vn8;
        }
        // the slot must be the one the table gives position ctx - 1
        patch = new_slot == static_cast<int64_t>(pb) * kBlockSize + new_off;
        if (!patch && lane == 0) report(a.err, PKV_DEVERR_SLOT);
      }

      for (int it = warp; it < n_iter; it += kConsumerWarps) {
        const int st = it % NS;
        if (!mbar_wait(&full_bar[st], (it / NS) & 1)) {
          ok = false;
          break;
        }
        if (patch && it == new_it) {
          uint8_t* kw = stages + st * kStageBytes + new_off * kRowBytes + lane * 8;
          *reinterpret_cast<uint2*>(kw) = kn8;
          *reinterpret_cast<uint2*>(kw + kTileBytes) = vn8;
          fence_proxy_async_shared();  // the stage is refilled by a bulk copy later
          __syncwarp();
        }
        const uint8_t* ks = stages + st * kStageBytes;
        const uint8_t* vs = ks + kTileBytes;
        const int tok0 = (b0 + it) * kBlockSize;

        // ---- scores: slot u holds token g + 4*(u ^ 2tb); 4 heads x this lane's 16 dims ----
        float sc4[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = g + 4 * (u ^ (2 * tb));
          float2 kf[8];
          unpack8x2(*reinterpret_cast<const uint4*>(ks + t * kRowBytes + j * 16), &kf[0]);
          unpack8x2(*reinterpret_cast<const uint4*>(ks + t * kRowBytes + 128 + j * 16), &kf[4]);
#pragma unroll
          for (int hs = 0; hs < 4; ++hs) {
            float2 x = __fmul2_rn(qf[hs][0], kf[0]);
#pragma unroll
            for (int e = 1; e < 8; ++e) x = __ffma2_rn(qf[hs][e], kf[e], x);
            sc4[u][hs] = x.x + x.y;
          }
        }
        // reduce-scatter over the 8 lanes of the group: heads by lane bits 2 and 1,
        // token pairs by lane bit 0 (slot orders above make every step select-free)
        float r2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float a0 = sc4[u][0] + __shfl_xor_sync(kFull, sc4[u][2], 4);
          const float a1 = sc4[u][1] + __shfl_xor_sync(kFull, sc4[u][3], 4);
          r2[u] = a0 + __shfl_xor_sync(kFull, a1, 2);
        }
        float s0 = r2[0] + __shfl_xor_sync(kFull, r2[2], 1);  // token tk0, head jj
        float s1 = r2[1] + __shfl_xor_sync(kFull, r2[3], 1);  // token tk1, head jj
        if (tok0 + kBlockSize > n_vis) {
          if (tok0 + tk0 >= n_vis) s0 = -INFINITY;
          if (tok0 + tk1 >= n_vis) s1 = -INFINITY;
        }

        // ---- online softmax (head jj, this block's 16 tokens) ----
        float mb = fmaxf(s0, s1);
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 1));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 8));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 16));
        const float m_new = fmaxf(m_run, mb);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float p0 = exp2_approx(s0 - m_use);
        const float p1 = exp2_approx(s1 - m_use);
        const float alpha = exp2_approx(m_run - m_use);
        l_run = fmaf(l_run, alpha, p0 + p1);
        m_run = m_new;
        pbuf[tk0 * 4 + jj] = p0;
        pbuf[tk1 * 4 + jj] = p1;
        if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float al = __shfl_sync(kFull, alpha, 2 * h);  // lane 2h holds head h
            const float2 al2 = make_float2(al, al);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[h][e] = __fmul2_rn(acc[h][e], al2);
          }
        }
        __syncwarp();

        // ---- weighted values: tokens hf, hf+2, ..., dims 8c..8c+7 ----
        const bool tail = tok0 + kBlockSize > n_vis;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const int t = hf + 2 * v;
          const float4 pw = *reinterpret_cast<const float4*>(pbuf + t * 4);
          uint4 vv = *reinterpret_cast<const uint4*>(vs + t * kRowBytes + c * 16);
          // last block: slots past the context may hold anything (even NaN patterns)
          if (tail && tok0 + t >= n_vis) vv = make_uint4(0, 0, 0, 0);
          float2 fv[4];
          unpack8x2(vv, fv);
          const float w4[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float2 w2 = make_float2(w4[h], w4[h]);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[h][e] = __ffma2_rn(w2, fv[e], acc[h][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);  // this warp is done with the stage
      }
      if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);

      // ---- merge: lanes, then warps ----
      float l_tot = l_run + __shfl_xor_sync(kFull, l_run, 1);
      l_tot += __shfl_xor_sync(kFull, l_tot, 8);
      l_tot += __shfl_xor_sync(kFull, l_tot, 16);
#pragma unroll
      for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[h][e].x += __shfl_xor_sync(kFull, acc[h][e].x, 16);
          acc[h][e].y += __shfl_xor_sync(kFull, acc[h][e].y, 16);
        }

      named_barrier_sync(1, kConsumerWarps * 32);  // all consumer warps are done with the stages
      float* acc_s = reinterpret_cast<float*>(stages);  // [4 warps][4 heads][128]
      if (hf == 0) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float4* dst = reinterpret_cast<float4*>(acc_s + (warp * 4 + h) * kHeadDim + 8 * c);
          dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
          dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
        }
      }
      if (g == 0 && (j & 1) == 0) {
        m_s[warp * 4 + jj] = m_run;
        l_s[warp * 4 + jj] = l_tot;
      }
      named_barrier_sync(1, kConsumerWarps * 32);

      const int h = warp;  // 0..3
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
      }
      const int64_t orow = qrow0 + h;
      if constexpr (kMode == SplitMode::kCluster) {
        *reinterpret_cast<float4*>(cta_o + h * kHeadDim + d0) = make_float4(o[0], o[1], o[2], o[3]);
        if (lane == 0) {
          cta_m[h] = mx;
          cta_l[h] = sum;
        }
      } else {
        if constexpr (kMode == SplitMode::kDirect) {
          if (has_prefix) {
            pdl_wait();  // the prefix pass wrote these partials
            fold_prefix(a, orow, d0, mx, sum, o);
          }
        }
        const float inv = (mx != -INFINITY && sum > 0.f) ? 1.f / sum : 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] *= inv;
        if constexpr (kMode == SplitMode::kDirect) {
          uint2 packed;
          packed.x = pack_bf16x2(o[0], o[1]);
          packed.y = pack_bf16x2(o[2], o[3]);
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + orow * kHeadDim + d0) = packed;
        } else {
          const int64_t slot = orow * a.part_slots + a.part_slot0 + split;
          *reinterpret_cast<float4*>(a.part_o + slot * kHeadDim + d0) = make_float4(o[0], o[1], o[2], o[3]);
          if (lane == 0) {
            a.part_lse[slot] = (mx == -INFINITY) ? -INFINITY : (mx + log2f(sum)) * kLn2;
            if (split == 0 && start == 0)
              for (int sl = 0; sl < a.part_slot0; ++sl) a.part_lse[orow * a.part_slots + sl] = -INFINITY;
          }
        }
      }
    }
  }

  if constexpr (kMode == SplitMode::kCluster) {
    // The leader waits for the prefix pass and issues the loads of its first
    // partials before the cluster merge, so their latency overlaps the merge.
    const bool lead = cluster_cta_rank() == 0 && warp < kConsumerWarps;
    float pre_ls[kPrefixChunk];
    float4 pre_v[kPrefixChunk];
    if (has_prefix && lead) {
      pdl_wait();  // the prefix pass wrote these partials
      load_prefix_chunk(a, qrow0 + warp, lane * 4, 0, pre_ls, pre_v);
    }
    // every CTA of the cluster has left its (max, sum, acc) in shared memory
    cluster_sync_all();
    if (lead) {
      const int h = warp;
      const int d0 = lane * 4;
      const uint32_t nranks = gridDim.y;  // cluster = all splits of this (row, KV head)
      // every rank's (max, sum, O) read at once: one round trip over the cluster
      float mr[kMaxClusterSplits], lr[kMaxClusterSplits];
      float4 vr[kMaxClusterSplits];
#pragma unroll
      for (int rk = 0; rk < kMaxClusterSplits; ++rk) {
        if (rk < static_cast<int>(nranks)) {
          mr[rk] = ld_cluster_f32(map_shared_to_rank(cta_m + h, rk));
          lr[rk] = ld_cluster_f32(map_shared_to_rank(cta_l + h, rk));
          vr[rk] = ld_cluster_f32x4(map_shared_to_rank(cta_o + h * kHeadDim + d0, rk));
        } else {
          mr[rk] = -INFINITY;
          lr[rk] = 0.f;
          vr[rk] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int rk = 0; rk < kMaxClusterSplits; ++rk) mx = fmaxf(mx, mr[rk]);
      float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f, sum = 0.f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int rk = 0; rk < kMaxClusterSplits; ++rk) {
          if (mr[rk] == -INFINITY) continue;
          const float sc = exp2_approx(mr[rk] - mx);
          sum = fmaf(lr[rk], sc, sum);
          o0 = fmaf(vr[rk].x, sc, o0);
          o1 = fmaf(vr[rk].y, sc, o1);
          o2 = fmaf(vr[rk].z, sc, o2);
          o3 = fmaf(vr[rk].w, sc, o3);
        }
      }
      if (has_prefix) {
        float o4[4] = {o0, o1, o2, o3};
        fold_prefix_chunk(pre_ls, pre_v, mx, sum, o4);
        fold_prefix(a, qrow0 + h, d0, mx, sum, o4, kPrefixChunk);  // slots past the first chunk
        o0 = o4[0];
        o1 = o4[1];
        o2 = o4[2];
        o3 = o4[3];
      }
      const float inv = (mx != -INFINITY && sum > 0.f) ? 1.f / sum : 0.f;
      uint2 packed;
      packed.x = pack_bf16x2(o0 * inv, o1 * inv);
      packed.y = pack_bf16x2(o2 * inv, o3 * inv);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + (qrow0 + h) * kHeadDim + d0) = packed;
    }
    // keep every CTA's shared memory alive until CTA 0 has read it
    cluster_sync_all();
  }
}

template <int NS, SplitMode kMode>
__global__ void __launch_bounds__(kThreads, PKV_DECODE_MIN_CTAS) paged_decode_kernel(const DecodeArgs a) {
  if (!a.overlap_previous) pdl_wait();  // inputs come from earlier grids in the stream
  pdl_trigger();
  paged_decode_body<NS, kMode>(a);
  if (a.overlap_previous) pdl_wait();  // complete only after the grid it overlapped
}

constexpr int kStages = PKV_DECODE_STAGES;

// Opt the kernel in to more than 48 KiB of dynamic shared memory, once per
// device (function attributes are per device context).
template <SplitMode kMode>
cudaError_t allow_smem(int bytes) {
  static std::atomic<bool> done[64];  // per device; host threads may race on a first call
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    e = cudaFuncSetAttribute(paged_decode_kernel<kStages, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_paged_decode(const DecodeArgs& a, cudaStream_t stream) {
  using L = DecodeSmem<kStages>;
  static_assert(L::kBytes <= 113 * 1024, "two CTAs per SM must fit in shared memory");
  const dim3 grid(static_cast<unsigned>(a.num_seqs * a.q_len), static_cast<unsigned>(a.num_splits),
                  static_cast<unsigned>(a.num_kv_heads));
  if (grid.x == 0) return cudaSuccess;
  if (a.num_splits == 1) {
    cudaError_t e = allow_smem<SplitMode::kDirect>(L::kBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(paged_decode_kernel<kStages, SplitMode::kDirect>, grid, dim3(kThreads), L::kBytes, stream, 1,
                      a);
  }
  if (a.part_o == nullptr) {
    if (a.num_splits > kMaxClusterSplits) return cudaErrorInvalidValue;
    cudaError_t e = allow_smem<SplitMode::kCluster>(L::kBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(paged_decode_kernel<kStages, SplitMode::kCluster>, grid, dim3(kThreads), L::kBytes, stream,
                      static_cast<unsigned>(a.num_splits), a);
  }
  cudaError_t e = allow_smem<SplitMode::kWorkspace>(L::kBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(paged_decode_kernel<kStages, SplitMode::kWorkspace>, grid, dim3(kThreads), L::kBytes, stream, 1,
                    a);
}

cudaError_t launch_paged_decode_workspace(const DecodeArgs& a, cudaStream_t stream) {
  using L = DecodeSmem<kStages>;
  const dim3 grid(static_cast<unsigned>(a.num_seqs * a.q_len), static_cast<unsigned>(a.num_splits),
                  static_cast<unsigned>(a.num_kv_heads));
  if (grid.x == 0) return cudaSuccess;
  cudaError_t e = allow_smem<SplitMode::kWorkspace>(L::kBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(paged_decode_kernel<kStages, SplitMode::kWorkspace>, grid, dim3(kThreads), L::kBytes, stream, 1,
                    a);
}

}  // namespace pkv
