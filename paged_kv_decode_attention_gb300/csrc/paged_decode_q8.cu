// paged_decode_q8.cu -- decode attention over a q8_0 paged KV cache, with the dequantisation inside the kernel: Q.K^T on the
// 5th-generation tensor cores, P.V on the CUDA cores, side by side.
//
// What it computes ("Chapter 8: Inference Optimization",
// clxhxhhr.top/posts/4341): the decode step of §8.1.1 over the block tables
// of §8.3.1, with K and V stored in the q8_0 format of §8.4.2 / Fig. 8-23 --
// every 32 consecutive values of a token's head vector share one FP16 scale
// s and keep 8-bit codes c, value = s * c.  Reading 34 instead of 64 bytes
// per group pays only if the conversion costs less than the bytes saved
// (§8.4.2, dT = dD / beta - T_c).  With 4 query heads per KV head a token
// costs 2 x 512 multiply-adds against 272 bytes read; at HBM speed an SM has
// about 12 cycles per token.  The work is split between two units that run
// concurrently:
//
//   S^T = K_codes . Qbd^T  on tcgen05 (M = 128 tokens, N = 16, K = 128 dims,
//        8 instructions per 128 tokens, ~4.4 cycles per token).  Qbd is
//        block-diagonal: row n = 4g + h holds query head h on the 32 dims of
//        group g and zeros elsewhere, so column 4g + h of S^T is group g's part
//        of the dot product and the softmax applies each group's K scale in
//        FP32 -- the codes stay exact (int8 -> FP16) and no scale is rounded.
//   O += P' . V_codes      on the FP32 pipes (~4 cycles per token): P' = p * sV
//        per (token, head, group), codes converted exactly to FP32.
//
// CTA = 15 warps (17 with four producers), one per SM, persistent: it walks
// work units u = blockIdx.x, + gridDim.x, ... (a unit is one (request, KV
// head, split)).
//   producers (warps 0-1, or 0-3): per 128-token tile, a K producer copies 8
//              blocks' K tiles (2176 B each) into the K ring and a V producer
//              their V tiles into the V ring, the latter once the tile's K has
//              landed; one bulk copy per lane.
//   next warp: MMA issuer (one thread): QK(i) into a double-buffered S in
//              tensor memory.
//   next 8   : attention, two groups of four that take alternate tiles.  In
//              a group, warp w (TMEM sub-partition w) owns tokens 32w .. 32w+31
//              of its tiles (thread = token for S) and keeps its own
//              online-softmax state (max, sum, O for 4 heads x 128 dims, lane =
//              4 dims); the eight states merge once per unit (log-sum-exp), so
//              no tile needs a cross-warp exchange.  The weights are taken
//              against a maximum that moves only when a score exceeds it by
//              more than 2^8, so most tiles skip the warp-wide reduction.
//   last 4   : dequantisation of the ring's K codes into a double-buffered
//              FP16 operand tile (128-byte swizzled rows), the unit's Qbd, and
//              a copy of the tile's K scales for the softmax, so that a K stage
//              is free as soon as its codes are converted.
// The fused-append instance (kFused) adds one warp: per unit holding its
// request's new token it quantises the new K and V rows as kv_append_q8 does
// and stores them in the pools, and the producers issue the copy of that
// token's tile only after the rows are in place, so the tile carries them and
// no other role changes.
// Every wait is bounded (about 2 s) and reports PKV_DEVERR_TIMEOUT instead of
// hanging; the roles exchange data only through mbarriers.
#include <cmath>
#include <cuda_fp16.h>

#include "pkv_common.cuh"
#include "pkv_kernels.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

#ifndef PKV_Q8_K_STAGES
#define PKV_Q8_K_STAGES 4
#endif
#ifndef PKV_Q8_V_STAGES
#define PKV_Q8_V_STAGES 4
#endif
constexpr int kKStages = PKV_Q8_K_STAGES;
constexpr int kVStages = PKV_Q8_V_STAGES;
#ifndef PKV_Q8_PRODUCERS
#define PKV_Q8_PRODUCERS 2
#endif
constexpr int kProducerWarps = PKV_Q8_PRODUCERS;  // half for the K ring, half for the V ring
constexpr int kPerRing = kProducerWarps / 2;     // warps per ring, taking tiles in turn
constexpr int kMmaWarp = kProducerWarps;
constexpr int kFirstAttnWarp = kMmaWarp + 1;
constexpr int kAttnWarps = 8;
constexpr int kFirstDqWarp = kFirstAttnWarp + kAttnWarps;
constexpr int kQ8Threads = (kFirstDqWarp + 4) * 32;
constexpr int kAppendWarp = kFirstDqWarp + 4;        // fused-append instance only
constexpr int kQ8ThreadsFused = kQ8Threads + 32;
constexpr int kReadySlots = 4;                       // fused append: units whose new rows are stored, a ring
constexpr int kQ8TileBlocks = 8;                               // blocks per 128-token tile
constexpr int kRawStageBytes = kQ8TileBlocks * kQ8TileBytes;   // 8 K (or V) tiles: 17408
constexpr int kOpHalfBytes = 128 * 128;                        // 128 rows x 64 FP16 values
constexpr int kOffKd = 0;                                      // K codes x 2, FP16 [128 tok][128 d]
constexpr int kOffQbd = kOffKd + 2 * 2 * kOpHalfBytes;         // Qbd, FP16 [16][128 d]
constexpr int kOffP = kOffQbd + 4096;                          // P' per attention warp: [32 tok][16] FP32
constexpr int kOffMl = kOffP + kAttnWarps * 2048;              // unit merge: max, sum [8 warps][4 heads]
constexpr int kScaleSlots = 4;                                 // K scales of a tile, for the softmax
constexpr int kOffSk = kOffMl + 2 * kAttnWarps * 4 * 4;        // [slot][128 tokens][4] FP16
constexpr int kOffRawK = kOffSk + kScaleSlots * 1024;          // K ring
constexpr int kOffRawV = kOffRawK + kKStages * kRawStageBytes;  // V ring
constexpr int kOffBarQ8 = kOffRawV + kVStages * kRawStageBytes;
constexpr int kSmemQ8 = kOffBarQ8 + 512;
static_assert(kSmemQ8 <= 227 * 1024, "shared memory per CTA");
static_assert(kOffRawK % 16 == 0 && kOffQbd % 1024 == 0 && kOffP % 16 == 0, "alignment");
constexpr uint32_t kTmemColsQ8 = 32;  // S buffers at columns 0 and 16
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazyMax = 8.f;  // log2 units: weights stay below 2^8 (FP32 throughout)

struct Q8Bars {
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t kd_full[2], kd_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t sk_full[kScaleSlots];
  uint64_t merge[2];
  uint64_t ready[kReadySlots], ready_empty[kReadySlots];  // fused append: a unit's new rows are in the pools
  uint32_t tmem_base;
};
static_assert(sizeof(Q8Bars) <= 512, "barrier area");

// One (request, KV head, split) of the launch; with the append fused in,
// also where the request's new token (position ctx - 1) falls: its tile of
// the unit and its logical block (new_tile -1 when another unit holds it).
struct Unit {
  int r, kvh, split, b0, b1, n_tiles, ctx_keys, ctx_raw;
  int new_tile, new_blk;
};

template <bool kFused = false>
__device__ __forceinline__ Unit unit_at(const DecodeArgs& a, int u) {
  Unit x;
  x.split = u % a.num_splits;
  const int row = u / a.num_splits;
  x.r = row / a.num_kv_heads;
  x.kvh = row - x.r * a.num_kv_heads;
  x.ctx_raw = a.context_lens[x.r];
  const int ctx = min(max(x.ctx_raw, 0), a.max_blocks * kBlockSize);
  const int nb = (ctx + kBlockSize - 1) / kBlockSize;
  x.b0 = x.split * a.blocks_per_split;
  x.b1 = min(nb, x.b0 + a.blocks_per_split);
  x.n_tiles = x.b1 > x.b0 ? (x.b1 - x.b0 + kQ8TileBlocks - 1) / kQ8TileBlocks : 0;
  x.ctx_keys = min(ctx, x.b1 * kBlockSize);
  x.new_tile = -1;
  x.new_blk = 0;
  if (kFused && x.ctx_raw > 0 && x.ctx_raw <= a.max_blocks * kBlockSize) {
    const int nbl = (x.ctx_raw - 1) / kBlockSize;
    if (nbl >= x.b0 && nbl < x.b1) {
      x.new_tile = (nbl - x.b0) / kQ8TileBlocks;
      x.new_blk = nbl;
    }
  }
  return x;
}

// Fused append: one warp stores its quantised row (lane l: codes of values
// 4l .. 4l+3; lanes 8g: group g's scale) at `slot` of one pool, as
// kv_append_q8 does; a slot outside the pool (or negative) stores nothing.
__device__ __forceinline__ void q8_store_row(const DecodeArgs& a, const void* cache, int64_t slot, int kvh,
                                             uint32_t codes, float d, int lane) {
  if (slot < 0 || slot >= static_cast<int64_t>(a.num_blocks) * kBlockSize) return;
  uint8_t* tile = static_cast<uint8_t*>(const_cast<void*>(cache)) +
                  ((slot / kBlockSize) * a.num_kv_heads + kvh) * static_cast<int64_t>(kQ8TileBytes);
  const int off = static_cast<int>(slot % kBlockSize);
  *reinterpret_cast<uint32_t*>(tile + off * kHeadDim + lane * 4) = codes;
  if ((lane & 7) == 0) *reinterpret_cast<__half*>(tile + kQ8CodeBytes + (off * 4 + (lane >> 3)) * 2) = __float2half_rn(d);
}

// Power-of-two shift e that brings the group's largest |q| below 2^15, so
// q * 2^-e converts to FP16 without overflow (exactly, for BF16 inputs in
// the normal range); 0 for any ordinary query.
__device__ __forceinline__ int q_shift(float amax) {
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;
  return e >= 15 ? e - 14 : 0;
}

__device__ __forceinline__ float pow2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// max |q| over the unit's 4 query heads x 128 dims (512 contiguous BF16),
// computed by one warp on its own.
__device__ __forceinline__ float group_q_absmax(const uint16_t* qg, int lane) {
  const uint4 a = reinterpret_cast<const uint4*>(qg)[lane];
  const uint4 b = reinterpret_cast<const uint4*>(qg)[lane + 32];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  return m;
}

// 8 int8 codes -> 8 FP16 values (exact): the biased byte c + 128 becomes the
// low mantissa byte of 1024 + (c + 128), then 1152 is subtracted.
__device__ __forceinline__ uint4 codes_to_f16(uint2 w) {
  const uint32_t a = w.x ^ 0x80808080u;
  const uint32_t b = w.y ^ 0x80808080u;
  constexpr uint32_t kMagic = 0x64646464u;
  uint32_t h[4] = {__byte_perm(a, kMagic, 0x4140), __byte_perm(a, kMagic, 0x4342), __byte_perm(b, kMagic, 0x4140),
                   __byte_perm(b, kMagic, 0x4342)};
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h[i]) : "r"(0x64806480u));
  return make_uint4(h[0], h[1], h[2], h[3]);
}

// 4 int8 codes -> 4 FP32 values (exact): c + 128 as the low mantissa byte of
// 2^23 + (c + 128), then 2^23 + 128 is subtracted.
__device__ __forceinline__ void codes_to_f32(uint32_t w, float2& c01, float2& c23) {
  const uint32_t x = w ^ 0x80808080u;
  constexpr uint32_t kMagic = 0x4B000000u;
  const float2 bias = make_float2(-8388736.f, -8388736.f);
  c01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, kMagic, 0x7650)),
                               __uint_as_float(__byte_perm(x, kMagic, 0x7651))), bias);
  c23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, kMagic, 0x7652)),
                               __uint_as_float(__byte_perm(x, kMagic, 0x7653))), bias);
}

__device__ __forceinline__ void half4_to_float(uint2 w, float* f) {
  const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
  const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
  f[0] = lo.x;
  f[1] = lo.y;
  f[2] = hi.x;
  f[3] = hi.y;
}

// P' of one warp: 32 tokens x 16 FP32 (4 groups x 4 heads); the 16-byte chunk
// of group q of token t sits at chunk position (q + t/2) % 4 of the token's
// 64-byte row, which keeps both the per-token writes and the per-group reads
// free of bank conflicts.
__device__ __forceinline__ uint32_t p_chunk(int t, int q) { return t * 64 + (((q + (t >> 1)) & 3) << 4); }

// Bounded wait on the CTA-wide unit-merge barrier (one arrival per attention warp).
__device__ __forceinline__ bool merge_sync(uint64_t* merge, uint32_t& n, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(&merge[n & 1]);
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&merge[n & 1], (n >> 1) & 1));
  ++n;
  return ok;
}

// q8_0 tiles: int8 codes + FP16 group scales, 2176 B per (block, KV head).
// kFused: the step's append fused in (a.k_new, a.v_new, a.slot_mapping set;
// token r is request r's new token), with one more warp; an instance of its
// own, so the plain decode carries none of it.
template <bool kFused>
__global__ void __launch_bounds__(kFused ? kQ8ThreadsFused : kQ8Threads, 1)
    paged_decode_q8_kernel(const DecodeArgs a) {
  static_assert(!kFused || kPerRing == 1, "the fused append's ready ring assumes one producer warp per ring");
  constexpr int kTile = kQ8TileBytes;
  pdl_trigger();
  extern __shared__ __align__(1024) uint8_t smem[];
  Q8Bars* bars = reinterpret_cast<Q8Bars*>(smem + kOffBarQ8);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_units = a.num_seqs * a.num_kv_heads * a.num_splits;
  const int hq = a.num_kv_heads * kGroup;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      // 128 dequant threads and the V producer (so no K stage is refilled
      // before the V producer has seen it land)
      mbar_init(&bars->k_empty[s], 128 + 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], kAttnWarps / 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->kd_full[s], 128);
      mbar_init(&bars->kd_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_empty[s], kAttnWarps / 2 * 32);
      mbar_init(&bars->merge[s], kAttnWarps);
    }
    for (int s = 0; s < kScaleSlots; ++s) mbar_init(&bars->sk_full[s], 128);
    for (int s = 0; s < kReadySlots; ++s) {
      mbar_init(&bars->ready[s], 32);                      // the append warp
      mbar_init(&bars->ready_empty[s], kProducerWarps);   // each producer warp, once it has waited
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&bars->tmem_base, kTmemColsQ8);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // The set-up above reads no input; everything below may read what earlier
  // grids in the stream write (e.g. this step's append), so wait for them here.
  pdl_wait();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t sbase = smem_addr(smem);
  bool ok = true;

  if (warp < kProducerWarps) {
    // ------------------------------ producers ------------------------------
    // Warp 0 copies each tile's 8 K tiles into the K ring; warp 1 copies its 8
    // V tiles into the V ring once the tile's K has landed, so that V arrives
    // about when the softmax needs it instead of occupying a stage for the
    // whole Q.K^T and softmax.  One copy per lane.  Block-table entries are
    // read 32 at a time (one per lane), one chunk ahead of use.
    const bool is_v = warp >= kPerRing;
    const int ppar = warp % kPerRing;  // this warp issues the tiles with i % kPerRing == ppar
    const int ns = is_v ? kVStages : kKStages;
    uint64_t* full = is_v ? bars->v_full : bars->k_full;
    uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
    uint8_t* ring = smem + (is_v ? kOffRawV : kOffRawK);
    const uint8_t* pool = static_cast<const uint8_t*>(is_v ? a.v_cache : a.k_cache);
    const uint64_t policy = l2_policy_evict_first();
    int i = 0;
    int nf = 0;  // units holding their request's new token so far (fused append)
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const Unit x = unit_at<kFused>(a, u);
      const int32_t* table = a.block_tables + static_cast<int64_t>(x.r) * a.max_blocks;
      // the load stays inside the table row whatever the context length, so it
      // need not wait for that length; entries past the unit's blocks are dropped
      auto entry = [&](int bi) -> int {
        const int raw = table[min(bi, a.max_blocks - 1)];
        return bi < x.b1 ? raw : 0;  // checked where used
      };
      int cur = entry(x.b0 + lane);
      int nxt = 0;
      for (int j = 0; j < x.n_tiles; ++j, ++i) {
        const int slot = j & 3;  // this tile's 8 entries in the current 32-entry chunk
        if (slot == 0) nxt = entry(x.b0 + j * kQ8TileBlocks + 32 + lane);  // the next chunk, read ahead
        int blk = __shfl_sync(0xffffffffu, cur, slot * kQ8TileBlocks + (lane & (kQ8TileBlocks - 1)));
        if (slot == 3) cur = nxt;
        if (i % kPerRing != ppar) continue;  // another warp's tile
        const int st = i % ns;
        const int nblk = min(kQ8TileBlocks, x.b1 - (x.b0 + j * kQ8TileBlocks));
        const bool copies = lane < nblk;
        if (copies && (blk < 0 || blk >= a.num_blocks)) {
          if (!is_v) report(a.err, PKV_DEVERR_BLOCK_ID);
          blk = 0;
        }
        if (lane == 0) {
          if (is_v) ok = mbar_wait(&bars->k_full[i % kKStages], (i / kKStages) & 1);  // K(i) landed
          if (ok && i >= ns) ok = mbar_wait(&empty[st], ((i / ns) & 1) ^ 1);
          if (kFused && ok && j == x.new_tile) {
            // fused append: the tile holding the new token is copied only once
            // the append warp has stored the new rows in the pools
            ok = mbar_wait(&bars->ready[nf % kReadySlots], (nf / kReadySlots) & 1);
            mbar_arrive(&bars->ready_empty[nf % kReadySlots]);
          }
          if (ok) mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(nblk) * kTile);
        }
        if (kFused && j == x.new_tile) ++nf;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (copies)
          bulk_copy_g2s(ring + st * kRawStageBytes + lane * kQ8TileBytes,
                        pool + (static_cast<int64_t>(blk) * a.num_kv_heads + x.kvh) * kTile, kTile,
                        &full[st], policy);
        __syncwarp();
        if (is_v && lane == 0) mbar_arrive(&bars->k_empty[i % kKStages]);
      }
    }
    if (lane == 0) {
      if (!ok) report(a.err, PKV_DEVERR_TIMEOUT);
      // no copy may still be landing when the CTA's shared memory is released
      for (int k = max(0, i - ns); k < i; ++k)
        if (k % kPerRing == ppar) mbar_wait(&full[k % ns], (k / ns) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_f16_f32(128, 16, false, false);
      int i = 0;
      const uint32_t qbd = sbase + kOffQbd;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const Unit x = unit_at(a, u);
        if (x.n_tiles == 0) continue;
        for (int j = 0; j < x.n_tiles; ++j, ++i) {
          const int b = i & 1;
          ok = mbar_wait(&bars->kd_full[b], (i >> 1) & 1);
          if (ok && i >= 2) ok = mbar_wait(&bars->s_empty[b], ((i - 2) >> 1) & 1);  // softmax(i-2) read S
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t kd = sbase + kOffKd + b * 2 * kOpHalfBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ka = kd + (kk >> 2) * kOpHalfBytes + 32 * (kk & 3);
            const uint32_t qa = qbd + (kk >> 2) * 2048 + 32 * (kk & 3);
            tc::mma_ss(tmem + b * 16, tc::smem_desc(ka, 16, 1024), tc::smem_desc(qa, 16, 1024), kIdS,
                       kk > 0 ? 1u : 0u);
          }
          tc::commit(&bars->s_full[b]);
          tc::commit(&bars->kd_empty[b]);
        }
      }
      if (!ok) report(a.err, PKV_DEVERR_TIMEOUT);
      // tensor memory is released only after the last MMA has finished
      if (i > 0) mbar_wait(&bars->kd_empty[(i - 1) & 1], ((i - 1) >> 1) & 1);
    }
    __syncwarp();
  } else if (warp < kFirstDqWarp) {
    // ------------------------------ attention ------------------------------
    const int aw = warp - kFirstAttnWarp;  // 0..7
    const int par = aw >> 2;           // this warp's tiles: i % 2 == par (it reads S buffer par)
    const int w = warp & 3;            // TMEM sub-partition: tokens 32w .. 32w+31 of a tile
    const int k = w * 32 + lane;       // this thread's token row of S
    const int g_own = lane >> 3;       // group of this lane's dims 4*lane .. 4*lane+3
    const uint32_t lane_off = static_cast<uint32_t>(w * 32) << 16;
    uint8_t* pw = smem + kOffP + aw * 2048;  // this warp's P' (and, at a unit's end, its O)
    float* ml = reinterpret_cast<float*>(smem + kOffMl);  // [max | sum][warp][head]
    // this thread's part of a unit's output: head aw % 4, dims (aw / 4) * 64 + 2*lane .. +1
    const int h_out = aw & 3;
    const int d_out = (aw >> 2) * 64 + 2 * lane;
    uint32_t nmerge = 0;
    int i = 0;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const Unit x = unit_at(a, u);
      const int64_t orow0 = static_cast<int64_t>(x.r) * hq + x.kvh * kGroup;
      if (threadIdx.x == kFirstAttnWarp * 32 && x.split == 0 && x.kvh == 0 && x.ctx_raw > a.max_blocks * kBlockSize)
        report(a.err, PKV_DEVERR_CONTEXT);
      // fused append: a slot for an empty row has no position ctx - 1 to go
      // to; the token is not stored and the caller's error is reported
      if (kFused && threadIdx.x == kFirstAttnWarp * 32 && x.split == 0 && x.kvh == 0 && x.ctx_raw <= 0 &&
          a.slot_mapping[x.r] >= 0)
        report(a.err, PKV_DEVERR_SLOT);
      const int64_t orow_out = orow0 + h_out;
      if (x.n_tiles == 0) {
        if (a.num_splits == 1)
          *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + orow_out * kHeadDim + d_out) = 0u;
        else if (lane == 0 && aw < 4)
          a.part_lse[orow_out * a.num_splits + x.split] = -INFINITY;
        continue;
      }
      const uint16_t* qg = static_cast<const uint16_t*>(a.q) + orow0 * kHeadDim;
      const float c0 = a.scale_log2 * pow2i(q_shift(group_q_absmax(qg, lane)));
      float m[4], l[4];
      float2 o[4][2];  // O[h][dims 4*lane + {0,1}], O[h][dims 4*lane + {2,3}]
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
        o[h][0] = o[h][1] = make_float2(0.f, 0.f);
      }
      for (int j = 0; j < x.n_tiles; ++j, ++i) {
        if ((i & 1) != par) continue;  // the other group's tile
        const int sb = par;
        const int vst = i % kVStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (i >> 1) & 1));
        if (!ok) break;
        tc::fence_after_sync();
        float s[16];  // column 4g + h: group g's part of head h's dot product
        tc::tmem_ld16(tmem + lane_off + sb * 16, s);
        tc::tmem_wait_ld();
        // this token's K scales, copied out of the K stage by the dequantisation;
        // read before S is released, which orders the read before the slot's reuse
        float sk[4] = {1.f, 1.f, 1.f, 1.f}, sv[4] = {1.f, 1.f, 1.f, 1.f};
        {
          const int sks = i % kScaleSlots;
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->sk_full[sks], (i / kScaleSlots) & 1));
          if (!ok) break;
          half4_to_float(*reinterpret_cast<const uint2*>(smem + kOffSk + sks * 1024 + k * 8), sk);
        }
        tc::fence_before_sync();
        mbar_arrive(&bars->s_empty[sb]);
        const uint8_t* rawv = smem + kOffRawV + vst * kRawStageBytes;
        const int so = (k >> 4) * kQ8TileBytes + kQ8CodeBytes + (k & 15) * 8;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->v_full[vst], (i / kVStages) & 1));
        if (!ok) break;
        half4_to_float(*reinterpret_cast<const uint2*>(rawv + so), sv);
        const bool valid = (x.b0 + j * kQ8TileBlocks) * kBlockSize + k < x.ctx_keys;
#pragma unroll
        for (int q = 0; q < 4; ++q) sv[q] = valid ? sv[q] : 0.f;  // a slot past the data may hold any bits
        float sc[4], alpha[4] = {1.f, 1.f, 1.f, 1.f};
        bool over = false;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float dot = sk[0] * s[h] + sk[1] * s[4 + h] + sk[2] * s[8 + h] + sk[3] * s[12 + h];
          sc[h] = valid ? c0 * dot : -INFINITY;
          over |= sc[h] > m[h] + kLazyMax || (m[h] == -INFINITY && valid);
        }
        const bool grew = __any_sync(0xffffffffu, over);  // warp-uniform
        if (grew) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float mt = sc[h];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            if (mt > m[h] + kLazyMax || (m[h] == -INFINITY && mt != -INFINITY)) {  // uniform: mt is the warp's
              alpha[h] = exp2_approx(m[h] - mt);  // 0 while m is -inf
              m[h] = mt;
            }
          }
        }
        // this token's weights P' = p * sV for the 4 groups x 4 heads
        float p[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          p[h] = (m[h] == -INFINITY || !valid) ? 0.f : exp2_approx(sc[h] - m[h]);
          l[h] = l[h] * alpha[h] + p[h];
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4*>(pw + p_chunk(lane, q)) =
              make_float4(p[0] * sv[q], p[1] * sv[q], p[2] * sv[q], p[3] * sv[q]);
        if (grew) {  // warp-uniform: the maxima are the warp's
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float2 a2 = make_float2(alpha[h], alpha[h]);
            o[h][0] = __fmul2_rn(o[h][0], a2);
            o[h][1] = __fmul2_rn(o[h][1], a2);
          }
        }
        __syncwarp();
        // O += P' V over the warp's 32 tokens: lane = dims 4*lane .. 4*lane+3.
        // Only keys that hold data: in a ragged last tile the other slots may
        // hold any bits, and a NaN scale pattern times a zero weight is NaN.
        const int nkeys = x.ctx_keys - (x.b0 + j * kQ8TileBlocks) * kBlockSize - 32 * w;
        const uint8_t* vrow = rawv + (2 * w) * kQ8TileBytes + 4 * lane;
        auto pv_keys = [&](int n) {
#pragma unroll 8
          for (int t = 0; t < n; ++t) {
            const uint32_t cw = *reinterpret_cast<const uint32_t*>(vrow + (t >> 4) * kQ8TileBytes + (t & 15) * 128);
            const float4 pv = *reinterpret_cast<const float4*>(pw + p_chunk(t, g_own));
            float2 c01, c23;
            codes_to_f32(cw, c01, c23);
            const float ph[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float2 p2 = make_float2(ph[h], ph[h]);
              o[h][0] = __ffma2_rn(p2, c01, o[h][0]);
              o[h][1] = __ffma2_rn(p2, c23, o[h][1]);
            }
          }
        };
        if (nkeys >= 32)
          pv_keys(32);  // every tile but a unit's last: a fixed trip count
        else
          pv_keys(nkeys);
        __syncwarp();  // P' is rewritten by the warp's next tile
        if (lane == 0) mbar_arrive(&bars->v_empty[vst]);
      }
      if (!ok) break;

      // ---- unit epilogue: merge the 8 warps' (max, sum, O); a warp without a
      // tile (or a key) in this unit contributes max -inf and sum 0 ----
      float lw[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        lw[h] = l[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lw[h] += __shfl_xor_sync(0xffffffffu, lw[h], off);
      }
      // O of this warp: [head][128 dims] FP32 over its own P' area
#pragma unroll
      for (int h = 0; h < 4; ++h)
        *reinterpret_cast<float4*>(pw + h * 512 + lane * 16) = make_float4(o[h][0].x, o[h][0].y, o[h][1].x, o[h][1].y);
      if (lane < 4) {
        const float mh = lane == 0 ? m[0] : lane == 1 ? m[1] : lane == 2 ? m[2] : m[3];
        const float lh = lane == 0 ? lw[0] : lane == 1 ? lw[1] : lane == 2 ? lw[2] : lw[3];
        ml[aw * 4 + lane] = mh;
        ml[kAttnWarps * 4 + aw * 4 + lane] = lh;
      }
      ok = merge_sync(bars->merge, nmerge, lane);
      if (!ok) break;
      float mx = -INFINITY;
#pragma unroll
      for (int v = 0; v < kAttnWarps; ++v) mx = fmaxf(mx, ml[v * 4 + h_out]);
      float den = 0.f;
      float2 num = make_float2(0.f, 0.f);
#pragma unroll
      for (int v = 0; v < kAttnWarps; ++v) {
        const float mv = ml[v * 4 + h_out];
        const float e = (mv == -INFINITY) ? 0.f : exp2_approx(mv - mx);
        den += e * ml[kAttnWarps * 4 + v * 4 + h_out];
        const float2 ov = *reinterpret_cast<const float2*>(smem + kOffP + v * 2048 + h_out * 512 + d_out * 4);
        num.x += e * ov.x;
        num.y += e * ov.y;
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      if (a.num_splits == 1) {
        *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + orow_out * kHeadDim + d_out) =
            pack_bf16x2(num.x * inv, num.y * inv);
      } else {
        const int64_t slot = orow_out * a.num_splits + x.split;
        *reinterpret_cast<float2*>(a.part_o + slot * kHeadDim + d_out) = make_float2(num.x * inv, num.y * inv);
        if (lane == 0 && aw < 4) a.part_lse[slot] = den > 0.f ? (mx + log2f(den)) * kLn2 : -INFINITY;
      }
      // every warp has read the others' partials before any P' area is written again
      ok = merge_sync(bars->merge, nmerge, lane);
    }
    if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
  } else if (warp < kAppendWarp) {
    // ------------------------------ K dequantisation (4 warps) ------------------------------
    const int t128 = threadIdx.x - kFirstDqWarp * 32;
    const int cc = t128 & 15;  // 16-byte output chunk of a row: dims 8cc .. 8cc+7
    const int rsub = t128 >> 4;
    const int c = cc & 7;
    const int rbase = rsub * 128 + cc * 8;  // + (jj>>1)*2176 + (jj&1)*1024 for row jj*8 + rsub
    const int wbase = (cc >> 3) * kOpHalfBytes + rsub * 128 + ((c ^ rsub) << 4);  // + jj*1024
    int i = 0;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const Unit x = unit_at(a, u);
      if (x.n_tiles == 0) continue;
      const int64_t orow0 = static_cast<int64_t>(x.r) * hq + x.kvh * kGroup;
      const uint16_t* qg = static_cast<const uint16_t*>(a.q) + orow0 * kHeadDim;
      const float qs = pow2i(-q_shift(group_q_absmax(qg, lane)));
      for (int j = 0; j < x.n_tiles; ++j, ++i) {
        const int st = i % kKStages;
        const int b = i & 1;
        ok = mbar_wait(&bars->k_full[st], (i / kKStages) & 1);
        if (ok && i >= 2) ok = mbar_wait(&bars->kd_empty[b], ((i - 2) >> 1) & 1);  // QK(i-2) done
        // the unit's first tile rewrites the query operand: the previous unit's last QK must be done
        if (ok && j == 0 && i >= 1) ok = mbar_wait(&bars->kd_empty[(i - 1) & 1], ((i - 1) >> 1) & 1);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint8_t* stage = smem + kOffRawK + st * kRawStageBytes;
        // token t128's K scales for the softmax (slot i % 4 was last read by the
        // softmax of tile i-4, which released S(i-4) before QK(i-2) ran)
        *reinterpret_cast<uint2*>(smem + kOffSk + (i % kScaleSlots) * 1024 + t128 * 8) =
              *reinterpret_cast<const uint2*>(stage + (t128 >> 4) * kQ8TileBytes + kQ8CodeBytes + (t128 & 15) * 8);
        if (j == 0) {
          // the unit's block-diagonal query operand
          const int d = t128;
          float qv[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) qv[h] = bf16_lo(qg[h * kHeadDim + d]) * qs;
          uint8_t* qb = smem + kOffQbd + (d >> 6) * 2048;
#pragma unroll
          for (int n = 0; n < 16; ++n)
            *reinterpret_cast<__half*>(qb + tc::sw128_offset(n, d & 63)) =
                __float2half_rn((n >> 2) == (d >> 5) ? qv[n & 3] : 0.f);
        }
        // all 16 loads first: stores to the operand tile could alias them for
        // the compiler, which would otherwise serialise load -> store pairs
        const uint8_t* raw = stage + rbase;
        uint8_t* dst = smem + kOffKd + b * 2 * kOpHalfBytes + wbase;
        uint2 wv[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          wv[jj] = *reinterpret_cast<const uint2*>(raw + (jj >> 1) * kQ8TileBytes + (jj & 1) * 1024);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          *reinterpret_cast<uint4*>(dst + jj * 1024) = codes_to_f16(wv[jj]);
        tc::fence_proxy_async_smem();  // the operand tiles are read by the tensor core
        mbar_arrive(&bars->kd_full[b]);
        mbar_arrive(&bars->sk_full[i % kScaleSlots]);
        mbar_arrive(&bars->k_empty[st]);
      }
    }
    if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
  } else if constexpr (kFused) {
    // ------------------------------ append (fused instance) ------------------------------
    // Per unit holding its request's new token: the K and V rows quantised as
    // kv_append_q8 quantises them and stored where it stores them, then made
    // visible to the producers' bulk copies (async proxy) and announced; the
    // tile holding the token is copied after that, so it carries the rows.
    // A slot other than the one the block table gives position ctx - 1 is
    // stored and reported (the result is then undefined, as documented).
    int nf = 0;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const Unit x = unit_at<true>(a, u);
      if (x.new_tile < 0) continue;
      const int sl = nf % kReadySlots;
      if (nf >= kReadySlots)  // both producers have passed the slot's previous unit
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->ready_empty[sl], ((nf / kReadySlots) - 1) & 1));
      if (!ok) break;
      const int64_t row = static_cast<int64_t>(x.r) * a.num_kv_heads + x.kvh;
      const uint2 kr = reinterpret_cast<const uint2*>(a.k_new)[row * (kHeadDim / 4) + lane];
      const uint2 vr = reinterpret_cast<const uint2*>(a.v_new)[row * (kHeadDim / 4) + lane];
      const int64_t slot = a.slot_mapping[x.r];
      const int pb = a.block_tables[static_cast<int64_t>(x.r) * a.max_blocks + x.new_blk];
      float kd, vd;
      const uint32_t kc = q8_0_quantize_lane(kr, kd);
      const uint32_t vc = q8_0_quantize_lane(vr, vd);
      q8_store_row(a, a.k_cache, slot, x.kvh, kc, kd, lane);
      q8_store_row(a, a.v_cache, slot, x.kvh, vc, vd, lane);
      if (slot >= 0 && slot != static_cast<int64_t>(pb) * kBlockSize + (x.ctx_raw - 1) % kBlockSize && lane == 0)
        report(a.err, PKV_DEVERR_SLOT);
      fence_proxy_async_global();  // the stores before the bulk copies that read them
      mbar_arrive(&bars->ready[sl]);
      ++nf;
    }
    if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemColsQ8);
  }
}

template <bool kFused>
cudaError_t allow_smem_q8() {
  static std::atomic<bool> done[64];  // per device; host threads may race on a first call
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    e = cudaFuncSetAttribute(paged_decode_q8_kernel<kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemQ8);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_paged_decode_q8(const DecodeArgs& a, int32_t grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (a.k_new != nullptr) {
    cudaError_t e = allow_smem_q8<true>();
    if (e != cudaSuccess) return e;
    return launch_pdl(paged_decode_q8_kernel<true>, dim3(static_cast<unsigned>(grid)), dim3(kQ8ThreadsFused),
                      kSmemQ8, stream, 1, a);
  }
  cudaError_t e = allow_smem_q8<false>();
  if (e != cudaSuccess) return e;
  return launch_pdl(paged_decode_q8_kernel<false>, dim3(static_cast<unsigned>(grid)), dim3(kQ8Threads), kSmemQ8,
                    stream, 1, a);
}

}  // namespace pkv
