// paged_decode_fp8_tc.cu -- decode attention (one query token per request)
// over a paged FP8 (E4M3) KV cache with both contractions on the
// 5th-generation tensor cores in their 8-bit mode: the K and V tiles go from
// HBM into shared memory by TMA and into the tensor core as they are, with no
// conversion pass and no converted operand copy.
//
// What it computes ("Chapter 8: Inference Optimization",
// clxhxhhr.top/posts/4341): the decode step of §8.1.1 reads the request's
// context KV through its block table (§8.3.1 / Fig. 8-10), with K and V held
// in FP8 and the query in BF16 (§8.4.4).  Softmax is blockwise with a running
// maximum and sum (the FlashAttention organisation §8.3.1 names).
//
// Per 256-token tile (16 blocks) of a (request, KV head, split) unit:
//   S^T = K . Qp^T   (kind::f8f6f4, A = K tile K-major, M = 128 tokens per
//                     half, K = 128 dims, N = 16: 2 x 4 instructions)
//   O^T += V^T . P^T (A = V tile read MN-major, M = 128 dims, K = 256 tokens,
//                     N = 16: 8 instructions)
// A tile is 256 tokens because the softmax's fixed cost per tile (the four
// warps agreeing on the maxima) is what bounds an SM: each thread takes two
// tokens per agreement.
// Both operands of an 8-bit MMA are 8-bit, so the BF16 query and the FP32
// weights enter as sums of E4M3 parts, which keeps them exact or nearly so:
//   - Qp rows 0-3 are the 4 query heads of the GQA group scaled by a power of
//     two sigma_h (the largest |q| lands in [128, 256)) and rounded to E4M3;
//     rows 4-7 are the E4M3 rounding of what that left.  A BF16 value has 8
//     significant bits and each part holds 4, so q * sigma_h = row h + row
//     4 + h exactly, down to E4M3's smallest step (2^-9, i.e. 2^-16 of the
//     largest element).  The softmax divides the scores by sigma_h again.
//   - P^T rows 0-3 are the weights times 2^6, rounded to E4M3, rows 4-7 the
//     rounding of the remainders: about 2^-8 relative per weight.  The
//     running maximum moves lazily (when a score exceeds it by more than
//     2^2), so a weight is at most 2^2 and 2^6 times it at most 2^8, inside
//     E4M3's range (448); the factor keeps the remainders of weights above
//     2^-8 out of E4M3's subnormal range.  The sum of the weights is kept in
//     FP32 from the unrounded values; the epilogue divides O by 2^6 again.
//
// The persistent CTAs stride through the units.  CTA = 8 warps:
//   warp 0 / 1 : K / V producer -- one TMA load per block (16 tokens x 128
//                bytes, 128-byte swizzle: the layout the MMA reads) into
//                3-stage K and V rings of 32 KiB stages; blocks past the unit's
//                range are fetched at an out-of-range row so TMA fills zeros.
//   warp 2     : MMA issuer (one thread): S into a double-buffered S and P.V
//                into the unit's O (double-buffered across units), each issued
//                as soon as its inputs are ready.
//   warp 3     : writes each unit's query operand Qp.
//   warps 4-7  : softmax, thread = token (TMEM lane) of each half tile, as in the
//                BF16 tensor-core decode: mask, scale into base 2, agree on
//                the tile's per-head maxima, rescale O in tensor memory when
//                the maximum moves, write P^T; at a unit's end O / l (BF16, or
//                a normalised split partial and its log-sum-exp).  Each tile
//                and unit end passes one barrier of the 4 warps where each
//                posts its health, so all four leave together if one gives up.
// Every wait is bounded and reports PKV_DEVERR_TIMEOUT instead of hanging.
#include <climits>
#include <cmath>
#include <cuda_fp16.h>

#include "pkv_common.cuh"
#include "pkv_kernels.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kFtStages = 3;
constexpr int kFtThreads = 256;
constexpr int kFtTileBlocks = 16;                          // blocks per tile
constexpr int kFtTileTokens = kFtTileBlocks * kBlockSize;  // 256 tokens: two 128-token halves
constexpr int kFtBoxBytes = kBlockSize * kHeadDim;         // one block's 16 x 128 bytes: 2 KiB
constexpr int kFtHalfBytes = 128 * kHeadDim;               // 128 tokens x 128 bytes: 16 KiB
constexpr int kFtStageBytes = 2 * kFtHalfBytes;            // K (or V) of one tile: 32 KiB
constexpr int kFtN = 16;                                   // MMA N
constexpr int kFtOpBytes = kFtN * 128;                     // Qp, or half of P^T: 16 rows x 128 bytes
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kFtStages * kFtStageBytes;
constexpr int kOffQp = kOffV + kFtStages * kFtStageBytes;  // 2 buffers (unit parity)
constexpr int kOffPt = kOffQp + 2 * kFtOpBytes;            // 2 buffers (tile parity) of 2 halves
constexpr int kOffX = kOffPt + 4 * kFtOpBytes;             // float [2][4 warps][8]: exchanges
constexpr int kOffKn = kOffX + 2 * 4 * 8 * 4;              // fused append: 2 new K rows (unit parity), E4M3
constexpr int kOffKnAt = kOffKn + 2 * kHeadDim;            // int [2]: where each row goes (tile << 8 | row), or -1
constexpr int kOffBar = kOffKnAt + 16;
constexpr int kSmemFt = kOffBar + 512;
constexpr uint32_t kColS = 0;    // S^T buffers at columns 0 and 32 (16 columns per half)
constexpr uint32_t kColO = 64;   // O^T buffers at columns 64 and 80
constexpr uint32_t kFtTmemCols = 128;
constexpr float kFtLazyMax = 2.f;       // base-2 units: weights stay at or below 2^2
constexpr float kFtPScale = 64.f;       // weights enter P^T times 2^6 (at most 2^8 < 448)
constexpr float kFtPUnscale = 1.f / 64.f;
constexpr float kFtLn2 = 0.6931471805599453f;
constexpr int kFtNamedBar = 1;          // the softmax warps' barrier

static_assert(kSmemFt <= 227 * 1024, "one CTA per SM");
static_assert(kFtTileTokens == 2 * 128, "a tile is two 128-token MMA halves");
static_assert(kOffV % 1024 == 0 && kOffQp % 1024 == 0 && kOffPt % 1024 == 0 && kFtOpBytes % 1024 == 0,
              "swizzled operands need 1 KiB alignment");
static_assert(kFtLazyMax + 6.f <= 8.f, "scaled weights must stay inside E4M3's range");

struct FtBars {
  uint64_t k_full[kFtStages];
  uint64_t k_empty[kFtStages];
  uint64_t v_full[kFtStages];
  uint64_t v_empty[kFtStages];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t p_full[2];
  uint64_t p_empty[2];
  uint64_t o_full[2];
  uint64_t o_empty[2];
  uint32_t tmem_base;
};
static_assert(sizeof(FtBars) <= 512, "barrier area");

struct FtUnit {
  int r, kvh, split, b0, b1, n_tiles, ctx_keys, ctx_raw;
  // fused append: the tile and tile row holding the request's new token
  // (position ctx - 1) and its logical block; new_tile = -1 when the unit
  // does not hold it or there is no append
  int new_tile, new_row, new_blk;
};

// Unit u: split fastest, then KV head, then request.  kFused: also where the
// request's new token falls (the fused append).
template <bool kFused>
__device__ __forceinline__ FtUnit ft_unit(const DecodeArgs& a, int u) {
  FtUnit x;
  x.split = u % a.num_splits;
  const int row = u / a.num_splits;
  x.r = row / a.num_kv_heads;
  x.kvh = row - x.r * a.num_kv_heads;
  x.ctx_raw = a.context_lens[x.r];
  const int ctx = min(max(x.ctx_raw, 0), a.max_blocks * kBlockSize);
  const int nb = (ctx + kBlockSize - 1) / kBlockSize;
  x.b0 = x.split * a.blocks_per_split;
  x.b1 = min(nb, x.b0 + a.blocks_per_split);
  x.n_tiles = x.b1 > x.b0 ? (x.b1 - x.b0 + kFtTileBlocks - 1) / kFtTileBlocks : 0;
  x.ctx_keys = min(ctx, x.b1 * kBlockSize);
  x.new_tile = -1;
  x.new_row = 0;
  x.new_blk = 0;
  if (kFused && x.ctx_raw > 0 && x.ctx_raw <= a.max_blocks * kBlockSize) {
    const int p = x.ctx_raw - 1;
    const int nbl = p / kBlockSize;
    if (nbl >= x.b0 && nbl < x.b1) {
      x.new_tile = (nbl - x.b0) / kFtTileBlocks;
      x.new_row = ((nbl - x.b0) % kFtTileBlocks) * kBlockSize + p % kBlockSize;
      x.new_blk = nbl;
    }
  }
  return x;
}

// Fused append: the caller's slot for the unit's new token, and whether it is
// the slot the block table gives that position (only then is the row patched
// into the tiles; any slot inside the pool is stored, as the append would).
__device__ __forceinline__ bool ft_new_slot(const DecodeArgs& a, const FtUnit& x, int64_t& slot) {
  slot = a.slot_mapping[x.r];
  const int pb = a.block_tables[static_cast<int64_t>(x.r) * a.max_blocks + x.new_blk];
  return slot >= 0 && slot == static_cast<int64_t>(pb) * kBlockSize + (x.ctx_raw - 1) % kBlockSize;
}

// Byte offset of the 4 E4M3 values of dims 4l .. 4l+3 of a 256-token stage's
// row `row` (two 128-row halves, 128-byte swizzle).
__device__ __forceinline__ uint32_t ft_row_word(int row, int l) {
  const int half = row >> 7, r = row & 127;
  return half * kFtHalfBytes + r * 128 + ((((l >> 2) ^ (r & 7)) & 7) << 4) + (l & 3) * 4;
}

// Producer warp: TMA loads of one tensor's tiles into its ring.  Lane b < 16
// issues the box of the tile's block b; block ids are read 32 at a time, one
// chunk ahead.
__device__ __forceinline__ bool ft_produce(const DecodeArgs& a, const CUtensorMap* map, uint8_t* ring,
                                           uint64_t* full, uint64_t* empty, int num_units, int lane) {
  const uint64_t policy = l2_policy_evict_first();
  const int oob_row = a.num_blocks * a.num_kv_heads * kBlockSize;  // first row past the pool
  bool ok = true;
  int i = 0;
  for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
    const FtUnit x = ft_unit<false>(a, u);
    if (x.n_tiles == 0) continue;
    const int32_t* table = a.block_tables + static_cast<int64_t>(x.r) * a.max_blocks;
    // the load stays inside the table row whatever the context length, so it
    // need not wait for that length; entries past the unit's blocks are dropped
    auto entry = [&](int bi) -> int {
      const int raw = table[min(bi, a.max_blocks - 1)];
      return bi < x.b1 ? raw : INT_MIN;  // checked where used
    };
    int cur = entry(x.b0 + lane);
    int nxt = INT_MIN;
    for (int j = 0; j < x.n_tiles; ++j, ++i) {
      const int slot = j & 1;  // this tile's 16 entries in the current 32-entry chunk
      if (slot == 0) nxt = entry(x.b0 + j * kFtTileBlocks + 32 + lane);
      const int blk = __shfl_sync(0xffffffffu, cur, slot * kFtTileBlocks + (lane & 15));
      if (slot == 1) cur = nxt;
      const int st = i % kFtStages;
      if (i >= kFtStages) ok = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((i / kFtStages) - 1) & 1));
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], kFtStageBytes);
      __syncwarp();
      if (lane < kFtTileBlocks) {
        int y = oob_row;
        if (blk != INT_MIN) {
          int b = blk;
          if (b < 0 || b >= a.num_blocks) {
            report(a.err, PKV_DEVERR_BLOCK_ID);
            b = 0;
          }
          y = (b * a.num_kv_heads + x.kvh) * kBlockSize;
        }
        tc::tma_load_2d(ring + st * kFtStageBytes + lane * kFtBoxBytes, map, 0, y, &full[st], policy);
      }
    }
  }
  // copies still in flight must land before shared memory is released
  if (lane == 0)
    for (int k = max(0, i - kFtStages); k < i; ++k) mbar_wait(&full[k % kFtStages], (k / kFtStages) & 1);
  return ok;
}

__device__ __forceinline__ float ft_sel4(const float* v, int k) {
  return k == 0 ? v[0] : k == 1 ? v[1] : k == 2 ? v[2] : v[3];
}

// Two FP32 values rounded to E4M3 (nearest even, saturating at +-448): `a`
// in the high byte, `b` in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

// The two E4M3 values of a pair back in FP32 (exact): low byte in lo, high byte in hi.
__device__ __forceinline__ void e4m3x2_to_f32x2(uint32_t pair, float& lo, float& hi) {
  uint32_t h2;
  const uint16_t p = static_cast<uint16_t>(pair);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(p));
  lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
  hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

// 4 BF16 values (two words) as 4 E4M3 bytes, rounded as the E4M3 append rounds.
__device__ __forceinline__ uint32_t bf16x4_to_e4m3x4(uint32_t w0, uint32_t w1) {
  return f32x2_to_e4m3x2(bf16_hi(w0), bf16_lo(w0)) | (f32x2_to_e4m3x2(bf16_hi(w1), bf16_lo(w1)) << 16);
}

// The power of two that brings a head's largest |q| (BF16 magnitude bits
// `amax_bits`) into [128, 256); 1 for an all-zero head.
__device__ __forceinline__ float q_sigma(uint32_t amax_bits) {
  if (amax_bits == 0) return 1.f;
  int e = static_cast<int>((amax_bits >> 7) & 0xffu) - 127;  // exponent of the largest |q|
  if (e < -126) e = -126;                                    // subnormal: treat as the smallest normal
  int s = 7 - e;
  s = s < -120 ? -120 : (s > 120 ? 120 : s);
  return __int_as_float((127 + s) << 23);
}

// kFused: the request's new token is stored and used in place of the row
// read (a.k_new, a.v_new, a.slot_mapping set); an instance of its own, so the
// plain decode carries none of that work.
template <bool kFused>
__global__ void __launch_bounds__(kFtThreads, 1)
    paged_decode_fp8_tc_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                               const DecodeArgs a) {
  pdl_trigger();
  extern __shared__ __align__(1024) uint8_t smem[];
  FtBars* bars = reinterpret_cast<FtBars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_units = a.num_seqs * a.num_kv_heads * a.num_splits;
  const int hq = a.num_kv_heads * kGroup;

  // ---------------- set-up ----------------
  // Qp and P^T rows past the ones written per unit / tile stay zero.
  for (int idx = threadIdx.x; idx < 6 * kFtOpBytes / 16; idx += kFtThreads)
    reinterpret_cast<uint4*>(smem + kOffQp)[idx] = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFtStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->q_full[b], 32);
      mbar_init(&bars->q_empty[b], 1);
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_empty[b], 128);
      mbar_init(&bars->p_full[b], 128);
      mbar_init(&bars->p_empty[b], 1);
      mbar_init(&bars->o_full[b], 1);
      mbar_init(&bars->o_empty[b], 128);
    }
    fence_barrier_init();
  }
  if (warp == 2) {
    tc::tmem_alloc(&bars->tmem_base, kFtTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tensor_map(&k_map);
    tc::prefetch_tensor_map(&v_map);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // The set-up above reads no input; everything below may read what earlier
  // grids in the stream write, so wait for them here.
  pdl_wait();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t sbase = smem_addr(smem);
  bool ok = true;

  if (warp == 0 || warp == 1) {
    // ------------------------------ producers ------------------------------
    ok = warp == 0 ? ft_produce(a, &k_map, smem + kOffK, bars->k_full, bars->k_empty, num_units, lane)
                   : ft_produce(a, &v_map, smem + kOffV, bars->v_full, bars->v_empty, num_units, lane);
    if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
  } else if (warp == 2) {
    // ------------------------------ MMA issuer ------------------------------
    // Two cursors walk the tile sequence: one issues S, the other P.V.  The
    // thread polls both and issues whichever is ready, so a P.V whose weights
    // are done never waits behind the next tile's K arrival.
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_e4m3_f32(128, kFtN, false, false);
      constexpr uint32_t kIdO = tc::idesc_e4m3_f32(128, kFtN, true, false);
      struct Cursor {
        int u, j, i, seq, n;  // unit, tile in unit, tile overall, unit ordinal, tiles of the unit
      };
      auto settle = [&](Cursor& c) {  // move to the first unit with a tile, from c.u on
        for (; c.u < num_units; c.u += gridDim.x) {
          c.n = ft_unit<false>(a, c.u).n_tiles;
          if (c.n > 0) return;
        }
      };
      auto advance = [&](Cursor& c) {
        ++c.i;
        if (++c.j < c.n) return;
        c.j = 0;
        ++c.seq;
        c.u += gridDim.x;
        settle(c);
      };
      Cursor cs{static_cast<int>(blockIdx.x), 0, 0, 0, 0};
      settle(cs);
      Cursor cp = cs;
      uint64_t t_idle = 0;
      // fused append, K side: the S cursor's unit's new K row (tile << 8 | tile
      // row, or -1), published with the unit's query operand
      int kp_at = -1;
      while (cp.u < num_units) {
        bool progressed = false;
        // ---- S of the next tile ----
        if (cs.u < num_units) {
          const int i = cs.i, st = i % kFtStages, sb = i & 1, ub = cs.seq & 1;
          bool ready = mbar_test_wait(&bars->k_full[st], (i / kFtStages) & 1);
          if (ready && cs.j == 0) ready = mbar_test_wait(&bars->q_full[ub], (cs.seq >> 1) & 1);
          if (ready && i >= 2) ready = mbar_test_wait(&bars->s_empty[sb], ((i >> 1) - 1) & 1);
          if (ready) {
            tc::fence_after_sync();
            const uint32_t kst = sbase + kOffK + st * kFtStageBytes;
            const uint32_t qp = sbase + kOffQp + ub * kFtOpBytes;
            if (kFused && cs.j == 0) kp_at = reinterpret_cast<const int*>(smem + kOffKnAt)[ub];
            if (kFused && kp_at >= 0 && (kp_at >> 8) == cs.j) {
              // the new token's K row (E4M3, from the query-operand warp)
              // written over the tile's row, 16-byte chunks to their swizzled places
              const int row = kp_at & 255, r = row & 127;
              const uint4* src = reinterpret_cast<const uint4*>(smem + kOffKn + ub * kHeadDim);
              uint8_t* dst = smem + kOffK + st * kFtStageBytes + (row >> 7) * kFtHalfBytes + r * 128;
#pragma unroll
              for (int ch = 0; ch < 8; ++ch) *reinterpret_cast<uint4*>(dst + ((ch ^ (r & 7)) << 4)) = src[ch];
              tc::fence_proxy_async_smem();  // the tensor core reads the patched row
            }
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // 32 dims (bytes) per step
                tc::mma_f8(tmem + kColS + 32 * sb + 16 * half,
                           tc::smem_desc(kst + half * kFtHalfBytes + 32 * kk, 16, 1024),
                           tc::smem_desc(qp + 32 * kk, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
            tc::commit(&bars->s_full[sb]);
            tc::commit(&bars->k_empty[st]);
            if (cs.j == cs.n - 1) tc::commit(&bars->q_empty[ub]);
            advance(cs);
            progressed = true;
          }
        }
        // ---- P.V of the oldest tile whose S is issued ----
        if (cp.i < cs.i) {
          const int i = cp.i, st = i % kFtStages, pb = i & 1, ub = cp.seq & 1;
          bool ready = mbar_test_wait(&bars->p_full[pb], (i >> 1) & 1) &&
                       mbar_test_wait(&bars->v_full[st], (i / kFtStages) & 1);
          // the first tile of a unit overwrites O: the epilogue that last read it must be done
          if (ready && cp.j == 0 && cp.seq >= 2)
            ready = mbar_test_wait(&bars->o_empty[ub], ((cp.seq >> 1) - 1) & 1);
          if (ready) {
            tc::fence_after_sync();
            const uint32_t vst = sbase + kOffV + st * kFtStageBytes;
            const uint32_t pt = sbase + kOffPt + pb * 2 * kFtOpBytes;
            // V read MN-major: the 128 dims of a token are one 128-byte
            // swizzled row (a single atom along M), 8-token groups 1 KiB apart;
            // P^T's tokens 128-255 are its second 16-row operand
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // 32 tokens per step
              tc::mma_f8(tmem + kColO + 16 * ub, tc::smem_desc(vst + 4096 * kk, kFtHalfBytes, 1024),
                         tc::smem_desc(pt + (kk >> 2) * kFtOpBytes + 32 * (kk & 3), 16, 1024), kIdO,
                         (cp.j > 0 || kk > 0) ? 1u : 0u);
            tc::commit(&bars->v_empty[st]);
            tc::commit(&bars->p_empty[pb]);
            if (cp.j == cp.n - 1) tc::commit(&bars->o_full[ub]);
            advance(cp);
            progressed = true;
          }
        }
        if (progressed) {
          t_idle = 0;
        } else if (t_idle == 0) {
          t_idle = global_timer_ns();
        } else if (global_timer_ns() - t_idle > kWaitLimitNs) {
          ok = false;
          break;
        }
      }
      if (!ok) report(a.err, PKV_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------ query operand ------------------------------
    // lane = (head h = lane / 8, dims 16 * (lane % 8) .. + 15)
    const int h = lane >> 3, c = lane & 7;
    int seq = 0;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const FtUnit x = ft_unit<kFused>(a, u);
      if (x.n_tiles == 0) continue;
      const int ub = seq & 1;
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(x.r) * hq + x.kvh * kGroup + h) * kHeadDim +
          16 * c);
      const uint4 w0 = src[0], w1 = src[1];
      // fused append, K side: lane l rounds dims 4l .. 4l+3 of the unit's new
      // K row to E4M3 as the append rounds and stores them where the append
      // would; the row goes to the MMA thread with the query operand, which
      // writes it over the tile's row.  The row is loaded with the slot, not
      // after it, so it costs no extra round trip before the first tile.
      uint2 kraw = make_uint2(0, 0);
      int64_t kslot = -1;
      bool kpatch = false;
      if (kFused && x.new_tile >= 0) {
        kraw = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.k_new) +
                                              (static_cast<int64_t>(x.r) * a.num_kv_heads + x.kvh) * kHeadDim)[lane];
        kpatch = ft_new_slot(a, x, kslot);
      }
      const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      uint32_t amax = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = max(amax, max(wv[e] & 0x7fffu, (wv[e] >> 16) & 0x7fffu));
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float sigma = q_sigma(amax);
      uint32_t hi[4], lo[4];  // 16 E4M3 bytes each, dim 16c + 4k + b in byte b of word k
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float xv[4], rv[4];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          xv[2 * b] = bf16_lo(wv[2 * k + b]) * sigma;
          xv[2 * b + 1] = bf16_hi(wv[2 * k + b]) * sigma;
        }
        const uint32_t h01 = f32x2_to_e4m3x2(xv[1], xv[0]), h23 = f32x2_to_e4m3x2(xv[3], xv[2]);
        float r0, r1, r2, r3;
        e4m3x2_to_f32x2(h01, r0, r1);
        e4m3x2_to_f32x2(h23, r2, r3);
        rv[0] = xv[0] - r0;  // exact in FP32
        rv[1] = xv[1] - r1;
        rv[2] = xv[2] - r2;
        rv[3] = xv[3] - r3;
        hi[k] = h01 | (h23 << 16);
        lo[k] = f32x2_to_e4m3x2(rv[1], rv[0]) | (f32x2_to_e4m3x2(rv[3], rv[2]) << 16);
      }
      int kn_at = -1;
      uint32_t kn_word = 0;
      if (kFused && kslot >= 0) {
        kn_word = bf16x4_to_e4m3x4(kraw.x, kraw.y);
        if (kslot < static_cast<int64_t>(a.num_blocks) * kBlockSize)
          *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(const_cast<void*>(a.k_cache)) +
                                       ((kslot / kBlockSize) * a.num_kv_heads + x.kvh) *
                                           static_cast<int64_t>(kFtBoxBytes) +
                                       (kslot % kBlockSize) * kHeadDim + 4 * lane) = kn_word;
        if (kpatch)
          kn_at = (x.new_tile << 8) | x.new_row;
        else if (lane == 0)
          report(a.err, PKV_DEVERR_SLOT);
      }
      if (seq >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_empty[ub], ((seq >> 1) - 1) & 1));
      if (!ok) break;
      uint8_t* dst = smem + kOffQp + ub * kFtOpBytes;
      *reinterpret_cast<uint4*>(dst + tc::sw128_offset_b8(h, 16 * c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(dst + tc::sw128_offset_b8(4 + h, 16 * c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      if (kFused) {
        reinterpret_cast<uint32_t*>(smem + kOffKn + ub * kHeadDim)[lane] = kn_word;
        if (lane == 0) reinterpret_cast<int*>(smem + kOffKnAt)[ub] = kn_at;
      }
      tc::fence_proxy_async_smem();
      mbar_arrive(&bars->q_full[ub]);
      ++seq;
    }
    if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
  } else {
    // ------------------------------ softmax ------------------------------
    const int w = warp & 3;           // TMEM sub-partition
    const int t = threadIdx.x - 128;  // tokens t and 128 + t of the tile (TMEM lane t); at a unit's end, the output dim
    const uint32_t lane_off = static_cast<uint32_t>(w * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + kOffX);  // [2][4][8]
    const bool direct = a.num_splits == 1;
    bool ok_all = true;  // uniform across the 4 warps: changes only right after an exchange
    // Exchanges among the 4 warps alternate between two buffers: each warp
    // writes its 4 values and its health flag into its row, passes the
    // barrier and reads all rows before the next exchange's barrier, so a
    // buffer is reused only after everyone has read it.
    int nx = 0;
    auto xbuf = [&]() -> float* { return xch + (nx & 1) * 32; };
    auto all_healthy = [&](float* buf) -> bool {
      if (lane == 4) buf[w * 8 + 4] = ok ? 1.f : 0.f;
      named_barrier_sync(kFtNamedBar, 128);
      ++nx;
      bool all = true;
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) all = all && buf[ww * 8 + 4] != 0.f;
      return all;
    };
    int i = 0, seq = 0;
    for (int u = blockIdx.x; u < num_units && ok_all; u += gridDim.x) {
      const FtUnit x = ft_unit<kFused>(a, u);
      const int64_t orow0 = static_cast<int64_t>(x.r) * hq + x.kvh * kGroup;
      if (threadIdx.x == 128 && x.split == 0 && x.kvh == 0 && x.ctx_raw > a.max_blocks * kBlockSize)
        report(a.err, PKV_DEVERR_CONTEXT);
      // fused append: a slot for an empty row has no position ctx - 1 to go
      // to; the token is not stored and the caller's error is reported
      if (kFused && threadIdx.x == 128 && x.split == 0 && x.kvh == 0 && x.ctx_raw <= 0 &&
          a.slot_mapping[x.r] >= 0)
        report(a.err, PKV_DEVERR_SLOT);
      if (x.n_tiles == 0) {  // padding row or a split past the context
        if (direct)
          reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + orow0 * kHeadDim)[t] = make_uint2(0, 0);
        else if (t < kGroup)
          a.part_lse[(orow0 + t) * a.num_splits + x.split] = -INFINITY;
        continue;
      }
      const int ub = seq & 1;
      // the query operand's scale of each head, taken from the query exactly
      // as the query-operand warp takes it: scores / sigma_h in base 2
      float c[4];
      {
        const int hh = lane >> 3, cc = lane & 7;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                          (orow0 + hh) * kHeadDim + 16 * cc);
        const uint4 w0 = src[0], w1 = src[1];
        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t amax = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = max(amax, max(wv[e] & 0x7fffu, (wv[e] >> 16) & 0x7fffu));
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float inv_sigma = 1.f / q_sigma(amax);  // a power of two: exact
#pragma unroll
        for (int h = 0; h < 4; ++h) c[h] = a.scale_log2 * __shfl_sync(0xffffffffu, inv_sigma, 8 * h);
      }
      // fused append, V side: the warp whose lanes own the new token's tile
      // row loads its V row (lane l: dims 4l .. 4l+3, rounded to E4M3 as the
      // append rounds) and writes it once that tile's V has landed
      bool vp_mine = false, vp_patch = false;
      int64_t vp_slot = -1;
      uint32_t vp_word = 0;
      if (kFused && x.new_tile >= 0 && ((x.new_row & 127) >> 5) == w) {
        vp_patch = ft_new_slot(a, x, vp_slot);
        vp_mine = vp_slot >= 0;
        const uint2 v = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.v_new) +
                                                       (static_cast<int64_t>(x.r) * a.num_kv_heads + x.kvh) *
                                                           kHeadDim)[lane];
        vp_word = bf16x4_to_e4m3x4(v.x, v.y);
      }
      float m[4], l[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
      for (int j = 0; j < x.n_tiles; ++j, ++i) {
        const int sb = i & 1;
        float s8[2][8] = {};
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (i >> 1) & 1));
        if (ok) {
          tc::fence_after_sync();
          // per half: heads 0..3 from the high parts, then from the remainders
          tc::tmem_ld8(tmem + lane_off + kColS + 32 * sb, s8[0]);
          tc::tmem_ld8(tmem + lane_off + kColS + 32 * sb + 16, s8[1]);
          tc::tmem_wait_ld();
          tc::fence_before_sync();
          mbar_arrive(&bars->s_empty[sb]);
        }
        const int tok0 = (x.b0 + j * kFtTileBlocks) * kBlockSize + t;  // token of half 0; half 1 is 128 further
        bool valid[2];
        float sc[2][4], mt[4];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          valid[hf] = tok0 + 128 * hf < x.ctx_keys;
#pragma unroll
          for (int h = 0; h < 4; ++h) sc[hf][h] = (ok && valid[hf]) ? c[h] * (s8[hf][h] + s8[hf][4 + h]) : -INFINITY;
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) mt[h] = fmaxf(sc[0][h], sc[1][h]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
          for (int h = 0; h < 4; ++h) mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], off));
        // agree on the tile's maxima (and on whether every warp is healthy)
        float* xs = xbuf();
        if (lane < 4) xs[w * 8 + lane] = ft_sel4(mt, lane);
        if (!all_healthy(xs)) {
          ok_all = false;
          break;
        }
        float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int ww = 0; ww < 4; ++ww) {
          const float4 v = *reinterpret_cast<const float4*>(xs + ww * 8);
          tm[0] = fmaxf(tm[0], v.x);
          tm[1] = fmaxf(tm[1], v.y);
          tm[2] = fmaxf(tm[2], v.z);
          tm[3] = fmaxf(tm[3], v.w);
        }
        // lazy running maximum: move it only when a score exceeds it by more than 2^2
        float alpha[4];
        bool grow_any = false;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const bool grow = tm[h] > m[h] + kFtLazyMax || (m[h] == -INFINITY && tm[h] != -INFINITY);
          alpha[h] = grow ? exp2_approx(m[h] - tm[h]) : 1.f;  // 0 while m is -inf
          if (grow) m[h] = tm[h];
          grow_any = grow_any || grow;
        }
        if (grow_any) {  // uniform
          if (j > 0) {
            // O holds weights taken against the old maxima: rescale this warp's 32 dims
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_empty[(i - 1) & 1], ((i - 1) >> 1) & 1));
            if (ok) {
              tc::fence_after_sync();
              float o[8];  // columns h (high parts) and 4 + h (remainders) of head h
              tc::tmem_ld8(tmem + lane_off + kColO + 16 * ub, o);
              tc::tmem_wait_ld();
              uint32_t ob[8];
#pragma unroll
              for (int h = 0; h < 8; ++h) ob[h] = __float_as_uint(o[h] * alpha[h & 3]);
              tc::tmem_st8(tmem + lane_off + kColO + 16 * ub, ob);
              tc::tmem_wait_st();
              tc::fence_before_sync();
            }
          }
#pragma unroll
          for (int h = 0; h < 4; ++h) l[h] *= alpha[h];
        }
        // the weights, and as E4M3 high parts and remainders times 2^6
        uint32_t phi[2][2], plo[2][2];  // [half][pair]: head 2k in the low byte, 2k + 1 in the high byte
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float p[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            p[h] = (sc[hf][h] == -INFINITY) ? 0.f : exp2_approx(sc[hf][h] - m[h]);
            l[h] += p[h];
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float x0 = p[2 * k] * kFtPScale, x1 = p[2 * k + 1] * kFtPScale;
            phi[hf][k] = f32x2_to_e4m3x2(x1, x0);
            float r0, r1;
            e4m3x2_to_f32x2(phi[hf][k], r0, r1);
            plo[hf][k] = f32x2_to_e4m3x2(x1 - r1, x0 - r0);
          }
        }
        // P^T buffer sb is free once P.V(i - 2) has read it
        if (ok && i >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_empty[sb], ((i >> 1) - 1) & 1));
        // slots past the data in the last real block may hold any bits (NaN
        // patterns included): zero those V rows, a zero weight is not enough
        bool garbage[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) garbage[hf] = !valid[hf] && tok0 + 128 * hf < x.b1 * kBlockSize;
        const bool vp_now = vp_mine && j == x.new_tile;  // warp-uniform
        if (ok && (vp_now || __any_sync(0xffffffffu, garbage[0] || garbage[1]))) {
          const int st = i % kFtStages;
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (i / kFtStages) & 1));
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            if (ok && garbage[hf]) {
              uint4* vrow = reinterpret_cast<uint4*>(smem + kOffV + st * kFtStageBytes + (128 * hf + t) * 128);
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) vrow[cc] = make_uint4(0, 0, 0, 0);
            }
          if (ok && vp_now) {
            // the new token's V row, stored where the append would and written over the tile's row
            if (vp_slot < static_cast<int64_t>(a.num_blocks) * kBlockSize)
              *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(const_cast<void*>(a.v_cache)) +
                                           ((vp_slot / kBlockSize) * a.num_kv_heads + x.kvh) *
                                               static_cast<int64_t>(kFtBoxBytes) +
                                           (vp_slot % kBlockSize) * kHeadDim + 4 * lane) = vp_word;
            if (vp_patch)
              *reinterpret_cast<uint32_t*>(smem + kOffV + st * kFtStageBytes + ft_row_word(x.new_row, lane)) =
                  vp_word;
          }
        }
        if (ok) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint8_t* pt = smem + kOffPt + (2 * sb + hf) * kFtOpBytes;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              pt[tc::sw128_offset_b8(h, t)] = static_cast<uint8_t>(phi[hf][h >> 1] >> (8 * (h & 1)));
              pt[tc::sw128_offset_b8(4 + h, t)] = static_cast<uint8_t>(plo[hf][h >> 1] >> (8 * (h & 1)));
            }
          }
          tc::fence_proxy_async_smem();  // P^T and zeroed V rows before the tensor core reads them
          mbar_arrive(&bars->p_full[sb]);
        }
      }
      if (!ok_all) break;

      // ---- unit epilogue: l over the 128 tokens, O / l from tensor memory ----
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int h = 0; h < 4; ++h) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
      float* xl = xbuf();
      if (lane < 4) xl[w * 8 + lane] = ft_sel4(l, lane);
      if (!all_healthy(xl)) {
        ok_all = false;
        break;
      }
      float lsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) {
        const float4 v = *reinterpret_cast<const float4*>(xl + ww * 8);
        lsum[0] += v.x;
        lsum[1] += v.y;
        lsum[2] += v.z;
        lsum[3] += v.w;
      }
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_full[ub], (seq >> 1) & 1));
      if (ok) {
        tc::fence_after_sync();
        float o8[8];
        tc::tmem_ld8(tmem + lane_off + kColO + 16 * ub, o8);  // dim t: heads 0..3, high parts then remainders
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        mbar_arrive(&bars->o_empty[ub]);
        float o[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) o[h] = (o8[h] + o8[4 + h]) * kFtPUnscale;
        if (direct) {
          uint16_t* dst = static_cast<uint16_t*>(a.out) + orow0 * kHeadDim + t;
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float inv = lsum[h] > 0.f ? 1.f / lsum[h] : 0.f;
            dst[h * kHeadDim] = static_cast<uint16_t>(pack_bf16x2(o[h] * inv, 0.f) & 0xffffu);
          }
        } else {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float inv = lsum[h] > 0.f ? 1.f / lsum[h] : 0.f;
            a.part_o[((orow0 + h) * a.num_splits + x.split) * kHeadDim + t] = o[h] * inv;
          }
          if (t < kGroup) {
            const float ls = ft_sel4(lsum, t);
            a.part_lse[(orow0 + t) * a.num_splits + x.split] =
                ls > 0.f ? (ft_sel4(m, t) + log2f(ls)) * kFtLn2 : -INFINITY;
          }
        }
      }
      ++seq;
    }
    if ((!ok || !ok_all) && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kFtTmemCols);
  }
}

template <bool kFused>
cudaError_t allow_smem_ft() {
  static std::atomic<bool> done[64];  // per device; host threads may race on a first call
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    e = cudaFuncSetAttribute(paged_decode_fp8_tc_kernel<kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemFt);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_paged_decode_fp8_tc(const DecodeArgs& a, int32_t grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (a.q_len != 1 || a.num_splits < 1 || (a.num_splits > 1 && (a.part_o == nullptr || a.part_lse == nullptr)))
    return cudaErrorInvalidValue;
  const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.num_kv_heads * kBlockSize;
  if (rows + kBlockSize >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  CUtensorMap kmap, vmap;
  if (!make_pool_map_e4m3(&kmap, a.k_cache, rows) || !make_pool_map_e4m3(&vmap, a.v_cache, rows))
    return cudaErrorInvalidValue;
  const bool fused = a.k_new != nullptr;
  if (fused && (a.v_new == nullptr || a.slot_mapping == nullptr)) return cudaErrorInvalidValue;
  cudaError_t e = fused ? allow_smem_ft<true>() : allow_smem_ft<false>();
  if (e != cudaSuccess) return e;
  return fused ? launch_pdl(paged_decode_fp8_tc_kernel<true>, dim3(static_cast<unsigned>(grid)), dim3(kFtThreads),
                            kSmemFt, stream, 1, kmap, vmap, a)
               : launch_pdl(paged_decode_fp8_tc_kernel<false>, dim3(static_cast<unsigned>(grid)), dim3(kFtThreads),
                            kSmemFt, stream, 1, kmap, vmap, a);
}

}  // namespace pkv
