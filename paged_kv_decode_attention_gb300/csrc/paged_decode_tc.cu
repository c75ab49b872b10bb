// paged_decode_tc.cu -- decode attention (one query token per request) over a
// paged BF16 KV cache for large batches: both contractions on the
// 5th-generation tensor cores, the KV stream held in flight by one persistent
// CTA per SM.
//
// What it computes ("Chapter 8: Inference Optimization",
// clxhxhhr.top/posts/4341): the decode step of §8.1.1 reads the request's
// context KV; §8.3.1 / Fig. 8-10 -- logical block j is found through the
// request's block table; §8.3.2 / Fig. 8-13 -- shared prefix blocks are plain
// table entries.  Softmax is blockwise with a running maximum and sum (online
// softmax, the FlashAttention organisation §8.3.1 names).
//
// Why tensor cores for a 4 FLOP/B step: decode is bound by the bytes in
// flight.  An SM must keep about 190 KB of K/V requests outstanding to cover
// the loaded HBM latency at its share of the bandwidth, which leaves room for
// one CTA; that CTA then has about 1.2 us per 64 KB tile, too little for FP32
// dot products of 4 heads x 128 tokens x 128 dims beside the softmax.  Per
// 128-token tile (8 blocks) of a (request, KV head, split) unit:
//   S^T = K . Qp^T   (A = K tile, M = 128 tokens, K = 128 dims, N = 16)
//   O^T += V^T . P^T (A = V tile read MN-major, M = 128 dims, K = 128 tokens, N = 16)
// with Qp rows 0-3 = the 4 query heads of the GQA group and P^T rows 0-3 the
// weights in BF16, rows 4-7 the BF16 rounding of their remainders (so P.V
// carries the weights to about 2^-17 relative), zeros elsewhere: 16
// tcgen05.mma per tile, while the CUDA cores exponentiate one score per
// (token, head).
//
// The persistent CTAs stride through the units.  CTA = 8 warps:
//   warp 0 / 1 : K / V producer -- TMA loads of 16-token x 64-dim boxes
//                (128-byte swizzle) of the tile's 8 blocks into 3-stage K and V
//                rings (32 KiB per stage); blocks past the unit's range are
//                fetched at an out-of-range row so TMA fills them with zeros.
//   warp 2     : MMA issuer (one thread): S into a double-buffered S and P.V
//                into the unit's O (double-buffered across units), each issued
//                as soon as its inputs are ready.
//   warp 3     : writes each unit's query operand Qp (BF16, as stored).
//   warps 4-7  : softmax, thread = token (TMEM lane) of the tile: masks keys
//                past the context, scales into base 2, agrees with the other 3
//                warps on the tile's per-head maxima, raises the running
//                maximum lazily (by more than 2^8 only, rescaling O in tensor
//                memory), writes P^T and, at a unit's end, O / l (BF16, or a
//                normalised split partial and its log-sum-exp).  Each tile and
//                unit end passes one barrier of the 4 warps where each posts
//                its health, so all four leave together if one gives up a wait.
// Every wait is bounded and reports PKV_DEVERR_TIMEOUT instead of hanging.
#include <climits>
#include <cmath>

#include "pkv_common.cuh"
#include "pkv_kernels.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kDtStages = 3;
constexpr int kDtThreads = 256;
constexpr int kDtTileBlocks = 8;                            // blocks per tile
constexpr int kDtTileTokens = kDtTileBlocks * kBlockSize;   // 128 tokens
constexpr int kDtHalfBytes = kDtTileTokens * 128;           // 64 dims x 128 tokens: 16 KiB
constexpr int kDtStageBytes = 2 * kDtHalfBytes;             // K (or V) of one tile: 32 KiB
constexpr int kDtN = 16;                                    // MMA N
constexpr int kDtOpHalf = kDtN * 128;                       // 16 rows x 64 elements: 2 KiB
constexpr int kDtOpBytes = 2 * kDtOpHalf;                   // Qp or P^T: 4 KiB
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kDtStages * kDtStageBytes;
constexpr int kOffQp = kOffV + kDtStages * kDtStageBytes;   // 2 buffers (unit parity)
constexpr int kOffPt = kOffQp + 2 * kDtOpBytes;             // 2 buffers (tile parity)
constexpr int kOffX = kOffPt + 2 * kDtOpBytes;              // float [2][4 warps][8]: exchanges
constexpr int kOffBar = kOffX + 2 * 4 * 8 * 4;
constexpr int kSmemDt = kOffBar + 256;
constexpr uint32_t kColS = 0;    // S^T buffers at columns 0 and 16
constexpr uint32_t kColO = 32;   // O^T buffers at columns 32 and 48
constexpr uint32_t kDtTmemCols = 64;
constexpr float kDtLazyMax = 8.f;  // base-2 units: weights stay below 2^8
constexpr float kDtLn2 = 0.6931471805599453f;
constexpr int kDtNamedBar = 1;     // the softmax warps' barrier

static_assert(kSmemDt <= 227 * 1024, "one CTA per SM");
static_assert(kOffV % 1024 == 0 && kOffQp % 1024 == 0 && kOffPt % 1024 == 0, "swizzled operands need 1 KiB alignment");

struct DtBars {
  uint64_t k_full[kDtStages];
  uint64_t k_empty[kDtStages];
  uint64_t v_full[kDtStages];
  uint64_t v_empty[kDtStages];
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
static_assert(sizeof(DtBars) <= 256, "barrier area");

struct DtUnit {
  int r, kvh, split, b0, b1, n_tiles, ctx_keys, ctx_raw;
};

// Unit u: split fastest, then KV head, then request.
__device__ __forceinline__ DtUnit dt_unit(const DecodeArgs& a, int u) {
  DtUnit x;
  x.split = u % a.num_splits;
  const int row = u / a.num_splits;
  x.r = row / a.num_kv_heads;
  x.kvh = row - x.r * a.num_kv_heads;
  x.ctx_raw = a.context_lens[x.r];
  const int ctx = min(max(x.ctx_raw, 0), a.max_blocks * kBlockSize);
  const int nb = (ctx + kBlockSize - 1) / kBlockSize;
  x.b0 = x.split * a.blocks_per_split;
  x.b1 = min(nb, x.b0 + a.blocks_per_split);
  x.n_tiles = x.b1 > x.b0 ? (x.b1 - x.b0 + kDtTileBlocks - 1) / kDtTileBlocks : 0;
  x.ctx_keys = min(ctx, x.b1 * kBlockSize);
  return x;
}

// Producer warp: TMA loads of one tensor's tiles into its ring.  Lane 2b + h
// issues the box of block b, dims 64h .. 64h+63; block ids are read 32 at a
// time, one chunk ahead.
__device__ __forceinline__ bool dt_produce(const DecodeArgs& a, const CUtensorMap* map, uint8_t* ring,
                                           uint64_t* full, uint64_t* empty, int num_units, int lane) {
  const uint64_t policy = l2_policy_evict_first();
  const int oob_row = a.num_blocks * a.num_kv_heads * kBlockSize;  // first row past the pool
  bool ok = true;
  int i = 0;
  for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
    const DtUnit x = dt_unit(a, u);
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
      const int slot = j & 3;  // this tile's 8 entries in the current 32-entry chunk
      if (slot == 0) nxt = entry(x.b0 + j * kDtTileBlocks + 32 + lane);
      const int blk = __shfl_sync(0xffffffffu, cur, slot * kDtTileBlocks + ((lane >> 1) & 7));
      if (slot == 3) cur = nxt;
      const int st = i % kDtStages;
      if (i >= kDtStages) ok = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((i / kDtStages) - 1) & 1));
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], kDtStageBytes);
      __syncwarp();
      if (lane < 2 * kDtTileBlocks) {
        int y = oob_row;
        if (blk != INT_MIN) {
          int b = blk;
          if (b < 0 || b >= a.num_blocks) {
            report(a.err, PKV_DEVERR_BLOCK_ID);
            b = 0;
          }
          y = (b * a.num_kv_heads + x.kvh) * kBlockSize;
        }
        const int bb = lane >> 1, h = lane & 1;
        tc::tma_load_2d(ring + st * kDtStageBytes + h * kDtHalfBytes + bb * (kBlockSize * 128), map, h * 64, y,
                        &full[st], policy);
      }
    }
  }
  // copies still in flight must land before shared memory is released
  if (lane == 0)
    for (int k = max(0, i - kDtStages); k < i; ++k) mbar_wait(&full[k % kDtStages], (k / kDtStages) & 1);
  return ok;
}

__device__ __forceinline__ float sel4(const float* v, int k) {
  return k == 0 ? v[0] : k == 1 ? v[1] : k == 2 ? v[2] : v[3];
}

__global__ void __launch_bounds__(kDtThreads, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                           const DecodeArgs a) {
  pdl_trigger();
  extern __shared__ __align__(1024) uint8_t smem[];
  DtBars* bars = reinterpret_cast<DtBars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_units = a.num_seqs * a.num_kv_heads * a.num_splits;
  const int hq = a.num_kv_heads * kGroup;

  // ---------------- set-up ----------------
  // Qp and P^T rows past the ones written per unit / tile stay zero.
  for (int idx = threadIdx.x; idx < 4 * kDtOpBytes / 16; idx += kDtThreads)
    reinterpret_cast<uint4*>(smem + kOffQp)[idx] = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDtStages; ++s) {
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
    tc::tmem_alloc(&bars->tmem_base, kDtTmemCols);
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
    ok = warp == 0 ? dt_produce(a, &k_map, smem + kOffK, bars->k_full, bars->k_empty, num_units, lane)
                   : dt_produce(a, &v_map, smem + kOffV, bars->v_full, bars->v_empty, num_units, lane);
    if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
  } else if (warp == 2) {
    // ------------------------------ MMA issuer ------------------------------
    // Two cursors walk the tile sequence: one issues S, the other P.V.  The
    // thread polls both and issues whichever is ready, so a P.V whose weights
    // are done never waits behind the next tile's K arrival.
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16_f32(128, kDtN, false, false);
      constexpr uint32_t kIdO = tc::idesc_bf16_f32(128, kDtN, true, false);
      struct Cursor {
        int u, j, i, seq, n;  // unit, tile in unit, tile overall, unit ordinal, tiles of the unit
      };
      auto settle = [&](Cursor& c) {  // move to the first unit with a tile, from c.u on
        for (; c.u < num_units; c.u += gridDim.x) {
          c.n = dt_unit(a, c.u).n_tiles;
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
      while (cp.u < num_units) {
        bool progressed = false;
        // ---- S of the next tile ----
        if (cs.u < num_units) {
          const int i = cs.i, st = i % kDtStages, sb = i & 1, ub = cs.seq & 1;
          bool ready = mbar_test_wait(&bars->k_full[st], (i / kDtStages) & 1);
          if (ready && cs.j == 0) ready = mbar_test_wait(&bars->q_full[ub], (cs.seq >> 1) & 1);
          if (ready && i >= 2) ready = mbar_test_wait(&bars->s_empty[sb], ((i >> 1) - 1) & 1);
          if (ready) {
            tc::fence_after_sync();
            const uint32_t kst = sbase + kOffK + st * kDtStageBytes;
            const uint32_t qp = sbase + kOffQp + ub * kDtOpBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // 16 dims per step
              tc::mma_bf16(tmem + kColS + 16 * sb,
                           tc::smem_desc(kst + (kk >> 2) * kDtHalfBytes + 32 * (kk & 3), 16, 1024),
                           tc::smem_desc(qp + (kk >> 2) * kDtOpHalf + 32 * (kk & 3), 16, 1024), kIdS,
                           kk > 0 ? 1u : 0u);
            tc::commit(&bars->s_full[sb]);
            tc::commit(&bars->k_empty[st]);
            if (cs.j == cs.n - 1) tc::commit(&bars->q_empty[ub]);
            advance(cs);
            progressed = true;
          }
        }
        // ---- P.V of the oldest tile whose S is issued ----
        if (cp.i < cs.i) {
          const int i = cp.i, st = i % kDtStages, pb = i & 1, ub = cp.seq & 1;
          bool ready = mbar_test_wait(&bars->p_full[pb], (i >> 1) & 1) &&
                       mbar_test_wait(&bars->v_full[st], (i / kDtStages) & 1);
          // the first tile of a unit overwrites O: the epilogue that last read it must be done
          if (ready && cp.j == 0 && cp.seq >= 2)
            ready = mbar_test_wait(&bars->o_empty[ub], ((cp.seq >> 1) - 1) & 1);
          if (ready) {
            tc::fence_after_sync();
            const uint32_t vst = sbase + kOffV + st * kDtStageBytes;
            const uint32_t pt = sbase + kOffPt + pb * kDtOpBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // 16 tokens per step
              tc::mma_bf16(tmem + kColO + 16 * ub, tc::smem_desc(vst + 2048 * kk, kDtHalfBytes, 1024),
                           tc::smem_desc(pt + (kk >> 2) * kDtOpHalf + 32 * (kk & 3), 16, 1024), kIdO,
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
    int seq = 0;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const DtUnit x = dt_unit(a, u);
      if (x.n_tiles == 0) continue;
      const int ub = seq & 1;
      if (seq >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_empty[ub], ((seq >> 1) - 1) & 1));
      if (!ok) break;
      // the group's 4 heads x 128 dims are 1 KiB contiguous: 64 chunks of 8 dims
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                        (static_cast<int64_t>(x.r) * hq + x.kvh * kGroup) * kHeadDim);
      uint8_t* dst = smem + kOffQp + ub * kDtOpBytes;
#pragma unroll
      for (int c = lane; c < 64; c += 32) {
        const int h = c >> 4, cc = c & 15;
        *reinterpret_cast<uint4*>(dst + (cc >> 3) * kDtOpHalf + tc::sw128_offset(h, (cc & 7) * 8)) = src[c];
      }
      tc::fence_proxy_async_smem();
      mbar_arrive(&bars->q_full[ub]);
      ++seq;
    }
    if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
  } else {
    // ------------------------------ softmax ------------------------------
    const int w = warp & 3;           // TMEM sub-partition
    const int t = threadIdx.x - 128;  // token of the tile (TMEM lane); at a unit's end, the output dim
    const uint32_t lane_off = static_cast<uint32_t>(w * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + kOffX);  // [2][4][8]
    const float c0 = a.scale_log2;
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
      named_barrier_sync(kDtNamedBar, 128);
      ++nx;
      bool all = true;
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) all = all && buf[ww * 8 + 4] != 0.f;
      return all;
    };
    int i = 0, seq = 0;
    for (int u = blockIdx.x; u < num_units && ok_all; u += gridDim.x) {
      const DtUnit x = dt_unit(a, u);
      const int64_t orow0 = static_cast<int64_t>(x.r) * hq + x.kvh * kGroup;
      if (threadIdx.x == 128 && x.split == 0 && x.kvh == 0 && x.ctx_raw > a.max_blocks * kBlockSize)
        report(a.err, PKV_DEVERR_CONTEXT);
      if (x.n_tiles == 0) {  // padding row or a split past the context
        if (direct)
          reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + orow0 * kHeadDim)[t] = make_uint2(0, 0);
        else if (t < kGroup)
          a.part_lse[(orow0 + t) * a.num_splits + x.split] = -INFINITY;
        continue;
      }
      const int ub = seq & 1;
      float m[4], l[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
      for (int j = 0; j < x.n_tiles; ++j, ++i) {
        const int sb = i & 1;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (i >> 1) & 1));
        if (ok) {
          tc::fence_after_sync();
          tc::tmem_ld4(tmem + lane_off + kColS + 16 * sb, s);
          tc::tmem_wait_ld();
          tc::fence_before_sync();
          mbar_arrive(&bars->s_empty[sb]);
        }
        const int tok = (x.b0 + j * kDtTileBlocks) * kBlockSize + t;
        const bool valid = tok < x.ctx_keys;
        float sc[4], mt[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          sc[h] = (ok && valid) ? c0 * s[h] : -INFINITY;
          mt[h] = sc[h];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
          for (int h = 0; h < 4; ++h) mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], off));
        // agree on the tile's maxima (and on whether every warp is healthy)
        float* xs = xbuf();
        if (lane < 4) xs[w * 8 + lane] = sel4(mt, lane);
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
        // lazy running maximum: move it only when a score exceeds it by more than 2^8
        float alpha[4];
        bool grow_any = false;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const bool grow = tm[h] > m[h] + kDtLazyMax || (m[h] == -INFINITY && tm[h] != -INFINITY);
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
              float o[8];  // columns h (high part) and 4 + h (remainder) of head h
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
        float p[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          p[h] = (sc[h] == -INFINITY) ? 0.f : exp2_approx(sc[h] - m[h]);
          l[h] += p[h];
        }
        // P^T buffer sb is free once P.V(i - 2) has read it
        if (ok && i >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_empty[sb], ((i >> 1) - 1) & 1));
        // slots past the data in the last real block may hold any bits (NaN
        // patterns included): zero those V rows, a zero weight is not enough
        const bool garbage = !valid && tok < x.b1 * kBlockSize;
        if (ok && __any_sync(0xffffffffu, garbage)) {
          const int st = i % kDtStages;
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (i / kDtStages) & 1));
          if (ok && garbage) {
            uint8_t* vt = smem + kOffV + st * kDtStageBytes;
#pragma unroll
            for (int c = 0; c < 16; ++c)
              *reinterpret_cast<uint4*>(vt + (c >> 3) * kDtHalfBytes + t * 128 + (c & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
          }
        }
        if (ok) {
          uint8_t* pt = smem + kOffPt + sb * kDtOpBytes + (t >> 6) * kDtOpHalf;
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const uint32_t hi = pack_bf16x2(p[h], 0.f) & 0xffffu;
            const float rest = p[h] - __uint_as_float(hi << 16);  // exact in FP32
            const uint32_t lo = pack_bf16x2(rest, 0.f) & 0xffffu;
            *reinterpret_cast<uint16_t*>(pt + tc::sw128_offset(h, t & 63)) = static_cast<uint16_t>(hi);
            *reinterpret_cast<uint16_t*>(pt + tc::sw128_offset(4 + h, t & 63)) = static_cast<uint16_t>(lo);
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
      if (lane < 4) xl[w * 8 + lane] = sel4(l, lane);
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
        for (int h = 0; h < 4; ++h) o[h] = o8[h] + o8[4 + h];
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
            const float ls = sel4(lsum, t);
            a.part_lse[(orow0 + t) * a.num_splits + x.split] = ls > 0.f ? (sel4(m, t) + log2f(ls)) * kDtLn2 : -INFINITY;
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
    tc::tmem_dealloc(tmem, kDtTmemCols);
  }
}

cudaError_t allow_smem_dt() {
  static std::atomic<bool> done[64];  // per device; host threads may race on a first call
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    e = cudaFuncSetAttribute(paged_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemDt);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_paged_decode_tc(const DecodeArgs& a, int32_t grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (a.q_len != 1 || a.num_splits < 1 || (a.num_splits > 1 && (a.part_o == nullptr || a.part_lse == nullptr)))
    return cudaErrorInvalidValue;
  const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.num_kv_heads * kBlockSize;
  if (rows + kBlockSize >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  CUtensorMap kmap, vmap;
  if (!make_pool_map(&kmap, a.k_cache, rows) || !make_pool_map(&vmap, a.v_cache, rows)) return cudaErrorInvalidValue;
  cudaError_t e = allow_smem_dt();
  if (e != cudaSuccess) return e;
  return launch_pdl(paged_decode_tc_kernel, dim3(static_cast<unsigned>(grid)), dim3(kDtThreads), kSmemDt, stream, 1,
                    kmap, vmap, a);
}

}  // namespace pkv
