// paged_chunk_tc.cu -- causal chunk attention on the 5th-generation tensor
// cores: 64 query rows (16 query positions x the 4 query heads of a GQA
// group) against the request's paged K/V, one KV head per CTA.
//
// What it computes ("Chapter 8: Inference Optimization",
// clxhxhhr.top/posts/4341): §8.2.3 and Fig. 8-8/8-9 -- of c new tokens after
// h cached ones, new token j attends to the first h + j tokens; §8.3.1 /
// Fig. 8-10 -- every K/V block is found through the request's block table;
// §8.5.2 -- verifying several positions reads the same KV.  With 16 positions
// x 4 heads the work is a dense contraction (64 rows against every 16-token
// tile), so S = Q K^T and O = P V run as tcgen05.mma with FP32 accumulators in
// tensor memory, and softmax runs in FP32 on the CUDA cores in between.
//
// CTA = 7 warps, one (request, row tile, split, KV head); 2 CTAs per SM:
//   warps 0, 6: TMA producers of K and of V.  A tile is 4 blocks (64 tokens):
//             for each block two 16x64 boxes (128-byte swizzle), issued by 8
//             lanes at once, land in that tensor's ring; blocks past the range
//             are fetched at an out-of-range row so TMA fills them with zeros.
//             A K stage is free once S has read it, a V stage once P.V has, so
//             the K ring refills while a tile's softmax and P.V still run.
//   warp 1  : MMA issuer (one thread).  S_j = Q K_j^T (M 64, N 64, 8 k-steps,
//             Q and K from shared memory) into a double-buffered TMEM S;
//             O += P_j V_j (M 64, N 128, 2 x 4 k-steps, P from TMEM, V from
//             shared memory) into TMEM O.  The thread polls both and issues
//             whichever is ready, so QK^T of the next tile overlaps the
//             softmax and neither waits behind the other.
//   warps 2-5: softmax.  Thread = one row (TMEM lanes 0-15 of each 32-lane
//             sub-partition hold an M=64 accumulator).  Scores are masked
//             (causal and context), scaled into base 2, exponentiated against
//             a lazily updated row max (O in TMEM is rescaled only when a row
//             max grows by more than 2^8), and written back over the S buffer
//             they came from as the A operands of the next PV MMAs: the BF16
//             weights, then the BF16 roundings of their remainders (so P.V
//             carries the weights to about 2^-17 relative, as an FP32 P
//             would within the output's BF16 rounding).
//   epilogue: O / l to BF16 (one split) or FP32 + lse (split-KV partials).
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pkv_common.cuh"
#include "pkv_kernels.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kTcThreads = 224;
constexpr int kVProdWarp = 6;
constexpr int kTileBlocks = 4;                        // KV blocks per tile
constexpr int kTileTokens = kTileBlocks * kBlockSize;  // 64
constexpr int kRows = 64;                             // 16 positions x 4 heads
constexpr int kQBytes = kRows * kHeadDim * 2;         // 16 KiB
constexpr int kHalfBytes = kTileTokens * 128;         // 64 tokens x 64 dims = 8 KiB
constexpr int kStageBytesTc = 2 * kHalfBytes;         // K (or V) of a tile, dims 0-63 then 64-127: 16 KiB
constexpr int kOffQ = 0;
// Ring depth (16 KiB per stage, a K ring and a V ring): with P kept in
// tensor memory, 16 KiB of Q plus 3 + 3 stages fit twice into an SM's shared
// memory (2 CTAs per SM, 96 KiB of K/V each).
constexpr int kTcStages = 3;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kTcStages * kStageBytesTc;
constexpr int kOffBar = kOffV + kTcStages * kStageBytesTc;
constexpr int kSmemTc = kOffBar + 256;
static_assert(kSmemTc <= 113 * 1024, "two CTAs per SM");
// Tensor memory: two S/P buffers of 64 columns (S_j in FP32; then P_j over
// it, its BF16 high parts in the first 32 columns and the BF16 remainders in
// the next 32), then O (128 columns).
constexpr int kNB = 2;
constexpr uint32_t kColO = kNB * 64;
constexpr uint32_t kTmemCols = 256;
constexpr float kRescaleThreshold = 8.f;  // log2 units: weights stay below 2^8
constexpr float kLn2 = 0.6931471805599453f;

struct TcBars {
  uint64_t k_full[kTcStages];
  uint64_t k_empty[kTcStages];
  uint64_t v_full[kTcStages];
  uint64_t v_empty[kTcStages];
  uint64_t s_full[kNB];
  uint64_t p_full[kNB];
  uint64_t o_done[kNB];
  uint64_t q_full;  // the softmax warps have staged Q
  uint32_t tmem_base;
};
static_assert(sizeof(TcBars) <= 256, "barrier area");

template <bool kSplit>
__device__ __forceinline__ void paged_chunk_tc_body(const CUtensorMap& k_map, const CUtensorMap& v_map,
                                                    const ChunkArgs& a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  TcBars* bars = reinterpret_cast<TcBars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---------------- set-up: barriers, TMEM (reads no input) ----------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int s = 0; s < kNB; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 128);
      mbar_init(&bars->o_done[s], 1);
    }
    mbar_init(&bars->q_full, 128);
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tensor_map(&k_map);
    tc::prefetch_tensor_map(&v_map);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // everything below may read what earlier grids in the stream write; the
  // grids launched after this one may start only now: the cascade's suffix
  // pass reads its inputs without waiting, so they must be complete when it starts
  pdl_wait();
  pdl_trigger();

  const bool cascade = a.group_seqs != nullptr;
  const int n_rt = (a.q_len + 15) / 16;  // row tiles per request (chunk mode)
  const int split = blockIdx.y;
  const int kvh = blockIdx.z;
  const int hq = a.num_kv_heads * kGroup;
  const int cap = a.max_blocks * kBlockSize;
  // Row m of the 64-row tile is (request row_req(m), query position row_pos(m), head m % 4).
  //   chunk mode  : one request, positions rt*16 + m/4 (q_len tokens, causal);
  //   cascade mode: member m/4 of prefix group blockIdx.x, its single query.
  int r = 0, rt = 0, table_row = 0, nb = 0, ctx_keys = 0;
  const int32_t* members = nullptr;
  if (cascade) {
    members = a.group_seqs + static_cast<int64_t>(blockIdx.x) * kCascadeGroup;
    table_row = members[0];
    nb = table_row >= 0 ? min(a.group_blocks[blockIdx.x], a.max_blocks) : 0;
    ctx_keys = nb * kBlockSize;  // prefix blocks are full: no garbage slots
  } else {
    r = blockIdx.x / n_rt;
    rt = blockIdx.x - r * n_rt;
    table_row = r;
    const int ctx = a.context_lens[r];
    if (ctx > cap && threadIdx.x == 0 && split == 0 && kvh == 0 && rt == 0) report(a.err, PKV_DEVERR_CONTEXT);
    // the last position of this row tile sees the most keys
    const int ip_last = min(a.q_len - 1, rt * 16 + 15);
    int n_vis_cta = ctx - a.q_len + 1 + ip_last;
    if (ctx <= 0 || n_vis_cta < 0) n_vis_cta = 0;
    n_vis_cta = min(n_vis_cta, cap);
    nb = (n_vis_cta + kBlockSize - 1) / kBlockSize;
    ctx_keys = min(max(ctx, 0), cap);  // keys holding data (the rest of the last block may be garbage)
  }
  auto row_req = [&](int m) -> int { return cascade ? members[m >> 2] : r; };
  auto row_pos = [&](int m) -> int { return cascade ? 0 : rt * 16 + (m >> 2); };
  const int b0 = split * a.blocks_per_split;
  const int b1 = min(nb, b0 + a.blocks_per_split);
  const int n_tiles = (b1 - b0 + kTileBlocks - 1) / kTileBlocks;

  // rows handled by softmax threads: warp w >= 2 owns TMEM sub-partition w % 4
  // Threads t and t+16 of a softmax warp share one row (TMEM lane t), each
  // taking half of its columns.
  const int quad = warp & 3;
  const int half = lane >> 4;
  const int row = quad * 16 + (lane & 15);
  const bool softmax_warp = warp >= 2 && warp < 6;
  const int rq = softmax_warp ? row_req(row) : -1;
  const int ip = row_pos(row);
  const int g = row & 3;
  const bool row_valid = softmax_warp && rq >= 0 && ip < a.q_len;
  const int64_t orow = (static_cast<int64_t>(rq) * a.q_len + ip) * hq + kvh * kGroup + g;
  const int64_t slot = orow * a.part_slots + a.part_slot0 + split;

  const uint32_t tmem = bars->tmem_base;
  const uint32_t sbase = smem_addr(smem);
  bool ok = true;

  if (n_tiles <= 0) {
    if (row_valid && half == 0) {
      if constexpr (kSplit) {
        a.part_lse[slot] = -INFINITY;
      } else {
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow * kHeadDim);
#pragma unroll
        for (int c = 0; c < kHeadDim * 2 / 16; ++c) o[c] = make_uint4(0, 0, 0, 0);
      }
    }
  } else if (warp == 0 || warp == kVProdWarp) {
    // ---------------------------- TMA producers ----------------------------
    const bool is_v = warp == kVProdWarp;
    uint64_t* full = is_v ? bars->v_full : bars->k_full;
    uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
    uint8_t* ring = smem + (is_v ? kOffV : kOffK);
    const CUtensorMap* map = is_v ? &v_map : &k_map;
    const uint64_t policy = l2_policy_evict_first();
    const int32_t* table = a.block_tables + static_cast<int64_t>(table_row) * a.max_blocks;
    const int oob_row = a.num_blocks * a.num_kv_heads * kBlockSize;  // first row past the pool
    const int n_blocks = b1 - b0;
    // block id of block base + lane of the range, INT_MIN past it
    auto chunk = [&](int base) -> int { return base + lane < n_blocks ? table[b0 + base + lane] : INT_MIN; };
    // its pool row (a bad id reads block 0); past the range, the first row
    // past the pool (zero fill)
    auto row_of = [&](int blk) -> int {
      if (blk == INT_MIN) return oob_row;
      if (blk < 0 || blk >= a.num_blocks) {
        report(a.err, PKV_DEVERR_BLOCK_ID);
        blk = 0;
      }
      return (blk * a.num_kv_heads + kvh) * kBlockSize;
    };
    // Block ids are read 32 at a time (8 tiles), one chunk ahead, and checked
    // only when their chunk is used, so the next chunk's load stays in flight.
    // The 8 boxes of a tile (4 blocks x two 64-dim halves) are issued by 8
    // lanes at once: lane 2b + c takes block b, half c.
    int cur = row_of(chunk(0)), nxt = INT_MIN;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int slot = j & 7;
      if (slot == 0) nxt = chunk((j + 8) * kTileBlocks);
      const int yy = __shfl_sync(0xffffffffu, cur, slot * kTileBlocks + ((lane >> 1) & 3));
      if (slot == 7) cur = row_of(nxt);
      const int st = j % kTcStages;
      if (j >= kTcStages) ok = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((j / kTcStages) & 1) ^ 1));
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], kStageBytesTc);
      __syncwarp();
      if (lane < 2 * kTileBlocks) {
        const int b = lane >> 1, c = lane & 1;
        tc::tma_load_2d(ring + st * kStageBytesTc + c * kHalfBytes + b * 2048, map, c * 64, yy, &full[st], policy);
      }
    }
    if (lane == 0) {
      if (!ok) report(a.err, PKV_DEVERR_TIMEOUT);
      // the last tiles' copies must land before shared memory is released
      for (int j = max(0, n_tiles - kTcStages); j < n_tiles; ++j) mbar_wait(&full[j % kTcStages], (j / kTcStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------- MMA issuer ----------------------------
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16_f32(kRows, kTileTokens, false, false);
      constexpr uint32_t kIdO = tc::idesc_bf16_f32(kRows, kHeadDim, false, true);
      // Two cursors: S_js needs its K tile and its buffer back (the P.V that
      // last read it done), P.V_jp needs P_jp.  The thread polls both and
      // issues whichever is ready, so neither waits behind the other.
      int js = 0, jp = 0;
      uint64_t t_idle = 0;
      ok = mbar_wait(&bars->q_full, 0);  // Q staged while the first K/V tiles are in flight
      while (ok && jp < n_tiles) {
        bool progressed = false;
        if (js < n_tiles) {
          const int st = js % kTcStages, sb = js % kNB;
          bool ready = mbar_test_wait(&bars->k_full[st], (js / kTcStages) & 1);
          if (ready && js >= kNB) ready = mbar_test_wait(&bars->o_done[sb], ((js / kNB) - 1) & 1);
          if (ready) {
            tc::fence_after_sync();
            const uint32_t kst = sbase + kOffK + st * kStageBytesTc;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t qa = sbase + kOffQ + (kk >> 2) * 8192 + 32 * (kk & 3);
              const uint32_t ka = kst + (kk >> 2) * kHalfBytes + 32 * (kk & 3);
              tc::mma_bf16(tmem + sb * 64, tc::smem_desc(qa, 16, 1024), tc::smem_desc(ka, 16, 1024), kIdS, kk > 0);
            }
            tc::commit(&bars->s_full[sb]);
            tc::commit(&bars->k_empty[st]);
            ++js;
            progressed = true;
          }
        }
        if (jp < js && mbar_test_wait(&bars->p_full[jp % kNB], (jp / kNB) & 1) &&
            mbar_test_wait(&bars->v_full[jp % kTcStages], (jp / kTcStages) & 1)) {
          tc::fence_after_sync();
          const int st = jp % kTcStages;
          // P_jp: 64 BF16 high parts per row packed in 32 columns, then the remainders
          const uint32_t ptm = tmem + (jp % kNB) * 64;
          const uint32_t vst = sbase + kOffV + st * kStageBytesTc;
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_bf16_tmem_a(tmem + kColO, ptm + 32 * part + 8 * kk,
                                  tc::smem_desc(vst + 2048 * kk, kHalfBytes, 1024), kIdO,
                                  (jp > 0 || part > 0 || kk > 0) ? 1u : 0u);
          tc::commit(&bars->o_done[jp % kNB]);
          tc::commit(&bars->v_empty[st]);
          ++jp;
          progressed = true;
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
  } else {
    // ---------------------------- softmax ----------------------------
    {
      // Q rows (position, head) -> 128-byte swizzled K-major tile, two 64-dim
      // halves, staged here rather than before the producer starts so that
      // these loads overlap the first K/V tiles' flight.  Thread t loads
      // 16-byte chunk t % 16 of rows t / 16 + 8k, k < 8, all loads issued
      // before the first store: the (member, query) chain costs two round
      // trips, not eight.
      const int t = threadIdx.x - 64;  // 0..127
      const int ch = t & 15;           // 16-byte chunk of the row
      const uint16_t* qbase = static_cast<const uint16_t*>(a.q);
      constexpr int kPerThread = kRows * 16 / 128;
      uint4 v[kPerThread];
#pragma unroll
      for (int k = 0; k < kPerThread; ++k) {
        const int m = (t >> 4) + 8 * k;
        const int ipm = row_pos(m);
        const int rm = row_req(m);
        v[k] = make_uint4(0, 0, 0, 0);
        if (rm >= 0 && ipm < a.q_len)
          v[k] = *reinterpret_cast<const uint4*>(
              qbase + ((static_cast<int64_t>(rm) * a.q_len + ipm) * hq + kvh * kGroup + (m & 3)) * kHeadDim + ch * 8);
      }
#pragma unroll
      for (int k = 0; k < kPerThread; ++k) {
        const int m = (t >> 4) + 8 * k;
        *reinterpret_cast<uint4*>(smem + kOffQ + (ch >> 3) * 8192 + tc::sw128_offset(m, (ch & 7) * 8)) = v[k];
      }
      tc::fence_proxy_async_smem();
      mbar_arrive(&bars->q_full);
    }
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    // keys this row may see inside this split: causal limit, context, and the
    // split's own block range (the tail tile's extra blocks arrive zero-filled)
    int n_vis_row = 0;
    if (row_valid) {
      const int ctx_r = a.context_lens[rq];
      n_vis_row = min(min(max(ctx_r - a.q_len + 1 + ip, 0), cap), b1 * kBlockSize);
    }
    const float c = a.scale_log2;  // > 0: the max of raw scores scales to the max of scaled ones
    float m_stale = -INFINITY;     // scaled max the weights are taken against (lags the true max by < 2^8)
    float l = 0.f;                 // this thread's half of the row's weight sum
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int sb = j % kNB;
      const int st = j % kTcStages;
      // keep `ok` warp-uniform: the tcgen05 loads below are warp-collective
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (j / kNB) & 1));
      if (!ok) break;
      tc::fence_after_sync();
      float s[32];  // raw scores of tokens half*32 .. half*32+31 of the tile
      tc::tmem_ld16x2_32<32>(tmem + lane_off + sb * 64, s);
      tc::tmem_wait_ld();
      const int tok0 = (b0 + j * kTileBlocks) * kBlockSize + half * 32;
      if (__any_sync(0xffffffffu, tok0 + 32 > n_vis_row)) {
#pragma unroll
        for (int e = 0; e < 32; ++e) s[e] = (tok0 + e < n_vis_row) ? s[e] : -INFINITY;
      }
      float mx;
      {
        float t8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t8[e] = fmaxf(fmaxf(s[e], s[e + 8]), fmaxf(s[e + 16], s[e + 24]));
        mx = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])), fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16)) * c;  // whole row, scaled
      }
      const bool grow = mx > m_stale + kRescaleThreshold;  // also true the first time a row sees a key
      const float m_new = grow ? mx : m_stale;
      const float alpha = grow ? exp2_approx(m_stale - m_new) : 1.f;  // 0 while m_stale is -inf
      if (__any_sync(0xffffffffu, grow && j > 0 && m_stale != -INFINITY)) {
        // O holds weights taken against the old maxima: rescale this warp's rows
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[(j - 1) % kNB], ((j - 1) / kNB) & 1));
        tc::fence_after_sync();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float o[32];
          tc::tmem_ld16x2_32<64>(tmem + lane_off + kColO + 32 * cc, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tc::tmem_st16x2_32<64>(tmem + lane_off + kColO + 32 * cc, o);
        }
        tc::tmem_wait_st();
      }
      l *= alpha;
      m_stale = m_new;
      const float nm = (m_stale == -INFINITY) ? 0.f : -m_stale;
      const float2 c2 = make_float2(c, c);
      const float2 nm2 = make_float2(nm, nm);
      // P_j overwrites the S_j buffer it came from, 2 BF16 per 32-bit column:
      // the weights' BF16 roundings, then the BF16 roundings of what they
      // left out, so P.V carries the weights to about 2^-17 relative
      uint32_t pk[16], pr[16];
      float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 x = __ffma2_rn(make_float2(s[2 * e], s[2 * e + 1]), c2, nm2);
        const float p0 = exp2_approx(x.x);
        const float p1 = exp2_approx(x.y);
        acc2 = __fadd2_rn(acc2, make_float2(p0, p1));
        pk[e] = pack_bf16x2(p0, p1);
        pr[e] = pack_bf16x2(p0 - __uint_as_float(pk[e] << 16), p1 - __uint_as_float(pk[e] & 0xffff0000u));
      }
      tc::tmem_st16x2_16<16>(tmem + lane_off + sb * 64, pk);
      tc::tmem_st16x2_16<16>(tmem + lane_off + sb * 64 + 32, pr);
      l += acc2.x + acc2.y;
      // slots past the request's data in its last block may hold anything: zero those V rows
      const int tile0 = (b0 + j * kTileBlocks) * kBlockSize;
      const int tile_end = tile0 + kTileTokens;
      if (ctx_keys < tile_end && ctx_keys > tile0 && (ctx_keys & (kBlockSize - 1)) != 0) {
        // V(j) may land after S(j): wait for it (its stage cannot move on
        // before this tile's P.V, which waits for these weights)
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (j / kTcStages) & 1));
        const int first = ctx_keys - tile0;                                // first garbage token of the tile
        const int last = min(kTileTokens, ((first + kBlockSize - 1) / kBlockSize) * kBlockSize);
        uint8_t* vt = smem + kOffV + st * kStageBytesTc;
        const int t128 = threadIdx.x - 64;
        for (int idx = t128; idx < (last - first) * 16; idx += 128) {
          const int tk = first + (idx >> 4);
          const int ch = idx & 15;  // 8 chunks in each 64-dim half
          *reinterpret_cast<uint4*>(vt + (ch >> 3) * kHalfBytes + tk * 128 + (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      tc::tmem_wait_st();
      tc::fence_proxy_async_smem();  // zeroed V rows, if any, before the PV MMA reads them
      tc::fence_before_sync();
      mbar_arrive(&bars->p_full[sb]);
    }
    if (!ok && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
    // ---- epilogue: this thread writes dims half*64 .. half*64+63 of its row ----
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[(n_tiles - 1) % kNB], ((n_tiles - 1) / kNB) & 1));
    tc::fence_after_sync();
    const float l_row = l + __shfl_xor_sync(0xffffffffu, l, 16);
    const float inv = (l_row > 0.f) ? 1.f / l_row : 0.f;
    const float lse = (l_row > 0.f) ? (m_stale + log2f(l_row)) * kLn2 : -INFINITY;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      float o[32];
      tc::tmem_ld16x2_32<64>(tmem + lane_off + kColO + 32 * cc, o);  // dims half*64 + 32cc .. +31
      tc::tmem_wait_ld();
      const int d0 = half * 64 + 32 * cc;
      if (row_valid && ok) {
        if constexpr (kSplit) {
          float4* dst = reinterpret_cast<float4*>(a.part_o + slot * kHeadDim + d0);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow * kHeadDim + d0);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = pack_bf16x2(o[8 * e] * inv, o[8 * e + 1] * inv);
            w.y = pack_bf16x2(o[8 * e + 2] * inv, o[8 * e + 3] * inv);
            w.z = pack_bf16x2(o[8 * e + 4] * inv, o[8 * e + 5] * inv);
            w.w = pack_bf16x2(o[8 * e + 6] * inv, o[8 * e + 7] * inv);
            dst[e] = w;
          }
        }
      }
    }
    if constexpr (kSplit) {
      if (row_valid && ok && half == 0) a.part_lse[slot] = lse;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kSplit>
__global__ void __launch_bounds__(kTcThreads, 2)
    paged_chunk_tc_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                          const ChunkArgs a) {
  paged_chunk_tc_body<kSplit>(k_map, v_map, a);  // waits for earlier grids after its set-up
}

// ---------------------------------------------------------------------------
// host side: tensor maps over a KV pool viewed as rows of 128 BF16
// ---------------------------------------------------------------------------

template <bool kSplit>
cudaError_t launch_chunk_variant(const CUtensorMap& kmap, const CUtensorMap& vmap, const ChunkArgs& a, dim3 grid,
                                 cudaStream_t stream) {
  static std::atomic<bool> done[64];  // per device; host threads may race on a first call
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    e = cudaFuncSetAttribute(paged_chunk_tc_kernel<kSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return launch_pdl(paged_chunk_tc_kernel<kSplit>, grid, dim3(kTcThreads), kSmemTc, stream, 1, kmap, vmap, a);
}

}  // namespace

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_pool_map(CUtensorMap* map, const void* pool, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim * 2)};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlockSize)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_pool_map_e4m3(CUtensorMap* map, const void* pool, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(kBlockSize)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_paged_chunk_tc(const ChunkArgs& a, int32_t grid_x, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.num_blocks) * a.num_kv_heads * kBlockSize;
  if (rows + kBlockSize >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  CUtensorMap kmap, vmap;
  if (!make_pool_map(&kmap, a.k_cache, rows) || !make_pool_map(&vmap, a.v_cache, rows)) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(grid_x), static_cast<unsigned>(a.num_splits),
                  static_cast<unsigned>(a.num_kv_heads));
  if (grid.x == 0) return cudaSuccess;
  // partials to the workspace (splits, or a cascade prefix pass), or BF16 out
  return a.part_o != nullptr ? launch_chunk_variant<true>(kmap, vmap, a, grid, stream)
                             : launch_chunk_variant<false>(kmap, vmap, a, grid, stream);
}

}  // namespace pkv
