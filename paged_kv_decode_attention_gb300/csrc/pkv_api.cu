// pkv_api.cu -- the exported C ABI of libpkv (declared in include/pkv.h).
//
// Host side only: argument validation, the split-KV heuristic, workspace
// carving and stream-ordered launches.  Nothing here allocates, frees or
// synchronises device memory (except pkv_get_device_error, which reads the
// error word and documents that it synchronises).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "pkv.h"
#include "pkv_common.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

// Device error word (PKV_DEVERR_* bits); one per device that loads the library.
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
// Per-device caches, filled on first use.  Host threads may race on a first
// use: each computes the same value and the stores are atomic.
std::atomic<unsigned int*> g_error_ptr[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];

}  // namespace

// Address of this device's error word, looked up once per device (with that
// device current, as cudaGetSymbolAddress requires).
unsigned int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned int* w = g_error_ptr[dev].load(std::memory_order_acquire);
  if (w == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    w = static_cast<unsigned int*>(p);
    g_error_ptr[dev].store(w, std::memory_order_release);
  }
  return w;
}

namespace {

unsigned int* error_word() { return device_error_word(); }

// SM count assumed when no device can be queried (host-only sizing): GB300.
constexpr int kGb300Sms = 152;

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kGb300Sms;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kGb300Sms;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

pkv_status check_cache(const pkv_cache_desc* c) {
  if (c == nullptr) return PKV_ERR_NULL;
  if (c->num_blocks < 0 || c->num_kv_heads <= 0) return PKV_ERR_SHAPE;
  if (c->block_size != kBlockSize || c->head_dim != kHeadDim) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Splits are made only when the un-split grid would leave the GPU
// under-filled: the decode kernel keeps 2 CTAs per SM busy, and one full wave
// of long-running CTAs beats several waves of short ones (each CTA pays a
// pipeline fill).  Each split keeps at least 16 blocks (256 tokens).
constexpr int kMinBlocksPerSplit = 16;
constexpr int kResidentCtasPerSm = 2;
constexpr int kTcMinBlocksPerSplit = 128;

// Decode batches with at least this many (request, KV head) rows per SM run
// on the persistent tensor-core kernel: with two CTAs per SM already busy,
// one CTA streaming 192 KiB of tiles per SM wastes less on per-CTA fill and
// drain (measured: 64 x 32K tokens 0.98 vs 0.88 of the HBM peak, 512 x 512
// 0.89 vs 0.80).
constexpr int kTcDecodeRowsPerSm = 2;
// Smaller batches go there too when the CTA-per-row kernel's one wave would
// leave more than a tenth of its slots (2 CTAs per SM) empty -- its CTAs each
// stream at a fixed rate, so empty slots are lost bandwidth -- provided there
// are at least 3/4 of a row per SM and requests of at least 128 blocks, where
// the persistent kernel's larger fixed cost is paid back.  Measured (fraction
// of the HBM peak, CTA-per-row vs persistent): 24 x 8K tokens 0.66 vs 0.89,
// 16 x 16K 0.91 vs 0.94, 32 x 32K 0.91 vs 1.01; 8 x 8K (a quarter row per SM)
// 0.77 vs 0.77; 37 x 2K (97 % of the slots filled) 0.86 vs 0.81.
constexpr int kTcDecodeMinBlocks = 128;

// Blocks per split of the CTA-per-row decode kernel: splits are made only
// when the un-split grid would leave the GPU under-filled, as many as fit in
// one wave -- a few CTAs spilling into a second wave would double the call's
// time -- each of at least kMinBlocksPerSplit blocks.
int32_t row_kernel_blocks_per_split(int64_t rows, int32_t max_blocks_per_seq, int32_t sm_count) {
  const int64_t slots = static_cast<int64_t>(kResidentCtasPerSm) * sm_count;
  if (rows <= 0 || max_blocks_per_seq <= kMinBlocksPerSplit) return max_blocks_per_seq;
  const int64_t splits = slots / rows;
  if (splits <= 1) return max_blocks_per_seq;
  int64_t bps = (max_blocks_per_seq + splits - 1) / splits;
  if (bps < kMinBlocksPerSplit) bps = kMinBlocksPerSplit;
  if (bps > max_blocks_per_seq) bps = max_blocks_per_seq;
  return static_cast<int32_t>(bps);
}

bool decode_on_tensor_cores(int64_t num_seqs, int64_t num_kv_heads, int32_t q_len, int32_t max_blocks_per_seq,
                            int sm_count) {
  if (q_len != 1) return false;
  const int64_t rows = num_seqs * num_kv_heads;
  if (rows >= static_cast<int64_t>(kTcDecodeRowsPerSm) * sm_count) return true;
  if (4 * rows < 3 * static_cast<int64_t>(sm_count) || max_blocks_per_seq < kTcDecodeMinBlocks) return false;
  const int32_t bps = row_kernel_blocks_per_split(rows, max_blocks_per_seq, sm_count);
  const int64_t ctas = rows * ((max_blocks_per_seq + bps - 1) / bps);
  return 10 * ctas < 9 * static_cast<int64_t>(kResidentCtasPerSm) * sm_count;
}

// Split size for the persistent kernels (one CTA per SM walking units of
// 8-block tiles): minimise the makespan -- the busiest CTA runs
// ceil(units / SMs) units, each costing its tiles plus about one tile of
// pipeline fill and epilogue -- with 2 tiles charged for the combine pass.
int32_t persistent_blocks_per_split(int64_t rows, int32_t max_blocks_per_seq, int32_t sm_count,
                                    int32_t tile_blocks = 8) {
  int32_t best = max_blocks_per_seq;
  int64_t best_cost = INT64_MAX;
  for (int32_t splits = 1; splits <= 64; ++splits) {
    int32_t bps = (max_blocks_per_seq + splits - 1) / splits;
    bps = (bps + tile_blocks - 1) / tile_blocks * tile_blocks;
    if (splits > 1 && bps < 2 * tile_blocks) break;
    if (bps > max_blocks_per_seq) bps = max_blocks_per_seq;
    const int64_t s_eff = (max_blocks_per_seq + bps - 1) / bps;
    const int64_t units = rows * s_eff;
    const int64_t per_cta = (units + sm_count - 1) / sm_count;
    // in tiles: the unit's tiles plus about one tile of set-up and drain, and
    // the combine pass when there is more than one split
    const int64_t cost = per_cta * ((bps + tile_blocks - 1) / tile_blocks + 1) + (s_eff > 1 ? 2 : 0);
    if (cost < best_cost) {
      best_cost = cost;
      best = bps;
    }
  }
  return best;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_NULL: return "PKV_ERR_NULL: a required pointer is NULL";
    case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE: a size is negative or inconsistent";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: shape not supported (block_size 16, head_dim 128, GQA 4)";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: split-KV workspace missing or too small";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA runtime call failed";
    case PKV_ERR_EXHAUSTED: return "PKV_ERR_EXHAUSTED: not enough free blocks in the pool";
  }
  return "unknown pkv_status";
}

pkv_status pkv_kv_append(void* k_cache, void* v_cache, const pkv_cache_desc* cache, const int64_t* slot_mapping,
                         const void* k_new, const void* v_new, int32_t num_tokens, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k_cache || !v_cache || !slot_mapping || !k_new || !v_new) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return PKV_ERR_UNSUPPORTED;
  unsigned int* err = error_word();
  cudaError_t e = launch_kv_append(k_cache, v_cache, cache->num_blocks, cache->num_kv_heads, slot_mapping,
                                   k_new, v_new, num_tokens, err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int32_t pkv_choose_kv_blocks_per_split(int32_t num_seqs, int32_t num_kv_heads, int32_t q_len,
                                       int32_t max_blocks_per_seq, int32_t sm_count) {
  if (max_blocks_per_seq <= 0) return 1;
  if (q_len >= kTcMinQLen) {
    // tensor-core chunk kernel: cap each CTA at ~1/8 of the longest request
    // (and never below 2048 tokens) so one long request cannot form the tail
    if (max_blocks_per_seq <= kTcMinBlocksPerSplit) return max_blocks_per_seq;
    int32_t bps = (max_blocks_per_seq + 7) / 8;
    return bps < kTcMinBlocksPerSplit ? kTcMinBlocksPerSplit : bps;
  }
  if (sm_count <= 0) sm_count = device_sm_count();
  const int64_t rows = static_cast<int64_t>(num_seqs) * (q_len > 0 ? q_len : 1) * num_kv_heads;
  if (decode_on_tensor_cores(num_seqs, num_kv_heads, q_len, max_blocks_per_seq, sm_count))
    return persistent_blocks_per_split(rows, max_blocks_per_seq, sm_count);
  return row_kernel_blocks_per_split(rows, max_blocks_per_seq, sm_count);
}

size_t pkv_workspace_size(int32_t num_seqs, int32_t q_len, int32_t num_q_heads, int32_t head_dim,
                          int32_t max_blocks_per_seq, int32_t kv_blocks_per_split) {
  if (num_seqs <= 0 || q_len <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
      kv_blocks_per_split <= 0 || kv_blocks_per_split >= max_blocks_per_seq)
    return 0;
  const size_t splits = (static_cast<size_t>(max_blocks_per_seq) + kv_blocks_per_split - 1) / kv_blocks_per_split;
  if (q_len < kTcMinQLen && splits <= static_cast<size_t>(kMaxClusterSplits) &&
      !decode_on_tensor_cores(num_seqs, num_q_heads / kGroup, q_len, max_blocks_per_seq, device_sm_count()))
    return 0;  // decode splits merge inside a thread-block cluster
  const size_t rows = static_cast<size_t>(num_seqs) * q_len * num_q_heads;
  return align_up(rows * splits * head_dim * sizeof(float), 256) + align_up(rows * splits * sizeof(float), 256);
}

}  // extern "C"

namespace {

// pkv_paged_attention's checks and launches.  fused (optional): the append
// fused into the CTA-per-row decode kernel (q_len 1; the caller has checked
// that this kernel runs).  dry_run: every check, no launch.
struct FusedAppend {
  const int64_t* slot_mapping;
  const void* k_new;
  const void* v_new;
};

pkv_status paged_attention_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                                const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                float scale, int32_t kv_blocks_per_split, void* workspace, size_t workspace_bytes,
                                void* stream, const FusedAppend* fused, bool dry_run) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || q_len < 1 || max_blocks_per_seq < 1 || kv_blocks_per_split < 0) return PKV_ERR_SHAPE;
  if (num_q_heads != kGroup * cache->num_kv_heads) return PKV_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return PKV_ERR_SHAPE;
  if (static_cast<int64_t>(num_seqs) * q_len > 0x7fffffff || cache->num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return PKV_ERR_UNSUPPORTED;

  int32_t bps = kv_blocks_per_split;
  if (bps == 0)
    bps = pkv_choose_kv_blocks_per_split(num_seqs, cache->num_kv_heads, q_len, max_blocks_per_seq, 0);
  if (bps > max_blocks_per_seq) bps = max_blocks_per_seq;
  const int32_t splits = (max_blocks_per_seq + bps - 1) / bps;
  if (splits > 65535) return PKV_ERR_UNSUPPORTED;

  DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.err = error_word();
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = cache->num_blocks;
  a.num_kv_heads = cache->num_kv_heads;
  a.num_seqs = num_seqs;
  a.q_len = q_len;
  a.blocks_per_split = bps;
  a.num_splits = splits;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.part_slots = splits;
  a.part_slot0 = 0;
  if (fused != nullptr) {
    a.slot_mapping = fused->slot_mapping;
    a.k_new = fused->k_new;
    a.v_new = fused->v_new;
  }
  const int32_t tc_grid_x = num_seqs * ((q_len + 15) / 16);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = device_sm_count();
  if (decode_on_tensor_cores(num_seqs, cache->num_kv_heads, q_len, max_blocks_per_seq, sms)) {
    const int64_t units = static_cast<int64_t>(num_seqs) * cache->num_kv_heads * splits;
    if (units > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    const int32_t grid = static_cast<int32_t>(units < sms ? units : sms);
    if (splits == 1) {
      if (dry_run) return PKV_OK;
      return launch_paged_decode_tc(a, grid, s) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
    }
    const size_t need = pkv_workspace_size(num_seqs, 1, num_q_heads, kHeadDim, max_blocks_per_seq, bps);
    if (workspace == nullptr || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_WORKSPACE;
    if (dry_run) return PKV_OK;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                          align_up(rows * splits * kHeadDim * sizeof(float), 256));
    if (launch_paged_decode_tc(a, grid, s) != cudaSuccess) return PKV_ERR_CUDA;
    return launch_attn_combine(out, nullptr, a.part_o, a.part_lse, static_cast<int32_t>(rows), splits, s) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
  }
  const bool tensor_cores = q_len >= kTcMinQLen;
  if (splits > kMaxClusterSplits || (tensor_cores && splits > 1)) {
    const size_t need = pkv_workspace_size(num_seqs, q_len, num_q_heads, kHeadDim, max_blocks_per_seq, bps);
    if (workspace == nullptr || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_WORKSPACE;
    if (dry_run) return PKV_OK;
    const size_t rows = static_cast<size_t>(num_seqs) * q_len * num_q_heads;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                          align_up(rows * splits * kHeadDim * sizeof(float), 256));
    if ((tensor_cores ? launch_paged_chunk_tc(a, tc_grid_x, s) : launch_paged_decode(a, s)) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (launch_attn_combine(out, nullptr, a.part_o, a.part_lse, static_cast<int32_t>(rows), splits, s) != cudaSuccess)
      return PKV_ERR_CUDA;
    return PKV_OK;
  }
  if (dry_run) return PKV_OK;
  return (tensor_cores ? launch_paged_chunk_tc(a, tc_grid_x, s) : launch_paged_decode(a, s)) == cudaSuccess ? PKV_OK
                                                                                                 : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                               float scale, int32_t kv_blocks_per_split, void* workspace, size_t workspace_bytes,
                               void* stream) {
  return paged_attention_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                              num_seqs, q_len, num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes,
                              stream, nullptr, false);
}

pkv_status pkv_paged_attention_append(void* out, const void* q, void* k_cache, void* v_cache,
                                      const pkv_cache_desc* cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                      int32_t q_len, int32_t num_q_heads, float scale, int32_t kv_blocks_per_split,
                                      void* workspace, size_t workspace_bytes, const int64_t* slot_mapping,
                                      const void* k_new, const void* v_new, int32_t num_tokens, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens > 0) {
    if (!k_cache || !v_cache || !slot_mapping || !k_new || !v_new) return PKV_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15) return PKV_ERR_UNSUPPORTED;
  }
  // every check of the attention first, so an error enqueues nothing
  st = paged_attention_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                            num_seqs, q_len, num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes,
                            stream, nullptr, true);
  if (st != PKV_OK) return st;
  // one launch when each request appends its one new token and the decode
  // runs on the CTA-per-row kernel; otherwise the append, then the attention
  const bool fuse = q_len == 1 && num_tokens == num_seqs && num_seqs > 0 &&
                    !decode_on_tensor_cores(num_seqs, cache->num_kv_heads, 1, max_blocks_per_seq, device_sm_count());
  if (fuse) {
    const FusedAppend f{slot_mapping, k_new, v_new};
    return paged_attention_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                                num_seqs, q_len, num_q_heads, scale, kv_blocks_per_split, workspace,
                                workspace_bytes, stream, &f, false);
  }
  if (num_tokens > 0) {
    st = pkv_kv_append(k_cache, v_cache, cache, slot_mapping, k_new, v_new, num_tokens, stream);
    if (st != PKV_OK) return st;
  }
  return paged_attention_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                              num_seqs, q_len, num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes,
                              stream, nullptr, false);
}

void pkv_cascade_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t num_groups, int32_t max_prefix_blocks,
                      int32_t max_suffix_blocks, int32_t sm_count, int32_t* prefix_blocks_per_split,
                      int32_t* suffix_blocks_per_split) {
  if (sm_count <= 0) sm_count = device_sm_count();
  // prefix pass: about a third of the SMs' worth of (group, split, head)
  // CTAs.  The suffix pass runs beside it and needs the rest: an SM holding a
  // tensor-core CTA has room for one decode CTA only, so many short prefix
  // CTAs would crowd the suffix out, and few long ones would finish last.
  int32_t pbps = max_prefix_blocks > 0 ? max_prefix_blocks : 1;
  const int64_t prows = static_cast<int64_t>(num_groups > 0 ? num_groups : 1) * num_kv_heads;
  const int64_t target = (sm_count + 2) / 3;
  if (max_prefix_blocks > 0 && prows < target) {
    const int64_t sp = (target + prows / 2) / prows;
    pbps = static_cast<int32_t>((max_prefix_blocks + sp - 1) / sp);
    pbps = ((pbps + 3) / 4) * 4;  // whole 4-block tiles
    if (pbps < 16) pbps = 16;
  }
  // suffix pass: the CTA-per-row decode kernel's split over the longest suffix
  const int32_t span = max_suffix_blocks > 0 ? max_suffix_blocks : 1;
  int32_t sbps = row_kernel_blocks_per_split(static_cast<int64_t>(num_seqs) * num_kv_heads, span, sm_count);
  if (prefix_blocks_per_split) *prefix_blocks_per_split = pbps;
  if (suffix_blocks_per_split) *suffix_blocks_per_split = sbps;
}

static int32_t ceil_div(int32_t a, int32_t b) { return (a + b - 1) / b; }

size_t pkv_cascade_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t max_prefix_blocks,
                                  int32_t max_suffix_blocks, int32_t prefix_blocks_per_split,
                                  int32_t suffix_blocks_per_split) {
  if (num_seqs <= 0 || num_q_heads <= 0 || max_suffix_blocks <= 0 || prefix_blocks_per_split <= 0 ||
      suffix_blocks_per_split <= 0)
    return 0;
  // the suffix pass merges on chip (and folds in the prefix partials) when it
  // needs at most kMaxClusterSplits splits; only then does it need no slots
  const int32_t ss = ceil_div(max_suffix_blocks, suffix_blocks_per_split);
  const size_t slots = static_cast<size_t>(max_prefix_blocks > 0 ? ceil_div(max_prefix_blocks, prefix_blocks_per_split) : 0) +
                       (ss > kMaxClusterSplits ? ss : 0);
  if (slots == 0) return 0;
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
  return align_up(rows * slots * kHeadDim * sizeof(float), 256) + align_up(rows * slots * sizeof(float), 256);
}

}  // extern "C"

namespace {

// pkv_paged_attention_cascade's checks and launches; fused and dry_run as for
// paged_attention_impl (the suffix pass always runs on the CTA-per-row kernel).
pkv_status cascade_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, float scale,
                        const int32_t* group_seqs, const int32_t* group_blocks, const int32_t* seq_prefix_blocks,
                        int32_t num_groups, int32_t max_prefix_blocks, int32_t max_suffix_blocks,
                        int32_t prefix_blocks_per_split, int32_t suffix_blocks_per_split, void* workspace,
                        size_t workspace_bytes, void* stream, const FusedAppend* fused, bool dry_run) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_blocks_per_seq < 1 || num_groups < 0 || max_prefix_blocks < 0 ||
      max_prefix_blocks > max_blocks_per_seq || max_suffix_blocks < 0 || max_suffix_blocks > max_blocks_per_seq ||
      prefix_blocks_per_split < 0 || suffix_blocks_per_split < 0)
    return PKV_ERR_SHAPE;
  if (max_suffix_blocks == 0) max_suffix_blocks = max_blocks_per_seq;
  if (num_q_heads != kGroup * cache->num_kv_heads) return PKV_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !seq_prefix_blocks) return PKV_ERR_NULL;
  if (num_groups > 0 && (!group_seqs || !group_blocks)) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return PKV_ERR_UNSUPPORTED;
  int32_t pbps = prefix_blocks_per_split, sbps = suffix_blocks_per_split;
  if (pbps == 0 || sbps == 0) {
    int32_t p0 = 0, s0 = 0;
    pkv_cascade_plan(num_seqs, cache->num_kv_heads, num_groups, max_prefix_blocks, max_suffix_blocks, 0, &p0, &s0);
    if (pbps == 0) pbps = p0;
    if (sbps == 0) sbps = s0;
  }
  const int32_t sp = (num_groups > 0 && max_prefix_blocks > 0) ? ceil_div(max_prefix_blocks, pbps) : 0;
  const int32_t ss = ceil_div(max_suffix_blocks, sbps);
  if (sp > 65535 || ss > 65535) return PKV_ERR_UNSUPPORTED;
  const size_t need = pkv_cascade_workspace_size(num_seqs, num_q_heads, max_prefix_blocks, max_suffix_blocks, pbps, sbps);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return PKV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_WORKSPACE;
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
  const bool on_chip = ss <= kMaxClusterSplits;  // suffix merges in a cluster and folds in the prefix
  const int32_t slots = sp + (on_chip ? 0 : ss);

  DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.err = error_word();
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = cache->num_blocks;
  a.num_kv_heads = cache->num_kv_heads;
  a.num_seqs = num_seqs;
  a.q_len = 1;
  a.scale_log2 = scale * 1.4426950408889634f;
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = slots > 0 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                         align_up(rows * slots * kHeadDim * sizeof(float), 256))
                              : nullptr;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.part_slots = slots;
  if (dry_run) return PKV_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (sp > 0) {
    // shared prefixes: each group's members x 4 heads as one 64-row tensor-core tile
    DecodeArgs p = a;
    p.blocks_per_split = pbps;
    p.num_splits = sp;
    p.part_slot0 = 0;
    p.group_seqs = group_seqs;
    p.group_blocks = group_blocks;
    if (launch_paged_chunk_tc(p, num_groups, s) != cudaSuccess) return PKV_ERR_CUDA;
  }
  // private suffixes (and requests outside every group) on the decode kernel
  a.blocks_per_split = sbps;
  a.num_splits = ss;
  a.seq_start_block = seq_prefix_blocks;
  a.overlap_previous = sp > 0 ? 1 : 0;  // the suffix pass runs beside the prefix pass
  if (fused != nullptr) {  // the new tokens lie in the suffixes: the suffix pass stores them
    a.slot_mapping = fused->slot_mapping;
    a.k_new = fused->k_new;
    a.v_new = fused->v_new;
  }
  if (on_chip) {
    // direct (one split) or cluster merge, folding in the prefix partials: no combine kernel
    a.part_o = nullptr;
    a.part_lse = nullptr;
    a.part_slots = 0;
    a.part_slot0 = 0;
    if (sp > 0) {
      a.prefix_o = part_o;
      a.prefix_lse = part_lse;
      a.prefix_slots = sp;
    }
    return launch_paged_decode(a, s) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
  a.part_slot0 = sp;
  if (launch_paged_decode_workspace(a, s) != cudaSuccess) return PKV_ERR_CUDA;
  if (launch_attn_combine(out, nullptr, a.part_o, a.part_lse, static_cast<int32_t>(rows), slots, s) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_cascade(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const pkv_cache_desc* cache, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                       int32_t num_q_heads, float scale, const int32_t* group_seqs,
                                       const int32_t* group_blocks, const int32_t* seq_prefix_blocks,
                                       int32_t num_groups, int32_t max_prefix_blocks, int32_t max_suffix_blocks,
                                       int32_t prefix_blocks_per_split, int32_t suffix_blocks_per_split,
                                       void* workspace, size_t workspace_bytes, void* stream) {
  return cascade_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                      num_q_heads, scale, group_seqs, group_blocks, seq_prefix_blocks, num_groups, max_prefix_blocks,
                      max_suffix_blocks, prefix_blocks_per_split, suffix_blocks_per_split, workspace,
                      workspace_bytes, stream, nullptr, false);
}

pkv_status pkv_paged_attention_cascade_append(
    void* out, const void* q, void* k_cache, void* v_cache, const pkv_cache_desc* cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, float scale,
    const int32_t* group_seqs, const int32_t* group_blocks, const int32_t* seq_prefix_blocks, int32_t num_groups,
    int32_t max_prefix_blocks, int32_t max_suffix_blocks, int32_t prefix_blocks_per_split,
    int32_t suffix_blocks_per_split, void* workspace, size_t workspace_bytes, const int64_t* slot_mapping,
    const void* k_new, const void* v_new, int32_t num_tokens, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens > 0) {
    if (!k_cache || !v_cache || !slot_mapping || !k_new || !v_new) return PKV_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15) return PKV_ERR_UNSUPPORTED;
  }
  // every check of the attention first, so an error enqueues nothing
  st = cascade_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                    num_q_heads, scale, group_seqs, group_blocks, seq_prefix_blocks, num_groups, max_prefix_blocks,
                    max_suffix_blocks, prefix_blocks_per_split, suffix_blocks_per_split, workspace, workspace_bytes,
                    stream, nullptr, true);
  if (st != PKV_OK) return st;
  if (num_tokens == num_seqs && num_seqs > 0) {
    const FusedAppend f{slot_mapping, k_new, v_new};
    return cascade_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                        num_q_heads, scale, group_seqs, group_blocks, seq_prefix_blocks, num_groups,
                        max_prefix_blocks, max_suffix_blocks, prefix_blocks_per_split, suffix_blocks_per_split,
                        workspace, workspace_bytes, stream, &f, false);
  }
  if (num_tokens > 0) {
    st = pkv_kv_append(k_cache, v_cache, cache, slot_mapping, k_new, v_new, num_tokens, stream);
    if (st != PKV_OK) return st;
  }
  return cascade_impl(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                      num_q_heads, scale, group_seqs, group_blocks, seq_prefix_blocks, num_groups, max_prefix_blocks,
                      max_suffix_blocks, prefix_blocks_per_split, suffix_blocks_per_split, workspace,
                      workspace_bytes, stream, nullptr, false);
}

pkv_status pkv_kv_append_q8_0(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                              const int64_t* slot_mapping, const void* k_new, const void* v_new, int32_t num_tokens,
                              void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k_cache || !v_cache || !slot_mapping || !k_new || !v_new) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return PKV_ERR_UNSUPPORTED;
  return launch_kv_append_q8(k_cache, v_cache, cache->num_blocks, cache->num_kv_heads, slot_mapping, k_new, v_new,
                             num_tokens, error_word(), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

int32_t pkv_choose_kv_blocks_per_split_q8_0(int32_t num_seqs, int32_t num_kv_heads, int32_t max_blocks_per_seq,
                                            int32_t sm_count) {
  if (max_blocks_per_seq <= 0) return 1;
  if (sm_count <= 0) sm_count = device_sm_count();
  const int64_t rows = static_cast<int64_t>(num_seqs > 0 ? num_seqs : 1) * (num_kv_heads > 0 ? num_kv_heads : 1);
  return persistent_blocks_per_split(rows, max_blocks_per_seq, sm_count);
}

int32_t pkv_choose_kv_blocks_per_split_fp8_e4m3(int32_t num_seqs, int32_t num_kv_heads, int32_t max_blocks_per_seq,
                                                int32_t sm_count) {
  if (max_blocks_per_seq <= 0) return 1;
  if (sm_count <= 0) sm_count = device_sm_count();
  const int64_t rows = static_cast<int64_t>(num_seqs > 0 ? num_seqs : 1) * (num_kv_heads > 0 ? num_kv_heads : 1);
  return persistent_blocks_per_split(rows, max_blocks_per_seq, sm_count, 16);
}

size_t pkv_workspace_size_q8_0(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                               int32_t kv_blocks_per_split) {
  if (num_seqs <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || kv_blocks_per_split <= 0 ||
      kv_blocks_per_split >= max_blocks_per_seq)
    return 0;
  const size_t splits = (static_cast<size_t>(max_blocks_per_seq) + kv_blocks_per_split - 1) / kv_blocks_per_split;
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
  return align_up(rows * splits * kHeadDim * sizeof(float), 256) + align_up(rows * splits * sizeof(float), 256);
}

}  // extern "C"

namespace {

// Decode over quantised pools (q8_0, or E4M3 when fp8): validation, split
// choice, workspace carving, the decode kernel and the combine pass.
pkv_status quantised_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, float scale,
                               int32_t kv_blocks_per_split, void* workspace, size_t workspace_bytes, void* stream,
                               bool fp8, const FusedAppend* fused = nullptr, bool dry_run = false) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_blocks_per_seq < 1 || kv_blocks_per_split < 0) return PKV_ERR_SHAPE;
  if (num_q_heads != kGroup * cache->num_kv_heads) return PKV_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * kBlockSize > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
  int32_t bps = kv_blocks_per_split;
  if (bps == 0)
    bps = fp8 ? pkv_choose_kv_blocks_per_split_fp8_e4m3(num_seqs, cache->num_kv_heads, max_blocks_per_seq, 0)
              : pkv_choose_kv_blocks_per_split_q8_0(num_seqs, cache->num_kv_heads, max_blocks_per_seq, 0);
  if (bps > max_blocks_per_seq) bps = max_blocks_per_seq;
  const int32_t splits = (max_blocks_per_seq + bps - 1) / bps;
  const int64_t units = static_cast<int64_t>(num_seqs) * cache->num_kv_heads * splits;
  if (units > 0x7fffffff) return PKV_ERR_UNSUPPORTED;

  DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.err = error_word();
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = cache->num_blocks;
  a.num_kv_heads = cache->num_kv_heads;
  a.num_seqs = num_seqs;
  a.q_len = 1;
  a.blocks_per_split = bps;
  a.num_splits = splits;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.part_slots = splits;
  if (fused != nullptr) {  // the decode kernel stores the new tokens
    a.slot_mapping = fused->slot_mapping;
    a.k_new = fused->k_new;
    a.v_new = fused->v_new;
  }
  const int sms = device_sm_count();
  const int32_t grid = static_cast<int32_t>(units < sms ? units : sms);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // E4M3 tiles feed the tensor cores' 8-bit path as they are; q8_0 codes are
  // dequantised inside the kernel
  auto launch = [&]() {
    return fp8 ? launch_paged_decode_fp8_tc(a, grid, s) : launch_paged_decode_q8(a, grid, s);
  };
  if (splits == 1) {
    if (dry_run) return PKV_OK;
    return launch() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
  const size_t need = pkv_workspace_size_q8_0(num_seqs, num_q_heads, max_blocks_per_seq, bps);
  if (workspace == nullptr || workspace_bytes < need) return PKV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_WORKSPACE;
  if (dry_run) return PKV_OK;
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        align_up(rows * splits * kHeadDim * sizeof(float), 256));
  if (launch() != cudaSuccess) return PKV_ERR_CUDA;
  return launch_attn_combine(out, nullptr, a.part_o, a.part_lse, static_cast<int32_t>(rows), splits, s) ==
                 cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_q8_0(void* out, const void* q, const void* k_cache, const void* v_cache,
                                    const pkv_cache_desc* cache, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                    int32_t num_q_heads, float scale, int32_t kv_blocks_per_split, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  return quantised_attention(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                             num_seqs, num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes, stream,
                             false);
}

pkv_status pkv_paged_attention_fp8_e4m3(void* out, const void* q, const void* k_cache, const void* v_cache,
                                        const pkv_cache_desc* cache, const int32_t* block_tables,
                                        int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                        int32_t num_q_heads, float scale, int32_t kv_blocks_per_split,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  return quantised_attention(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                             num_seqs, num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes, stream,
                             true);
}

}  // extern "C"

namespace {

// The quantising append and the decode over a quantised cache as one call:
// one launch when token r is request r's new token, else the append, then
// the attention.  Every check runs before anything is enqueued.
pkv_status quantised_attention_append(void* out, const void* q, void* k_cache, void* v_cache,
                                      const pkv_cache_desc* cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                      int32_t num_q_heads, float scale, int32_t kv_blocks_per_split, void* workspace,
                                      size_t workspace_bytes, const int64_t* slot_mapping, const void* k_new,
                                      const void* v_new, int32_t num_tokens, void* stream, bool fp8) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens > 0) {
    if (!k_cache || !v_cache || !slot_mapping || !k_new || !v_new) return PKV_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
         reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
      return PKV_ERR_UNSUPPORTED;
  }
  st = quantised_attention(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                           num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes, stream, fp8, nullptr,
                           true);
  if (st != PKV_OK) return st;
  if (num_tokens == num_seqs && num_seqs > 0) {
    const FusedAppend f{slot_mapping, k_new, v_new};
    return quantised_attention(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                               num_seqs, num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes, stream,
                               fp8, &f, false);
  }
  if (num_tokens > 0) {
    st = fp8 ? pkv_kv_append_fp8_e4m3(k_cache, v_cache, cache, slot_mapping, k_new, v_new, num_tokens, stream)
             : pkv_kv_append_q8_0(k_cache, v_cache, cache, slot_mapping, k_new, v_new, num_tokens, stream);
    if (st != PKV_OK) return st;
  }
  return quantised_attention(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                             num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes, stream, fp8);
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_q8_0_append(void* out, const void* q, void* k_cache, void* v_cache,
                                           const pkv_cache_desc* cache, const int32_t* block_tables,
                                           int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                           int32_t num_q_heads, float scale, int32_t kv_blocks_per_split,
                                           void* workspace, size_t workspace_bytes, const int64_t* slot_mapping,
                                           const void* k_new, const void* v_new, int32_t num_tokens, void* stream) {
  return quantised_attention_append(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                                    num_seqs, num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes,
                                    slot_mapping, k_new, v_new, num_tokens, stream, false);
}

pkv_status pkv_paged_attention_fp8_e4m3_append(void* out, const void* q, void* k_cache, void* v_cache,
                                               const pkv_cache_desc* cache, const int32_t* block_tables,
                                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                                               int32_t num_seqs, int32_t num_q_heads, float scale,
                                               int32_t kv_blocks_per_split, void* workspace, size_t workspace_bytes,
                                               const int64_t* slot_mapping, const void* k_new, const void* v_new,
                                               int32_t num_tokens, void* stream) {
  return quantised_attention_append(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                                    num_seqs, num_q_heads, scale, kv_blocks_per_split, workspace, workspace_bytes,
                                    slot_mapping, k_new, v_new, num_tokens, stream, true);
}

pkv_status pkv_kv_append_fp8_e4m3(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                                  const int64_t* slot_mapping, const void* k_new, const void* v_new,
                                  int32_t num_tokens, void* stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k_cache || !v_cache || !slot_mapping || !k_new || !v_new) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return PKV_ERR_UNSUPPORTED;
  return launch_kv_append_fp8(k_cache, v_cache, cache->num_blocks, cache->num_kv_heads, slot_mapping, k_new, v_new,
                              num_tokens, error_word(), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

pkv_status pkv_attn_combine(void* out, float* out_lse, const float* partial_o, const float* partial_lse,
                            int32_t num_rows, int32_t head_dim, int32_t num_splits, void* stream) {
  if (num_rows < 0 || num_splits < 1) return PKV_ERR_SHAPE;
  if (head_dim != kHeadDim) return PKV_ERR_UNSUPPORTED;
  if (num_rows == 0) return PKV_OK;
  if (!out || !partial_o || !partial_lse) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(out) & 7) || (reinterpret_cast<uintptr_t>(partial_o) & 15) ||
      (reinterpret_cast<uintptr_t>(partial_lse) & 3))
    return PKV_ERR_UNSUPPORTED;
  return launch_attn_combine(out, out_lse, partial_o, partial_lse, num_rows, num_splits,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

pkv_status pkv_get_device_error(uint32_t* host_word, int32_t reset) {
  if (host_word == nullptr) return PKV_ERR_NULL;
  unsigned int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return PKV_ERR_CUDA;
  *host_word = v;
  if (reset) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // extern "C"
