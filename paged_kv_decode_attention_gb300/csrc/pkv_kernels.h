// pkv_kernels.h -- host-side launchers of libpkv's kernels (internal).
// The exported C ABI (pkv_api.cu) validates arguments and calls these.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

namespace pkv {

// Launch `kernel` on `stream` with programmatic stream serialization: its
// CTAs may be scheduled while the previous grid in the stream finishes; every
// kernel of this library starts with pdl_wait() before reading any input, so
// results are the same as with a plain launch.  cluster_y > 1 also groups
// the grid's y dimension into thread-block clusters of that size.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       unsigned cluster_y, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_y > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = cluster_y;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Splits of one (row, KV head) up to this count run as one thread-block
// cluster and merge through distributed shared memory (no workspace); more
// splits go through the workspace and the combine kernel.
constexpr int kMaxClusterSplits = 8;

// One decode/split launch: grid (rows, splits, kv heads); see paged_decode.cu.
struct DecodeArgs {
  void* out;                  // BF16 [B][q_len][Hq][D]; written when num_splits == 1
  const void* q;              // BF16 [B][q_len][Hq][D]
  const void* k_cache;        // BF16 [num_blocks][Hkv][16][D]
  const void* v_cache;
  const int32_t* block_tables;  // [B][max_blocks]
  const int32_t* context_lens;  // [B]
  float* part_o;              // FP32 [B*q_len*Hq][num_splits][D]; NULL = cluster merge
  float* part_lse;            // FP32 [B*q_len*Hq][num_splits]
  unsigned int* err;          // device error word
  int32_t max_blocks;
  int32_t num_blocks;
  int32_t num_kv_heads;
  int32_t num_seqs;
  int32_t q_len;
  int32_t blocks_per_split;
  int32_t num_splits;
  float scale_log2;           // scale * log2(e)
  // Workspace slots per row and the first slot this launch writes (split s
  // goes to slot part_slot0 + s); both default to (num_splits, 0).
  int32_t part_slots;
  int32_t part_slot0;
  // Decode: per-request first block (suffix after a shared prefix handled
  // elsewhere); NULL = 0.  Rows whose start is 0 also mark slots
  // [0, part_slot0) empty (-inf) so the combine ignores them.
  const int32_t* seq_start_block;
  // Tensor-core kernel, cascade mode: group g's members are
  // group_seqs[16g .. 16g+15] (-1 = none) and share blocks [0, group_blocks[g]).
  const int32_t* group_seqs;
  const int32_t* group_blocks;
  // Decode in direct or cluster mode for a cascade: the prefix pass's
  // normalised partials (prefix_slots per output row, natural-log lse) are
  // merged into the final result of rows whose request has a prefix.
  const float* prefix_o;
  const float* prefix_lse;
  int32_t prefix_slots;
  // Decode launched right after the cascade's prefix pass: that pass lets
  // the grids after it start only once it has waited for the grids before it,
  // so this decode's inputs are complete when it starts; it starts at once
  // (overlapping the pass) and waits for the pass only before it exits.
  int32_t overlap_previous;
  // Append fused into the decode kernel (q_len 1, CTA-per-row kernel): token
  // r of k_new/v_new ([num_seqs][Hkv][128] BF16) is request r's new token, at
  // position context_lens[r] - 1, stored at slot_mapping[r] (< 0 = not
  // stored).  The CTA whose block range holds that position writes the row
  // into the pools and uses it in place of the tile's stale row.  NULL = no
  // append.
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
};

cudaError_t launch_kv_append(void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                             const int64_t* slot_mapping, const void* k_new, const void* v_new,
                             int32_t num_tokens, unsigned int* err, cudaStream_t stream);

// num_splits == 1: direct; part_o == NULL: cluster merge (num_splits <= kMaxClusterSplits);
// otherwise partials to the workspace (the caller then runs the combine kernel).
cudaError_t launch_paged_decode(const DecodeArgs& a, cudaStream_t stream);
// Always writes split partials to the workspace (any number of splits).
cudaError_t launch_paged_decode_workspace(const DecodeArgs& a, cudaStream_t stream);

// Queries per request at or above which the tensor-core chunk kernel runs
// (16 positions x 4 heads = 64 rows, one tcgen05 M=64 tile).
constexpr int kTcMinQLen = 16;

// Chunked causal attention on tensor cores (paged_chunk_tc.cu).  Same fields
// as DecodeArgs; num_splits > 1 always goes through the workspace.  With
// group_seqs set (cascade mode) the grid's x index is a prefix group, the 64
// rows are its 16 members x 4 heads (q_len 1) and the keys are the group's
// shared prefix blocks, read through the first member's table row.
using ChunkArgs = DecodeArgs;
cudaError_t launch_paged_chunk_tc(const ChunkArgs& a, int32_t grid_x, cudaStream_t stream);

// Tensor map over a BF16 KV pool viewed as `rows` rows of 128 elements, boxes
// of 16 rows x 64 elements with the 128-byte swizzle (paged_chunk_tc.cu).
bool make_pool_map(CUtensorMap* map, const void* pool, int64_t rows);

// Tensor map over an E4M3 KV pool viewed as `rows` rows of 128 bytes, boxes
// of 16 rows x 128 bytes with the 128-byte swizzle (paged_chunk_tc.cu).
bool make_pool_map_e4m3(CUtensorMap* map, const void* pool, int64_t rows);
// Decode (q_len 1) with QK^T and PV on tensor cores, `grid` persistent CTAs
// striding over the (request, KV head, split) units; num_splits > 1 writes
// workspace partials for the combine kernel (paged_decode_tc.cu).
cudaError_t launch_paged_decode_tc(const DecodeArgs& a, int32_t grid, cudaStream_t stream);

// Members per cascade group: 16 requests x 4 heads = one 64-row tile.
constexpr int kCascadeGroup = 16;

// q8_0 KV (pools of kQ8TileBytes per (block, kv head)): quantising append,
// and decode (q_len 1) on tensor cores, `grid` persistent CTAs walking the
// (request, KV head, split) units; num_splits > 1 writes workspace partials.
cudaError_t launch_kv_append_q8(void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                                const int64_t* slot_mapping, const void* k_new, const void* v_new,
                                int32_t num_tokens, unsigned int* err, cudaStream_t stream);
cudaError_t launch_paged_decode_q8(const DecodeArgs& a, int32_t grid, cudaStream_t stream);
// Decode (q_len 1) over E4M3 pools with both contractions on the tensor
// cores' 8-bit path, `grid` persistent CTAs striding over the (request, KV
// head, split) units; num_splits > 1 writes workspace partials
// (paged_decode_fp8_tc.cu).
cudaError_t launch_paged_decode_fp8_tc(const DecodeArgs& a, int32_t grid, cudaStream_t stream);
// FP8 (E4M3) KV: rounding append (pools of kFp8TileBytes per (block, kv head)).
cudaError_t launch_kv_append_fp8(void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                                 const int64_t* slot_mapping, const void* k_new, const void* v_new,
                                 int32_t num_tokens, unsigned int* err, cudaStream_t stream);

// Device error word of the current device (PKV_DEVERR_* bits).
unsigned int* device_error_word();

// Copies whole blocks (all KV heads) of both pools; block_bytes per block,
// a multiple of 16.
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, int32_t num_blocks, int64_t block_bytes,
                               const int32_t* src, const int32_t* dst, int32_t num_pairs, unsigned int* err,
                               cudaStream_t stream);

cudaError_t launch_attn_combine(void* out, float* out_lse, const float* part_o, const float* part_lse,
                                int32_t num_rows, int32_t num_splits, cudaStream_t stream);

}  // namespace pkv
