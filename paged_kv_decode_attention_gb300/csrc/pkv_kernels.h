// pkv_kernels.h -- host-side launchers of libpkv's kernels (internal).
// The exported C ABI (pkv_api.cu) validates arguments and calls these.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

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
};

cudaError_t launch_kv_append(void* k_cache, void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                             const int64_t* slot_mapping, const void* k_new, const void* v_new,
                             int32_t num_tokens, unsigned int* err, cudaStream_t stream);

// num_splits == 1: direct; part_o == NULL: cluster merge (num_splits <= kMaxClusterSplits);
// otherwise partials to the workspace (the caller then runs the combine kernel).
cudaError_t launch_paged_decode(const DecodeArgs& a, cudaStream_t stream);

// Queries per request at or above which the tensor-core chunk kernel runs
// (16 positions x 4 heads = 64 rows, one tcgen05 M=64 tile).
constexpr int kTcMinQLen = 16;

// Chunked causal attention on tensor cores (paged_chunk_tc.cu).  Same fields
// as DecodeArgs; num_splits > 1 always goes through the workspace.
using ChunkArgs = DecodeArgs;
cudaError_t launch_paged_chunk_tc(const ChunkArgs& a, cudaStream_t stream);

cudaError_t launch_attn_combine(void* out, float* out_lse, const float* part_o, const float* part_lse,
                                int32_t num_rows, int32_t num_splits, cudaStream_t stream);

}  // namespace pkv
