// decode_graph.cu -- a decode step of several layers (per layer: append the
// step's new tokens, then attention) captured as one CUDA graph per buffer
// set, for the two alternating ("ping-pong") buffer sets of a decode loop.
//
// Why ("Chapter 8: Inference Optimization", clxhxhhr.top/posts/4341, §8.6.3;
// "Popping the GPU bubble", §3): with CUDA graphs off, a decode round spends
// a roughly fixed time submitting kernels one by one from the host; a graph
// replays the whole step with one launch.  A graph needs fixed buffer
// addresses, and a pipelined loop needs two buffer sets so the host can
// prepare one step while the GPU runs the other.
//
// The step is recorded by calling this library's own entry points inside a
// stream capture: the graph runs exactly the kernels of the direct calls,
// with the same validation (a call that fails aborts the capture and create
// returns its status).  Capture runs on a private non-blocking stream in
// relaxed mode, so the entry points' one-time per-device set-up (function
// attributes, symbol lookups) may happen inside it.
#include <cstdint>
#include <new>

#include <cuda_runtime.h>

#include "pkv.h"

struct pkv_decode_graph {
  cudaGraphExec_t exec[2];
};

namespace {

constexpr size_t kBf16RowBytes = 128 * 2;  // one head vector

pkv_status append_layer(const pkv_decode_graph_desc& d, const pkv_decode_graph_buffers& b, int l,
                        cudaStream_t s) {
  const size_t kv_layer = static_cast<size_t>(d.num_tokens) * d.cache.num_kv_heads * kBf16RowBytes;
  const void* kn = static_cast<const uint8_t*>(b.k_new) + l * kv_layer;
  const void* vn = static_cast<const uint8_t*>(b.v_new) + l * kv_layer;
  switch (d.kv_format) {
    case PKV_KV_BF16:
      return pkv_kv_append(d.k_caches[l], d.v_caches[l], &d.cache, b.slot_mapping, kn, vn, d.num_tokens, s);
    case PKV_KV_Q8_0:
      return pkv_kv_append_q8_0(d.k_caches[l], d.v_caches[l], &d.cache, b.slot_mapping, kn, vn, d.num_tokens, s);
    case PKV_KV_FP8_E4M3:
      return pkv_kv_append_fp8_e4m3(d.k_caches[l], d.v_caches[l], &d.cache, b.slot_mapping, kn, vn, d.num_tokens,
                                    s);
    default:
      return PKV_ERR_UNSUPPORTED;
  }
}

pkv_status attend_layer(const pkv_decode_graph_desc& d, const pkv_decode_graph_buffers& b, int l, cudaStream_t s) {
  const size_t q_layer = static_cast<size_t>(d.num_seqs) * d.q_len * d.num_q_heads * kBf16RowBytes;
  const void* q = static_cast<const uint8_t*>(b.q) + l * q_layer;
  void* out = static_cast<uint8_t*>(b.out) + l * q_layer;
  const void* kc = d.k_caches[l];
  const void* vc = d.v_caches[l];
  switch (d.kv_format) {
    case PKV_KV_BF16:
      if (d.num_groups > 0)
        return pkv_paged_attention_cascade(out, q, kc, vc, &d.cache, b.block_tables, d.max_blocks_per_seq,
                                           b.context_lens, d.num_seqs, d.num_q_heads, d.scale, b.group_seqs,
                                           b.group_blocks, b.seq_prefix_blocks, d.num_groups, d.max_prefix_blocks,
                                           d.max_suffix_blocks, d.prefix_blocks_per_split,
                                           d.suffix_blocks_per_split, d.workspace, d.workspace_bytes, s);
      return pkv_paged_attention(out, q, kc, vc, &d.cache, b.block_tables, d.max_blocks_per_seq, b.context_lens,
                                 d.num_seqs, d.q_len, d.num_q_heads, d.scale, d.kv_blocks_per_split, d.workspace,
                                 d.workspace_bytes, s);
    case PKV_KV_Q8_0:
      return pkv_paged_attention_q8_0(out, q, kc, vc, &d.cache, b.block_tables, d.max_blocks_per_seq,
                                      b.context_lens, d.num_seqs, d.num_q_heads, d.scale, d.kv_blocks_per_split,
                                      d.workspace, d.workspace_bytes, s);
    case PKV_KV_FP8_E4M3:
      return pkv_paged_attention_fp8_e4m3(out, q, kc, vc, &d.cache, b.block_tables, d.max_blocks_per_seq,
                                          b.context_lens, d.num_seqs, d.num_q_heads, d.scale,
                                          d.kv_blocks_per_split, d.workspace, d.workspace_bytes, s);
    default:
      return PKV_ERR_UNSUPPORTED;
  }
}

// The append and the attention as one call (pkv_paged_attention_append, its
// cascade form, or the q8_0 / E4M3 one), which fuses them into one kernel
// when it can.
pkv_status append_attend_layer(const pkv_decode_graph_desc& d, const pkv_decode_graph_buffers& b, int l,
                               cudaStream_t s) {
  const size_t q_layer = static_cast<size_t>(d.num_seqs) * d.q_len * d.num_q_heads * kBf16RowBytes;
  const size_t kv_layer = static_cast<size_t>(d.num_tokens) * d.cache.num_kv_heads * kBf16RowBytes;
  const void* kn = static_cast<const uint8_t*>(b.k_new) + l * kv_layer;
  const void* vn = static_cast<const uint8_t*>(b.v_new) + l * kv_layer;
  if (d.kv_format == PKV_KV_Q8_0)
    return pkv_paged_attention_q8_0_append(
        static_cast<uint8_t*>(b.out) + l * q_layer, static_cast<const uint8_t*>(b.q) + l * q_layer, d.k_caches[l],
        d.v_caches[l], &d.cache, b.block_tables, d.max_blocks_per_seq, b.context_lens, d.num_seqs, d.num_q_heads,
        d.scale, d.kv_blocks_per_split, d.workspace, d.workspace_bytes, b.slot_mapping, kn, vn, d.num_tokens, s);
  if (d.kv_format == PKV_KV_FP8_E4M3)
    return pkv_paged_attention_fp8_e4m3_append(
        static_cast<uint8_t*>(b.out) + l * q_layer, static_cast<const uint8_t*>(b.q) + l * q_layer, d.k_caches[l],
        d.v_caches[l], &d.cache, b.block_tables, d.max_blocks_per_seq, b.context_lens, d.num_seqs, d.num_q_heads,
        d.scale, d.kv_blocks_per_split, d.workspace, d.workspace_bytes, b.slot_mapping, kn, vn, d.num_tokens, s);
  if (d.num_groups > 0)
    return pkv_paged_attention_cascade_append(
        static_cast<uint8_t*>(b.out) + l * q_layer, static_cast<const uint8_t*>(b.q) + l * q_layer, d.k_caches[l],
        d.v_caches[l], &d.cache, b.block_tables, d.max_blocks_per_seq, b.context_lens, d.num_seqs, d.num_q_heads,
        d.scale, b.group_seqs, b.group_blocks, b.seq_prefix_blocks, d.num_groups, d.max_prefix_blocks,
        d.max_suffix_blocks, d.prefix_blocks_per_split, d.suffix_blocks_per_split, d.workspace, d.workspace_bytes,
        b.slot_mapping, kn, vn, d.num_tokens, s);
  return pkv_paged_attention_append(static_cast<uint8_t*>(b.out) + l * q_layer,
                                    static_cast<const uint8_t*>(b.q) + l * q_layer, d.k_caches[l], d.v_caches[l],
                                    &d.cache, b.block_tables, d.max_blocks_per_seq, b.context_lens, d.num_seqs,
                                    d.q_len, d.num_q_heads, d.scale, d.kv_blocks_per_split, d.workspace,
                                    d.workspace_bytes, b.slot_mapping, kn, vn, d.num_tokens, s);
}

// Host-side checks of the description (the calls check the rest).
pkv_status check_desc(const pkv_decode_graph_desc& d) {
  if (d.num_layers < 1 || d.num_tokens < 0 || d.num_seqs < 0 || d.q_len < 1 || d.num_q_heads < 1)
    return PKV_ERR_SHAPE;
  if (d.kv_format != PKV_KV_BF16 && d.kv_format != PKV_KV_Q8_0 && d.kv_format != PKV_KV_FP8_E4M3)
    return PKV_ERR_UNSUPPORTED;
  if (d.num_groups < 0) return PKV_ERR_SHAPE;
  if ((d.kv_format != PKV_KV_BF16 || d.num_groups > 0) && d.q_len != 1) return PKV_ERR_UNSUPPORTED;
  if (d.kv_format != PKV_KV_BF16 && d.num_groups > 0) return PKV_ERR_UNSUPPORTED;
  if (d.cache.num_kv_heads < 1) return PKV_ERR_SHAPE;
  if (d.k_caches == nullptr || d.v_caches == nullptr) return PKV_ERR_NULL;
  for (int l = 0; l < d.num_layers; ++l)
    if (d.k_caches[l] == nullptr || d.v_caches[l] == nullptr) return PKV_ERR_NULL;
  for (int s = 0; s < 2; ++s) {
    const pkv_decode_graph_buffers& b = d.set[s];
    if (b.q == nullptr || b.out == nullptr || b.block_tables == nullptr || b.context_lens == nullptr)
      return PKV_ERR_NULL;
    if (d.num_tokens > 0 && (b.k_new == nullptr || b.v_new == nullptr || b.slot_mapping == nullptr))
      return PKV_ERR_NULL;
    if (d.num_groups > 0 && (b.group_seqs == nullptr || b.group_blocks == nullptr || b.seq_prefix_blocks == nullptr))
      return PKV_ERR_NULL;
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_decode_graph_create(const pkv_decode_graph_desc* desc, pkv_decode_graph** graph) {
  if (graph == nullptr || desc == nullptr) return PKV_ERR_NULL;
  *graph = nullptr;
  const pkv_decode_graph_desc& d = *desc;
  pkv_status st = check_desc(d);
  if (st != PKV_OK) return st;
  pkv_decode_graph* g = new (std::nothrow) pkv_decode_graph{};
  if (g == nullptr) return PKV_ERR_CUDA;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
    delete g;
    return PKV_ERR_CUDA;
  }
  for (int s = 0; s < 2 && st == PKV_OK; ++s) {
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
      st = PKV_ERR_CUDA;
      break;
    }
    pkv_status call = PKV_OK;
    for (int l = 0; l < d.num_layers && call == PKV_OK; ++l) {
      if (d.num_tokens > 0) {
        call = append_attend_layer(d, d.set[s], l, cs);  // the append fused where the shape allows
        continue;
      }
      if (d.num_tokens > 0) call = append_layer(d, d.set[s], l, cs);
      if (call == PKV_OK) call = attend_layer(d, d.set[s], l, cs);
    }
    cudaGraph_t captured = nullptr;
    const cudaError_t e = cudaStreamEndCapture(cs, &captured);
    if (call != PKV_OK)
      st = call;
    else if (e != cudaSuccess || captured == nullptr)
      st = PKV_ERR_CUDA;
    else if (cudaGraphInstantiate(&g->exec[s], captured, 0) != cudaSuccess)
      st = PKV_ERR_CUDA;
    if (captured != nullptr) cudaGraphDestroy(captured);
  }
  cudaStreamDestroy(cs);
  if (st != PKV_OK) {
    pkv_decode_graph_destroy(g);
    return st;
  }
  *graph = g;
  return PKV_OK;
}

pkv_status pkv_decode_graph_launch(pkv_decode_graph* graph, int32_t buffer_set, void* stream) {
  if (graph == nullptr) return PKV_ERR_NULL;
  if (buffer_set != 0 && buffer_set != 1) return PKV_ERR_SHAPE;
  return cudaGraphLaunch(graph->exec[buffer_set], static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK
                                                                                                   : PKV_ERR_CUDA;
}

void pkv_decode_graph_destroy(pkv_decode_graph* graph) {
  if (graph == nullptr) return;
  for (int s = 0; s < 2; ++s)
    if (graph->exec[s] != nullptr) cudaGraphExecDestroy(graph->exec[s]);
  delete graph;
}

}  // extern "C"
