// pkv_static_workspace.cu -- pkv_paged_attention_static_workspace: the
// attention entry point for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: code that runs where
// the allocator must not be entered (inside a custom memory manager or an
// allocation callback, or under a framework that forbids allocation on its
// hot path), and plain C callers that hold no CUDA allocator at all.  For
// them this entry point takes the split-KV partial results in a fixed
// scratch array compiled into the library instead of a caller workspace.  It
// then forwards to pkv_paged_attention, so the kernels and results are the
// same.
//
// The array is a file-scope __device__ variable.  Every GPU that loads
// libpkv holds it until the process exits.  In host code its name is only a
// host-side stand-in, so the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and cached.  That happens on
// the first call made on a device, so that first call should come before any
// stream capture.  The cache is per device and safe for concurrent first calls
// from several host threads; a cudaDeviceReset of a device leaves its cached
// address stale, so this entry point is not for use on that device after a
// reset.  All calls on a device share the one array: calls that may
// overlap on the GPU (different streams without ordering between them) race
// on it.  Nothing in it needs to start at zero, because each call writes every
// partial log-sum-exp it later reads and only reads partial outputs it wrote.
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "pkv.h"

namespace {

static __device__ __align__(256) uint8_t g_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_static_workspace_ptr[kMaxDevices];
std::mutex g_static_workspace_lookup;

// Device address of this device's copy of the array (looked up once per
// device; a first call racing another thread's waits for its lookup).
void* static_workspace_address(pkv_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *st = PKV_ERR_CUDA;
    return nullptr;
  }
  void* p = g_static_workspace_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_static_workspace_lookup);
    p = g_static_workspace_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) {
        *st = PKV_ERR_CUDA;
        return nullptr;
      }
      g_static_workspace_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *st = PKV_OK;
  return p;
}

}  // namespace

extern "C" pkv_status pkv_paged_attention_static_workspace(
    void* out, const void* q, const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
    int32_t q_len, int32_t num_q_heads, float scale, int32_t kv_blocks_per_split, void* stream) {
  if (cache == nullptr) return PKV_ERR_NULL;
  if (num_seqs < 0 || q_len < 1 || max_blocks_per_seq < 1 || kv_blocks_per_split < 0) return PKV_ERR_SHAPE;
  // resolve the split exactly as pkv_paged_attention does, to size the scratch
  int32_t bps = kv_blocks_per_split;
  if (bps == 0)
    bps = pkv_choose_kv_blocks_per_split(num_seqs, cache->num_kv_heads, q_len, max_blocks_per_seq, 0);
  if (bps > max_blocks_per_seq) bps = max_blocks_per_seq;
  const size_t need =
      pkv_workspace_size(num_seqs, q_len, num_q_heads, cache->head_dim, max_blocks_per_seq, bps);
  if (need > PKV_STATIC_WORKSPACE_BYTES) return PKV_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    pkv_status st = PKV_OK;
    ws = static_workspace_address(&st);
    if (st != PKV_OK) return st;
  }
  return pkv_paged_attention(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                             num_seqs, q_len, num_q_heads, scale, bps, ws, need > 0 ? PKV_STATIC_WORKSPACE_BYTES : 0,
                             stream);
}
