// pa_decode_no_alloc: pa_decode with its split-K scratch taken from a
// fixed-size array that the library itself holds in device memory, for
// callers that cannot allocate device memory.
//
// The scratch is a file-scope __device__ array. Host code cannot use its name
// as a device address (on the host the name is only a stand-in), so each
// device's address is looked up once with cudaGetSymbolAddress, with that
// device current, and cached.
#include <cuda_runtime.h>
#include <stdio.h>

#include <atomic>

#include "internal.h"
#include "pagedattn.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device

__device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];

int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  char msg[256];
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    return pa::set_error(PA_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, sizeof(msg), "device index %d", dev);
    return pa::set_error(PA_ERR_UNSUPPORTED, msg);
  }
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess) {
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(no-alloc scratch): %s",
               cudaGetErrorString(e));
      return pa::set_error(PA_ERR_CUDA, msg);
    }
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" size_t pa_decode_no_alloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int pa_decode_no_alloc(void* out, const void* query, const void* key_cache,
                                  const void* value_cache, const int32_t* block_tables,
                                  const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size, float scale,
                                  int max_blocks_per_seq, int num_blocks, int partition_tokens,
                                  pa_dtype dtype, pa_dtype out_dtype, cudaStream_t stream) {
  const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim,
                                                max_blocks_per_seq, block_size, partition_tokens);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "pa_decode_no_alloc: these sizes need %zu bytes of split-K scratch; the built-in "
             "scratch holds %zu (use pa_decode with a caller-owned workspace, or longer "
             "partitions)", need, kNoAllocScratchBytes);
    return pa::set_error(PA_ERR_WORKSPACE, msg);
  }
  void* ws = nullptr;
  if (need > 0 && num_seqs > 0) {
    int rc = scratch_address(&ws);
    if (rc != PA_OK) return rc;
    // the header and arrival counters at the start of the scratch must be
    // zero; the previous call's contents are still there
    const size_t counters = pa::kWorkspaceHeader + static_cast<size_t>(num_seqs) * num_q_heads * sizeof(int);
    cudaError_t e = cudaMemsetAsync(ws, 0, counters, stream);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaMemsetAsync(no-alloc scratch counters): %s",
               cudaGetErrorString(e));
      return pa::set_error(PA_ERR_CUDA, msg);
    }
  }
  return pa_decode(out, query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, block_size, scale, max_blocks_per_seq,
                   num_blocks, partition_tokens, dtype, out_dtype, ws,
                   ws ? kNoAllocScratchBytes : 0, stream);
}
