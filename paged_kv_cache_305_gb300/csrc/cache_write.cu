// Cache write: copy each new token's K and V rows into its slot of the paged
// pool. vLLM performs this write for the token being decoded before the
// attention kernel runs ("PagedAttention by hand", Setup, Step 1, and the
// Code section). With the [blocks, B, Hkv, d] layout the
// [Hkv, d] rows of one token are contiguous both in the source and at the
// slot, so the copy is one contiguous run of Hkv * d * 2 bytes per tensor,
// moved in 16-byte vectors.
#include <cuda_runtime.h>

#include "internal.h"

namespace pa {
namespace {

constexpr int kThreads = 128;

// One CTA per token; its threads stride over the row's 16-byte chunks.
__global__ void __launch_bounds__(kThreads)
reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                         uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                         const int64_t* __restrict__ slot_mapping, int chunks,
                         long long num_slots, unsigned long long* bad) {
  const int t = blockIdx.x;
  const long long slot = slot_mapping[t];
  if (slot < 0) return;  // nothing to write for this token
  if (slot >= num_slots) {
    if (threadIdx.x == 0) atomicAdd(bad, 1ull);
    return;
  }
  const uint4* ks = key + static_cast<size_t>(t) * chunks;
  const uint4* vs = value + static_cast<size_t>(t) * chunks;
  uint4* kd = key_cache + static_cast<size_t>(slot) * chunks;
  uint4* vd = value_cache + static_cast<size_t>(slot) * chunks;
  for (int c = threadIdx.x; c < chunks; c += kThreads) {
    const uint4 k = __ldg(ks + c);
    const uint4 v = __ldg(vs + c);
    kd[c] = k;
    vd[c] = v;
  }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                     void* value_cache, const int64_t* slot_mapping,
                                     int num_tokens, int row_bytes, long long num_slots,
                                     unsigned long long* bad, cudaStream_t stream) {
  reshape_and_cache_kernel<<<num_tokens, kThreads, 0, stream>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value),
      static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), slot_mapping,
      row_bytes / 16, num_slots, bad);
  return cudaGetLastError();
}

}  // namespace pa
