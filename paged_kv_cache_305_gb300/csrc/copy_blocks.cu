// Whole-block copies inside the K and V pools: the device half of
// copy-on-write ("PagedAttention by hand", Why divide memory into physical
// blocks?: allocate a fresh physical block, copy that one block's contents,
// then write into the copy). A block is B * Hkv * d contiguous 16-bit values
// in the [blocks, B, Hkv, d] layout, moved in 16-byte vectors.
#include <cuda_runtime.h>

#include "internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
copy_blocks_kernel(uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                   const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                   int num_copies, long long block_chunks, int num_blocks,
                   unsigned long long* bad) {
  for (int i = blockIdx.y; i < num_copies; i += gridDim.y) {
    const int s = src[i], d = dst[i];
    if (static_cast<unsigned>(s) >= static_cast<unsigned>(num_blocks) ||
        static_cast<unsigned>(d) >= static_cast<unsigned>(num_blocks)) {
      if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(bad, 1ull);  // skipped, counted
      continue;
    }
    if (s == d) continue;
    const uint4* ks = key_cache + static_cast<size_t>(s) * block_chunks;
    const uint4* vs = value_cache + static_cast<size_t>(s) * block_chunks;
    uint4* kd = key_cache + static_cast<size_t>(d) * block_chunks;
    uint4* vd = value_cache + static_cast<size_t>(d) * block_chunks;
    for (long long c = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; c < block_chunks;
         c += static_cast<long long>(gridDim.x) * kThreads) {
      const uint4 k = ks[c];
      const uint4 v = vs[c];
      kd[c] = k;
      vd[c] = v;
    }
  }
}

}  // namespace

cudaError_t launch_copy_blocks(void* key_cache, void* value_cache, const int32_t* src,
                               const int32_t* dst, int num_copies, long long block_bytes,
                               int num_blocks, unsigned long long* bad, cudaStream_t stream) {
  const long long chunks = block_bytes / 16;
  long long gx = (chunks + kThreads - 1) / kThreads;
  if (gx > 64) gx = 64;
  const int gy = num_copies < 65535 ? num_copies : 65535;
  copy_blocks_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), kThreads, 0,
                       stream>>>(static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), src,
                                 dst, num_copies, chunks, num_blocks, bad);
  return cudaGetLastError();
}

}  // namespace pa
