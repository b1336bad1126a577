// Paged decode attention for sm_103a.
//
// What is computed: for each sequence s and query head hq, softmax(scale *
// K q) V over the sequence's tokens, where token t's K/V row lives in
// physical block table[s][t / B] at offset t % B ("Paged Attention > The
// PagedAttention Algorithm", Standard Attention vs PagedAttention; the
// result equals standard attention on the gathered rows). No gathered copy is
// made: rows are read straight from the paged pool into shared memory
// (Optimized CUDA Kernels: attention computed directly on the paged
// structure, one block at a time, with a running max and running sum).
//
// Work decomposition: one CTA per (partition, kv head, sequence). A
// partition is `partition_tokens` consecutive tokens; all G = Hq / Hkv query
// heads of the kv head are handled by the same CTA, so every K/V byte is read
// from HBM once per call. Inside the CTA, each of the 4 warps owns every 4th
// 16-token tile of the partition and runs its own cp.async ring of
// STAGES tiles (K and V, 16 rows each), so the main loop has no CTA-wide
// barrier. Per tile a warp computes the scores of 16 query-head rows (the
// group, zero-padded) against 16 tokens with m16n8k16 tensor-core products,
// updates the online softmax in fp32 (base-2 exponent), and accumulates
// P.V with the same instruction (weights as a 16-bit head plus a 16-bit
// remainder, so their rounding stays far below the output tolerance). The 4 warps' states are then merged by
// log-sum-exp; a partition that is not a sequence's only one stores
// (normalised output, lse) to the workspace, and the last partition CTA of a
// (sequence, kv head) to arrive merges all partitions and writes `out`.
//
// Shared-memory rows are 16-byte-chunk XOR swizzled (chunk ^ (row & 7)) so
// that the 8 row addresses of every ldmatrix phase fall in distinct banks.
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileTokens = 16;  // tokens per warp tile (the k extent of the P.V product)
constexpr int kRows = 16;        // query-head rows of one tensor-core tile
constexpr int kStages = 3;       // cp.async ring depth per warp

template <int D>
struct Geometry {
  static constexpr int kRowBytes = D * 2;                    // one K or V row
  static constexpr int kChunks = kRowBytes / 16;             // 16-byte chunks per row
  static constexpr int kTileBytes = kTileTokens * kRowBytes;  // 16 rows
  static constexpr int kStageBytes = 2 * kTileBytes;          // K tile + V tile
  static constexpr int kPipeBytes = kWarps * kStages * kStageBytes;
  static constexpr int kQBytes = kRows * kRowBytes;
  static constexpr int kMLBytes = kWarps * 2 * kRows * 4;  // per-warp row max and sum
  static constexpr int kFacBytes = (kWarps + 2) * kRows * 4;
  static constexpr int kFixedBytes = kQBytes + kPipeBytes + kMLBytes + kFacBytes;
  static constexpr int kOStride = D + 4;  // fp32 row stride of a warp's merged output
  static_assert(kRows * kOStride * 4 <= kStages * kStageBytes, "merge area must fit a warp ring");
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk ^ (row & 7)) << 4);
}

template <typename Ty, int D>
__global__ void __launch_bounds__(kThreads)
paged_decode_kernel(const DecodeArgs a) {
  using Geo = Geometry<D>;
  using T = typename Ty::T;
  constexpr int kRowBytes = Geo::kRowBytes;
  constexpr int kChunks = Geo::kChunks;
  constexpr int kKSteps = D / 16;  // k-steps of the q.K product over head_dim
  constexpr int kNTiles = D / 8;   // n-tiles of the P.V product over head_dim
  constexpr int kRowsPerCopy = 32 / kChunks;          // rows one warp-wide copy covers
  constexpr int kCopies = kTileTokens / kRowsPerCopy;  // copies per lane per tensor per tile

  const int part = blockIdx.x;
  const int h = blockIdx.y;
  const int s = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int shift = a.block_shift;
  const int bmask = (1 << shift) - 1;
  const int G = a.group;

  // ---- sequence length and this CTA's token range --------------------------
  const int Lmax = a.max_blocks_per_seq << shift;
  int L = a.seq_lens[s];
  if (L < 0 || L > Lmax) {
    if (part == 0 && h == 0 && tid == 0) atomicAdd(a.bad, 1ull);
    L = min(max(L, 0), Lmax);
  }
  const int Pt = a.partition_tokens;
  const int nparts = L > 0 ? (L + Pt - 1) / Pt : 1;
  if (part >= nparts) return;
  const int t0 = part * Pt;  // a multiple of the block size
  const int ntok = min(Pt, L - t0);  // 0 only when L == 0

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sPipe = smem + Geo::kQBytes;
  float* sML = reinterpret_cast<float*>(sPipe + Geo::kPipeBytes);  // [warp][m|l][row]
  float* sFac = sML + kWarps * 2 * kRows;  // [warp][row] weights, then [row] 1/sum, [row] lse
  int* sTab = reinterpret_cast<int*>(sFac + (kWarps + 2) * kRows);
  __shared__ int sLast;

  // ---- this partition's slice of the block table (checked) ----------------
  const int nblk = (ntok + bmask) >> shift;
  const int32_t* trow = a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + (t0 >> shift);
  for (int i = tid; i < nblk; i += kThreads) {
    int phys = trow[i];
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) {
      atomicAdd(a.bad, 1ull);
      phys = -1;  // rows of a rejected block read as zeros
    }
    sTab[i] = phys;
  }
  // ---- the group's query rows, zero-padded to 16 rows ----------------------
  const T* qg = static_cast<const T*>(a.query) +
                (static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(h) * G) * D;
  for (int i = tid; i < kRows * kChunks; i += kThreads) {
    const int r = i / kChunks, c = i % kChunks;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < G) v = *reinterpret_cast<const uint4*>(qg + r * D + c * 8);
    *reinterpret_cast<uint4*>(sQ + r * kRowBytes + swz(r, c)) = v;
  }
  __syncthreads();

  // q as the A operand of the score product, kept in registers
  uint32_t qa[kKSteps][4];
  {
    const int mi = lane >> 3, rr = lane & 7;
    const int row = rr + ((mi & 1) << 3);
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
      const int c = 2 * kk + (mi >> 1);
      ldmatrix_x4(qa[kk], smem_u32(sQ + row * kRowBytes + swz(row, c)));
    }
  }

  // ---- per-warp pipelined token loop --------------------------------------
  const int ntiles = (ntok + kTileTokens - 1) / kTileTokens;
  const int my_tiles = warp < ntiles ? (ntiles - warp + kWarps - 1) / kWarps : 0;
  unsigned char* wpipe = sPipe + warp * kStages * Geo::kStageBytes;
  const size_t slot_stride = static_cast<size_t>(a.num_kv_heads) * D;  // elements per slot
  const T* kbase = static_cast<const T*>(a.key_cache) + static_cast<size_t>(h) * D;
  const T* vbase = static_cast<const T*>(a.value_cache) + static_cast<size_t>(h) * D;
  const int cc = lane % kChunks;  // this lane's 16-byte chunk of a row
  const int cr = lane / kChunks;  // this lane's first row of a tile

  auto load_tile = [&](int it, int stage) {
    const int tb = (warp + it * kWarps) * kTileTokens;  // partition-relative first token
    unsigned char* sk = wpipe + stage * Geo::kStageBytes;
    unsigned char* sv = sk + Geo::kTileBytes;
#pragma unroll
    for (int i = 0; i < kCopies; ++i) {
      const int r = cr + i * kRowsPerCopy;
      const int t = tb + r;
      const int phys = t < ntok ? sTab[t >> shift] : -1;
      const bool ok = phys >= 0;
      const size_t slot = ok ? (static_cast<size_t>(phys) << shift) + (t & bmask) : 0;
      const uint32_t off = r * kRowBytes + swz(r, cc);
      cp_async_16(smem_u32(sk + off), kbase + slot * slot_stride + cc * 8, ok);
      cp_async_16(smem_u32(sv + off), vbase + slot * slot_stride + cc * 8, ok);
    }
  };

  float m0 = -INFINITY, m1 = -INFINITY;  // running max of rows lane/4 and lane/4 + 8
  float l0 = 0.f, l1 = 0.f;              // this lane's share of the running sums
  float o[kNTiles][4];
#pragma unroll
  for (int n = 0; n < kNTiles; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < my_tiles) load_tile(i, i);
    cp_async_commit();
  }

  const float sl2 = a.scale_log2;
  const int tq = 2 * (lane & 3);  // first token column this lane holds in an 8-token n-tile

  for (int it = 0; it < my_tiles; ++it) {
    cp_async_wait<kStages - 2>();
    __syncwarp();
    {
      const int nx = it + kStages - 1;
      if (nx < my_tiles) load_tile(nx, nx % kStages);
      cp_async_commit();
    }
    const unsigned char* sk = wpipe + (it % kStages) * Geo::kStageBytes;
    const unsigned char* sv = sk + Geo::kTileBytes;
    const int valid = ntok - (warp + it * kWarps) * kTileTokens;  // >= 1

    // scores: [16 rows] x [16 tokens] as two m16n8 tiles
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int tok = rr + ((mi >> 1) << 3);
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        uint32_t b[4];
        ldmatrix_x4(b, smem_u32(sk + tok * kRowBytes + swz(tok, 2 * kk + (mi & 1))));
        Ty::mma(sa, qa[kk], b[0], b[1]);
        Ty::mma(sb, qa[kk], b[2], b[3]);
      }
    }
    // x[0..3]: row lane/4, tokens tq, tq+1, tq+8, tq+9; x[4..7]: row lane/4+8
    float x[8] = {sa[0] * sl2, sa[1] * sl2, sb[0] * sl2, sb[1] * sl2,
                  sa[2] * sl2, sa[3] * sl2, sb[2] * sl2, sb[3] * sl2};
    if (valid < kTileTokens) {
      const int tk[4] = {tq, tq + 1, tq + 8, tq + 9};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (tk[j] >= valid) x[j] = x[j + 4] = -INFINITY;
      }
    }
    float mx0 = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    float mx1 = fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);
    m0 = n0;
    m1 = n1;
    // weights, as A fragments: rows lane/4 (pa[0], pa[2]) and lane/4 + 8 (pa[1], pa[3]).
    // Each fp32 weight is split into a 16-bit head and the 16-bit rounding of
    // the remainder; both go through the P.V product, so the weights carry
    // about 16 significant bits instead of the input type's 8 or 11.
    float p[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      p[j] = ex2(x[j] - n0);
      p[j + 4] = ex2(x[j + 4] - n1);
    }
    uint32_t pa[4], pl[4];
    pa[0] = Ty::pack(p[0], p[1]);
    pa[1] = Ty::pack(p[4], p[5]);
    pa[2] = Ty::pack(p[2], p[3]);
    pa[3] = Ty::pack(p[6], p[7]);
    {
      const int src[4][2] = {{0, 1}, {4, 5}, {2, 3}, {6, 7}};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 hd = Ty::unpack(pa[j]);
        pl[j] = Ty::pack(p[src[j][0]] - hd.x, p[src[j][1]] - hd.y);
      }
    }
    l0 = l0 * al0 + ((p[0] + p[1]) + (p[2] + p[3]));
    l1 = l1 * al1 + ((p[4] + p[5]) + (p[6] + p[7]));
    if (__any_sync(0xffffffffu, (al0 != 1.f) | (al1 != 1.f))) {
#pragma unroll
      for (int n = 0; n < kNTiles; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
    }
    // O += P V: V rows are the k dimension, read transposed
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int tok = rr + ((mi & 1) << 3);
#pragma unroll
      for (int j = 0; j < kNTiles / 2; ++j) {
        uint32_t b[4];
        ldmatrix_x4_trans(b, smem_u32(sv + tok * kRowBytes + swz(tok, 2 * j + (mi >> 1))));
        Ty::mma(o[2 * j], pa, b[0], b[1]);
        Ty::mma(o[2 * j + 1], pa, b[2], b[3]);
        Ty::mma(o[2 * j], pl, b[0], b[1]);
        Ty::mma(o[2 * j + 1], pl, b[2], b[3]);
      }
    }
  }
  cp_async_wait<0>();

  // ---- merge the warps (log-sum-exp) -------------------------------------
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __syncwarp();
  {
    float* sO = reinterpret_cast<float*>(wpipe);
    const int r0 = lane >> 2;
#pragma unroll
    for (int n = 0; n < kNTiles; ++n) {
      const int col = n * 8 + tq;
      *reinterpret_cast<float2*>(sO + r0 * Geo::kOStride + col) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(sO + (r0 + 8) * Geo::kOStride + col) = make_float2(o[n][2], o[n][3]);
    }
    if ((lane & 3) == 0) {
      sML[(warp * 2 + 0) * kRows + r0] = m0;
      sML[(warp * 2 + 0) * kRows + r0 + 8] = m1;
      sML[(warp * 2 + 1) * kRows + r0] = l0;
      sML[(warp * 2 + 1) * kRows + r0 + 8] = l1;
    }
  }
  __syncthreads();
  if (tid < kRows) {
    const int r = tid;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sML[(w * 2) * kRows + r]);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = (M == -INFINITY) ? 0.f : ex2(sML[(w * 2) * kRows + r] - M);
      sFac[w * kRows + r] = f;
      tot += f * sML[(w * 2 + 1) * kRows + r];
    }
    sFac[kWarps * kRows + r] = tot > 0.f ? 1.f / tot : 0.f;
    sFac[(kWarps + 1) * kRows + r] = tot > 0.f ? M + __log2f(tot) : -INFINITY;
  }
  __syncthreads();

  const size_t row0 = static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(h) * G;
  if (nparts == 1) {
    for (int i = tid; i < G * (D / 2); i += kThreads) {
      const int g = i / (D / 2), c = 2 * (i % (D / 2));
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float* sO = reinterpret_cast<const float*>(sPipe + w * kStages * Geo::kStageBytes);
        const float f = sFac[w * kRows + g];
        v0 += f * sO[g * Geo::kOStride + c];
        v1 += f * sO[g * Geo::kOStride + c + 1];
      }
      const float inv = sFac[kWarps * kRows + g];
      const size_t o_idx = (row0 + g) * D + c;
      if (a.out_f32) {
        *reinterpret_cast<float2*>(static_cast<float*>(a.out) + o_idx) = make_float2(v0 * inv, v1 * inv);
      } else {
        *reinterpret_cast<uint32_t*>(static_cast<T*>(a.out) + o_idx) = Ty::pack(v0 * inv, v1 * inv);
      }
    }
    return;
  }

  // ---- split-K: store this partition, the last arrival combines -----------
  const int P = a.max_partitions;
  for (int i = tid; i < G * D; i += kThreads) {
    const int g = i / D, c = i % D;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* sO = reinterpret_cast<const float*>(sPipe + w * kStages * Geo::kStageBytes);
      v += sFac[w * kRows + g] * sO[g * Geo::kOStride + c];
    }
    a.ws_out[((row0 + g) * P + part) * D + c] = v * sFac[kWarps * kRows + g];
  }
  if (tid < G) a.ws_lse[(row0 + tid) * P + part] = sFac[(kWarps + 1) * kRows + tid];
  __threadfence();
  __syncthreads();
  int* counter = a.ws_count + static_cast<size_t>(s) * a.num_kv_heads + h;
  if (tid == 0) sLast = (atomicAdd(counter, 1) == nparts - 1);
  __syncthreads();
  if (!sLast) return;
  __threadfence();

  // per-row max and 1/sum of the partition weights
  float* sRed = reinterpret_cast<float*>(sPipe);  // [row] max, [row] 1/sum, then weights
  for (int g = warp; g < G; g += kWarps) {
    const float* lse = a.ws_lse + (row0 + g) * P;
    float M = -INFINITY;
    for (int p = lane; p < nparts; p += 32) M = fmaxf(M, __ldcg(lse + p));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float tot = 0.f;
    for (int p = lane; p < nparts; p += 32) tot += ex2(__ldcg(lse + p) - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    if (lane == 0) {
      sRed[g] = M;
      sRed[kRows + g] = 1.f / tot;
    }
  }
  __syncthreads();
  float* sW = sRed + 2 * kRows;
  const int cap = (Geo::kPipeBytes / 4 - 2 * kRows) / G;  // weights per row that fit
  constexpr int kGStride = kThreads / D;                  // rows handled per pass
  constexpr int kAcc = kRows / kGStride;
  const int col = tid % D;
  const int gfirst = tid / D;
  float acc[kAcc];
#pragma unroll
  for (int k = 0; k < kAcc; ++k) acc[k] = 0.f;
  for (int p0 = 0; p0 < nparts; p0 += cap) {
    const int np = min(cap, nparts - p0);
    for (int i = tid; i < G * np; i += kThreads) {
      const int g = i / np, p = i % np;
      sW[g * np + p] = ex2(__ldcg(a.ws_lse + (row0 + g) * P + p0 + p) - sRed[g]) * sRed[kRows + g];
    }
    __syncthreads();
    for (int p = 0; p < np; ++p) {
#pragma unroll
      for (int k = 0; k < kAcc; ++k) {
        const int g = gfirst + k * kGStride;
        if (g < G) acc[k] += sW[g * np + p] * __ldcg(a.ws_out + ((row0 + g) * P + p0 + p) * D + col);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int k = 0; k < kAcc; ++k) {
    const int g = gfirst + k * kGStride;
    if (g < G) {
      const size_t o_idx = (row0 + g) * D + col;
      if (a.out_f32) {
        static_cast<float*>(a.out)[o_idx] = acc[k];
      } else {
        static_cast<T*>(a.out)[o_idx] = Ty::cvt(acc[k]);
      }
    }
  }
  if (tid == 0) *counter = 0;  // ready for the next call on this workspace
}

template <typename Ty, int D>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
  const int B = 1 << a.block_shift;
  const int entries = (a.partition_tokens + B - 1) / B;
  const size_t smem = static_cast<size_t>(Geometry<D>::kFixedBytes) + 4 * static_cast<size_t>(entries);
  auto kern = paged_decode_kernel<Ty, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_partitions, a.num_kv_heads, a.num_seqs);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t decode_smem_bytes(int head_dim, int table_entries) {
  const size_t fixed = head_dim == 64 ? Geometry<64>::kFixedBytes : Geometry<128>::kFixedBytes;
  return fixed + 4 * static_cast<size_t>(table_entries);
}

cudaError_t launch_decode(const DecodeArgs& a, int head_dim, bool bf16, cudaStream_t stream) {
  if (bf16) {
    return head_dim == 64 ? launch_typed<BF16, 64>(a, stream) : launch_typed<BF16, 128>(a, stream);
  }
  return head_dim == 64 ? launch_typed<F16, 64>(a, stream) : launch_typed<F16, 128>(a, stream);
}

}  // namespace pa
