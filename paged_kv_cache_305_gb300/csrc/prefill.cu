// Paged causal prefill (chunked prefill) for sm_103a.
//
// What is computed: sequence s has L = seq_lens[s] tokens in the paged cache,
// the last Q of which are new; their queries (rows query_start[s] ..
// query_start[s+1]-1) attend causally: query j sits at position L - Q + j and
// sees tokens 0 .. L - Q + j ("PagedAttention" glossary, How It Works: the
// blockwise formula with query index i; read token by token). K/V rows come
// straight from the physical blocks through the block table.
//
// Work decomposition: one CTA per (query tile, kv head, sequence). A query
// tile is 64 rows = Mq query positions x the G heads of the kv head
// (Mq = 64 / G), so each K/V tile read from the cache serves every query head
// of the group. The CTA walks the key tiles (64 tokens) from the first up to
// the tile holding its last query's position, double-buffered with cp.async;
// table ids for the next tile are loaded a tile ahead. Each warp owns 16 rows:
// S = q K^T and O = P V with m16n8k16 tensor-core products, an online softmax
// per row in fp32 (base-2 exponents), a causal mask per row on the diagonal
// tiles, and weights entering P V as a 16-bit head plus a 16-bit remainder.
// Query tiles are launched last-first, so the longest (most key tiles) start
// first.
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerCta = 64;  // query rows (positions x heads)
constexpr int kKeyTile = 64;     // tokens per key tile
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk ^ (row & 7)) << 4);
}

template <int D>
struct PGeo {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kChunks = kRowBytes / 16;
  static constexpr int kQBytes = kRowsPerCta * kRowBytes;
  static constexpr int kTileBytes = kKeyTile * kRowBytes;  // one K or V tile
  static constexpr int kSmem = kQBytes + 2 * 2 * kTileBytes;
  static constexpr int kRowGroups = kThreads / kChunks;      // rows loaded per pass
  static constexpr int kRowsPerThread = kKeyTile / kRowGroups;
};

template <typename Ty, int D>
__global__ void __launch_bounds__(kThreads, 2)
paged_prefill_kernel(const PrefillArgs a) {
  using Geo = PGeo<D>;
  using T = typename Ty::T;
  constexpr int kRowBytes = Geo::kRowBytes;
  constexpr int kChunks = Geo::kChunks;
  constexpr int kKSteps = D / 16;
  constexpr int kDTiles = D / 8;  // n-tiles of P V over head_dim
  constexpr int kTokTiles = kKeyTile / 8;  // n-tiles of q K^T over a key tile
  constexpr int kRPT = Geo::kRowsPerThread;

  const int qt = gridDim.x - 1 - blockIdx.x;  // longest tiles first
  const int h = blockIdx.y;
  const int s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.group;
  const int Mq = kRowsPerCta / G;  // query positions per tile
  const int shift = a.block_shift, bmask = (1 << shift) - 1;
  const int Lmax = a.max_blocks_per_seq << shift;

  int L = a.seq_lens[s];
  const int q0 = a.query_start[s];
  int Q = a.query_start[s + 1] - q0;
  if (L < 0 || L > Lmax || Q < 0 || Q > L) {
    if (qt == 0 && h == 0 && tid == 0) atomicAdd(a.bad, 1ull);
    L = min(max(L, 0), Lmax);
    Q = min(max(Q, 0), L);
  }
  const int j0 = qt * Mq;  // first query position index of this tile
  if (j0 >= Q) return;
  const int jn = min(Mq, Q - j0);            // query positions in this tile
  const int last_pos = L - Q + j0 + jn - 1;  // the tile's furthest position
  const int ntiles = last_pos / kKeyTile + 1;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sKV = smem + Geo::kQBytes;  // [stage][K|V][64 rows]

  // ---- query rows: r -> (position j0 + r / G, head h*G + r % G) -------------
  const T* qbase = static_cast<const T*>(a.query);
  for (int i = tid; i < kRowsPerCta * kChunks; i += kThreads) {
    const int r = i / kChunks, c = i % kChunks;
    const int jj = r / G, g = r % G;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (jj < jn && r < Mq * G) {
      const size_t row = static_cast<size_t>(q0 + j0 + jj) * a.num_q_heads + static_cast<size_t>(h) * G + g;
      v = *reinterpret_cast<const uint4*>(qbase + row * D + c * 8);
    }
    *reinterpret_cast<uint4*>(sQ + r * kRowBytes + swz(r, c)) = v;
  }

  // ---- key/value tile loads ---------------------------------------------------
  const size_t slot_stride = static_cast<size_t>(a.num_kv_heads) * D;
  const T* kbase = static_cast<const T*>(a.key_cache) + static_cast<size_t>(h) * D;
  const T* vbase = static_cast<const T*>(a.value_cache) + static_cast<size_t>(h) * D;
  const int cc = tid % kChunks, rg = tid / kChunks;
  const int32_t* trow = a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq;
  int ids[kRPT];
  auto load_ids = [&](int kt) {
#pragma unroll
    for (int i = 0; i < kRPT; ++i) {
      const int t = kt * kKeyTile + rg + i * Geo::kRowGroups;
      ids[i] = (kt < ntiles && t < L) ? __ldg(trow + (t >> shift)) : -1;
    }
  };
  auto issue = [&](int kt, int buf) {
    unsigned char* sk = sKV + buf * 2 * Geo::kTileBytes;
    unsigned char* sv = sk + Geo::kTileBytes;
#pragma unroll
    for (int i = 0; i < kRPT; ++i) {
      const int r = rg + i * Geo::kRowGroups;
      const int t = kt * kKeyTile + r;
      const int phys = ids[i];
      const bool in = t < L;
      const bool ok = in && static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks);
      if (in && !ok && cc == 0) atomicAdd(a.bad, 1ull);
      const size_t slot = ok ? (static_cast<size_t>(phys) << shift) + (t & bmask) : 0;
      const uint32_t off = r * kRowBytes + swz(r, cc);
      cp_async_16(smem_u32(sk + off), kbase + slot * slot_stride + cc * 8, ok);
      cp_async_16(smem_u32(sv + off), vbase + slot * slot_stride + cc * 8, ok);
    }
    cp_async_commit();
  };

  load_ids(0);
  issue(0, 0);
  load_ids(1);
  __syncthreads();  // q tile in shared memory

  uint32_t qa[kKSteps][4];
  {
    const int mi = lane >> 3, rr = lane & 7;
    const int row = warp * 16 + rr + ((mi & 1) << 3);
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk)
      ldmatrix_x4(qa[kk], smem_u32(sQ + row * kRowBytes + swz(row, 2 * kk + (mi >> 1))));
  }
  // causal limit of this lane's two rows (warp*16 + lane/4, + 8)
  const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
  const int lim0 = (r0 / G < jn && r0 < Mq * G) ? L - Q + j0 + r0 / G : last_pos;
  const int lim1 = (r1 / G < jn && r1 < Mq * G) ? L - Q + j0 + r1 / G : last_pos;
  const int tq = 2 * (lane & 3);
  const float sl2 = a.scale_log2;

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[kDTiles][4];
#pragma unroll
  for (int n = 0; n < kDTiles; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  for (int kt = 0; kt < ntiles; ++kt) {
    if (kt + 1 < ntiles) {
      issue(kt + 1, (kt + 1) & 1);
      load_ids(kt + 2);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const unsigned char* sk = sKV + (kt & 1) * 2 * Geo::kTileBytes;
    const unsigned char* sv = sk + Geo::kTileBytes;
    const int tbase = kt * kKeyTile;

    // S = q K^T: 16 rows x 64 tokens
    float sc[kTokTiles][4];
#pragma unroll
    for (int n = 0; n < kTokTiles; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
    {
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
#pragma unroll
        for (int tp = 0; tp < kTokTiles / 2; ++tp) {
          const int tok = tp * 16 + rr + ((mi >> 1) << 3);
          uint32_t b[4];
          ldmatrix_x4(b, smem_u32(sk + tok * kRowBytes + swz(tok, 2 * kk + (mi & 1))));
          Ty::mma(sc[2 * tp], qa[kk], b[0], b[1]);
          Ty::mma(sc[2 * tp + 1], qa[kk], b[2], b[3]);
        }
      }
    }
    // mask, row max
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < kTokTiles; ++n) {
      const int t = tbase + n * 8 + tq;
      sc[n][0] = t <= lim0 ? sc[n][0] * sl2 : -INFINITY;
      sc[n][1] = t + 1 <= lim0 ? sc[n][1] * sl2 : -INFINITY;
      sc[n][2] = t <= lim1 ? sc[n][2] * sl2 : -INFINITY;
      sc[n][3] = t + 1 <= lim1 ? sc[n][3] * sl2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // a fully masked tile leaves a row at its previous (finite) max
    const float al0 = n0 == -INFINITY ? 1.f : ex2(m0 - n0);
    const float al1 = n1 == -INFINITY ? 1.f : ex2(m1 - n1);
    m0 = n0;
    m1 = n1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int n = 0; n < kTokTiles; ++n) {
      sc[n][0] = n0 == -INFINITY ? 0.f : ex2(sc[n][0] - n0);
      sc[n][1] = n0 == -INFINITY ? 0.f : ex2(sc[n][1] - n0);
      sc[n][2] = n1 == -INFINITY ? 0.f : ex2(sc[n][2] - n1);
      sc[n][3] = n1 == -INFINITY ? 0.f : ex2(sc[n][3] - n1);
      rs0 += sc[n][0] + sc[n][1];
      rs1 += sc[n][2] + sc[n][3];
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
    if (__any_sync(kFull, (al0 != 1.f) | (al1 != 1.f))) {
#pragma unroll
      for (int n = 0; n < kDTiles; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
    }
    // O += P V over the tile's four 16-token k-steps
    {
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int ks = 0; ks < kKeyTile / 16; ++ks) {
        const float* pa0 = sc[2 * ks];
        const float* pa1 = sc[2 * ks + 1];
        uint32_t ph[4], pl[4];
        ph[0] = Ty::pack(pa0[0], pa0[1]);
        ph[1] = Ty::pack(pa0[2], pa0[3]);
        ph[2] = Ty::pack(pa1[0], pa1[1]);
        ph[3] = Ty::pack(pa1[2], pa1[3]);
        {
          const float2 d0 = Ty::unpack(ph[0]), d1 = Ty::unpack(ph[1]);
          const float2 d2 = Ty::unpack(ph[2]), d3 = Ty::unpack(ph[3]);
          pl[0] = Ty::pack(pa0[0] - d0.x, pa0[1] - d0.y);
          pl[1] = Ty::pack(pa0[2] - d1.x, pa0[3] - d1.y);
          pl[2] = Ty::pack(pa1[0] - d2.x, pa1[1] - d2.y);
          pl[3] = Ty::pack(pa1[2] - d3.x, pa1[3] - d3.y);
        }
        const int tok = ks * 16 + rr + ((mi & 1) << 3);
#pragma unroll
        for (int jj = 0; jj < kDTiles / 2; ++jj) {
          uint32_t b[4];
          ldmatrix_x4_trans(b, smem_u32(sv + tok * kRowBytes + swz(tok, 2 * jj + (mi >> 1))));
          Ty::mma(o[2 * jj], ph, b[0], b[1]);
          Ty::mma(o[2 * jj + 1], ph, b[2], b[3]);
          Ty::mma(o[2 * jj], pl, b[0], b[1]);
          Ty::mma(o[2 * jj + 1], pl, b[2], b[3]);
        }
      }
    }
    __syncthreads();  // this buffer is refilled two tiles from now
  }

  // ---- normalise and store ----------------------------------------------------
  l0 += __shfl_xor_sync(kFull, l0, 1);
  l1 += __shfl_xor_sync(kFull, l1, 1);
  l0 += __shfl_xor_sync(kFull, l0, 2);
  l1 += __shfl_xor_sync(kFull, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? r1 : r0;
    const int jj = r / G, g = r % G;
    if (jj >= jn || r >= Mq * G) continue;
    const size_t row = static_cast<size_t>(q0 + j0 + jj) * a.num_q_heads + static_cast<size_t>(h) * G + g;
    const float inv = half ? inv1 : inv0;
#pragma unroll
    for (int n = 0; n < kDTiles; ++n) {
      const float v0 = o[n][half * 2] * inv, v1 = o[n][half * 2 + 1] * inv;
      const size_t oi = row * D + n * 8 + tq;
      if (a.out_f32) {
        *reinterpret_cast<float2*>(static_cast<float*>(a.out) + oi) = make_float2(v0, v1);
      } else {
        *reinterpret_cast<uint32_t*>(static_cast<T*>(a.out) + oi) = Ty::pack(v0, v1);
      }
    }
  }
}

template <typename Ty, int D>
cudaError_t launch_p(const PrefillArgs& a, int max_query_len, cudaStream_t stream) {
  const int Mq = kRowsPerCta / a.group;
  const int tiles = (max_query_len + Mq - 1) / Mq;
  if (tiles < 1) return cudaSuccess;
  auto kern = paged_prefill_kernel<Ty, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PGeo<D>::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(tiles, a.num_kv_heads, a.num_seqs), kThreads, PGeo<D>::kSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, int head_dim, bool bf16, int max_query_len,
                           cudaStream_t stream) {
  if (bf16) {
    return head_dim == 64 ? launch_p<BF16, 64>(a, max_query_len, stream)
                          : launch_p<BF16, 128>(a, max_query_len, stream);
  }
  return head_dim == 64 ? launch_p<F16, 64>(a, max_query_len, stream)
                        : launch_p<F16, 128>(a, max_query_len, stream);
}

}  // namespace pa
