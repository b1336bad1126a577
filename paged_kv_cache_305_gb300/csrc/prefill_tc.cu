// Paged causal prefill on the tcgen05 tensor cores (block sizes 1..64).
//
// The operation ("PagedAttention" glossary, How It Works: the blockwise
// formula with query index i, read token by token): query j of sequence s's
// Q-token chunk sits at position L - Q + j and attends to tokens
// 0 .. L - Q + j of the paged cache.
//
// One CTA per (query tile, kv head, sequence). A query tile is 128 rows =
// 128 / G positions x the G heads of the kv head (the product's M), so each
// K/V tile serves every query head of the group. Key tiles are 64 tokens.
// Roles (8 warps):
//   warps 0-3  one thread per query row: loads the query tile, then for every
//              key tile reads its row of S = q K^T from tensor memory (and at
//              once frees the S columns for the next tile's product), applies
//              the causal limit (only in warps holding a diagonal tile: a
//              warp-uniform branch, so other tiles carry no per-element
//              selects), keeps the running max / sum (base 2), writes the
//              weights into tensor memory (fp16 inputs: rounded to fp16, and
//              the sum adds those rounded weights; bf16: a 16-bit head plus
//              the 16-bit rounding of the remainder), and rescales its output
//              row when the max has grown by more than 2^8 since the last
//              rescale; finally divides by the sum and stores the row.
//   warps 4, 5 producers of the K and the V tiles (each on its own, so K
//              runs ahead of V): whole blocks of 8+ tokens by TMA (one box
//              per block, the whole head dim, straight from the block
//              table), partial / out-of-range blocks by plain loads
//              with zero fill; blocks under 8 tokens row by row with 16-byte
//              cp.async; two stages, a K stage reused as soon as its S is done.
//   warp 6     one thread issues S_{j+1} = Q K_{j+1}^T (smem x smem, M=128,
//              N=64) as soon as the softmax has read S_j;
//   warp 7     one thread issues O += P_j V_j (weights from tensor memory, V
//              from smem read MN-major, N = head dim): one product for fp16,
//              the head and the remainder for bf16.
// Tensor memory (256 columns): S at 0, P at 64, O at 128, so the product of
// the next S overlaps the whole softmax of the current tile. All waits are
// bounded; a wait that gives up is counted and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;  // query rows per CTA = product M
constexpr int kKeys = 64;   // tokens per key tile = N of S
constexpr int kStages = 2;
constexpr int kThreads = 256;
constexpr int kKWarp = 4;    // producer of K tiles
constexpr int kVWarp = 5;    // producer of V tiles
constexpr int kMmaWarp = 6;  // one thread issues the S products
constexpr int kPvWarp = 7;   // one thread issues the P V products
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;    // S, 64 fp32 columns
constexpr uint32_t kColP = 64;   // P: 32 columns of packed 16-bit heads, 32 of remainders
constexpr uint32_t kColO = 128;  // O, head_dim fp32 columns
constexpr float kRescaleLog2 = 8.f;
// fp16 inputs: the weights carry a factor 2^6 (at most 2^14 under the lazy
// rescale), so weights down to 2^-20 of the reference max stay normal fp16
constexpr float kWeightLog2Offset = 6.f;
constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct TcGeo {
  static constexpr int kHalves = D / 64;           // 128-byte row slices of the head dim
  static constexpr int kQHalf = kRows * 128;        // one slice of the query tile
  static constexpr int kQBytes = kHalves * kQHalf;
  // K and V tiles: 8-token groups of the whole head dim (kGroupBytes), in
  // a group the 64-element slices one after the other, each 8 rows of 128
  // bytes; one group of one block is exactly what a cache block holds for
  // 8 of its tokens, so a whole block lands with one copy
  static constexpr int kGroupBytes = kHalves * 1024;
  static constexpr int kTileBytes = kKeys * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K then V
  static constexpr int kBarOff = kQBytes + kStages * kStageBytes;
  // barriers + alignment slack; at least 80 KB so that no more than two CTAs
  // (2 x 256 tensor-memory columns) share an SM
  static constexpr int kSmem = kBarOff + 128 + 1024 > 80 * 1024 ? kBarOff + 128 + 1024 : 80 * 1024;
};
static_assert(kStages == 2, "stage and S buffer of tile j are both j & 1");

// barrier slots (8 bytes each) after the tiles
// Every batch of products is followed by exactly one tcgen05.commit, on one
// barrier; whoever needs that batch finished waits on that barrier (the K
// producer on S, the V producer on P V), so nothing depends on how a commit
// relates to earlier ones.
// Barriers that a waiter could otherwise see two phases ahead are kept per
// tile parity ([2]).
enum : int {
  kBarKFull = 0,   // [2] K tile landed
  kBarVFull = 2,   // [2] V tile landed
  kBarSFull = 4,   // [2] S_j done: S in tensor memory, K stage free
  kBarPFull = 6,   // weights P_j (and any O rescale) in tensor memory
  kBarSFree = 7,   // S_j read into registers: the S columns may be overwritten
  kBarODone = 8,   // [2] P_j V done: O updated, V stage and P columns free
  kBarQFull = 10,  // query tile in shared memory
  kTmemSlot = 11,  // 4-byte TMEM base address
  kBarNever = 12,  // nothing arrives here: the wait of a stalled test launch
};

// Offset of 16-byte chunk (chunk & 7) of row `row` inside one 128-byte-row
// slice (the slice itself, chunk >> 3, is added by the caller).
__device__ __forceinline__ uint32_t sw_off(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// Offset of 16-byte chunk c of token t inside a K or V tile.
template <int D>
__device__ __forceinline__ uint32_t kv_off(int t, int c) {
  return static_cast<uint32_t>((t >> 3) * TcGeo<D>::kGroupBytes + (c >> 3) * 1024) +
         sw_off(t & 7, c);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Packed pairs of fp32 (one 64-bit register) and the paired fp32 multiply-add
// of sm_100-family cores, plus the three-input max: fewer instructions in the
// per-row softmax.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// acc + the two fp16 halves of h, each added exactly as fp32 (mixed-precision add)
__device__ __forceinline__ float add_f16x2(float acc, uint32_t h) {
  asm("{\n .reg .f16 lo, hi;\n mov.b32 {lo, hi}, %1;\n add.rn.f32.f16 %0, lo, %0;\n"
      " add.rn.f32.f16 %0, hi, %0;\n}"
      : "+f"(acc)
      : "r"(h));
  return acc;
}

// Two bf16 values to fp16, round to nearest even (exact inside fp16's normal
// range; beyond +-65504 the result is inf).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return F16::pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Bounded wait made uniform across the warp: every lane of a warp that
// executes warp-collective tensor-memory instructions must take the same path.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(kFull, tc::mbar_wait(bar, parity));
}

// SINGLE: fp16 weights in one P V product with fp16 V (fp16 caches, or bf16
// caches whose value rows were first converted to an fp16 copy, v16);
// otherwise bf16 weights as a head plus the rounding of the remainder.
template <typename Ty, int D, bool SINGLE>
__global__ void __launch_bounds__(kThreads, 2)
paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using Geo = TcGeo<D>;
  using T = typename Ty::T;
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  constexpr int kKSteps = D / 16;

  const int qt = gridDim.x - 1 - blockIdx.x;  // longest tiles first
  const int h = blockIdx.y;
  const int s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.group;
  const int P = kRows / G;  // query positions per tile
  const int shift = a.block_shift;
  const int Lmax = a.max_blocks_per_seq << shift;

  int L = a.seq_lens[s];
  const int q0 = a.query_start[s];
  int Q = a.query_start[s + 1] - q0;
  if (L < 0 || L > Lmax || Q < 0 || Q > L) {
    if (qt == 0 && h == 0 && tid == 0) atomicAdd(a.bad, 1ull);
    L = min(max(L, 0), Lmax);
    Q = min(max(Q, 0), L);
  }
  const int j0 = qt * P;
  if (j0 >= Q) return;
  const int jn = min(P, Q - j0);
  const int last_pos = L - Q + j0 + jn - 1;
  const int ntiles = last_pos / kKeys + 1;

  extern __shared__ unsigned char raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = tc::smem_u32(sm);
  const uint32_t sKV = sQ + Geo::kQBytes;
  const uint32_t bars = sQ + Geo::kBarOff;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  auto sK = [&](int st) { return sKV + static_cast<uint32_t>(st * Geo::kStageBytes); };
  auto sV = [&](int st) { return sK(st) + static_cast<uint32_t>(Geo::kTileBytes); };

  // blocks under 8 tokens arrive row by row: every producer lane signals its
  // own copies' completion on the tile's barrier
  const bool row_copies = shift < 3;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar(kBarKFull + i), row_copies ? 32 : 1);
      tc::mbar_init(bar(kBarVFull + i), row_copies ? 32 : 1);
      tc::mbar_init(bar(kBarSFull + i), 1);
      tc::mbar_init(bar(kBarODone + i), 1);
    }
    tc::mbar_init(bar(kBarPFull), 128);
    tc::mbar_init(bar(kBarSFree), 128);
    tc::mbar_init(bar(kBarQFull), 128);
    tc::mbar_init(bar(kBarNever), 1);
    tc::mbar_init_fence();
  }
  if (warp == 0) tc::tmem_alloc(bar(kTmemSlot), kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + Geo::kBarOff + 8 * kTmemSlot);
  bool ok = true;

  if (warp < 4) {
    // ---------------- query tile: row r = (position j0 + r / G, head h*G + r % G)
    // every load issued before any store, so their latencies overlap
    const T* qb = static_cast<const T*>(a.query);
    constexpr int kPer = kRows * kChunks / 128;  // 16-byte chunks per thread
    uint4 qv[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + 128 * k;
      const int r = i / kChunks, c = i % kChunks;
      const int jj = r / G, g = r % G;
      qv[k] = make_uint4(0u, 0u, 0u, 0u);
      if (r < P * G && jj < jn) {
        const size_t row = static_cast<size_t>(q0 + j0 + jj) * a.num_q_heads +
                           static_cast<size_t>(h) * G + g;
        qv[k] = __ldg(reinterpret_cast<const uint4*>(qb + row * D) + c);
      }
    }
    const uint32_t sign = a.scale_log2 < 0.f ? 0x80008000u : 0u;  // q.k*scale == (-q).k*|scale|
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + 128 * k;
      const int r = i / kChunks, c = i % kChunks;
      const uint4 v = make_uint4(qv[k].x ^ sign, qv[k].y ^ sign, qv[k].z ^ sign, qv[k].w ^ sign);
      st_shared_v4(sQ + (c >> 3) * Geo::kQHalf + sw_off(r, c), v);
    }
    tc::fence_async_smem();
    tc::mbar_arrive(bar(kBarQFull));

    // ---------------- softmax: thread tid owns query row tid (TMEM lane tid)
    const int r = tid;
    const bool row_valid = r < P * G && r / G < jn;
    const int qp = row_valid ? L - Q + j0 + r / G : last_pos;  // causal limit
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl2 = fabsf(a.scale_log2);  // the query tile carries the sign
    float m = -INFINITY, l = 0.f;  // running max (base-2 units) and sum of weights
    for (int j = 0; j < ntiles; ++j) {
      ok = warp_wait(bar(kBarSFull + (j & 1)), (j >> 1) & 1);
      if (!ok) break;
      tc::tc_fence_after();
      float sv[kKeys];
      {
        uint32_t x0[16], x1[16], x2[16], x3[16];
        tc::tmem_ld16(lane_addr + kColS, x0);
        tc::tmem_ld16(lane_addr + kColS + 16, x1);
        tc::tmem_ld16(lane_addr + kColS + 32, x2);
        tc::tmem_ld16(lane_addr + kColS + 48, x3);
        tc::tmem_ld_wait16(x0);
        tc::tmem_ld_wait16(x1);
        tc::tmem_ld_wait16(x2);
        tc::tmem_ld_wait16(x3);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          sv[i] = __uint_as_float(x0[i]);
          sv[16 + i] = __uint_as_float(x1[i]);
          sv[32 + i] = __uint_as_float(x2[i]);
          sv[48 + i] = __uint_as_float(x3[i]);
        }
      }
      // S_j is in registers: S_{j+1} may now be written into the same columns
      tc::tc_fence_before();
      tc::mbar_arrive(bar(kBarSFree));
      // tokens kb + c with c > lim are past this row's causal limit; a warp
      // with any such row takes the masked path, the others carry no
      // per-element selects (warp-uniform branch)
      const int lim = qp - j * kKeys;
      const bool diag = __any_sync(kFull, lim < kKeys - 1);
      bool rescale = false;
      float alpha = 1.f;
      uint32_t ph[32], pl[32];
      auto weights = [&](auto masked) {
        constexpr bool kMasked = decltype(masked)::value;
        if constexpr (kMasked) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) sv[c] = c > lim ? -INFINITY : sv[c];
        }
        // row max of the raw scores: four chains of three-input maxima
        float mx4[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float* v = sv + 16 * q4;
          float mq = max3(v[0], v[1], v[2]);
#pragma unroll
          for (int c = 3; c < 15; c += 2) mq = max3(mq, v[c], v[c + 1]);
          mx4[q4] = fmaxf(mq, v[15]);
        }
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        const float mn = fmaxf(m, mx == -INFINITY ? -INFINITY : mx * sl2);
        rescale = __any_sync(kFull, mn > m + kRescaleLog2);
        if (rescale) {
          alpha = ex2(m - mn);  // 0 on the first tile (m = -inf)
          l *= alpha;
          m = mn;
        }
        // weights 2^(s*sl2 - m), the exponent arguments by paired fp32
        // multiply-adds. SINGLE: the fp16 rounding of each weight (scaled by
        // 2^6), one product with fp16 V, and the row sum adds exactly those
        // rounded weights, so a weight's rounding error cancels between the
        // weighted sum and the sum. Otherwise (bf16 V): a bf16 head (the
        // upper half of the fp32 weight, taken by byte selection) and the
        // bf16 rounding of the remainder, two products (the operands of one
        // product share a type).
        constexpr float kOff = SINGLE ? kWeightLog2Offset : 0.f;
        const uint64_t sl2x2 = f2(sl2, sl2), nmx2 = f2(kOff - m, kOff - m);
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = 2 * i;
          float2 arg = f2_split(f2_fma(f2(sv[c], sv[c + 1]), sl2x2, nmx2));
          if constexpr (kMasked) {  // exact zeros past the limit (also for a zero scale)
            arg.x = c > lim ? -INFINITY : arg.x;
            arg.y = c + 1 > lim ? -INFINITY : arg.y;
          }
          const float p0 = ex2(arg.x), p1 = ex2(arg.y);
          if constexpr (!SINGLE) {
            rs[i & 3] += p0;
            rs[i & 3] += p1;
            const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
            ph[i] = __byte_perm(b0, b1, 0x7632);
            pl[i] = Ty::pack(p0 - __uint_as_float(b0 & 0xffff0000u),
                             p1 - __uint_as_float(b1 & 0xffff0000u));
          } else {
            ph[i] = F16::pack(p0, p1);
            rs[i & 3] = add_f16x2(rs[i & 3], ph[i]);
          }
        }
        l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      };
      if (diag)
        weights(std::true_type{});
      else
        weights(std::false_type{});
      if (j > 0) {
        // P_{j-1} V must be done before P_j overwrites its columns and O is rescaled
        ok = warp_wait(bar(kBarODone + ((j - 1) & 1)), ((j - 1) >> 1) & 1);
        if (!ok) break;
        tc::tc_fence_after();
        if (rescale) {
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            uint32_t x[16];
            tc::tmem_ld16(lane_addr + kColO + 16 * c, x);
            tc::tmem_ld_wait16(x);
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = __float_as_uint(__uint_as_float(x[i]) * alpha);
            tc::tmem_st16(lane_addr + kColO + 16 * c, x);
          }
        }
      }
      {
        uint32_t w[16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = ph[16 * hh + i];
          tc::tmem_st16(lane_addr + kColP + 16 * hh, w);  // weights (two products: head part)
          if constexpr (!SINGLE) {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pl[16 * hh + i];
            tc::tmem_st16(lane_addr + kColP + 32 + 16 * hh, w);  // weights, remainder
          }
        }
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar(kBarPFull));
    }
    if (ok) ok = warp_wait(bar(kBarODone + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1);
    if (ok) {
      tc::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t row = static_cast<size_t>(q0 + j0 + r / G) * a.num_q_heads +
                         static_cast<size_t>(h) * G + r % G;
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        uint32_t x[16];
        tc::tmem_ld16(lane_addr + kColO + 16 * c, x);
        tc::tmem_ld_wait16(x);
        if (!row_valid) continue;
        if (a.out_f32) {
          float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + row * D + 16 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            o[i] = make_float4(__uint_as_float(x[4 * i]) * inv, __uint_as_float(x[4 * i + 1]) * inv,
                               __uint_as_float(x[4 * i + 2]) * inv,
                               __uint_as_float(x[4 * i + 3]) * inv);
        } else {
          uint4* o = reinterpret_cast<uint4*>(static_cast<T*>(a.out) + row * D + 16 * c);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            uint4 w;
            w.x = Ty::pack(__uint_as_float(x[8 * i]) * inv, __uint_as_float(x[8 * i + 1]) * inv);
            w.y = Ty::pack(__uint_as_float(x[8 * i + 2]) * inv, __uint_as_float(x[8 * i + 3]) * inv);
            w.z = Ty::pack(__uint_as_float(x[8 * i + 4]) * inv, __uint_as_float(x[8 * i + 5]) * inv);
            w.w = Ty::pack(__uint_as_float(x[8 * i + 6]) * inv, __uint_as_float(x[8 * i + 7]) * inv);
            o[i] = w;
          }
        }
      }
    }
  } else if (warp == kKWarp || warp == kVWarp) {
    // ---------------- producers: K (or V) tiles of 64 tokens through the block table
    const bool is_v = warp == kVWarp;
    // bf16 caches with SINGLE: the V tiles come from the fp16 copy of the
    // value rows that the conversion pass wrote, block blk of sequence s at
    // block s * max_blocks_per_seq + blk (rejected block ids there are zeros)
    const bool from_v16 = SINGLE && Ty::kIsBf16 && is_v;
    if (from_v16) {
      // the copy is written by the conversion grid just before this one,
      // which may still be running (programmatic dependent launch): wait for
      // it to finish, then order its writes before this warp's TMA reads
      asm volatile("griddepcontrol.wait;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    const T* cache = static_cast<const T*>(from_v16 ? a.v16 : (is_v ? a.value_cache : a.key_cache));
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    const int full0 = is_v ? kBarVFull : kBarKFull;
    const int empty0 = is_v ? kBarODone : kBarSFull;  // stage free once S_j / P_j V is done
    const int B = 1 << shift;
    if (lane == 0 && B >= 8) tc::prefetch_tensormap(map);  // no map below 8
    const int nb = kKeys >> shift;  // blocks per tile (1..8)
    const int32_t* trow = a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq;
    const size_t slot_stride = static_cast<size_t>(a.num_kv_heads) * D;
    // lane i < nb describes block i of a tile: its id (-1: none / out of
    // range) and how many of its B tokens lie before L
    auto block_of = [&](int jt, int& id, int& valid) {
      id = -1;
      valid = 0;
      if (lane < nb && jt < ntiles) {
        const int blk = jt * nb + lane;
        valid = min(max(L - (blk << shift), 0), B);
        if (valid > 0) {
          if (from_v16) {
            id = s * a.max_blocks_per_seq + blk;
          } else {
            id = __ldg(trow + blk);
            if (static_cast<unsigned>(id) >= static_cast<unsigned>(a.num_blocks)) {
              if (!is_v) atomicAdd(a.bad, 1ull);  // counted once, by the K producer
              id = -1;
            }
          }
        }
      }
    };
    // one tensor (K or V) of tile j into stage st: rows of blocks that are
    // not whole and valid by plain loads (zeros past L), whole blocks by TMA,
    // one copy per lane (lane = block * halves + half)
    auto fill = [&](const T* cache, const CUtensorMap* map, uint32_t dst0, uint32_t full_bar,
                    int id, int valid, unsigned whole) {
      if (whole != (1u << nb) - 1u) {
        for (int i = 0; i < nb; ++i) {
          const int idi = __shfl_sync(kFull, id, i);
          const int vi = __shfl_sync(kFull, valid, i);
          if ((whole >> i) & 1u) continue;
          // lane: chunk lane % kChunks of rows lane / kChunks + kLaneRows * u;
          // batches of eight copies per lane: loads first, then stores
          constexpr int kLaneRows = 32 / kChunks;
          const int c = lane % kChunks;
          const T* src = cache + (static_cast<size_t>(max(idi, 0)) << shift) * slot_stride +
                         static_cast<size_t>(h) * D + c * 8;
          for (int t0 = lane / kChunks; t0 < B; t0 += 8 * kLaneRows) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int t = t0 + kLaneRows * u;
              v[u] = make_uint4(0u, 0u, 0u, 0u);
              if (t < vi && idi >= 0)
                v[u] = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(t) * slot_stride));
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int t = t0 + kLaneRows * u;
              if (t < B) st_shared_v4(dst0 + kv_off<D>(i * B + t, c), v[u]);
            }
          }
        }
        tc::fence_async_smem();
      }
      __syncwarp();
      if (lane == 0)
        tc::mbar_arrive_expect_tx(full_bar, static_cast<uint32_t>(__popc(whole)) * B * D * 2);
      __syncwarp();
      if ((whole >> lane) & 1u)  // lane i: block i, all B / 8 groups, whole head dim
        tc::tma_load_5d(dst0 + static_cast<uint32_t>(lane * B * D * 2), map, full_bar, 0, 0, 0,
                        id << (shift - 3), h);
    };
    if (B < 8) {
      // Blocks smaller than a swizzle atom: every row by a 16-byte cp.async
      // (zero fill past L and for rejected ids), two rows per warp
      // instruction. Each lane then arrives on the tile's barrier when its
      // copies have landed (cp.async.mbarrier.arrive.noinc, 32 arrivals per
      // tile); the product thread makes them visible to the tensor cores
      // (fence.proxy.async) after its wait.
      constexpr int kCopies = kKeys * kChunks / 32;  // per lane per tile
      // lane l holds the block ids of rows l and l + 32 of a tile (-1: none)
      // lane l holds the cache slots of rows l and l + 32 of a tile (-1:
      // past L or a rejected block id); slots stay below 2^31
      auto row_slots = [&](int jt, int (&sr)[2]) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int t = jt * kKeys + lane + 32 * u;
          sr[u] = -1;
          if (jt < ntiles && t < L) {
            if (from_v16) {
              sr[u] = ((s * a.max_blocks_per_seq + (t >> shift)) << shift) + (t & (B - 1));
            } else {
              const int id = __ldg(trow + (t >> shift));
              if (static_cast<unsigned>(id) < static_cast<unsigned>(a.num_blocks))
                sr[u] = (id << shift) + (t & (B - 1));
              else if (!is_v && (t & (B - 1)) == 0)
                atomicAdd(a.bad, 1ull);  // counted once per block, by the K producer
            }
          }
        }
      };
      // this lane's 16-byte chunk of a row: c = lane % kChunks, rows
      // kLaneRows * k + lane / kChunks
      constexpr int kLaneRows = 32 / kChunks;
      const int c = lane % kChunks, r0 = lane / kChunks;
      const T* cbase = cache + static_cast<size_t>(h) * D + c * 8;
      int sn[2];
      row_slots(0, sn);
      int j = 0;
      for (; j < ntiles; ++j) {
        const int st = j & 1;
        const int sr[2] = {sn[0], sn[1]};
        row_slots(j + 1, sn);  // next tile's table entries, ahead of time
        if (j >= kStages) {
          ok = warp_wait(bar(empty0 + st), ((j >> 1) - 1) & 1);
          if (!ok) break;
        }
        const uint32_t dst0 = is_v ? sV(st) : sK(st);
#pragma unroll
        for (int k = 0; k < kCopies; ++k) {
          const int row = kLaneRows * k + r0;
          // every lane of this copy reads rows in the same half of the tile
          const int slot = __shfl_sync(kFull, sr[(kLaneRows * k) >> 5], row & 31);
          const bool okr = slot >= 0;
          cp_async_16(dst0 + kv_off<D>(row, c),
                      cbase + static_cast<size_t>(okr ? slot : 0) * slot_stride, okr);
        }
        tc::cp_async_mbar_arrive_noinc(bar(full0 + st));
      }
      // copies still in flight (only after a wait gave up) land before exit
      for (int jj = max(0, j - kStages); jj < j; ++jj)
        tc::mbar_wait(bar(full0 + (jj & 1)), (jj >> 1) & 1);
    } else {
    int id_n, valid_n;
    block_of(0, id_n, valid_n);
    int j = 0;
    for (; j < ntiles; ++j) {
      const int st = j & 1;
      const int id = id_n, valid = valid_n;
      block_of(j + 1, id_n, valid_n);  // next tile's table entries, ahead of time
      const unsigned whole = __ballot_sync(kFull, lane < nb && id >= 0 && valid == B);
      if (j >= kStages) {
        ok = warp_wait(bar(empty0 + st), ((j >> 1) - 1) & 1);
        if (!ok) break;
      }
      fill(cache, map, is_v ? sV(st) : sK(st), bar(full0 + st), id, valid, whole);
    }
    // copies still in flight (only after a wait gave up) must land before exit
    for (int jj = max(0, j - kStages); jj < j; ++jj)
      tc::mbar_wait(bar(full0 + (jj & 1)), (jj >> 1) & 1);
    }
  } else if ((warp == kMmaWarp || warp == kPvWarp) && lane == 0) {
    // ---------------- products: S_j by one thread (warp kMmaWarp), P_j V by
    // another (warp kPvWarp), so the next S never queues behind the issue of
    // a P V; descriptors built once, moved by adding (byte offset >> 4) to
    // the start-address field. Each thread's commits track its own products.
    const uint32_t id_s = tc::idesc_f16(kRows, kKeys, Ty::kIsBf16, false);
    // P V: fp16 weights with fp16 V, or bf16 weight parts with bf16 V
    const uint32_t id_o = tc::idesc_f16(kRows, D, SINGLE ? false : Ty::kIsBf16, true);
    const uint64_t dq0 = tc::sdesc_sw128(sQ, 16, 1024);
    // K read K-major: 8-token groups kGroupBytes apart (SBO)
    const uint64_t dk0 = tc::sdesc_sw128(sK(0), 16, Geo::kGroupBytes);
    // V read MN-major: 8-token groups kGroupBytes apart (SBO), the two
    // 64-element slices of the head dim 1024 bytes apart (LBO)
    const uint64_t dv0 = tc::sdesc_sw128(sV(0), Geo::kHalves > 1 ? 1024 : 16, Geo::kGroupBytes);
    constexpr uint64_t kStageStep = Geo::kStageBytes >> 4;
    constexpr uint64_t kVStep = (2 * Geo::kGroupBytes) >> 4;  // 16 tokens
    auto kstep = [](int ks) {  // K-major: slice ks / 4, 32 bytes per 16 elements
      return static_cast<uint64_t>(((ks >> 2) * 1024 + (ks & 3) * 32) >> 4);
    };
    uint32_t last_bar = 0, last_parity = 0;  // this thread's latest commit
    // a stalled test launch first waits on a barrier that nothing signals:
    // the wait runs out, no product is issued, and every warp winds down
    if (a.stall_for_test) ok = tc::mbar_wait(bar(kBarNever), 0);
    if (warp == kMmaWarp) {
      for (int j = 0; j < ntiles && ok; ++j) {
        // S_j overwrites S_{j-1}: wait until the softmax has read it
        ok = (j == 0 ? tc::mbar_wait(bar(kBarQFull), 0)
                     : tc::mbar_wait(bar(kBarSFree), (j - 1) & 1)) &&
             tc::mbar_wait(bar(kBarKFull + (j & 1)), (j >> 1) & 1);
        if (!ok) break;
        tc::tc_fence_after();
        if (row_copies) tc::fence_async_smem();  // rows written by cp.async, seen by the products
        const int st = j & 1;
        const uint64_t dk = dk0 + st * kStageStep;
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks) {
          const uint64_t qoff =
              static_cast<uint64_t>(((ks >> 2) * Geo::kQHalf + (ks & 3) * 32) >> 4);
          tc::mma_ss(tmem + kColS, dq0 + qoff, dk + kstep(ks), id_s, ks > 0 ? 1u : 0u);
        }
        tc::tc_commit(bar(kBarSFull + st));
        last_bar = bar(kBarSFull + st);
        last_parity = (j >> 1) & 1;
      }
    } else {
      for (int j = 0; j < ntiles && ok; ++j) {
        const int b = j & 1;
        ok = tc::mbar_wait(bar(kBarPFull), j & 1) &&
             tc::mbar_wait(bar(kBarVFull + b), (j >> 1) & 1);
        if (!ok) break;
        tc::tc_fence_after();
        if (row_copies) tc::fence_async_smem();
        const uint32_t colP = tmem + kColP;
        const uint64_t dv = dv0 + b * kStageStep;
        // fp16: one product; bf16: the weights' head part, then the remainder
#pragma unroll
        for (int part = 0; part < (SINGLE ? 1 : 2); ++part) {
#pragma unroll
          for (int ks = 0; ks < kKeys / 16; ++ks)
            tc::mma_ts(tmem + kColO, colP + part * 32 + ks * 8, dv + ks * kVStep,
                       id_o, (j > 0 || part > 0 || ks > 0) ? 1u : 0u);
        }
        tc::tc_commit(bar(kBarODone + b));
        last_bar = bar(kBarODone + b);
        last_parity = (j >> 1) & 1;
      }
    }
    // nothing this thread issued may still be running when the CTA ends
    if (last_bar != 0) tc::mbar_wait(last_bar, last_parity);
  }

  if (!ok && lane == 0) atomicAdd(a.timeouts, 1ull);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Conversion pass for bf16 caches: the value rows of every sequence, in
// logical order, to an fp16 copy: block j of sequence s (its B slots x Hkv x
// d) at block s * max_blocks_per_seq + j of v16, so the prefill's V tiles are
// fp16 and P V is one product. One CTA per (block j, sequence s); only the
// rows before the sequence's length are written (the prefill reads no
// others); a rejected block id gives zero rows (the prefill's K producer
// counts it). Values beyond fp16's range become +-inf.
template <int D>
__global__ void __launch_bounds__(256) v16_convert_kernel(const PrefillArgs a) {
  // the prefill launched after this kernel may start its CTAs once every CTA
  // here has started (programmatic dependent launch); only its V producer
  // waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int j = blockIdx.x, s = blockIdx.y;
  const int shift = a.block_shift;
  const int B = 1 << shift;
  const int Lmax = a.max_blocks_per_seq << shift;
  const int L = min(max(a.seq_lens[s], 0), Lmax);
  const int rows = min(L - (j << shift), B);
  if (rows <= 0) return;
  const int id = __ldg(a.block_tables + static_cast<size_t>(s) * a.max_blocks_per_seq + j);
  const bool ok = static_cast<unsigned>(id) < static_cast<unsigned>(a.num_blocks);
  const size_t row_chunks = static_cast<size_t>(a.num_kv_heads) * D / 8;  // 16-byte chunks per slot
  const size_t n = static_cast<size_t>(rows) * row_chunks;
  const uint4* src = reinterpret_cast<const uint4*>(a.value_cache) +
                     (static_cast<size_t>(ok ? id : 0) << shift) * row_chunks;
  uint4* dst = reinterpret_cast<uint4*>(a.v16) +
               ((static_cast<size_t>(s) * a.max_blocks_per_seq + j) << shift) * row_chunks;
  for (size_t i = threadIdx.x; i < n; i += 256) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (ok) {
      const uint4 v = __ldg(src + i);
      w = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                     bf16x2_to_f16x2(v.w));
    }
    dst[i] = w;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (f == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && p != nullptr) {
      f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

// One cache [num_blocks * B slots, Hkv, d] viewed, innermost first, as
// (64 elements of a head-dim slice, 8 slots of a group, d / 64 slices,
// slot groups, kv head); a box is one block of one kv head: (64, 8, d / 64,
// B / 8, 1), which lands in the tile layout of the products (8-token groups
// of the whole head dim, 128-byte swizzle). Only for B >= 8 (a multiple of 8
// slots); smaller blocks are copied row by row and get no map.
bool encode_cache_map(CUtensorMap* map, const void* cache, bool bf16, long long num_slots, int hkv,
                      int d, int block_size) {
  if (block_size < 8) {
    *map = CUtensorMap{};
    return true;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(hkv) * d * 2;  // bytes per slot
  const cuuint64_t dims[5] = {64, 8, static_cast<cuuint64_t>(d / 64),
                              static_cast<cuuint64_t>(num_slots / 8), static_cast<cuuint64_t>(hkv)};
  const cuuint64_t strides[4] = {row, 128, 8 * row, static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[5] = {64, 8, static_cast<cuuint32_t>(d / 64),
                             static_cast<cuuint32_t>(block_size / 8), 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
             const_cast<void*>(cache), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// after_convert: launched right behind the conversion pass as a programmatic
// dependent launch (its CTAs may start while the pass is finishing).
template <typename Ty, int D, bool SINGLE>
cudaError_t launch_kernel(const CUtensorMap& km, const CUtensorMap& vm, const PrefillArgs& a,
                          int tiles, bool after_convert, cudaStream_t stream) {
  auto kern = paged_prefill_tc_kernel<Ty, D, SINGLE>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcGeo<D>::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, a.num_kv_heads, a.num_seqs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = TcGeo<D>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_convert ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, km, vm, a);
}

template <typename Ty, int D>
cudaError_t launch_tc(const PrefillArgs& a, int max_query_len, cudaStream_t stream) {
  const int P = kRows / a.group;
  const int tiles = (max_query_len + P - 1) / P;
  if (tiles < 1) return cudaSuccess;
  const int B = 1 << a.block_shift;
  const long long slots = static_cast<long long>(a.num_blocks) << a.block_shift;
  CUtensorMap km, vm;
  if (!encode_cache_map(&km, a.key_cache, Ty::kIsBf16, slots, a.num_kv_heads, D, B))
    return cudaErrorInvalidValue;
  if (Ty::kIsBf16 && a.v16 != nullptr) {
    // bf16 with a workspace: the value rows to fp16 first, then one P V product
    const long long vslots =
        static_cast<long long>(a.num_seqs) * a.max_blocks_per_seq << a.block_shift;
    if (!encode_cache_map(&vm, a.v16, false, vslots, a.num_kv_heads, D, B))
      return cudaErrorInvalidValue;
    v16_convert_kernel<D><<<dim3(a.max_blocks_per_seq, a.num_seqs), 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_kernel<Ty, D, true>(km, vm, a, tiles, true, stream);
  }
  if (!encode_cache_map(&vm, a.value_cache, Ty::kIsBf16, slots, a.num_kv_heads, D, B))
    return cudaErrorInvalidValue;
  return launch_kernel<Ty, D, !Ty::kIsBf16>(km, vm, a, tiles, false, stream);
}

}  // namespace

bool prefill_tc_supported(int block_size, long long num_slots) {
  return block_size >= 1 && block_size <= 64 && num_slots <= 0x7fffffffll;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, int head_dim, bool bf16, int max_query_len,
                              cudaStream_t stream) {
  if (bf16) {
    return head_dim == 64 ? launch_tc<BF16, 64>(a, max_query_len, stream)
                          : launch_tc<BF16, 128>(a, max_query_len, stream);
  }
  return head_dim == 64 ? launch_tc<F16, 64>(a, max_query_len, stream)
                        : launch_tc<F16, 128>(a, max_query_len, stream);
}

}  // namespace pa
