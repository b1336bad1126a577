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
// Work decomposition. A "row" is one (sequence, kv head); all G = Hq / Hkv
// query heads of the kv head are computed together, so every K/V byte is read
// from HBM once per call. A row is cut into partitions of `partition_tokens`
// tokens (split-K). The kernel is persistent: a grid of (SMs x CTAs per SM)
// CTAs, each taking a contiguous run of partitions in (sequence, kv head,
// partition) order, balanced by tokens (plus a fixed cost per partition).
// Consecutive partitions of one row inside a CTA form a "segment": the online
// softmax simply continues across their boundary. A segment that is a whole
// row writes `out`; a row cut between CTAs leaves one piece per CTA (fp32
// normalised output + base-2 log-sum-exp) in the workspace, and the last CTA
// to finish a piece of that row merges the pieces in order and writes `out`.
//
// Inside a CTA, each of the 4 warps owns every 4th 16-token tile of each
// segment and streams K/V through its own cp.async ring, which runs on across
// segment boundaries. Table ids are loaded several tiles ahead into registers
// (one per lane for one of the tile's 16 rows) and handed out by shuffles.
// Per tile a warp computes the scores of 16 query-head rows (the group,
// zero-padded) against 16 tokens with m16n8k16 tensor-core products, updates
// the online softmax in fp32 with base-2 exponents, and accumulates P.V with
// the same instruction (weights as a 16-bit head plus a 16-bit remainder, so
// their rounding stays far below the output tolerance). At a segment end the
// four warps' states are merged by log-sum-exp through shared memory.
//
// Shared-memory K/V/q rows are 16-byte-chunk XOR swizzled (chunk ^ (row & 7))
// so the 8 row addresses of every ldmatrix phase fall in distinct banks.
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileTokens = 16;  // tokens per warp tile (the k extent of the P.V product)
constexpr int kRows = 16;        // query-head rows of one tensor-core tile
constexpr int kIdDepth = 4;      // tiles whose table ids are in flight ahead of their copies
constexpr unsigned kFull = 0xffffffffu;

struct Seg {
  int s, h;      // sequence, kv head
  int t0, t1;    // token range [t0, t1)
  int ntiles;    // 16-token tiles in the range
  int piece;     // -1: the segment is the whole row; else its piece index
  int npieces;   // pieces of the row (when piece >= 0)
  int pad;
};

template <int D, int STAGES>
struct Geometry {
  static constexpr int kRowBytes = D * 2;                    // one K or V row
  static constexpr int kChunks = kRowBytes / 16;             // 16-byte chunks per row
  static constexpr int kTileBytes = kTileTokens * kRowBytes;  // 16 rows
  static constexpr int kStageBytes = 2 * kTileBytes;          // K tile + V tile
  static constexpr int kPipeBytes = kWarps * STAGES * kStageBytes;
  static constexpr int kQBytes = kRows * kRowBytes;
  static constexpr int kMLBytes = kWarps * 2 * kRows * 4;  // per-warp row max and sum
  static constexpr int kFacBytes = (kWarps + 2) * kRows * 4;
  static constexpr int kSegBytes = kMaxSegments * static_cast<int>(sizeof(Seg));
  static constexpr int kFixedBytes = kQBytes + kPipeBytes + kMLBytes + kFacBytes + kSegBytes;
  static constexpr int kOStride = D + 4;  // fp32 row stride of a warp's state in the merge area
  static constexpr int kQRegs = kRows * kChunks / kThreads;  // 16-byte q chunks per thread
  static_assert(kRows * kChunks % kThreads == 0, "q chunks must divide among threads");
  static_assert(kPipeBytes >= kWarps * 8, "the schedule scan reuses the ring area");
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk ^ (row & 7)) << 4);
}

// Owner CTA of scheduling position `pos` in [0, W): floor(pos * C / W). The
// host checks that W * C fits in 63 bits.
__device__ __forceinline__ int owner_of(long long pos, int C, long long W) {
  return static_cast<int>((pos * C) / W);
}
// First scheduling position owned by CTA c: ceil(c * W / C) (LLONG_MAX past the end).
__device__ __forceinline__ long long first_pos(int c, int C, long long W) {
  if (c >= C) return LLONG_MAX;
  const long long q = W / C, r = W % C;
  return static_cast<long long>(c) * q + (static_cast<long long>(c) * r + C - 1) / C;
}

template <typename Ty, int D, int STAGES>
__global__ void __launch_bounds__(kThreads)
paged_decode_kernel(const DecodeArgs a) {
  using Geo = Geometry<D, STAGES>;
  using T = typename Ty::T;
  constexpr int kRowBytes = Geo::kRowBytes;
  constexpr int kChunks = Geo::kChunks;
  constexpr int kKSteps = D / 16;  // k-steps of the q.K product over head_dim
  constexpr int kNTiles = D / 8;   // n-tiles of the P.V product over head_dim
  constexpr int kRowsPerCopy = 32 / kChunks;          // rows one warp-wide copy covers
  constexpr int kCopies = kTileTokens / kRowsPerCopy;  // copies per lane per tensor per tile
  constexpr int kOS = Geo::kOStride;

  const int cta = blockIdx.x;
  const int C = gridDim.x;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int shift = a.block_shift;
  const int bmask = (1 << shift) - 1;
  const int G = a.group;
  const int S = a.num_seqs;
  const int Hkv = a.num_kv_heads;
  const int Pt = a.partition_tokens;
  const int Lmax = a.max_blocks_per_seq << shift;
  const long long UW = static_cast<long long>(Pt) + kUnitCost;  // weight of a full partition

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sPipe = smem + Geo::kQBytes;
  float* sML = reinterpret_cast<float*>(sPipe + Geo::kPipeBytes);  // [warp][m|l][row]
  float* sFac = sML + kWarps * 2 * kRows;  // [warp][row] weights, [row] 1/sum, [row] lse
  Seg* sSeg = reinterpret_cast<Seg*>(sFac + (kWarps + 2) * kRows);
  float* sMerge =
      reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(sSeg) + Geo::kSegBytes);
  __shared__ long long sW[3];  // base position of the first / last unit's sequence
  __shared__ int sRange[6];    // first unit (s, h, p), end unit (s, h, p)
  __shared__ int sFlag;

  auto clamp_len = [&](int L) { return L < 0 ? 0 : (L > Lmax ? Lmax : L); };
  auto nparts_of = [&](int L) { return L > 0 ? (L + Pt - 1) / Pt : 1; };

  // ======================= schedule ========================================
  // Every CTA computes the same prefix of sequence weights: a sequence of
  // length L has ceil(L / Pt) partitions per kv head (one if L is 0), each
  // weighing its tokens plus kUnitCost. CTA c owns the partitions whose start
  // position lies in [first_pos(c), first_pos(c + 1)).
  const int per = (S + kThreads - 1) / kThreads;
  const int s_lo = min(S, tid * per), s_hi = min(S, s_lo + per);
  long long mine = 0;
  for (int s = s_lo; s < s_hi; ++s) {
    const int raw = a.seq_lens[s];
    const int L = clamp_len(raw);
    if (raw != L && cta == 0) atomicAdd(a.bad, 1ull);
    mine += static_cast<long long>(Hkv) * (L + static_cast<long long>(nparts_of(L)) * kUnitCost);
  }
  long long incl = mine;  // inclusive scan within the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long v = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += v;
  }
  long long* sScan = reinterpret_cast<long long*>(sPipe);
  if (lane == 31) sScan[warp] = incl;
  if (tid == 0) {
    sRange[0] = S; sRange[1] = 0; sRange[2] = 0;
    sRange[3] = S; sRange[4] = 0; sRange[5] = 0;
  }
  __syncthreads();
  long long base = incl - mine;
  for (int w = 0; w < warp; ++w) base += sScan[w];
  long long Wtot = 0;
  for (int w = 0; w < kWarps; ++w) Wtot += sScan[w];
  const long long tau_b = first_pos(cta, C, Wtot);
  const long long tau_e = first_pos(cta + 1, C, Wtot);
  // the first partition at or after position tau, found by the thread whose
  // chunk of sequences holds tau
  for (int which = 0; which < 2; ++which) {
    const long long tau = which == 0 ? tau_b : tau_e;
    const bool claim = (tid == 0 && tau <= 0) || (mine > 0 && base < tau && tau <= base + mine);
    if (!claim) continue;
    long long sb = base;
    int rs = s_hi, rh = 0, rp = 0;
    long long rbase = base + mine;
    for (int s = s_lo; s < s_hi; ++s) {
      const int L = clamp_len(a.seq_lens[s]);
      const int np = nparts_of(L);
      const long long w = L + static_cast<long long>(np) * kUnitCost;
      const long long se = sb + Hkv * w;
      if (tau <= sb) {
        rs = s; rh = 0; rp = 0; rbase = sb;
        break;
      }
      if (tau < se) {
        const long long r = tau - sb;
        int h = static_cast<int>(r / w);
        long long p = (r - h * w + UW - 1) / UW;
        if (p >= np) {
          p = 0;
          ++h;
        }
        if (h >= Hkv) {
          rs = s + 1; rh = 0; rp = 0; rbase = se;
        } else {
          rs = s; rh = h; rp = static_cast<int>(p); rbase = sb;
        }
        break;
      }
      sb = se;
    }
    sRange[which * 3 + 0] = rs;
    sRange[which * 3 + 1] = rh;
    sRange[which * 3 + 2] = rp;
    sW[1 + which] = rbase;
  }
  __syncthreads();
  const long long Rb = static_cast<long long>(sRange[0]) * Hkv + sRange[1];
  const int pb = sRange[2];
  const long long Re = static_cast<long long>(sRange[3]) * Hkv + sRange[4];
  const int pe = sRange[5];
  if (Rb == Re && pb == pe) return;  // this CTA owns no partition
  const long long nseg_total = (Re - Rb) + (pe > 0 ? 1 : 0);

  // ======================= per-warp state ===================================
  unsigned char* wpipe = sPipe + warp * STAGES * Geo::kStageBytes;
  const size_t slot_stride = static_cast<size_t>(Hkv) * D;  // elements per slot
  const T* kcache = static_cast<const T*>(a.key_cache);
  const T* vcache = static_cast<const T*>(a.value_cache);
  const int cc = lane % kChunks;  // this lane's 16-byte chunk of a row
  const int cr = lane / kChunks;  // this lane's first row of a tile
  const float sl2 = a.scale_log2;
  const int tq = 2 * (lane & 3);  // first token column this lane holds in an 8-token n-tile
  const int P = a.max_partitions;

  uint32_t qa[kKSteps][4];
  float m0, m1, l0, l1;
  float o[kNTiles][4];
  auto reset_state = [&]() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int n = 0; n < kNTiles; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  };
  auto load_qa = [&]() {
    const int mi = lane >> 3, rr = lane & 7;
    const int row = rr + ((mi & 1) << 3);
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
      const int c = 2 * kk + (mi >> 1);
      ldmatrix_x4(qa[kk], smem_u32(sQ + row * kRowBytes + swz(row, c)));
    }
  };
  // q rows of a segment, as this thread's share of 16-byte chunks (zero rows >= G)
  uint4 qreg[Geo::kQRegs];
  auto fetch_q = [&](const Seg& g) {
    const T* qg = static_cast<const T*>(a.query) +
                  (static_cast<size_t>(g.s) * a.num_q_heads + static_cast<size_t>(g.h) * G) * D;
#pragma unroll
    for (int k = 0; k < Geo::kQRegs; ++k) {
      const int i = tid + k * kThreads;
      const int r = i / kChunks, c = i % kChunks;
      qreg[k] = r < G ? *reinterpret_cast<const uint4*>(qg + r * D + c * 8)
                      : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  auto store_q = [&]() {
#pragma unroll
    for (int k = 0; k < Geo::kQRegs; ++k) {
      const int i = tid + k * kThreads;
      const int r = i / kChunks, c = i % kChunks;
      *reinterpret_cast<uint4*>(sQ + r * kRowBytes + swz(r, c)) = qreg[k];
    }
  };

  for (long long b0 = 0; b0 < nseg_total; b0 += kMaxSegments) {
    const int nseg = static_cast<int>(min(static_cast<long long>(kMaxSegments), nseg_total - b0));
    // ---- segment records of this batch -------------------------------------
    if (tid < nseg) {
      const long long R = Rb + b0 + tid;
      const int s = static_cast<int>(R / Hkv), h = static_cast<int>(R % Hkv);
      const int L = clamp_len(a.seq_lens[s]);
      const int np = nparts_of(L);
      const int pf = R == Rb ? pb : 0;
      const int pl = R == Re ? pe : np;
      Seg g;
      g.s = s;
      g.h = h;
      g.t0 = pf * Pt;
      g.t1 = static_cast<int>(min(static_cast<long long>(pl) * Pt, static_cast<long long>(L)));
      g.ntiles = (g.t1 - g.t0 + kTileTokens - 1) / kTileTokens;
      g.piece = -1;
      g.npieces = 1;
      g.pad = 0;
      if (!(pf == 0 && pl == np)) {
        // a row cut between CTAs: walk its owners in order to find this CTA's
        // piece index and the number of pieces
        const long long w = L + static_cast<long long>(np) * kUnitCost;
        const long long rowbase = R == Rb ? sW[1] + static_cast<long long>(sRange[1]) * w
                                          : sW[2] + static_cast<long long>(sRange[4]) * w;
        int c = owner_of(rowbase, C, Wtot);
        int k = 0, me = -1;
        while (true) {
          if (c == cta) me = k;
          if (c + 1 >= C) break;
          const long long pn = (first_pos(c + 1, C, Wtot) - rowbase + UW - 1) / UW;
          if (pn >= np) break;
          c = owner_of(rowbase + pn * UW, C, Wtot);
          ++k;
        }
        g.piece = me;
        g.npieces = k + 1;
      }
      sSeg[tid] = g;
    }
    __syncthreads();
    // q of the first segment
    fetch_q(sSeg[0]);
    store_q();
    __syncthreads();
    load_qa();
    reset_state();
    if (nseg > 1) fetch_q(sSeg[1]);

    // ---- tile iterators over this warp's tiles of the batch ------------------
    // (segment, tile j): the warp's tiles are j = warp, warp + 4, ... of each segment
    auto advance = [&](int& sg, int& j) {
      j += kWarps;
      while (sg < nseg && j >= sSeg[sg].ntiles) {
        ++sg;
        j = warp;
      }
    };
    // table id of row (lane & 15) of a tile (validated when the copy is issued)
    auto load_id = [&](int sg, int j) -> int {
      if (sg >= nseg) return 0;
      const Seg& g = sSeg[sg];
      const int t = g.t0 + j * kTileTokens + (lane & 15);
      if (t >= g.t1) return 0;
      return __ldg(a.block_tables + static_cast<size_t>(g.s) * a.max_blocks_per_seq + (t >> shift));
    };
    int id_sg = 0, id_j = warp - kWarps;
    advance(id_sg, id_j);
    int is_sg = id_sg, is_j = id_j;
    int idq[kIdDepth];
#pragma unroll
    for (int k = 0; k < kIdDepth; ++k) {
      idq[k] = load_id(id_sg, id_j);
      advance(id_sg, id_j);
    }
    int issued = 0;
    auto issue = [&]() {
      if (is_sg < nseg) {
        const Seg& g = sSeg[is_sg];
        const int tb = g.t0 + is_j * kTileTokens;
        unsigned char* sk = wpipe + (issued % STAGES) * Geo::kStageBytes;
        unsigned char* sv = sk + Geo::kTileBytes;
        const T* kb = kcache + static_cast<size_t>(g.h) * D + cc * 8;
        const T* vb = vcache + static_cast<size_t>(g.h) * D + cc * 8;
#pragma unroll
        for (int i = 0; i < kCopies; ++i) {
          const int r = cr + i * kRowsPerCopy;
          const int phys = __shfl_sync(kFull, idq[0], r);
          const int t = tb + r;
          const bool in = t < g.t1;
          const bool ok = in && static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks);
          if (in && !ok && cc == 0) atomicAdd(a.bad, 1ull);  // rejected id: its rows read as zero
          const size_t slot = ok ? (static_cast<size_t>(phys) << shift) + (t & bmask) : 0;
          const uint32_t off = r * kRowBytes + swz(r, cc);
          cp_async_16(smem_u32(sk + off), kb + slot * slot_stride, ok);
          cp_async_16(smem_u32(sv + off), vb + slot * slot_stride, ok);
        }
        ++issued;
        advance(is_sg, is_j);
      }
#pragma unroll
      for (int k = 0; k + 1 < kIdDepth; ++k) idq[k] = idq[k + 1];
      idq[kIdDepth - 1] = load_id(id_sg, id_j);
      advance(id_sg, id_j);
      cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < STAGES - 1; ++i) issue();
    int consumed = 0;

    for (int sg = 0; sg < nseg; ++sg) {
      const Seg g = sSeg[sg];
      // ---- this warp's tiles of the segment --------------------------------
      for (int j = warp; j < g.ntiles; j += kWarps) {
        cp_async_wait<STAGES - 2>();
        __syncwarp();
        issue();
        const unsigned char* sk = wpipe + (consumed % STAGES) * Geo::kStageBytes;
        const unsigned char* sv = sk + Geo::kTileBytes;
        ++consumed;
        const int valid = g.t1 - (g.t0 + j * kTileTokens);  // >= 1

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
          for (int e = 0; e < 4; ++e) {
            if (tk[e] >= valid) x[e] = x[e + 4] = -INFINITY;
          }
        }
        float mx0 = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        float mx1 = fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);
        m0 = n0;
        m1 = n1;
        // weights as A fragments: rows lane/4 (pa[0], pa[2]) and lane/4 + 8
        // (pa[1], pa[3]); each is a 16-bit head (pa) plus the 16-bit rounding of
        // the remainder (pl), so the weights keep about 16 significant bits
        float p[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          p[e] = ex2(x[e] - n0);
          p[e + 4] = ex2(x[e + 4] - n1);
        }
        uint32_t pa[4], pl[4];
        pa[0] = Ty::pack(p[0], p[1]);
        pa[1] = Ty::pack(p[4], p[5]);
        pa[2] = Ty::pack(p[2], p[3]);
        pa[3] = Ty::pack(p[6], p[7]);
        {
          const int src[4][2] = {{0, 1}, {4, 5}, {2, 3}, {6, 7}};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 hd = Ty::unpack(pa[e]);
            pl[e] = Ty::pack(p[src[e][0]] - hd.x, p[src[e][1]] - hd.y);
          }
        }
        l0 = l0 * al0 + ((p[0] + p[1]) + (p[2] + p[3]));
        l1 = l1 * al1 + ((p[4] + p[5]) + (p[6] + p[7]));
        if (__any_sync(kFull, (al0 != 1.f) | (al1 != 1.f))) {
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
          for (int jj = 0; jj < kNTiles / 2; ++jj) {
            uint32_t b[4];
            ldmatrix_x4_trans(b, smem_u32(sv + tok * kRowBytes + swz(tok, 2 * jj + (mi >> 1))));
            Ty::mma(o[2 * jj], pa, b[0], b[1]);
            Ty::mma(o[2 * jj + 1], pa, b[2], b[3]);
            Ty::mma(o[2 * jj], pl, b[0], b[1]);
            Ty::mma(o[2 * jj + 1], pl, b[2], b[3]);
          }
        }
      }

      // ---- segment end: merge the four warps (log-sum-exp) --------------------
      l0 += __shfl_xor_sync(kFull, l0, 1);
      l1 += __shfl_xor_sync(kFull, l1, 1);
      l0 += __shfl_xor_sync(kFull, l0, 2);
      l1 += __shfl_xor_sync(kFull, l1, 2);
      {
        float* sMw = sMerge + warp * G * kOS;
        const int r0 = lane >> 2;
        if (r0 < G) {
#pragma unroll
          for (int n = 0; n < kNTiles; ++n)
            *reinterpret_cast<float2*>(sMw + r0 * kOS + n * 8 + tq) = make_float2(o[n][0], o[n][1]);
        }
        if (r0 + 8 < G) {
#pragma unroll
          for (int n = 0; n < kNTiles; ++n)
            *reinterpret_cast<float2*>(sMw + (r0 + 8) * kOS + n * 8 + tq) =
                make_float2(o[n][2], o[n][3]);
        }
        if ((lane & 3) == 0) {
          sML[(warp * 2 + 0) * kRows + r0] = m0;
          sML[(warp * 2 + 0) * kRows + r0 + 8] = m1;
          sML[(warp * 2 + 1) * kRows + r0] = l0;
          sML[(warp * 2 + 1) * kRows + r0 + 8] = l1;
        }
      }
      __syncthreads();
      if (tid < G) {
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
      const bool more = sg + 1 < nseg;
      if (more) store_q();  // q of the next segment (every warp is past its ldmatrix of this one)
      __syncthreads();
      if (more) {
        load_qa();
        if (sg + 2 < nseg) fetch_q(sSeg[sg + 2]);
      }
      reset_state();

      const size_t row0 = static_cast<size_t>(g.s) * a.num_q_heads + static_cast<size_t>(g.h) * G;
      auto merged = [&](int gr, int c) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += sFac[w * kRows + gr] * sMerge[(w * G + gr) * kOS + c];
        return v * sFac[kWarps * kRows + gr];
      };
      if (g.piece < 0) {
        for (int i = tid; i < G * (D / 2); i += kThreads) {
          const int gr = i / (D / 2), c = 2 * (i % (D / 2));
          const float v0 = merged(gr, c), v1 = merged(gr, c + 1);
          const size_t oi = (row0 + gr) * D + c;
          if (a.out_f32) {
            *reinterpret_cast<float2*>(static_cast<float*>(a.out) + oi) = make_float2(v0, v1);
          } else {
            *reinterpret_cast<uint32_t*>(static_cast<T*>(a.out) + oi) = Ty::pack(v0, v1);
          }
        }
      } else {
        // store this piece; the last of the row's pieces to arrive merges them in order
        for (int i = tid; i < G * D; i += kThreads) {
          const int gr = i / D, c = i % D;
          a.ws_out[((row0 + gr) * P + g.piece) * D + c] = merged(gr, c);
        }
        if (tid < G) a.ws_lse[(row0 + tid) * P + g.piece] = sFac[(kWarps + 1) * kRows + tid];
        __syncthreads();
        int* counter = a.ws_count + static_cast<size_t>(g.s) * Hkv + g.h;
        if (tid == 0) {
          __threadfence();
          const int prev = atomicAdd(counter, 1);
          sFlag = prev == g.npieces - 1;
          if (sFlag) __threadfence();
        }
        __syncthreads();
        if (sFlag) {
          const int n = g.npieces;
          for (int i = tid; i < G * D; i += kThreads) {
            const int gr = i / D, c = i % D;
            const float* lse = a.ws_lse + (row0 + gr) * P;
            const float* po = a.ws_out + (row0 + gr) * P * D + c;
            float M = -INFINITY;
            for (int k = 0; k < n; ++k) M = fmaxf(M, __ldcg(lse + k));
            float num = 0.f, den = 0.f;
            int k = 0;
            for (; k + 4 <= n; k += 4) {
              float lv[4], ov[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                lv[e] = __ldcg(lse + k + e);
                ov[e] = __ldcg(po + static_cast<size_t>(k + e) * D);
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float wgt = ex2(lv[e] - M);
                den += wgt;
                num += wgt * ov[e];
              }
            }
            for (; k < n; ++k) {
              const float wgt = ex2(__ldcg(lse + k) - M);
              den += wgt;
              num += wgt * __ldcg(po + static_cast<size_t>(k) * D);
            }
            const float v = num / den;
            const size_t oi = (row0 + gr) * D + c;
            if (a.out_f32) {
              static_cast<float*>(a.out)[oi] = v;
            } else {
              static_cast<T*>(a.out)[oi] = Ty::cvt(v);
            }
          }
          if (tid == 0) *counter = 0;  // ready for the next call on this workspace
        }
      }
      __syncthreads();  // the merge area, factors and flag are reused at the next segment end
    }
    cp_async_wait<0>();
  }
}

template <typename Ty, int D, int STAGES>
cudaError_t plan_typed(int group, int* ctas_per_sm, size_t* smem) {
  const size_t bytes = static_cast<size_t>(Geometry<D, STAGES>::kFixedBytes) +
                       static_cast<size_t>(kWarps) * group * Geometry<D, STAGES>::kOStride * 4;
  auto kern = paged_decode_kernel<Ty, D, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, bytes);
  if (e != cudaSuccess) return e;
  *ctas_per_sm = n;
  *smem = bytes;
  return cudaSuccess;
}

template <typename Ty, int D, int STAGES>
cudaError_t launch_typed(const DecodeArgs& a, long long grid, size_t smem, cudaStream_t stream) {
  paged_decode_kernel<Ty, D, STAGES><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename Ty, int D>
cudaError_t launch_d(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  // three ring stages when two CTAs still fit on an SM, else two
  int n3 = 0, n2 = 0;
  size_t m3 = 0, m2 = 0;
  cudaError_t e = plan_typed<Ty, D, 3>(a.group, &n3, &m3);
  if (e != cudaSuccess) return e;
  int stages = 3, per_sm = n3;
  size_t smem = m3;
  if (n3 < 2) {
    e = plan_typed<Ty, D, 2>(a.group, &n2, &m2);
    if (e != cudaSuccess) return e;
    if (n2 > n3) {
      stages = 2;
      per_sm = n2;
      smem = m2;
    }
  }
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  long long grid = static_cast<long long>(per_sm) * num_sms;
  const long long units =
      static_cast<long long>(a.num_seqs) * a.num_kv_heads * a.max_partitions;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  return stages == 3 ? launch_typed<Ty, D, 3>(a, grid, smem, stream)
                     : launch_typed<Ty, D, 2>(a, grid, smem, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int head_dim, bool bf16, int num_sms,
                          cudaStream_t stream) {
  if (bf16) {
    return head_dim == 64 ? launch_d<BF16, 64>(a, num_sms, stream)
                          : launch_d<BF16, 128>(a, num_sms, stream);
  }
  return head_dim == 64 ? launch_d<F16, 64>(a, num_sms, stream)
                        : launch_d<F16, 128>(a, num_sms, stream);
}

}  // namespace pa
