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
// Work decomposition. The G = Hq / Hkv query heads of a kv head are computed
// together, so every K/V byte is read from HBM once per call. Kv heads are
// taken in groups of Hc (4, 2 or 1, dividing Hkv); a "row" is one (sequence,
// head group), cut into partitions of `partition_tokens` tokens (split-K).
// The kernel is persistent: a grid of (SMs x CTAs per SM) CTAs, each taking a
// contiguous run of partitions in (sequence, head group, partition) order,
// balanced by tokens (plus a fixed cost per partition). Consecutive
// partitions of one row inside a CTA form a "segment": the online softmax
// simply continues across their boundary. A segment that is a whole row
// writes `out`; a row cut between CTAs leaves one piece per CTA and head
// (fp32 normalised output + base-2 log-sum-exp) in the workspace, and the
// last piece of a head to arrive merges its pieces in order and writes `out`.
//
// Inside a CTA the 4 warps are spread over the Hc heads of the group (4 / Hc
// warps per head, splitting the head's 16-token tiles round-robin), so at any
// time the warps read the same token slots of adjacent heads: with Hc = 4 one
// slot's reads are 4 x d x 2 contiguous bytes. Each warp streams K/V through
// its own cp.async ring, which runs on across segment boundaries; table ids
// are loaded several tiles ahead into registers (one per lane for one of the
// tile's 16 rows) and handed out by shuffles. Per 16-token tile a warp
// computes S^T = K q^T with m16n8k16 tensor-core products (16 tokens x 8 query
// heads per product, so a group of up to 8 heads costs one product per 16
// dims), updates the online softmax per head in fp32 with base-2 exponents,
// transposes the weights in registers (movmatrix) into the B operand, and
// accumulates O^T = V^T P^T with the same instruction (weights as a 16-bit
// head plus a 16-bit remainder, so their rounding stays far below the output
// tolerance). At a segment end a warp that owns its head alone finalizes from
// registers; warps sharing a head first merge through shared memory.
//
// Shared-memory K/V rows are 16-byte-chunk XOR swizzled (chunk ^ (row & 7)) so
// the 8 row addresses of every ldmatrix phase fall in distinct banks.
#include <cuda_runtime.h>
#include <limits.h>

#include <atomic>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileTokens = 16;  // tokens per warp tile (the k extent of the P.V product)
constexpr int kRows = 16;        // query-head rows of one tensor-core tile
constexpr int kIdDepth = 8;      // tiles whose table ids are in flight ahead of their copies
constexpr int kDynMaxParts = 32;  // rows with more partitions get no dynamic ones
constexpr unsigned kFull = 0xffffffffu;

struct Seg {
  int s, hg;     // sequence, kv-head group
  int t0, t1;    // token range [t0, t1)
  int ntiles;    // 16-token tiles in the range
  int piece;     // -1: the segment is the whole row; else its piece index
  int npieces;   // pieces of the row (when piece >= 0)
  int L;         // the sequence's length
};

template <int D, int STAGES>
struct Geometry {
  static constexpr int kRowBytes = D * 2;                    // one K or V row
  static constexpr int kChunks = kRowBytes / 16;             // 16-byte chunks per row
  static constexpr int kTileBytes = kTileTokens * kRowBytes;  // 16 rows
  static constexpr int kStageBytes = 2 * kTileBytes;          // K tile + V tile
  static constexpr int kPipeBytes = kWarps * STAGES * kStageBytes;
  static constexpr int kMLBytes = kWarps * 2 * kRows * 4;  // per-warp row max and sum
  static constexpr int kSegBytes = kMaxSegments * static_cast<int>(sizeof(Seg));
  static constexpr int kFixedBytes = kPipeBytes + kMLBytes + kSegBytes;
  static constexpr int kOStride = D + 4;  // fp32 row stride of a warp's state in the merge area
  static_assert(kPipeBytes >= 2 * kWarps * 8, "the schedule scan reuses the ring area");
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

// APPEND: the step's new K/V rows are given (pa_decode_append): the tile
// holding each sequence's newest token reads that row from them and stores
// it into its cache slot. Without it the kernel carries none of that code.
template <typename Ty, int D, int STAGES, int NT, bool APPEND>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 3 : 2)
paged_decode_kernel(const DecodeArgs a) {
  using Geo = Geometry<D, STAGES>;
  using T = typename Ty::T;
  constexpr int kRowBytes = Geo::kRowBytes;
  constexpr int kChunks = Geo::kChunks;
  constexpr int kKSteps = D / 16;  // k-steps of the q.K product over head_dim
  constexpr int kMT = D / 16;      // 16-dim m-tiles of the P.V product over head_dim
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
  const int Hc = a.heads_per_cta;
  const int NG = Hkv / Hc;          // head groups per sequence (rows per sequence)
  const int Wh = kWarps / Hc;       // warps per head
  const int hi = warp / Wh;         // this warp's head within the group
  const int ws = warp % Wh;         // this warp's share of the head's tiles
  const int Pt = a.partition_tokens;
  const int Lmax = a.max_blocks_per_seq << shift;
  const long long UW = static_cast<long long>(Pt) + kUnitCost;  // weight of a full partition

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sPipe = smem;
  float* sML = reinterpret_cast<float*>(sPipe + Geo::kPipeBytes);  // [warp][m|l][row]
  Seg* sSeg = reinterpret_cast<Seg*>(sML + kWarps * 2 * kRows);
  float* sMerge =  // [warp][G][kOS], present only when warps share a head
      reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(sSeg) + Geo::kSegBytes);
  __shared__ long long sW[3];  // base position of the first / last unit's row
  __shared__ int sRange[6];    // first unit (hg, s, p), end unit (hg, s, p)

  auto clamp_len = [&](int L) { return L < 0 ? 0 : (L > Lmax ? Lmax : L); };
  auto nparts_of = [&](int L) { return L > 0 ? (L + Pt - 1) / Pt : 1; };
  // The trailing d partitions of every row of sequence s are handed out one
  // by one at run time (claimed through a counter in the workspace) to the
  // CTAs that finish their static share first; the rest of the row (its
  // "lead", at least one partition) is split statically. d is a function of
  // the data alone: about dyn_percent % of the partitions of a row of up to
  // 4 partitions and twice that share of a longer row's, the fraction
  // rounded up or down by a fixed per-sequence offset.
  auto dyn_of = [&](int np, int s) -> int {
    // long rows (more than kDynMaxParts partitions) keep a static split: they
    // balance well already, and their many pieces would make the merge long
    if (a.dyn_percent <= 0 || np < 2 || np > kDynMaxParts) return 0;
    const long long pct = np <= 4 ? a.dyn_percent : 2 * a.dyn_percent;
    const long long off = (static_cast<unsigned>(s) * 2654435761u) % 100u;
    const long long d = (static_cast<long long>(np) * pct + off) / 100;
    return static_cast<int>(min(d, static_cast<long long>(np - 1)));
  };
  struct Lead {
    int L, npl, d;  // length, lead partitions, dynamic partitions
    long long w;    // weight of the lead: its tokens + kUnitCost per partition
  };
  auto lead_of = [&](int s) -> Lead {
    Lead r;
    r.L = clamp_len(a.seq_lens[s]);
    const int np = nparts_of(r.L);
    r.d = dyn_of(np, s);
    r.npl = np - r.d;
    r.w = min(static_cast<long long>(r.L), static_cast<long long>(r.npl) * Pt) +
          static_cast<long long>(r.npl) * kUnitCost;
    return r;
  };

  // ======================= schedule ========================================
  // Rows are taken head-group-major: row R = hg * S + s, so the rows of one
  // head group over all sequences are consecutive and sequences that share
  // prefix blocks (consecutive in the batch) re-read them back to back, from
  // L2. The lead of a row of length L has npl partitions (one if L is 0),
  // each weighing its tokens plus kUnitCost; every CTA computes the same
  // prefix of these weights over the sequences (one pass, Wseq), and the
  // positions of head group hg are offset by hg * Wseq. CTA c owns the lead
  // partitions whose start position lies in [first_pos(c), first_pos(c + 1)).
  const int per = (S + kThreads - 1) / kThreads;
  const int s_lo = min(S, tid * per), s_hi = min(S, s_lo + per);
  long long mine = 0, dmine = 0;
  for (int s = s_lo; s < s_hi; ++s) {
    const int raw = a.seq_lens[s];
    const Lead ld = lead_of(s);
    if (raw != ld.L && cta == 0) atomicAdd(a.bad, 1ull);
    mine += ld.w;
    dmine += ld.d;
  }
  long long incl = mine;  // inclusive scan within the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long v = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += v;
  }
  long long dincl = dmine;  // the same for the dynamic partitions
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long v = __shfl_up_sync(kFull, dincl, off);
    if (lane >= off) dincl += v;
  }
  long long* sScan = reinterpret_cast<long long*>(sPipe);
  if (lane == 31) {
    sScan[warp] = incl;
    sScan[kWarps + warp] = dincl;
  }
  if (tid == 0) {
    sRange[0] = NG; sRange[1] = 0; sRange[2] = 0;
    sRange[3] = NG; sRange[4] = 0; sRange[5] = 0;
    sW[1] = sW[2] = 0;
  }
  __syncthreads();
  long long base = incl - mine, dbase = dincl - dmine;  // this thread's chunk starts
  for (int w = 0; w < warp; ++w) {
    base += sScan[w];
    dbase += sScan[kWarps + w];
  }
  long long Wseq = 0, Dseq = 0;
  for (int w = 0; w < kWarps; ++w) {
    Wseq += sScan[w];
    Dseq += sScan[kWarps + w];
  }
  const long long Wtot = Wseq * NG;
  const long long Dtot = a.ws_claim != nullptr ? Dseq * NG : 0;  // dynamic partitions
  const long long tau_b = first_pos(cta, C, Wtot);
  const long long tau_e = first_pos(cta + 1, C, Wtot);
  // the first lead partition at or after position tau, found by the thread
  // whose chunk of sequences holds tau's offset within its head group
  for (int which = 0; which < 2; ++which) {
    const long long tau = which == 0 ? tau_b : tau_e;
    if (tau >= Wtot) continue;  // past the last partition: the default (NG, 0, 0)
    const int hg = static_cast<int>(tau / Wseq);
    const long long off = tau - hg * Wseq;
    const bool claim = (tid == 0 && off <= 0) || (mine > 0 && base < off && off <= base + mine);
    if (!claim) continue;
    long long sb = base;
    int rs = s_hi, rp = 0;
    long long rbase = base + mine;
    for (int s = s_lo; s < s_hi; ++s) {
      const Lead ld = lead_of(s);
      const long long se = sb + ld.w;
      if (off <= sb) {
        rs = s; rp = 0; rbase = sb;
        break;
      }
      if (off < se) {
        const long long p = (off - sb + UW - 1) / UW;
        if (p >= ld.npl) {
          rs = s + 1; rp = 0; rbase = se;
        } else {
          rs = s; rp = static_cast<int>(p); rbase = sb;
        }
        break;
      }
      sb = se;
    }
    // (hg, S) is the first row of the next head group
    sRange[which * 3 + 0] = hg;
    sRange[which * 3 + 1] = rs;
    sRange[which * 3 + 2] = rp;
    sW[1 + which] = static_cast<long long>(hg) * Wseq + rbase;  // the row's base position
  }
  __syncthreads();
  const long long Rb = static_cast<long long>(sRange[0]) * S + sRange[1];
  const int pb = sRange[2];
  const long long Re = static_cast<long long>(sRange[3]) * S + sRange[4];
  const int pe = sRange[5];
  const long long nseg_total =
      (Rb == Re && pb == pe) ? 0 : (Re - Rb) + (pe > 0 ? 1 : 0);  // static segments

  // static lead pieces of the row whose lead starts at position rowbase and
  // has npl partitions: their number, and the index of the one CTA c0 owns
  auto lead_pieces = [&](long long rowbase, int npl, int c0, int* me) -> int {
    int c = owner_of(rowbase, C, Wtot);
    int k = 0;
    *me = -1;
    while (true) {
      if (c == c0) *me = k;
      if (c + 1 >= C) break;
      const long long pn = (first_pos(c + 1, C, Wtot) - rowbase + UW - 1) / UW;
      if (pn >= npl) break;
      c = owner_of(rowbase + pn * UW, C, Wtot);
      ++k;
    }
    return k + 1;
  };

  // ======================= per-warp state ===================================
  unsigned char* wpipe = sPipe + warp * STAGES * Geo::kStageBytes;
  const size_t slot_stride = static_cast<size_t>(Hkv) * D;  // elements per slot
  const T* kcache = static_cast<const T*>(a.key_cache);
  const T* vcache = static_cast<const T*>(a.value_cache);
  const int cc = lane % kChunks;  // this lane's 16-byte chunk of a row
  const int cr = lane / kChunks;  // this lane's first row of a tile
  const float sl2 = a.scale_log2;
  const int r8 = lane >> 2;       // fragment row this lane holds (token of a score tile, dim of an output tile)
  const int tq = 2 * (lane & 3);  // first fragment column this lane holds (query head)
  const int P = a.max_partitions;

  // q as the B operand of the score product (B[d][head] = q[head][d]), the
  // running max / sum of the heads this lane holds (nt*8 + tq, +1), and the
  // output accumulator O^T[d][head] as MT tiles of 16 dims x 8*NT heads
  uint32_t qb[kKSteps][NT][2];
  float mrun[NT][2], lrun[NT][2];
  float o[kMT][NT][4];
  auto reset_state = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mrun[nt][0] = mrun[nt][1] = -INFINITY;
      lrun[nt][0] = lrun[nt][1] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
  };
  auto load_q = [&](const Seg& g) {
    const T* qh = static_cast<const T*>(a.query) +
                  (static_cast<size_t>(g.s) * a.num_q_heads +
                   static_cast<size_t>(g.hg * Hc + hi) * G) * D;
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int head = nt * 8 + r8;
        const T* qr = qh + head * D + kk * 16 + tq;
        qb[kk][nt][0] = head < G ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
        qb[kk][nt][1] = head < G ? *reinterpret_cast<const uint32_t*>(qr + 8) : 0u;
      }
    }
  };

  // one dynamic partition: the record of the u-th one (head group u / Dseq,
  // sequences in order, each row's trailing partitions in order), written
  // by the thread whose chunk of sequences holds it
  auto locate_unit = [&](unsigned long long u) {
    const int hg = static_cast<int>(u / static_cast<unsigned long long>(Dseq));
    const long long off = static_cast<long long>(u) - static_cast<long long>(hg) * Dseq;
    if (!(dmine > 0 && dbase <= off && off < dbase + dmine)) return;
    long long acc_d = dbase, acc_w = base;
    for (int s = s_lo; s < s_hi; ++s) {
      const Lead ld = lead_of(s);
      if (off < acc_d + ld.d) {
        const int i = static_cast<int>(off - acc_d);
        int me;
        const int ns = lead_pieces(static_cast<long long>(hg) * Wseq + acc_w, ld.npl, -1, &me);
        Seg g;
        g.s = s;
        g.hg = hg;
        g.t0 = (ld.npl + i) * Pt;
        g.t1 = static_cast<int>(min(static_cast<long long>(g.t0) + Pt, static_cast<long long>(ld.L)));
        g.ntiles = (g.t1 - g.t0 + kTileTokens - 1) / kTileTokens;
        g.piece = ns + i;
        g.npieces = ns + ld.d;
        g.L = ld.L;
        sSeg[0] = g;
        return;
      }
      acc_d += ld.d;
      acc_w += ld.w;
    }
  };

  // Batches of segment records: the static segments (kMaxSegments at a time),
  // then one claimed dynamic partition at a time until none is left.
  __shared__ unsigned long long sClaim;
  long long b0 = 0;
  for (;;) {
    int nseg;
    if (b0 < nseg_total) {
      nseg = static_cast<int>(min(static_cast<long long>(kMaxSegments), nseg_total - b0));
      // ---- static segment records of this batch ---------------------------------
      if (tid < nseg) {
        const long long R = Rb + b0 + tid;
        const int hg = static_cast<int>(R / S), s = static_cast<int>(R % S);
        const Lead ld = lead_of(s);
        const int pf = R == Rb ? pb : 0;
        const int pl = R == Re ? pe : ld.npl;
        Seg g;
        g.s = s;
        g.hg = hg;
        g.t0 = pf * Pt;
        g.t1 = static_cast<int>(min(static_cast<long long>(pl) * Pt, static_cast<long long>(ld.L)));
        g.ntiles = (g.t1 - g.t0 + kTileTokens - 1) / kTileTokens;
        g.piece = -1;
        g.npieces = 1;
        g.L = ld.L;
        const bool cut = !(pf == 0 && pl == ld.npl);
        if (cut || ld.d > 0) {
          // a row cut between CTAs, or one with dynamic partitions: its lead
          // pieces in CTA order come first, then one piece per dynamic partition
          int me = 0, ns = 1;
          if (cut) ns = lead_pieces(R == Rb ? sW[1] : sW[2], ld.npl, cta, &me);
          g.piece = me;
          g.npieces = ns + ld.d;
        }
        sSeg[tid] = g;
      }
      b0 += nseg;
    } else {
      if (Dtot == 0) break;
      if (tid == 0) sClaim = atomicAdd(a.ws_claim, 1ull);
      __syncthreads();
      const unsigned long long u = sClaim;
      if (u >= static_cast<unsigned long long>(Dtot)) break;  // uniform
      locate_unit(u);
      nseg = 1;
    }
    __syncthreads();
    load_q(sSeg[0]);
    reset_state();

    // ---- tile iterators over this warp's tiles of the batch ------------------
    // (segment, tile j): the warp's tiles are j = ws, ws + Wh, ... of each segment
    auto advance = [&](int& sg, int& j) {
      j += Wh;
      while (sg < nseg && j >= sSeg[sg].ntiles) {
        ++sg;
        j = ws;
      }
    };
    // cache slot of row (lane & 15) of a tile: kNoSlot past the segment's
    // end and for a rejected block id (counted once per row, its rows read
    // as zero); the copies then need one shuffle and one multiply each
    constexpr uint32_t kNoSlot = 0xffffffffu;
    auto load_id = [&](int sg, int j) -> uint32_t {
      if (sg >= nseg) return kNoSlot;
      const Seg& g = sSeg[sg];
      const int t = g.t0 + j * kTileTokens + (lane & 15);
      if (t >= g.t1) return kNoSlot;
      const int phys = __ldg(a.block_tables + static_cast<size_t>(g.s) * a.max_blocks_per_seq + (t >> shift));
      if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) {
        if (lane < 16) atomicAdd(a.bad, 1ull);
        return kNoSlot;
      }
      return (static_cast<uint32_t>(phys) << shift) + static_cast<uint32_t>(t & bmask);
    };
    int id_sg = 0, id_j = ws - Wh;
    advance(id_sg, id_j);
    int is_sg = id_sg, is_j = id_j;
    uint32_t idq[kIdDepth];
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
        const int h = g.hg * Hc + hi;
        const size_t hoff = static_cast<size_t>(h) * D + cc * 8;
        const T* kb = kcache + hoff;
        const T* vb = vcache + hoff;
        // with new K/V given, the one tile holding the sequence's newest token
        // (warp-uniform test) reads that row from them; the compute step then
        // stores it into its slot
        const bool fresh_tile = APPEND && g.t1 == g.L && tb + kTileTokens >= g.L;
        const int fresh_r = fresh_tile ? g.L - 1 - tb : -1;
        auto copy = [&](int i, bool check_fresh) {
          const int r = cr + i * kRowsPerCopy;
          const uint32_t sl = __shfl_sync(kFull, idq[0], r);
          const bool ok = sl != kNoSlot;
          const size_t slot = ok ? sl : 0u;
          const uint32_t off = r * kRowBytes + swz(r, cc);
          if (check_fresh && r == fresh_r) {
            const size_t nrow = (static_cast<size_t>(g.s) * Hkv + h) * D + cc * 8;
            cp_async_16(smem_u32(sk + off), static_cast<const T*>(a.new_key) + nrow, true);
            cp_async_16(smem_u32(sv + off), static_cast<const T*>(a.new_value) + nrow, true);
          } else {
            cp_async_16(smem_u32(sk + off), kb + slot * slot_stride, ok);
            cp_async_16(smem_u32(sv + off), vb + slot * slot_stride, ok);
          }
        };
        if (fresh_tile) {
#pragma unroll
          for (int i = 0; i < kCopies; ++i) copy(i, true);
        } else {
#pragma unroll
          for (int i = 0; i < kCopies; ++i) copy(i, false);
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
    for (int i = 0; i < STAGES - 1; ++i) issue();  // the loop issues the STAGES-th ahead
    int consumed = 0;

    for (int sg = 0; sg < nseg; ++sg) {
      const Seg g = sSeg[sg];
      // ---- this warp's tiles of the segment --------------------------------
      for (int j = ws; j < g.ntiles; j += Wh) {
        // refill the slot the previous tile used before waiting, so STAGES
        // tiles are in flight while this one lands
        __syncwarp();
        issue();
        cp_async_wait<STAGES - 1>();
        __syncwarp();
        const unsigned char* sk = wpipe + (consumed % STAGES) * Geo::kStageBytes;
        const unsigned char* sv = sk + Geo::kTileBytes;
        ++consumed;
        const int valid = g.t1 - (g.t0 + j * kTileTokens);  // >= 1
        if (APPEND && g.t1 == g.L && valid <= kTileTokens && lane < kChunks) {
          // the tile holds the newest token: its row (from the new K/V, now in
          // shared memory) goes to its cache slot; a rejected block id stores
          // nothing (already counted when the tile was loaded)
          const int fresh_phys = __ldg(a.block_tables + static_cast<size_t>(g.s) * a.max_blocks_per_seq +
                                       ((g.L - 1) >> shift));
          if (static_cast<unsigned>(fresh_phys) < static_cast<unsigned>(a.num_blocks)) {
            const int r = valid - 1;
            const size_t dst = ((static_cast<size_t>(fresh_phys) << shift) + ((g.L - 1) & bmask)) * slot_stride +
                               static_cast<size_t>(g.hg * Hc + hi) * D + lane * 8;
            const uint32_t off = r * kRowBytes + swz(r, lane);
            *reinterpret_cast<uint4*>(const_cast<T*>(kcache) + dst) = *reinterpret_cast<const uint4*>(sk + off);
            *reinterpret_cast<uint4*>(const_cast<T*>(vcache) + dst) = *reinterpret_cast<const uint4*>(sv + off);
          }
        }

        // scores S^T[token][head] = K q^T: 16 tokens x 8*NT heads. The k-steps
        // alternate between two accumulators to halve the dependent chain.
        float sc[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][0][e] = sc[nt][1][e] = 0.f;
        {
          const int mi = lane >> 3, rr = lane & 7;
          const int tok = rr + ((mi & 1) << 3);
#pragma unroll
          for (int kk = 0; kk < kKSteps; ++kk) {
            uint32_t ka[4];
            ldmatrix_x4(ka, smem_u32(sk + tok * kRowBytes + swz(tok, 2 * kk + (mi >> 1))));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) Ty::mma(sc[nt][kk & 1], ka, qb[kk][nt][0], qb[kk][nt][1]);
          }
        }
        // per head (column): lane holds tokens r8 and r8 + 8 for heads nt*8 + tq, +1
        const bool lo_ok = r8 < valid, hi_ok = r8 + 8 < valid;
        uint32_t ph[NT][2], pl[NT][2];  // weights as B fragments: 16-bit head, 16-bit remainder
        float al[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float x[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = (sc[nt][0][e] + sc[nt][1][e]) * sl2;
          if (!lo_ok) x[0] = x[1] = -INFINITY;
          if (!hi_ok) x[2] = x[3] = -INFINITY;
          float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            mx[c] = fmaxf(mx[c], __shfl_xor_sync(kFull, mx[c], 4));
            mx[c] = fmaxf(mx[c], __shfl_xor_sync(kFull, mx[c], 8));
            mx[c] = fmaxf(mx[c], __shfl_xor_sync(kFull, mx[c], 16));
            const float mn = fmaxf(mrun[nt][c], mx[c]);
            al[nt][c] = ex2(mrun[nt][c] - mn);
            mrun[nt][c] = mn;
          }
          float p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) p[e] = ex2(x[e] - mrun[nt][e & 1]);
          lrun[nt][0] = lrun[nt][0] * al[nt][0] + (p[0] + p[2]);
          lrun[nt][1] = lrun[nt][1] * al[nt][1] + (p[1] + p[3]);
          // C-fragment pairs (token row, two heads) transposed into B-fragment
          // pairs (head row, two tokens): tokens 0-7 and 8-15
          const uint32_t h0 = Ty::pack(p[0], p[1]), h1 = Ty::pack(p[2], p[3]);
          const float2 d0 = Ty::unpack(h0), d1 = Ty::unpack(h1);
          const uint32_t r0v = Ty::pack(p[0] - d0.x, p[1] - d0.y);
          const uint32_t r1v = Ty::pack(p[2] - d1.x, p[3] - d1.y);
          ph[nt][0] = movmatrix_trans(h0);
          ph[nt][1] = movmatrix_trans(h1);
          pl[nt][0] = movmatrix_trans(r0v);
          pl[nt][1] = movmatrix_trans(r1v);
        }
        bool rescale = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) rescale |= (al[nt][0] != 1.f) | (al[nt][1] != 1.f);
        if (__any_sync(kFull, rescale)) {
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              o[mt][nt][0] *= al[nt][0];
              o[mt][nt][1] *= al[nt][1];
              o[mt][nt][2] *= al[nt][0];
              o[mt][nt][3] *= al[nt][1];
            }
        }
        // O^T[d][head] += V^T P^T: A = V^T read transposed from the [token][d] tile
        {
          const int mi = lane >> 3, rr = lane & 7;
          const int tok = rr + ((mi >> 1) << 3);
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt) {
            uint32_t va[4];
            ldmatrix_x4_trans(va, smem_u32(sv + tok * kRowBytes + swz(tok, 2 * mt + (mi & 1))));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              Ty::mma(o[mt][nt], va, ph[nt][0], ph[nt][1]);
              Ty::mma(o[mt][nt], va, pl[nt][0], pl[nt][1]);
            }
          }
        }
      }

      // ---- segment end --------------------------------------------------------
      // full per-head sums: add the partial sums of the 8 lanes holding the same heads
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          lrun[nt][c] += __shfl_xor_sync(kFull, lrun[nt][c], 4);
          lrun[nt][c] += __shfl_xor_sync(kFull, lrun[nt][c], 8);
          lrun[nt][c] += __shfl_xor_sync(kFull, lrun[nt][c], 16);
        }
      if (Wh > 1) {
        // warps sharing a head: the others hand their state to the head's first warp
        if (ws != 0) {
          float* sMw = sMerge + warp * G * kOS;
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int head = nt * 8 + tq + (e & 1), d = mt * 16 + r8 + ((e & 2) << 2);
                if (head < G) sMw[head * kOS + d] = o[mt][nt][e];
              }
          if (r8 == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                sML[(warp * 2 + 0) * kRows + nt * 8 + tq + c] = mrun[nt][c];
                sML[(warp * 2 + 1) * kRows + nt * 8 + tq + c] = lrun[nt][c];
              }
          }
        }
        __syncthreads();
        if (ws == 0) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int head = nt * 8 + tq + c;
              float M = mrun[nt][c];
              for (int w = warp + 1; w < warp + Wh; ++w) M = fmaxf(M, sML[(w * 2) * kRows + head]);
              const float f = M == -INFINITY ? 0.f : ex2(mrun[nt][c] - M);
              lrun[nt][c] *= f;
#pragma unroll
              for (int mt = 0; mt < kMT; ++mt) {
                o[mt][nt][c] *= f;
                o[mt][nt][c + 2] *= f;
              }
              for (int w = warp + 1; w < warp + Wh; ++w) {
                const float gw = M == -INFINITY ? 0.f : ex2(sML[(w * 2) * kRows + head] - M);
                lrun[nt][c] += gw * sML[(w * 2 + 1) * kRows + head];
                if (head < G) {
                  const float* sMw = sMerge + w * G * kOS + head * kOS;
#pragma unroll
                  for (int mt = 0; mt < kMT; ++mt) {
                    o[mt][nt][c] += gw * sMw[mt * 16 + r8];
                    o[mt][nt][c + 2] += gw * sMw[mt * 16 + r8 + 8];
                  }
                }
              }
              mrun[nt][c] = M;
            }
        }
        __syncthreads();  // the merge area is reused at the next segment end
      }

      if (ws == 0) {
        // finalize this warp's head: query heads nt*8 + tq (+1) of its group (those < G)
        const int h = g.hg * Hc + hi;
        const size_t row0 = static_cast<size_t>(g.s) * a.num_q_heads + static_cast<size_t>(h) * G;
        float inv[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) inv[nt][c] = lrun[nt][c] > 0.f ? 1.f / lrun[nt][c] : 0.f;
        if (g.piece < 0) {
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int head = nt * 8 + tq + (e & 1), d = mt * 16 + r8 + ((e & 2) << 2);
                if (head < G) {
                  const float v = o[mt][nt][e] * inv[nt][e & 1];
                  const size_t oi = (row0 + head) * D + d;
                  if (a.out_f32) {
                    static_cast<float*>(a.out)[oi] = v;
                  } else {
                    static_cast<T*>(a.out)[oi] = Ty::cvt(v);
                  }
                }
              }
        } else {
          // store this piece; the head's last piece to arrive merges them in order
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int head = nt * 8 + tq + (e & 1), d = mt * 16 + r8 + ((e & 2) << 2);
                if (head < G) a.ws_out[((row0 + head) * P + g.piece) * D + d] = o[mt][nt][e] * inv[nt][e & 1];
              }
          if (r8 == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int head = nt * 8 + tq + c;
                if (head < G)
                  a.ws_lse[(row0 + head) * P + g.piece] =
                      lrun[nt][c] > 0.f ? mrun[nt][c] + __log2f(lrun[nt][c]) : -INFINITY;
              }
          }
          __syncwarp();
          int* counter = a.ws_count + static_cast<size_t>(g.s) * Hkv + h;
          int last = 0;
          if (lane == 0) {
            __threadfence();
            last = atomicAdd(counter, 1) == g.npieces - 1;
            if (last) __threadfence();
          }
          last = __shfl_sync(kFull, last, 0);
          if (last) {
            // merge the head's pieces: lane handles 4 consecutive columns of a row
            const int n = g.npieces;
            constexpr int kC4 = D / 4;
            for (int e = lane; e < G * kC4; e += 32) {
              const int gr = e / kC4, c4 = e % kC4;
              const float* lse = a.ws_lse + (row0 + gr) * P;
              const float* po = a.ws_out + (row0 + gr) * P * D + c4 * 4;
              float M = -INFINITY;
              for (int k = 0; k < n; ++k) M = fmaxf(M, __ldcg(lse + k));
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              float den = 0.f;
              int k = 0;
              for (; k + 4 <= n; k += 4) {
                float lv[4];
                float4 ov[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  lv[u] = __ldcg(lse + k + u);
                  ov[u] = __ldcg(reinterpret_cast<const float4*>(po + static_cast<size_t>(k + u) * D));
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float wgt = M == -INFINITY ? 0.f : ex2(lv[u] - M);
                  den += wgt;
                  acc.x += wgt * ov[u].x;
                  acc.y += wgt * ov[u].y;
                  acc.z += wgt * ov[u].z;
                  acc.w += wgt * ov[u].w;
                }
              }
              for (; k < n; ++k) {
                const float wgt = M == -INFINITY ? 0.f : ex2(__ldcg(lse + k) - M);
                const float4 ov = __ldcg(reinterpret_cast<const float4*>(po + static_cast<size_t>(k) * D));
                den += wgt;
                acc.x += wgt * ov.x;
                acc.y += wgt * ov.y;
                acc.z += wgt * ov.z;
                acc.w += wgt * ov.w;
              }
              const float iv = den > 0.f ? 1.f / den : 0.f;
              const size_t oi = (row0 + gr) * D + c4 * 4;
              if (a.out_f32) {
                *reinterpret_cast<float4*>(static_cast<float*>(a.out) + oi) =
                    make_float4(acc.x * iv, acc.y * iv, acc.z * iv, acc.w * iv);
              } else {
                uint2 pk;
                pk.x = Ty::pack(acc.x * iv, acc.y * iv);
                pk.y = Ty::pack(acc.z * iv, acc.w * iv);
                *reinterpret_cast<uint2*>(static_cast<T*>(a.out) + oi) = pk;
              }
            }
            if (lane == 0) *counter = 0;  // ready for the next call on this workspace
          }
        }
      }
      reset_state();
      if (sg + 1 < nseg) load_q(sSeg[sg + 1]);
    }
    cp_async_wait<0>();
    __syncthreads();  // the segment records are rewritten for the next batch
  }
  if (a.ws_claim != nullptr && tid == 0) {
    // the last CTA to finish (every claim made) leaves the counters at zero
    __threadfence();
    if (atomicAdd(a.ws_done, 1u) == static_cast<unsigned>(C - 1)) {
      atomicExch(a.ws_claim, 0ull);
      atomicExch(a.ws_done, 0u);
    }
  }
}

template <typename Ty, int D, int STAGES, int NT, bool APPEND>
cudaError_t plan_typed(const DecodeArgs& a, int* ctas_per_sm, size_t* smem) {
  const int warps_per_head = kWarps / a.heads_per_cta;
  const size_t merge = warps_per_head > 1 ? static_cast<size_t>(kWarps) * a.group *
                                                Geometry<D, STAGES>::kOStride * 4
                                          : 0;
  const size_t bytes = static_cast<size_t>(Geometry<D, STAGES>::kFixedBytes) + merge;
  // the attribute is an upper bound shared by every call of this kernel: set it
  // to the largest request (a full merge area for 16 query heads)
  const size_t most = static_cast<size_t>(Geometry<D, STAGES>::kFixedBytes) +
                      static_cast<size_t>(kWarps) * kMaxGroup * Geometry<D, STAGES>::kOStride * 4;
  auto kern = paged_decode_kernel<Ty, D, STAGES, NT, APPEND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(most));
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, bytes);
  if (e != cudaSuccess) return e;
  *ctas_per_sm = n;
  *smem = bytes;
  return cudaSuccess;
}

template <typename Ty, int D, int STAGES, int NT, bool APPEND>
cudaError_t launch_typed(const DecodeArgs& a, long long grid, size_t smem, cudaStream_t stream) {
  paged_decode_kernel<Ty, D, STAGES, NT, APPEND>
      <<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

// Launch plans (ring depth, CTAs per SM, shared memory) cached per device
// and kernel variant, so the occupancy query runs once, not on every call.
constexpr int kPlanDevices = 64;
constexpr int kPlanSlots = 2 * 2 * 2 * 2 * (kMaxGroup + 1) * 3;
std::atomic<unsigned long long> g_plans[kPlanDevices][kPlanSlots];

template <typename Ty, int D, int NT, bool APPEND>
cudaError_t launch_d(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int hc_slot = a.heads_per_cta == 4 ? 2 : (a.heads_per_cta == 2 ? 1 : 0);
  const int slot = ((((APPEND ? 1 : 0) * 2 + (Ty::kIsBf16 ? 1 : 0)) * 2 + (D == 128 ? 1 : 0)) * 2 +
                    (NT - 1)) * (kMaxGroup + 1) * 3 + a.group * 3 + hc_slot;
  unsigned long long plan = (dev >= 0 && dev < kPlanDevices) ? g_plans[dev][slot].load() : 0ull;
  if (plan == 0) {
    // the ring depth that fits the most CTAs on an SM (three stages on a tie)
    int n3 = 0, n2 = 0;
    size_t m3 = 0, m2 = 0;
    e = plan_typed<Ty, D, 3, NT, APPEND>(a, &n3, &m3);
    if (e != cudaSuccess) return e;
    e = plan_typed<Ty, D, 2, NT, APPEND>(a, &n2, &m2);
    if (e != cudaSuccess) return e;
    const bool three = n3 >= n2;
    const unsigned long long per = static_cast<unsigned long long>(three ? n3 : n2);
    const unsigned long long mem = three ? m3 : m2;
    if (per < 1) return cudaErrorInvalidConfiguration;
    plan = (three ? 1ull : 2ull) | (per << 2) | (mem << 16);
    if (dev >= 0 && dev < kPlanDevices) g_plans[dev][slot].store(plan);
  }
  const bool three = (plan & 3ull) == 1ull;
  const int per_sm = static_cast<int>((plan >> 2) & 0x3fffull);
  const size_t smem = static_cast<size_t>(plan >> 16);
  long long grid = static_cast<long long>(per_sm) * num_sms;
  const long long units = static_cast<long long>(a.num_seqs) *
                          (a.num_kv_heads / a.heads_per_cta) * a.max_partitions;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  return three ? launch_typed<Ty, D, 3, NT, APPEND>(a, grid, smem, stream)
               : launch_typed<Ty, D, 2, NT, APPEND>(a, grid, smem, stream);
}

template <typename Ty, int D>
cudaError_t launch_g(const DecodeArgs& a, int num_sms, cudaStream_t stream) {
  if (a.new_key != nullptr)
    return a.group <= 8 ? launch_d<Ty, D, 1, true>(a, num_sms, stream)
                        : launch_d<Ty, D, 2, true>(a, num_sms, stream);
  return a.group <= 8 ? launch_d<Ty, D, 1, false>(a, num_sms, stream)
                      : launch_d<Ty, D, 2, false>(a, num_sms, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int head_dim, bool bf16, int num_sms,
                          cudaStream_t stream) {
  if (bf16) {
    return head_dim == 64 ? launch_g<BF16, 64>(a, num_sms, stream)
                          : launch_g<BF16, 128>(a, num_sms, stream);
  }
  return head_dim == 64 ? launch_g<F16, 64>(a, num_sms, stream)
                        : launch_g<F16, 128>(a, num_sms, stream);
}

}  // namespace pa
