// ibp_decode_pipe.cuh - the per-row fetch and decode steps shared by the
// specialised gather-decompress kernel (k_decompress_fast) and the fused
// gather-decompress + pooling kernel (k_bag).
//
// « Algorithme central », step 3 (Décompression): a warp reads a row's
// compressed segment into shared memory, derives each lane's starting bit
// offset with warp primitives, and rebuilds its words by putting the Bitval
// bits back at the Mask positions; « Intégration au système »: only the
// compressed part of a fixed-size slot is read, and a bitmask in GPU memory
// says which rows are compressed.
//
// A warp works on groups of G rows.  Per group, three steps, each
// warp-collective (every lane of the warp calls them, with lane q < G
// holding row q's id):
//   issue_prefix  the first `pre` words of every row (which hold the S
//                 participation headers) -> shared stage, by cp.async;
//   row_info      from the landed headers: the row's kind (raw, compressed,
//                 bad id, corrupt), its stream length Lw, and where each
//                 segment's fields start in its row's stream;
//   issue_rest    the words [pre, Lw) of each row (W for raw rows);
// and then, per row, decode_row / decode_segments (one word per lane and
// segment) or, with PAIR, decode_row_pairs / decode_pairs_at (two
// consecutive words per lane and 64-word block), with a caller-supplied sink
// that stores the rebuilt words (gather) or adds them up (pooling).
//
// Shapes are compile-time: W = 32 * SC words per row, at most R runs of kept
// bits per word, uniform plan (TAB = false: one Mask/Bitval for every word
// position, constants in registers) or per-word tables (TAB = true, staged
// once per CTA in shared memory, with NPL e-planes for the field offsets),
// slot layout or packed layout (PK).
#pragma once

#include <cuda_runtime.h>

#include "ibp_internal.cuh"

namespace ibp {

constexpr uint32_t kAll = 0xFFFFFFFFu;

// Words of a per-word table entry in shared memory: {run masks, packed run
// shifts, Bitval & Mask}: 4 words for up to two runs, 8 for up to four.
template <int R>
struct TabEntry {
  static constexpr uint32_t EW = R <= 2 ? 4u : 8u;
};

template <int SC, int R, int NPL, bool TAB>
struct TabShape {
  static constexpr uint32_t W = 32u * SC;
  static constexpr uint32_t ENT = TAB ? W * TabEntry<R>::EW : 0u;
  static constexpr uint32_t EPL = TAB && NPL > 0 ? ((SC * NPL + 31u) / 32u) * 32u : 0u;
  static constexpr uint32_t WORDS = ENT + EPL;  // shared words before the warp stages
};

// NP > 1 (rows of 32 or 64 segments whose slots are in device memory): each
// row is NP tasks of SC / NP segments, and a group is one task.  A task's
// stage holds the row's S header words and then only the part of the stream
// that its segments' fields occupy (at most W / NP words plus alignment), so
// stages stay smaller than a row's and more warps fit on an SM; each task
// re-reads the row's headers.
// SHORT (rows of 8 or 16 segments whose stored streams are mostly at most
// W / 4 words, slots in device memory): a stage row holds RW = W / 4 words,
// so stages are a quarter of the size; a row whose stream is longer is
// decoded from its slot in device memory, and a raw row is copied from it.
template <int SC, uint32_t GW, int NP = 1, bool SHORT = false>
struct FastShape {
  static constexpr uint32_t W = 32u * SC;
  static constexpr uint32_t RW = SHORT ? W / 4u : W;  // words per stage row
  static constexpr uint32_t G = NP > 1 ? 1u : (GW / W >= 1 ? GW / W : 1u);  // rows (tasks) per group
  static constexpr uint32_t STAGE = NP > 1 ? SC + W / NP + 32u : G * RW + 32u;  // words per stage
  static constexpr uint32_t CH = W / 4;                    // 16-byte chunks per row
  static constexpr uint32_t CB = (CH + 31) / 32;           // chunk blocks of 32 per row
};

// Row ids are carried as 32-bit values: kNoRow marks "no row" (past the end
// of the work), kBadId an id outside [0, n_rows).
constexpr int32_t kNoRow = -1, kBadId = -2;

// Word offset of a row in the slots (PK: in the packed buffer) and the number
// of words it occupies there.
struct RowPos {
  uint64_t off;
  uint32_t ext;
};

// PAIR (rows of two or more segments): the decode of a compressed row gives
// each lane two consecutive words of every 64-word block (decode_pairs_at),
// written with one 8-byte store per lane; the per-word tables are then staged
// in the order the lanes read them (see init).
template <int R, int SC, int NPL, bool TAB, bool PK, uint32_t GW, int NP = 1, bool PAIR = false,
          bool SHORT = false>
struct RowPipe {
  using F = FastShape<SC, GW, NP, SHORT>;
  using T = TabShape<SC, R, NPL, TAB>;
  static constexpr uint32_t W = F::W, G = F::G, CB = F::CB, RW = F::RW;
  static constexpr uint32_t EW = TabEntry<R>::EW;
  static constexpr uint32_t PCB = NP > 1 ? (SC / 4 + 31) / 32 : CB;  // chunk blocks a prefix can span
  static constexpr uint32_t SEGP = SC / NP;  // segments of a task
  static constexpr uint32_t WP = W / NP;     // output words of a task
  static_assert(NP == 1 || (!PK && SC >= 32 && (SEGP == 16 || SEGP == 32)), "tasks of 16 or 32 segments, slot layout");
  static_assert(!PAIR || SC >= 2, "pairs need 64-word blocks");
  static_assert(!SHORT || (PAIR && !PK && NP == 1 && SC >= 8), "short stage rows: pair decode, slots, whole rows");

  uint32_t lane, lt, lanebit;
  uint32_t half, j0, plt, pbit0, pbit1;  // PAIR: segment 2k + half, positions j0, j0 + 1
  uint32_t p, pscale, bm;  // uniform: popcount(Mask), -, Bitval & Mask; tables: p_min, p_scale
  uint32_t rm[R], rs[R];   // uniform: runs of kept bits and their shifts
  const uint32_t* tab;     // shared: [W][EW] per-word entries (TAB)
  const uint32_t* epl;     // shared: [SC][NPL] e-planes (TAB, NPL > 0)
  const uint32_t* slots;
  const uint32_t* bitmask;
  const uint64_t* offsets;  // PK
  uint32_t pre, pre_ch;     // prefix in words (multiple of 4, <= W) and in 16-byte chunks
  uint32_t n_rows32;
  bool reuse;               // row copies also allocate in L1 (IBP_HINT_ROW_REUSE)

  // Per-thread set-up.  TAB: the block's threads stage the plan's tables into
  // smem and meet at a barrier, so every thread of the block must call this
  // before any warp leaves.
  __device__ __forceinline__ void init(const PlanView& pv, const uint32_t* slots_, const uint32_t* bitmask_,
                                       const uint64_t* offsets_, uint64_t n_rows, uint32_t pre_, uint32_t* smem) {
    lane = threadIdx.x & 31u;
    lt = lanemask_lt();
    lanebit = 1u << lane;
    half = lane >> 4;
    j0 = 2u * (lane & 15u);
    plt = (1u << j0) - 1u;
    pbit0 = 1u << j0;
    pbit1 = pbit0 << 1;
    p = TAB ? pv.p_min : pv.u_p;
    pscale = pv.p_scale;
    bm = pv.u_bm;
#pragma unroll
    for (int k = 0; k < R; ++k) {
      rm[k] = pv.u_rmask[k];
      rs[k] = pv.u_rsh[k];
    }
    tab = smem;
    epl = smem + T::ENT;
    if constexpr (TAB) {
      for (uint32_t w = threadIdx.x; w < W; w += blockDim.x) {
        // PAIR: word w = 64 k + 2 L + i (lane L, i = 0, 1) goes to entry
        // 64 k + 32 i + L, so that the 32 lanes' reads of their i-th words are
        // 32 consecutive entries
        const uint32_t slot = PAIR ? ((w & ~63u) | ((w & 1u) << 5) | ((w & 63u) >> 1)) : w;
        uint32_t* e = smem + slot * EW;
#pragma unroll
        for (int k = 0; k < (EW == 4 ? 2 : 4); ++k) e[k] = k < R ? __ldg(pv.rmask + k * W + w) : 0u;
        e[EW == 4 ? 2 : 4] = __ldg(pv.rshift + w);
        e[EW == 4 ? 3 : 5] = __ldg(pv.bm + w);
      }
      if constexpr (NPL > 0) {
        for (uint32_t i = threadIdx.x; i < SC * NPL; i += blockDim.x)
          smem[T::ENT + i] = __ldg(pv.eplanes + (i / NPL) * kPlanes + (i % NPL));
      }
      __syncthreads();
    }
    slots = slots_;
    bitmask = bitmask_;
    offsets = offsets_;
    pre = pre_;
    pre_ch = pre_ >> 2;
    n_rows32 = static_cast<uint32_t>(n_rows);  // < 2^31 (checked by the launchers)
    reuse = (pv.hints & IBP_HINT_ROW_REUSE) != 0;
  }

  // An id as the pipeline carries it.
  __device__ __forceinline__ int32_t check_id(int64_t id) const {
    return (id >= 0 && static_cast<uint64_t>(id) < n_rows32) ? static_cast<int32_t>(id) : kBadId;
  }

  __device__ __forceinline__ RowPos row_pos(int32_t id) const {
    if constexpr (PK) {
      if (id < 0) return {0, 0};
      const uint64_t lo = offsets[id], hi = offsets[id + 1];
      const uint64_t ext = hi > lo ? hi - lo : 0;
      return {lo, static_cast<uint32_t>(ext < W ? ext : W)};
    } else {
      return {static_cast<uint64_t>(id >= 0 ? id : 0) * W, W};
    }
  }

  // Prefix of a group: the row's bitmask word into bmw, and lane i copies
  // chunk i (+32 ...) of every row's first `pre` words.  Warp-collective.
  __device__ __forceinline__ void issue_prefix(uint32_t* sb, int32_t id, RowPos rp, uint32_t& bmw) const {
    if (id >= 0) bmw = ld_u32(bitmask + (static_cast<uint32_t>(id) >> 5));
#pragma unroll
    for (uint32_t q = 0; q < G; ++q) {
      const int32_t idq = __shfl_sync(kAll, id, q);
      uint64_t offq;
      if constexpr (PK)
        offq = __shfl_sync(kAll, static_cast<unsigned long long>(rp.off), q);
      else
        offq = static_cast<uint64_t>(idq) * W;
      // PK: a row shorter than the prefix is corrupt (row_info says so) and
      // is not read
      bool ok = idq >= 0;
      if constexpr (PK) ok = ok && __shfl_sync(kAll, rp.ext, q) >= pre;
      if (ok) {
        const uint32_t* src = slots + offq;
        uint32_t* dst = sb + q * RW;
        // blocks of 32 chunks up to the prefix's last (a task's prefix, its
        // row's headers, is at most one block)
#pragma unroll
        for (uint32_t b = 0; b < PCB; ++b) {
          if (32u * b >= pre_ch) break;  // warp-uniform
          const uint32_t c = lane + 32u * b;
          if (c < pre_ch) cp_row16(reuse, dst + 4u * c, src + 4u * c);
        }
      }
    }
  }

  // Bits that the matching words of segment s save against 32 bits each.
  __device__ __forceinline__ uint32_t seg_saved(uint32_t H, uint32_t s) const {
    uint32_t c = p * __popc(H);
    if constexpr (TAB && NPL > 0) {
#pragma unroll
      for (int k = 0; k < NPL; ++k) c += pscale * (__popc(H & epl[s * NPL + k]) << k);
    }
    return c;
  }

  // Stream bits that segment s of a row occupies (headers aside): 32 per
  // word, less what its matching words save.  At most 1024 for any header.
  __device__ __forceinline__ uint32_t seg_bits(uint32_t H, uint32_t s) const { return 1024u - seg_saved(H, s); }

  // The group's segments, flat: segment f = q * SC + s is segment s of row q,
  // for NSEG = G * SC segments (at most 32, or 64 for one row of 64 segments).
  static constexpr uint32_t NSEG = G * SC;
  static_assert(NSEG <= 32 || (G == 1 && SC == 64), "segments of a group: one or two per lane");

  // Where each segment's fields start in its row's stream: segment f's base
  // is held by lane f (in `lo`; segments 32 .. 63 in `hi`).
  struct Bases {
    uint32_t lo, hi;
  };

  // From the landed headers of a group: every segment's base (the row's S
  // header words, then the fields of its earlier segments: a segmented
  // exclusive warp scan of the segments' stream bits, one segment per lane),
  // and, to lane q < G, the length in bits of row q's stream.  Replaces a
  // serial walk over the headers with log2(SC) shuffle steps per group, and
  // lets the decode of a segment take its base with one shuffle, without a
  // dependency on the segments before it.  Warp-collective.
  __device__ __forceinline__ void seg_scan(const uint32_t* sb, Bases& b, uint32_t& row_bits) const {
    constexpr uint32_t SW = SC < 32 ? SC : 32;  // lanes per row in the scan
    auto bits_of = [&](uint32_t f) -> uint32_t {
      if (f >= NSEG) return 0u;
      const uint32_t q = f / SC, s = f % SC;
      return seg_bits(sb[q * RW + s], s);
    };
    auto scan = [&](uint32_t v) -> uint32_t {  // inclusive, within groups of SW lanes
#pragma unroll
      for (uint32_t d = 1; d < SW; d <<= 1) {
        const uint32_t t = __shfl_up_sync(kAll, v, d);
        if ((lane & (SW - 1)) >= d) v += t;
      }
      return v;
    };
    const uint32_t a = bits_of(lane);
    const uint32_t ia = scan(a);
    b.lo = 32u * SC + ia - a;
    if constexpr (NSEG > 32) {
      const uint32_t tot_a = __shfl_sync(kAll, ia, 31);
      const uint32_t c = bits_of(lane + 32);
      const uint32_t ic = scan(c);
      b.hi = 32u * SC + tot_a + ic - c;
      row_bits = 32u * SC + tot_a + __shfl_sync(kAll, ic, 31);
    } else {
      b.hi = 0;
      const uint32_t src = (lane < G ? lane : 0u) * SC + SC - 1u;  // last segment of row `lane`
      row_bits = 32u * SC + __shfl_sync(kAll, ia, src);
    }
  }

  // The base of segment s of row q (warp-uniform q, s).
  __device__ __forceinline__ uint32_t seg_base(const Bases& b, uint32_t q, uint32_t s) const {
    const uint32_t f = q * SC + s;
    if constexpr (NSEG > 32)
      return __shfl_sync(kAll, f < 32 ? b.lo : b.hi, f & 31u);
    else
      return __shfl_sync(kAll, b.lo, f);
  }

  // Kind and stream length of lane q's row of a group whose prefix has landed
  // in sb, and the group's segment bases.  Warp-collective (seg_scan).
  //
  // NP > 1: the group is part `part` of a row, and nt encodes the 16-byte
  // chunks [c0, c1) of the slot that the task needs after the headers, as
  // (c0 << 16) | c1: for a compressed row, the words that its segments' fields
  // occupy (and the word after the last field, which the decode's two-word read
  // may touch, within the row); for a raw row, its WP words.
  __device__ __forceinline__ void row_info(const uint32_t* sb, int32_t id, RowPos rp, uint32_t bmw, uint32_t& kind,
                                           uint32_t& nt, Bases& bases, uint32_t part = 0) const {
    uint32_t row_bits;
    seg_scan(sb, bases, row_bits);
    uint32_t lo_bit = 0, hi_bit = 0;
    if constexpr (NP > 1) {  // warp-collective: every lane takes the shuffles
      lo_bit = seg_base(bases, 0, part * SEGP);
      const uint32_t nx = seg_base(bases, 0, (part + 1 < NP ? part + 1 : part) * SEGP);
      hi_bit = part + 1 < NP ? nx : row_bits;
    }
    kind = kNone;
    nt = 0;
    if (id == kNoRow) return;
    if (id == kBadId) {
      kind = kBadRange;
      return;
    }
    if (!((bmw >> (static_cast<uint32_t>(id) & 31u)) & 1u)) {
      kind = (PK && rp.ext < W) ? kCorrupt : kRaw;
      if constexpr (NP > 1)
        nt = ((part * (WP / 4u)) << 16) | ((part + 1u) * (WP / 4u));
      else
        nt = (kind == kRaw && !SHORT) ? W : 0u;  // SHORT: a raw row is copied from its slot
      return;
    }
    if (PK && rp.ext < pre) {
      kind = kCorrupt;
      return;
    }
    const uint32_t Lw = (row_bits + 31u) >> 5;
    if (Lw >= W || (PK && ((Lw + 3u) & ~3u) > rp.ext)) {
      kind = kCorrupt;
      return;
    }
    kind = kComp;
    if constexpr (NP > 1) {
      // lo_bit < hi_bit <= row_bits < 32 W; the last field starts below hi_bit
      const uint32_t ws = lo_bit >> 5;
      const uint32_t we = min(W, ((hi_bit - 1u) >> 5) + 2u);
      nt = ((ws >> 2) << 16) | ((we + 3u) >> 2);
    } else {
      nt = Lw;
      if (SHORT && Lw > RW) kind = kCompSlot;  // decoded from its slot
    }
  }

  // Rest of a group: [pre, Lw) of compressed rows, [pre, W) of raw rows.
  // Warp-collective.
  __device__ __forceinline__ void issue_rest(uint32_t* sb, int32_t id, RowPos rp, uint32_t kind, uint32_t nt) const {
    if constexpr (NP > 1) {
      // one task per group, held by lane 0: chunks [c0, c1) of its row to
      // stage words SC + 4 (c - c0)
      const uint32_t k0 = __shfl_sync(kAll, kind, 0);
      if (k0 != kRaw && k0 != kComp) return;
      const uint32_t n0 = __shfl_sync(kAll, nt, 0);
      const uint32_t c0 = n0 >> 16, c1 = n0 & 0xFFFFu;
      const uint32_t* src = slots + static_cast<uint64_t>(__shfl_sync(kAll, id, 0)) * W;
      for (uint32_t c = c0 + lane; c < c1; c += 32) cp_row16(reuse, sb + SC + 4u * (c - c0), src + 4u * c);
      return;
    }
    const bool need = (kind == kRaw || kind == kComp) && nt > pre;
    for (uint32_t mk = __ballot_sync(kAll, need); mk; mk &= mk - 1) {
      const uint32_t q = __ffs(mk) - 1;
      const uint32_t ntq = __shfl_sync(kAll, nt, q);
      uint64_t offq;
      if constexpr (PK)
        offq = __shfl_sync(kAll, static_cast<unsigned long long>(rp.off), q);
      else
        offq = static_cast<uint64_t>(__shfl_sync(kAll, id, q)) * W;
      const uint32_t* src = slots + offq;
      uint32_t* dst = sb + q * RW;
      for (uint32_t c = pre_ch + lane; c < ((ntq + 3u) >> 2); c += 32) cp_row16(reuse, dst + 4u * c, src + 4u * c);
    }
  }

  // Word lane + 32 s of a compressed row whose stream is in pb, given the bit
  // where segment s's fields start (base, the same in every lane).
  __device__ __forceinline__ uint32_t decode_word(const uint32_t* pb, uint32_t H, uint32_t s, uint32_t base) const {
    uint32_t P = base + 32u * lane - p * __popc(H & lt);
    if constexpr (TAB && NPL > 0) {
      uint32_t e_lt = 0;
#pragma unroll
      for (int k = 0; k < NPL; ++k) e_lt += __popc(H & epl[s * NPL + k] & lt) << k;
      P -= pscale * e_lt;
    }
    const uint32_t* q = pb + (P >> 5);
    const uint32_t v = __funnelshift_r(q[0], q[1], P);
    uint32_t y;
    if constexpr (TAB) {
      const uint32_t* e = tab + (32u * s + lane) * EW;
      const uint4 e0 = *reinterpret_cast<const uint4*>(e);
      if constexpr (EW == 4) {
        const uint32_t m2[2] = {e0.x, e0.y};
        y = deposit_runs_packed<(R < 2 ? R : 2)>(v, m2, e0.z) | e0.w;
      } else {
        const uint4 e1 = *reinterpret_cast<const uint4*>(e + 4);
        const uint32_t m4[4] = {e0.x, e0.y, e0.z, e0.w};
        y = deposit_runs_packed<R>(v, m4, e1.x) | e1.y;
      }
    } else {
      y = deposit_runs<R>(v, rm, rs) | bm;
    }
    return (H & lanebit) ? y : v;
  }

  // Decodes segments [s_lo, s_lo + NS) of row q of the group (compressed,
  // stream in pb): sink(j, y) receives word lane + 32 (s_lo + j), j = 0 ..
  // NS-1, in order.  Each segment's base comes from the group's Bases.
  // The headers are at hb[0 .. SC), and stream bit k at bit (k - bias) of pb
  // (bias 0 and pb = hb unless a task's stage holds only part of the stream:
  // then bias = 32 (first stream word staged - its stage word)).
  template <uint32_t NS, class Sink>
  __device__ __forceinline__ void decode_segments(const uint32_t* hb, const uint32_t* pb, uint32_t q, uint32_t s_lo,
                                                  const Bases& bases, Sink&& sink, uint32_t bias = 0) const {
    decode_segments_at<NS>(hb, pb, s_lo, [&](uint32_t j) { return seg_base(bases, q, s_lo + j) - bias; }, sink);
  }

  // As decode_segments, with base_of(j) giving the base of segment s_lo + j
  // (warp-uniform), in stream bits of pb.
  template <uint32_t NS, class BaseOf, class Sink>
  __device__ __forceinline__ void decode_segments_at(const uint32_t* hb, const uint32_t* pb, uint32_t s_lo,
                                                     BaseOf&& base_of, Sink&& sink) const {
    if constexpr (NS >= 4 && NS % 4 == 0) {
      if (s_lo % 4 == 0) {
#pragma unroll
        for (uint32_t j = 0; j < NS; j += 4) {
          const uint4 h = *reinterpret_cast<const uint4*>(hb + s_lo + j);
          const uint32_t s = s_lo + j;
          sink(j, decode_word(pb, h.x, s, base_of(j)));
          sink(j + 1, decode_word(pb, h.y, s + 1, base_of(j + 1)));
          sink(j + 2, decode_word(pb, h.z, s + 2, base_of(j + 2)));
          sink(j + 3, decode_word(pb, h.w, s + 3, base_of(j + 3)));
        }
        return;
      }
    }
#pragma unroll
    for (uint32_t j = 0; j < NS; ++j) {
      const uint32_t s = s_lo + j;
      sink(j, decode_word(pb, hb[s], s, base_of(j)));
    }
  }

  // PAIR: segments [s_lo, s_lo + NS) of a compressed row as NS / 2 blocks of
  // 64 words.  In block k lane L rebuilds positions j0 = 2 (L mod 16) and
  // j0 + 1 of segment s_lo + 2k + L / 16, i.e. words 2L and 2L + 1 of the
  // block: its first field starts at the segment's base plus the bits of the
  // segment's words below j0 (a popcount of the header, as in decode_word),
  // and its second field right after the first (32 bits on, less what the
  // first word saves if it matches: p, plus p_scale times its e-plane
  // value, all from registers, so that both fields' reads issue at once).
  // sink(k, y0, y1) receives the two words.  base_of(j) gives the base of
  // segment s_lo + j (j differs between the two half-warps), in stream bits
  // of pb; s_lo is even.
  template <uint32_t NS, class BaseOf, class Sink>
  __device__ __forceinline__ void decode_pairs_at(const uint32_t* hb, const uint32_t* pb, uint32_t s_lo,
                                                  BaseOf&& base_of, Sink&& sink) const {
    static_assert(NS % 2 == 0, "whole blocks");
#pragma unroll
    for (uint32_t k = 0; k < NS / 2; ++k) {
      const uint32_t s = s_lo + 2u * k + half;
      const uint32_t H = hb[s];
      uint32_t P0 = base_of(2u * k + half) + 32u * j0 - p * __popc(H & plt);
      uint32_t sv0 = p;  // bits the first word saves if it matches
      if constexpr (TAB && NPL > 0) {
        uint32_t e_lt = 0, e0 = 0;
#pragma unroll
        for (int kk = 0; kk < NPL; ++kk) {
          const uint32_t E = epl[s * NPL + kk];
          e_lt += __popc(H & E & plt) << kk;
          e0 |= ((E >> j0) & 1u) << kk;
        }
        P0 -= pscale * e_lt;
        sv0 += pscale * e0;
      }
      const uint32_t P1 = P0 + 32u - ((H & pbit0) ? sv0 : 0u);
      uint32_t y[2];
#pragma unroll
      for (uint32_t i = 0; i < 2; ++i) {
        const uint32_t P = i == 0 ? P0 : P1;
        const uint32_t* q = pb + (P >> 5);
        const uint32_t v = __funnelshift_r(q[0], q[1], P);
        uint32_t d;
        if constexpr (TAB) {
          const uint32_t* e = tab + (64u * (s_lo / 2u + k) + 32u * i + lane) * EW;
          const uint4 e0 = *reinterpret_cast<const uint4*>(e);
          if constexpr (EW == 4) {
            const uint32_t m2[2] = {e0.x, e0.y};
            d = deposit_runs_packed<(R < 2 ? R : 2)>(v, m2, e0.z) | e0.w;
          } else {
            const uint4 e1 = *reinterpret_cast<const uint4*>(e + 4);
            const uint32_t m4[4] = {e0.x, e0.y, e0.z, e0.w};
            d = deposit_runs_packed<R>(v, m4, e1.x) | e1.y;
          }
        } else {
          d = deposit_runs<R>(v, rm, rs) | bm;
        }
        y[i] = (H & (i == 0 ? pbit0 : pbit1)) ? d : v;
      }
      sink(k, y[0], y[1]);
    }
  }

  // PAIR: the whole of row q; sink(k, y0, y1) gets words 64 k + 2 lane and
  // 64 k + 2 lane + 1.
  template <class Sink>
  __device__ __forceinline__ void decode_row_pairs(const uint32_t* pb, uint32_t q, const Bases& bases,
                                                   Sink&& sink) const {
    decode_pairs_at<SC>(pb, pb, 0u, [&](uint32_t j) { return seg_base_pair(bases, q, j); }, sink);
  }

  // As decode_row_pairs, with the row's headers at hb and its stream at pb
  // (SHORT: a row too long for its stage row, read from its slot).
  template <class Sink>
  __device__ __forceinline__ void decode_row_pairs_from(const uint32_t* hb, const uint32_t* pb, uint32_t q,
                                                        const Bases& bases, Sink&& sink) const {
    decode_pairs_at<SC>(hb, pb, 0u, [&](uint32_t j) { return seg_base_pair(bases, q, j); }, sink);
  }

  // PAIR: the base of segment j of row q where j = 2k + half differs between
  // the half-warps; both segments of a block sit in the same 32 lanes of the
  // scan (f is even for the block's first), so the register is warp-uniform.
  __device__ __forceinline__ uint32_t seg_base_pair(const Bases& b, uint32_t q, uint32_t j) const {
    const uint32_t f = q * SC + j;
    if constexpr (NSEG > 32)
      return __shfl_sync(kAll, (f & ~1u) < 32 ? b.lo : b.hi, f & 31u);
    else
      return __shfl_sync(kAll, b.lo, f);
  }

  // NP > 1: the bases of task `part`'s SEGP segments, less `bias`, gathered
  // into one register (lane j holds segment part * SEGP + j's), so that each
  // segment's base is one shuffle with a compile-time lane.
  __device__ __forceinline__ uint32_t task_bases(const Bases& b, uint32_t part, uint32_t bias) const {
    const uint32_t f = part * SEGP + (lane % SEGP);
    uint32_t v;
    if constexpr (NSEG > 32)
      v = __shfl_sync(kAll, part * SEGP < 32 ? b.lo : b.hi, f & 31u);
    else
      v = __shfl_sync(kAll, b.lo, f);
    return v - bias;
  }

  // The whole of row q: sink(s, y) gets word lane + 32 s, s = 0 .. SC-1.
  template <class Sink>
  __device__ __forceinline__ void decode_row(const uint32_t* pb, uint32_t q, const Bases& bases, Sink&& sink) const {
    decode_segments<SC>(pb, pb, q, 0u, bases, sink);
  }
};

}  // namespace ibp
