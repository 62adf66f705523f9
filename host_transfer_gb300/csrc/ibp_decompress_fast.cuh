// ibp_decompress_fast.cuh - gather/contiguous decompress specialised for the
// common plan shapes: rows are a whole number of 32-word segments
// (W = 32 * SC, SC a power of two up to 64), the kept bits of every word
// form at most four runs, buffers are 16-byte aligned and row ids fit in 31
// bits.  Two modes: TAB = false, every word position shares one Mask/Bitval
// (uniform plan), whose constants sit in registers; TAB = true, per-word
// Masks, whose deposit runs and Bitval are staged once per CTA in shared
// memory and whose field offsets use the e-planes of the plan (NPL of them).
// Instantiated by ibp_decompress_fast_u.cu (uniform) and
// ibp_decompress_fast_t.cu (tables).  The method is the same as k_decompress (« Algorithme
// central », step 3: a warp stages a row's compressed segment in shared
// memory, computes each lane's bit offset with warp primitives and puts the
// Bitval bits back); what changes is that W, the rows per group G and the
// segment count are compile-time constants, so every loop unrolls, headers
// are read with 16-byte shared loads, the deposit constants sit in
// registers, and the prefetch maps lane i to 16-byte chunk i of each row.
//
// Pipeline per warp (as in k_decompress): ids of group j+3 -> registers;
// prefix [0, pre) of the G rows of group j+2 -> shared stage (cp.async);
// kinds of group j+1 from its landed headers, then the rest [pre, Lw) of
// its rows -> shared stage (cp.async); decode of group j.  Stages are G rows
// of W words (W a multiple of 32: a row's 128-byte global lines land on
// 128-byte shared-memory lines) plus 32 words for the decoder's read of one
// word past a row.
#pragma once

#include <cuda_runtime.h>

#include "ibp_internal.cuh"

namespace ibp {

constexpr int kFastWarps = 8;
constexpr int kFastStages = 3;  // shared-memory stages per warp (D >= 3)
constexpr uint32_t kAll = 0xFFFFFFFFu;
// Words per group (GW; rows per group G = GW / W, at least 1).  512 by
// default; 256 for copies that also allocate in L1 (IBP_HINT_ROW_REUSE on
// host-mapped slots): the smaller stages leave more of the SM's on-chip
// memory to L1, which is where repeated rows are found.
constexpr uint32_t kGroupWords = 512;
constexpr uint32_t kGroupWordsReuse = 256;
// Slots in device memory (measured): uniform plans take 768-word groups (dense
// HBM 2395 -> 2580 GB/s: longer straight-line decode blocks), per-word-table
// plans 1024 (sparse HBM 2167 -> 2299 GB/s: two 512-word rows per group).
constexpr uint32_t kGroupWordsDev = 768;
constexpr uint32_t kGroupWordsDevTable = 1024;

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

template <int SC, uint32_t GW>
struct FastShape {
  static constexpr uint32_t W = 32u * SC;
  static constexpr uint32_t G = GW / W >= 1 ? GW / W : 1u;  // rows per group
  static constexpr uint32_t STAGE = G * W + 32u;           // words per stage
  static constexpr uint32_t CH = W / 4;                    // 16-byte chunks per row
  static constexpr uint32_t CB = (CH + 31) / 32;           // chunk blocks of 32 per row
};

// PK = false: row r of the table is slots[r * W ..]; PK = true: the packed
// layout, row r is slots[offsets[r] .. offsets[r + 1]) (its stored words
// rounded up to 16 bytes), and a row whose stream would reach past that
// extent is corrupt.
// MP = true (plan sets, contiguous decode, table path): CTA row blockIdx.y
// decodes rows [y * rows_per_plan, (y + 1) * rows_per_plan) of the table with
// plan y of a.plans (a device array of plan views).
// CTAs per SM the register allocation is sized for, where that causes no
// spills (measured on one GB300): uniform plans up to W = 1024 with 512-word
// groups fit four (+1 % on dense and DLRM rows); with the larger groups of
// device slots shared memory holds two, and a two-CTA budget leaves the
// straight-line decode its registers; per-word-table plans up to W = 512 with
// at most one e-plane fit three with 512-word groups (instead of the two that
// 107 registers allowed: +9 % for device slots, -2 % over the host link, so
// host slots keep the compiler's choice) and two with 1024-word groups; other
// shapes keep the compiler's choice.
template <int SC, int NPL, bool TAB, bool MP, bool DEV, uint32_t GW>
constexpr int fast_min_blocks() {
  if (!TAB) return DEV ? 2 : (SC <= 32 ? 4 : 1);
  if (DEV && !MP && SC <= 16 && NPL <= 1) return GW >= 1024 ? 2 : 3;
  return 1;
}

// DEV only selects the register budget (fast_min_blocks).
template <int R, int SC, int NPL, bool TAB, bool PK, uint32_t GW, bool MP = false, bool DEV = false>
__global__ void __launch_bounds__(kFastWarps * 32, (fast_min_blocks<SC, NPL, TAB, MP, DEV, GW>())) k_decompress_fast(const DecodeArgs a) {
  static_assert(!MP || (TAB && !PK), "plan sets decode through the table path, slot layout");
  using F = FastShape<SC, GW>;
  using T = TabShape<SC, R, NPL, TAB>;
  constexpr uint32_t W = F::W, G = F::G, STAGE = F::STAGE, CB = F::CB;
  constexpr uint32_t EW = TabEntry<R>::EW;
  extern __shared__ __align__(128) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t nw_cta = blockDim.x >> 5;
  uint32_t* const tab = smem;             // [W][EW] per-word entries (TAB)
  uint32_t* const epl = smem + T::ENT;    // [SC][NPL] e-planes (TAB, NPL > 0)
  constexpr int D = kFastStages;
  uint32_t* const stages = smem + T::WORDS + warp * static_cast<uint32_t>(D) * STAGE;
  const uint32_t lt = lanemask_lt();
  const uint32_t lanebit = 1u << lane;

  // this CTA's plan, row range and output
  PlanView pv;
  if constexpr (MP)
    pv = a.plans[blockIdx.y];
  else
    pv = a.pv;
  const uint64_t n_out = MP ? a.rows_per_plan : a.n_out;
  const uint64_t first = MP ? a.first + blockIdx.y * a.rows_per_plan : a.first;
  uint32_t* const out = MP ? a.out + blockIdx.y * a.rows_per_plan * (32ull * SC) : a.out;

  // plan constants: uniform Mask (TAB = false) or the per-word tables
  const uint32_t p = TAB ? pv.p_min : pv.u_p;
  const uint32_t pscale = pv.p_scale;
  const uint32_t bm = pv.u_bm;
  uint32_t rm[R], rs[R];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    rm[k] = pv.u_rmask[k];
    rs[k] = pv.u_rsh[k];
  }
  if constexpr (TAB) {
    // Stage the tables once per CTA; every thread reaches this barrier
    // before any warp leaves.
    for (uint32_t w = threadIdx.x; w < W; w += blockDim.x) {
      uint32_t* e = tab + w * EW;
#pragma unroll
      for (int k = 0; k < (EW == 4 ? 2 : 4); ++k) e[k] = k < R ? __ldg(pv.rmask + k * W + w) : 0u;
      e[EW == 4 ? 2 : 4] = __ldg(pv.rshift + w);
      e[EW == 4 ? 3 : 5] = __ldg(pv.bm + w);
    }
    if constexpr (NPL > 0) {
      for (uint32_t i = threadIdx.x; i < SC * NPL; i += blockDim.x)
        epl[i] = __ldg(pv.eplanes + (i / NPL) * kPlanes + (i % NPL));
    }
    __syncthreads();
  }
  const bool reuse = (pv.hints & IBP_HINT_ROW_REUSE) != 0;
  const uint32_t pre = MP ? pv.pre : a.pre;  // multiple of 4, <= W
  const uint32_t pre_ch = pre >> 2;    // prefix chunks per row
  const uint32_t n_rows32 = static_cast<uint32_t>(a.n_rows);  // < 2^31 (checked by the launcher)

  // Warp gw owns groups gw, gw + nwarps, ...; group g is output rows
  // g*G .. g*G + G - 1 and lane q < G owns row g*G + q.
  const uint64_t n_groups = (n_out + G - 1) / G;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * nw_cta + warp;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * nw_cta;
  // Programmatic dependent launch: the next kernel of the stream may start
  // its CTAs as this grid's CTAs exit (its prologue overlaps this grid's
  // drain), and every CTA waits for the previous grid to complete, with its
  // memory visible, before touching per-call data (ids, bitmask, slots,
  // output, status).  The plan tables read above are written only when the
  // plan is created.  Without the launch attribute both are no-ops.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (gw >= n_groups) return;  // warp-uniform; only warp-level syncs below
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint64_t J = (n_groups - gw + nwarps - 1) / nwarps;
  const uint64_t row_step = nwarps * G;  // first row of group j+1 minus first row of group j

  // Row ids are carried as 32-bit values; -1 marks "no row" (past the end of
  // the output) and kBadId an id outside [0, n_rows).
  constexpr int32_t kNoRow = -1, kBadId = -2;
  auto load_id = [&](uint64_t j, uint64_t rbase) -> int32_t {
    const uint64_t i = rbase + lane;
    if (j >= J || lane >= G || i >= n_out) return kNoRow;
    const int64_t id = a.ids ? a.ids[i] : static_cast<int64_t>(first + i);
    return (id >= 0 && static_cast<uint64_t>(id) < n_rows32) ? static_cast<int32_t>(id) : kBadId;
  };

  // Word offset of a row in the slots (PK: in the packed buffer) and the
  // number of words it occupies there.
  struct RowPos {
    uint64_t off;
    uint32_t ext;
  };
  auto row_pos = [&](int32_t id) -> RowPos {
    if constexpr (PK) {
      if (id < 0) return {0, 0};
      const uint64_t lo = a.offsets[id], hi = a.offsets[id + 1];
      const uint64_t ext = hi > lo ? hi - lo : 0;
      return {lo, static_cast<uint32_t>(ext < W ? ext : W)};
    } else {
      return {static_cast<uint64_t>(id >= 0 ? id : 0) * W, W};
    }
  };

  // Prefix of group j: lane i copies chunk i (+32 ...) of every row.
  auto issue_prefix = [&](uint64_t j, uint32_t* sb, int32_t id, RowPos rp, uint32_t& bmw) {
    if (id >= 0) bmw = ld_u32(a.bitmask + (static_cast<uint32_t>(id) >> 5));
    if (j >= J) return;
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
        const uint32_t* src = a.slots + offq;
        uint32_t* dst = sb + q * W;
#pragma unroll
        for (uint32_t b = 0; b < CB; ++b) {
          const uint32_t c = lane + 32u * b;
          if (c < pre_ch) cp_row16(reuse, dst + 4u * c, src + 4u * c);
        }
      }
    }
  };

  // Bits that the matching words of a row save against 32 bits each (p per
  // match, plus pscale * e for the e-planes of per-word plans), summed over
  // its S headers.  Rows of 8 or more segments: one header per lane, G rows
  // in ceil(G / (32 / SC)) passes, each row's sum by a warp reduction and
  // kept by lane q for row q (warp-collective: every lane calls it).
  // Shorter rows: lane q walks its own row's headers.
  auto saved_bits = [&](const uint32_t* sb) -> uint32_t {
    auto seg_saved = [&](uint32_t H, uint32_t s) -> uint32_t {
      uint32_t c = p * __popc(H);
      if constexpr (TAB && NPL > 0) {
#pragma unroll
        for (int k = 0; k < NPL; ++k) c += pscale * (__popc(H & epl[s * NPL + k]) << k);
      }
      return c;
    };
    uint32_t mine = 0;
    if constexpr (SC >= 8) {
      constexpr uint32_t RPP = SC >= 32 ? 1u : 32u / SC;  // rows per pass
      const uint32_t qo = SC >= 32 ? 0u : lane / SC;       // this lane's row in a pass
#pragma unroll
      for (uint32_t q0 = 0; q0 < G; q0 += RPP) {
        uint32_t c = 0;
        if (q0 + qo < G) {
          const uint32_t* hb = sb + (q0 + qo) * W;
#pragma unroll
          for (uint32_t s = SC >= 32 ? lane : lane % SC; s < SC; s += 32) c += seg_saved(hb[s], s);
        }
#pragma unroll
        for (uint32_t r = 0; r < RPP; ++r) {
          if (q0 + r >= G) break;
          const uint32_t t = __reduce_add_sync(kAll, qo == r ? c : 0u);
          if (lane == q0 + r) mine = t;
        }
      }
    } else {
      if (lane < G) {
        const uint32_t* hb = sb + lane * W;
        if constexpr (SC >= 4) {
#pragma unroll
          for (uint32_t s = 0; s < SC; s += 4) {
            const uint4 h = *reinterpret_cast<const uint4*>(hb + s);
            mine += seg_saved(h.x, s) + seg_saved(h.y, s + 1) + seg_saved(h.z, s + 2) + seg_saved(h.w, s + 3);
          }
        } else {
#pragma unroll
          for (uint32_t s = 0; s < SC; ++s) mine += seg_saved(hb[s], s);
        }
      }
    }
    return mine;
  };

  // Kind and stream length of lane q's row of group j (headers in stage).
  // Warp-collective (saved_bits).
  auto row_info = [&](const uint32_t* sb, int32_t id, RowPos rp, uint32_t bmw, uint32_t& kind,
                      uint32_t& nt) {
    const uint32_t saved = saved_bits(sb);
    kind = kNone;
    nt = 0;
    if (id == kNoRow) return;
    if (id == kBadId) {
      kind = kBadRange;
      return;
    }
    if (!((bmw >> (static_cast<uint32_t>(id) & 31u)) & 1u)) {
      kind = (PK && rp.ext < W) ? kCorrupt : kRaw;
      nt = kind == kRaw ? W : 0u;
      return;
    }
    if (PK && rp.ext < pre) {
      kind = kCorrupt;
      return;
    }
    const uint32_t Lw = (32u * (SC + W) - saved + 31u) >> 5;
    if (Lw >= W || (PK && ((Lw + 3u) & ~3u) > rp.ext)) {
      kind = kCorrupt;
      return;
    }
    kind = kComp;
    nt = Lw;
  };

  // Rest of group j: [pre, Lw) of compressed rows, [pre, W) of raw rows.
  auto issue_rest = [&](uint64_t j, uint32_t* sb, int32_t id, RowPos rp, uint32_t kind, uint32_t nt) {
    if (j >= J) return;
    const bool need = (kind == kRaw || kind == kComp) && nt > pre;
    for (uint32_t mk = __ballot_sync(kAll, need); mk; mk &= mk - 1) {
      const uint32_t q = __ffs(mk) - 1;
      const uint32_t ntq = __shfl_sync(kAll, nt, q);
      uint64_t offq;
      if constexpr (PK)
        offq = __shfl_sync(kAll, static_cast<unsigned long long>(rp.off), q);
      else
        offq = static_cast<uint64_t>(__shfl_sync(kAll, id, q)) * W;
      const uint32_t* src = a.slots + offq;
      uint32_t* dst = sb + q * W;
      for (uint32_t c = pre_ch + lane; c < ((ntq + 3u) >> 2); c += 32) cp_row16(reuse, dst + 4u * c, src + 4u * c);
    }
  };

  auto decode_row = [&](const uint32_t* pb, uint32_t* o) {
    uint32_t base = 32u * SC + 32u * lane;
    auto seg = [&](uint32_t H, uint32_t s) {
      uint32_t P = base - p * __popc(H & lt);
      uint32_t step = 1024u - p * __popc(H);
      if constexpr (TAB && NPL > 0) {
        uint32_t e_lt = 0, e_all = 0;
#pragma unroll
        for (int k = 0; k < NPL; ++k) {
          const uint32_t Ek = H & epl[s * NPL + k];
          e_lt += __popc(Ek & lt) << k;
          e_all += __popc(Ek) << k;
        }
        P -= pscale * e_lt;
        step -= pscale * e_all;
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
      o[32u * s] = (H & lanebit) ? y : v;
      base += step;
    };
    if constexpr (SC >= 4) {
#pragma unroll
      for (uint32_t s = 0; s < SC; s += 4) {
        const uint4 h = *reinterpret_cast<const uint4*>(pb + s);
        seg(h.x, s);
        seg(h.y, s + 1);
        seg(h.z, s + 2);
        seg(h.w, s + 3);
      }
    } else {
#pragma unroll
      for (uint32_t s = 0; s < SC; ++s) seg(pb[s], s);
    }
  };

  auto decode_group = [&](const uint32_t* sb, uint64_t rbase, uint32_t kind) {
    uint32_t* const obase = out + rbase * W + lane;
    const uint32_t comp = __ballot_sync(kAll, kind == kComp);
    const uint32_t raw = __ballot_sync(kAll, kind == kRaw);
    const bool bad = kind == kBadRange || kind == kCorrupt;
    const uint32_t badm = __ballot_sync(kAll, bad);
    constexpr uint32_t kGroupBits = G >= 32 ? kAll : (1u << G) - 1u;
    if (!TAB && comp == kGroupBits) {
      // uniform plan, every row compressed (the common case): straight-line
      // code, so the rows' independent offset chains and shared loads can
      // overlap
#pragma unroll
      for (uint32_t q = 0; q < G; ++q) decode_row(sb + q * W, obase + q * W);
    } else {
#pragma unroll
      for (uint32_t q = 0; q < G; ++q) {
        if ((comp >> q) & 1u) decode_row(sb + q * W, obase + q * W);
      }
    }
    if (raw | badm) {
      if (bad) record_status(pv.status, kind == kBadRange ? IBP_ERANGE : IBP_ECORRUPT);
      for (uint32_t q = 0; q < G; ++q) {
        const bool r = (raw >> q) & 1u, z = (badm >> q) & 1u;
        if (!(r | z)) continue;
        uint32_t* orow = obase - lane + q * W;
        const uint4* prow = reinterpret_cast<const uint4*>(sb + q * W);
#pragma unroll
        for (uint32_t b = 0; b < CB; ++b) {
          const uint32_t c = lane + 32u * b;
          if (c < F::CH) reinterpret_cast<uint4*>(orow)[c] = r ? prow[c] : make_uint4(0, 0, 0, 0);
        }
      }
    }
  };

  // Pipeline over D stages: at iteration j, st[k] holds group j + k.  Per
  // iteration: load the ids of group j+D, issue the prefix of group j+D-1,
  // read the kinds of group j+1 from its landed headers and issue its rest,
  // decode group j.  cp.async groups are committed in the order prefix(j+D-1),
  // rest(j+1); the prologue commits an empty group after each of its first
  // D-2 prefixes so that every iteration sees the same order.  Then the
  // prefix of j+1 is complete once at most 2D-4 groups are pending (rest(j+D-3)
  // .. prefix(j+D-1)), and the rest of j once at most 2 are (prefix(j+D-1),
  // rest(j+1)).
  // PK: a group's ids are loaded one iteration before its row offsets, and
  // its offsets one iteration before its prefix, so ids run D+1 groups ahead.
  constexpr int IA = PK ? D + 1 : D;
  uint64_t rb0 = gw * G;  // first output row of group j
  int32_t idr[IA + 1];    // ids of groups j .. j+IA
  RowPos rpr[D + 1];      // row positions of groups j .. j+D (PK: loaded; else from the id)
  uint32_t bmr[D];        // bitmask words of groups j .. j+D-1
  uint32_t* st[D];
#pragma unroll
  for (int i = 0; i < IA; ++i) idr[i] = load_id(i, rb0 + i * row_step);
#pragma unroll
  for (int i = 0; i < D; ++i) {
    st[i] = stages + i * STAGE;
    bmr[i] = 0;
    rpr[i] = row_pos(idr[i]);
  }
#pragma unroll
  for (int i = 0; i < D - 1; ++i) {
    issue_prefix(i, st[i], idr[i], rpr[i], bmr[i]);
    cp_commit();
    if (i < D - 2) cp_commit();
  }
  cp_wait<2 * D - 4>();
  __syncwarp();
  uint32_t kind0, nt0;
  row_info(st[0], idr[0], rpr[0], bmr[0], kind0, nt0);
  issue_rest(0, st[0], idr[0], rpr[0], kind0, nt0);
  cp_commit();

  for (uint64_t j = 0; j < J; ++j, rb0 += row_step) {
    idr[IA] = load_id(j + IA, rb0 + IA * row_step);
    if constexpr (PK) rpr[D] = row_pos(idr[D]);
    issue_prefix(j + D - 1, st[D - 1], idr[D - 1], rpr[D - 1], bmr[D - 1]);
    cp_commit();
    cp_wait<2 * D - 4>();
    __syncwarp();
    uint32_t kind1, nt1;
    row_info(st[1], idr[1], rpr[1], bmr[1], kind1, nt1);
    issue_rest(j + 1, st[1], idr[1], rpr[1], kind1, nt1);
    cp_commit();
    cp_wait<2>();
    __syncwarp();
    decode_group(st[0], rb0, kind0);
    __syncwarp();
    kind0 = kind1;
    uint32_t* const t = st[0];
#pragma unroll
    for (int i = 0; i < D - 1; ++i) st[i] = st[i + 1];
    st[D - 1] = t;
#pragma unroll
    for (int i = 0; i < IA; ++i) idr[i] = idr[i + 1];
#pragma unroll
    for (int i = 0; i < D; ++i) rpr[i] = rpr[i + 1];
    if constexpr (!PK) rpr[D - 1] = row_pos(idr[D - 1]);
#pragma unroll
    for (int i = 0; i < D - 1; ++i) bmr[i] = bmr[i + 1];
    bmr[D - 1] = 0;
  }
  cp_wait<0>();
}

template <int R, int SC, int NPL, bool TAB, bool PK, uint32_t GW, bool MP = false, bool DEV = false>
static int launch_fast_t(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  using F = FastShape<SC, GW>;
  using T = TabShape<SC, R, NPL, TAB>;
  const size_t per_warp = 4ull * kFastStages * F::STAGE;
  const size_t fixed = 4ull * T::WORDS;
  size_t warps = (220ull * 1024 - fixed) / per_warp;
  if (warps > static_cast<size_t>(kFastWarps)) warps = kFastWarps;
  if (warps < 1) return IBP_EINVAL;
  const size_t smem = fixed + warps * per_warp;
  auto kern = k_decompress_fast<R, SC, NPL, TAB, PK, GW, MP, DEV>;
  // One-time set-up per device: the shared-memory opt-in and the occupancy
  // for this launch shape.
  static int occ_cache[64] = {0};
  const int dev = plan->device;
  if (dev < 0 || dev >= 64) return IBP_EINVAL;
  int occ = occ_cache[dev];
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    // Row-reuse copies are served from L1: prefer a quarter of the SM's
    // on-chip memory as shared memory and leave the rest to L1 (DLRM rows,
    // Zipf ids: 279 -> 286 GB/s; a smaller share left too few CTAs).
    if (GW == kGroupWordsReuse && e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 25);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, static_cast<int>(warps * 32), smem);
    if (e != cudaSuccess || occ < 1) {
      set_cuda_error(e, "set-up of k_decompress_fast");
      cudaGetLastError();
      return IBP_ECUDA;
    }
    occ_cache[dev] = occ;
  }
  const uint64_t groups = ((MP ? a.rows_per_plan : a.n_out) + F::G - 1) / F::G;
  const uint64_t need = (groups + warps - 1) / warps;
  uint64_t cap = static_cast<uint64_t>(occ) * sm_count(dev);
  if (MP) cap = cap / a.n_plans > 0 ? cap / a.n_plans : 1;  // CTAs per plan
  const dim3 grid(static_cast<unsigned>(need < cap ? need : cap), MP ? a.n_plans : 1u);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(warps * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // Programmatic dependent launch only for a grid that fills the GPU: with
  // fewer CTAs than it holds, the next launches' CTAs would be placed at once
  // and wait there, grid after grid (a small grid measured 1.6x slower).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = grid.x * grid.y >= cap * (MP ? a.n_plans : 1u) ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) {
    set_cuda_error(e, "k_decompress_fast");
    cudaGetLastError();
    return IBP_ECUDA;
  }
  return check_launch("k_decompress_fast");
}

template <int R, int NPL, bool TAB, bool PK, uint32_t GW, bool DEV = false>
static int launch_fast_sc(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  switch (plan->S) {
    case 1: return launch_fast_t<R, 1, NPL, TAB, PK, GW, false, DEV>(plan, a, stream);
    case 2: return launch_fast_t<R, 2, NPL, TAB, PK, GW, false, DEV>(plan, a, stream);
    case 4: return launch_fast_t<R, 4, NPL, TAB, PK, GW, false, DEV>(plan, a, stream);
    case 8: return launch_fast_t<R, 8, NPL, TAB, PK, GW, false, DEV>(plan, a, stream);
    case 16: return launch_fast_t<R, 16, NPL, TAB, PK, GW, false, DEV>(plan, a, stream);
    case 32: return launch_fast_t<R, 32, NPL, TAB, PK, GW, false, DEV>(plan, a, stream);
    default: return launch_fast_t<R, 64, NPL, TAB, PK, GW, false, DEV>(plan, a, stream);
  }
}

template <bool PK, uint32_t GW, bool DEV = false>
static int launch_fast_uniform_t(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  switch (plan->max_runs) {
    case 1: return launch_fast_sc<1, 0, false, PK, GW, DEV>(plan, a, stream);
    case 2: return launch_fast_sc<2, 0, false, PK, GW, DEV>(plan, a, stream);
    case 3: return launch_fast_sc<3, 0, false, PK, GW, DEV>(plan, a, stream);
    default: return launch_fast_sc<4, 0, false, PK, GW, DEV>(plan, a, stream);
  }
}

template <int R, bool PK, uint32_t GW, bool DEV = false>
static int launch_table_r(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  switch (plan->view.npl) {
    case 0: return launch_fast_sc<R, 0, true, PK, GW, DEV>(plan, a, stream);
    case 1: return launch_fast_sc<R, 1, true, PK, GW, DEV>(plan, a, stream);
    default: return launch_fast_sc<R, 6, true, PK, GW, DEV>(plan, a, stream);
  }
}

template <bool PK, uint32_t GW, bool DEV = false>
static int launch_fast_table_t(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  return plan->max_runs <= 2 ? launch_table_r<2, PK, GW, DEV>(plan, a, stream)
                             : launch_table_r<4, PK, GW, DEV>(plan, a, stream);
}

template <int R, int NPL>
static int launch_fast_set_sc(const ibp_plan* plan0, DecodeArgs& a, cudaStream_t stream) {
  switch (plan0->S) {
    case 1: return launch_fast_t<R, 1, NPL, true, false, kGroupWords, true>(plan0, a, stream);
    case 2: return launch_fast_t<R, 2, NPL, true, false, kGroupWords, true>(plan0, a, stream);
    case 4: return launch_fast_t<R, 4, NPL, true, false, kGroupWords, true>(plan0, a, stream);
    case 8: return launch_fast_t<R, 8, NPL, true, false, kGroupWords, true>(plan0, a, stream);
    case 16: return launch_fast_t<R, 16, NPL, true, false, kGroupWords, true>(plan0, a, stream);
    default: return launch_fast_t<R, 32, NPL, true, false, kGroupWords, true>(plan0, a, stream);
  }
}

// One translation unit each (compiled in parallel): slot layout uniform and
// table plans on host slots (kGroupWords) and on device slots
// (kGroupWordsDev, kGroupWordsDevTable), with the row-reuse hint
// (kGroupWordsReuse), packed layout uniform (device setting) and table plans.
int launch_fast_uniform(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);
int launch_fast_uniform_dev(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);
int launch_fast_uniform_reuse(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);
int launch_fast_table(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);
int launch_fast_table_dev(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);
int launch_fast_table_reuse(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);
int launch_fast_uniform_packed(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);
int launch_fast_table_packed(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream);

}  // namespace ibp
