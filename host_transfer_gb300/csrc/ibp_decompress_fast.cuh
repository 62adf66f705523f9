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

#include "ibp_decode_pipe.cuh"

namespace ibp {

constexpr int kFastWarps = 8;
constexpr int kFastStages = 3;  // shared-memory stages per warp (D >= 3)
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
// Compressed rows of two or more segments under per-word tables, from device
// memory (slots or the packed cache), are rebuilt two consecutive words per
// lane and written with 8-byte stores (RowPipe's PAIR decode): one header
// popcount, one base shuffle and one store per two words (sparse rows from
// HBM 2869 -> 2948 GB/s, packed 0.383 -> 0.400 of the HBM peak; with the
// straight-line group decode below, 0.58 -> 0.62 against one word per lane).
// Decodes that wait on the host link keep one word per lane and the fewer
// registers that allows.  Uniform plans keep one word per lane and segment:
// there a half-warp's fields sit one segment after the other's (56 words for
// dense rows), their shared-memory reads conflict two ways, and the pairs
// measured no faster on dense rows (2938 -> 2904 GB/s) and slower on DLRM
// rows (2849 -> 2748 GB/s).
constexpr bool kPairUniform = false;
constexpr bool kPairTable = true;
// A group whose rows are all compressed is decoded as straight-line code (no
// per-row branch), so the rows' offset chains and shared-memory loads overlap:
// always for uniform plans, and for per-word tables of at most two runs per
// word (sparse rows from HBM, two rows per group: 2957 -> 3476 GB/s, 0.53 ->
// 0.62 of the HBM peak; packed 0.47 -> 0.51), on device slots only.  Tables of
// up to four runs keep the per-row branch (straight-line code there spilled
// registers), and so do host slots and plan sets: their decode waits on the
// link, and the straight-line groups of up to eight rows took more registers
// (80 -> 135) and so fewer CTAs (per-head K/V plan sets from host slots
// 227 -> 174 GB/s).
constexpr bool kStraightTable = true;
// Rows whose stored streams are mostly short (at most W / 4 words, as
// ibp_plan_tune_prefix records) take stage rows of W / 4 words when their
// slots are in device memory (per-word tables of up to two runs and one
// e-plane, rows of 256 or 512 words): the stages shrink to a quarter, so the
// register budget (80, three CTAs of eight warps) rather than shared memory
// bounds the warps per SM, and the rare longer rows are decoded from their
// slots.  Sparse rows from HBM 3476 -> 3775 GB/s (0.62 -> 0.67 of the HBM
// peak); a four-CTA budget (64 registers) measured 0.55.  The small stages
// also make room for a deeper pipeline: four stages 0.67 -> 0.68 (five 0.64,
// six 0.61: the extra stages' state costs registers); a prefix of RW words,
// so that no row of at most RW words needs a second fetch, measured 0.66;
// seven or six warps per CTA (97 or 113 registers) 0.61 and 0.60.
constexpr bool kShortRows = true;
constexpr int kShortStages = 4;  // shared-memory stages per warp with short stage rows

// PK = false: row r of the table is slots[r * W ..]; PK = true: the packed
// layout, row r is slots[offsets[r] .. offsets[r + 1]) (its stored words
// rounded up to 16 bytes), and a row whose stream would reach past that
// extent is corrupt.
// MP = true (plan sets, contiguous decode, table path): CTA row blockIdx.y
// decodes rows [y * rows_per_plan, (y + 1) * rows_per_plan) of the table with
// plan y of a.plans (a device array of plan views).
// CTAs per SM the register allocation is sized for, where that causes no
// spills (measured on one GB300): uniform plans up to W = 1024 with 512-word
// groups fit four (+1 % on dense and DLRM rows); with the 768-word groups of
// device slots shared memory holds three, and a three-CTA budget (80
// registers) keeps them all resident; per-word-table plans up to W = 512 with
// at most one e-plane fit three with 512-word groups (instead of the two that
// 107 registers allowed: +9 % for device slots, -2 % over the host link, so
// host slots keep the compiler's choice) and two with 1024-word groups; other
// shapes keep the compiler's choice.
// Rows split into tasks (NP > 1): a register budget for three CTAs (tasks of
// 32 segments, whose stages leave two CTAs per SM, measured the same with a
// budget for two).
// Short stage rows (SHORT) leave room for four CTAs or more; a budget for
// three measured best (see kShortRows).
template <int SC, int NPL, bool TAB, bool MP, bool DEV, uint32_t GW, int NP = 1, bool SHORT = false>
constexpr int fast_min_blocks() {
  if (NP > 1 || SHORT) return 3;
  if (!TAB) return DEV ? (SC <= 32 ? 3 : 1) : (SC <= 32 ? 4 : 1);
  if (DEV && !MP && SC <= 16 && NPL <= 1) return GW >= 1024 ? 2 : 3;
  return 1;
}

// DEV (slots or packed cache in device memory) selects the register budget
// (fast_min_blocks) and, for per-word tables, the pair decode and the
// straight-line groups.  NP > 1: every row
// is NP tasks of SC / NP segments (RowPipe), for rows of 32 or 64 segments
// whose slots are in device memory.
template <int R, int SC, int NPL, bool TAB, bool PK, uint32_t GW, bool MP = false, bool DEV = false, int NP = 1,
          bool SHORT = false>
__global__ void __launch_bounds__(kFastWarps * 32, (fast_min_blocks<SC, NPL, TAB, MP, DEV, GW, NP, SHORT>()))
    k_decompress_fast(const DecodeArgs a) {
  static_assert(!MP || (TAB && !PK), "plan sets decode through the table path, slot layout");
  static_assert(NP == 1 || !MP, "plan sets decode whole rows");
  constexpr bool PAIR = SC >= 2 && (TAB ? kPairTable && DEV : kPairUniform);
  using Pipe = RowPipe<R, SC, NPL, TAB, PK, GW, NP, PAIR, SHORT>;
  using F = typename Pipe::F;
  using T = typename Pipe::T;
  constexpr uint32_t W = F::W, G = F::G, STAGE = F::STAGE, CB = F::CB, RW = F::RW;
  extern __shared__ __align__(128) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t nw_cta = blockDim.x >> 5;
  constexpr int D = SHORT ? kShortStages : kFastStages;
  uint32_t* const stages = smem + T::WORDS + warp * static_cast<uint32_t>(D) * STAGE;

  // this CTA's plan, row range and output
  PlanView pv;
  if constexpr (MP)
    pv = a.plans[blockIdx.y];
  else
    pv = a.pv;
  const uint64_t n_out = (MP ? a.rows_per_plan : a.n_out) * NP;  // rows, or tasks
  const uint64_t first = MP ? a.first + blockIdx.y * a.rows_per_plan : a.first;
  uint32_t* const out = MP ? a.out + blockIdx.y * a.rows_per_plan * (32ull * SC) : a.out;

  // plan constants, and the per-word tables staged once per CTA (every
  // thread reaches the barrier inside before any warp leaves)
  Pipe pp;
  pp.init(pv, a.slots, a.bitmask, a.offsets, a.n_rows, NP > 1 ? SC : (MP ? pv.pre : a.pre), smem);

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
  // IBP_HINT_EARLY_FETCH (the caller states that the previous kernel wrote
  // none of this call's inputs): the wait moves after the pipeline's prologue,
  // so the first ids and prefixes are fetched while the previous grid drains;
  // every write still comes after the wait.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (gw >= n_groups) return;  // warp-uniform; only warp-level syncs below
  const bool early = (pv.hints & IBP_HINT_EARLY_FETCH) != 0;  // CTA-uniform
  if (!early) asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint64_t J = (n_groups - gw + nwarps - 1) / nwarps;
  const uint64_t row_step = nwarps * G;  // first row of group j+1 minus first row of group j

  auto load_id = [&](uint64_t j, uint64_t rbase) -> int32_t {
    const uint64_t i = rbase + lane;
    if (j >= J || lane >= G || i >= n_out) return kNoRow;
    const uint64_t r = i / NP;  // output row (NP > 1: of task i)
    return pp.check_id(a.ids ? a.ids[r] : static_cast<int64_t>(first + r));
  };
  // NP > 1: the part of its row that the task of group j (first task rbase) is
  auto part_of = [&](uint64_t rbase) -> uint32_t { return static_cast<uint32_t>(rbase % NP); };

  // NP > 1: one task; its words WP * part .. of output row rbase / NP.
  auto decode_task = [&](const uint32_t* sb, uint64_t rbase, uint32_t kind, uint32_t nt,
                         const typename Pipe::Bases& bases) {
    const uint32_t k0 = __shfl_sync(kAll, kind, 0);
    if (k0 == kNone) return;
    const uint32_t part = part_of(rbase);
    uint32_t* const orow = out + (rbase / NP) * W + part * Pipe::WP;
    if (k0 == kComp) {
      const uint32_t c0 = __shfl_sync(kAll, nt, 0) >> 16;
      const uint32_t tb = pp.task_bases(bases, part, 128u * c0 - 32u * SC);
      if constexpr (PAIR) {
        uint2* const o2 = reinterpret_cast<uint2*>(orow) + lane;
        pp.template decode_pairs_at<Pipe::SEGP>(
            sb, sb, part * Pipe::SEGP, [&](uint32_t j) { return __shfl_sync(kAll, tb, j); },
            [&](uint32_t k, uint32_t y0, uint32_t y1) { o2[32u * k] = make_uint2(y0, y1); });
      } else {
        uint32_t* const o = orow + lane;
        pp.template decode_segments_at<Pipe::SEGP>(
            sb, sb, part * Pipe::SEGP, [&](uint32_t j) { return __shfl_sync(kAll, tb, j); },
            [&](uint32_t j, uint32_t y) { o[32u * j] = y; });
      }
      return;
    }
    if (k0 != kRaw && lane == 0) record_status(pv.status, k0 == kBadRange ? IBP_ERANGE : IBP_ECORRUPT);
    const uint4* prow = reinterpret_cast<const uint4*>(sb + SC);
#pragma unroll
    for (uint32_t c = lane; c < Pipe::WP / 4; c += 32)
      reinterpret_cast<uint4*>(orow)[c] = k0 == kRaw ? prow[c] : make_uint4(0, 0, 0, 0);
  };

  // id: lane q < G holds row q's id (SHORT: rows read from their slots).
  auto decode_group = [&](const uint32_t* sb, uint64_t rbase, uint32_t kind, const typename Pipe::Bases& bases,
                          int32_t id) {
    uint32_t* const obase = out + rbase * W + lane;
    const uint32_t comp = __ballot_sync(kAll, kind == kComp);
    const uint32_t raw = __ballot_sync(kAll, kind == kRaw);
    const bool bad = kind == kBadRange || kind == kCorrupt;
    const uint32_t badm = __ballot_sync(kAll, bad);
    constexpr uint32_t kGroupBits = G >= 32 ? kAll : (1u << G) - 1u;
    // row q of the group, compressed: one 4-byte store per lane and segment,
    // or (PAIR) one 8-byte store per lane and 64-word block
    auto decode_comp = [&](uint32_t q) {
      if constexpr (PAIR) {
        uint2* const o2 = reinterpret_cast<uint2*>(obase - lane + q * W) + lane;
        pp.decode_row_pairs(sb + q * RW, q, bases,
                            [&](uint32_t k, uint32_t y0, uint32_t y1) { o2[32u * k] = make_uint2(y0, y1); });
      } else {
        uint32_t* o = obase + q * W;
        pp.decode_row(sb + q * W, q, bases, [&](uint32_t s, uint32_t y) { o[32u * s] = y; });
      }
    };
    if ((!TAB || (kStraightTable && R <= 2 && DEV && !MP)) && comp == kGroupBits) {
      // every row compressed (the common case): straight-line code, so the
      // rows' independent offset chains and shared loads can overlap
#pragma unroll
      for (uint32_t q = 0; q < G; ++q) decode_comp(q);
    } else {
#pragma unroll
      for (uint32_t q = 0; q < G; ++q) {
        if ((comp >> q) & 1u) decode_comp(q);
      }
    }
    if constexpr (SHORT) {
      // rows that have no stage row: compressed rows longer than RW words,
      // decoded from their slots (headers from the stage), and raw rows,
      // copied from their slots in 16-byte chunks; then bad ids and corrupt
      // rows, zero-filled
      const uint32_t slotm = __ballot_sync(kAll, kind == kCompSlot);
      for (uint32_t m = slotm | raw | badm; m; m &= m - 1) {
        const uint32_t q = __ffs(m) - 1;
        const int32_t idq = __shfl_sync(kAll, id, q);
        uint32_t* const orow = obase - lane + q * W;
        if ((slotm >> q) & 1u) {
          uint2* const o2 = reinterpret_cast<uint2*>(orow) + lane;
          pp.decode_row_pairs_from(sb + q * RW, a.slots + static_cast<uint64_t>(idq) * W, q, bases,
                                   [&](uint32_t k, uint32_t y0, uint32_t y1) { o2[32u * k] = make_uint2(y0, y1); });
        } else {
          const bool r = (raw >> q) & 1u;
          const uint4* const prow = reinterpret_cast<const uint4*>(a.slots + static_cast<uint64_t>(r ? idq : 0) * W);
#pragma unroll
          for (uint32_t b = 0; b < CB; ++b) {
            const uint32_t c = lane + 32u * b;
            if (c < F::CH) reinterpret_cast<uint4*>(orow)[c] = r ? prow[c] : make_uint4(0, 0, 0, 0);
          }
        }
      }
      if (bad) record_status(pv.status, kind == kBadRange ? IBP_ERANGE : IBP_ECORRUPT);
      return;
    }
    if (raw == kGroupBits) {
      // every row raw (e.g. K/V rows of 64 words that no Mask compresses): the
      // group's rows are contiguous in the stage and in the output, so one
      // flat copy in 16-byte chunks keeps every lane busy
      const uint4* src = reinterpret_cast<const uint4*>(sb);
      uint4* dst = reinterpret_cast<uint4*>(obase - lane);
#pragma unroll
      for (uint32_t c = lane; c < G * W / 4; c += 32) dst[c] = src[c];
      return;
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
    rpr[i] = pp.row_pos(idr[i]);
  }
#pragma unroll
  for (int i = 0; i < D - 1; ++i) {
    if (static_cast<uint64_t>(i) < J) pp.issue_prefix(st[i], idr[i], rpr[i], bmr[i]);
    cp_commit();
    if (i < D - 2) cp_commit();
  }
  cp_wait<2 * D - 4>();
  __syncwarp();
  uint32_t kind0, nt0;
  typename Pipe::Bases bases0;
  pp.row_info(st[0], idr[0], rpr[0], bmr[0], kind0, nt0, bases0, part_of(rb0));
  pp.issue_rest(st[0], idr[0], rpr[0], kind0, nt0);
  cp_commit();
  if (early) asm volatile("griddepcontrol.wait;" ::: "memory");  // before the first write

  for (uint64_t j = 0; j < J; ++j, rb0 += row_step) {
    idr[IA] = load_id(j + IA, rb0 + IA * row_step);
    if constexpr (PK) rpr[D] = pp.row_pos(idr[D]);
    if (j + D - 1 < J) pp.issue_prefix(st[D - 1], idr[D - 1], rpr[D - 1], bmr[D - 1]);
    cp_commit();
    cp_wait<2 * D - 4>();
    __syncwarp();
    uint32_t kind1, nt1;
    typename Pipe::Bases bases1;
    pp.row_info(st[1], idr[1], rpr[1], bmr[1], kind1, nt1, bases1, part_of(rb0 + row_step));
    if (j + 1 < J) pp.issue_rest(st[1], idr[1], rpr[1], kind1, nt1);
    cp_commit();
    cp_wait<2>();
    __syncwarp();
    if constexpr (NP > 1)
      decode_task(st[0], rb0, kind0, nt0, bases0);
    else
      decode_group(st[0], rb0, kind0, bases0, idr[0]);
    __syncwarp();
    kind0 = kind1;
    nt0 = nt1;
    bases0 = bases1;
    uint32_t* const t = st[0];
#pragma unroll
    for (int i = 0; i < D - 1; ++i) st[i] = st[i + 1];
    st[D - 1] = t;
#pragma unroll
    for (int i = 0; i < IA; ++i) idr[i] = idr[i + 1];
#pragma unroll
    for (int i = 0; i < D; ++i) rpr[i] = rpr[i + 1];
    if constexpr (!PK) rpr[D - 1] = pp.row_pos(idr[D - 1]);
#pragma unroll
    for (int i = 0; i < D - 1; ++i) bmr[i] = bmr[i + 1];
    bmr[D - 1] = 0;
  }
  cp_wait<0>();
}

template <int R, int SC, int NPL, bool TAB, bool PK, uint32_t GW, bool MP = false, bool DEV = false, int NP = 1,
          bool SHORT = false>
static int launch_fast_t(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  using F = FastShape<SC, GW, NP, SHORT>;
  using T = TabShape<SC, R, NPL, TAB>;
  const size_t per_warp = 4ull * (SHORT ? kShortStages : kFastStages) * F::STAGE;
  const size_t fixed = 4ull * T::WORDS;
  size_t warps = (220ull * 1024 - fixed) / per_warp;
  if (warps > static_cast<size_t>(kFastWarps)) warps = kFastWarps;
  if (warps < 1) return IBP_EINVAL;
  const size_t smem = fixed + warps * per_warp;
  auto kern = k_decompress_fast<R, SC, NPL, TAB, PK, GW, MP, DEV, NP, SHORT>;
  // One-time set-up per device: the shared-memory opt-in and the occupancy
  // for this launch shape.
  static std::atomic<int> occ_cache[64];  // per device, any host thread
  const int dev = plan->device;
  if (dev < 0 || dev >= 64) return IBP_EINVAL;
  int occ = occ_cache[dev].load(std::memory_order_relaxed);
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
    occ_cache[dev].store(occ, std::memory_order_relaxed);
  }
  const uint64_t groups = ((MP ? a.rows_per_plan : a.n_out) * NP + F::G - 1) / F::G;
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
    // rows of 32 and 64 segments in device memory: two tasks per row (of 16
    // and 32 segments; 2048-word rows in four tasks of 16: 13.3 us per LLM
    // weight launch from HBM, in two of 32: 11.9 us, and the layer step 0.81
    // -> 0.94 of the HBM peak, the next launches' CTAs finding room beside
    // the two CTAs per SM that the larger stages leave)
    case 32: return launch_fast_t<R, 32, NPL, TAB, PK, GW, false, DEV, (DEV && !PK ? 2 : 1)>(plan, a, stream);
    default: return launch_fast_t<R, 64, NPL, TAB, PK, GW, false, DEV, (DEV && !PK ? 2 : 1)>(plan, a, stream);
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

// Short stage rows (slots in device memory, per-word tables, rows of 8 or 16
// segments, at most one e-plane), two rows per group: with four (256-word
// rows in 1024-word groups) the straight-line group spilled registers.
template <int R>
static int launch_fast_short(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  const bool e0 = plan->view.npl == 0;
  if (plan->S == 8)
    return e0 ? launch_fast_t<R, 8, 0, true, false, 512, false, true, 1, true>(plan, a, stream)
              : launch_fast_t<R, 8, 1, true, false, 512, false, true, 1, true>(plan, a, stream);
  return e0 ? launch_fast_t<R, 16, 0, true, false, 1024, false, true, 1, true>(plan, a, stream)
            : launch_fast_t<R, 16, 1, true, false, 1024, false, true, 1, true>(plan, a, stream);
}

template <bool PK, uint32_t GW, bool DEV = false>
static int launch_fast_table_t(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  // rows of 8 or 16 segments in device memory whose stored streams are
  // mostly at most W / 4 words (ibp_plan_tune_prefix found so), at most two
  // runs of kept bits per word, at most one e-plane: stage rows of W / 4 words
  if constexpr (DEV && !PK && kShortRows) {
    if (plan->short_rows && plan->max_runs <= 2 && plan->view.npl <= 1 && a.pre <= plan->W / 4u &&
        (plan->S == 8 || plan->S == 16)) {
      if (plan->max_runs <= 1) return launch_fast_short<1>(plan, a, stream);
      return launch_fast_short<2>(plan, a, stream);
    }
  }
  // one run of kept bits per word and at most one e-plane (the sparse tables'
  // plans): a one-run deposit per word instead of two
  if (plan->max_runs <= 1 && plan->view.npl <= 1)
    return plan->view.npl == 0 ? launch_fast_sc<1, 0, true, PK, GW, DEV>(plan, a, stream)
                               : launch_fast_sc<1, 1, true, PK, GW, DEV>(plan, a, stream);
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
