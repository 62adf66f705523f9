// ibp_bag.cuh - gather-decompress fused with sum / mean pooling (an
// "embedding bag"): the rows of each bag are decoded and added into per-lane
// float accumulators; decoded rows never go to HBM, only one pooled row per
// bag does.
//
// « Résultats »: IBP's rows feed DLRM embedding tables and GNN feature
// aggregation, whose consumer pools the rows of each bag; « Algorithme
// central », step 3 (last point): fetching overlaps the logic that consumes
// the data.  Pooling (the reading, as in the oracle): out[b] = the rows of
// ids[offsets[b] .. offsets[b+1]) added as IEEE single values in that order
// from +0.0, or that sum divided by the bag size (mean; an empty bag gives
// zeros).  A bag with offsets outside 0 <= offsets[b] <= offsets[b+1] <= n_ids
// gives zeros and IBP_ERANGE; a bad id or a corrupt slot decodes to a zero
// row that still counts in the bag's size (IBP_ERANGE / IBP_ECORRUPT).
//
// The fetch and decode steps are those of k_decompress_fast (RowPipe in
// ibp_decode_pipe.cuh: same plan shapes, same three-stage cp.async pipeline
// of prefix, then rest, per group of G rows).
// What differs is the unit of work: warp gw owns bags gw, gw + nwarps, ...; a
// cursor cuts each bag into groups of at most G consecutive ids (a group
// never spans two bags; an empty or invalid bag is one group of no rows), and
// the decode of a group adds its rows, in order, into the lanes'
// accumulators (word lane + 32 s in acc[s]; under per-word tables, when a
// warp pools whole rows, word 64 k + 2 lane + i in acc[2 k + i]); the group
// that ends a bag writes the bag's output row.
#pragma once

#include "ibp_decompress_fast.cuh"

namespace ibp {

// BF16: every decoded word holds two bfloat16 elements (element 2j in bits
// 0-15), each widened exactly to float and pooled on its own; the output row
// has 2W floats.
// CS > 1 (column split, for few bags on device slots): a team of CS
// consecutive warps takes each bag; all of them fetch its rows (the repeats
// are L2 hits) and warp `part` of the team decodes and pools only segments
// [part * SC/CS, (part + 1) * SC/CS), skipping the earlier segments' fields by
// their headers.  Each column is still added in bag order.
template <int R, int SC, int NPL, bool TAB, uint32_t GW, bool BF16, int CS = 1>
__global__ void __launch_bounds__(kFastWarps * 32) k_bag(const BagArgs ba) {
  static_assert(CS >= 1 && SC % CS == 0, "a warp pools whole segments");
  constexpr uint32_t SPW = SC / CS;  // segments this warp pools
  // per-word tables: two consecutive words per lane (as in k_decompress_fast)
  // where a warp pools whole rows (sparse bags from host slots 967 -> 979-984
  // GB/s); warps of a team keep one word per lane (with pairs, sparse bags
  // from HBM in teams of two: 2196 -> 1981 GB/s)
  constexpr bool PAIR = TAB && kPairTable && CS == 1 && SPW % 2 == 0;
  using Pipe = RowPipe<R, SC, NPL, TAB, false, GW, 1, PAIR>;
  using F = typename Pipe::F;
  using T = typename Pipe::T;
  constexpr uint32_t W = F::W, G = F::G, STAGE = F::STAGE;
  constexpr int D = kFastStages;
  extern __shared__ __align__(128) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t nw_cta = blockDim.x >> 5;
  uint32_t* const stages = smem + T::WORDS + warp * static_cast<uint32_t>(D) * STAGE;

  const PlanView pv = ba.d.pv;
  const int64_t* const ids = ba.d.ids;
  Pipe pp;
  pp.init(pv, ba.d.slots, ba.d.bitmask, nullptr, ba.d.n_rows, ba.d.pre, smem);
  const uint64_t n_bags = ba.n_bags;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * nw_cta + warp;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * nw_cta;
  // Programmatic dependent launch, as in k_decompress_fast: the next kernel
  // may start as this grid drains; wait for the previous grid before
  // touching per-call data.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint64_t team = gw / CS, nteams = nwarps / CS;  // warps per CTA are a multiple of CS
  const uint32_t s_lo = CS == 1 ? 0u : static_cast<uint32_t>(gw % CS) * SPW;
  if (team >= n_bags) return;  // warp-uniform; only warp-level syncs below
  // IBP_HINT_EARLY_FETCH: as in k_decompress_fast, the prologue's reads (bag
  // offsets, ids, bitmask words, prefixes) may come before the wait; every
  // write (pooled rows, status word) comes after it.
  const bool early = (pv.hints & IBP_HINT_EARLY_FETCH) != 0;
  if (!early) asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- the cursor over this warp's bags (warp-uniform state) ----
  struct Grp {
    uint64_t bag;  // n_bags: no group
    uint64_t pos;  // first id position
    uint32_t n;    // ids in the group (<= G)
    uint32_t last;  // the group ends its bag
    uint32_t bad;   // the bag's offsets are invalid
  };
  uint64_t cb = team, cp = 0, ce = 0;
  uint32_t cbad = 0;
  auto open_bag = [&]() {
    const int64_t lo = ba.offsets[cb], hi = ba.offsets[cb + 1];
    const bool ok = lo >= 0 && lo <= hi && static_cast<uint64_t>(hi) <= ba.n_ids;
    cp = ok ? static_cast<uint64_t>(lo) : 0;
    ce = ok ? static_cast<uint64_t>(hi) : 0;
    cbad = ok ? 0u : 1u;
  };
  open_bag();
  auto next_group = [&]() -> Grp {
    Grp g{n_bags, 0, 0, 0, 0};
    if (cb >= n_bags) return g;
    const uint64_t left = ce - cp;
    g.bag = cb;
    g.pos = cp;
    g.n = static_cast<uint32_t>(left < G ? left : G);
    g.last = left <= G ? 1u : 0u;
    g.bad = cbad;
    cp += g.n;
    if (g.last) {
      cb += nteams;
      if (cb < n_bags) open_bag();
    }
    return g;
  };

  // Row ids of a group: lane q < n holds the id at position pos + q.
  auto load_id = [&](const Grp& g) -> int32_t {
    if (g.bag >= n_bags || lane >= g.n) return kNoRow;
    return pp.check_id(ids[g.pos + lane]);
  };

  constexpr uint32_t NA = BF16 ? 2 * SPW : SPW;  // accumulators per lane
  float acc[NA];
#pragma unroll
  for (uint32_t s = 0; s < NA; ++s) acc[s] = 0.0f;
  uint64_t cnt = 0;  // ids of the current bag seen so far
  // Word j of this lane (j < SPW) is word lane + 32 (s_lo + j) of a row, or
  // (PAIR) word 64 (j / 2) + 2 lane + j % 2 of segments s_lo ...
  auto word_of = [&](uint32_t j) -> uint32_t {
    return PAIR ? 32u * s_lo + 64u * (j / 2u) + 2u * lane + (j % 2u) : lane + 32u * (s_lo + j);
  };
  // add decoded word w (this lane's word j of a row)
  auto add_word = [&](uint32_t j, uint32_t w) {
    if constexpr (BF16) {
      acc[2 * j] = __fadd_rn(acc[2 * j], __uint_as_float(w << 16));
      acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], __uint_as_float(w & 0xFFFF0000u));
    } else {
      acc[j] = __fadd_rn(acc[j], __uint_as_float(w));
    }
  };
  auto add_row = [&](const uint32_t* pb, uint32_t q, const typename Pipe::Bases& bases) {
    if constexpr (PAIR) {
      pp.template decode_pairs_at<SPW>(
          pb, pb, s_lo, [&](uint32_t j) { return pp.seg_base_pair(bases, q, s_lo + j); },
          [&](uint32_t k, uint32_t y0, uint32_t y1) {
            add_word(2u * k, y0);
            add_word(2u * k + 1u, y1);
          });
    } else {
      pp.template decode_segments<SPW>(pb, pb, q, s_lo, bases, [&](uint32_t j, uint32_t y) { add_word(j, y); });
    }
  };

  // Add group g's rows in order; the group that ends a bag writes it out.
  auto consume = [&](const Grp& g, const uint32_t* sb, uint32_t kind, const typename Pipe::Bases& bases) {
    const uint32_t comp = __ballot_sync(kAll, kind == kComp);
    const uint32_t raw = __ballot_sync(kAll, kind == kRaw);
    const bool bad = kind == kBadRange || kind == kCorrupt;
    if (bad) record_status(pv.status, kind == kBadRange ? IBP_ERANGE : IBP_ECORRUPT);
    constexpr uint32_t kGroupBits = G >= 32 ? kAll : (1u << G) - 1u;
    if ((!TAB || (kStraightTable && R <= 2)) && comp == kGroupBits) {
      // every row compressed: straight-line code, so the rows' decode work
      // overlaps (the additions still follow the row order)
#pragma unroll
      for (uint32_t q = 0; q < G; ++q) add_row(sb + q * W, q, bases);
    } else {
#pragma unroll
      for (uint32_t q = 0; q < G; ++q) {
        if ((comp >> q) & 1u) {
          add_row(sb + q * W, q, bases);
        } else if ((raw >> q) & 1u) {
#pragma unroll
          for (uint32_t j = 0; j < SPW; ++j) add_word(j, sb[q * W + word_of(j)]);
        }
      }
    }
    cnt += g.n;
    if (g.last) {
      if (g.bad && lane == 0) record_status(pv.status, IBP_ERANGE);
      const float c = static_cast<float>(cnt);
      const bool div = ba.mean && cnt;
      if constexpr (BF16) {
        float2* const o = reinterpret_cast<float2*>(ba.out + g.bag * (2 * W));
#pragma unroll
        for (uint32_t j = 0; j < SPW; ++j) {
          const float lo = acc[2 * j], hi = acc[2 * j + 1];
          o[word_of(j)] = div ? make_float2(__fdiv_rn(lo, c), __fdiv_rn(hi, c)) : make_float2(lo, hi);
        }
      } else {
        float* const o = ba.out + g.bag * W;
#pragma unroll
        for (uint32_t j = 0; j < SPW; ++j) o[word_of(j)] = div ? __fdiv_rn(acc[j], c) : acc[j];
      }
#pragma unroll
      for (uint32_t s = 0; s < NA; ++s) acc[s] = 0.0f;
      cnt = 0;
    }
  };

  // Pipeline over D stages, as in k_decompress_fast: at iteration j, st[k]
  // holds group j + k; cp.async groups are committed in the order
  // prefix(j+D-1), rest(j+1), with empty commits in the prologue.
  Grp gr[D + 1];
  int32_t idr[D + 1];
  uint32_t bmr[D];
  uint32_t* st[D];
#pragma unroll
  for (int i = 0; i < D; ++i) {
    gr[i] = next_group();
    idr[i] = load_id(gr[i]);
    st[i] = stages + i * STAGE;
    bmr[i] = 0;
  }
#pragma unroll
  for (int i = 0; i < D - 1; ++i) {
    pp.issue_prefix(st[i], idr[i], pp.row_pos(idr[i]), bmr[i]);
    cp_commit();
    if (i < D - 2) cp_commit();
  }
  cp_wait<2 * D - 4>();
  __syncwarp();
  uint32_t kind0, nt0;
  typename Pipe::Bases bases0;
  pp.row_info(st[0], idr[0], pp.row_pos(idr[0]), bmr[0], kind0, nt0, bases0);
  pp.issue_rest(st[0], idr[0], pp.row_pos(idr[0]), kind0, nt0);
  cp_commit();
  if (early) asm volatile("griddepcontrol.wait;" ::: "memory");  // before the first write

  while (gr[0].bag < n_bags) {
    gr[D] = next_group();
    idr[D] = load_id(gr[D]);
    pp.issue_prefix(st[D - 1], idr[D - 1], pp.row_pos(idr[D - 1]), bmr[D - 1]);
    cp_commit();
    cp_wait<2 * D - 4>();
    __syncwarp();
    uint32_t kind1, nt1;
    typename Pipe::Bases bases1;
    pp.row_info(st[1], idr[1], pp.row_pos(idr[1]), bmr[1], kind1, nt1, bases1);
    pp.issue_rest(st[1], idr[1], pp.row_pos(idr[1]), kind1, nt1);
    cp_commit();
    cp_wait<2>();
    __syncwarp();
    consume(gr[0], st[0], kind0, bases0);
    __syncwarp();
    kind0 = kind1;
    bases0 = bases1;
    uint32_t* const t = st[0];
#pragma unroll
    for (int i = 0; i < D - 1; ++i) st[i] = st[i + 1];
    st[D - 1] = t;
#pragma unroll
    for (int i = 0; i < D; ++i) {
      gr[i] = gr[i + 1];
      idr[i] = idr[i + 1];
    }
#pragma unroll
    for (int i = 0; i < D - 1; ++i) bmr[i] = bmr[i + 1];
    bmr[D - 1] = 0;
  }
  cp_wait<0>();
}

template <int R, int SC, int NPL, bool TAB, uint32_t GW, bool BF16, int CS = 1>
static int launch_bag_t(const ibp_plan* plan, BagArgs& a, cudaStream_t stream) {
  using F = FastShape<SC, GW>;
  using T = TabShape<SC, R, NPL, TAB>;
  const size_t per_warp = 4ull * kFastStages * F::STAGE;
  const size_t fixed = 4ull * T::WORDS;
  size_t warps = (220ull * 1024 - fixed) / per_warp;
  if (warps > static_cast<size_t>(kFastWarps)) warps = kFastWarps;
  if (warps < 1) return IBP_EINVAL;
  const size_t smem = fixed + warps * per_warp;
  if (warps % CS != 0) return IBP_EINVAL;  // a team's warps share a CTA
  auto kern = k_bag<R, SC, NPL, TAB, GW, BF16, CS>;
  static std::atomic<int> occ_cache[64];  // per device, any host thread
  const int dev = plan->device;
  if (dev < 0 || dev >= 64) return IBP_EINVAL;
  int occ = occ_cache[dev].load(std::memory_order_relaxed);
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, static_cast<int>(warps * 32), smem);
    if (e != cudaSuccess || occ < 1) {
      set_cuda_error(e, "set-up of k_bag");
      cudaGetLastError();
      return IBP_ECUDA;
    }
    occ_cache[dev].store(occ, std::memory_order_relaxed);
  }
  const uint64_t need = (a.n_bags * CS + warps - 1) / warps;
  const uint64_t cap = static_cast<uint64_t>(occ) * sm_count(dev);
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(static_cast<unsigned>(warps * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // Programmatic dependent launch only for device slots and a grid of at
  // least half the GPU's CTAs (measured: with far fewer CTAs the next
  // launches' CTAs are placed at once and wait, 1.6x slower for 1,024 bags in
  // 128 CTAs; 2,048 bags in 256 CTAs gain 3 %; over the host link it cost
  // 3 % on DLRM bags).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (a.d.dev_slots && 2ull * grid >= cap) ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) {
    set_cuda_error(e, "k_bag");
    cudaGetLastError();
    return IBP_ECUDA;
  }
  return check_launch("k_bag");
}

template <int R, int NPL, bool TAB, uint32_t GW, bool BF16, int CS = 1>
static int launch_bag_sc(const ibp_plan* plan, BagArgs& a, cudaStream_t stream) {
  switch (plan->S) {
    case 1: return launch_bag_t<R, 1, NPL, TAB, GW, BF16, (CS <= 1 ? CS : 1)>(plan, a, stream);
    case 2: return launch_bag_t<R, 2, NPL, TAB, GW, BF16, (CS <= 2 ? CS : 1)>(plan, a, stream);
    case 4: return launch_bag_t<R, 4, NPL, TAB, GW, BF16, (CS <= 4 ? CS : 1)>(plan, a, stream);
    case 8: return launch_bag_t<R, 8, NPL, TAB, GW, BF16, (CS <= 8 ? CS : 1)>(plan, a, stream);
    default: return launch_bag_t<R, 16, NPL, TAB, GW, BF16, (CS <= 16 ? CS : 1)>(plan, a, stream);
  }
}

template <int R, uint32_t GW, bool BF16, int CS = 1>
static int launch_bag_table(const ibp_plan* plan, BagArgs& a, cudaStream_t stream) {
  switch (plan->view.npl) {
    case 0: return launch_bag_sc<R, 0, true, GW, BF16, CS>(plan, a, stream);
    case 1: return launch_bag_sc<R, 1, true, GW, BF16, CS>(plan, a, stream);
    default: return launch_bag_sc<R, 6, true, GW, BF16, CS>(plan, a, stream);
  }
}

template <uint32_t GW, bool BF16, int CS = 1>
static int launch_bag_gw(const ibp_plan* plan, BagArgs& a, cudaStream_t stream) {
  if (!plan->uniform) {
    if (plan->max_runs <= 1 && plan->view.npl <= 1)  // one-run deposits, as in the decoder
      return plan->view.npl == 0 ? launch_bag_sc<1, 0, true, GW, BF16, CS>(plan, a, stream)
                                 : launch_bag_sc<1, 1, true, GW, BF16, CS>(plan, a, stream);
    return plan->max_runs <= 2 ? launch_bag_table<2, GW, BF16, CS>(plan, a, stream)
                               : launch_bag_table<4, GW, BF16, CS>(plan, a, stream);
  }
  switch (plan->max_runs) {
    case 1: return launch_bag_sc<1, 0, false, GW, BF16, CS>(plan, a, stream);
    case 2: return launch_bag_sc<2, 0, false, GW, BF16, CS>(plan, a, stream);
    case 3: return launch_bag_sc<3, 0, false, GW, BF16, CS>(plan, a, stream);
    default: return launch_bag_sc<4, 0, false, GW, BF16, CS>(plan, a, stream);
  }
}

// Instantiation units (compiled in parallel), one per group size.
int launch_bag_256(const ibp_plan* plan, BagArgs& a, cudaStream_t stream);
int launch_bag_512(const ibp_plan* plan, BagArgs& a, cudaStream_t stream);
int launch_bag_1024(const ibp_plan* plan, BagArgs& a, cudaStream_t stream);
int launch_bag_bf16(const ibp_plan* plan, BagArgs& a, cudaStream_t stream);  // 512-word groups
// 1024-word groups, teams of 2 or 4 warps per bag (device slots, few bags)
int launch_bag_1024_split(const ibp_plan* plan, BagArgs& a, cudaStream_t stream, int cs);

}  // namespace ibp
