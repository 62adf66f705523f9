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
// The fetch and decode are those of k_decompress_fast (same plan shapes, same
// three-stage cp.async pipeline of prefix, then rest, per group of G rows).
// What differs is the unit of work: warp gw owns bags gw, gw + nwarps, ...; a
// cursor cuts each bag into groups of at most G consecutive ids (a group
// never spans two bags; an empty or invalid bag is one group of no rows), and
// the decode of a group adds its rows, in order, into the lanes'
// accumulators (word lane + 32 s in acc[s]); the group that ends a bag
// writes the bag's output row.
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
  using F = FastShape<SC, GW>;
  using T = TabShape<SC, R, NPL, TAB>;
  constexpr uint32_t W = F::W, G = F::G, STAGE = F::STAGE, CB = F::CB;
  constexpr uint32_t EW = TabEntry<R>::EW;
  constexpr int D = kFastStages;
  extern __shared__ __align__(128) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t nw_cta = blockDim.x >> 5;
  uint32_t* const tab = smem;
  uint32_t* const epl = smem + T::ENT;
  uint32_t* const stages = smem + T::WORDS + warp * static_cast<uint32_t>(D) * STAGE;
  const uint32_t lt = lanemask_lt();
  const uint32_t lanebit = 1u << lane;

  const PlanView pv = ba.d.pv;
  const uint32_t* const slots = ba.d.slots;
  const uint32_t* const bitmask = ba.d.bitmask;
  const int64_t* const ids = ba.d.ids;
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
  const uint32_t pre = ba.d.pre;  // multiple of 4, <= W
  const uint32_t pre_ch = pre >> 2;
  const uint32_t n_rows32 = static_cast<uint32_t>(ba.d.n_rows);  // < 2^31 (checked by the launcher)
  const uint64_t n_bags = ba.n_bags;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * nw_cta + warp;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * nw_cta;
  // Programmatic dependent launch, as in k_decompress_fast: the next kernel
  // may start as this grid drains; wait for the previous grid before
  // touching per-call data.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr uint32_t SPW = SC / CS;  // segments this warp pools
  const uint64_t team = gw / CS, nteams = nwarps / CS;  // warps per CTA are a multiple of CS
  const uint32_t s_lo = CS == 1 ? 0u : static_cast<uint32_t>(gw % CS) * SPW;
  if (team >= n_bags) return;  // warp-uniform; only warp-level syncs below
  asm volatile("griddepcontrol.wait;" ::: "memory");

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
  constexpr int32_t kNoRow = -1, kBadId = -2;
  auto load_id = [&](const Grp& g) -> int32_t {
    if (g.bag >= n_bags || lane >= g.n) return kNoRow;
    const int64_t id = ids[g.pos + lane];
    return (id >= 0 && static_cast<uint64_t>(id) < n_rows32) ? static_cast<int32_t>(id) : kBadId;
  };

  auto issue_prefix = [&](uint32_t* sb, int32_t id, uint32_t& bmw) {
    if (id >= 0) bmw = ld_u32(bitmask + (static_cast<uint32_t>(id) >> 5));
#pragma unroll
    for (uint32_t q = 0; q < G; ++q) {
      const int32_t idq = __shfl_sync(kAll, id, q);
      if (idq >= 0) {
        const uint32_t* src = slots + static_cast<uint64_t>(idq) * W;
        uint32_t* dst = sb + q * W;
#pragma unroll
        for (uint32_t b = 0; b < CB; ++b) {
          const uint32_t c = lane + 32u * b;
          if (c < pre_ch) cp_row16(reuse, dst + 4u * c, src + 4u * c);
        }
      }
    }
  };

  // Bits saved by the matching words of lane q's row (summed over its
  // headers), as in k_decompress_fast: rows of 8 or more segments take one
  // header per lane and a warp reduction per row (warp-collective), shorter
  // rows a walk by lane q.
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
      const uint32_t qo = SC >= 32 ? 0u : lane / SC;
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

  // Warp-collective (saved_bits).
  auto row_info = [&](const uint32_t* sb, int32_t id, uint32_t bmw, uint32_t& kind, uint32_t& nt) {
    const uint32_t saved = saved_bits(sb);
    kind = kNone;
    nt = 0;
    if (id == kNoRow) return;
    if (id == kBadId) {
      kind = kBadRange;
      return;
    }
    if (!((bmw >> (static_cast<uint32_t>(id) & 31u)) & 1u)) {
      kind = kRaw;
      nt = W;
      return;
    }
    const uint32_t Lw = (32u * (SC + W) - saved + 31u) >> 5;
    if (Lw >= W) {
      kind = kCorrupt;
      return;
    }
    kind = kComp;
    nt = Lw;
  };

  auto issue_rest = [&](uint32_t* sb, int32_t id, uint32_t kind, uint32_t nt) {
    const bool need = (kind == kRaw || kind == kComp) && nt > pre;
    for (uint32_t mk = __ballot_sync(kAll, need); mk; mk &= mk - 1) {
      const uint32_t q = __ffs(mk) - 1;
      const uint32_t ntq = __shfl_sync(kAll, nt, q);
      const uint32_t* src = slots + static_cast<uint64_t>(__shfl_sync(kAll, id, q)) * W;
      uint32_t* dst = sb + q * W;
      for (uint32_t c = pre_ch + lane; c < ((ntq + 3u) >> 2); c += 32) cp_row16(reuse, dst + 4u * c, src + 4u * c);
    }
  };

  constexpr uint32_t NA = BF16 ? 2 * SPW : SPW;  // accumulators per lane
  float acc[NA];
#pragma unroll
  for (uint32_t s = 0; s < NA; ++s) acc[s] = 0.0f;
  uint64_t cnt = 0;  // ids of the current bag seen so far
  // add decoded word w (word lane + 32 (s_lo + s) of a row)
  auto add_word = [&](uint32_t s, uint32_t w) {
    if constexpr (BF16) {
      acc[2 * s] = __fadd_rn(acc[2 * s], __uint_as_float(w << 16));
      acc[2 * s + 1] = __fadd_rn(acc[2 * s + 1], __uint_as_float(w & 0xFFFF0000u));
    } else {
      acc[s] = __fadd_rn(acc[s], __uint_as_float(w));
    }
  };

  auto add_row = [&](const uint32_t* pb) {
    uint32_t base = 32u * SC + 32u * lane;
    // segment s of the row, pooled into accumulator j
    auto seg = [&](uint32_t H, uint32_t s, uint32_t j) {
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
      add_word(j, (H & lanebit) ? y : v);
      base += step;
    };
    if constexpr (CS > 1) {
      // step over the fields of the segments before this warp's slice
      for (uint32_t s = 0; s < s_lo; ++s) {
        const uint32_t H = pb[s];
        uint32_t step = 1024u - p * __popc(H);
        if constexpr (TAB && NPL > 0) {
          uint32_t e_all = 0;
#pragma unroll
          for (int k = 0; k < NPL; ++k) e_all += __popc(H & epl[s * NPL + k]) << k;
          step -= pscale * e_all;
        }
        base += step;
      }
#pragma unroll
      for (uint32_t j = 0; j < SPW; ++j) seg(pb[s_lo + j], s_lo + j, j);
    } else if constexpr (SC >= 4) {
#pragma unroll
      for (uint32_t s = 0; s < SC; s += 4) {
        const uint4 h = *reinterpret_cast<const uint4*>(pb + s);
        seg(h.x, s, s);
        seg(h.y, s + 1, s + 1);
        seg(h.z, s + 2, s + 2);
        seg(h.w, s + 3, s + 3);
      }
    } else {
#pragma unroll
      for (uint32_t s = 0; s < SC; ++s) seg(pb[s], s, s);
    }
  };

  // Add group g's rows in order; the group that ends a bag writes it out.
  auto consume = [&](const Grp& g, const uint32_t* sb, uint32_t kind) {
    const uint32_t comp = __ballot_sync(kAll, kind == kComp);
    const uint32_t raw = __ballot_sync(kAll, kind == kRaw);
    const bool bad = kind == kBadRange || kind == kCorrupt;
    if (bad) record_status(pv.status, kind == kBadRange ? IBP_ERANGE : IBP_ECORRUPT);
    constexpr uint32_t kGroupBits = G >= 32 ? kAll : (1u << G) - 1u;
    if (!TAB && comp == kGroupBits) {
      // uniform plan, every row compressed: straight-line code, so the rows'
      // decode work overlaps (the additions still follow the row order)
#pragma unroll
      for (uint32_t q = 0; q < G; ++q) add_row(sb + q * W);
    } else {
#pragma unroll
      for (uint32_t q = 0; q < G; ++q) {
        if ((comp >> q) & 1u) {
          add_row(sb + q * W);
        } else if ((raw >> q) & 1u) {
#pragma unroll
          for (uint32_t j = 0; j < SPW; ++j) add_word(j, sb[q * W + 32u * (s_lo + j) + lane]);
        }
      }
    }
    cnt += g.n;
    if (g.last) {
      if (g.bad && lane == 0) record_status(pv.status, IBP_ERANGE);
      const float c = static_cast<float>(cnt);
      const bool div = ba.mean && cnt;
      if constexpr (BF16) {
        float2* const o = reinterpret_cast<float2*>(ba.out + g.bag * (2 * W)) + lane + 32u * s_lo;
#pragma unroll
        for (uint32_t j = 0; j < SPW; ++j) {
          const float lo = acc[2 * j], hi = acc[2 * j + 1];
          o[32u * j] = div ? make_float2(__fdiv_rn(lo, c), __fdiv_rn(hi, c)) : make_float2(lo, hi);
        }
      } else {
        float* const o = ba.out + g.bag * W + lane + 32u * s_lo;
#pragma unroll
        for (uint32_t j = 0; j < SPW; ++j) o[32u * j] = div ? __fdiv_rn(acc[j], c) : acc[j];
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
    issue_prefix(st[i], idr[i], bmr[i]);
    cp_commit();
    if (i < D - 2) cp_commit();
  }
  cp_wait<2 * D - 4>();
  __syncwarp();
  uint32_t kind0, nt0;
  row_info(st[0], idr[0], bmr[0], kind0, nt0);
  issue_rest(st[0], idr[0], kind0, nt0);
  cp_commit();

  while (gr[0].bag < n_bags) {
    gr[D] = next_group();
    idr[D] = load_id(gr[D]);
    issue_prefix(st[D - 1], idr[D - 1], bmr[D - 1]);
    cp_commit();
    cp_wait<2 * D - 4>();
    __syncwarp();
    uint32_t kind1, nt1;
    row_info(st[1], idr[1], bmr[1], kind1, nt1);
    issue_rest(st[1], idr[1], kind1, nt1);
    cp_commit();
    cp_wait<2>();
    __syncwarp();
    consume(gr[0], st[0], kind0);
    __syncwarp();
    kind0 = kind1;
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
  static int occ_cache[64] = {0};
  const int dev = plan->device;
  if (dev < 0 || dev >= 64) return IBP_EINVAL;
  int occ = occ_cache[dev];
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, static_cast<int>(warps * 32), smem);
    if (e != cudaSuccess || occ < 1) {
      set_cuda_error(e, "set-up of k_bag");
      cudaGetLastError();
      return IBP_ECUDA;
    }
    occ_cache[dev] = occ;
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
  if (!plan->uniform)
    return plan->max_runs <= 2 ? launch_bag_table<2, GW, BF16, CS>(plan, a, stream)
                               : launch_bag_table<4, GW, BF16, CS>(plan, a, stream);
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
