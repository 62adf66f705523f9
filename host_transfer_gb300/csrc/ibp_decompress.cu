// ibp_decompress.cu - warp-parallel gather-decompress of IBP slots.
//
// « Algorithme central », step 3 (Décompression): a warp of 32 threads
// cooperatively reads a contiguous compressed segment from CPU memory into a
// shared-memory workspace; warp primitives give each thread the starting bit
// offset of the word it owns; each thread rebuilds its word by putting the
// Bitval bits back at the Mask positions; asynchronous memory accesses
// overlap the fetch of later rows with the decoding of the current ones.
// « Intégration au système »: only the compressed prefix of a fixed-size slot
// is read, and a bitmask in GPU memory says which rows are compressed.
//
// GB300 design.  Each warp owns groups of G consecutive output rows (G = 32
// for 32-word rows down to 1 for rows of 1 K words and more) and runs a
// three-deep software pipeline over its groups:
//   ids of group j+3 -> registers            (plain loads)
//   headers of group j+2 -> shared memory     (cp.async, 16 B)
//   payload of group j+1 -> shared memory     (cp.async, 16 B, only the
//                                              compressed prefix)
//   decode of group j: one lane per word, 32 words per step
// so a warp keeps the payload of G rows plus the headers of G more rows in
// flight while it decodes.  cp.async reads mapped pinned host memory and HBM
// alike.  Offsets: when every word position has the same Mask the offset of
// lane i within a segment is 32 i - p * popc(H & lanemask_lt) (p = popcount
// of the Mask); otherwise a 5-step shuffle scan of the per-word field
// lengths.  Reinsertion: y = deposit(v) | (Bitval & Mask) with deposit done by
// up to four precomputed runs of kept bits, or by the five-step parallel-
// suffix expand for masks with more runs.
#include <cuda_runtime.h>

#include "ibp_internal.cuh"

namespace ibp {

constexpr int kDecWarpsMax = 8;
constexpr uint32_t kFull = 0xFFFFFFFFu;

template <bool UNIFORM, int R>
__device__ __forceinline__ uint32_t rebuild_word(const PlanView& pv, uint32_t v, uint32_t w) {
  if constexpr (UNIFORM) {
    if constexpr (R > 0)
      return deposit_runs<R>(v, pv.u_rmask, pv.u_rsh) | pv.u_bm;
    else
      return expand5(v, pv.u_mv, pv.u_keep) | pv.u_bm;
  } else {
    const uint32_t W = pv.W;
    if constexpr (R > 0) {
      uint32_t rm[R], rs[R];
      const uint32_t sh = __ldg(pv.rshift + w);
#pragma unroll
      for (int k = 0; k < R; ++k) {
        rm[k] = __ldg(pv.rmask + k * W + w);
        rs[k] = (sh >> (8 * k)) & 0xFFu;
      }
      return deposit_runs<R>(v, rm, rs) | __ldg(pv.bm + w);
    } else {
      uint32_t mv[5];
#pragma unroll
      for (int i = 0; i < 5; ++i) mv[i] = __ldg(pv.mv + i * W + w);
      return expand5(v, mv, ~__ldg(pv.mask + w)) | __ldg(pv.bm + w);
    }
  }
}

// Decode one compressed row whose stream (headers first) is in pb; write its
// W words to orow.  General form: any W, per-word tables or uniform scalars.
template <bool UNIFORM, int R>
__device__ __forceinline__ void decode_row(const PlanView& pv, const uint32_t* __restrict__ pb,
                                           uint32_t* __restrict__ orow, uint32_t lane,
                                           uint32_t lt) {
  const uint32_t W = pv.W, S = pv.S;
  uint32_t base = 32u * S;  // stream bit of segment s's first field
  for (uint32_t s = 0; s < S; ++s) {
    const uint32_t H = pb[s];
    const uint32_t w = 32u * s + lane;
    const uint32_t flag = (H >> lane) & 1u;
    uint32_t off, seg;
    if constexpr (UNIFORM) {
      const uint32_t nwords = min(32u, W - 32u * s);
      off = 32u * lane - pv.u_p * __popc(H & lt);
      seg = 32u * nwords - pv.u_p * __popc(H);
    } else {
      const uint32_t len = (w < W) ? (flag ? 32u - __ldg(pv.pcnt + w) : 32u) : 0u;
      uint32_t incl = len;
#pragma unroll
      for (uint32_t d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += t;
      }
      off = incl - len;
      seg = __shfl_sync(kFull, incl, 31);
    }
    if (w < W) {
      const uint32_t P = base + off;
      const uint32_t lo = pb[P >> 5];
      const uint32_t hi = pb[(P >> 5) + 1];
      const uint32_t v = __funnelshift_r(lo, hi, P & 31u);
      orow[w] = flag ? rebuild_word<UNIFORM, R>(pv, v, w) : v;
    }
    base += seg;
  }
}

// Uniform plan, W a multiple of 32: every segment is full and every word has
// the same Mask, so lane i's field in segment s starts at bit
//   32 S + 1024 s + 32 i - p * (matching words before it),
// read with one funnel shift over two shared-memory words.
template <int R>
__device__ __forceinline__ void decode_row_fast(const PlanView& pv, const uint32_t* __restrict__ pb,
                                                uint32_t* __restrict__ orow, uint32_t lane,
                                                uint32_t lt) {
  const uint32_t S = pv.S, p = pv.u_p;
  const uint32_t lanebit = 1u << lane;
  uint32_t base = 32u * S + 32u * lane;
  uint32_t* o = orow + lane;
#pragma unroll 4
  for (uint32_t s = 0; s < S; ++s) {
    const uint32_t H = pb[s];
    const uint32_t P = base - p * __popc(H & lt);
    const uint32_t* q = pb + (P >> 5);
    const uint32_t v = __funnelshift_r(q[0], q[1], P);
    uint32_t y;
    if constexpr (R > 0)
      y = deposit_runs<R>(v, pv.u_rmask, pv.u_rsh) | pv.u_bm;
    else
      y = expand5(v, pv.u_mv, pv.u_keep) | pv.u_bm;
    o[32u * s] = (H & lanebit) ? y : v;
    base += 1024u - p * __popc(H);
  }
}

template <bool UNIFORM, int R>
__global__ void __launch_bounds__(kDecWarpsMax * 32) k_decompress(const DecodeArgs a) {
  extern __shared__ __align__(16) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t nw_cta = blockDim.x >> 5;
  const uint32_t G = a.G, W = a.pv.W, S = a.pv.S, rowcap = a.rowcap;
  // Stage = G rows of rowcap words (a multiple of 32, so a row's 128-byte
  // global lines land on 128-byte shared-memory lines) plus 32 words for the
  // decoder's one-word read past the last row.
  const uint32_t stage_words = G * rowcap + 32u;
  uint32_t* const stages = smem + warp * 3u * stage_words;  // [3] stages
  const uint32_t lt = lanemask_lt();
  const bool fast = UNIFORM && (W & 31u) == 0;

  const uint64_t n_groups = (a.n_out + G - 1) / G;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * nw_cta + warp;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * nw_cta;
  if (gw >= n_groups) return;  // warp-uniform; only warp-level syncs below
  const uint64_t J = (n_groups - gw + nwarps - 1) / nwarps;
  // Lane q < G of group j owns output row row_first + j * row_step + q.
  const uint64_t row_first = gw * G;
  const uint64_t row_step = nwarps * G;
  const uint32_t pre = a.pre;
  const bool reuse = (a.pv.hints & IBP_HINT_ROW_REUSE) != 0;

  auto present = [&](uint64_t j) -> bool {
    return j < J && lane < G && row_first + j * row_step + lane < a.n_out;
  };
  auto in_table = [&](int64_t id) -> bool {
    return id >= 0 && static_cast<uint64_t>(id) < a.n_rows;
  };
  auto load_id = [&](uint64_t j) -> int64_t {
    if (!present(j)) return -1;
    const uint64_t i = row_first + j * row_step + lane;
    return a.ids ? a.ids[i] : static_cast<int64_t>(a.first + i);
  };
  // Words [0, pre) of every row of group j (its headers and the part of the
  // stream that every compressed row has), and the row's bitmask word.
  auto issue_prefix = [&](uint64_t j, uint32_t* sb, int64_t id, uint32_t& bmw) {
    const bool ok = present(j) && in_table(id);
    if (ok) bmw = ld_u32(a.bitmask + (static_cast<uint64_t>(id) >> 5));
    if (j >= J) return;
    const unsigned long long src_l =
        reinterpret_cast<unsigned long long>(a.slots + static_cast<uint64_t>(ok ? id : 0) * W);
    for (uint32_t m = __ballot_sync(kFull, ok); m; m &= m - 1) {
      const uint32_t q = __ffs(m) - 1;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(__shfl_sync(kFull, src_l, q));
      uint32_t* dst = sb + q * rowcap;
      if (a.vec) {
        for (uint32_t c = lane; c < (pre >> 2); c += 32) cp_row16(reuse, dst + 4u * c, src + 4u * c);
      } else {
        for (uint32_t k = lane; k < pre; k += 32) cp_async4(dst + k, src + k);
      }
    }
  };

  // Row kind and words to read, from the headers of group j (lane q).
  auto row_info = [&](uint64_t j, const uint32_t* sb, int64_t id, uint32_t bmw, uint32_t& kind,
                      uint32_t& nt) {
    kind = kNone;
    nt = 0;
    if (!present(j)) return;
    if (!in_table(id)) {
      kind = kBadRange;
      return;
    }
    if (!((bmw >> (static_cast<uint64_t>(id) & 31u)) & 1u)) {
      kind = kRaw;
      nt = W;
      return;
    }
    const uint32_t* hb = sb + lane * rowcap;
    uint32_t drop = 0;  // sum of popcount(Mask) over the matching words
    // Lane q starts at header q mod S: rows are rowcap words apart (a
    // multiple of 32), so reading header s on every lane would hit one bank.
    uint32_t s = lane % S;
    for (uint32_t t = 0; t < S; ++t, s = (s + 1 == S) ? 0 : s + 1) {
      const uint32_t H = hb[s];
      if (s == S - 1) {
        const uint32_t nb = W - 32u * s;
        if (nb < 32u && (H >> nb)) {
          kind = kCorrupt;
          return;
        }
      }
      if constexpr (UNIFORM) {
        drop += __popc(H);
      } else {
#pragma unroll
        for (int k = 0; k < kPlanes; ++k) drop += __popc(H & __ldg(a.pv.planes + s * kPlanes + k)) << k;
      }
    }
    if constexpr (UNIFORM) drop *= a.pv.u_p;
    const uint32_t bits = 32u * (S + W) - drop;
    const uint32_t Lw = (bits + 31u) >> 5;
    if (Lw >= W) {
      kind = kCorrupt;
      return;
    }
    kind = kComp;
    nt = Lw;
  };

  // The rest of each row of group j: words [pre, Lw) of a compressed row,
  // [pre, W) of a raw one.  Usually nothing for dense data.
  auto issue_rest = [&](uint64_t j, uint32_t* sb, int64_t id, uint32_t kind, uint32_t nt) {
    if (j >= J) return;
    const bool need = (kind == kRaw || kind == kComp) && nt > pre;
    const uint32_t needmask = __ballot_sync(kFull, need);
    if (!needmask) return;
    const unsigned long long src_l =
        reinterpret_cast<unsigned long long>(a.slots + static_cast<uint64_t>(need ? id : 0) * W);
    for (uint32_t m = needmask; m; m &= m - 1) {
      const uint32_t q = __ffs(m) - 1;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(__shfl_sync(kFull, src_l, q));
      const uint32_t ntq = __shfl_sync(kFull, nt, q);
      uint32_t* dst = sb + q * rowcap;
      if (a.vec) {
        for (uint32_t c = (pre >> 2) + lane; c < ((ntq + 3u) >> 2); c += 32) cp_row16(reuse, dst + 4u * c, src + 4u * c);
      } else {
        for (uint32_t k = pre + lane; k < ntq; k += 32) cp_async4(dst + k, src + k);
      }
    }
  };

  auto decode_group = [&](uint64_t j, const uint32_t* sb, uint32_t kind) {
    uint32_t* const obase = a.out + (row_first + j * row_step) * W;
    for (uint32_t m = __ballot_sync(kFull, kind == kComp); m; m &= m - 1) {
      const uint32_t q = __ffs(m) - 1;
      if (fast) {
        decode_row_fast<R>(a.pv, sb + q * rowcap, obase + static_cast<uint64_t>(q) * W, lane, lt);
      } else {
        decode_row<UNIFORM, R>(a.pv, sb + q * rowcap, obase + static_cast<uint64_t>(q) * W, lane, lt);
      }
    }
    for (uint32_t m = __ballot_sync(kFull, kind == kRaw); m; m &= m - 1) {
      const uint32_t q = __ffs(m) - 1;
      const uint32_t* pb = sb + q * rowcap;
      uint32_t* orow = obase + static_cast<uint64_t>(q) * W;
      if (a.vec) {
        for (uint32_t c = lane; c < (W >> 2); c += 32)
          reinterpret_cast<uint4*>(orow)[c] = reinterpret_cast<const uint4*>(pb)[c];
      } else {
        for (uint32_t k = lane; k < W; k += 32) orow[k] = pb[k];
      }
    }
    const bool bad = kind == kBadRange || kind == kCorrupt;
    if (bad) record_status(a.pv.status, kind == kBadRange ? IBP_ERANGE : IBP_ECORRUPT);
    for (uint32_t m = __ballot_sync(kFull, bad); m; m &= m - 1) {
      const uint32_t q = __ffs(m) - 1;
      uint32_t* orow = obase + static_cast<uint64_t>(q) * W;
      for (uint32_t k = lane; k < W; k += 32) orow[k] = 0u;
    }
  };

  // Pipeline, per iteration j: ids of group j+3 (registers), prefix of group
  // j+2 (cp.async), kinds of group j+1 from its landed headers and the rest of
  // its rows (cp.async), decode of group j.  Group j lives in stage j % 3.
  // Commit order per iteration: prefix(j+2), rest(j+1); so before the rest of
  // j+1 is issued, prefix(j+1) is complete once at most two groups (rest(j),
  // prefix(j+2)) are pending, and before the decode of j, rest(j) is complete
  // once at most two (prefix(j+2), rest(j+1)) are.
  int64_t id0 = load_id(0), id1 = load_id(1), id2 = load_id(2);
  uint32_t* st0 = stages;                    // stage of group j
  uint32_t* st1 = stages + stage_words;      // stage of group j + 1
  uint32_t* st2 = stages + 2 * stage_words;  // stage of group j + 2
  uint32_t bm0 = 0, bm1 = 0;
  issue_prefix(0, st0, id0, bm0);
  cp_commit();
  issue_prefix(1, st1, id1, bm1);
  cp_commit();
  cp_wait<1>();
  __syncwarp();
  uint32_t kind0, nt0;
  row_info(0, st0, id0, bm0, kind0, nt0);
  issue_rest(0, st0, id0, kind0, nt0);
  cp_commit();

  for (uint64_t j = 0; j < J; ++j) {
    const int64_t id3 = load_id(j + 3);
    uint32_t bm2 = 0;
    issue_prefix(j + 2, st2, id2, bm2);
    cp_commit();
    cp_wait<2>();
    __syncwarp();
    uint32_t kind1, nt1;
    row_info(j + 1, st1, id1, bm1, kind1, nt1);
    issue_rest(j + 1, st1, id1, kind1, nt1);
    cp_commit();
    cp_wait<2>();
    __syncwarp();
    decode_group(j, st0, kind0);
    __syncwarp();
    id1 = id2;
    id2 = id3;
    bm1 = bm2;
    kind0 = kind1;
    uint32_t* const t = st0;
    st0 = st1;
    st1 = st2;
    st2 = t;
  }
  cp_wait<0>();
}

template <bool U, int R>
static int launch_t(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  const size_t per_warp = 4ull * 3ull * (a.G * a.rowcap + 32ull);
  const size_t budget = 220ull * 1024;
  size_t warps = budget / per_warp;
  if (warps > static_cast<size_t>(kDecWarpsMax)) warps = kDecWarpsMax;
  if (warps < 1) return IBP_EINVAL;
  const size_t smem = warps * per_warp;
  auto kern = k_decompress<U, R>;
  // One-time set-up per device: the shared-memory opt-in and the occupancy
  // for this launch shape (smem depends only on the row width).
  static std::atomic<int> occ_cache[64];  // per device, any host thread
  static size_t occ_smem[64] = {0};
  const int dev = plan->device;
  if (dev < 0 || dev >= 64) return IBP_EINVAL;
  int occ = occ_cache[dev].load(std::memory_order_relaxed);
  if (occ == 0 || occ_smem[dev] != smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, static_cast<int>(warps * 32), smem);
    if (e != cudaSuccess || occ < 1) {
      set_cuda_error(e, "set-up of k_decompress");
      cudaGetLastError();
      return IBP_ECUDA;
    }
    occ_cache[dev].store(occ, std::memory_order_relaxed);
    occ_smem[dev] = smem;
  }
  const uint64_t groups = (a.n_out + a.G - 1) / a.G;
  const uint64_t need = (groups + warps - 1) / warps;
  const uint64_t cap = static_cast<uint64_t>(occ) * sm_count(dev);
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  kern<<<grid, static_cast<unsigned>(warps * 32), smem, stream>>>(a);
  return check_launch("k_decompress");
}

int launch_decompress(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  if (fast_decompress_applies(plan, a)) return launch_decompress_fast(plan, a, stream);
  const uint32_t runs = plan->max_runs;
  const int R = runs <= static_cast<uint32_t>(kMaxRuns) ? (runs == 0 ? 1 : static_cast<int>(runs)) : 0;
  if (plan->uniform) {
    switch (R) {
      case 1: return launch_t<true, 1>(plan, a, stream);
      case 2: return launch_t<true, 2>(plan, a, stream);
      case 3: return launch_t<true, 3>(plan, a, stream);
      case 4: return launch_t<true, 4>(plan, a, stream);
      default: return launch_t<true, 0>(plan, a, stream);
    }
  }
  switch (R) {
    case 1: return launch_t<false, 1>(plan, a, stream);
    case 2: return launch_t<false, 2>(plan, a, stream);
    case 3: return launch_t<false, 3>(plan, a, stream);
    case 4: return launch_t<false, 4>(plan, a, stream);
    default: return launch_t<false, 0>(plan, a, stream);
  }
}

}  // namespace ibp
