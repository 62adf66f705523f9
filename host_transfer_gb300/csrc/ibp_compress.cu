// ibp_compress.cu - IBP compression of rows into fixed-size in-place slots.
//
// « Algorithme central », step 2 (Compression): each chunk (here one 32-bit
// word) is tested against Bitval at the invariant positions; on a match the
// invariant bits are removed and the remaining ones shifted together; a
// participation bit says whether the chunk was compressed; the GPU does this
// directly on CPU memory through zero-copy mappings.  « Intégration au
// système »: the result goes back into the row's fixed-size buffer and a
// bitmask in GPU memory records which rows are compressed.
//
// GB300 design: one warp per row, 32 words per step (one per lane).  The
// participation header of a segment is the warp ballot of the match flags;
// the bit offset of each lane's field is 32 i - p * popc(H & lanemask_lt)
// for a uniform Mask, else a shuffle scan; fields are OR-ed into a zeroed
// shared-memory stream with shared atomics (a field spans at most two
// words).  A warp handles 32 consecutive rows so that it writes one whole
// bitmask word; the next row is prefetched with cp.async while the current
// one is packed.
#include <cuda_runtime.h>

#include "ibp_internal.cuh"

namespace ibp {

constexpr int kCompWarpsMax = 8;
constexpr uint32_t kFullMask = 0xFFFFFFFFu;

template <bool UNIFORM, int R>
__device__ __forceinline__ void word_params(const PlanView& pv, uint32_t w, uint32_t& m,
                                            uint32_t& bmv, uint32_t& p) {
  if constexpr (UNIFORM) {
    m = pv.u_mask;
    bmv = pv.u_bm;
    p = pv.u_p;
  } else {
    m = __ldg(pv.mask + w);
    bmv = __ldg(pv.bm + w);
    p = __ldg(pv.pcnt + w);
  }
}

template <bool UNIFORM, int R>
__device__ __forceinline__ uint32_t strip_word(const PlanView& pv, uint32_t x, uint32_t w,
                                               uint32_t m) {
  if constexpr (UNIFORM) {
    if constexpr (R > 0)
      return extract_runs<R>(x, pv.u_rmask, pv.u_rsh);
    else
      return compress5(x, pv.u_mv, pv.u_keep);
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
      return extract_runs<R>(x, rm, rs);
    } else {
      uint32_t mv[5];
#pragma unroll
      for (int i = 0; i < 5; ++i) mv[i] = __ldg(pv.mv + i * W + w);
      return compress5(x, mv, ~m);
    }
  }
}

template <bool UNIFORM, int R>
__global__ void __launch_bounds__(kCompWarpsMax * 32, 2) k_compress(const CompressArgs a) {
  extern __shared__ __align__(16) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t nw_cta = blockDim.x >> 5;
  const uint32_t W = a.pv.W, S = a.pv.S, rowcap = a.rowcap;
  uint32_t* const xbuf = smem + warp * 3u * rowcap;  // [2][rowcap] rows
  uint32_t* const sbuf = xbuf + 2u * rowcap;         // [rowcap] stream
  const uint32_t lt = lanemask_lt();

  const uint64_t nblk = (a.n_rows + 31) / 32;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * nw_cta;

  auto load_row = [&](uint64_t row, uint32_t* dst) {
    const uint32_t* src = a.rows + row * W;
    if (a.vec) {
      for (uint32_t c = lane; c < (W >> 2); c += 32) cp_async16(dst + 4u * c, src + 4u * c);
    } else {
      for (uint32_t k = lane; k < W; k += 32) cp_async4(dst + k, src + k);
    }
  };

  for (uint64_t rb = static_cast<uint64_t>(blockIdx.x) * nw_cta + warp; rb < nblk; rb += nwarps) {
    const uint64_t r0 = rb * 32;
    const uint64_t left = a.n_rows - r0;
    const uint32_t nr = left < 32 ? static_cast<uint32_t>(left) : 32u;
    uint32_t bits = 0;
    unsigned long long stored = 0;
    load_row(r0, xbuf);
    cp_commit();
    for (uint32_t r = 0; r < nr; ++r) {
      if (r + 1 < nr) load_row(r0 + r + 1, xbuf + ((r + 1) & 1u) * rowcap);
      cp_commit();
      for (uint32_t k = lane; k < rowcap; k += 32) sbuf[k] = 0u;
      cp_wait<1>();
      __syncwarp();
      const uint32_t* x = xbuf + (r & 1u) * rowcap;
      uint32_t base = 32u * S;
      for (uint32_t s = 0; s < S; ++s) {
        const uint32_t w = 32u * s + lane;
        const bool valid = w < W;
        uint32_t m = 0, bmv = 0, p = 0;
        if (valid) word_params<UNIFORM, R>(a.pv, w, m, bmv, p);
        const uint32_t xv = valid ? x[w] : 0u;
        const bool flag = valid && ((xv ^ bmv) & m) == 0u;
        const uint32_t H = __ballot_sync(kFullMask, flag);
        const uint32_t len = valid ? (flag ? 32u - p : 32u) : 0u;
        uint32_t off, seg;
        if constexpr (UNIFORM) {
          const uint32_t nwords = min(32u, W - 32u * s);
          off = 32u * lane - a.pv.u_p * __popc(H & lt);
          seg = 32u * nwords - a.pv.u_p * __popc(H);
        } else {
          uint32_t incl = len;
#pragma unroll
          for (uint32_t d = 1; d < 32; d <<= 1) {
            const uint32_t t = __shfl_up_sync(kFullMask, incl, d);
            if (lane >= d) incl += t;
          }
          off = incl - len;
          seg = __shfl_sync(kFullMask, incl, 31);
        }
        if (len) {
          const uint32_t v = flag ? strip_word<UNIFORM, R>(a.pv, xv, w, m) : xv;
          const uint32_t P = base + off;
          const uint32_t k0 = P >> 5, sh = P & 31u;
          // only streams shorter than the row are kept: later words are moot
          if (k0 < W) atomicOr(&sbuf[k0], v << sh);
          if (sh + len > 32u && k0 + 1 < W) atomicOr(&sbuf[k0 + 1], v >> (32u - sh));
        }
        if (lane == 0) sbuf[s] = H;
        base += seg;
      }
      __syncwarp();
      const uint32_t Lw = (base + 31u) >> 5;
      uint32_t* dst = a.slots + (r0 + r) * W;
      if (Lw < W) {
        if (a.vec) {
          for (uint32_t c = lane; c < (W >> 2); c += 32) {
            uint4 q = reinterpret_cast<const uint4*>(sbuf)[c];
            const uint32_t k = 4u * c;
            if (k + 0 >= Lw) q.x = 0u;
            if (k + 1 >= Lw) q.y = 0u;
            if (k + 2 >= Lw) q.z = 0u;
            if (k + 3 >= Lw) q.w = 0u;
            reinterpret_cast<uint4*>(dst)[c] = q;
          }
        } else {
          for (uint32_t k = lane; k < W; k += 32) dst[k] = k < Lw ? sbuf[k] : 0u;
        }
        bits |= 1u << r;
        stored += Lw;
      } else {
        if (a.vec) {
          for (uint32_t c = lane; c < (W >> 2); c += 32)
            reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(x)[c];
        } else {
          for (uint32_t k = lane; k < W; k += 32) dst[k] = x[k];
        }
        stored += W;
      }
      __syncwarp();
    }
    if (lane == 0) {
      a.bitmask[rb] = bits;
      if (a.stored) atomicAdd(a.stored, stored);
    }
  }
  cp_wait<0>();
}

template <bool U, int R>
static int launch_t(const ibp_plan* plan, CompressArgs& a, cudaStream_t stream) {
  const size_t per_warp = 4ull * 3ull * a.rowcap;
  size_t warps = (220ull * 1024) / per_warp;
  if (warps > static_cast<size_t>(kCompWarpsMax)) warps = kCompWarpsMax;
  if (warps < 1) return IBP_EINVAL;
  const size_t smem = warps * per_warp;
  auto kern = k_compress<U, R>;
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
      set_cuda_error(e, "set-up of k_compress");
      cudaGetLastError();
      return IBP_ECUDA;
    }
    occ_cache[dev].store(occ, std::memory_order_relaxed);
    occ_smem[dev] = smem;
  }
  const uint64_t blocks32 = (a.n_rows + 31) / 32;
  const uint64_t need = (blocks32 + warps - 1) / warps;
  const uint64_t cap = static_cast<uint64_t>(occ) * sm_count(dev);
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  kern<<<grid, static_cast<unsigned>(warps * 32), smem, stream>>>(a);
  return check_launch("k_compress");
}

int launch_compress(const ibp_plan* plan, CompressArgs& a, cudaStream_t stream) {
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
