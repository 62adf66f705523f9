// ibp_gather_raw.cu - uncompressed row gather, the baseline that IBP's
// gather-decompress is measured against (the "ideal uncompressed transfer"
// of the rows a batch needs, « Résultats » of the paper summary).
//
// Enough independent loads stay in flight per SM that the copy is bound by
// the link (zero-copy host memory) or by HBM, not by latency.
#include <cuda_runtime.h>

#include "ibp_internal.cuh"

namespace ibp {

constexpr int kRawThreads = 256;
constexpr uint32_t kRawRows = 8;  // rows a warp has in flight

// A warp copies kRawRows rows at a time: lane q < kRawRows loads row q's id,
// then every lane loads one 16-byte (or 4-byte) chunk of each of the rows
// before storing any, so each lane keeps kRawRows independent loads in flight.
template <bool VEC>
__global__ void __launch_bounds__(kRawThreads) k_gather_raw(const uint32_t* __restrict__ rows,
                                                            uint64_t n_rows, uint32_t W,
                                                            const int64_t* __restrict__ ids,
                                                            uint64_t n_ids, uint32_t* __restrict__ out) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t gw = (static_cast<uint64_t>(blockIdx.x) * kRawThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = (static_cast<uint64_t>(gridDim.x) * kRawThreads) >> 5;
  const uint32_t cw = VEC ? 4u : 1u;
  const uint32_t per_row = W / cw;
  for (uint64_t i0 = gw * kRawRows; i0 < n_ids; i0 += nwarps * kRawRows) {
    int64_t id = -1;
    if (lane < kRawRows && i0 + lane < n_ids) id = ids[i0 + lane];
    const bool ok = id >= 0 && static_cast<uint64_t>(id) < n_rows;
    const unsigned long long src_l =
        reinterpret_cast<unsigned long long>(rows + static_cast<uint64_t>(ok ? id : 0) * W);
    const uint32_t okm = __ballot_sync(0xFFFFFFFFu, ok);
    for (uint32_t cb = 0; cb < per_row; cb += 32) {
      const uint32_t c = cb + lane;
      uint4 v[kRawRows];
#pragma unroll
      for (uint32_t u = 0; u < kRawRows; ++u) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(__shfl_sync(0xFFFFFFFFu, src_l, u));
        v[u] = make_uint4(0, 0, 0, 0);
        if (((okm >> u) & 1u) && c < per_row) {
          if (VEC)
            v[u] = *reinterpret_cast<const uint4*>(src + c * cw);
          else
            v[u].x = src[c];
        }
      }
#pragma unroll
      for (uint32_t u = 0; u < kRawRows; ++u) {
        if (i0 + u < n_ids && c < per_row) {
          uint32_t* dst = out + (i0 + u) * W + c * cw;
          if (VEC)
            *reinterpret_cast<uint4*>(dst) = v[u];
          else
            *dst = v[u].x;
        }
      }
    }
  }
}

int launch_gather_raw(const uint32_t* rows, uint64_t n_rows, uint32_t W, const int64_t* ids,
                      uint64_t n_ids, uint32_t* out, bool vec, int device, cudaStream_t stream) {
  const uint64_t warps_needed = (n_ids + kRawRows - 1) / kRawRows;
  const uint64_t need = (warps_needed * 32 + kRawThreads - 1) / kRawThreads;
  const uint64_t cap = 8ull * sm_count(device);
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  if (vec)
    k_gather_raw<true><<<grid, kRawThreads, 0, stream>>>(rows, n_rows, W, ids, n_ids, out);
  else
    k_gather_raw<false><<<grid, kRawThreads, 0, stream>>>(rows, n_rows, W, ids, n_ids, out);
  return check_launch("k_gather_raw");
}

}  // namespace ibp
