// ibp_gather_raw.cu - uncompressed row gather, the baseline that IBP's
// gather-decompress is measured against (the "ideal uncompressed transfer"
// of the rows a batch needs, « Résultats » of the paper summary).
//
// Each thread copies 16-byte chunks of the flat (row, chunk) space, four
// independent chunks in flight per thread, so the copy is bound by the link
// (zero-copy host memory) or by HBM, not by latency.
#include <cuda_runtime.h>

#include "ibp_internal.cuh"

namespace ibp {

constexpr int kRawThreads = 256;
constexpr int kRawUnroll = 4;

template <bool VEC>
__global__ void __launch_bounds__(kRawThreads) k_gather_raw(const uint32_t* __restrict__ rows,
                                                            uint64_t n_rows, uint32_t W,
                                                            const int64_t* __restrict__ ids,
                                                            uint64_t n_ids, uint32_t* __restrict__ out) {
  const uint32_t cw = VEC ? 4u : 1u;          // words per chunk
  const uint32_t per_row = W / cw;             // chunks per row (W % 4 == 0 when VEC)
  const uint64_t total = n_ids * per_row;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kRawThreads;
  for (uint64_t c0 = static_cast<uint64_t>(blockIdx.x) * kRawThreads + threadIdx.x; c0 < total;
       c0 += stride * kRawUnroll) {
    uint4 v[kRawUnroll];
    uint64_t dsto[kRawUnroll];
#pragma unroll
    for (int u = 0; u < kRawUnroll; ++u) {
      const uint64_t c = c0 + u * stride;
      dsto[u] = ~0ull;
      v[u] = make_uint4(0, 0, 0, 0);
      if (c < total) {
        const uint64_t i = c / per_row;
        const uint32_t k = static_cast<uint32_t>(c - i * per_row);
        const int64_t id = __ldg(ids + i);
        dsto[u] = i * W + k * cw;
        if (id >= 0 && static_cast<uint64_t>(id) < n_rows) {
          const uint32_t* src = rows + static_cast<uint64_t>(id) * W + k * cw;
          if (VEC)
            v[u] = *reinterpret_cast<const uint4*>(src);
          else
            v[u].x = *src;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kRawUnroll; ++u) {
      if (dsto[u] == ~0ull) continue;
      if (VEC)
        *reinterpret_cast<uint4*>(out + dsto[u]) = v[u];
      else
        out[dsto[u]] = v[u].x;
    }
  }
}

int launch_gather_raw(const uint32_t* rows, uint64_t n_rows, uint32_t W, const int64_t* ids,
                      uint64_t n_ids, uint32_t* out, bool vec, int device, cudaStream_t stream) {
  const uint64_t chunks = n_ids * (vec ? W / 4 : W);
  const uint64_t need = (chunks + kRawThreads * kRawUnroll - 1) / (kRawThreads * kRawUnroll);
  const uint64_t cap = 8ull * sm_count(device);
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  if (vec)
    k_gather_raw<true><<<grid, kRawThreads, 0, stream>>>(rows, n_rows, W, ids, n_ids, out);
  else
    k_gather_raw<false><<<grid, kRawThreads, 0, stream>>>(rows, n_rows, W, ids, n_ids, out);
  return check_launch("k_gather_raw");
}

}  // namespace ibp
