// ibp_lengths.cu - words a reader fetches for each requested row.
//
// « Intégration au système »: in-place compression allocates fixed-size
// buffers but reads only the compressed part; this kernel reports that part's
// length per row (Lw for a compressed row, W for a raw one), from the row's
// participation headers.  Used to size transfers and packed caches and to
// count the bytes a gather actually moves.
#include <cuda_runtime.h>

#include "ibp_internal.cuh"

namespace ibp {

__global__ void k_row_lengths(const PlanView pv, const uint32_t* __restrict__ slots, uint64_t n_rows,
                              const uint32_t* __restrict__ bitmask, const int64_t* __restrict__ ids,
                              uint64_t n_ids, uint32_t* __restrict__ lengths) {
  const uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_ids) return;
  const int64_t id = ids[i];
  const uint32_t W = pv.W, S = pv.S;
  if (id < 0 || static_cast<uint64_t>(id) >= n_rows) {
    lengths[i] = 0;
    record_status(pv.status, IBP_ERANGE);
    return;
  }
  if (!((ld_u32(bitmask + (static_cast<uint64_t>(id) >> 5)) >> (id & 31)) & 1u)) {
    lengths[i] = W;
    return;
  }
  const uint32_t* h = slots + static_cast<uint64_t>(id) * W;
  uint32_t drop = 0;
  for (uint32_t s = 0; s < S; ++s) {
    uint32_t H = ld_u32(h + s);
    if (s == S - 1 && W - 32u * s < 32u) H &= (1u << (W - 32u * s)) - 1u;
    for (int k = 0; k < kPlanes; ++k) drop += __popc(H & __ldg(pv.planes + s * kPlanes + k)) << k;
  }
  const uint32_t Lw = (32u * (S + W) - drop + 31u) >> 5;
  lengths[i] = Lw < W ? Lw : W;
}

int launch_row_lengths(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                       const uint32_t* bitmask, const int64_t* ids, uint64_t n_ids,
                       uint32_t* lengths, cudaStream_t stream) {
  const unsigned threads = 256;
  const uint64_t blocks = (n_ids + threads - 1) / threads;
  k_row_lengths<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(plan->view, slots, n_rows, bitmask,
                                                                       ids, n_ids, lengths);
  return check_launch("k_row_lengths");
}

// Histogram of the fetched length of n_sample evenly spaced rows (row
// i * n_rows / n_sample), in 16-byte chunks: hist[c] = rows that occupy c
// chunks, c <= ceil(W / 4).  Raw rows and rows whose headers announce W words
// or more count as W words.
__global__ void k_length_hist(const PlanView pv, const uint32_t* __restrict__ slots, uint64_t n_rows,
                              const uint32_t* __restrict__ bitmask, uint64_t n_sample,
                              uint32_t* __restrict__ hist) {
  extern __shared__ uint32_t h_s[];
  const uint32_t W = pv.W, S = pv.S;
  const uint32_t nb = (W + 3u) / 4u + 1u;
  for (uint32_t b = threadIdx.x; b < nb; b += blockDim.x) h_s[b] = 0;
  __syncthreads();
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_sample; i += stride) {
    const uint64_t r = i * n_rows / n_sample;
    uint32_t len = W;
    if ((ld_u32(bitmask + (r >> 5)) >> (r & 31u)) & 1u) {
      const uint32_t* h = slots + r * W;
      uint32_t drop = 0;
      for (uint32_t s = 0; s < S; ++s) {
        uint32_t H = ld_u32(h + s);
        if (s == S - 1 && W - 32u * s < 32u) H &= (1u << (W - 32u * s)) - 1u;
        for (int k = 0; k < kPlanes; ++k) drop += __popc(H & __ldg(pv.planes + s * kPlanes + k)) << k;
      }
      const uint32_t Lw = (32u * (S + W) - drop + 31u) >> 5;
      len = Lw < W ? Lw : W;
    }
    atomicAdd(h_s + (len + 3u) / 4u, 1u);
  }
  __syncthreads();
  for (uint32_t b = threadIdx.x; b < nb; b += blockDim.x)
    if (h_s[b]) atomicAdd(hist + b, h_s[b]);
}

int launch_length_hist(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                       const uint32_t* bitmask, uint64_t n_sample, uint32_t* hist, cudaStream_t stream) {
  const unsigned threads = 256;
  const uint64_t want = (n_sample + threads - 1) / threads;
  const uint64_t cap = 4ull * sm_count(plan->device);
  const size_t smem = 4ull * ((plan->W + 3u) / 4u + 1u);
  k_length_hist<<<static_cast<unsigned>(want < cap ? want : cap), threads, smem, stream>>>(
      plan->view, slots, n_rows, bitmask, n_sample, hist);
  return check_launch("k_length_hist");
}

}  // namespace ibp
