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

}  // namespace ibp
