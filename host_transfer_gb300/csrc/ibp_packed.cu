// ibp_packed.cu - the packed cache layout.
//
// « Intégration au système », cache compression: compressing the tensors a
// GPU software cache holds raises its effective capacity.  Fixed-size slots
// (the in-place layout of the host transfers) save no space, so a cache keeps
// each row's stored words only - Lw for a compressed row, W for a raw one,
// rounded up to 4 words so that every row starts on a 16-byte boundary - back
// to back, with offsets[r] the word where row r starts and offsets[n] the
// total.  The stream of a row is the same as in its slot.
#include <cuda_runtime.h>

#include "ibp_internal.cuh"

namespace ibp {

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;  // per thread
constexpr uint64_t kScanBlock = kScanThreads * kScanItems;

// offsets[r + 1] = stored words of row r rounded up to 4; offsets[0] = 0.
__global__ void k_packed_lengths(const PlanView pv, const uint32_t* __restrict__ slots,
                                 uint64_t n_rows, const uint32_t* __restrict__ bitmask,
                                 uint64_t* __restrict__ offsets) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  const uint32_t W = pv.W, S = pv.S;
  for (uint64_t r = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < n_rows; r += stride) {
    if (r == 0) offsets[0] = 0;
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
      len = Lw < W ? Lw : W;  // a corrupt row is stored whole; its decode reports it
    }
    offsets[r + 1] = (len + 3u) & ~3u;
  }
}

// Inclusive scan of each block's kScanBlock items in place; block totals to
// partials.
__global__ void __launch_bounds__(kScanThreads) k_scan_local(uint64_t* __restrict__ v, uint64_t n,
                                                             uint64_t* __restrict__ partials) {
  __shared__ uint64_t warp_sums[kScanThreads / 32];
  const uint64_t base = static_cast<uint64_t>(blockIdx.x) * kScanBlock + threadIdx.x * kScanItems;
  uint64_t x[kScanItems];
  uint64_t run = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    x[i] = base + i < n ? v[base + i] : 0;
    run += x[i];
    x[i] = run;  // inclusive within the thread
  }
  // exclusive scan of the thread totals across the block
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t incl = run;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= static_cast<uint32_t>(d)) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint64_t ws = warp_sums[lane];
    uint64_t wi = ws;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, wi, d);
      if (lane >= static_cast<uint32_t>(d)) wi += t;
    }
    warp_sums[lane] = wi - ws;  // exclusive
  }
  __syncthreads();
  const uint64_t before = warp_sums[warp] + incl - run;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i)
    if (base + i < n) v[base + i] = x[i] + before;
  if (threadIdx.x == kScanThreads - 1) partials[blockIdx.x] = before + run;
}

// Exclusive scan of the block totals (one block, any count).
__global__ void __launch_bounds__(kScanThreads) k_scan_partials(uint64_t* __restrict__ partials, uint64_t nb) {
  __shared__ uint64_t warp_sums[kScanThreads / 32];
  __shared__ uint64_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (uint64_t b0 = 0; b0 < nb; b0 += kScanThreads) {
    const uint64_t i = b0 + threadIdx.x;
    const uint64_t x = i < nb ? partials[i] : 0;
    uint64_t incl = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= static_cast<uint32_t>(d)) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const uint64_t ws = warp_sums[lane];
      uint64_t wi = ws;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, wi, d);
        if (lane >= static_cast<uint32_t>(d)) wi += t;
      }
      warp_sums[lane] = wi - ws;
    }
    __syncthreads();
    const uint64_t c = carry;
    if (i < nb) partials[i] = c + warp_sums[warp] + incl - x;
    __syncthreads();
    if (threadIdx.x == kScanThreads - 1) carry = c + warp_sums[warp] + incl;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kScanThreads) k_scan_add(uint64_t* __restrict__ v, uint64_t n,
                                                           const uint64_t* __restrict__ partials) {
  const uint64_t add = partials[blockIdx.x];
  const uint64_t base = static_cast<uint64_t>(blockIdx.x) * kScanBlock + threadIdx.x * kScanItems;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i)
    if (base + i < n) v[base + i] += add;
}

int launch_packed_offsets(const ibp_plan* plan, const uint32_t* slots, uint64_t n_rows,
                          const uint32_t* bitmask, uint64_t* offsets, cudaStream_t stream) {
  const uint64_t want = (n_rows + 255) / 256;
  const uint64_t cap = 16ull * sm_count(plan->device);
  k_packed_lengths<<<static_cast<unsigned>(want < cap ? want : cap), 256, 0, stream>>>(
      plan->view, slots, n_rows, bitmask, offsets);
  int rc = check_launch("k_packed_lengths");
  if (rc != IBP_OK) return rc;
  // inclusive scan of offsets[1 .. n_rows]
  const uint64_t nb = (n_rows + kScanBlock - 1) / kScanBlock;
  if (nb > 0x7FFFFFFFull) return IBP_EINVAL;
  uint64_t* partials = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&partials), nb * sizeof(uint64_t), stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return IBP_ENOMEM;
  }
  k_scan_local<<<static_cast<unsigned>(nb), kScanThreads, 0, stream>>>(offsets + 1, n_rows, partials);
  rc = check_launch("k_scan_local");
  if (rc == IBP_OK) {
    k_scan_partials<<<1, kScanThreads, 0, stream>>>(partials, nb);
    rc = check_launch("k_scan_partials");
  }
  if (rc == IBP_OK) {
    k_scan_add<<<static_cast<unsigned>(nb), kScanThreads, 0, stream>>>(offsets + 1, n_rows, partials);
    rc = check_launch("k_scan_add");
  }
  e = cudaFreeAsync(partials, stream);
  if (rc == IBP_OK && e != cudaSuccess) {
    set_cuda_error(e, "cudaFreeAsync");
    rc = IBP_ECUDA;
  }
  return rc;
}

// A warp per row: the row's stored words (16-byte chunks) from its slot to
// its place in the packed buffer.
__global__ void k_pack(const uint32_t* __restrict__ slots, uint64_t n_rows, uint32_t W,
                       const uint64_t* __restrict__ offsets, uint32_t* __restrict__ packed) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t gw = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nw = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;
  for (uint64_t r = gw; r < n_rows; r += nw) {
    const uint64_t lo = offsets[r], hi = offsets[r + 1];
    uint64_t len = hi > lo ? hi - lo : 0;
    if (len > W) len = W;
    const uint4* src = reinterpret_cast<const uint4*>(slots + r * W);
    uint4* dst = reinterpret_cast<uint4*>(packed + lo);
    for (uint32_t c = lane; c < (len >> 2); c += 32) dst[c] = src[c];
  }
}

int launch_pack(const uint32_t* slots, uint64_t n_rows, uint32_t W, const uint64_t* offsets,
                uint32_t* packed, int device, cudaStream_t stream) {
  const uint64_t want = (n_rows * 32 + 255) / 256;
  const uint64_t cap = 16ull * sm_count(device);
  k_pack<<<static_cast<unsigned>(want < cap ? want : cap), 256, 0, stream>>>(slots, n_rows, W, offsets,
                                                                            packed);
  return check_launch("k_pack");
}

}  // namespace ibp
