// ibp_preprocess.cu - Mask/Bitval from a sample of rows, and the per-word
// decode tables of a plan.
//
// « Algorithme central », step 1 (Prétraitement): the bit positions that hold
// the same value in at least a fraction T of the sampled tensors form the
// Mask; their values form Bitval; both are kept in GPU memory and reused for
// the whole dataset.
#include <cuda_runtime.h>

#include <cmath>

#include "ibp_internal.cuh"

namespace ibp {

constexpr int kCountThreads = 128;
constexpr uint64_t kRowsPerCountBlock = 2048;  // at least; more when grid.y would pass 65535

// ones[w*32 + b] += number of sampled rows with bit b of word w set.
// Threads run along w (coalesced rows); blockIdx.y takes a slice of rows; each
// thread keeps 32 counters in registers and adds them once at the end.
__global__ void __launch_bounds__(kCountThreads) k_count_ones(const uint32_t* __restrict__ sample,
                                                              uint64_t s_rows, uint32_t W,
                                                              uint64_t rows_per_block,
                                                              uint32_t* __restrict__ ones) {
  const uint32_t w = blockIdx.x * kCountThreads + threadIdx.x;
  if (w >= W) return;
  const uint64_t r0 = static_cast<uint64_t>(blockIdx.y) * rows_per_block;
  if (r0 >= s_rows) return;
  const uint64_t r1 = min(s_rows, r0 + rows_per_block);
  uint32_t c[32];
#pragma unroll
  for (int b = 0; b < 32; ++b) c[b] = 0;
  const uint32_t* p = sample + r0 * W + w;
  for (uint64_t r = r0; r < r1; ++r, p += W) {
    const uint32_t x = __ldg(p);
#pragma unroll
    for (int b = 0; b < 32; ++b) c[b] += (x >> b) & 1u;
  }
#pragma unroll
  for (int b = 0; b < 32; ++b)
    if (c[b]) atomicAdd(&ones[w * 32 + b], c[b]);
}

// Threshold t = ceil(T * s_rows) in IEEE double; a bit is invariant when at
// least t rows agree on it, and its Bitval bit is the majority value (a tie
// gives 0).
__global__ void k_mask_from_counts(const uint32_t* __restrict__ ones, uint64_t s_rows, uint32_t W,
                                   double T, uint32_t* __restrict__ mask,
                                   uint32_t* __restrict__ bitval) {
  const uint32_t w = blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= W) return;
  const uint64_t t = static_cast<uint64_t>(ceil(T * static_cast<double>(s_rows)));
  uint32_t m = 0, v = 0;
#pragma unroll 4
  for (int b = 0; b < 32; ++b) {
    const uint64_t n1 = ones[w * 32 + b];
    const uint64_t n0 = s_rows - n1;
    if ((n1 > n0 ? n1 : n0) >= t) {
      m |= 1u << b;
      if (n1 > n0) v |= 1u << b;
    }
  }
  mask[w] = m;
  bitval[w] = v;
}

int launch_preprocess(const uint32_t* sample, uint64_t s_rows, uint32_t W, double T,
                      uint32_t* mask, uint32_t* bitval, cudaStream_t stream) {
  uint32_t* ones = nullptr;
  const size_t bytes = 32ull * W * sizeof(uint32_t);
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&ones), bytes, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return IBP_ENOMEM;
  }
  e = cudaMemsetAsync(ones, 0, bytes, stream);
  if (e != cudaSuccess) {
    set_cuda_error(e, "cudaMemsetAsync");
    cudaFreeAsync(ones, stream);
    return IBP_ECUDA;
  }
  uint64_t per_block = kRowsPerCountBlock;
  if ((s_rows + per_block - 1) / per_block > 65535) per_block = (s_rows + 65534) / 65535;
  const uint64_t yblocks = (s_rows + per_block - 1) / per_block;
  dim3 grid((W + kCountThreads - 1) / kCountThreads, static_cast<unsigned>(yblocks));
  k_count_ones<<<grid, kCountThreads, 0, stream>>>(sample, s_rows, W, per_block, ones);
  int rc = check_launch("k_count_ones");
  if (rc == IBP_OK) {
    k_mask_from_counts<<<(W + 127) / 128, 128, 0, stream>>>(ones, s_rows, W, T, mask, bitval);
    rc = check_launch("k_mask_from_counts");
  }
  e = cudaFreeAsync(ones, stream);
  if (rc == IBP_OK && e != cudaSuccess) {
    set_cuda_error(e, "cudaFreeAsync");
    rc = IBP_ECUDA;
  }
  return rc;
}

int launch_count_and_threshold(const uint32_t* sample, uint64_t s_rows, uint32_t W, double T,
                               uint32_t* ones, uint32_t* mask, uint32_t* bitval,
                               cudaStream_t stream) {
  uint64_t per_block = kRowsPerCountBlock;
  if ((s_rows + per_block - 1) / per_block > 65535) per_block = (s_rows + 65534) / 65535;
  const uint64_t yblocks = (s_rows + per_block - 1) / per_block;
  dim3 grid((W + kCountThreads - 1) / kCountThreads, static_cast<unsigned>(yblocks));
  k_count_ones<<<grid, kCountThreads, 0, stream>>>(sample, s_rows, W, per_block, ones);
  int rc = check_launch("k_count_ones");
  if (rc != IBP_OK) return rc;
  k_mask_from_counts<<<(W + 127) / 128, 128, 0, stream>>>(ones, s_rows, W, T, mask, bitval);
  return check_launch("k_mask_from_counts");
}

// ---------------------------------------------------------------------------
// Plan tables

struct PlanSummary {
  uint32_t nonuniform;
  uint32_t max_runs;
  uint32_t min_kept;
  uint32_t max_kept;
  unsigned long long sum_kept;  // kept bits over all word positions
  uint32_t present_lo;          // bit p set: some word has popcount(Mask) = p (p < 32)
  uint32_t present_hi;          // some word has popcount(Mask) = 32
};

// One thread per word position; one warp per 32-word segment (for the bit
// planes).  The block size is a multiple of 32 and every lane reaches the
// ballots.
__global__ void k_plan_tables(PlanView v, PlanSummary* sum) {
  const uint32_t W = v.W;
  const uint32_t w = blockIdx.x * blockDim.x + threadIdx.x;
  const bool in = w < W;
  uint32_t* mask = const_cast<uint32_t*>(v.mask);
  uint32_t* bm = const_cast<uint32_t*>(v.bm);
  uint32_t p = 0;
  if (in) {
    const uint32_t m = mask[w];
    const uint32_t b = bm[w] & m;
    bm[w] = b;
    p = __popc(m);
    const_cast<uint32_t*>(v.pcnt)[w] = p;
    const uint32_t keep = ~m;
    // runs of kept bits, low to high
    uint32_t x = keep, src = 0, nruns = 0, shifts = 0;
    uint32_t rm[kMaxRuns] = {0, 0, 0, 0};
    while (x) {
      const uint32_t lo = __ffs(x) - 1;
      const uint32_t y = x >> lo;
      const uint32_t len = (y == 0xFFFFFFFFu) ? 32u : static_cast<uint32_t>(__ffs(~y) - 1);
      const uint32_t run = (len == 32 ? 0xFFFFFFFFu : ((1u << len) - 1u)) << lo;
      if (nruns < kMaxRuns) {
        rm[nruns] = run;
        shifts |= (lo - src) << (8 * nruns);
      }
      src += len;
      ++nruns;
      x &= ~run;
    }
#pragma unroll
    for (int k = 0; k < kMaxRuns; ++k) const_cast<uint32_t*>(v.rmask)[k * W + w] = rm[k];
    const_cast<uint32_t*>(v.rshift)[w] = shifts;
    // move masks of the five-step compress/expand of `keep`
    uint32_t mk = ~keep << 1, mm = keep;
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      uint32_t mp = mk ^ (mk << 1);
      mp ^= mp << 2;
      mp ^= mp << 4;
      mp ^= mp << 8;
      mp ^= mp << 16;
      const uint32_t mvi = mp & mm;
      const_cast<uint32_t*>(v.mv)[i * W + w] = mvi;
      mm = (mm ^ mvi) | (mvi >> (1u << i));
      mk &= ~mp;
    }
    atomicMax(&sum->max_runs, nruns);
    atomicMin(&sum->min_kept, 32u - p);
    atomicMax(&sum->max_kept, 32u - p);
    atomicAdd(&sum->sum_kept, static_cast<unsigned long long>(32u - p));
    if (p < 32u)
      atomicOr(&sum->present_lo, 1u << p);
    else
      atomicOr(&sum->present_hi, 1u);
    if (m != mask[0] || b != (bm[0] & mask[0])) atomicOr(&sum->nonuniform, 1u);
  }
  // bit planes of popcount(Mask) per segment
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t seg = w / 32;
#pragma unroll
  for (int k = 0; k < kPlanes; ++k) {
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, in && ((p >> k) & 1u));
    if (lane == 0 && seg < v.S) const_cast<uint32_t*>(v.planes)[seg * kPlanes + k] = bal;
  }
}

// eplanes[s*6+k] bit i = bit k of (pcnt[32s+i] - p_min) / p_scale.
__global__ void k_plan_eplanes(PlanView v) {
  const uint32_t w = blockIdx.x * blockDim.x + threadIdx.x;
  const bool in = w < v.W;
  const uint32_t e = in ? (v.pcnt[w] - v.p_min) / v.p_scale : 0u;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t seg = w / 32;
#pragma unroll
  for (int k = 0; k < kPlanes; ++k) {
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, in && ((e >> k) & 1u));
    if (lane == 0 && seg < v.S) const_cast<uint32_t*>(v.eplanes)[seg * kPlanes + k] = bal;
  }
}

static uint32_t gcd_u32(uint32_t a, uint32_t b) {
  while (b) {
    const uint32_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

int build_plan_tables(ibp_plan* plan) {
  PlanSummary h = {0, 0, 32, 0, 0, 0, 0};
  PlanSummary* d = nullptr;
  cudaError_t e = cudaMalloc(&d, sizeof(PlanSummary));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return IBP_ENOMEM;
  }
  e = cudaMemcpy(d, &h, sizeof(h), cudaMemcpyHostToDevice);
  const uint32_t threads = 256;
  const uint32_t blocks = (plan->W + threads - 1) / threads;
  if (e == cudaSuccess) {
    k_plan_tables<<<blocks, threads>>>(plan->view, d);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(&h, d, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) {
    set_cuda_error(e, "k_plan_tables");
    cudaGetLastError();
    return IBP_ECUDA;
  }
  // popcounts present -> p_min, p_scale (gcd of the differences), npl
  {
    PlanView& v = plan->view;
    uint32_t pmin = 32, pmax = 0, g = 0;
    for (uint32_t q = 0; q <= 32; ++q) {
      const bool has = q < 32 ? ((h.present_lo >> q) & 1u) : (h.present_hi & 1u);
      if (!has) continue;
      if (q < pmin) pmin = q;
      if (q > pmax) pmax = q;
    }
    for (uint32_t q = pmin; q <= 32; ++q) {
      const bool has = q < 32 ? ((h.present_lo >> q) & 1u) : (h.present_hi & 1u);
      if (has && q > pmin) g = gcd_u32(g, q - pmin);
    }
    v.p_min = pmin;
    v.p_scale = g ? g : 1u;
    const uint32_t emax = (pmax - pmin) / v.p_scale;
    v.npl = emax == 0 ? 0u : (emax == 1 ? 1u : 6u);
    k_plan_eplanes<<<(plan->W + 255) / 256, 256>>>(v);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      set_cuda_error(e, "k_plan_eplanes");
      cudaGetLastError();
      return IBP_ECUDA;
    }
  }
  plan->uniform = h.nonuniform ? 0u : 1u;
  plan->max_runs = h.max_runs;
  plan->min_kept = h.min_kept;
  plan->max_kept = h.max_kept;
  // Shortest stream a compressed row can have (every word matching): the
  // words a reader needs for any row, whatever its headers say.
  const uint64_t min_bits = 32ull * plan->S + h.sum_kept;
  const uint64_t lmin = (min_bits + 31) / 32;
  plan->lmin = static_cast<uint32_t>(lmin < plan->W ? lmin : plan->W);
  PlanView& v = plan->view;
  // word 0's entries become the uniform scalars (used only when uniform)
  uint32_t w0[13];
  const uint32_t* src[13] = {v.mask, v.bm, v.pcnt, v.rmask, v.rmask + plan->W,
                             v.rmask + 2 * plan->W, v.rmask + 3 * plan->W, v.rshift, v.mv,
                             v.mv + plan->W, v.mv + 2 * plan->W, v.mv + 3 * plan->W,
                             v.mv + 4 * plan->W};
  for (int i = 0; i < 13; ++i) {
    e = cudaMemcpy(&w0[i], src[i], 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
      set_cuda_error(e, "plan scalars");
      cudaGetLastError();
      return IBP_ECUDA;
    }
  }
  v.u_mask = w0[0];
  v.u_bm = w0[1];
  v.u_p = w0[2];
  v.u_keep = ~w0[0];
  for (int k = 0; k < kMaxRuns; ++k) {
    v.u_rmask[k] = w0[3 + k];
    v.u_rsh[k] = (w0[7] >> (8 * k)) & 0xFFu;
  }
  for (int i = 0; i < 5; ++i) v.u_mv[i] = w0[8 + i];
  return IBP_OK;
}

}  // namespace ibp
