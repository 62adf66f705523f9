// ibp_decompress_fast_set.cu - plan-set instantiations of the specialised
// decompress kernel (ibp_decompress_fast.cuh): contiguous decode of a table
// whose consecutive row blocks each have their own plan (finer Mask
// granularity, e.g. one plan per attention head of a KV cache).  Every plan of
// the set goes through the per-word-table path sized for the set's most runs
// of kept bits and e-planes; a uniform plan's tables hold its one Mask at
// every position and its e-planes are zero, so it decodes there unchanged.
#include "ibp_decompress_fast.cuh"

namespace ibp {

template <int R>
static int launch_fast_set_r(const ibp_plan* plan0, uint32_t npl, DecodeArgs& a, cudaStream_t stream) {
  switch (npl) {
    case 0: return launch_fast_set_sc<R, 0>(plan0, a, stream);
    case 1: return launch_fast_set_sc<R, 1>(plan0, a, stream);
    default: return launch_fast_set_sc<R, 6>(plan0, a, stream);
  }
}

int launch_fast_set(const ibp_plan* plan0, uint32_t max_runs, uint32_t npl, DecodeArgs& a, cudaStream_t stream) {
  return max_runs <= 2 ? launch_fast_set_r<2>(plan0, npl, a, stream) : launch_fast_set_r<4>(plan0, npl, a, stream);
}

}  // namespace ibp
