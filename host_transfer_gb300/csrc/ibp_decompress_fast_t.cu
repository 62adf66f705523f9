// ibp_decompress_fast_t.cu - per-word-table instantiations of the
// specialised decompress kernel (ibp_decompress_fast.cuh): plans whose word
// positions have different Masks, with up to four runs of kept bits per word
// and 0, 1 or 6 e-planes.
#include "ibp_decompress_fast.cuh"

namespace ibp {

template <int R>
static int launch_table_r(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  switch (plan->view.npl) {
    case 0: return launch_fast_sc<R, 0, true>(plan, a, stream);
    case 1: return launch_fast_sc<R, 1, true>(plan, a, stream);
    default: return launch_fast_sc<R, 6, true>(plan, a, stream);
  }
}

int launch_fast_table(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  return plan->max_runs <= 2 ? launch_table_r<2>(plan, a, stream) : launch_table_r<4>(plan, a, stream);
}

}  // namespace ibp
