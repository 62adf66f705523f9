// ibp_decompress_fast_t.cu - per-word-table instantiations (slot layout) of
// the specialised decompress kernel (ibp_decompress_fast.cuh): plans whose
// word positions have different Masks, with up to four runs of kept bits per
// word and 0, 1 or 6 e-planes.
#include "ibp_decompress_fast.cuh"

namespace ibp {

int launch_fast_table(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  return launch_fast_table_t<false, kGroupWords>(plan, a, stream);
}

}  // namespace ibp
