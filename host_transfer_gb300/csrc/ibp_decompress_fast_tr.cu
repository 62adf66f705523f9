// ibp_decompress_fast_tr.cu - per-word-table instantiations (slot layout) of
// the specialised decompress kernel (ibp_decompress_fast.cuh) with the small
// groups used for row-reuse copies from host-mapped slots.
#include "ibp_decompress_fast.cuh"

namespace ibp {

int launch_fast_table_reuse(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  return launch_fast_table_t<false, kGroupWordsReuse>(plan, a, stream);
}

}  // namespace ibp
