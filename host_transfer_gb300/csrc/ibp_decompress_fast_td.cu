// ibp_decompress_fast_td.cu - per-word-table instantiations (slot layout) of
// the specialised decompress kernel (ibp_decompress_fast.cuh) for slots in
// device memory: 1024-word groups, and a register budget sized for the CTAs
// that shared memory then holds.
#include "ibp_decompress_fast.cuh"

namespace ibp {

int launch_fast_table_dev(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  return launch_fast_table_t<false, kGroupWordsDevTable, true>(plan, a, stream);
}

}  // namespace ibp
