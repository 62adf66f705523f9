// ibp_decompress_fast_tp.cu - per-word-table instantiations of the
// specialised decompress kernel (ibp_decompress_fast.cuh) for the packed
// cache layout.  The packed buffer lives in device memory, so these take the
// device-slot launch shape: 1024-word groups and the device register budget
// (sparse rows from the packed cache 2205 -> 2593 GB/s, 0.39 -> 0.46 of the
// HBM peak; 512-word groups with three CTAs per SM: 2505 GB/s).
#include "ibp_decompress_fast.cuh"

namespace ibp {

int launch_fast_table_packed(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  return launch_fast_table_t<true, kGroupWordsDevTable, true>(plan, a, stream);
}

}  // namespace ibp
