// ibp_decompress_fast_up.cu - uniform-plan instantiations of the specialised
// decompress kernel (ibp_decompress_fast.cuh) for the packed cache layout, with
// the device-slot group size (a packed cache lives in HBM).
#include "ibp_decompress_fast.cuh"

namespace ibp {

int launch_fast_uniform_packed(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  return launch_fast_uniform_t<true, kGroupWordsDev, true>(plan, a, stream);
}

}  // namespace ibp
