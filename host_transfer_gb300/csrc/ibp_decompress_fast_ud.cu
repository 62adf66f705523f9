// ibp_decompress_fast_ud.cu - uniform-plan instantiations (slot layout) of the
// specialised decompress kernel (ibp_decompress_fast.cuh) for slots in device
// memory: 768-word groups and a two-CTA register budget.
#include "ibp_decompress_fast.cuh"

namespace ibp {

int launch_fast_uniform_dev(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  return launch_fast_uniform_t<false, kGroupWordsDev, true>(plan, a, stream);
}

}  // namespace ibp
