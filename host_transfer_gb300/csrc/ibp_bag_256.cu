// ibp_bag_256.cu - instantiations of the fused gather-decompress and pooling
// kernel (ibp_bag.cuh) with 256-word groups.
#include "ibp_bag.cuh"

namespace ibp {

int launch_bag_256(const ibp_plan* plan, BagArgs& a, cudaStream_t stream) {
  return launch_bag_gw<256u, false>(plan, a, stream);
}

}  // namespace ibp
