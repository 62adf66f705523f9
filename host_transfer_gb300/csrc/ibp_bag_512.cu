// ibp_bag_512.cu - instantiations of the fused gather-decompress and pooling
// kernel (ibp_bag.cuh) with 512-word groups.
#include "ibp_bag.cuh"

namespace ibp {

int launch_bag_512(const ibp_plan* plan, BagArgs& a, cudaStream_t stream) {
  return launch_bag_gw<512u, false>(plan, a, stream);
}

}  // namespace ibp
