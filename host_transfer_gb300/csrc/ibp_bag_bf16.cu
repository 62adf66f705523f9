// ibp_bag_bf16.cu - instantiations of the fused gather-decompress and pooling
// kernel (ibp_bag.cuh) for rows of bfloat16 pairs, with 512-word groups.
#include "ibp_bag.cuh"

namespace ibp {

int launch_bag_bf16(const ibp_plan* plan, BagArgs& a, cudaStream_t stream) {
  return launch_bag_gw<512u, true>(plan, a, stream);
}

}  // namespace ibp
