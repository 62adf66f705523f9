// ibp_bag_split.cu - instantiations of the fused gather-decompress and pooling
// kernel (ibp_bag.cuh) with 1024-word groups and teams of 2 or 4 warps per
// bag, which split each row's segments (few bags on device slots).
#include "ibp_bag.cuh"

namespace ibp {

int launch_bag_1024_split(const ibp_plan* plan, BagArgs& a, cudaStream_t stream, int cs) {
  return cs >= 4 ? launch_bag_gw<1024u, false, 4>(plan, a, stream) : launch_bag_gw<1024u, false, 2>(plan, a, stream);
}

}  // namespace ibp
