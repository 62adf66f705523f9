// ibp_bag.cu - the choice of group size for the fused gather-decompress and
// pooling kernel (ibp_bag.cuh), measured on the dense GNN, sparse GNN and DLRM
// tables (bags of 32 ids): host-mapped slots read with the row-reuse hint
// take 256-word groups (the smaller stages leave more of the SM's on-chip
// memory to L1, where repeated rows are found), other host-mapped slots 512;
// slots in device memory take 1024-word groups for W >= 128 (more rows in
// flight per warp: one bag is one warp's sequence of rows) and 512 below.
// Rows of bfloat16 pairs take 512-word groups.  Few bags on device slots are
// pooled by teams of 2 or 4 warps per bag (column split).
#include "ibp_bag.cuh"

namespace ibp {

int launch_bag(const ibp_plan* plan, BagArgs& a, cudaStream_t stream) {
  if (!fast_decompress_applies(plan, a.d) || plan->S > 16u) return IBP_EINVAL;
  if (a.bf16) return launch_bag_bf16(plan, a, stream);
  if (!a.d.dev_slots) return (a.d.pv.hints & IBP_HINT_ROW_REUSE) ? launch_bag_256(plan, a, stream)
                                                                   : launch_bag_512(plan, a, stream);
  if (plan->W < 128u) return launch_bag_512(plan, a, stream);
  // Few bags: a team of warps per bag, each pooling a slice of the segments,
  // while the bags leave the GPU's warp slots free (two CTAs of eight warps
  // per SM with these groups).
  const uint64_t slots_free = 16ull * sm_count(plan->device);
  if (plan->S >= 4 && 4 * a.n_bags <= slots_free) return launch_bag_1024_split(plan, a, stream, 4);
  if (plan->S >= 2 && 2 * a.n_bags <= slots_free) return launch_bag_1024_split(plan, a, stream, 2);
  return launch_bag_1024(plan, a, stream);
}

}  // namespace ibp
