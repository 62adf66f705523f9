// ibp_decompress_fast_u.cu - uniform-plan instantiations (slot layout) of the
// specialised decompress kernel (ibp_decompress_fast.cuh), and the choice
// between the specialised kernels and the general one.
#include "ibp_decompress_fast.cuh"

namespace ibp {

int launch_fast_uniform(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  return launch_fast_uniform_t<false, kGroupWords>(plan, a, stream);
}

bool fast_decompress_applies(const ibp_plan* plan, const DecodeArgs& a) {
  const uint32_t S = plan->S;
  const bool pow2_segments = S == 1 || S == 2 || S == 4 || S == 8 || S == 16 || S == 32 || S == 64;
  const bool runs_ok = plan->max_runs >= 1 && plan->max_runs <= static_cast<uint32_t>(kMaxRuns);
  // per-word tables: W words x 16 or 32 bytes of shared memory per CTA
  const bool table_ok = plan->uniform || plan->W <= 1024u;
  return runs_ok && table_ok && plan->W == 32u * S && pow2_segments && a.vec &&
         a.n_rows < (1ull << 31) && (a.pre % 4u) == 0;
}

int launch_decompress_fast(const ibp_plan* plan, DecodeArgs& a, cudaStream_t stream) {
  if (a.offsets)
    return plan->uniform ? launch_fast_uniform_packed(plan, a, stream)
                         : launch_fast_table_packed(plan, a, stream);
  if ((a.pv.hints & IBP_HINT_ROW_REUSE) && !a.dev_slots)
    return plan->uniform ? launch_fast_uniform_reuse(plan, a, stream) : launch_fast_table_reuse(plan, a, stream);
  if (plan->uniform) return a.dev_slots ? launch_fast_uniform_dev(plan, a, stream) : launch_fast_uniform(plan, a, stream);
  return a.dev_slots ? launch_fast_table_dev(plan, a, stream) : launch_fast_table(plan, a, stream);
}

}  // namespace ibp
