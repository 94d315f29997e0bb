// mk_step_d128_q8.cu -- instantiations of the step kernel for head_dim 128 over a q8_0 KV cache.
#include "mk_kernel.cuh"

namespace mk {

cudaError_t configure_d128_q8(size_t smem) { return configure_all<128, true>(smem); }
cudaError_t launch_d128_q8(const Params& p, int tb, size_t smem, cudaStream_t s) {
  return launch_any<128, true>(p, tb, smem, s);
}
cudaError_t occupancy_d128_q8(int* blocks, size_t smem) { return occupancy_d<128, true>(blocks, smem); }

}  // namespace mk
