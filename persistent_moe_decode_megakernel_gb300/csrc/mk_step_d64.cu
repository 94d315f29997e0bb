// mk_step_d64.cu -- instantiations of the step kernel for head_dim 64.
#include "mk_kernel.cuh"

namespace mk {

cudaError_t configure_d64(size_t smem) { return configure_all<64, false>(smem); }
cudaError_t launch_d64(const Params& p, int tb, size_t smem, cudaStream_t s) { return launch_any<64, false>(p, tb, smem, s); }
cudaError_t occupancy_d64(int* blocks, size_t smem) { return occupancy_d<64, false>(blocks, smem); }

}  // namespace mk
