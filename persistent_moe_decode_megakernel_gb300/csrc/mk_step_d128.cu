// mk_step_d128.cu -- instantiations of the step kernel for head_dim 128.
#include "mk_kernel.cuh"

namespace mk {

cudaError_t configure_d128(size_t smem) { return configure_all<128, false>(smem); }
cudaError_t launch_d128(const Params& p, int tb, size_t smem, cudaStream_t s) { return launch_any<128, false>(p, tb, smem, s); }
cudaError_t occupancy_d128(int* blocks, size_t smem) { return occupancy_d<128, false>(blocks, smem); }

size_t smem_bytes_impl() { return sizeof(Smem) + 1024; }

}  // namespace mk
