// mk_launch.cu -- dispatch from the host library to the step-kernel instantiations.
#include <cuda_runtime.h>

#include "mk_layout.h"

namespace mk {

cudaError_t configure_d128(size_t smem);
cudaError_t configure_d64(size_t smem);
cudaError_t configure_d128_q8(size_t smem);
cudaError_t launch_d128(const Params& p, int tb, size_t smem, cudaStream_t s);
cudaError_t launch_d128_q8(const Params& p, int tb, size_t smem, cudaStream_t s);
cudaError_t launch_d64(const Params& p, int tb, size_t smem, cudaStream_t s);
cudaError_t occupancy_d128(int* blocks, size_t smem);
cudaError_t occupancy_d64(int* blocks, size_t smem);
cudaError_t occupancy_d128_q8(int* blocks, size_t smem);
size_t smem_bytes_impl();

size_t smem_bytes() { return smem_bytes_impl(); }

// rows of the batch held in registers at once by a GEMV tile
int tb_for_batch(int B) { return B <= 1 ? 1 : (B <= 2 ? 2 : 4); }
// the instantiation of a step (see launch_any): 5 for the tcgen05 one (batches of kTcMinBatch
// rows or more), 4 for 3-4 rows; batches of 1-2 rows run a narrow one with the small-batch MoE
// path (1, 2) or, where the step cannot take it, with the general path (11, 12)
int tb_for_step(const Params& p) {
  if (p.tc) return 5;
  const int tb = tb_for_batch(p.B);
  return tb == 4 ? 4 : p.small_moe ? tb : 10 + tb;
}

cudaError_t configure_kernels(int D, bool kv_q8) {
  if (kv_q8) return D == 128 ? configure_d128_q8(smem_bytes()) : cudaErrorInvalidValue;
  return D == 128 ? configure_d128(smem_bytes()) : configure_d64(smem_bytes());
}

cudaError_t occupancy(int D, bool kv_q8, int* blocks) {
  if (kv_q8) return D == 128 ? occupancy_d128_q8(blocks, smem_bytes()) : cudaErrorInvalidValue;
  return D == 128 ? occupancy_d128(blocks, smem_bytes()) : occupancy_d64(blocks, smem_bytes());
}

cudaError_t launch_step(const Params& p, cudaStream_t s) {
  const int tb = tb_for_step(p);
  if (p.kv_q8) return p.D == 128 ? launch_d128_q8(p, tb, smem_bytes(), s) : cudaErrorInvalidValue;
  return p.D == 128 ? launch_d128(p, tb, smem_bytes(), s) : launch_d64(p, tb, smem_bytes(), s);
}

}  // namespace mk
