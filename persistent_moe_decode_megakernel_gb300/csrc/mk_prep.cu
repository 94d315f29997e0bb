// mk_prep.cu -- one-time weight preparation at context creation: the transposed copy of
// each layer's down projections used by the small-batch MoE path.
//
// w_down of one expert is [H][F] (a hidden row holds its F weights); the copy is [F][H],
// so that the down-projection weights of one FFN row -- the row a block's gate/up unit
// produces -- are one contiguous H-element run that a bulk copy moves in one piece.
#include <cuda_runtime.h>
#include <stdint.h>

namespace mk {
namespace {

// 32 x 32 tiles through shared memory (padded against bank conflicts); grid (F/32, H/32, E)
__global__ void transpose_down_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, int H, int F) {
  __shared__ uint16_t tile[32][33];
  const size_t ex = static_cast<size_t>(blockIdx.z) * H * F;
  const int f0 = blockIdx.x * 32, h0 = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int h = h0 + r, f = f0 + threadIdx.x;
    if (h < H && f < F) tile[r][threadIdx.x] = in[ex + static_cast<size_t>(h) * F + f];
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int f = f0 + r, h = h0 + threadIdx.x;
    if (f < F && h < H) out[ex + static_cast<size_t>(f) * H + h] = tile[threadIdx.x][r];
  }
}

}  // namespace

// out[e][f][h] = in[e][h][f] for E experts (bf16 bit patterns); enqueued on stream s
cudaError_t transpose_down(const uint16_t* in, uint16_t* out, int E, int H, int F, cudaStream_t s) {
  const dim3 grid((F + 31) / 32, (H + 31) / 32, E);
  transpose_down_kernel<<<grid, dim3(32, 8), 0, s>>>(in, out, H, F);
  return cudaGetLastError();
}

}  // namespace mk
