// mk_noalloc.cu -- paged GQA decode attention that allocates no device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's memory pool or allocator hooks, sandboxed plug-ins handed only
// pre-allocated buffers, or paths where an allocation would synchronise the
// device at a bad moment.  mk_create needs a workspace, so such callers cannot
// use the step kernel; this entry point gives them the attention part of the
// step with no allocation at all.  Its only scratch -- the split-K partial
// softmax states and an error word -- lives in one file-scope __device__ array
// of fixed size (4 MiB), which every GPU that loads the library keeps until
// the process exits.
//
// The split structure is the one the step kernel uses: each (row, KV head)
// is cut into up to nsplit page ranges; a first kernel computes every range's
// (max, sum, un-normalised output) with an online softmax, a second merges the
// ranges in range order.  The number of ranges is chosen so that the partials
// fit the scratch; shapes that do not fit even one range per (row, KV head)
// are rejected.

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "mk.h"

namespace mk {
void set_last_error(int code, const char* text);
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB
constexpr int kHeaderFloats = 64;                            // error word + padding, cleared every call
constexpr int kMaxDevices = 64;
constexpr int kBlock = 256;
constexpr int kPosBlock = 64;                                // positions scored per online-softmax step
constexpr int kMaxRows = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

struct RowLens {
  int32_t len[kMaxRows];
};

__device__ __forceinline__ float bf16f(uint16_t u) { return __uint_as_float(static_cast<uint32_t>(u) << 16); }

// One block per (range, KV head, row): online softmax over the range's positions.
// Partial layout: [row][kv head][range][head in group][D + 2] = (o[D], max, sum).
template <int D>
__global__ void __launch_bounds__(kBlock) split_kernel(const float* __restrict__ q, const uint16_t* __restrict__ kv,
                                                       const int32_t* __restrict__ bt, RowLens lens, int Hq, int Hkv,
                                                       int ps, int num_pages, int maxpg, int pages_per_range,
                                                       int nrange, float scale, float* __restrict__ scratch) {
  const int r = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = Hq / Hkv;
  const int tid = threadIdx.x;
  __shared__ float qs[8][D];
  __shared__ float sc[8][kPosBlock];
  __shared__ float mrun[8], lrun[8], corr[8];
  int* err = reinterpret_cast<int*>(scratch);
  float* part = scratch + kHeaderFloats;
  for (int i = tid; i < G * D; i += kBlock) {
    const int h = i / D, d = i % D;
    qs[h][d] = q[(static_cast<size_t>(b) * Hq + kvh * G + h) * D + d] * scale;
  }
  if (tid < G) { mrun[tid] = -INFINITY; lrun[tid] = 0.f; }
  constexpr int kPer = 8 * D / kBlock;   // output values per thread (G*D <= 8*D)
  float o[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) o[i] = 0.f;
  __syncthreads();
  const int Lc = lens.len[b];
  const int npg = (Lc + ps - 1) / ps;
  const int pg0 = r * pages_per_range, pg1 = min(npg, pg0 + pages_per_range);
  const int t_end = min(pg1 * ps, Lc);
  const size_t plane = static_cast<size_t>(Hkv) * ps * D;   // one K (or V) plane of a page
  for (int t0 = pg0 * ps; t0 < t_end; t0 += kPosBlock) {
    for (int i = tid; i < G * kPosBlock; i += kBlock) {
      const int h = i / kPosBlock, j = i % kPosBlock, t = t0 + j;
      float s = -INFINITY;
      if (t < t_end) {
        const int page = bt[static_cast<size_t>(b) * maxpg + t / ps];
        if (page >= 0 && page < num_pages) {
          const uint16_t* krow = kv + static_cast<size_t>(page) * 2 * plane + (static_cast<size_t>(kvh) * ps + t % ps) * D;
          float acc = 0.f;
          for (int d = 0; d < D; ++d) acc = fmaf(qs[h][d], bf16f(krow[d]), acc);
          s = acc;
        } else {
          atomicExch(err, MK_ERR_DEVICE_BOUNDS);
        }
      }
      sc[h][j] = s;
    }
    __syncthreads();
    if (tid < G) {
      float mx = mrun[tid];
      for (int j = 0; j < kPosBlock; ++j) mx = fmaxf(mx, sc[tid][j]);
      const float c = mrun[tid] == -INFINITY ? 0.f : __expf(mrun[tid] - mx);
      float sum = 0.f;
      for (int j = 0; j < kPosBlock; ++j) {
        const float pj = sc[tid][j] == -INFINITY ? 0.f : __expf(sc[tid][j] - mx);
        sc[tid][j] = pj;
        sum += pj;
      }
      corr[tid] = c;
      lrun[tid] = lrun[tid] * c + sum;
      if (mx != -INFINITY) mrun[tid] = mx;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = tid + kBlock * i;
      if (idx < G * D) {
        const int h = idx / D, d = idx % D;
        float acc = o[i] * corr[h];
        for (int j = 0; j < kPosBlock; ++j) {
          const float pj = sc[h][j];
          if (pj != 0.f) {
            const int t = t0 + j;
            const int page = bt[static_cast<size_t>(b) * maxpg + t / ps];
            const uint16_t* vrow =
                kv + static_cast<size_t>(page) * 2 * plane + plane + (static_cast<size_t>(kvh) * ps + t % ps) * D;
            acc = fmaf(pj, bf16f(vrow[d]), acc);
          }
        }
        o[i] = acc;
      }
    }
    __syncthreads();
  }
  float* dst = part + ((static_cast<size_t>(b) * Hkv + kvh) * nrange + r) * G * (D + 2);
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int idx = tid + kBlock * i;
    if (idx < G * D) {
      const int h = idx / D, d = idx % D;
      dst[h * (D + 2) + d] = o[i];
    }
  }
  if (tid < G) {
    dst[tid * (D + 2) + D] = mrun[tid];
    dst[tid * (D + 2) + D + 1] = lrun[tid];
  }
}

// One block per (KV head, row): merge the ranges in range order.
template <int D>
__global__ void __launch_bounds__(kBlock) merge_kernel(int Hq, int Hkv, int nrange, const float* __restrict__ scratch,
                                                       float* __restrict__ out, int32_t* status_out) {
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int G = Hq / Hkv;
  const float* part = scratch + kHeaderFloats + (static_cast<size_t>(b) * Hkv + kvh) * nrange * G * (D + 2);
  for (int idx = threadIdx.x; idx < G * D; idx += kBlock) {
    const int h = idx / D, d = idx % D;
    float M = -INFINITY;
    for (int r = 0; r < nrange; ++r) M = fmaxf(M, part[(r * G + h) * (D + 2) + D]);
    float L = 0.f, acc = 0.f;
    for (int r = 0; r < nrange; ++r) {
      const float* pr = part + (r * G + h) * (D + 2);
      const float f = pr[D] == -INFINITY ? 0.f : __expf(pr[D] - M);
      L += f * pr[D + 1];
      acc = fmaf(f, pr[d], acc);
    }
    // a row none of whose pages was in range has no positions (L == 0): it gets zeros, and the
    // bounds error in the scratch's error word is its only report
    out[(static_cast<size_t>(b) * Hq + kvh * G + h) * D + d] = L > 0.f ? acc / L : 0.f;
  }
  if (status_out != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    *status_out = *reinterpret_cast<const int*>(scratch);
}

int fail(int code, const char* text) {
  mk::set_last_error(code, text);
  return code;
}

// Device address of the scratch array on the current device, looked up once per device.
int scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MK_ERR_UNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return fail(MK_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<float*>(g_scratch_addr[dev]);
  return MK_OK;
}

}  // namespace

extern "C" int mk_paged_attention_noalloc(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                          int32_t page_size, int32_t num_pages, int32_t max_pages_per_seq,
                                          const float* q, const int32_t* seq_lens, const int32_t* block_tables,
                                          const void* kv_layer, float* out, int32_t* status_out, mk_stream_t stream) {
  mk::set_last_error(MK_OK, "");
  if (batch < 1 || batch > kMaxRows) return fail(MK_ERR_INVALID_ARG, "batch outside 1..64");
  if (num_q_heads < 1 || num_kv_heads < 1 || page_size < 1 || num_pages < 1 || max_pages_per_seq < 1)
    return fail(MK_ERR_INVALID_ARG, "sizes must be > 0");
  if (num_q_heads % num_kv_heads) return fail(MK_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  if (head_dim != 64 && head_dim != 128) return fail(MK_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  const int G = num_q_heads / num_kv_heads;
  if (G > 8) return fail(MK_ERR_UNSUPPORTED, "more than 8 query heads per KV head");
  if (!seq_lens) return fail(MK_ERR_INVALID_ARG, "seq_lens is NULL");
  RowLens lens;
  int max_npg = 0;
  const int64_t max_len = static_cast<int64_t>(max_pages_per_seq) * page_size;
  // positions and page offsets are 32-bit on the device
  if (max_len > (int64_t(1) << 30)) return fail(MK_ERR_UNSUPPORTED, "max_pages_per_seq*page_size above 2^30");
  for (int b = 0; b < batch; ++b) {
    if (seq_lens[b] < 1 || seq_lens[b] > max_len) return fail(MK_ERR_INVALID_ARG, "a seq_len is outside 1..max_pages_per_seq*page_size");
    lens.len[b] = seq_lens[b];
    max_npg = std::max(max_npg, (seq_lens[b] + page_size - 1) / page_size);
  }
  // ranges per (row, KV head) so that the partials fit the scratch
  const size_t per_range = static_cast<size_t>(batch) * num_kv_heads * G * (head_dim + 2) * sizeof(float);
  const size_t room = kNoAllocScratchBytes - kHeaderFloats * sizeof(float);
  if (per_range > room) {
    char msg[200];
    snprintf(msg, sizeof msg, "batch x heads needs %zu bytes of scratch per range; the fixed scratch holds %zu",
             per_range, room);
    return fail(MK_ERR_UNSUPPORTED, msg);
  }
  int nrange = static_cast<int>(std::min<size_t>(room / per_range, 64));
  nrange = std::min(nrange, max_npg);
  const int pages_per_range = (max_npg + nrange - 1) / nrange;
  nrange = (max_npg + pages_per_range - 1) / pages_per_range;
  if (!q || !block_tables || !kv_layer || !out) return fail(MK_ERR_INVALID_ARG, "a pointer argument is NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(kv_layer) |
       reinterpret_cast<uintptr_t>(block_tables)) & 3u)
    return fail(MK_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
  float* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(scratch, 0, kHeaderFloats * sizeof(float), s);   // the error word starts at zero
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, cudaGetErrorString(e));
  const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim)));
  const dim3 g1(nrange, num_kv_heads, batch), g2(num_kv_heads, batch);
  const uint16_t* kv = static_cast<const uint16_t*>(kv_layer);
  if (head_dim == 128) {
    split_kernel<128><<<g1, kBlock, 0, s>>>(q, kv, block_tables, lens, num_q_heads, num_kv_heads, page_size, num_pages,
                                            max_pages_per_seq, pages_per_range, nrange, scale, scratch);
    merge_kernel<128><<<g2, kBlock, 0, s>>>(num_q_heads, num_kv_heads, nrange, scratch, out, status_out);
  } else {
    split_kernel<64><<<g1, kBlock, 0, s>>>(q, kv, block_tables, lens, num_q_heads, num_kv_heads, page_size, num_pages,
                                           max_pages_per_seq, pages_per_range, nrange, scale, scratch);
    merge_kernel<64><<<g2, kBlock, 0, s>>>(num_q_heads, num_kv_heads, nrange, scratch, out, status_out);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MK_ERR_CUDA, cudaGetErrorString(e));
  return MK_OK;
}
