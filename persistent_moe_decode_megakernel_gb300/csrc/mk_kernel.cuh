// mk_kernel.cuh -- the persistent decode-step kernel for GB300 (sm_103a).
//
// One thread block per SM stays resident for the whole step ("Inside the
// megakernel serving engine for North Mini Code", section "What is a
// Megakernel?").  Each block walks its own host-built task list.  A task waits
// for the tiles that produce what it reads, not for a whole phase: every value
// one block hands to another is an 8-byte tagged word -- the fp32 or int32 value and this step's
// tag, written with one relaxed store -- and the reader polls the words it
// needs until they carry the step's tag.  No counter, fence or barrier sits
// between blocks; every wait is bounded by a %globaltimer watchdog that records
// an error and ends the step.
//
// Block layout: two consumer warpgroups and one producer warpgroup.  One
// producer thread streams the operand each tile reads from HBM -- weight rows
// with 1-D bulk copies, KV pages with 2-D TMA boxes (128-byte swizzle) -- into a
// two-slot shared-memory ring (completion on mbarriers, L2 evict-first).
// Weights never depend on activations and the cached KV never depends on this
// step, so the producer runs ahead across every data wait; its only wait is for
// the layer's routing, because expert weights are chosen by it.  The producer
// warpgroup hands its registers to the consumers (setmaxnreg).
//
// Consumers: GEMV rows on CUDA cores in fp32 at batches of 1-2 rows (RMSNorm
// fused into the staging of the input), mma.sync tensor-core tiles for wider
// batches; paged GQA attention on mma.sync tiles with an online softmax.
//
// Work kinds (task list entries, see mk_debug.h), per layer:
//   QKV     RMSNorm + fused QKV rows               reads the layer input (all rows)
//   ATTN    this block's split items of the step's attention plan: RoPE, the KV
//           append (split 0), partial (max, sum, output) per split
//                                                  reads q, k, v of its (row, KV head)
//           then the block merges a slice of the outputs of every pair it holds a
//           split of, over all that pair's splits   reads their partials
//   OPROJ   O-proj rows + residual                 reads the attention output (all)
//   ROUTER  RMSNorm + router rows (a few experts)  reads x after attention (all)
//   MOE     every block routes the batch itself from the router logits (softmax,
//           top-k, weights, active experts, a cost-balanced split of the gate/up
//           units over the blocks) and hands the result to its producer; then
//           small batches: the block's gate/up units and the same FFN rows of the
//             transposed down projection, an on-chip [B][H] partial, published and
//             summed per hidden row by the row's owner block  reads every block's partial
//           wider batches: gate/up units -> SwiGLU outputs; down projection by
//             hidden rows of every active expert      reads every unit's SwiGLU outputs
//   HEAD    final RMSNorm + LM-head rows           reads the last layer's output (all)
// The last block to finish clears the step's flags (abort, finish count).

#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "mk_layout.h"

namespace mk {
namespace {  // internal linkage: each instantiation unit gets its own copy

// --------------------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(tx) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// 2-D tiled TMA load of box (x, y) of the tensor map into shared memory (completion on an mbarrier)
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], "
      "[%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// 3-D tiled TMA load of box (x, y, z) of the tensor map into shared memory (completion on an mbarrier)
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z, uint64_t* bar,
                                            uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, "
      "%4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// 4-D tiled TMA load of box (x, y, z, w) of the tensor map into shared memory (completion on an mbarrier)
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int x, int y, int z, int w,
                                            uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, "
      "%4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a(16x16 bf16, row) * b(16x8 bf16, col), fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// Signed bytes -> fp16, exactly: with its sign bit flipped a byte b is the unsigned b + 128, and
// the fp16 whose high byte is 0x64 and low byte is u has the value 1024 + u; subtracting 1152
// leaves b.  (fp16 keeps every integer below 2048 exactly.)
__device__ __forceinline__ uint32_t s8_to_f16x2(uint32_t x, uint32_t sel) {   // the two bytes sel picks
  const uint32_t h = __byte_perm(x ^ 0x80808080u, 0x64646464u, sel);
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), __half2half2(__ushort_as_half(0x6480u)));
  return *reinterpret_cast<const uint32_t*>(&v);
}
// the two signed bytes in the low half of u (first in bits 0-7) -> f16x2
__device__ __forceinline__ uint32_t s8x2_f16x2(uint32_t u) { return s8_to_f16x2(u, 0x4140u); }
// d += a(16x16 f16, row) * b(16x8 f16, col), fp32 accumulate (a pure register operation: the
// compiler may schedule it freely)
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// two floats -> f16x2 (first in the low half), and the f16x2 of what rounding left over
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const __half2 r = __floats2half2_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}
// ---- tcgen05: 5th-generation tensor cores, accumulators in tensor memory ----------------------
// Shared-memory matrix descriptor of a K-major operand with the 128-byte swizzle: start address,
// (unused) leading offset, 1024 bytes between 8-row groups, descriptor version 1, swizzle mode 2.
// Advancing K by 16 bf16 within the 128-byte swizzle row adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16 with bf16 A and B (both K-major) and an fp32 accumulator
__device__ __forceinline__ uint32_t tc_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// D (tensor memory) = A * B^T, or += when acc
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc)));
}
// the same, issued by one elected lane of a converged warp (the whole warp computes the operands,
// so that they are warp-uniform)
__device__ __forceinline__ void tc_mma_elect(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc)));
}
__device__ __forceinline__ void tc_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
// one arrival on bar once every tensor-core operation this thread issued so far has completed
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 8 consecutive accumulator columns of this warp's 32 lanes (one per thread), waited for
__device__ __forceinline__ void tc_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float f16_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }
// two floats -> bf16x2 (first in the low half), and the bf16x2 of what rounding left over
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 r = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}
// two floats -> three bf16x2 terms (high, middle, low) whose sum keeps the floats' 24-bit
// significands: each term is the bf16 rounding of what the previous ones left over
__device__ __forceinline__ void split3_bf16x2(float a, float b, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float a1 = a - __low2float(h), b1 = b - __high2float(h);
  const __nv_bfloat162 m = __floats2bfloat162_rn(a1, b1);
  const __nv_bfloat162 r = __floats2bfloat162_rn(a1 - __low2float(m), b1 - __high2float(m));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  mid = *reinterpret_cast<const uint32_t*>(&m);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}
// L2 prefetch of a contiguous byte range (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// ---- tagged 8-byte words: value in the low half, step tag in the high half
__device__ __forceinline__ uint64_t ll_pack(float v, uint32_t tag) {
  return static_cast<uint64_t>(__float_as_uint(v)) | (static_cast<uint64_t>(tag) << 32);
}
__device__ __forceinline__ void ll_st(uint64_t* p, float v, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(ll_pack(v, tag)) : "memory");
}
__device__ __forceinline__ void ll_st2(uint64_t* p, float a, float b, uint32_t tag) {   // 16-byte aligned
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(ll_pack(a, tag)), "l"(ll_pack(b, tag))
               : "memory");
}
// Tagged loads are volatile (never merged or hoisted out of a polling loop) but carry no
// memory clobber, so the compiler may issue a batch of them before the first is used:
// each word is validated by its own tag, not by ordering against other accesses.
__device__ __forceinline__ uint64_t ll_ld(const uint64_t* p) {
  uint64_t x;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(x) : "l"(p));
  return x;
}
__device__ __forceinline__ void ll_ld2(const uint64_t* p, uint64_t& a, uint64_t& b) {   // 16-byte aligned
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}
__device__ __forceinline__ bool ll_ok(uint64_t x, uint32_t tag) { return static_cast<uint32_t>(x >> 32) == tag; }
__device__ __forceinline__ float ll_f(uint64_t x) { return __uint_as_float(static_cast<uint32_t>(x)); }

__device__ __forceinline__ void cbar() {  // all consumer threads
  __syncwarp();
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}
// barrier over the consumer threads that also ANDs a flag
__device__ __forceinline__ bool cbar_and(bool v) {
  uint32_t r;
  __syncwarp();
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kConsumerThreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf1(uint16_t u) { return __uint_as_float(static_cast<uint32_t>(u) << 16); }
__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
__device__ __forceinline__ uint16_t to_bf16_bits(float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&h);
}
// DL consecutive bf16 values of a K or V row in shared memory -> fp32
template <int DL>
__device__ __forceinline__ void unpack_row(const uint16_t* src, float (&out)[DL]) {
  if constexpr (DL == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(src);
    out[0] = bf_lo(w.x); out[1] = bf_hi(w.x); out[2] = bf_lo(w.y); out[3] = bf_hi(w.y);
  } else {
    static_assert(DL == 2, "head_dim 64 or 128");
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
    out[0] = bf_lo(w); out[1] = bf_hi(w);
  }
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Greedy selection state over (value, index) pairs: m1 the largest value, i1 its lowest index,
// m2 the largest value at any other index.
struct Top2 {
  float m1, m2;
  int i1;
};
__device__ __forceinline__ void top2_add(Top2& t, float v, int i) {
  if (v > t.m1 || (v == t.m1 && i < t.i1)) { t.m2 = t.m1; t.m1 = v; t.i1 = i; }
  else t.m2 = fmaxf(t.m2, v);
}
__device__ __forceinline__ void top2_merge(Top2& t, const Top2& o) {   // (m1 >= m2 on both sides)
  if (o.m1 > t.m1 || (o.m1 == t.m1 && o.i1 < t.i1)) {
    t.m2 = fmaxf(t.m1, o.m2);
    t.m1 = o.m1;
    t.i1 = o.i1;
  } else {
    t.m2 = fmaxf(t.m2, o.m1);
  }
}
__device__ __forceinline__ void top2_warp(Top2& t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Top2 x;
    x.m1 = __shfl_xor_sync(0xffffffffu, t.m1, o);
    x.m2 = __shfl_xor_sync(0xffffffffu, t.m2, o);
    x.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
    top2_merge(t, x);
  }
}

// Two warp sums at once (a[tb] and b[tb] for every tb): afterwards lanes 0-15 hold the sums
// of a and lanes 16-31 the sums of b.  Five shuffles per tb instead of ten.
template <int TB>
__device__ __forceinline__ void warp_sum2(float (&a)[TB], const float (&b)[TB]) {
  const bool hi = (threadIdx.x & 16) != 0;
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) {
    float keep = hi ? b[tb] : a[tb];
    const float send = hi ? a[tb] : b[tb];
    keep += __shfl_xor_sync(0xffffffffu, send, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
    a[tb] = keep;
  }
}

// Division by a divisor fixed for a loop (1 <= d < 2^16), exact for 0 <= n < 2^16: with
// m = ceil(2^32 / d) = m * d - 2^32 + ... the error term e = m * d - 2^32 < d, and n * e < 2^32,
// so floor(n * m / 2^32) = floor(n / d).  One wide multiply instead of a division routine.
struct FastDiv {
  uint32_t d;
  uint64_t m;
  __device__ __forceinline__ explicit FastDiv(int d_) : d(static_cast<uint32_t>(d_)), m(0xffffffffull / static_cast<uint32_t>(d_) + 1ull) {}
  __device__ __forceinline__ int div(int n) const { return static_cast<int>((static_cast<uint64_t>(n) * m) >> 32); }
};

// The per-tile timeline (mk_debug_trace) exists only in builds with MK_TRACE=1; elsewhere every
// trace write folds away at compile time.
__device__ __forceinline__ bool tr_on(const Params& p) { return kTrace && p.trace != nullptr; }

// --------------------------------------------------------------------------- shared memory
constexpr int kCmbItems = 16;   // split items one attention merge group takes at most
enum : uint8_t { R_EMBED = 1, R_GEMV = 2, R_ATTN = 3, R_GU = 4, R_DOWN = 5, R_END = 6, R_ROUTE = 7,
                 R_DT = 9, R_RED = 10,    // small-batch MoE: transposed down rows; partial-sum reduction
                 R_TC = 11,               // wide batch: a tcgen05 GEMV chunk
                 R_YRED = 12 };           // wide batch: sum the per-slot down-projection outputs of own rows
// GEMV stream kinds beyond the task ops (MK_OP_QKV / OPROJ / ROUTER / HEAD)
enum : int { R_OP_GU = 100 };

struct Meta {
  uint8_t kind, op, first, last;
  uint16_t layer, n;     // rows (GEMV/GU/DOWN) or pages (ATTN) in this chunk
  uint32_t row0;         // first row / FFN row / hidden row / page index of the chunk
  uint32_t idx;          // task index (GEMV/EMBED) / item index (ATTN) / active expert (GU/DOWN)
  uint32_t e;            // expert id (GU/DOWN)
  uint32_t aux;          // row tile (DOWN)
  uint32_t lo, hi;       // tile range
  uint32_t pad[8];       // pad[0..1]: issue time of the record (timeline builds)
};
static_assert(sizeof(Meta) == 64, "meta size");


struct __align__(1024) Smem {
  uint8_t ring[kSlots][kSlotBytes];
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  Meta meta[kSlots];
  union {
    float seg[2][kMaxRowsPerChunk][kConsumerWarps][4];   // GEMV segment sums [record parity][row][segment][batch row]
    float attn[kAttnScratch];
  } scr;
  float rstd[kMaxBatch];
  float ssred[kConsumerWarps][4];
  int32_t slot_of[kMaxBatch];
  int32_t rids[kMaxBatch * kMaxTopK];
  float rval[kMaxBatch * kMaxTopK];
  float rmax[kMaxBatch], rz[kMaxBatch], rsum[kMaxBatch];
  int32_t ecnt[kMaxExperts];
  int32_t rcache[kMaxBatch * kMaxTopK];   // this layer's routing ids, cached by the first MoE item of the block
  float rwcache[kMaxBatch * kMaxTopK];    // and their combine weights
  // routing: logits; down projection: products, x_mid, SwiGLU inputs; tcgen05 tiles: the staged
  // input slices (1024-byte aligned for the 128-byte swizzle)
  alignas(1024) float moe[kMoeScratch];
  int32_t wlist[kConsumerWarps][kMaxBatch];   // per warp: (row, slot) pairs routed to one expert
  int32_t elist[kMaxBatch];               // gate/up run: (row, slot) pairs routed to its expert
  int32_t eact[kMaxExperts];              // this layer's active experts, ascending
  int32_t ecost[kMaxExperts];             // cost of one gate/up unit of each, and the cost prefix
  int32_t ecum[kMaxExperts + 1];
  int32_t nact;
  int32_t gu_lo, gu_hi;                   // this block's gate/up units
  float hsm[kSmallMaxB * kMaxUnits];      // small-batch MoE: weighted SwiGLU outputs of this block's units
  uint64_t route_bar;                     // consumers -> producer: routing of the layer is in shared memory
  int32_t ykey;                           // layer whose normalised MoE input scr.attn holds, or -1
  uint32_t prod_count, cons_count;
  int32_t flag;
  int32_t is_last;
  uint32_t tag;          // this step's tag, read from the uploaded step data
  // tcgen05 tiles: the consumers post one request per staged input slice; one warp of the producer
  // warpgroup issues its MMAs
  struct TcReq {
    uint32_t a;       // shared address of the slice's first A unit (units of an M-block consecutive)
    uint32_t x;       // shared address of the input buffer (terms bp * 128 bytes apart)
    uint32_t d;       // tensor-memory address of the first M-block's accumulators
    uint32_t idesc;
    uint32_t nmc, nu; // M-blocks, A units per M-block (2: gate, up)
    uint32_t ustride; // bytes between A units
    uint32_t dstride, dunit;   // accumulator columns between M-blocks, between a block's units
    uint32_t dh, dlo; // high-term accumulator, first lower-term accumulator (columns from a unit's)
    uint32_t bp;      // N columns (and rows of an input term)
    uint32_t flags;   // 1 accumulate high, 2 accumulate lower, 4 release the ring record, 8 stop, T << 4,
                      // (buffer + 1) << 8, 1 << 16 the pass's last request, ring slot << 20
    uint32_t pad_[3];
  };
  TcReq tcreq[kTcReqs];
  uint64_t reqbar[kTcReqs]; // consumers (all) -> issuer: request i is written and its slice staged
  uint64_t ackbar[kTcReqs]; // issuer -> consumers: request i has been read
  uint64_t xbar[kTcXBufs];  // tcgen05 tiles: the tensor cores have read input slice buffer i
  uint64_t wbar;            // tcgen05 tiles: the tensor cores have read the issuer's current record
  uint64_t pbar;            // tcgen05 tiles: the current pass's MMAs have completed (issuer -> consumers)
  uint32_t tmem_base;       // tensor-memory address of this block's accumulators (wide batches)
  // attention merge: the split items of the group being merged (gathered words from g0, split
  // scales from fs in the scratch; att: the output's word offset; m: FastDiv multiplier of nsl)
  struct CmbItem {
    int32_t g0, ns, o0, nsl, fs, first, att, pad_;
    uint64_t m;
  };
  CmbItem cmb[kCmbItems];
};

static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory (with the 1024-byte alignment pad) exceeds 227 KB");

// --------------------------------------------------------------------------- errors / waits
// wait: MK_WAIT_* for a timeout (what the wait was on), 0 for a bounds error; observed: the ring
// record (timeout on the ring) or the bad value (bounds); tag: the step tag a data wait needed
__device__ __noinline__ void record_error(const Params& p, int code, int op, int layer, uint32_t wait, uint32_t observed,
                             uint32_t tag, int detail, bool abort) {
  if (atomicCAS(&p.status->code, 0, code) == 0) {
    p.status->op = op;
    p.status->layer = layer;
    p.status->cta = blockIdx.x;
    p.status->wait = wait;
    p.status->observed = observed;
    p.status->tag = tag;
    p.status->detail = detail;
    __threadfence();
  }
  if (abort) atomicExch(&p.flags[F_ABORT], 1u);
}

__device__ __forceinline__ bool aborted(const Params& p) {
  return *reinterpret_cast<const volatile uint32_t*>(&p.flags[F_ABORT]) != 0u;
}

// A tagged read that found a stale tag re-polls the word in place (no call, so that the
// registers of the surrounding unrolled code stay put), bounded by the watchdog and
// giving up if another block aborted the step; ok turns false when it gives up, and the
// caller records the timeout once (ll_timeout) outside its hot loops.
#define LL_FIX(x, ptr, tag, op, layer, ok)                                                  \
  do {                                                                                      \
    if (!ll_ok((x), (tag))) {                                                               \
      const uint64_t t0_ = globaltimer();                                                   \
      for (uint32_t it_ = 1;; ++it_) {                                                      \
        (x) = ll_ld(ptr);                                                                   \
        if (ll_ok((x), (tag))) break;                                                       \
        if ((it_ & 15u) == 0u && (aborted(p) || globaltimer() - t0_ > p.watchdog_ns)) {     \
          (ok) = false;                                                                     \
          break;                                                                            \
        }                                                                                   \
      }                                                                                     \
    }                                                                                       \
  } while (0)

__device__ __noinline__ void ll_timeout(const Params& p, int op, int layer, uint32_t tag) {
  record_error(p, MK_ERR_TIMEOUT, op, layer, MK_WAIT_DATA, 0, tag, -1, true);
}

// A batch of tagged loads written between LL_RETRY_BEGIN and LL_RETRY_END(ok) ORs the
// stale-tag bits of every word it reads into st_; the batch runs again until one pass sees
// only current tags (bounded by the watchdog and the abort flag; ok turns false when it
// gives up).  The first pass is the common case.  Plain loops, no closures: the
// destinations stay in registers.
#define LL_RETRY_BEGIN                  \
  {                                     \
    uint64_t t0_ = 0;                   \
    for (uint32_t it_ = 0;; ++it_) {    \
      uint32_t st_ = 0;
#define LL_RETRY_END(ok)                                                                  \
      if (st_ == 0u) break;                                                               \
      if (it_ == 0u) {                                                                    \
        t0_ = globaltimer();                                                              \
      } else if ((it_ & 15u) == 0u && (aborted(p) || globaltimer() - t0_ > p.watchdog_ns)) { \
        (ok) = false;                                                                     \
        break;                                                                            \
      }                                                                                   \
    }                                                                                     \
  }
// True once the watchdog has run out for a wait that started at t0, or the step was aborted.
__device__ __noinline__ bool ll_expired(const Params& p, uint64_t t0) {
  return aborted(p) || globaltimer() - t0 > p.watchdog_ns;
}

// Gather n tagged words into shared-memory floats: dst[i] = value of word addr(i), i over
// this thread's indices threadIdx.x + k * kConsumerThreads.  Loads go out kB at a time (8: the
// body is inlined at every call site, and instruction fetch of the step's short phases is
// dear: 16 at a time measured 9 % slower at batch 1, 4 at a time 1 % slower); a
// batch is issued again for the words whose tags were stale, all of them at once, until
// every word is current (one loaded L2 round trip per pass, the same code for the first and
// the later passes).  False if the watchdog or an abort ended the wait.
template <int kB = 8, class Addr>
__device__ __forceinline__ bool ll_gather(const Params& p, int n, Addr addr, float* dst, uint32_t tag) {
  #pragma unroll 1
  for (int base = threadIdx.x; base < n; base += kB * kConsumerThreads) {
    uint32_t want = kB >= 32 ? 0xffffffffu : (1u << kB) - 1u;   // words of this batch not yet seen with the step's tag
    uint64_t t0 = 0;
    #pragma unroll 1
    for (uint32_t it = 0;; ++it) {
      uint64_t x[kB];
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        const int i = base + k * kConsumerThreads;
        x[k] = (i < n && ((want >> k) & 1u)) ? ll_ld(addr(i)) : 0ull;
      }
      uint32_t stale = 0;
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        const int i = base + k * kConsumerThreads;
        if (i < n && ((want >> k) & 1u)) {
          if (ll_ok(x[k], tag)) dst[i] = ll_f(x[k]);
          else stale |= 1u << k;
        }
      }
      want = stale;
      if (want == 0u) break;
      if (it == 0u) t0 = globaltimer();
      else if ((it & 15u) == 0u && ll_expired(p, t0)) return false;
    }
  }
  return true;
}

// stale-tag bits of a word (0 when current)
__device__ __forceinline__ uint32_t ll_stale(uint64_t x, uint32_t tag) { return static_cast<uint32_t>(x >> 32) ^ tag; }

// one warp: wait until record c has landed in its slot.  Warps consume records
// independently; false (warp-uniform) if the step was aborted meanwhile.
__device__ bool warp_wait_record(const Params& p, Smem& S, uint32_t c) {
  const int s = static_cast<int>(c % kSlots);
  const uint32_t ph = (c / kSlots) & 1u;
  bool ok = mbar_try_wait(&S.full[s], ph);
  if (!ok) {
    const uint64_t t0 = globaltimer();
    #pragma unroll 1
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(&S.full[s], ph)) { ok = true; break; }
      if ((it & 63u) == 0u) {
        if (aborted(p)) break;
        if (globaltimer() - t0 > p.watchdog_ns) {
          if ((threadIdx.x & 31) == 0) record_error(p, MK_ERR_TIMEOUT, 0, -1, MK_WAIT_RING, c, 0, -1, true);
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// one warp: done reading record c's slot
__device__ __forceinline__ void warp_release_record(Smem& S, uint32_t c) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&S.empty[c % kSlots]);
}

// barrier over the group of `nw` consecutive warps containing this warp (nw in {1, 2, 4, 8}) that ANDs a flag
__device__ __forceinline__ bool group_bar_and(bool v, int nw) {
  if (nw == 1) return __all_sync(0xffffffffu, v);
  if (nw == kConsumerWarps) return cbar_and(v);
  uint32_t r;
  const uint32_t id = 2u + static_cast<uint32_t>((threadIdx.x >> 5) / nw);
  const uint32_t cnt = 32u * static_cast<uint32_t>(nw);
  __syncwarp();
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(cnt)
      : "memory");
  return r != 0;
}

// --------------------------------------------------------------------------- tcgen05 split-K
// The rows of this block's split-K group (KS consecutive blocks) of a dense tile kind.
__device__ __forceinline__ void tc_group_rows(const Params& p, int op, int KS, uint32_t& glo, uint32_t& ghi) {
  const int g0 = (static_cast<int>(blockIdx.x) / KS) * KS, g1 = g0 + KS;
  if (op == MK_OP_ROUTER) {
    const int rr = router_tile_rows(p.E, p.n_ctas, p.max_batch);
    glo = static_cast<uint32_t>(g0 * rr);
    ghi = static_cast<uint32_t>(min(p.E, g1 * rr));
  } else {
    const uint64_t n = op == MK_OP_QKV ? static_cast<uint64_t>(p.nqkv) : static_cast<uint64_t>(p.H);
    glo = static_cast<uint32_t>(n * g0 / p.n_ctas);
    ghi = static_cast<uint32_t>(n * g1 / p.n_ctas);
  }
}

// --------------------------------------------------------------------------- producer
// Q8: the KV pool holds q8_0 blocks (codes and scales) instead of bf16 values.  TC: the
// tcgen05 paths of wide batches are compiled in (the widest instantiation only: the code the
// narrower kernels never run would still cost them instruction fetch).  SMALL: the small-batch
// MoE path, the only one of the narrow instantiations (the host launches the widest one for
// every step that cannot take it).
template <bool Q8, bool TC, bool SMALL>
struct Producer {
  const Params& p;
  Smem& S;
  uint32_t c = 0;
  uint32_t pev = 0;   // producer trace events (written from the end of the block's trace area)
  uint32_t rphase = 0;  // parity of the next routing hand-over from the consumers
  uint64_t pol, pol_reuse;
  __device__ Producer(const Params& p_, Smem& S_) : p(p_), S(S_) {
    pol = policy_evict_first();
    pol_reuse = policy_evict_normal();
  }

  // Warm L2 with (at most kPrefetchBytes of) a task's weights or KV pages, so that the ring's
  // copies of a phase that starts after a dependency wait come from L2.  Done for the block's
  // first task only: one task ahead throughout the step measured 0.8 % slower at batch 1
  // (its code, fetched every task, costs more than the warm copies save).
  static constexpr uint32_t kPrefetchBytes = 256u * 1024u;
  __device__ void prefetch_task(const mk_task& t) {
    switch (t.op) {
      case MK_OP_QKV:
      case MK_OP_OPROJ:
      case MK_OP_ROUTER:
      case MK_OP_HEAD: {
        const LayerW& lw = p.layers[t.op == MK_OP_HEAD ? 0 : t.layer];
        const uint16_t* W = t.op == MK_OP_QKV ? lw.w_qkv : t.op == MK_OP_OPROJ ? lw.w_o
                          : t.op == MK_OP_ROUTER ? lw.w_router : p.lm_head;
        const int K = t.op == MK_OP_OPROJ ? p.Hq * p.D : p.H;
        const uint64_t bytes = static_cast<uint64_t>(t.hi - t.lo) * K * 2u;
        prefetch_l2(W + static_cast<size_t>(t.lo) * K, static_cast<uint32_t>(bytes < kPrefetchBytes ? bytes : kPrefetchBytes));
        break;
      }
      case MK_OP_ATTN: {
        const int cta = blockIdx.x;
        // one page of K (or V) of one KV head (q8_0: its codes; the small scale runs are not warmed)
        const uint32_t blk = static_cast<uint32_t>(p.ps) * p.D * (Q8 ? 1u : 2u);
        uint32_t done = 0;
        #pragma unroll 1
        for (int it = p.item_off[cta]; it < p.item_off[cta + 1] && done < kPrefetchBytes; ++it) {
          const mk_attn_item item = p.items[it];
          const int32_t* btrow = p.block_tables + static_cast<size_t>(item.b) * p.maxpg;
          #pragma unroll 1
          for (uint32_t pg = item.page_lo; pg < item.page_hi && done < kPrefetchBytes; ++pg) {
            const int32_t page = btrow[pg];
            if (page < 0 || page >= p.P) continue;
            if constexpr (Q8) {
              const uint8_t* base = reinterpret_cast<const uint8_t*>(p.kv) + t.layer * p.kv_layer_bytes;
              const size_t kb = ((static_cast<size_t>(page) * 2) * p.Hkv + item.kvh) * p.ps * p.D;
              prefetch_l2(base + kb, blk);
              prefetch_l2(base + kb + static_cast<size_t>(p.Hkv) * p.ps * p.D, blk);
            } else {
              const size_t kb = (((static_cast<size_t>(t.layer) * p.P + page) * 2) * p.Hkv + item.kvh) * p.ps * p.D;
              prefetch_l2(p.kv + kb, blk);
              prefetch_l2(p.kv + kb + static_cast<size_t>(p.Hkv) * p.ps * p.D, blk);
            }
            done += 2 * blk;
          }
        }
        break;
      }
      default: break;
    }
  }

  // wait for the slot of record c to be free; false if the step was aborted
  __device__ bool acquire() {
    const int s = static_cast<int>(c % kSlots);
    const uint32_t ph = ((c / kSlots) & 1u) ^ 1u;
    if (mbar_try_wait(&S.empty[s], ph)) return true;
    const uint64_t t0 = globaltimer();
    #pragma unroll 1
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(&S.empty[s], ph)) return true;
      if ((it & 63u) == 0u) {
        if (aborted(p)) return false;
        if (globaltimer() - t0 > p.watchdog_ns) {
          record_error(p, MK_ERR_TIMEOUT, 0, -1, MK_WAIT_RING, c, 0, -1, true);
          return false;
        }
      }
    }
  }
  __device__ Meta& meta() {
    Meta& m = S.meta[c % kSlots];
    if (tr_on(p)) {
      const uint64_t t = globaltimer();
      m.pad[0] = static_cast<uint32_t>(t);
      m.pad[1] = static_cast<uint32_t>(t >> 32);
    }
    return m;
  }
  __device__ uint8_t* slot() { return S.ring[c % kSlots]; }
  __device__ uint64_t* full() { return &S.full[c % kSlots]; }

  __device__ bool emit_control(uint8_t kind, const mk_task& t, uint32_t idx) {
    if (!acquire()) return false;
    Meta& m = meta();
    m.kind = kind; m.op = static_cast<uint8_t>(t.op); m.first = 1; m.last = 1;
    m.layer = t.layer; m.n = 0; m.row0 = t.lo; m.idx = idx; m.e = 0; m.aux = 0;
    m.lo = t.lo; m.hi = t.hi;
    mbar_arrive(full());
    ++c;
    return true;
  }

  __device__ bool gemv_tile(const mk_task& t, uint32_t ti) {
    const uint16_t* W;
    int K;
    const LayerW& lw = p.layers[t.op == MK_OP_HEAD ? 0 : t.layer];
    switch (t.op) {
      case MK_OP_QKV: W = lw.w_qkv; K = p.H; break;
      case MK_OP_OPROJ: W = lw.w_o; K = p.Hq * p.D; break;
      case MK_OP_ROUTER: W = lw.w_router; K = p.H; break;
      default: W = p.lm_head; K = p.H; break;
    }
    int rpc = gemv_rows_per_chunk(K);
    if (!SMALL && p.B > kSmallMaxB && rpc > 16) rpc &= ~15;   // tensor-core tiles of wide batches: whole 16-row tiles
    // A batch wider than one register group (groups of 4 rows) is served group-major: the tile
    // is streamed once per group (aux = group), so the consumers stage each group's input once
    // per tile; the repeated reads of the tile come from L2 (evict-normal while it is reused).
    const int ng = (!SMALL && p.B > 2) ? (p.B + wide_group_rows(K) - 1) / wide_group_rows(K) : 1;
    const uint64_t pl = ng > 1 ? pol_reuse : pol;
    #pragma unroll 1
    for (int g = 0; g < ng; ++g) {
      #pragma unroll 1
      for (uint32_t r0 = t.lo; r0 < t.hi; r0 += rpc) {
        const uint32_t n = min(static_cast<uint32_t>(rpc), t.hi - r0);
        if (!acquire()) return false;
        Meta& m = meta();
        m.kind = R_GEMV; m.op = static_cast<uint8_t>(t.op); m.first = (g == 0 && r0 == t.lo);
        m.last = (g == ng - 1 && r0 + n >= t.hi);
        m.layer = t.layer; m.n = static_cast<uint16_t>(n); m.row0 = r0; m.idx = ti; m.e = 0;
        m.aux = static_cast<uint32_t>(g);
        m.lo = t.lo; m.hi = t.hi;
        const uint32_t bytes = n * static_cast<uint32_t>(K) * 2u;
        mbar_arrive_expect_tx(full(), bytes);
        bulk_g2s(slot(), W + static_cast<size_t>(r0) * K, bytes, full(), g == ng - 1 ? pol : pl);
        ++c;
      }
    }
    return true;
  }

  // Wide batches on tcgen05: the tile's weight rows as A operand units of MB rows x 64 columns
  // (K-major, 128-byte swizzle; TMA boxes of 16 rows, rows past the tile left as they are: their
  // accumulator rows are never read).  Gate/up runs have two units per (slice, M-block): the
  // expert's gate rows, then the same FFN rows of its up projection.  A pass covers as many
  // M-blocks as the tensor memory holds accumulators for (accs per M-block, each MB rows x the
  // N columns); within a pass, records go slice by slice, each with up to kTcChunkBytes of
  // units: several slices of all the pass's M-blocks, or one slice of a group of M-blocks.
  // Meta: row0 the first M-block, n the M-blocks, aux the first slice | slices << 16, pad[2] the
  // pass's M-blocks (first | end << 16), pad[4] the N columns the passes were sized for.
  __device__ bool tc_emit(const mk_task& t, uint32_t ti, uint8_t op, const uint64_t* map, int K, int R, int y0, int y1,
                          int nu, int accs, int ncols, uint32_t e, uint32_t idx, uint32_t aux_flag, int s_lo = 0,
                          int s_hi = -1, uint32_t own_lo = 0, uint32_t own_hi = 0) {
    const int MB = tc_mblock(R), nmb = (R + MB - 1) / MB;
    const int pmb = min(nmb, kTcCols / (accs * ncols));
    const int upc = kTcChunkBytes / (nu * MB * 128);   // (slice, M-block) pairs per record
    const int ns = s_hi < 0 ? (K + 63) / 64 : s_hi;     // (the end of this block's slices)
    #pragma unroll 1
    for (int m0 = 0; m0 < nmb; m0 += pmb) {
      const int m1 = min(nmb, m0 + pmb), nm = m1 - m0;
      const int mg = nm < upc ? nm : upc;
      const int nsc = nm < upc ? upc / nm : 1;
      #pragma unroll 1
      for (int s0 = s_lo; s0 < ns; s0 += nsc) {
        const int s1 = min(ns, s0 + nsc);
        #pragma unroll 1
        for (int ma = m0; ma < m1; ma += mg) {
          const int mb1 = min(m1, ma + mg);
          if (!acquire()) return false;
          Meta& m = meta();
          m.kind = R_TC; m.op = op;
          m.first = (m0 == 0 && s0 == s_lo && ma == m0); m.last = (m1 == nmb && s1 == ns && mb1 == m1);
          m.layer = t.layer; m.n = static_cast<uint16_t>(mb1 - ma); m.row0 = static_cast<uint32_t>(ma);
          m.idx = idx; m.e = e;
          m.aux = static_cast<uint32_t>(s0) | (static_cast<uint32_t>(s1 - s0) << 16);
          m.lo = t.lo; m.hi = t.hi;
          m.pad[2] = static_cast<uint32_t>(m0) | (static_cast<uint32_t>(m1) << 16);
          m.pad[3] = aux_flag;
          m.pad[4] = static_cast<uint32_t>(ncols);
          m.pad[5] = own_lo;
          m.pad[6] = static_cast<uint32_t>(s_lo) | (static_cast<uint32_t>(ns) << 16);
          m.pad[7] = own_hi;
          uint32_t bytes = 0;
          #pragma unroll 1
          for (int mm = ma; mm < mb1; ++mm) bytes += static_cast<uint32_t>((min(MB, R - mm * MB) + 15) / 16) * 2048u;
          mbar_arrive_expect_tx(full(), bytes * static_cast<uint32_t>((s1 - s0) * nu));
          uint8_t* dst = slot();
          #pragma unroll 1
          for (int sl = s0; sl < s1; ++sl) {
            #pragma unroll 1
            for (int mm = ma; mm < mb1; ++mm) {
              const int rows = min(MB, R - mm * MB);
              #pragma unroll 1
              for (int un = 0; un < nu; ++un) {
                const int u = ((sl - s0) * (mb1 - ma) + (mm - ma)) * nu + un;
                const int y = (un == 0 ? y0 : y1) + mm * MB;
                #pragma unroll 1
                for (int j = 0; j * 16 < rows; ++j)
                  tma_load_2d(dst + u * MB * 128 + j * 2048, map, 64 * sl, y + 16 * j, full(), pol);
              }
            }
          }
          ++c;
        }
      }
    }
    return true;
  }
  __device__ bool tc_tile(const mk_task& t, uint32_t ti) {
    const int K = t.op == MK_OP_OPROJ ? p.Hq * p.D : p.H;
    const uint64_t* map = p.wmaps + static_cast<size_t>(tc_map_index(t.op, t.layer, p.L)) * 16;
    const int KS = tc_ksplit(t.op, p.n_ctas, p.n_router_tiles, t.op == MK_OP_QKV ? p.nqkv : p.H, K);
    const int ns = (K + 63) / 64;
    mk_task tt = t;
    int s_lo = 0, s_hi = ns;
    if (KS > 1) {   // the group's rows, this block's share of K
      tc_group_rows(p, t.op, KS, tt.lo, tt.hi);
      const int q = static_cast<int>(blockIdx.x) % KS;
      s_lo = q * ns / KS;
      s_hi = (q + 1) * ns / KS;
    }
    return tc_emit(tt, ti, static_cast<uint8_t>(t.op), map, K, static_cast<int>(tt.hi - tt.lo), static_cast<int>(tt.lo), 0,
                   1, tc_accs(t.op, p.B, K), tc_batch_cols(p.B), 0u, ti, static_cast<uint32_t>(KS), s_lo, s_hi, t.lo,
                   t.hi);
  }

  // Up to kIdBatch page ids of a chunk, read with independent loads (the block table is not
  // written during a step), so that their latencies overlap instead of adding up per page.
  static constexpr int kIdBatch = 8;
  __device__ __forceinline__ void page_ids(const int32_t* src, uint32_t n, int32_t (&ids)[kIdBatch]) const {
    #pragma unroll
    for (int j = 0; j < kIdBatch; ++j) ids[j] = static_cast<uint32_t>(j) < n ? __ldg(src + j) : 0;
  }
  // a page id outside the pool is recorded and replaced by page 0, which keeps the slot's byte
  // count; the step's result is then flagged invalid
  __device__ __forceinline__ int32_t checked_page(int32_t page, int layer, uint32_t pos) const {
    if (page < 0 || page >= p.P) {
      record_error(p, MK_ERR_DEVICE_BOUNDS, MK_OP_ATTN, layer, 0u, static_cast<uint32_t>(page), 0,
                   static_cast<int>(pos), false);
      return 0;
    }
    return page;
  }

  // KV pages of this block's attention items: one TMA box per page holds its K rows then its
  // V rows for the item's KV head, each as [dim half][position][64 dims] (128-byte swizzle);
  // page i of a chunk sits at i * 2 * page_size * D * 2 bytes of the slot.
  __device__ bool attn_items(const mk_task& t) {
    if constexpr (Q8) return attn_items_q8(t);
    const int cta = blockIdx.x;
    const int ppc = pages_per_chunk(p.ps, p.D);
    const uint32_t box = 2u * static_cast<uint32_t>(p.ps) * p.D * 2u;   // K and V of one page
    #pragma unroll 1
    for (int it = p.item_off[cta]; it < p.item_off[cta + 1]; ++it) {
      const mk_attn_item item = p.items[it];
      const int32_t* btrow = p.block_tables + static_cast<size_t>(item.b) * p.maxpg;
      #pragma unroll 1
      for (uint32_t pg = item.page_lo; pg < item.page_hi; pg += ppc) {
        const uint32_t n = min(static_cast<uint32_t>(ppc), item.page_hi - pg);
        int32_t ids[kIdBatch];
        page_ids(btrow + pg, n, ids);   // in flight across the slot wait
        if (!acquire()) return false;
        Meta& m = meta();
        m.kind = R_ATTN; m.op = MK_OP_ATTN; m.first = (pg == item.page_lo); m.last = (pg + n >= item.page_hi);
        m.layer = t.layer; m.n = static_cast<uint16_t>(n); m.row0 = pg; m.idx = static_cast<uint32_t>(it);
        m.e = 0; m.aux = 0; m.lo = item.page_lo; m.hi = item.page_hi;
        mbar_arrive_expect_tx(full(), n * box);
        uint8_t* dst = slot();
        #pragma unroll 1
        for (uint32_t i0 = 0; i0 < n; i0 += kIdBatch) {
          if (i0 > 0) page_ids(btrow + pg + i0, n - i0, ids);
          #pragma unroll
          for (int j = 0; j < kIdBatch; ++j) {
            const uint32_t i = i0 + j;
            if (i >= n) break;
            const int32_t page = checked_page(ids[j], t.layer, pg + i);
            tma_load_4d(dst + i * box, p.kv_map, 0, item.kvh * p.ps, 0, (t.layer * p.P + page) * 2, full(), pol);
          }
        }
        ++c;
      }
    }
    // the consumers then merge this block's share of every pair it holds a split of, with no
    // record of their own: both slots are free meanwhile for the weights of the next tile
    return true;
  }

  // q8_0 cache: per page, the K codes and V codes of the item's KV head (3-D TMA boxes of
  // page_size rows of head_dim bytes, 128-byte swizzle) and their scale runs (1-D bulk copies).
  // A slot holds [K codes][V codes][K scales][V scales], each for pages_per_chunk_q8 pages.
  __device__ bool attn_items_q8(const mk_task& t) {
    const int cta = blockIdx.x;
    const int ppc = pages_per_chunk_q8(p.ps, p.D);
    const int rows_cap = ppc * p.ps;
    const uint32_t cbox = static_cast<uint32_t>(p.ps) * p.D;                 // codes of one page, one head
    const uint32_t srow = static_cast<uint32_t>(p.D / 32) * 2u;              // scale bytes of one row
    const uint32_t sbox = static_cast<uint32_t>(p.ps) * srow;                // scales of one page, one head
    const uint8_t* sbase = reinterpret_cast<const uint8_t*>(p.kv) + t.layer * p.kv_layer_bytes + p.kv_code_bytes;
#pragma unroll 1
    for (int it = p.item_off[cta]; it < p.item_off[cta + 1]; ++it) {
      const mk_attn_item item = p.items[it];
      const int32_t* btrow = p.block_tables + static_cast<size_t>(item.b) * p.maxpg;
#pragma unroll 1
      for (uint32_t pg = item.page_lo; pg < item.page_hi; pg += ppc) {
        const uint32_t n = min(static_cast<uint32_t>(ppc), item.page_hi - pg);
        int32_t ids[kIdBatch];
        page_ids(btrow + pg, n, ids);   // in flight across the slot wait
        if (!acquire()) return false;
        Meta& m = meta();
        m.kind = R_ATTN; m.op = MK_OP_ATTN; m.first = (pg == item.page_lo); m.last = (pg + n >= item.page_hi);
        m.layer = t.layer; m.n = static_cast<uint16_t>(n); m.row0 = pg; m.idx = static_cast<uint32_t>(it);
        m.e = 0; m.aux = 0; m.lo = item.page_lo; m.hi = item.page_hi;
        mbar_arrive_expect_tx(full(), 2u * n * (cbox + sbox));
        uint8_t* dst = slot();
        uint8_t* sd = dst + static_cast<size_t>(2 * rows_cap) * p.D;
#pragma unroll 1
        for (uint32_t i0 = 0; i0 < n; i0 += kIdBatch) {
          if (i0 > 0) page_ids(btrow + pg + i0, n - i0, ids);
#pragma unroll
          for (int j = 0; j < kIdBatch; ++j) {
            const uint32_t i = i0 + j;
            if (i >= n) break;
            const int32_t page = checked_page(ids[j], t.layer, pg + i);
            const int rowk = ((page * 2) * p.Hkv + item.kvh) * p.ps;   // row of the layer's code plane
            const int rowv = rowk + p.Hkv * p.ps;
            tma_load_3d(dst + i * cbox, p.kv_map, 0, rowk, t.layer, full(), pol);
            tma_load_3d(dst + static_cast<size_t>(rows_cap) * p.D + i * cbox, p.kv_map, 0, rowv, t.layer, full(), pol);
            bulk_g2s(sd + i * sbox, sbase + static_cast<size_t>(rowk) * srow, sbox, full(), pol);
            bulk_g2s(sd + rows_cap * srow + i * sbox, sbase + static_cast<size_t>(rowv) * srow, sbox, full(), pol);
          }
        }
        ++c;
      }
    }
    return true;
  }

  // MoE records of layer l.  First a routing record: the consumers of this block read the
  // router logits, route every row of the batch and split the layer's gate/up units over the
  // blocks, all in shared memory, then hand over.  Gate/up: this block's units (FFN rows of
  // active experts) as chunks of gate rows followed by as many up rows; one run of chunks per
  // expert.  Down: this block's hidden rows [lo, hi) of every active expert, several experts'
  // row blocks per chunk.
  __device__ bool moe_tasks(const mk_task& t) {
    const int l = t.layer;
    // the layer's expert weight pointers are loaded before the routing wait, so that the first
    // expert copy goes out as soon as the routing arrives (0.5 % at batch 1)
    const uint16_t* w_gu = p.layers[l].w_gate_up;
    const uint16_t* w_dn = p.layers[l].w_down;
    const uint16_t* w_dt = p.layers[l].w_down_t;
    asm volatile("" ::"l"(w_gu), "l"(w_dn), "l"(w_dt));
    if (!moe_control(R_ROUTE, l, 0u, 0u)) return false;
    const uint64_t t0 = tr_on(p) ? globaltimer() : 0;
    {
      const uint64_t tw = globaltimer();
      #pragma unroll 1
      for (uint32_t it = 1; !mbar_try_wait(&S.route_bar, rphase); ++it) {
        if ((it & 63u) == 0u) {
          if (aborted(p)) return false;
          if (globaltimer() - tw > p.watchdog_ns) {
            record_error(p, MK_ERR_TIMEOUT, MK_OP_MOE, l, MK_WAIT_ROUTE, 0, 0, -1, true);
            return false;
          }
        }
      }
      rphase ^= 1u;
    }
    if (tr_on(p) && pev < static_cast<uint32_t>(p.trace_cap) / 2) {
      uint64_t* e = p.trace + (static_cast<size_t>(blockIdx.x) * p.trace_cap + p.trace_cap - 1 - pev) * 4;
      e[0] = t0;
      e[1] = globaltimer();
      e[2] = e[1];
      e[3] = static_cast<uint64_t>(MK_OP_MOE) | (static_cast<uint64_t>(l) << 8) |
             (static_cast<uint64_t>(TR_PRODUCER_ROUTE_WAIT) << 24);
      ++pev;
    }
    const int cta = blockIdx.x;
    const int nact = S.nact;
    const int u0 = S.gu_lo, u1 = S.gu_hi;
    const int H = p.H, F = p.F;
    if constexpr (SMALL) return small_moe_tasks(l, u0, u1, w_gu, w_dt);
    // gate/up
    const int fpc = gemv_rows_per_chunk(H) / 2;    // gate rows (and as many up rows) per chunk
    if (u0 >= u1) {
      if (!moe_control(R_GU, l, 0u, 1u)) return false;
    }
    if (TC && p.tc) {
      // wide batch: each expert run on tcgen05, its routed pairs as the N columns
      const uint64_t* map = p.wmaps + static_cast<size_t>(tc_map_index(MK_OP_MOE, l, p.L)) * 16;
      #pragma unroll 1
      for (int u = u0; u < u1;) {
        const int a = u / F, f0 = u - a * F;
        const int fend = min(F, u1 - a * F);
        const int e = S.eact[a];
        mk_task tt;
        tt.op = MK_OP_MOE; tt.layer = static_cast<uint16_t>(l);
        tt.lo = static_cast<uint32_t>(f0); tt.hi = static_cast<uint32_t>(fend); tt.reserved = 0;
        const uint32_t lastgu = (a * F + fend >= u1) ? 1u : 0u;
        if (!tc_emit(tt, 0u, MK_OP_MOE, map, H, fend - f0, e * 2 * F + f0, e * 2 * F + F + f0, 2, 4,
                     tc_batch_cols(S.ecnt[e]), static_cast<uint32_t>(e), static_cast<uint32_t>(a), lastgu))
          return false;
        u = a * F + fend;
      }
    }
    #pragma unroll 1
    for (int u = (TC && p.tc) ? u1 : u0; u < u1;) {
      const int a = u / F, f0 = u - a * F;
      const int fend = min(F, u1 - a * F);
      const uint32_t lastgu = (a * F + fend >= u1) ? 1u : 0u;
      const int e = S.eact[a];
      const uint16_t* gate = w_gu + static_cast<size_t>(e) * 2 * F * H;
      // an expert whose routed rows exceed one register group (groups of 4 rows, batches of 3
      // or more) is streamed once per group (group in aux >> 1), so each group's input is
      // staged once per run; the repeated reads come from L2
      const int ng = p.B > 2 ? (S.ecnt[e] + wide_group_rows(H) - 1) / wide_group_rows(H) : 1;
      #pragma unroll 1
      for (int g = 0; g < ng; ++g) {
        #pragma unroll 1
        for (int f = f0; f < fend; f += fpc) {
          const int n = min(fpc, fend - f);
          if (!acquire()) return false;
          Meta& m = meta();
          m.kind = R_GU; m.op = MK_OP_MOE; m.first = (g == 0 && f == f0); m.last = (g == ng - 1 && f + n >= fend);
          m.layer = static_cast<uint16_t>(l); m.n = static_cast<uint16_t>(n); m.row0 = f;
          m.idx = static_cast<uint32_t>(a); m.e = static_cast<uint32_t>(e);
          m.aux = lastgu | (static_cast<uint32_t>(g) << 1);
          m.lo = f0; m.hi = fend;
          const uint32_t bytes = static_cast<uint32_t>(n) * H * 2u;
          const uint64_t pl = g == ng - 1 ? pol : pol_reuse;
          mbar_arrive_expect_tx(full(), 2u * bytes);
          bulk_g2s(slot(), gate + static_cast<size_t>(f) * H, bytes, full(), pl);
          bulk_g2s(slot() + bytes, gate + static_cast<size_t>(F + f) * H, bytes, full(), pl);
          ++c;
        }
      }
      u = a * F + fend;
    }
    // down
    const uint32_t r0 = static_cast<uint32_t>(static_cast<uint64_t>(H) * cta / p.n_ctas);
    const uint32_t r1 = static_cast<uint32_t>(static_cast<uint64_t>(H) * (cta + 1) / p.n_ctas);
    if (TC && p.tc) {
      // wide batch: (active expert, 128-row block) units dealt evenly over the blocks, consecutive
      // units of one expert forming one run (contiguous hidden rows); each run on tcgen05 writes its
      // pairs' weighted outputs, then the block sums the slots of its own hidden rows
      const uint64_t* map = p.wmaps + static_cast<size_t>(tc_map_index(kTcOpDown, l, p.L)) * 16;
      const int nrb = (H + kTcDownRows - 1) / kTcDownRows;
      // the gate/up cost prefix (F units per expert) scaled to nrb units per expert
      const int ua = moe_gu_start(cta, p.n_ctas, S.ecum, S.ecost, nact, nrb, nrb, F);
      const int ub = moe_gu_start(cta + 1, p.n_ctas, S.ecum, S.ecost, nact, nrb, nrb, F);
      #pragma unroll 1
      for (int u = ua; u < ub;) {
        const int a = u / nrb, rb = u - a * nrb;
        const int rend = min(nrb, rb + (ub - u));
        const int e = S.eact[a];
        mk_task tt;
        tt.op = static_cast<uint16_t>(kTcOpDown); tt.layer = static_cast<uint16_t>(l);
        tt.lo = static_cast<uint32_t>(rb * kTcDownRows); tt.hi = static_cast<uint32_t>(min(H, rend * kTcDownRows));
        tt.reserved = 0;
        if (!tc_emit(tt, 0u, static_cast<uint8_t>(kTcOpDown), map, F, static_cast<int>(tt.hi - tt.lo),
                     e * H + static_cast<int>(tt.lo), 0, 1, 2, tc_batch_cols(S.ecnt[e]), static_cast<uint32_t>(e),
                     static_cast<uint32_t>(a), 0u))
          return false;
        u += rend - rb;
      }
      return moe_control(R_YRED, l, r0, r1);
    }
    const uint32_t rowb = static_cast<uint32_t>(F) * 2u;
    if (r1 <= r0 || nact == 0) return moe_control(R_DOWN, l, r0, r1);
    const int rpc = min(static_cast<int>(r1 - r0), static_cast<int>(kSlotBytes / rowb));
    bool first = true;
    #pragma unroll 1
    for (int rb = static_cast<int>(r0); rb < static_cast<int>(r1); rb += rpc) {
      const int nrc = min(rpc, static_cast<int>(r1) - rb);
      const int epc = max(1, min(255, static_cast<int>(kSlotBytes / (nrc * rowb))));
      #pragma unroll 1
      for (int a = 0; a < nact; a += epc) {
        const int ne = min(epc, nact - a);
        if (!acquire()) return false;
        Meta& m = meta();
        m.kind = R_DOWN; m.op = MK_OP_MOE; m.first = first;
        m.last = (rb + nrc >= static_cast<int>(r1)) && (a + ne >= nact);
        m.layer = static_cast<uint16_t>(l); m.n = static_cast<uint16_t>(ne); m.row0 = static_cast<uint32_t>(rb);
        m.idx = static_cast<uint32_t>(a); m.e = 0; m.aux = static_cast<uint32_t>(nrc);
        m.lo = r0; m.hi = r1;
        const uint32_t bytes = static_cast<uint32_t>(nrc) * rowb;
        mbar_arrive_expect_tx(full(), static_cast<uint32_t>(ne) * bytes);
        #pragma unroll 1
        for (int k = 0; k < ne; ++k) {
          const uint16_t* down = w_dn + (static_cast<size_t>(S.eact[a + k]) * H + rb) * F;
          bulk_g2s(slot() + k * bytes, down, bytes, full(), pol);
        }
        ++c;
        first = false;
      }
    }
    return true;
  }

  // Small-batch MoE records of layer l: this block's gate/up units [u0, u1) in groups of at
  // most two gate/up chunks, each group followed by one chunk of the same FFN rows of the
  // transposed down projection (so a group's SwiGLU outputs are consumed on this SM); the
  // consumers run all of them as one tile.  Then the reduction record: publish this block's
  // partial output, sum every block's partials for the block's own hidden rows.
  __device__ bool small_moe_tasks(int l, int u0, int u1, const uint16_t* w_gu, const uint16_t* w_dt) {
    const int H = p.H, F = p.F;
    const int fpc = gemv_rows_per_chunk(H) / 2;   // 2 * fpc transposed down rows fill at most one slot
    #pragma unroll 1
    for (int u = u0; u < u1;) {
      const int a = u / F, f0 = u - a * F;
      const int fend = min(F, u1 - a * F);
      const int e = S.eact[a];
      const uint16_t* gate = w_gu + static_cast<size_t>(e) * 2 * F * H;
      #pragma unroll 1
      for (int g0 = f0; g0 < fend; g0 += 2 * fpc) {
        const int gend = min(fend, g0 + 2 * fpc);
        #pragma unroll 1
        for (int f = g0; f < gend; f += fpc) {
          const int n = min(fpc, gend - f);
          if (!acquire()) return false;
          Meta& m = meta();
          m.kind = R_GU; m.op = MK_OP_MOE; m.first = (f == g0); m.last = (f + n >= gend);
          m.layer = static_cast<uint16_t>(l); m.n = static_cast<uint16_t>(n); m.row0 = f;
          m.idx = static_cast<uint32_t>(a); m.e = static_cast<uint32_t>(e); m.aux = 0u;   // the tile runs on
          m.lo = g0; m.hi = gend;
          const uint32_t bytes = static_cast<uint32_t>(n) * H * 2u;
          mbar_arrive_expect_tx(full(), 2u * bytes);
          bulk_g2s(slot(), gate + static_cast<size_t>(f) * H, bytes, full(), pol);
          bulk_g2s(slot() + bytes, gate + static_cast<size_t>(F + f) * H, bytes, full(), pol);
          ++c;
        }
        if (!acquire()) return false;
        Meta& m = meta();
        m.kind = R_DT; m.op = MK_OP_MOE; m.first = 1;
        m.last = (a * F + gend >= u1);   // the block's last group ends the gate/up tile
        m.layer = static_cast<uint16_t>(l); m.n = static_cast<uint16_t>(gend - g0); m.row0 = g0;
        m.idx = static_cast<uint32_t>(a); m.e = static_cast<uint32_t>(e);
        m.aux = static_cast<uint32_t>(a * F + g0 - u0);   // unit index of the chunk's first row
        m.lo = g0; m.hi = gend;
        const uint32_t bytes = static_cast<uint32_t>(gend - g0) * H * 2u;
        mbar_arrive_expect_tx(full(), bytes);
        bulk_g2s(slot(), w_dt + (static_cast<size_t>(e) * F + g0) * H, bytes, full(), pol);
        ++c;
      }
      u = a * F + fend;
    }
    const uint32_t r0 = static_cast<uint32_t>(static_cast<uint64_t>(H) * blockIdx.x / p.n_ctas);
    const uint32_t r1 = static_cast<uint32_t>(static_cast<uint64_t>(H) * (blockIdx.x + 1) / p.n_ctas);
    return moe_control(R_RED, l, r0, r1);
  }

  // an empty MoE record: a block with no gate/up units or no hidden rows still signals
  __device__ bool moe_control(uint8_t kind, int l, uint32_t lo, uint32_t hi, uint8_t op = MK_OP_MOE) {
    if (!acquire()) return false;
    Meta& m = meta();
    m.kind = kind; m.op = op; m.first = 1; m.last = 1;
    m.layer = static_cast<uint16_t>(l); m.n = 0; m.row0 = lo; m.idx = 0; m.e = 0; m.aux = 1;
    m.lo = lo; m.hi = hi;
    mbar_arrive(full());
    ++c;
    return true;
  }

  __device__ void run() {
    const int cta = blockIdx.x;
    if (p.task_off[cta] < p.task_off[cta + 1]) prefetch_task(p.tasks[p.task_off[cta]]);
    #pragma unroll 1
    for (int ti = p.task_off[cta]; ti < p.task_off[cta + 1]; ++ti) {
      const mk_task t = p.tasks[ti];
      bool ok = true;
      switch (t.op) {
        case MK_OP_EMBED: ok = emit_control(R_EMBED, t, static_cast<uint32_t>(ti)); break;
        case MK_OP_QKV:
        case MK_OP_OPROJ:
        case MK_OP_ROUTER:
        case MK_OP_HEAD: ok = (TC && p.tc) ? tc_tile(t, static_cast<uint32_t>(ti)) : gemv_tile(t, static_cast<uint32_t>(ti)); break;
        case MK_OP_ATTN: ok = attn_items(t); break;
        case MK_OP_MOE: ok = moe_tasks(t); break;
        case MK_OP_END: ok = emit_control(R_END, t, static_cast<uint32_t>(ti)); break;
        default: break;
      }
      if (!ok) break;
    }
    S.prod_count = c;
    if (tr_on(p)) p.trace[static_cast<size_t>(blockIdx.x) * p.trace_cap * 4 + 2] = pev;
  }
};

// --------------------------------------------------------------------------- GEMV pieces
// A chunk holds rows of length K (bf16, row-major).  A row is cut into S
// segments (S a power of two) so that one segment of the input vector -- at
// most 2048/TB values per row of the batch -- fits in registers: 8/TB
// 16-byte units per lane.  Warp w owns segment w % S of rows w/S, w/S + 8/S,
// ...: each lane dots its units of the row from shared memory against its
// register slice, and one warp reduction finishes the segment.  With S == 1 a
// warp finishes whole rows on its own; with S > 1 the segment sums meet in
// shared memory behind one barrier.
template <int TB>
struct Seg {
  static constexpr int kUnits = 8 / TB;   // 16-byte units per lane held in registers (64 floats in all)
  int K, S, KS, U;                         // segments per row, segment length, units per segment
  int s, rg, RPG;                          // this warp's segment, its first row, row stride
  __device__ explicit Seg(int K_, int min_s = 1) : K(K_) {
    S = min_s;
    while (S < kConsumerWarps && S * (256 * kUnits / 8) * 8 < K) S <<= 1;
    KS = ((K + S - 1) / S + 7) & ~7;
    U = KS >> 3;
    const int w = threadIdx.x >> 5;
    s = w & (S - 1);
    rg = w / S;
    RPG = kConsumerWarps / S;
    full = (U == 32 * kUnits) && (S * KS == K);
  }
  bool full;   // every lane owns all kUnits units of its segment (no bounds checks needed)
  // element offset in the row of this lane's j-th unit, or -1
  __device__ __forceinline__ int unit(int j) const {
    const int u = (threadIdx.x & 31) + 32 * j;
    const int e = s * KS + u * 8;
    return (u < U && e < K) ? e : -1;
  }
};

__device__ __forceinline__ void unpack8(const uint4 w, float (&f)[8]) {
  f[0] = bf_lo(w.x); f[1] = bf_hi(w.x); f[2] = bf_lo(w.y); f[3] = bf_hi(w.y);
  f[4] = bf_lo(w.z); f[5] = bf_hi(w.z); f[6] = bf_lo(w.w); f[7] = bf_hi(w.w);
}

// this lane's partial dot products of one row (row points at the row in shared memory);
// independent partial sums per unit pair break the FMA dependency chain
template <int TB>
__device__ __forceinline__ void row_dot(const uint8_t* row, const Seg<TB>& sg, const float (&y)[8 / TB][8][TB],
                                        float (&acc)[TB]) {
  constexpr int NU = Seg<TB>::kUnits;
  float part[TB][2];
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) { part[tb][0] = 0.f; part[tb][1] = 0.f; }
  if (sg.full) {
    const uint8_t* base = row + (sg.s * sg.KS + (threadIdx.x & 31) * 8) * 2;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
      float wf[8];
      unpack8(*reinterpret_cast<const uint4*>(base + j * 512), wf);
#pragma unroll
      for (int tb = 0; tb < TB; ++tb)
#pragma unroll
        for (int q = 0; q < 8; ++q) part[tb][q & 1] = fmaf(wf[q], y[j][q][tb], part[tb][q & 1]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < NU; ++j) {
      const int e = sg.unit(j);
      if (e >= 0) {
        float wf[8];
        unpack8(*reinterpret_cast<const uint4*>(row + e * 2), wf);
#pragma unroll
        for (int tb = 0; tb < TB; ++tb)
#pragma unroll
          for (int q = 0; q < 8; ++q) part[tb][q & 1] = fmaf(wf[q], y[j][q][tb], part[tb][q & 1]);
      }
    }
  }
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) acc[tb] += part[tb][0] + part[tb][1];
}

template <int TB>
__device__ __forceinline__ int pick_i(const int (&a)[TB], int i) {
  int v = a[0];
#pragma unroll
  for (int k = 1; k < TB; ++k)
    if (i == k) v = a[k];
  return v;
}

template <int TB>
__device__ __forceinline__ float pick(const float (&a)[TB], int i) {
  float v = a[0];
#pragma unroll
  for (int k = 1; k < TB; ++k)
    if (i == k) v = a[k];
  return v;
}

// 8 consecutive tagged words, re-polling until every one carries the step's tag (the
// unstaged SwiGLU input of wide batches); ok is false if the watchdog or an abort ended it.
// Returned by value so that the caller's registers never need an address.
struct H8 { float v[8]; bool ok; };
__device__ __noinline__ H8 load_h8(const Params& p, const uint64_t* src, uint32_t tag) {
  H8 r;
  r.ok = true;
  const uint64_t t0 = globaltimer();
  #pragma unroll 1
  for (uint32_t it = 1;; ++it) {
    uint32_t st = 0;
#pragma unroll
    for (int q = 0; q < 8; q += 2) {
      uint64_t a, b;
      ll_ld2(src + q, a, b);
      st |= ll_stale(a, tag) | ll_stale(b, tag);
      r.v[q] = ll_f(a);
      r.v[q + 1] = ll_f(b);
    }
    if (st == 0u) return r;
    if ((it & 15u) == 0u && (aborted(p) || globaltimer() - t0 > p.watchdog_ns)) { r.ok = false; return r; }
  }
}

// --------------------------------------------------------------------------- tcgen05 issuer
// One warp of the producer warpgroup (wide batches): takes the consumers' requests in order, one
// per staged input slice, and issues its MMAs (one elected lane; operands computed by the whole
// warp, so they are warp-uniform), then the commits it asks for.  Ends at the stop request the
// consumers post at the end of the step.
__device__ void tc_issuer(const Params& p, Smem& S) {
  const int lane = threadIdx.x & 31;
  uint32_t wph = 0;
  #pragma unroll 1
  for (uint32_t r = 0;; ++r) {
    const int slot = static_cast<int>(r % kTcReqs);
    const uint32_t ph = (r / kTcReqs) & 1u;
    if (!mbar_try_wait(&S.reqbar[slot], ph)) {
      const uint64_t t0 = globaltimer();
      bool got = false;
      #pragma unroll 1
      for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(&S.reqbar[slot], ph)) { got = true; break; }
        // the consumers post until the end of the step, even an aborted one; this bound only
        // guards against a fault of this kernel
        if ((it & 255u) == 0u && globaltimer() - t0 > 4u * p.watchdog_ns + 1000000000ull) break;
      }
      if (!got) {
        if (lane == 0) record_error(p, MK_ERR_TIMEOUT, 0, -1, MK_WAIT_RING, r, 0, -2, true);
        return;
      }
    }
    const Smem::TcReq q = S.tcreq[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.ackbar[slot]);
    if (q.flags & 8u) return;
    tc_fence_after();
    const uint32_t T = (q.flags >> 4) & 15u;
    const uint64_t xd = tc_desc_sw128(q.x);
    const uint64_t td = static_cast<uint64_t>((q.bp * 128u) >> 4);   // one input term
    const bool acc_hi = (q.flags & 1u) != 0u, acc_lo = (q.flags & 2u) != 0u;
    #pragma unroll 1
    for (uint32_t mi = 0; mi < q.nmc; ++mi) {
      #pragma unroll 1
      for (uint32_t un = 0; un < q.nu; ++un) {
        const uint64_t ad = tc_desc_sw128(q.a + (mi * q.nu + un) * q.ustride);
        const uint32_t du = q.d + mi * q.dstride + un * q.dunit;
        #pragma unroll
        for (int k16 = 0; k16 < 4; ++k16) {
          tc_mma_elect(du + q.dh, ad + 2 * k16, xd + 2 * k16, q.idesc, acc_hi || k16 > 0);
          #pragma unroll 1
          for (uint32_t t = 1; t < T; ++t)
            tc_mma_elect(du + q.dlo + (t - 1u) * q.bp, ad + 2 * k16, xd + t * td + 2 * k16, q.idesc, acc_lo || k16 > 0);
        }
      }
    }
    const uint32_t xb = (q.flags >> 8) & 15u;
    if (xb != 0u) tc_commit_elect(&S.xbar[xb - 1u]);
    if (q.flags & 4u) {
      // the ring record is released (for all consumer warps) once the tensor cores have read it;
      // at the end of a pass, the consumers may then read the accumulators
      tc_commit_elect(&S.wbar);
      {
        const uint64_t t0 = globaltimer();
        #pragma unroll 1
        for (uint32_t it = 1; !mbar_try_wait(&S.wbar, wph); ++it)
          if ((it & 255u) == 0u && globaltimer() - t0 > p.watchdog_ns) break;
        wph ^= 1u;
      }
      __syncwarp();
      if (lane == 0) {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&S.empty[q.flags >> 20])),
                     "r"(static_cast<uint32_t>(kConsumerWarps))
                     : "memory");
        if (q.flags & (1u << 16)) mbar_arrive(&S.pbar);
      }
    }
  }
}

// --------------------------------------------------------------------------- consumer
// Warps consume ring records independently (each waits for and releases every
// record of a tile); block-wide barriers are taken only at tile boundaries --
// the dependency wait at a tile's start and the signal at its end -- and, where
// S warps split a row, over those S warps only.
// Every consumer function is inlined into the dispatch loop, so the consumer's state
// (record index, flags) and the small arrays passed between its functions stay in
// registers (the consumer warpgroups hold 216 each).  A call that took the object's
// address would put that state in local memory, and with nearly all of the SM's L1
// given to shared memory, those accesses would miss to L2 after every barrier.
// TB: rows per register group (1, 2 or 4); W: the tcgen05 instantiation (batches of
// kTcMinBatch rows or more: every GEMV a tcgen05 tile), which carries none of the CUDA-core and
// mma.sync GEMV code, as the others carry none of the tcgen05 code; SM: the small-batch MoE
// path (narrow instantiations only), else the general one (or tcgen05).  The host picks the
// instantiation by the step's batch and path.
template <int TB, int D, bool Q8, bool W, bool SM>
struct Consumer {
  static_assert(!SM || (TB <= kSmallMaxB && !W), "the small-batch MoE path serves 1-2 rows");
  static constexpr bool kSmallMoe = SM;
  const Params& p;
  Smem& S;
  uint32_t c = 0;       // this warp's current record
  bool wok = true;      // this warp has not seen the step abort
  uint32_t nev = 1;     // trace events written (event 0 is the header)
  uint64_t twait = 0;   // when the current tile's dependency was met

  uint32_t tg;          // this step's tag (read from the step data at kernel start)
  __device__ Consumer(const Params& p_, Smem& S_) : p(p_), S(S_), tg(S_.tag) {}

  __device__ void trace_event(uint32_t kind, const Meta& m, uint64_t t0) {
    if (!tr_on(p) || threadIdx.x != 0) return;
    if (nev < static_cast<uint32_t>(p.trace_cap) / 2) {
      uint64_t* e = p.trace + (static_cast<size_t>(blockIdx.x) * p.trace_cap + nev) * 4;
      e[0] = t0;
      e[1] = twait ? twait : t0;
      e[2] = globaltimer();
      e[3] = static_cast<uint64_t>(m.op) | (static_cast<uint64_t>(m.layer) << 8) | (static_cast<uint64_t>(kind) << 24) |
             (static_cast<uint64_t>(m.kind == R_GU || m.kind == R_DOWN ? m.aux | (m.kind == R_DOWN ? 0x80000000u : 0u)
                                                                       : m.idx) << 32);
      ++nev;
    }
  }

  // a timestamped point inside a tile (tracing only)
  __device__ void trace_mark(uint32_t id, int layer, uint32_t val = 0) {
    if (!tr_on(p) || threadIdx.x != 0) return;
    if (nev < static_cast<uint32_t>(p.trace_cap) / 2) {
      const uint64_t t = globaltimer();
      uint64_t* ev = p.trace + (static_cast<size_t>(blockIdx.x) * p.trace_cap + nev) * 4;
      ev[0] = t; ev[1] = t; ev[2] = t;
      ev[3] = static_cast<uint64_t>(id) | (static_cast<uint64_t>(layer) << 8) | (static_cast<uint64_t>(TR_MARK) << 24) |
              (static_cast<uint64_t>(val) << 32);
      ++nev;
    }
  }

  __device__ const Meta& meta() const { return S.meta[c % kSlots]; }
  __device__ const uint8_t* slot() const { return S.ring[c % kSlots]; }

  // chunk timeline (tracing only): issue time, when warp 0 saw the data, when it released the slot
  uint64_t tchunk = 0;
  __device__ void trace_chunk_seen() {
    if (tr_on(p) && threadIdx.x == 0) tchunk = globaltimer();
  }
  __device__ void trace_chunk_done() {
    if (!tr_on(p) || threadIdx.x != 0) return;
    if (nev < static_cast<uint32_t>(p.trace_cap) / 2) {
      const Meta& m = meta();
      uint64_t* ev = p.trace + (static_cast<size_t>(blockIdx.x) * p.trace_cap + nev) * 4;
      ev[0] = static_cast<uint64_t>(m.pad[0]) | (static_cast<uint64_t>(m.pad[1]) << 32);
      ev[1] = tchunk;
      ev[2] = globaltimer();
      ev[3] = static_cast<uint64_t>(m.op) | (static_cast<uint64_t>(m.layer) << 8) |
              (static_cast<uint64_t>(TR_CHUNK) << 24) | (static_cast<uint64_t>(c) << 32);
      ++nev;
    }
  }

  // this warp moves to the next record of the current tile; false if the step aborted
  __device__ bool next_rec() {
    trace_chunk_done();
    warp_release_record(S, c);
    ++c;
    if (!warp_wait_record(p, S, c)) {
      wok = false;
      return false;
    }
    trace_chunk_seen();
    return true;
  }

  // ------------------------------------------------------------------ inputs
  // residual-stream vector xidx (layer input 2l, after attention 2l+1), row b
  __device__ __forceinline__ uint64_t* xrow(int xidx, int b) const {
    return p.X + (static_cast<size_t>(xidx) * p.max_batch + b) * p.H;
  }

  // ------------------------------------------------------------------ EMBED
  __device__ __forceinline__ bool embed() {
    const Meta m = meta();
    const int H = p.H;
    #pragma unroll 1
    for (int b = 0; b < p.B; ++b) {
      int tok = __ldg(p.tokens + b);
      if (tok < 0 || tok >= p.V) {
        if (threadIdx.x == 0)
          record_error(p, MK_ERR_DEVICE_BOUNDS, MK_OP_EMBED, -1, 0u, static_cast<uint32_t>(tok), 0, b,
                       false);
        tok = 0;
      }
      const uint16_t* row = p.embed + static_cast<size_t>(tok) * H;
      uint64_t* x = p.X + static_cast<size_t>(b) * H;
      #pragma unroll 1
      for (uint32_t col = m.lo + threadIdx.x; col < m.hi; col += kConsumerThreads) ll_st(x + col, bf1(row[col]), tg);
    }
    return true;
  }

  // ------------------------------------------------------------------ GEMV streams
  struct OutMap {
    uint64_t* base;       // tagged output of (row 0 of the batch, slot 0, matrix row 0), or null
    float* plain;         // untagged output (logits)
    size_t sb, sj;        // strides per batch row and per routing slot
    const uint64_t* resid;  // O-proj: residual input rows this block wrote itself, else null
    const float* bias;    // router bias by matrix row, or null
    float* hs;            // small-batch MoE: on-chip weighted SwiGLU outputs [kSmallMaxB][kMaxUnits], or null
    int hoff;             // unit index (relative to the block's first) of FFN row 0 of the tile's expert
  };

  __device__ __forceinline__ OutMap out_map(int op, int l) const {
    const size_t MB = p.max_batch, xs = MB * p.H;
    OutMap o{nullptr, nullptr, 0, 0, nullptr, nullptr, nullptr, 0};
    switch (op) {
      case MK_OP_QKV: o.base = p.QKV + l * MB * p.nqkv; o.sb = p.nqkv; break;
      case MK_OP_OPROJ: o.base = p.X + (2 * l + 1) * xs; o.sb = p.H; o.resid = p.X + 2 * l * xs; break;
      case MK_OP_ROUTER: o.base = p.RLOG + l * MB * p.E; o.sb = p.E; o.bias = p.layers[l].router_bias; break;
      case MK_OP_HEAD: o.plain = p.logits; o.sb = p.V; break;
      default: o.base = p.HB + l * MB * p.K * p.F; o.sb = static_cast<size_t>(p.K) * p.F; o.sj = p.F; break;
    }
    return o;
  }

  // result v (v2: the matching up row for gate/up) of matrix row `row` for batch row b, slot j;
  // rv: the residual input of that element when the caller already loaded it (O-proj), else NAN
  __device__ __forceinline__ void put(const OutMap& o, bool gu, uint32_t row, int b, int j, float v, float v2,
                                      float rv = NAN) {
    if (j < 0) return;
    const size_t off = static_cast<size_t>(b) * o.sb + static_cast<size_t>(j) * o.sj + row;
    if (gu) {
      v = (v / (1.0f + expf(-v))) * v2;
      // small-batch MoE: the combine weight is applied here, and the down projection of this
      // block's own units reads the value from shared memory
      if constexpr (kSmallMoe) {
        const int u = o.hoff + static_cast<int>(row);
        if (o.hs != nullptr && u >= 0 && u < kMaxUnits) o.hs[b * kMaxUnits + u] = v * S.rwcache[b * p.K + j];
      }
    }
    if (o.resid != nullptr) v += isnan(rv) ? ll_f(ll_ld(o.resid + off)) : rv;
    if (o.bias != nullptr) v += __ldg(o.bias + row);
    if (o.base != nullptr) ll_st(o.base + off, v, tg);
    else o.plain[off] = v;
  }

  // Stage the GEMV input of rows rb[0..nt) once per block in shared memory (dst, [nt][K] fp32,
  // RMS-normalised for the kinds that have a norm), so that the block reads each tagged input
  // word once instead of once per warp.  One round of loads: the gains go out with the tagged
  // words, and each row's sum of squares is reduced from the staged values themselves.
  __device__ __forceinline__ bool stage_input(int kind, int l, int K, const int (&rb)[TB], int nt, uint32_t tag,
                                           float* dst) {
    const uint16_t* g = nullptr;
    int xidx = 0;
    if (kind == 0) { g = p.layers[l].attn_norm; xidx = 2 * l; }
    else if (kind == 2) { g = p.layers[l].ffn_norm; xidx = 2 * l + 1; }
    else if (kind == 3) { g = p.final_norm; xidx = 2 * p.L; }
    const uint64_t* src[TB];
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      const int b = tb < nt ? rb[tb] : rb[0];
      src[tb] = kind == 1 ? p.ATT + (static_cast<size_t>(l) * p.max_batch + b) * (p.Hq * p.D) : xrow(xidx, b);
    }
    cbar();   // the previous group's input has been read
    // this thread's columns for the normalisation: 4 at k4 = 4 * tid + 1024 * j
    constexpr int kG = kMaxK / (4 * kConsumerThreads);
    uint2 gw[kG];
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      const int k4 = 4 * threadIdx.x + 4 * kConsumerThreads * j;
      gw[j] = (g != nullptr && k4 < K) ? __ldg(reinterpret_cast<const uint2*>(g + k4)) : make_uint2(0u, 0u);
    }
    const uint64_t* s0 = src[0];
    const uint64_t* s1 = src[TB > 1 ? 1 : 0];
    const uint64_t* s2 = src[TB > 2 ? 2 : 0];
    const uint64_t* s3 = src[TB > 3 ? 3 : 0];
    const FastDiv dK(K);   // nt * K <= the scratch size < 2^16
    // (the widest instantiation stages groups of 3-4 rows, 32 loads per thread per pass: 2 %
    // faster at batch 64; the narrow ones keep 8, where the inlined code size matters more)
    bool ok = ll_gather<TB == 4 ? 32 : 8>(p, nt * K, [=](int i) {
      const int tb = dK.div(i), k = i - tb * K;
      return (tb == 0 ? s0 : tb == 1 ? s1 : tb == 2 ? s2 : s3) + k;
    }, dst, tag);
    if (g != nullptr) {
      cbar();   // every staged value is in shared memory
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
      float ss[TB];
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) ss[tb] = 0.f;
#pragma unroll
      for (int j = 0; j < kG; ++j) {
        const int k4 = 4 * threadIdx.x + 4 * kConsumerThreads * j;
        if (k4 < K) {
#pragma unroll
          for (int tb = 0; tb < TB; ++tb) {
            if (tb < nt) {
              const float4 v = *reinterpret_cast<const float4*>(dst + tb * K + k4);
              ss[tb] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
          }
        }
      }
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) {
        const float w = warp_sum(ss[tb]);
        if (lane == 0) S.ssred[warp][tb] = w;
      }
      cbar();
      float r[TB];
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) t += S.ssred[w][tb];
        r[tb] = 1.0f / sqrtf(t / static_cast<float>(K) + p.eps);
      }
#pragma unroll
      for (int j = 0; j < kG; ++j) {
        const int k4 = 4 * threadIdx.x + 4 * kConsumerThreads * j;
        if (k4 < K) {
#pragma unroll
          for (int tb = 0; tb < TB; ++tb) {
            if (tb < nt) {
              float4* q = reinterpret_cast<float4*>(dst + tb * K + k4);
              float4 v = *q;
              v.x = (v.x * r[tb]) * bf_lo(gw[j].x);
              v.y = (v.y * r[tb]) * bf_hi(gw[j].x);
              v.z = (v.z * r[tb]) * bf_lo(gw[j].y);
              v.w = (v.w * r[tb]) * bf_hi(gw[j].y);
              *q = v;
            }
          }
        }
      }
    }
    cbar();
    return ok;
  }

  // this warp's segment of the staged input rows (yc, [nt][K]) into registers
  __device__ __forceinline__ void load_y_staged(const float* yc, const Seg<TB>& sg, int K, int nt,
                                                float (&y)[8 / TB][8][TB]) {
#pragma unroll
    for (int j = 0; j < Seg<TB>::kUnits; ++j) {
      const int e = sg.unit(j);
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (e >= 0 && tb < nt) {
          a = *reinterpret_cast<const float4*>(yc + tb * K + e);
          b = *reinterpret_cast<const float4*>(yc + tb * K + e + 4);
        }
        y[j][0][tb] = a.x; y[j][1][tb] = a.y; y[j][2][tb] = a.z; y[j][3][tb] = a.w;
        y[j][4][tb] = b.x; y[j][5][tb] = b.y; y[j][6][tb] = b.z; y[j][7][tb] = b.w;
      }
    }
  }

  __device__ __forceinline__ bool stream_load(const Seg<TB>& sg, bool moe, int kind, int l, int b0, int nt,
                                              uint32_t tag, int op, int (&rb)[TB], int (&rj)[TB],
                                              float (&y)[8 / TB][8][TB], const float*& ysrc) {
    ysrc = nullptr;
    if (moe) {
      expert_rows(b0, nt, rb, rj);
    } else {
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) { rb[tb] = b0 + tb; rj[tb] = 0; }
    }
    if (nt * sg.K <= kMoeScratch) {
      // the router input of a batch that fits is the MoE input: stage it into the cache
      const bool cache = op == MK_OP_ROUTER && sg.S == 1 && p.B <= TB && p.B * sg.K <= kAttnScratch;
      float* dst = cache ? S.scr.attn : S.moe;
      const bool ok = stage_input(kind, l, sg.K, rb, nt, tag, dst);
      if (cache && threadIdx.x == 0) S.ykey = l;
      load_y_staged(dst, sg, sg.K, nt, y);
      ysrc = dst;
      return ok;
    }
    return false;   // unreachable: register groups are sized so that their input fits the scratch
  }

  // Wide batches: one chunk of n weight rows (gate/up: n gate rows, then their n up rows)
  // against the staged input rows of the current register group, on tensor cores.
  // mma.m16n8k16 (bf16 operands, fp32 accumulation): A = 16 weight rows, B = 16 input
  // positions of the group's rows as the 8 columns (rows nt..7 zero).  The input is split into
  // bf16 terms (high, middle, low), one MMA each into separate accumulators; the weights are
  // exact.  Two terms keep ~16 bits of the fp32 input (relative error of a dot product ~3e-6
  // of its terms' magnitude), the third all of it.  The MMA issue rate bounds these tiles, so
  // three (`exact`) serve only the QKV projection: the step rounds its k and v to bf16 for
  // the cache, and a component that cancels to near zero must keep fp32 accuracy there.  The warps split K; a lane's 16-byte load of a weight row
  // (8 positions) feeds two k-steps, and the input positions are permuted alike (the terms of a
  // dot product may be taken in any order).  The warps' partial sums meet in shared memory.
  __device__ __forceinline__ void mma_chunk(const OutMap& om, bool gu, bool exact, int n, int K, uint32_t row0,
                                            const uint8_t* wsm, const float* ys, int nt, const int (&rb)[TB],
                                            const int (&rj)[TB], int par) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int NR = gu ? 2 * n : n;   // weight rows in the chunk, at most kMaxRowsPerChunk
    const bool two = NR > 16;        // a second 16-row tile
    const int KP = (K + 31) >> 5;    // 32-position steps of K, split over the warps
    const int kp0 = warp * KP / kConsumerWarps, kp1 = (warp + 1) * KP / kConsumerWarps;
    const uint8_t* wrow = wsm + static_cast<size_t>(g) * K * 2;   // rows g, g + 8, g + 16, g + 24
    const size_t r8 = static_cast<size_t>(8) * K * 2;
    const float* xrow = ys + static_cast<size_t>(g) * K;
    const bool xin = g < nt;
    float acc[2][3][4];   // [row tile][high, middle, low term of the input][fragment]
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int h = 0; h < 3; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[m][h][i] = 0.f;
    for (int kp = kp0; kp < kp1; ++kp) {
      const int k = kp * 32 + 8 * t;   // this lane's 8 positions (K is a multiple of 8)
      const bool kin = k < K;
      uint4 wa[4];
#pragma unroll
      for (int h = 0; h < 4; ++h)
        wa[h] = (kin && g + 8 * h < NR) ? *reinterpret_cast<const uint4*>(wrow + h * r8 + k * 2) : make_uint4(0u, 0u, 0u, 0u);
      float4 xv[2];
#pragma unroll
      for (int s = 0; s < 2; ++s)
        xv[s] = (kin && xin) ? *reinterpret_cast<const float4*>(xrow + k + 4 * s) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        // k-step s: fragment positions (2t, 2t+1) and (2t+8, 2t+9) are the lane's positions
        // 4s, 4s+1 and 4s+2, 4s+3
        uint32_t bh0, bm0, bl0, bh1, bm1, bl1;
        split3_bf16x2(xv[s].x, xv[s].y, bh0, bm0, bl0);
        split3_bf16x2(xv[s].z, xv[s].w, bh1, bm1, bl1);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          if (m == 1 && !two) break;
          const uint4 u0 = wa[2 * m], u1 = wa[2 * m + 1];
          const uint32_t a[4] = {s ? u0.z : u0.x, s ? u1.z : u1.x, s ? u0.w : u0.y, s ? u1.w : u1.y};
          mma_bf16(acc[m][0], a, bh0, bh1);
          mma_bf16(acc[m][1], a, bm0, bm1);
          if (exact) mma_bf16(acc[m][2], a, bl0, bl1);
        }
      }
    }
    // the partial sums share storage with the MoE input cache, which may be this chunk's input
    if (ys == S.scr.attn) cbar();
    if (threadIdx.x == 0) S.ykey = -1;
    float (*seg)[kConsumerWarps][4] = S.scr.seg[par];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      if (m == 1 && !two) break;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = 16 * m + g + (i >= 2 ? 8 : 0), col = 2 * t + (i & 1);
        if (col < 4 && row < NR) seg[row][warp][col] = acc[m][0][i] + (acc[m][1][i] + acc[m][2][i]);
      }
    }
    cbar();
    const int r = threadIdx.x >> 2, tb = threadIdx.x & 3;
    if (r < n && tb < nt) {
      float v = 0.f, v2 = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        v += seg[r][w][tb];
        if (gu) v2 += seg[n + r][w][tb];
      }
      put(om, gu, row0 + r, pick_i<TB>(rb, tb), pick_i<TB>(rj, tb), v, v2);
    }
  }

  __device__ __forceinline__ bool stream_gemv(int op) {
    constexpr bool kGroups = TB == 4;   // only the widest instantiation sees batches wider than its registers
    const int l = meta().layer;
    const uint32_t lo = meta().lo, hi = meta().hi;
    const int e = static_cast<int>(meta().e);
    const int nf0 = meta().n;
    const bool gu = op == R_OP_GU;
    const bool moe = gu;
    twait = globaltimer();
    const int B = p.B;
    const int lane = threadIdx.x & 31;
    const int K = op == MK_OP_OPROJ ? p.Hq * p.D : p.H;
    // (the small-batch MoE path keeps whole rows per warp: split rows would reuse the storage of
    // the cached MoE input, which every gate/up tile of the layer reads)
    const Seg<TB> sg(K, gu && !kSmallMoe ? (nf0 >= kConsumerWarps ? 1 : kConsumerWarps / nf0) : 1);
    // GEMV input: 0 x_in/attn_norm, 1 attention output, 2 x_mid/ffn_norm, 3 x_final/final_norm
    const int kind = op == MK_OP_QKV ? 0 : op == MK_OP_OPROJ ? 1 : (op == MK_OP_ROUTER || gu) ? 2 : 3;
    // the test hook waits for a tag that is never written
    const uint32_t tag = (op == MK_OP_OPROJ && l == p.stall_layer) ? (tg ^ 0x80000000u) : tg;
    const int eop = gu ? MK_OP_MOE : op;
    trace_mark(10 + (op == MK_OP_ROUTER ? 0 : moe ? 20 : 40), l);
    // Gate/up with the whole batch in one register group and the MoE input cached: y is the
    // same for every expert, so all of this block's runs (one per expert) form one tile and
    // only the routing slots change between runs.
    const bool gu_fused = gu && B <= TB && S.ykey == l;
    const int cnt = gu_fused ? B : moe ? expert_pairs(e) : B;
    const int GR = kGroups ? wide_group_rows(K) : TB;   // rows per register group (at most TB)
    const int ngroups = kGroups ? (cnt + GR - 1) / GR : 1;
    OutMap om = out_map(op, l);
    if (kSmallMoe && gu) {
      om.hs = S.hsm;
      om.hoff = static_cast<int>(meta().idx) * p.F - S.gu_lo;
    }
    int rb[TB], rj[TB];
    float y[8 / TB][8][TB];
    const float* ysrc = nullptr;   // the staged input rows of the current group, when staged
    bool ok = true;
    if (gu_fused) {
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) { rb[tb] = tb; rj[tb] = tb < B ? slot_of(tb, e) : -1; }
      load_y_smem(sg, rb, B, y);
    } else {
      ok = stream_load(sg, moe, kind, l, 0, min(cnt, GR), tag, eop, rb, rj, y, ysrc);
    }
    int cur_g = 0;   // register group whose input is staged
    // segment sums share storage with the MoE input cache: every warp has its input first
    if (sg.S > 1) cbar();
    trace_mark(11 + (op == MK_OP_ROUTER ? 0 : moe ? 20 : 40), l);
    for (;;) {
      const int n = meta().n;
      const uint32_t row0 = meta().row0;
      const bool last = meta().last;
      const uint8_t* wsm = slot();
      const int par = c & 1;
      ok = true;
      // tiles and expert runs of wide batches arrive group-major (the record's register group is
      // its aux, or aux >> 1 for gate/up): a group's input is staged when its first chunk arrives
      const bool gmajor = kGroups && !gu_fused && ngroups > 1;
      const int g_lo = gmajor ? static_cast<int>(moe ? meta().aux >> 1 : meta().aux) : 0;
      const int g_hi = gmajor ? g_lo + 1 : ngroups;
      for (int g = g_lo; g < g_hi && ok; ++g) {
        const int b0 = g * GR;
        const int nt = min(GR, cnt - b0);
        if (kGroups && ngroups > 1 && (!gmajor || g != cur_g)) {
          ok = stream_load(sg, moe, kind, l, b0, nt, tag, eop, rb, rj, y, ysrc) && ok;
          cur_g = g;
        }
        if constexpr (TB == 4) {
          if (ysrc != nullptr) {   // the group's input is staged: the chunk runs on tensor cores
            mma_chunk(om, gu, op == MK_OP_QKV, n, K, row0, wsm, ysrc, nt, rb, rj, par);
            continue;
          }
        }
        if (sg.S == 1 && om.resid == nullptr) {
          // whole rows per warp, two dot products in flight and one paired reduction:
          // gate/up: the row's gate and up; otherwise rows r and r + RPG
          const int step = gu ? sg.RPG : 2 * sg.RPG;
          for (int r = sg.rg; r < n; r += step) {
            const int r2 = gu ? n + r : r + sg.RPG;
            float a[TB], b[TB];
#pragma unroll
            for (int tb = 0; tb < TB; ++tb) { a[tb] = 0.f; b[tb] = 0.f; }
            row_dot<TB>(wsm + static_cast<size_t>(r) * K * 2, sg, y, a);
            if (gu || r2 < n) row_dot<TB>(wsm + static_cast<size_t>(r2) * K * 2, sg, y, b);
            warp_sum2<TB>(a, b);
            if (gu) {
              float up[TB];
#pragma unroll
              for (int tb = 0; tb < TB; ++tb) up[tb] = __shfl_xor_sync(0xffffffffu, a[tb], 16);
              if (lane < nt)
                put(om, true, row0 + r, pick_i<TB>(rb, lane), pick_i<TB>(rj, lane), pick<TB>(a, lane),
                    pick<TB>(up, lane));
            } else {
              const int tb = lane & 15;
              const int rr = lane < 16 ? r : r2;
              if (tb < nt && rr < n)
                put(om, false, row0 + rr, pick_i<TB>(rb, tb), pick_i<TB>(rj, tb), pick<TB>(a, tb), 0.f);
            }
          }
          continue;
        }
        for (int r = sg.rg; r < n; r += sg.RPG) {
          float acc[TB], acc2[TB];
#pragma unroll
          for (int tb = 0; tb < TB; ++tb) { acc[tb] = 0.f; acc2[tb] = 0.f; }
          row_dot<TB>(wsm + static_cast<size_t>(r) * K * 2, sg, y, acc);
          if (gu) row_dot<TB>(wsm + static_cast<size_t>(n + r) * K * 2, sg, y, acc2);
#pragma unroll
          for (int tb = 0; tb < TB; ++tb) {
            acc[tb] = warp_sum(acc[tb]);
            if (gu) acc2[tb] = warp_sum(acc2[tb]);
          }
          if (sg.S == 1) {
            if (lane < nt)
              put(om, gu, row0 + r, pick_i<TB>(rb, lane), pick_i<TB>(rj, lane), pick<TB>(acc, lane),
                  pick<TB>(acc2, lane));
          } else if (lane < nt) {
            S.scr.seg[par][r][sg.s][lane] = pick<TB>(acc, lane);
            if (gu) S.scr.seg[par][kMaxRowsPerChunk / 2 + r][sg.s][lane] = pick<TB>(acc2, lane);
          }
        }
        if (sg.S > 1) {
          if (threadIdx.x == 0) S.ykey = -1;   // seg shares storage with the MoE input cache
          // the S warps of this row group meet; segment 0's warp finishes the rows.  Its residual
          // inputs (O-proj) are loaded before the barrier so that their latency overlaps the wait.
          float rv[4] = {NAN, NAN, NAN, NAN};
          if (om.resid != nullptr && sg.s == 0 && lane < nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = sg.rg + sg.RPG * i;
              if (r < n) rv[i] = ll_f(ll_ld(om.resid + static_cast<size_t>(pick_i<TB>(rb, lane)) * om.sb + row0 + r));
            }
          }
          ok = group_bar_and(ok, sg.S);
          if (ok && sg.s == 0 && lane < nt) {
            int i = 0;
            #pragma unroll 1
            for (int r = sg.rg; r < n; r += sg.RPG, ++i) {
              float v = 0.f, v2 = 0.f;
              #pragma unroll 1
              for (int q = 0; q < sg.S; ++q) {
                v += S.scr.seg[par][r][q][lane];
                if (gu) v2 += S.scr.seg[par][kMaxRowsPerChunk / 2 + r][q][lane];
              }
              put(om, gu, row0 + r, pick_i<TB>(rb, lane), pick_i<TB>(rj, lane), v, v2,
                  i == 0 ? rv[0] : i == 1 ? rv[1] : i == 2 ? rv[2] : i == 3 ? rv[3] : NAN);
            }
          }
          if (kGroups && ngroups > 1) ok = group_bar_and(ok, sg.S);   // seg is reused by the next group
        }
      }
      if (!ok) { wok = false; break; }
      if (last && (!gu_fused || (meta().aux & 1u))) break;
      bool got = next_rec();
      if (kSmallMoe && gu) {
        // small-batch MoE: the block's gate/up chunks and the transposed down chunk after each
        // group are one tile; the warps move through it together (a down chunk reads every
        // warp's SwiGLU outputs of the group)
        if (!cbar_and(got)) break;
        if (meta().kind == R_DT) {
          moe_dt();
          if (meta().last) break;
          got = next_rec();
          if (!cbar_and(got)) break;
        }
      } else if (!got) {
        break;
      }
      if (last) {   // the next gate/up run of this block: its expert's slots
        const int e2 = static_cast<int>(meta().e);
#pragma unroll
        for (int tb = 0; tb < TB; ++tb) rj[tb] = tb < B ? slot_of(tb, e2) : -1;
        if (kSmallMoe && gu) om.hoff = static_cast<int>(meta().idx) * p.F - S.gu_lo;
      }
    }
    if (!ok) ll_timeout(p, eop, l, tg);
    if (!cbar_and(wok && ok)) return false;
    if (op == MK_OP_HEAD && p.next_token != nullptr) head_top2(lo, hi);
    return true;
  }

  // ------------------------------------------------------------------ wide batches on tcgen05
  uint32_t xst = 0;   // per input buffer i: bit i a commit on xbar[i] not yet waited for, bit 4 + i its parity
  uint32_t pph = 0;   // parity of the next pbar phase
  bool tc_held = false;   // the last record was a tcgen05 record, released by the issuing warp

  // Post request rq (every consumer thread, after its share of the slice is staged and fenced):
  // thread 0 writes the fields once the issuer has read the slot's previous request; each thread's
  // arrival releases its staged writes to the issuer.
  uint32_t rq = 0;
  __device__ __forceinline__ void tc_post(uint32_t a, uint32_t x, uint32_t d, uint32_t idesc, int nmc, int nu,
                                          int ustride, int dstride, int dunit, int dh, int dlo, int bp, uint32_t flags) {
    const int slot = static_cast<int>(rq % kTcReqs);
    if (threadIdx.x == 0) {
      if (rq >= static_cast<uint32_t>(kTcReqs)) tc_wait(&S.ackbar[slot], ((rq / kTcReqs) - 1u) & 1u);
      Smem::TcReq& r = S.tcreq[slot];
      r.a = a; r.x = x; r.d = d; r.idesc = idesc;
      r.nmc = static_cast<uint32_t>(nmc); r.nu = static_cast<uint32_t>(nu); r.ustride = static_cast<uint32_t>(ustride);
      r.dstride = static_cast<uint32_t>(dstride); r.dunit = static_cast<uint32_t>(dunit);
      r.dh = static_cast<uint32_t>(dh); r.dlo = static_cast<uint32_t>(dlo); r.bp = static_cast<uint32_t>(bp);
      r.flags = flags;
    }
    mbar_arrive(&S.reqbar[slot]);
    ++rq;
  }
  // the issuing warp's last request (every consumer thread, at the end of the step)
  __device__ __forceinline__ void tc_stop() { tc_post(0u, 0u, 0u, 0u, 0, 0, 0, 0, 0, 0, 0, 0, 8u); }

  // every consumer thread: wait for a phase of a tensor-core commit barrier (the work behind it
  // depends on no other block, so the limit only guards against a fault of this kernel)
  __device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t ph) {
    if (mbar_try_wait(bar, ph)) return true;
    const uint64_t t0 = globaltimer();
    #pragma unroll 1
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(bar, ph)) return true;
      if ((it & 63u) == 0u && globaltimer() - t0 > p.watchdog_ns) return false;
    }
  }

  // Input slice s (columns 64s .. 64s + 63 of every batch row): thread i takes pieces i and i + 256
  // (row i/8, 8 columns from 64s + 8(i%8)), 8 tagged words each.  tc_issue starts all 16 loads
  // (one L2 round trip per slice); tc_stage waits for them, re-polls stale words inline (no call: the caller's registers stay put), and stores
  // T bf16 terms of the fp32 value (high, then what it left, ...) into xb: term t of row b at
  // xb + t*Bp*128 + b*128, its 16-byte piece j at piece j ^ (b & 7) (the K-major layout with the
  // 128-byte swizzle).  A normalised input takes its gain here; the row's 1/rms is applied to the
  // accumulators (a dot product is linear in it), from the sums of squares collected in ss.
  // Columns at or past K are zero.
  __device__ __forceinline__ int tc_row(const int32_t* rows, int n) const { return rows != nullptr ? rows[n] : n; }
  __device__ __forceinline__ void tc_issue(const uint64_t* xbase, size_t xstride, int K, int s, int nrows,
                                           const int32_t* rows, uint64_t (&w)[16]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = threadIdx.x + h * kConsumerThreads;
      const int n = i >> 3, k = 64 * s + 8 * (i & 7);
      if (n < nrows && k < K) {
        const uint64_t* src = xbase + static_cast<size_t>(tc_row(rows, n)) * xstride + k;
#pragma unroll
        for (int q = 0; q < 8; q += 2) ll_ld2(src + q, w[8 * h + q], w[8 * h + q + 1]);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) w[8 * h + q] = 0ull;
      }
    }
  }
  __device__ __forceinline__ bool tc_stage(const uint64_t* xbase, size_t xstride, const uint16_t* g, int K, int s,
                                           int nrows, const int32_t* rows, int T, uint8_t* xb, int Bp, uint32_t tag,
                                           uint64_t (&w)[16], float (&ss)[2]) {
    const int B = nrows;
    // stale words (this step's tag not there yet): re-poll both pieces until every word is fresh
    uint32_t st = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = threadIdx.x + h * kConsumerThreads;
      if ((i >> 3) < B && 64 * s + 8 * (i & 7) < K) {
#pragma unroll
        for (int q = 0; q < 8; ++q) st |= (ll_stale(w[8 * h + q], tag) != 0u ? 1u : 0u) << h;
      }
    }
    bool ok = true;
    if (st != 0u) {
      const uint64_t t0 = globaltimer();
      #pragma unroll 1
      for (uint32_t it = 1; st != 0u; ++it) {
        uint32_t still = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if ((st >> h) & 1u) {
            const int i = threadIdx.x + h * kConsumerThreads;
            const uint64_t* src = xbase + static_cast<size_t>(tc_row(rows, i >> 3)) * xstride + 64 * s + 8 * (i & 7);
#pragma unroll
            for (int q = 0; q < 8; q += 2) ll_ld2(src + q, w[8 * h + q], w[8 * h + q + 1]);
#pragma unroll
            for (int q = 0; q < 8; ++q) still |= (ll_stale(w[8 * h + q], tag) != 0u ? 1u : 0u) << h;
          }
        }
        st = still;
        if (st != 0u && (it & 15u) == 0u && (aborted(p) || globaltimer() - t0 > p.watchdog_ns)) {
          ok = false;
          break;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = threadIdx.x + h * kConsumerThreads;
      const int b = i >> 3, cg = i & 7, k = 64 * s + 8 * cg;
      if (b >= B) continue;
      float x[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) x[q] = ll_f(w[8 * h + q]);   // zero past K
      float a = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) a = fmaf(x[q], x[q], a);
      ss[h] += a;
      if (g != nullptr && k < K) {
        const uint4 gu = __ldg(reinterpret_cast<const uint4*>(g + k));
        x[0] *= bf_lo(gu.x); x[1] *= bf_hi(gu.x); x[2] *= bf_lo(gu.y); x[3] *= bf_hi(gu.y);
        x[4] *= bf_lo(gu.z); x[5] *= bf_hi(gu.z); x[6] *= bf_lo(gu.w); x[7] *= bf_hi(gu.w);
      }
      uint8_t* dst = xb + b * 128 + ((cg ^ (b & 7)) << 4);
      uint4 hi, mid, lo;
      if (T == 3) {
        split3_bf16x2(x[0], x[1], hi.x, mid.x, lo.x);
        split3_bf16x2(x[2], x[3], hi.y, mid.y, lo.y);
        split3_bf16x2(x[4], x[5], hi.z, mid.z, lo.z);
        split3_bf16x2(x[6], x[7], hi.w, mid.w, lo.w);
        *reinterpret_cast<uint4*>(dst + 2 * Bp * 128) = lo;
      } else {
        split_bf16x2(x[0], x[1], hi.x, mid.x);
        split_bf16x2(x[2], x[3], hi.y, mid.y);
        split_bf16x2(x[4], x[5], hi.z, mid.z);
        split_bf16x2(x[6], x[7], hi.w, mid.w);
      }
      *reinterpret_cast<uint4*>(dst) = hi;
      *reinterpret_cast<uint4*>(dst + Bp * 128) = mid;
    }
    return ok;
  }

  // The fp32 sum of one M-block's accumulators for 8 columns of this warp's lanes: the lower
  // terms (lowest first), then the nhg high-term accumulators that received a slice
  __device__ __forceinline__ void tc_sum_accs(uint32_t ta, int Bp, int T, int KG, int nhg, float (&v)[8]) {
    tc_ld8(ta + (KG + T - 2) * Bp, v);
    #pragma unroll 1
    for (int a = KG + T - 3; a >= KG; --a) {
      float w[8];
      tc_ld8(ta + a * Bp, w);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] += w[j];
    }
    #pragma unroll 1
    for (int a = nhg - 1; a >= 0; --a) {
      float w[8];
      tc_ld8(ta + a * Bp, w);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] += w[j];
    }
  }

  // Split-K: this block's partial sums of the group's rows (its share of K, no norm) to
  // PSK[l][op][block][row][b], and its share of each input row's sum of squares to PSQ.
  __device__ __forceinline__ void tc_epilogue_split(int op, int l, int R, int MB, int m0, int m1, int Bp, int T, int KG,
                                                    int nhg, const float (&ss)[2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, hh = warp >> 2;
    const int half = Bp >> 1;
    const int r_in = MB == 128 ? 32 * q + lane : 16 * q + lane;
    const bool lane_ok = MB == 128 || lane < 16;
    const int B = p.B;
    const size_t blk = (static_cast<size_t>(l) * 3 + tc_split_slot(op)) * p.n_ctas + blockIdx.x;
    uint64_t* dst = p.PSK + blk * p.psk_cap;
    #pragma unroll 1
    for (int m = m0; m < m1; ++m) {
      const int row = m * MB + r_in;
      const uint32_t ta = S.tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                          static_cast<uint32_t>((m - m0) * (KG + T - 1) * Bp + hh * half);
      #pragma unroll 1
      for (int c8 = 0; c8 < half; c8 += 8) {
        float v[8];
        tc_sum_accs(ta + c8, Bp, T, KG, nhg, v);
        if (lane_ok && row < R) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int b = hh * half + c8 + j;
            if (b < B) ll_st(dst + static_cast<size_t>(row) * B + b, v[j], tg);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float v = ss[h];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      const int b = (threadIdx.x >> 3) + 32 * h;
      if ((threadIdx.x & 7) == 0 && b < B) ll_st(p.PSQ + blk * p.max_batch + b, v, tg);
    }
  }

  // Split-K: this block's own rows [own_lo, own_hi) from the KS partials of its group (in block
  // order) and, for normalised inputs, 1/rms from the group's sums of squares; then the tile's
  // epilogue (residual, bias, tagged outputs).
  __device__ __forceinline__ bool tc_finalize(int op, int l, bool norm, int K, int KS, uint32_t glo, uint32_t own_lo,
                                              uint32_t own_hi) {
    const int B = p.B;
    const int nown = static_cast<int>(own_hi - own_lo), roff = static_cast<int>(own_lo - glo);
    if (nown <= 0) return true;
    const int g0 = (static_cast<int>(blockIdx.x) / KS) * KS;
    const size_t blk0 = (static_cast<size_t>(l) * 3 + tc_split_slot(op)) * p.n_ctas + g0;
    const uint64_t* psk = p.PSK + blk0 * p.psk_cap;
    const uint64_t* psq = p.PSQ + blk0 * p.max_batch;
    const int per = nown * B;             // one block's words for these rows
    float* Y = S.moe;                     // [KS][nown][B], then [KS][B]
    const int cap = p.psk_cap;
    const int maxb = p.max_batch;
    const FastDiv dper(per), dB(B);
    bool ok = ll_gather(p, KS * per + KS * B, [=](int i) -> const uint64_t* {
      if (i < KS * per) {
        const int q = dper.div(i), r = i - q * per;
        return psk + static_cast<size_t>(q) * cap + static_cast<size_t>(roff) * B + r;
      }
      const int j = i - KS * per, q = dB.div(j);
      return psq + static_cast<size_t>(q) * maxb + (j - q * B);
    }, Y, tg);
    if (!cbar_and(ok)) return false;
    const OutMap om = out_map(op, l);
    #pragma unroll 1
    for (int i = threadIdx.x; i < per; i += kConsumerThreads) {
      const int r = i / B, b = i - r * B;
      float d = 0.f;
      #pragma unroll 1
      for (int q = 0; q < KS; ++q) d += Y[q * per + i];
      if (norm) {
        float t = 0.f;
        #pragma unroll 1
        for (int q = 0; q < KS; ++q) t += Y[KS * per + q * B + b];
        d *= 1.0f / sqrtf(t / static_cast<float>(K) + p.eps);
      }
      put(om, false, own_lo + r, b, 0, d, 0.f);
    }
    return true;
  }

  // Accumulators of M-blocks [m0, m1) of the pass to the outputs: per M-block KG accumulators of
  // the high term and one per lower term, summed here in fp32 (low terms first).  Warp w reads
  // tensor-memory lanes
  // 32(w % 4) .. + 31 (M = 128: row = lane; M = 64: rows 16(w % 4) + lane for lanes < 16) and
  // half w / 4 of the batch columns.
  __device__ __forceinline__ void tc_epilogue(const OutMap& om, bool norm, uint32_t lo, int R, int MB, int m0, int m1,
                                              int Bp, int T, int KG, int nhg, int nrows, bool gu) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, hh = warp >> 2;
    const int half = Bp >> 1;
    const int r_in = MB == 128 ? 32 * q + lane : 16 * q + lane;
    const bool lane_ok = MB == 128 || lane < 16;
    #pragma unroll 1
    for (int m = m0; m < m1; ++m) {
      const int row = m * MB + r_in;
      const int NA = gu ? 4 : KG + T - 1;
      const uint32_t ta = S.tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                          static_cast<uint32_t>((m - m0) * NA * Bp + hh * half);
      #pragma unroll 1
      for (int c8 = 0; c8 < half; c8 += 8) {
        if (gu) {
          // gate (high, low accumulators) and up (high, low) of this lane's FFN row: SwiGLU of the
          // pair's normalised input, to the pair's (row, slot)
          float gh[8], gl[8], uh[8], ul[8];
          tc_ld8(ta + Bp + c8, gl);
          tc_ld8(ta + c8, gh);
          tc_ld8(ta + 3 * Bp + c8, ul);
          tc_ld8(ta + 2 * Bp + c8, uh);
          if (lane_ok && row < R) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int n = hh * half + c8 + j;
              if (n < nrows) {
                const int ent = S.elist[n];
                const int b = ent / p.K, slot = ent - b * p.K;
                const float r = S.rstd[n];
                put(om, true, lo + row, b, slot, (gl[j] + gh[j]) * r, (ul[j] + uh[j]) * r);
              }
            }
          }
          continue;
        }
        float v[8];
        tc_sum_accs(ta + c8, Bp, T, KG, nhg, v);
        if (lane_ok && row < R) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int b = hh * half + c8 + j;
            if (b < p.B) put(om, false, lo + row, b, 0, norm ? v[j] * S.rstd[b] : v[j], 0.f);
          }
        }
      }
    }
  }

  // Down projection run: accumulators (high, low term) of hidden rows x pairs; each pair's value,
  // times its combine weight, to YD[l][row][slot][hidden row].
  __device__ __forceinline__ void tc_epilogue_down(int l, uint32_t lo, int R, int MB, int m0, int m1, int Bp, int nrows) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, hh = warp >> 2;
    const int half = Bp >> 1;
    const int r_in = MB == 128 ? 32 * q + lane : 16 * q + lane;
    const bool lane_ok = MB == 128 || lane < 16;
    uint64_t* yd = p.YD + static_cast<size_t>(l) * p.max_batch * p.K * p.H;
    #pragma unroll 1
    for (int m = m0; m < m1; ++m) {
      const int row = m * MB + r_in;
      const uint32_t ta = S.tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                          static_cast<uint32_t>((m - m0) * 2 * Bp + hh * half);
      #pragma unroll 1
      for (int c8 = 0; c8 < half; c8 += 8) {
        float hi8[8], lo8[8];
        tc_ld8(ta + Bp + c8, lo8);
        tc_ld8(ta + c8, hi8);
        if (lane_ok && row < R) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int n = hh * half + c8 + j;
            if (n < nrows) {
              const int ent = S.elist[n];   // b * K + slot
              ll_st(yd + static_cast<size_t>(ent) * p.H + lo + row, S.rwcache[ent] * (lo8[j] + hi8[j]), tg);
            }
          }
        }
      }
    }
  }

  // Wide batch: x_out of this block's hidden rows [lo, hi) = x_mid + the slots' weighted down
  // outputs, summed in slot order (the small-batch and register-group paths' order).
  __device__ __forceinline__ bool y_reduce() {
    const int l = meta().layer;
    const int r0 = static_cast<int>(meta().lo), nrow = static_cast<int>(meta().hi) - r0;
    twait = globaltimer();
    if (nrow <= 0) return true;
    const int B = p.B, K = p.K;
    const size_t xs = static_cast<size_t>(p.max_batch) * p.H;
    const uint64_t* yd = p.YD + static_cast<size_t>(l) * p.max_batch * K * p.H;
    float* Y = S.moe;   // [B][K][nrow]
    const FastDiv dn(nrow);
    bool ok = ll_gather(p, B * K * nrow, [=](int i) {
      const int bj = dn.div(i), r = i - bj * nrow;
      return yd + static_cast<size_t>(bj) * p.H + r0 + r;
    }, Y, tg);
    if (!ok) ll_timeout(p, MK_OP_MOE, l, tg);
    if (!cbar_and(ok)) return false;
    #pragma unroll 1
    for (int i = threadIdx.x; i < B * nrow; i += kConsumerThreads) {
      const int b = i / nrow, r = i - b * nrow;
      float acc = 0.f;
      #pragma unroll 1
      for (int j = 0; j < K; ++j) acc += Y[(b * K + j) * nrow + r];
      const size_t off = static_cast<size_t>(b) * p.H + r0 + r;
      ll_st(p.X + (2 * static_cast<size_t>(l) + 2) * xs + off,
            ll_f(ll_ld(p.X + (2 * static_cast<size_t>(l) + 1) * xs + off)) + acc, tg);
    }
    return true;
  }

  // A dense GEMV tile (QKV, O-proj, router, LM head) of a wide batch on tcgen05: for each record,
  // per slice, the consumers stage the batch's input slice (unless an earlier record of the pass
  // did), then one thread issues the MMAs of the record's units of that slice into the pass's
  // accumulators; the record's slot is released once the tensor cores have read it.  At the end
  // of a pass the accumulators go to the outputs.
  __device__ __forceinline__ bool tc_gemv() {
    const int op = meta().op, l = meta().layer;
    const uint32_t lo = meta().lo, hi = meta().hi;
    const int R = static_cast<int>(hi - lo);
    // gate/up of one expert run, or a run of one expert's down projection: the N columns are the
    // (row, slot) pairs routed to the expert
    const bool gu = op == MK_OP_MOE, dn = op == kTcOpDown;
    const int K = op == MK_OP_OPROJ ? p.Hq * p.D : dn ? p.F : p.H;
    // input kinds: 0 x_in/attn_norm, 1 un-normalised (attention output; SwiGLU outputs), 2
    // x_mid/ffn_norm, 3 x_final/final_norm
    const int kind = op == MK_OP_QKV ? 0 : (op == MK_OP_OPROJ || dn) ? 1 : (op == MK_OP_ROUTER || gu) ? 2 : 3;
    int nrows = p.B;
    const int32_t* rows = nullptr;
    if (gu || dn) {
      nrows = expert_pairs(static_cast<int>(meta().e));   // S.elist; ends with a barrier
      if (gu) {   // gate/up reads the pairs' x_mid rows; the down projection their SwiGLU rows
        if (threadIdx.x < nrows) S.wlist[0][threadIdx.x] = S.elist[threadIdx.x] / p.K;
        cbar();
        rows = S.wlist[0];
      } else {
        rows = S.elist;
      }
    }
    const int T = gu ? 2 : tc_terms(op), KG = gu ? 1 : tc_hi_groups(op, p.B, K);
    const int NA = gu ? 4 : KG + T - 1;
    // the N columns the producer sized the passes for (the routing both sides computed agrees;
    // the check keeps every accumulator address inside the allocation regardless)
    const int Bp = static_cast<int>(meta().pad[4]), MB = tc_mblock(R);
    // this block's slices of K [s_lo, ns) (split-K groups: a share; KS > 1 only for dense tiles)
    const int s_lo = static_cast<int>(meta().pad[6] & 0xffffu), ns = static_cast<int>(meta().pad[6] >> 16);
    const int KS = (gu || dn) ? 1 : static_cast<int>(meta().pad[3]);
    const uint32_t own_lo = meta().pad[5], own_hi = meta().pad[7];
    const int nhg = min(KG, ns - s_lo);   // high-term accumulators that receive a slice
    if (Bp != tc_batch_cols(nrows)) {
      if (threadIdx.x == 0)
        record_error(p, MK_ERR_DEVICE_BOUNDS, op, l, 0u, static_cast<uint32_t>(nrows), 0, Bp, true);
      cbar();
      return false;
    }
    const uint32_t xsz = static_cast<uint32_t>(T * Bp * 128);
    const int NX = min(kTcXBufs, static_cast<int>((kMoeScratch * 4) / xsz));
    const uint16_t* g = kind == 0 ? p.layers[l].attn_norm : kind == 2 ? p.layers[l].ffn_norm
                      : kind == 3 ? p.final_norm : nullptr;
    const uint64_t* xbase;
    size_t xstride;
    if (dn) {
      xstride = static_cast<size_t>(p.F);
      xbase = p.HB + static_cast<size_t>(l) * p.max_batch * p.K * xstride;
    } else if (kind == 1) {
      xstride = static_cast<size_t>(p.Hq) * p.D;
      xbase = p.ATT + static_cast<size_t>(l) * p.max_batch * xstride;
    } else {
      const int xidx = kind == 0 ? 2 * l : kind == 2 ? 2 * l + 1 : 2 * p.L;
      xstride = static_cast<size_t>(p.H);
      xbase = p.X + static_cast<size_t>(xidx) * p.max_batch * xstride;
    }
    // the test hook waits for a tag that is never written
    const uint32_t tag = (op == MK_OP_OPROJ && l == p.stall_layer) ? (tg ^ 0x80000000u) : tg;
    uint8_t* xb0 = reinterpret_cast<uint8_t*>(S.moe);
    const uint32_t idesc = tc_idesc_bf16(MB, Bp);
    twait = globaltimer();
    float ss[2] = {0.f, 0.f};
    int staged = 0, pass_m0 = -1;
    bool ok = true;
    uint64_t xw[16];   // the tagged words of the slice being staged
    #pragma unroll 1
    for (;;) {
      const int ma = static_cast<int>(meta().row0), nmc = meta().n;
      const int s0 = static_cast<int>(meta().aux & 0xffffu), nsc = static_cast<int>(meta().aux >> 16);
      const int pm0 = static_cast<int>(meta().pad[2] & 0xffffu), pm1 = static_cast<int>(meta().pad[2] >> 16);
      const bool last = meta().last;
      if (pm0 != pass_m0) { pass_m0 = pm0; staged = 0; ss[0] = 0.f; ss[1] = 0.f; }
      const uint32_t wa = smem_u32(slot());
      #pragma unroll 1
      for (int si = 0; si < nsc; ++si) {
        const int sl = s0 + si, buf = sl % NX;
        if (sl >= staged) {
          if ((xst >> buf) & 1u) {   // the tensor cores must have read the buffer's previous slice
            ok = tc_wait(&S.xbar[buf], (xst >> (4 + buf)) & 1u) && ok;
            xst ^= (1u << buf) | (1u << (4 + buf));
          }
          tc_issue(xbase, xstride, K, sl, nrows, rows, xw);
          ok = tc_stage(xbase, xstride, g, K, sl, nrows, rows, T, xb0 + buf * xsz, Bp, tag, xw, ss) && ok;
          fence_proxy_async_smem();   // generic writes, read by the tensor cores (async proxy)
          staged = sl + 1;
        }
        // the slice's MMAs go to the issuing warp; the record's last slice also commits the ring
        // record (its slot is refilled only after the tensor cores have read it)
        const bool last_use = ma + nmc == pm1;   // the slice's last record in this pass
        const int nu = gu ? 2 : 1;
        const bool pass_end = last_use && sl == ns - 1;
        const int rs = sl - s_lo;   // the slice's place in this block's share
        tc_post(wa + static_cast<uint32_t>(si * nmc * nu * MB * 128), smem_u32(xb0) + static_cast<uint32_t>(buf) * xsz,
                S.tmem_base + static_cast<uint32_t>((ma - pm0) * NA * Bp), idesc, nmc, nu, MB * 128, NA * Bp, 2 * Bp,
                (rs % KG) * Bp, KG * Bp, Bp,
                (rs >= KG ? 1u : 0u) | (rs > 0 ? 2u : 0u) | (si + 1 == nsc ? 4u : 0u) | (static_cast<uint32_t>(T) << 4) |
                    (last_use ? static_cast<uint32_t>(buf + 1) << 8 : 0u) | (pass_end ? 1u << 16 : 0u) |
                    (static_cast<uint32_t>(c % kSlots) << 20));
        if (last_use) xst |= 1u << buf;
      }
      // (the issuing warp releases the record once the tensor cores have read it)
      if (ma + nmc == pm1 && s0 + nsc == ns) {
        ok = tc_wait(&S.pbar, pph) && ok;   // the pass's MMAs have completed
        pph ^= 1u;
        ok = cbar_and(ok);
        if (!ok) break;
        // the pass is complete: its rows' norms, then the accumulators to the outputs
        if (kind != 1) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v = ss[h];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            const int b = (threadIdx.x >> 3) + 32 * h;
            if ((threadIdx.x & 7) == 0 && b < nrows) S.rstd[b] = 1.0f / sqrtf(v / static_cast<float>(K) + p.eps);
          }
        }
        cbar();
        tc_fence_after();
        if (dn) tc_epilogue_down(l, lo, R, MB, pm0, pm1, Bp, nrows);
        else if (KS > 1) {
          // split-K: publish this block's partials (and sums of squares), then finalise its own
          // rows from the group's
          tc_epilogue_split(op, l, R, MB, pm0, pm1, Bp, T, KG, nhg, ss);
          tc_fence_before();
          ok = tc_finalize(op, l, kind != 1, K, KS, lo, own_lo, own_hi) && ok;
        } else {
          tc_epilogue(out_map(gu ? int(R_OP_GU) : op, l), kind != 1, lo, R, MB, pm0, pm1, Bp, T, KG, nhg, nrows, gu);
        }
        tc_fence_before();   // these reads precede the next pass's MMAs (behind the next barrier)
      }
      if (last) break;
      ++c;
      if (!warp_wait_record(p, S, c)) { ok = false; wok = false; break; }
    }
    tc_held = true;   // (run() must not release the tile's last record either)
    if (!ok) ll_timeout(p, op, l, tg);
    if (!cbar_and(wok && ok)) return false;
    if (op == MK_OP_HEAD && p.next_token != nullptr) head_top2(lo, hi);
    return true;
  }

  // Greedy selection, first level: this block's (max, index, second) of its LM-head rows
  // [lo, hi) for every row of the batch, from the logits it has just written (a block
  // barrier separates the writes from these reads), into p.argp.
  __device__ __forceinline__ void head_top2(uint32_t lo, uint32_t hi) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    #pragma unroll 1
    for (int b = 0; b < p.B; ++b) {
      Top2 t{-INFINITY, -INFINITY, 0x7fffffff};
      const float* row = p.logits + static_cast<size_t>(b) * p.V;
      #pragma unroll 1
      for (uint32_t r = lo + threadIdx.x; r < hi; r += kConsumerThreads) top2_add(t, row[r], static_cast<int>(r));
      top2_warp(t);
      if (lane == 0) {
        S.ssred[warp][0] = t.m1;
        S.ssred[warp][1] = t.m2;
        S.ssred[warp][2] = __int_as_float(t.i1);
      }
      cbar();
      if (threadIdx.x == 0) {
        Top2 a{S.ssred[0][0], S.ssred[0][1], __float_as_int(S.ssred[0][2])};
        #pragma unroll 1
        for (int w = 1; w < kConsumerWarps; ++w) {
          const Top2 o{S.ssred[w][0], S.ssred[w][1], __float_as_int(S.ssred[w][2])};
          top2_merge(a, o);
        }
        float* out = p.argp + (static_cast<size_t>(blockIdx.x) * p.max_batch + b) * 4;
        out[0] = a.m1;
        out[1] = a.m2;
        out[2] = __int_as_float(a.i1);
      }
      cbar();
    }
  }

  // Ranks of every (row, expert) pair of the batch (see route_local): the consumer threads
  // form G groups, one row each at a time; in a group, 8 threads split the row's logits into
  // slices of at most LEN values held in registers, and the candidates (experts) are dealt
  // over the group's slots.  Each thread counts its slice's values above the candidate (ties:
  // lower index first); the 8 partial counts meet by shuffles.  Pairs ranked below top_k are
  // recorded with their logit, and each chosen expert's row count is incremented.
  template <int LEN>
  __device__ __forceinline__ void rank_rows(const float* lg) {
    const int B = p.B, E = p.E, K = p.K;
    const int G = B >= 8 ? 8 : B >= 4 ? 4 : B >= 2 ? 2 : 1;
    const int gsz = kConsumerThreads / G;
    const int grp = threadIdx.x / gsz, gt = threadIdx.x - grp * gsz;
    const int part = gt & 7, slot = gt >> 3, nslot = gsz >> 3;
    const int e_lo = part * E / 8, e_hi = (part + 1) * E / 8;   // at most LEN values (E <= 8 * LEN)
    const int ncand = (E + nslot - 1) / nslot;
    #pragma unroll 1
    for (int b0 = 0; b0 < B; b0 += G) {   // uniform trip counts: the shuffles below
      const int b = b0 + grp;
      const bool bon = b < B;
      const float* row = lg + (bon ? b : 0) * E;
      float sl[LEN];
#pragma unroll
      for (int k = 0; k < LEN; ++k) sl[k] = (e_lo + k < e_hi) ? row[e_lo + k] : -INFINITY;
      #pragma unroll 1
      for (int j = 0; j < ncand; ++j) {
        const int e = slot + j * nslot;
        const bool on = bon && e < E;
        const float v = row[on ? e : 0];
        int r0 = 0, r1 = 0;
#pragma unroll
        for (int k = 0; k < LEN; ++k) {
          // padding (-inf, index past the slice) never counts: finite logits only exceed it
          const int c = static_cast<int>(sl[k] > v) +
                        (static_cast<int>(sl[k] == v) & static_cast<int>(e_lo + k < e) & static_cast<int>(e_lo + k < e_hi));
          if (k & 1) r1 += c; else r0 += c;
        }
        int rank = r0 + r1;
        rank += __shfl_xor_sync(0xffffffffu, rank, 1);
        rank += __shfl_xor_sync(0xffffffffu, rank, 2);
        rank += __shfl_xor_sync(0xffffffffu, rank, 4);
        if (on && part == 0 && rank < K) {
          S.rids[b * K + rank] = e;
          S.rval[b * K + rank] = v;
          atomicAdd(&S.ecnt[e], 1);
        }
      }
    }
  }

  // Top-k of every row for wider batches: a warp per row holds the row's logits in registers
  // (up to 8 per lane) and runs k rounds of a warp argmax over (value, lower index); each
  // round's winner is recorded in rank order and taken out of the row.  Exact, with the same
  // tie rule as rank_rows.
  __device__ __forceinline__ void topk_rows_warp(const float* lg) {
    const int B = p.B, E = p.E, K = p.K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    #pragma unroll 1
    for (int b = warp; b < B; b += kConsumerWarps) {
      float v[kMaxExperts / 32];
#pragma unroll
      for (int k = 0; k < kMaxExperts / 32; ++k) {
        const int e = lane + 32 * k;
        v[k] = e < E ? lg[b * E + e] : -INFINITY;
      }
      // logits as unsigned keys in the same order (-0 taken as +0, so that equal logits have
      // equal keys); a key of 0 is below every logit
      uint32_t key[kMaxExperts / 32];
#pragma unroll
      for (int k = 0; k < kMaxExperts / 32; ++k) {
        const uint32_t u = __float_as_uint(v[k] + 0.f);
        key[k] = lane + 32 * k < E ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
      }
      uint32_t taken = 0;   // this lane's values already chosen (bit k)
      #pragma unroll 1
      for (int j = 0; j < K; ++j) {
        // this lane's best (a strict > keeps the lower expert of equal keys), then the warp's
        // largest key and the lowest expert holding it, one warp reduction each
        uint32_t bk = 0u;
        int bi = 0x7fffffff;
#pragma unroll
        for (int k = 0; k < kMaxExperts / 32; ++k)
          if (!((taken >> k) & 1u) && key[k] > bk) { bk = key[k]; bi = lane + 32 * k; }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        bi = static_cast<int>(__reduce_min_sync(0xffffffffu, bk == mk ? static_cast<uint32_t>(bi) : 0x7fffffffu));
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == 0) {
          S.rids[b * K + j] = bi;
          S.rval[b * K + j] = __uint_as_float((mk & 0x80000000u) ? (mk & 0x7fffffffu) : ~mk);
          atomicAdd(&S.ecnt[bi], 1);
        }
      }
    }
  }

  // ------------------------------------------------------------------ routing (every block)
  // Every block routes the whole batch itself from the router logits (tagged words the
  // router tiles wrote), so the MoE of a layer needs nothing else from another block.
  // Top-k by logit, ties to the lower expert index: an expert's rank is the number of
  // experts with a larger logit plus those with an equal logit and a lower index; every
  // (row, expert) pair counts its own rank against the row's logits in shared memory, the
  // comparisons of a pair split over up to 8 threads.  Weights: exp(r - max) over the chosen
  // experts, renormalised over them (or over all experts when norm_topk == 0).  Then the
  // active experts, the cost split of the gate/up units over the blocks, and (batches that
  // fit) the normalised MoE input, all in shared memory; the block's producer is released to
  // stream the experts.
  __device__ __forceinline__ bool route_local() {
    const int l = meta().layer;
    const int B = p.B, E = p.E, K = p.K, H = p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* lg = S.moe;   // [B][E]
    twait = globaltimer();
    trace_mark(15, l);
    bool ok = true;
    // the normalised MoE input of every row stays in shared memory when it fits; x_mid is
    // complete before the router logits are, so it is staged first (unless the router tile
    // of this block already left it there)
    const bool cache_in = B <= TB && B * H <= kAttnScratch;
    if (cache_in && S.ykey != l) {
      int rb[TB];
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) rb[tb] = tb;
      ok = stage_input(2, l, H, rb, B, tg, S.scr.attn);
    }
    {
      const uint64_t* rl = p.RLOG + static_cast<size_t>(l) * p.max_batch * E;
      ok = ll_gather(p, B * E, [=](int i) { return rl + i; }, lg, tg) && ok;
    }
    #pragma unroll 1
    for (int e = threadIdx.x; e < E; e += kConsumerThreads) S.ecnt[e] = 0;
    if (!ok) ll_timeout(p, MK_OP_ROUTER, l, tg);
    if (!cbar_and(ok)) return false;
    trace_mark(16, l);
    if (!p.norm_topk) {   // weights over all experts need each row's max and normaliser
      #pragma unroll 1
      for (int b = warp; b < B; b += kConsumerWarps) {
        float mx = -INFINITY;
        #pragma unroll 1
        for (int e = lane; e < E; e += 32) mx = fmaxf(mx, lg[b * E + e]);
        mx = warp_max(mx);
        float z = 0.f;
        #pragma unroll 1
        for (int e = lane; e < E; e += 32) z += expf(lg[b * E + e] - mx);
        z = warp_sum(z);
        if (lane == 0) { S.rmax[b] = mx; S.rz[b] = z; }
      }
    }
    if (W && B >= 8) topk_rows_warp(lg);   // (only the tcgen05 instantiation sees such batches)
    else if (E <= 128) rank_rows<16>(lg);
    else rank_rows<32>(lg);
    cbar();
    trace_mark(18, l);
    // small-batch MoE: the logits are consumed; the scratch becomes the [B][H] partial output
    // (and a row that is not routed to a unit's expert contributes zero to it)
    if constexpr (kSmallMoe) {
      #pragma unroll 1
      for (int i = threadIdx.x; i < B * H; i += kConsumerThreads) S.moe[i] = 0.f;
      #pragma unroll 1
      for (int i = threadIdx.x; i < B * kMaxUnits; i += kConsumerThreads) S.hsm[i] = 0.f;
    }
    // combine weights (a warp per row, a lane per slot) ...
    #pragma unroll 1
    for (int b = warp; b < B; b += kConsumerWarps) {
      const int j = lane < K ? lane : 0;
      const float mx = p.norm_topk ? S.rval[b * K] : S.rmax[b];   // rank 0 holds the row's largest logit
      const float ex = expf(S.rval[b * K + j] - mx);
      const float sum = warp_sum(lane < K ? ex : 0.f);
      if (lane < K) {
        const int i = b * K + lane;
        const float wgt = p.norm_topk ? ex / sum : ex / S.rz[b];
        S.rcache[i] = S.rids[i];
        S.rwcache[i] = wgt;
        if (blockIdx.x == 0) {   // a copy for inspection
          p.RIDS[static_cast<size_t>(l) * p.max_batch * K + i] = S.rids[i];
          p.RW[static_cast<size_t>(l) * p.max_batch * K + i] = wgt;
        }
      }
    }
    // ... while the last warp lists the active experts and their gate/up cost prefix
    if (warp == kConsumerWarps - 1) {
      int nact = 0;
      #pragma unroll 1
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool on = e < E && S.ecnt[e] > 0;
        const uint32_t ball = __ballot_sync(0xffffffffu, on);
        if (on) S.eact[nact + __popc(ball & ((1u << lane) - 1u))] = e;
        nact += __popc(ball);
      }
      if (lane == 0) S.nact = nact;
      __syncwarp();
      // 8 experts per lane, then a warp scan
      int32_t loc[kMaxExperts / 32];
      int32_t run = 0;
#pragma unroll
      for (int k = 0; k < kMaxExperts / 32; ++k) {
        const int a = lane * (kMaxExperts / 32) + k;
        const int32_t cst = a < nact ? moe_unit_cost(S.ecnt[S.eact[a]], W) : 0;
        if (a < nact) S.ecost[a] = cst;
        run += cst * p.F;
        loc[k] = run;
      }
      int32_t x = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const int32_t before = x - run;
#pragma unroll
      for (int k = 0; k < kMaxExperts / 32; ++k) {
        const int a = lane * (kMaxExperts / 32) + k;
        if (a < nact) S.ecum[a + 1] = before + loc[k];
      }
      if (lane == 0) S.ecum[0] = 0;
      __syncwarp();
      // this block's gate/up units (the two ends by two lanes at once); the producer needs only
      // the active list and this range, so this warp hands them over at once (the arrival
      // releases the warp's writes, ordered by the warp barrier) while the other warps finish
      // the combine weights
      if (lane < 2) {
        const int32_t u = moe_gu_start(blockIdx.x + lane, p.n_ctas, S.ecum, S.ecost, nact, p.F);
        if (lane == 0) S.gu_lo = u; else S.gu_hi = u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.route_bar);
    }
    if (threadIdx.x == 0) S.ykey = cache_in ? l : -1;
    cbar();
    trace_mark(17, l);
    return true;
  }

  // (row, slot) pairs routed to expert e, ascending, into S.elist; returns their number
  __device__ int expert_pairs(int e) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, n = p.B * p.K;
    if (warp == 0) {
      int cnt = 0;
      #pragma unroll 1
      for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        const bool hit = i < n && S.rcache[i] == e;
        const uint32_t bal = __ballot_sync(0xffffffffu, hit);
        if (hit) S.elist[cnt + __popc(bal & ((1u << lane) - 1u))] = i;
        cnt += __popc(bal);
      }
      if (lane == 0) S.flag = cnt;
    }
    cbar();
    return S.flag;
  }

  // inputs of up to TB (row, slot) pairs from the cached MoE input
  __device__ __forceinline__ void load_y_smem(const Seg<TB>& sg, const int (&rb)[TB], int nt,
                                              float (&y)[8 / TB][8][TB]) {
    const float* yc = S.scr.attn;
#pragma unroll
    for (int j = 0; j < Seg<TB>::kUnits; ++j) {
      const int e = sg.unit(j);
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (e >= 0 && tb < nt) {
          a = *reinterpret_cast<const float4*>(yc + rb[tb] * p.H + e);
          b = *reinterpret_cast<const float4*>(yc + rb[tb] * p.H + e + 4);
        }
        y[j][0][tb] = a.x; y[j][1][tb] = a.y; y[j][2][tb] = a.z; y[j][3][tb] = a.w;
        y[j][4][tb] = b.x; y[j][5][tb] = b.y; y[j][6][tb] = b.z; y[j][7][tb] = b.w;
      }
    }
  }

  // routing slot of expert e in batch row b, or -1
  __device__ __forceinline__ int slot_of(int b, int e) const {
    int s = -1;
    #pragma unroll 1
    for (int j = 0; j < p.K; ++j)
      if (S.rcache[b * p.K + j] == e) s = j;
    return s;
  }

  // pairs b0 .. b0+nt-1 of the current expert's list: (row, slot); slot -1 past the end
  __device__ __forceinline__ void expert_rows(int b0, int nt, int (&rb)[TB], int (&rj)[TB]) {
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      const int ent = tb < nt ? S.elist[b0 + tb] : 0;
      rb[tb] = ent / p.K;
      rj[tb] = tb < nt ? ent - rb[tb] * p.K : -1;
    }
  }

  // ------------------------------------------------------------------ MoE down projection + combine
  // (row, slot) pairs of the batch routed to expert e, ascending, into this warp's list
  __device__ int warp_expert_pairs(int e, int* wl) {
    const int lane = threadIdx.x & 31, n = p.B * p.K;
    int cnt = 0;
    #pragma unroll 1
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      const bool hit = i < n && S.rcache[i] == e;
      const uint32_t bal = __ballot_sync(0xffffffffu, hit);
      if (hit) wl[cnt + __popc(bal & ((1u << lane) - 1u))] = i;
      cnt += __popc(bal);
    }
    __syncwarp();
    return cnt;
  }

  // SwiGLU activations of up to TD (row, slot) pairs into registers, from the shared-memory
  // copy (hc) or from the tagged global buffer
  // The same from the tagged global buffer for pair groups of wide batches: the loads of half
  // the units go out together (one L2 round trip per half; a stale word sends its half again)
  template <int TD>
  __device__ __forceinline__ bool load_h_pairs_ll(const Seg<TD>& sg, int l, const int* pr, int nt,
                                                  float (&y)[8 / TD][8][TD]) {
    constexpr int kU = Seg<TD>::kUnits;
    const uint64_t* src[TD];
#pragma unroll
    for (int tb = 0; tb < TD; ++tb)
      src[tb] = p.HB + (static_cast<size_t>(l) * p.max_batch * p.K + pr[tb < nt ? tb : 0]) * p.F;
    bool ok = true;
#pragma unroll
    for (int h0 = 0; h0 < kU; h0 += kU / 2) {
      LL_RETRY_BEGIN
#pragma unroll
      for (int j = h0; j < h0 + kU / 2; ++j) {
        const int e = sg.unit(j);
#pragma unroll
        for (int tb = 0; tb < TD; ++tb) {
          if (e >= 0 && tb < nt) {
#pragma unroll
            for (int q = 0; q < 8; q += 2) {
              uint64_t a, b;
              ll_ld2(src[tb] + e + q, a, b);
              st_ |= ll_stale(a, tg) | ll_stale(b, tg);
              y[j][q][tb] = ll_f(a);
              y[j][q + 1][tb] = ll_f(b);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) y[j][q][tb] = 0.f;
          }
        }
      }
      LL_RETRY_END(ok)
    }
    return ok;
  }

  template <int TD>
  __device__ __forceinline__ bool load_h_pairs(const Seg<TD>& sg, int l, const float* hc, const int* pr, int nt,
                                               float (&y)[8 / TD][8][TD]) {
    if constexpr (TD > 1 && TB == 4) {   // (batches of two take the small-batch path by default)
      if (hc == nullptr) return load_h_pairs_ll<TD>(sg, l, pr, nt, y);
    }
    bool ok = true;
#pragma unroll
    for (int j = 0; j < Seg<TD>::kUnits; ++j) {
      const int e = sg.unit(j);
#pragma unroll
      for (int tb = 0; tb < TD; ++tb) {
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (e >= 0 && tb < nt) {
          const int i = pr[tb];   // row * K + slot
          if (hc != nullptr) {
            const float4 a = *reinterpret_cast<const float4*>(hc + static_cast<size_t>(i) * p.F + e);
            const float4 b = *reinterpret_cast<const float4*>(hc + static_cast<size_t>(i) * p.F + e + 4);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
          } else {
            const H8 h = load_h8(p, p.HB + (static_cast<size_t>(l) * p.max_batch * p.K + i) * p.F + e, tg);
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = h.v[q];
            ok = h.ok && ok;
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) y[j][q][tb] = v[q];
      }
    }
    return ok;
  }

  // This block owns hidden rows [lo, hi) of every active expert's down projection.  A chunk
  // holds `n` experts' blocks of `aux` rows (rows row0 .. row0+aux-1), experts idx .. idx+n-1 of
  // the layer's active list, one block after the other.  Warp w takes a contiguous share of
  // the chunk's rows; for each expert in its share it lists the (row, slot) pairs routed there
  // and dots their SwiGLU activations with the rows.  Every product w_j * (Wd_j . h_j) lands once
  // in shared memory; after the last chunk the slots are summed in slot order and added to
  // x_mid.
  template <int TD>
  __device__ __forceinline__ bool moe_down_t() {
    const Meta m0 = meta();
    const int l = m0.layer;
    const int B = p.B, K = p.K, F = p.F;
    const int r0 = static_cast<int>(m0.lo), nrow = static_cast<int>(m0.hi) - r0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t xs = static_cast<size_t>(p.max_batch) * p.H;
    twait = globaltimer();
    if (m0.n == 0) return true;   // no hidden rows here, or nothing routed
    float* P = S.moe;                                  // [B][K][nrow] products
    float* XM = P + B * K * nrow;                      // [B][nrow] x_mid of the block's rows
    const int hoff = (B * K * nrow + B * nrow + 3) & ~3;
    float* hc = (hoff + B * K * F <= kMoeScratch) ? S.moe + hoff : nullptr;   // [B][K][F] SwiGLU inputs
    trace_mark(40, l);
    bool ok = true;
    {
      // x_mid of the block's own rows (written by its O-proj tile), and the SwiGLU inputs
      #pragma unroll 1
      for (int i = threadIdx.x; i < B * nrow; i += kConsumerThreads) {
        const int t = i / nrow, r = i - t * nrow;
        XM[i] = ll_f(ll_ld(p.X + (2 * static_cast<size_t>(l) + 1) * xs + static_cast<size_t>(t) * p.H + r0 + r));
      }
      if (hc != nullptr) {
        const uint64_t* src = p.HB + static_cast<size_t>(l) * p.max_batch * K * F;
        ok = ll_gather(p, B * K * F, [=](int i) { return src + i; }, hc, tg);
      }
      if (!ok) ll_timeout(p, MK_OP_MOE, l, tg);
      if (!cbar_and(ok)) return false;
    }
    trace_mark(41, l);
    const Seg<TD> sg(F);
    int* wl = S.wlist[warp];
    for (;;) {
      const int ne = meta().n, nrc = static_cast<int>(meta().aux), rb0 = static_cast<int>(meta().row0);
      const int a0 = static_cast<int>(meta().idx);
      const bool last = meta().last;
      const uint8_t* wsm = slot();
      if constexpr (TB == 4) {
        if (B >= 16) {
          // wide batches: the chunk's (expert, group of TD pairs) units are dealt over the
          // warps; a warp fetches its pairs' SwiGLU inputs once and runs all of the expert's
          // rows in the chunk against them
          int gbase = 0;   // pair groups of the chunk's earlier experts
          #pragma unroll 1
          for (int ai = 0; ai < ne; ++ai) {
            const int cnt = warp_expert_pairs(S.eact[a0 + ai], wl);
            const int ng = (cnt + TD - 1) / TD;
            const int i0 = ai * nrc, iend = i0 + nrc;
            #pragma unroll 1
            for (int g = (warp + kConsumerWarps - gbase % kConsumerWarps) % kConsumerWarps; g < ng;
                 g += kConsumerWarps) {
              const int g0 = g * TD, nt = min(TD, cnt - g0);
              float y[8 / TD][8][TD];
              ok = load_h_pairs<TD>(sg, l, hc, wl + g0, nt, y) && ok;
              for (int ii = i0; ii < iend; ii += 2) {
                float a[TD], b[TD];
#pragma unroll
                for (int tb = 0; tb < TD; ++tb) { a[tb] = 0.f; b[tb] = 0.f; }
                row_dot<TD>(wsm + static_cast<size_t>(ii) * F * 2, sg, y, a);
                if (ii + 1 < iend) row_dot<TD>(wsm + static_cast<size_t>(ii + 1) * F * 2, sg, y, b);
                warp_sum2<TD>(a, b);
                const int tb = lane & 15;
                const int row = lane < 16 ? ii : ii + 1;
                if (tb < nt && row < iend) {
                  const int pi = wl[g0 + tb];
                  P[pi * nrow + rb0 + (row - i0) - r0] = S.rwcache[pi] * pick<TD>(a, tb);
                }
              }
            }
            gbase += ng;
          }
          if (last) break;
          if (!next_rec()) break;
          continue;
        }
      }
      const int R = ne * nrc;
      const int i1 = (warp + 1) * R / kConsumerWarps;
      #pragma unroll 1
      for (int i = warp * R / kConsumerWarps; i < i1;) {
        const int ai = i / nrc;
        const int iend = min(i1, (ai + 1) * nrc);
        const int cnt = warp_expert_pairs(S.eact[a0 + ai], wl);
        #pragma unroll 1
        for (int g0 = 0; g0 < cnt; g0 += TD) {
          const int nt = min(TD, cnt - g0);
          float y[8 / TD][8][TD];
          ok = load_h_pairs<TD>(sg, l, hc, wl + g0, nt, y) && ok;
          for (int ii = i; ii < iend; ii += 2) {
            // two rows in flight, one paired reduction (lanes 0-15: row ii, 16-31: row ii+1)
            float a[TD], b[TD];
#pragma unroll
            for (int tb = 0; tb < TD; ++tb) { a[tb] = 0.f; b[tb] = 0.f; }
            row_dot<TD>(wsm + static_cast<size_t>(ii) * F * 2, sg, y, a);
            if (ii + 1 < iend) row_dot<TD>(wsm + static_cast<size_t>(ii + 1) * F * 2, sg, y, b);
            warp_sum2<TD>(a, b);
            const int tb = lane & 15;
            const int row = lane < 16 ? ii : ii + 1;
            if (tb < nt && row < iend) {
              const int pi = wl[g0 + tb];
              const int r = rb0 + (row - ai * nrc) - r0;
              P[pi * nrow + r] = S.rwcache[pi] * pick<TD>(a, tb);
            }
          }
        }
        i = iend;
      }
      if (last) break;
      if (!next_rec()) break;
    }
    if (!ok) ll_timeout(p, MK_OP_MOE, l, tg);
    if (!cbar_and(wok && ok)) return false;
    trace_mark(42, l);
    // combine in slot order, residual
    #pragma unroll 1
    for (int t = warp; t < B; t += kConsumerWarps) {
      #pragma unroll 1
      for (int r = lane; r < nrow; r += 32) {
        float acc = 0.f;
        #pragma unroll 1
        for (int j = 0; j < K; ++j) acc += P[(t * K + j) * nrow + r];
        ll_st(p.X + (2 * static_cast<size_t>(l) + 2) * xs + static_cast<size_t>(t) * p.H + r0 + r,
              XM[t * nrow + r] + acc, tg);
      }
    }
    return true;
  }

  __device__ bool moe_down() { return moe_down_t<(TB > 2 ? 2 : TB)>(); }

  // ------------------------------------------------------------------ small-batch MoE
  // One chunk of the transposed down projection: rows f = row0 .. row0+n-1 of expert idx
  // ([H] each, bf16), whose weighted SwiGLU outputs this block computed in the preceding
  // gate/up tile.  Thread t owns the 8-column groups c = 8 * (t + 256 k) of the [B][H] partial
  // output in shared memory: it adds h_b[f] * Wd^T[f][c..c+8) for every row f (no reductions).
  __device__ __forceinline__ bool moe_dt() {
    const Meta m0 = meta();
    const int H = p.H, B = p.B, n = m0.n, u0 = static_cast<int>(m0.aux);
    twait = globaltimer();
    const uint8_t* wsm = slot();
    float* acc = S.moe;
    const float* hs = S.hsm;
    for (int c8 = threadIdx.x * 8; c8 < H; c8 += kConsumerThreads * 8) {
      float a[kSmallMaxB][8];
#pragma unroll
      for (int tb = 0; tb < kSmallMaxB; ++tb) {
        float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
        if (tb < B) {
          x0 = *reinterpret_cast<const float4*>(acc + tb * H + c8);
          x1 = *reinterpret_cast<const float4*>(acc + tb * H + c8 + 4);
        }
        a[tb][0] = x0.x; a[tb][1] = x0.y; a[tb][2] = x0.z; a[tb][3] = x0.w;
        a[tb][4] = x1.x; a[tb][5] = x1.y; a[tb][6] = x1.z; a[tb][7] = x1.w;
      }
#pragma unroll 4
      for (int r = 0; r < n; ++r) {
        float wf[8];
        unpack8(*reinterpret_cast<const uint4*>(wsm + (static_cast<size_t>(r) * H + c8) * 2), wf);
        const int u = u0 + r < kMaxUnits ? u0 + r : kMaxUnits - 1;
#pragma unroll
        for (int tb = 0; tb < kSmallMaxB; ++tb) {
          if (tb < B) {
            const float h = hs[tb * kMaxUnits + u];
#pragma unroll
            for (int q = 0; q < 8; ++q) a[tb][q] = fmaf(h, wf[q], a[tb][q]);
          }
        }
      }
#pragma unroll
      for (int tb = 0; tb < kSmallMaxB; ++tb) {
        if (tb < B) {
          *reinterpret_cast<float4*>(acc + tb * H + c8) = make_float4(a[tb][0], a[tb][1], a[tb][2], a[tb][3]);
          *reinterpret_cast<float4*>(acc + tb * H + c8 + 4) = make_float4(a[tb][4], a[tb][5], a[tb][6], a[tb][7]);
        }
      }
    }
    return true;   // the next record starts behind a block barrier
  }

  // Reduction record of the small-batch MoE: publish this block's [B][H] partial output, then
  // for the block's hidden rows [lo, hi): gather every block's partial (one batch of loads),
  // sum them in block order per lane group and by a warp reduction, add x_mid, and write the
  // layer output.
  __device__ __forceinline__ bool moe_reduce() {
    const Meta m0 = meta();
    const int l = m0.layer, B = p.B, H = p.H, N = p.n_ctas;
    const int r0 = static_cast<int>(m0.lo), nrow = static_cast<int>(m0.hi) - r0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t xs = static_cast<size_t>(p.max_batch) * H;
    twait = globaltimer();
    trace_mark(40, l);
    {
      uint64_t* mine = p.PT + (static_cast<size_t>(l) * N + blockIdx.x) * kSmallMaxB * H;
      #pragma unroll 1
      for (int i = threadIdx.x * 2; i < B * H; i += kConsumerThreads * 2) ll_st2(mine + i, S.moe[i], S.moe[i + 1], tg);
    }
    cbar();   // the partial output has been read out of the scratch
    if (nrow <= 0) return true;
    // one batch of loads: x_mid of the block's rows ([B][nrow], written by its O-proj tile),
    // then every block's partial for them ([B][N][nrow])
    const int ni = B * nrow;
    const uint64_t* xmid = p.X + (2 * static_cast<size_t>(l) + 1) * xs + r0;
    const uint64_t* pt = p.PT + static_cast<size_t>(l) * N * kSmallMaxB * H + r0;
    const FastDiv dnr(nrow), dbn(N * nrow);   // indices below ni + B * N * nrow <= the scratch size < 2^16
    bool ok = ll_gather(p, ni + B * N * nrow, [=](int i) {
      if (i < ni) {
        const int b = dnr.div(i);
        return xmid + static_cast<size_t>(b) * H + (i - b * nrow);
      }
      const int q = i - ni, b = dbn.div(q), rem = q - b * N * nrow;
      const int j = dnr.div(rem), rr = rem - j * nrow;
      return pt + (static_cast<size_t>(j) * kSmallMaxB + b) * H + rr;
    }, S.moe, tg);
    if (!ok) ll_timeout(p, MK_OP_MOE, l, tg);
    if (!cbar_and(ok)) return false;
    trace_mark(42, l);
    const float* part = S.moe + ni;
    #pragma unroll 1
    for (int k = 0; k * kConsumerWarps < ni; ++k) {   // warp-uniform trip count
      const int it = warp + k * kConsumerWarps;
      const int b = it < ni ? it / nrow : 0, rr = it - b * nrow;
      float v = 0.f;
      if (it < ni)
        #pragma unroll 1
        for (int j = lane; j < N; j += 32) v += part[(b * N + j) * nrow + rr];
      v = warp_sum(v);
      if (it < ni && lane == 0)
        ll_st(p.X + (2 * static_cast<size_t>(l) + 2) * xs + static_cast<size_t>(b) * H + r0 + rr, S.moe[it] + v, tg);
    }
    return true;
  }


  // ------------------------------------------------------------------ attention split item
  // Tensor cores: per 16 positions, S^T (positions x 8 grouped query heads) = K . Q^T with K
  // loaded by ldmatrix from the swizzled tiles and Q^T held in registers, then an online
  // softmax per head and O^T (dims x heads) += V^T . P^T, V^T by ldmatrix.trans and P^T by a
  // register transpose of the score fragment.  Q and P are split into bf16 hi + lo parts
  // (two MMAs each) so that the products keep ~16 bits: K and V are exact in bf16.
  // Warp w takes the 16-position tiles w, w+8, ... of each chunk; at the end of the item
  // the warps merge their (max, sum, output) states and the split's partial goes to
  // global memory; the last split of (row, KV head) merges all splits in split order.
  // A bf16 chunk is page-major: page i holds its K then its V, each as [dim half][position][64
  // dims] in lines of 128 bytes, and 16-byte piece j of line n sits at piece j ^ (n & 7) (TMA
  // 128-byte swizzle; every page starts on a 1024-byte boundary, page_size is a multiple of 8).
  // kv_line: the line of dims 0 .. 63 of chunk position r of K (which = 0) or V (which = 1);
  // kv_at: the byte offset of dims d .. d + 7 of that position.
  __device__ __forceinline__ int kv_line(int which, int r) const {
    const int pg = r / p.ps;
    return (2 * pg + which) * (D / 64) * p.ps + (r - pg * p.ps);
  }
  // the same for position r0 + x of a 16-position tile whose first page is pg0 = r0 / page_size
  // (x < 16, so at most one page boundary lies inside the tile)
  __device__ __forceinline__ int kv_line_in(int which, int r0, int pg0, int x) const {
    int pg = pg0, rr = r0 - pg0 * p.ps + x;
    if (rr >= p.ps) { rr -= p.ps; ++pg; }
    return (2 * pg + which) * (D / 64) * p.ps + rr;
  }
  __device__ __forceinline__ uint32_t kv_at(int line0, int d) const {
    const int n = line0 + (d >> 6) * p.ps;
    return static_cast<uint32_t>(n * 128 + ((((d & 63) >> 3) ^ (n & 7)) << 4) + (d & 7) * 2);
  }

  // q8_0 chunks: the slot holds [K codes][V codes][K scales][V scales] of pages_per_chunk_q8 pages,
  // codes as rows of D bytes with the TMA 128-byte swizzle (16-byte piece j of row r at piece
  // j ^ (r & 7)), scales as rows of D / 32 f16.  A warp takes 32 rows at a time (two 16-row
  // halves under one softmax update).  Codes become fp16 exactly, straight into MMA fragments:
  //  * S^T = K Q^T per 32-dim block: ldmatrix (b16) hands lane (g, t) bytes 4t .. 4t + 3 of a
  //    16-byte piece of rows g and g + 8; q's fragment takes its dims in that order.  Each
  //    block's partial is multiplied by the row's K scale.
  //  * O^T += V^T P^T per 32-dim block: ldmatrix.trans (b16) hands lane (g, t) dims 2g, 2g + 1
  //    of rows 2t and 2t + 1, so output row g of tile m is dim 16m + 2g and row g + 8 is dim
  //    16m + 2g + 1 (undone where o is stored).  The rows' V scales are folded into P.
  // P carries a factor 2^6 (in the exponent, so ls carries it too and o / ls is unchanged) that
  // keeps small P x scale products out of fp16's subnormal range.  Rows past the sequence are
  // masked (their codes are finite; their V scales are replaced by 0).
  static __device__ __forceinline__ uint32_t swz8(int r, int c) {
    return static_cast<uint32_t>(r * D + ((((c >> 4) ^ r) & 7) << 4) + (c & 15));
  }
  static __device__ __forceinline__ uint2 lds_v2(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
  }
  static __device__ __forceinline__ void f16x4_f32(uint2 v, float (&f)[4]) {
    const __half2 a = *reinterpret_cast<const __half2*>(&v.x), b = *reinterpret_cast<const __half2*>(&v.y);
    f[0] = __low2float(a); f[1] = __high2float(a); f[2] = __low2float(b); f[3] = __high2float(b);
  }
  __device__ __forceinline__ void attn_chunks_q8(int Lc, int pos, const uint16_t* kvcur, float (&o)[D / 16][4],
                                                 float (&mx)[2], float (&ls)[2]) {
    constexpr int NB = D / 32;   // scale blocks per row
    static_assert(NB == 4, "one 8-byte load holds a row's scales");
    constexpr float kLnP = 4.15888308336f;   // ln(2^6)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lpc = lane >> 4;   // ldmatrix row and piece of this lane
    const uint4* qf = reinterpret_cast<const uint4*>(S.scr.attn);
    const int rows_cap = pages_per_chunk_q8(p.ps, D) * p.ps;
    for (;;) {
      const int p0 = static_cast<int>(meta().row0) * p.ps;            // first position of the chunk
      const int npos = min(static_cast<int>(meta().n) * p.ps, Lc - p0);
      const bool last = meta().last;
      uint8_t* sl8 = const_cast<uint8_t*>(slot());
      const uint32_t Kc = smem_u32(sl8);
      const uint32_t Vc = Kc + rows_cap * D;
      const uint32_t Ks = Kc + 2 * rows_cap * D;                       // K scales, 8 bytes a row
      const uint32_t Vs = Ks + rows_cap * NB * 2;
#pragma unroll 1
      for (int tile = warp; tile * 32 < npos; tile += kConsumerWarps) {
        const int r0 = tile * 32;
        if (pos >= p0 + r0 && pos < p0 + r0 + 32) {
          // this token's codes and scales are not in the copied page yet: put them in its rows
          const int rr = pos - p0;
          const uint8_t* c8 = reinterpret_cast<const uint8_t*>(kvcur);
#pragma unroll 1
          for (int cidx = lane; cidx < 2 * (D / 16); cidx += 32) {
            const int which = cidx / (D / 16), d = (cidx - which * (D / 16)) * 16;
            const uint4 v = *reinterpret_cast<const uint4*>(c8 + which * D + d);
            const uint32_t a = (which ? Vc : Kc) + swz8(rr, d);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          }
          if (lane < 2 * NB) {
            const uint16_t* s8 = reinterpret_cast<const uint16_t*>(c8 + 2 * D);
            uint16_t* sc16 = reinterpret_cast<uint16_t*>(sl8 + 2 * rows_cap * D);
            (lane < NB ? sc16 : sc16 + rows_cap * NB)[rr * NB + (lane % NB)] = s8[lane];
          }
          fence_proxy_async_smem();   // these generic writes precede the slot's next TMA fill
          __syncwarp();
        }
        // S^T = K Q^T for both halves, block by block
        float sc[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ra = r0 + 16 * h + g;
          float kd[2][4];
          f16x4_f32(lds_v2(Ks + ra * (NB * 2)), kd[0]);
          f16x4_f32(lds_v2(Ks + (ra + 8) * (NB * 2)), kd[1]);
          sc[h][0] = sc[h][1] = sc[h][2] = sc[h][3] = 0.f;
          const int lr = r0 + 16 * h + lrow;
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            uint32_t x[4];   // rows g, g + 8 of piece 2b, then of piece 2b + 1
            ldsm_x4(Kc + swz8(lr, 16 * (2 * b + lpc)), x);
            float ab[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const uint32_t xa = x[2 * h2], xb = x[2 * h2 + 1];
              const uint32_t a[4] = {s8_to_f16x2(xa, 0x4140u), s8_to_f16x2(xb, 0x4140u), s8_to_f16x2(xa, 0x4342u),
                                     s8_to_f16x2(xb, 0x4342u)};
              const uint4 q = qf[(2 * b + h2) * 32 + lane];
              mma_f16(ab, a, q.x, q.y);
              mma_f16(ab, a, q.z, q.w);
            }
            sc[h][0] = fmaf(ab[0], kd[0][b], sc[h][0]);
            sc[h][1] = fmaf(ab[1], kd[0][b], sc[h][1]);
            sc[h][2] = fmaf(ab[2], kd[1][b], sc[h][2]);
            sc[h][3] = fmaf(ab[3], kd[1][b], sc[h][3]);
          }
          if (ra >= npos) { sc[h][0] = -INFINITY; sc[h][1] = -INFINITY; }
          if (ra + 8 >= npos) { sc[h][2] = -INFINITY; sc[h][3] = -INFINITY; }
        }
        // online softmax per head column (heads 2t, 2t+1 on this lane), over the 32 rows
        float pr[2][2][2], cr[2];   // [half][row g / g + 8][head]
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float tm = fmaxf(fmaxf(sc[0][j], sc[0][j + 2]), fmaxf(sc[1][j], sc[1][j + 2]));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
          const float mn = fmaxf(mx[j], tm);
          const float me = mn - kLnP;
          cr[j] = mx[j] == -INFINITY ? 0.f : __expf(mx[j] - mn);
          float sum = 0.f;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            pr[h][0][j] = sc[h][j] == -INFINITY ? 0.f : __expf(sc[h][j] - me);
            pr[h][1][j] = sc[h][j + 2] == -INFINITY ? 0.f : __expf(sc[h][j + 2] - me);
            sum += pr[h][0][j] + pr[h][1][j];
          }
          ls[j] = ls[j] * cr[j] + sum;
          mx[j] = mn;
        }
#pragma unroll
        for (int mm = 0; mm < D / 16; ++mm) {
          o[mm][0] *= cr[0]; o[mm][1] *= cr[1]; o[mm][2] *= cr[0]; o[mm][3] *= cr[1];
        }
        // O^T += V^T P^T, per half and block, with the block's V scales in P
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ra = r0 + 16 * h + g;
          float vd[2][4];
          f16x4_f32(lds_v2(Vs + ra * (NB * 2)), vd[0]);
          f16x4_f32(lds_v2(Vs + (ra + 8) * (NB * 2)), vd[1]);
          const bool va_on = ra < npos, vb_on = ra + 8 < npos;
          const int lr = r0 + 16 * h + lrow;
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const float va = va_on ? vd[0][b] : 0.f, vb = vb_on ? vd[1][b] : 0.f;
            uint32_t xa_h, xa_l, xb_h, xb_l;
            split_f16x2(pr[h][0][0] * va, pr[h][0][1] * va, xa_h, xa_l);
            split_f16x2(pr[h][1][0] * vb, pr[h][1][1] * vb, xb_h, xb_l);
            const uint32_t b0h = movmatrix_t(xa_h), b0l = movmatrix_t(xa_l);
            const uint32_t b1h = movmatrix_t(xb_h), b1l = movmatrix_t(xb_l);
            uint32_t y[4];   // rows 0-7 and 8-15 of piece 2b, then of piece 2b + 1, transposed
            ldsm_x4_t(Vc + swz8(lr, 16 * (2 * b + lpc)), y);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t a[4] = {s8_to_f16x2(y[2 * u], 0x4240u), s8_to_f16x2(y[2 * u], 0x4341u),
                                     s8_to_f16x2(y[2 * u + 1], 0x4240u), s8_to_f16x2(y[2 * u + 1], 0x4341u)};
              mma_f16(o[2 * b + u], a, b0h, b1h);
              mma_f16(o[2 * b + u], a, b0l, b1l);
            }
          }
        }
      }
      if (last) break;
      if (!next_rec()) break;
    }
  }

  __device__ __forceinline__ bool attn_item() {
    constexpr int KS = D / 16;                              // k-steps over head dims (Q K^T)
    constexpr int MT = D / 16;                              // 16-dim tiles of the output (P V)
    const Meta m0 = meta();
    const int l = m0.layer;
    twait = globaltimer();
    const mk_attn_item item = p.items[m0.idx];
    const int b = item.b, kvh = item.kvh, Gq = p.G;
    const int Lc = p.seq_lens[b];
    const int pos = Lc - 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    // Q^T as the B operand of S^T = K Q^T, one 16-byte fragment per (k-step, lane):
    // lane (g, t) holds head g at dims 16s + 2t (+1) and 16s + 2t + 8 (+1) (with a q8_0 cache:
    // dims 16s + 4t .. 16s + 4t + 3, the order its K fragments are read in), hi then lo parts
    // of the rotated, scaled q (zero for heads at or above G); then this token's k and v.
    // Every tagged load of the prologue is issued before the first is used.
    uint4* qf = reinterpret_cast<uint4*>(S.scr.attn);                     // [KS][32]
    uint16_t* kvcur = reinterpret_cast<uint16_t*>(S.scr.attn + KS * 32 * 4);  // [2][D]
    if (threadIdx.x == 0) S.ykey = -1;                                // the MoE input cache shares this storage
    const uint64_t* qkv = p.QKV + (static_cast<size_t>(l) * p.max_batch + b) * p.nqkv;
    const float* cs = p.rope_cos + static_cast<size_t>(b) * (D / 2);
    const float* sn = p.rope_sin + static_cast<size_t>(b) * (D / 2);
    bool ok = true;
    {
      const int i = threadIdx.x;
      const bool qunit = i < KS * 32;
      const int s2 = i >> 5, gg = (i >> 2) & 7, tt = i & 3;
      const bool qon = qunit && gg < Gq;
      const uint64_t* qh = qkv + (kvh * Gq + gg) * D;
      const bool kvon = i < D;
      const uint64_t* kh = qkv + (p.Hq + kvh) * D;
      const uint64_t* vh = qkv + (p.Hq + p.Hkv + kvh) * D;
      const int dk = i, dko = i < D / 2 ? i + D / 2 : i - D / 2;
      // words: q (raw, rotation partner) x 4 dims, k (raw, partner), v
      const uint64_t* wp[11];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int d = Q8 ? 16 * s2 + 4 * tt + j : 16 * s2 + 2 * tt + 8 * (j >> 1) + (j & 1);
        wp[2 * j] = qh + d;
        wp[2 * j + 1] = qh + (d < D / 2 ? d + D / 2 : d - D / 2);
      }
      wp[8] = kh + dk; wp[9] = kh + dko; wp[10] = vh + dk;
      const uint32_t need = (qon ? 0xffu : 0u) | (kvon ? 0x700u : 0u);
      uint64_t w[11];
#pragma unroll
      for (int k = 0; k < 11; ++k) w[k] = ((need >> k) & 1u) ? ll_ld(wp[k]) : 0ull;
      uint32_t stale = 0;
#pragma unroll
      for (int k = 0; k < 11; ++k) stale |= static_cast<uint32_t>(((need >> k) & 1u) && !ll_ok(w[k], tg)) << k;
      if (stale != 0u) {   // re-poll the stale words, all of them per sweep
        const uint64_t t0 = globaltimer();
        #pragma unroll 1
        for (uint32_t it = 1; stale != 0u; ++it) {
#pragma unroll
          for (int k = 0; k < 11; ++k)
            if ((stale >> k) & 1u) w[k] = ll_ld(wp[k]);
          uint32_t still = 0;
#pragma unroll
          for (int k = 0; k < 11; ++k) still |= static_cast<uint32_t>(((stale >> k) & 1u) && !ll_ok(w[k], tg)) << k;
          stale = still;
          if (stale != 0u && (it & 15u) == 0u && (aborted(p) || globaltimer() - t0 > p.watchdog_ns)) {
            ok = false;
            break;
          }
        }
      }
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (qon) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int d = Q8 ? 16 * s2 + 4 * tt + j : 16 * s2 + 2 * tt + 8 * (j >> 1) + (j & 1);
          const int dh = d % (D / 2);
          const float raw = ll_f(w[2 * j]), other = ll_f(w[2 * j + 1]);
          const float c = __ldg(cs + dh), sv = __ldg(sn + dh);
          v[j] = (d < D / 2 ? raw * c - other * sv : raw * c + other * sv) * p.scale;
        }
      }
      if (qunit) {
        uint4 f;
        if constexpr (Q8) {   // the q8_0 tile multiplies codes in fp16 (exact) by fp16 parts of q
          split_f16x2(v[0], v[1], f.x, f.z);
          split_f16x2(v[2], v[3], f.y, f.w);
        } else {
          split_bf16x2(v[0], v[1], f.x, f.z);
          split_bf16x2(v[2], v[3], f.y, f.w);
        }
        qf[i] = f;
      }
      if constexpr (Q8) {
        // q8_0 blocks of this token's k (after RoPE) and v, from their fp32 values: a warp per 32
        // dims (warps past head_dim / 32 take part in the reductions with zeros)
        float kf = 0.f, vf = 0.f;
        if (kvon) {
          const float raw = ll_f(w[8]), other = ll_f(w[9]);
          const float c = __ldg(cs + (i % (D / 2))), sv = __ldg(sn + (i % (D / 2)));
          kf = i < D / 2 ? raw * c - other * sv : raw * c + other * sv;
          vf = ll_f(w[10]);
        }
        const float ka = warp_max(fabsf(kf)), va = warp_max(fabsf(vf));
        if (kvon) {
          const float dk = ka / 127.0f, dv = va / 127.0f;
          const float ik = dk != 0.f ? 1.0f / dk : 0.f, iv = dv != 0.f ? 1.0f / dv : 0.f;
          uint8_t* c8 = reinterpret_cast<uint8_t*>(kvcur);          // [2][D] codes, then [2][D/32] scales
          c8[i] = static_cast<uint8_t>(static_cast<int8_t>(roundf(kf * ik)));
          c8[D + i] = static_cast<uint8_t>(static_cast<int8_t>(roundf(vf * iv)));
          if ((i & 31) == 0) {
            uint16_t* s8 = reinterpret_cast<uint16_t*>(c8 + 2 * D);
            s8[i >> 5] = __half_as_ushort(__float2half_rn(dk));
            s8[D / 32 + (i >> 5)] = __half_as_ushort(__float2half_rn(dv));
          }
        }
      } else if (kvon) {
        const float raw = ll_f(w[8]), other = ll_f(w[9]);
        const float c = __ldg(cs + (i % (D / 2))), sv = __ldg(sn + (i % (D / 2)));
        kvcur[i] = to_bf16_bits(i < D / 2 ? raw * c - other * sv : raw * c + other * sv);
        kvcur[D + i] = to_bf16_bits(ll_f(w[10]));
      }
    }
    if (!ok) ll_timeout(p, MK_OP_ATTN, l, tg);
    if (!cbar_and(ok)) return false;
    if (item.split == 0) {
      // append this token's k and v to the cache
      const int pg = pos / p.ps, sl = pos % p.ps;
      const int32_t page = __ldg(p.block_tables + static_cast<size_t>(b) * p.maxpg + pg);
      if (page >= 0 && page < p.P) {
        if constexpr (Q8) {
          uint8_t* base = reinterpret_cast<uint8_t*>(p.kv) + l * p.kv_layer_bytes;
          const size_t rowk = ((static_cast<size_t>(page) * 2) * p.Hkv + kvh) * p.ps + sl;
          const size_t rowv = rowk + static_cast<size_t>(p.Hkv) * p.ps;
          const uint8_t* c8 = reinterpret_cast<const uint8_t*>(kvcur);
#pragma unroll 1
          for (int d = threadIdx.x; d < D; d += kConsumerThreads) {
            base[rowk * D + d] = c8[d];
            base[rowv * D + d] = c8[D + d];
          }
          if (threadIdx.x < D / 32) {
            uint16_t* sb = reinterpret_cast<uint16_t*>(base + p.kv_code_bytes);
            const uint16_t* s8 = reinterpret_cast<const uint16_t*>(c8 + 2 * D);
            sb[rowk * (D / 32) + threadIdx.x] = s8[threadIdx.x];
            sb[rowv * (D / 32) + threadIdx.x] = s8[D / 32 + threadIdx.x];
          }
        } else {
          const size_t kb = (((static_cast<size_t>(l) * p.P + page) * 2 * p.Hkv + kvh) * p.ps + sl) * D;
          const size_t vb = kb + static_cast<size_t>(p.Hkv) * p.ps * D;
#pragma unroll 1
          for (int d = threadIdx.x; d < D; d += kConsumerThreads) {
            p.kv[kb + d] = kvcur[d];
            p.kv[vb + d] = kvcur[D + d];
          }
        }
      } else if (threadIdx.x == 0) {
        record_error(p, MK_ERR_DEVICE_BOUNDS, MK_OP_ATTN, l, 0u, static_cast<uint32_t>(page), 0, pg,
                     false);
      }
    }
    trace_mark(61, l);
    float o[MT][4];
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) o[mm][0] = o[mm][1] = o[mm][2] = o[mm][3] = 0.f;
    float mx[2] = {-INFINITY, -INFINITY}, ls[2] = {0.f, 0.f};   // heads 2t, 2t+1 (ls: this lane's share)

    if constexpr (Q8) {
      attn_chunks_q8(Lc, pos, kvcur, o, mx, ls);
    } else for (;;) {
      const int p0 = static_cast<int>(meta().row0) * p.ps;            // first position of the chunk
      const int npos = min(static_cast<int>(meta().n) * p.ps, Lc - p0);
      const bool last = meta().last;
      const uint32_t Kb = smem_u32(slot());
      for (int tile = warp; tile * 16 < npos; tile += kConsumerWarps) {
        const int r0 = tile * 16;
        bool patched = false;
        if (pos >= p0 + r0 && pos < p0 + r0 + 16) {
          // this token's k and v are not in the copied page yet: put them in its rows
          const int rr = pos - p0;
          #pragma unroll 1
          for (int cidx = lane; cidx < 2 * (D / 8); cidx += 32) {
            const int which = cidx / (D / 8), d = (cidx - which * (D / 8)) * 8;
            const uint4 v = *reinterpret_cast<const uint4*>(kvcur + which * D + d);
            const uint32_t a = Kb + kv_at(kv_line(which, rr), d);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          }
          patched = true;
        }
        if (r0 + 16 > npos) {
          // rows past the sequence: zero them so that 0-probability rows cannot carry NaN into P V
          #pragma unroll 1
          for (int cidx = lane; cidx < 16 * 2 * (D / 8); cidx += 32) {
            const int rr = r0 + cidx / (2 * (D / 8));
            const int rem = cidx % (2 * (D / 8));
            const int which = rem / (D / 8), d = (rem - which * (D / 8)) * 8;
            if (rr >= npos) {
              const uint32_t a = Kb + kv_at(kv_line(which, rr), d);
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
            }
          }
          patched = true;
        }
        if (patched) {
          fence_proxy_async_smem();   // these generic writes precede the slot's next TMA fill
          __syncwarp();
        }
        // S^T = K Q^T for this tile
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        const int pg0 = r0 / p.ps;
        const int lk = kv_line_in(0, r0, pg0, (lane & 7) + ((lane >> 3) & 1) * 8);
        const int lv = kv_line_in(1, r0, pg0, (lane & 7) + (lane >> 4) * 8);
#pragma unroll
        for (int s2 = 0; s2 < KS; ++s2) {
          uint32_t a[4];
          ldsm_x4(Kb + kv_at(lk, 16 * s2 + (lane >> 4) * 8), a);
          const uint4 q = qf[s2 * 32 + lane];
          mma_bf16(sc, a, q.x, q.y);
          mma_bf16(sc, a, q.z, q.w);
        }
        if (r0 + g >= npos) { sc[0] = -INFINITY; sc[1] = -INFINITY; }
        if (r0 + g + 8 >= npos) { sc[2] = -INFINITY; sc[3] = -INFINITY; }
        // online softmax per head column (heads 2t, 2t+1 on this lane)
        float pa[2], pb[2], cr[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float tm = fmaxf(sc[j], sc[j + 2]);
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
          tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
          const float mn = fmaxf(mx[j], tm);
          cr[j] = mx[j] == -INFINITY ? 0.f : __expf(mx[j] - mn);
          pa[j] = sc[j] == -INFINITY ? 0.f : __expf(sc[j] - mn);
          pb[j] = sc[j + 2] == -INFINITY ? 0.f : __expf(sc[j + 2] - mn);
          ls[j] = ls[j] * cr[j] + pa[j] + pb[j];
          mx[j] = mn;
        }
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) {
          o[mm][0] *= cr[0]; o[mm][1] *= cr[1]; o[mm][2] *= cr[0]; o[mm][3] *= cr[1];
        }
        // P^T as the B operand (positions x heads), hi and lo parts
        uint32_t xa_h, xa_l, xb_h, xb_l;
        split_bf16x2(pa[0], pa[1], xa_h, xa_l);
        split_bf16x2(pb[0], pb[1], xb_h, xb_l);
        const uint32_t b0h = movmatrix_t(xa_h), b0l = movmatrix_t(xa_l);
        const uint32_t b1h = movmatrix_t(xb_h), b1l = movmatrix_t(xb_l);
        // O^T += V^T P^T
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) {
          uint32_t a[4];
          ldsm_x4_t(Kb + kv_at(lv, 16 * mm + ((lane >> 3) & 1) * 8), a);
          mma_bf16(o[mm], a, b0h, b1h);
          mma_bf16(o[mm], a, b0l, b1l);
        }
      }
      if (last) break;
      if (!next_rec()) break;
    }
    if (!cbar_and(wok)) return false;
    trace_mark(62, l);

    // sums over the 8 lanes that share each head pair
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      ls[j] += __shfl_xor_sync(0xffffffffu, ls[j], 4);
      ls[j] += __shfl_xor_sync(0xffffffffu, ls[j], 8);
      ls[j] += __shfl_xor_sync(0xffffffffu, ls[j], 16);
    }
    // merge the 8 warps' states in one step: each warp stores (O^T fragment, max, sum) into the
    // slot it still holds (the producer refills it only after the release that follows), then
    // each thread folds the 8 states of 4 output dims of one head, in warp order
    constexpr int kStride = kMaxG * D + 2 * kMaxG;
    static_assert(kConsumerWarps * kStride * 4 <= kSlotBytes, "the warps' merge states must fit in the held slot");
    float* st = reinterpret_cast<float*>(const_cast<uint8_t*>(slot()));
    {
      float* dst = st + warp * kStride;
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) {
        // output rows of tile mm: dims 16mm + g and 16mm + g + 8 (q8_0: 16mm + 2g and 16mm + 2g + 1)
        const int d0 = Q8 ? 16 * mm + 2 * g : 16 * mm + g;
        const int d1 = Q8 ? d0 + 1 : d0 + 8;
        dst[(2 * t) * D + d0] = o[mm][0];
        dst[(2 * t + 1) * D + d0] = o[mm][1];
        dst[(2 * t) * D + d1] = o[mm][2];
        dst[(2 * t + 1) * D + d1] = o[mm][3];
      }
      if (g == 0) {
        dst[kMaxG * D + 2 * t] = mx[0];
        dst[kMaxG * D + 2 * t + 1] = mx[1];
        dst[kMaxG * D + kMaxG + 2 * t] = ls[0];
        dst[kMaxG * D + kMaxG + 2 * t + 1] = ls[1];
      }
    }
    cbar();
    {
      // a split's partial state (output, max, normaliser) for the merge; an unsplit pair's
      // state is the attention output itself, written at once (the same arithmetic as a merge
      // of one split: every output times 1 / L)
      const bool whole = item.nsplit == 1;
      uint64_t* po = whole ? p.ATT + (static_cast<size_t>(l) * p.max_batch + b) * (p.Hq * D) + static_cast<size_t>(kvh) * Gq * D
                           : p.PO + (static_cast<size_t>(l) * p.max_items + m0.idx) * (kMaxG * D);
      uint64_t* pml = p.PML + (static_cast<size_t>(l) * p.max_items + m0.idx) * (2 * kMaxG);
      #pragma unroll 1
      for (int q4 = threadIdx.x; q4 * 4 < Gq * D; q4 += kConsumerThreads) {
        const int h = (q4 * 4) / D, d = q4 * 4 - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, st[w * kStride + kMaxG * D + h]);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float mw = st[w * kStride + kMaxG * D + h];
          const float f = mw == -INFINITY ? 0.f : __expf(mw - M);
          L += f * st[w * kStride + kMaxG * D + kMaxG + h];
          const float4 ov = *reinterpret_cast<const float4*>(st + w * kStride + h * D + d);
          acc.x += f * ov.x; acc.y += f * ov.y; acc.z += f * ov.z; acc.w += f * ov.w;
        }
        if (whole) {
          const float invL = 1.f / L;
          acc.x *= invL; acc.y *= invL; acc.z *= invL; acc.w *= invL;
        }
        ll_st2(po + h * D + d, acc.x, acc.y, tg);
        ll_st2(po + h * D + d + 2, acc.z, acc.w, tg);
        if (d == 0 && !whole) ll_st2(pml + 2 * h, M, L, tg);
      }
    }
    fence_proxy_async_smem();   // the generic writes into the slot precede its next TMA fill
    trace_mark(63, l);
    return true;
  }

  // This block's share of merging the splits of every (row, KV head) pair it holds a split
  // of (pairs in one piece were written out by their item): split s of n merges outputs
  // [s*G*D/n, (s+1)*G*D/n) of the pair over all n splits, in split order, from their tagged
  // partials, and writes them as the attention output.  The block's split items go in groups
  // whose words fit the scratch, each group with one gather (one wait for the slowest split):
  // then a warp per (item, head) finds the head's max and normaliser over the splits (a lane
  // per split) and leaves each split's scale exp(m_s - M) / L, and 8 lanes per output sum the
  // splits.
  __device__ __forceinline__ bool attn_combine(int l) {
    trace_mark(66, l);
    const int Gq = p.G;
    const int GD = Gq * D;
    const int cta = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i_end = p.item_off[cta + 1];
    twait = globaltimer();
    bool ok = true;
    int it = p.item_off[cta];
    #pragma unroll 1
    for (;;) {
      // the next group: split items, gathered words [g0, g0 + 2*ns*G + ns*nsl) each, then their
      // split scales at fs (every thread walks the same items and takes the same group)
      int nk = 0, gtot = 0, ftot = 0;
      Smem::CmbItem e0{};   // the group's first item, also in registers (a group of one, the
                            // batch-1 case, needs no table and no barrier for it)
      // batches of one or two rows have at most 2 * Hkv pairs, so every block holds one item;
      // their kernels keep the one-item code alone (instruction fetch is dear at batch 1)
      constexpr int kmax = W ? kCmbItems : 1;
      #pragma unroll 1
      for (; it < i_end && nk < kmax; ++it) {
        const mk_attn_item item = p.items[it];
        const int ns = item.nsplit;
        if (ns <= 1) continue;
        const int o0 = item.split * GD / ns, nsl = (item.split + 1) * GD / ns - o0;
        const int nw = 2 * ns * Gq + ns * nsl;
        if (nk > 0 && gtot + nw + ftot + ns * Gq > kMoeScratch) break;
        Smem::CmbItem e;
        e.g0 = gtot; e.ns = ns; e.o0 = o0; e.nsl = nsl; e.fs = ftot; e.pad_ = 0;
        e.first = p.pair_first[item.b * p.Hkv + item.kvh];
        e.att = (l * p.max_batch + item.b) * (p.Hq * D) + item.kvh * GD;
        e.m = FastDiv(nsl).m;
        if (nk == 0) e0 = e;
        if (threadIdx.x == 0) S.cmb[nk] = e;
        ++nk; gtot += nw; ftot += ns * Gq;
      }
      if (nk == 0) break;
      const float* g = S.moe;
      float* fsb = S.moe + gtot;
      const FastDiv d2g(2 * Gq);
      const uint64_t* pml0 = p.PML + static_cast<size_t>(l) * p.max_items * (2 * kMaxG);
      const uint64_t* po0 = p.PO + static_cast<size_t>(l) * p.max_items * (kMaxG * D);
      const Smem::CmbItem* tab = S.cmb;
      auto word = [=](const Smem::CmbItem& e, int j) {   // gathered word j of item e
        const int nml = 2 * e.ns * Gq;
        if (j < nml) {
          const int sp = d2g.div(j);
          return pml0 + static_cast<size_t>(e.first + sp) * (2 * kMaxG) + (j - sp * 2 * Gq);
        }
        j -= nml;
        const int sp = static_cast<int>((static_cast<uint64_t>(j) * e.m) >> 32);
        return po0 + static_cast<size_t>(e.first + sp) * (kMaxG * D) + e.o0 + (j - sp * e.nsl);
      };
      if (!W || nk == 1) {
        ok = ll_gather(p, gtot, [=](int i) { return word(e0, i); }, S.moe + 0, tg) && ok;
      } else {
        cbar();   // the table
        ok = ll_gather(p, gtot, [=](int i) {
          int k = 0;
          while (k + 1 < nk && i >= tab[k + 1].g0) ++k;
          return word(tab[k], i - tab[k].g0);
        }, S.moe + 0, tg) && ok;
      }
      if (!ok) ll_timeout(p, MK_OP_ATTN, l, tg);
      if (!cbar_and(ok)) return false;
      trace_mark(64, l);
      #pragma unroll 1
      for (int x = warp; x < nk * Gq; x += kConsumerWarps) {
        const int k = x / Gq, h = x - k * Gq;
        const Smem::CmbItem e = (!W || nk == 1) ? e0 : tab[k];
        const float* ml = g + e.g0;
        float* fs = fsb + e.fs;
        float M = -INFINITY;
        #pragma unroll 1
        for (int sp = lane; sp < e.ns; sp += 32) M = fmaxf(M, ml[(sp * Gq + h) * 2]);
        M = warp_max(M);
        float L = 0.f;
        #pragma unroll 1
        for (int sp = lane; sp < e.ns; sp += 32) {
          const float m = ml[(sp * Gq + h) * 2];
          L += (m == -INFINITY ? 0.f : __expf(m - M)) * ml[(sp * Gq + h) * 2 + 1];
        }
        L = warp_sum(L);
        const float invL = 1.f / L;
        #pragma unroll 1
        for (int sp = lane; sp < e.ns; sp += 32) {
          const float m = ml[(sp * Gq + h) * 2];
          fs[sp * Gq + h] = (m == -INFINITY ? 0.f : __expf(m - M)) * invL;
        }
      }
      cbar();
      const int og = threadIdx.x >> 3, sub = threadIdx.x & 7;
      #pragma unroll 1
      for (int k = 0; k < nk; ++k) {
        const Smem::CmbItem e = (!W || nk == 1) ? e0 : tab[k];
        const float* part = g + e.g0 + 2 * e.ns * Gq;
        const float* fs = fsb + e.fs;
        uint64_t* att = p.ATT + static_cast<size_t>(e.att);
        #pragma unroll 1
        for (int base = 0; base < e.nsl; base += kConsumerThreads / 8) {   // uniform trip count: the shuffles below
          const int oi = base + og;
          float acc = 0.f;
          if (oi < e.nsl) {
            const int h = (e.o0 + oi) / D;
            #pragma unroll 1
            for (int sp = sub; sp < e.ns; sp += 8) acc += fs[sp * Gq + h] * part[sp * e.nsl + oi];
          }
          acc += __shfl_xor_sync(0xffffffffu, acc, 1);
          acc += __shfl_xor_sync(0xffffffffu, acc, 2);
          acc += __shfl_xor_sync(0xffffffffu, acc, 4);
          if (oi < e.nsl && sub == 0) ll_st(att + e.o0 + oi, acc, tg);
        }
      }
      cbar();   // the scratch and the table are reused by the next group
    }
    trace_mark(65, l);
    return true;
  }

  // ------------------------------------------------------------------ main loop
  __device__ void run() {
    for (;;) {
      bool ok = warp_wait_record(p, S, c);
      trace_chunk_seen();
      if (!cbar_and(ok)) break;   // every warp starts a tile together
      const Meta m0 = meta();
      const uint64_t t0 = tr_on(p) ? globaltimer() : 0;
      twait = 0;
      wok = true;
      switch (m0.kind) {
        case R_EMBED: ok = embed(); break;
        case R_GEMV:
        case R_GU:   // one inlined copy of the GEMV stream serves both kinds
          if constexpr (W) ok = m0.kind == R_GU && meta().n == 0;   // (only a block's empty gate/up share)
          else ok = (m0.kind == R_GU && meta().n == 0) ? true : stream_gemv(m0.kind == R_GU ? int(R_OP_GU) : int(m0.op));
          break;
        case R_ATTN: ok = attn_item(); break;
        case R_TC:
          if constexpr (W) ok = tc_gemv();
          break;
        case R_YRED:
          if constexpr (W) ok = y_reduce();
          break;
        case R_DOWN:   // the general MoE path: the widest instantiation only
          if constexpr (!kSmallMoe && !W) ok = moe_down();
          break;
        case R_ROUTE: ok = route_local(); break;
        case R_DT:   // small-batch MoE records exist only for batches of at most kSmallMaxB rows
          if constexpr (kSmallMoe) ok = moe_dt();
          break;
        case R_RED:
          if constexpr (kSmallMoe) ok = moe_reduce();
          break;
        default: break;
      }
      if (!ok) break;
      if (m0.kind != R_END) trace_event(m0.kind == R_ATTN || m0.kind == R_GU || m0.kind == R_DOWN || m0.kind == R_DT ||
                                                m0.kind == R_RED ? TR_ITEM : TR_TILE,
                                        m0, t0);
      trace_chunk_done();
      // after its last attention item the block merges its splits' partials; that needs no ring
      // slot, so the record is released first and the producer streams on meanwhile
      const bool merge = m0.kind == R_ATTN && static_cast<int>(m0.idx) == p.item_off[blockIdx.x + 1] - 1;
      if (tc_held) tc_held = false;
      else warp_release_record(S, c);
      ++c;
      if (merge && !attn_combine(m0.layer)) break;
      if (m0.kind == R_END) break;
    }
    if ((threadIdx.x & 31) == 0) atomicMin(&S.cons_count, c);
    if (threadIdx.x == 0 && tr_on(p)) {
      uint64_t* h = p.trace + static_cast<size_t>(blockIdx.x) * p.trace_cap * 4;
      h[0] = nev;
    }
  }
};

// --------------------------------------------------------------------------- the kernel
template <int TB, int D, bool Q8, bool W, bool SM>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the ring holds 128-byte-swizzled TMA tiles, whose pattern repeats every 1024 bytes
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + pad);
  const int tid = threadIdx.x;
  if (tid == 0) {
    #pragma unroll 1
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    mbar_init(&S.route_bar, 1);
    #pragma unroll 1
    for (int i = 0; i < kTcXBufs; ++i) mbar_init(&S.xbar[i], 1);
    #pragma unroll 1
    for (int i = 0; i < kTcReqs; ++i) {
      mbar_init(&S.reqbar[i], kConsumerThreads);
      mbar_init(&S.ackbar[i], 1);
    }
    mbar_init(&S.wbar, 1);
    mbar_init(&S.pbar, 1);
    S.prod_count = 0;
    S.cons_count = 0xffffffffu;
    S.ykey = -1;
    S.tag = *p.step_tag;   // a replayed launch (CUDA graph) gets a fresh tag through the step data
    if (tr_on(p)) p.trace[static_cast<size_t>(blockIdx.x) * p.trace_cap * 4 + 1] = globaltimer();
    fence_mbar_init();
  }
  if constexpr (W) {
    // wide batches: warp 0 takes all of this SM's tensor memory for the tcgen05 accumulators
    if (p.tc && (tid >> 5) == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&S.tmem_base)),
                   "r"(kTcCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
  }
  __syncthreads();
  if constexpr (W) tc_fence_after();
  {
    // every block warms a slice of the small per-layer vectors (norm gains) in L2, so that
    // their first read in a layer is an L2 hit rather than a DRAM access behind the stream
    const int n_lines = (2 * p.L + 1) * ((p.H * 2 + 127) / 128);
    #pragma unroll 1
    for (int i = blockIdx.x * kThreads + tid; i < n_lines; i += gridDim.x * kThreads) {
      const int lines_per = (p.H * 2 + 127) / 128;
      const int v = i / lines_per, ln = i - v * lines_per;
      const uint16_t* base = v == 2 * p.L ? p.final_norm : (v & 1) ? p.layers[v >> 1].ffn_norm : p.layers[v >> 1].attn_norm;
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(reinterpret_cast<const uint8_t*>(base) + ln * 128));
    }
  }
  if (tid >= kConsumerThreads) {
    // producer warpgroup: one thread streams, the rest only lend their registers
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    if (tid == kConsumerThreads) {
      Producer<Q8, W, SM> prod(p, S);
      prod.run();
    }
    if constexpr (W) {
      if (p.tc && (tid >> 5) == (kConsumerThreads >> 5) + 1) tc_issuer(p, S);   // the next warp
    }
    __syncwarp();
    asm volatile("bar.sync 12, 128;" ::: "memory");
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kLaunchRegs));
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
    {
      Consumer<TB, D, Q8, W, SM> cons(p, S);
      cons.run();
      if constexpr (W) {
        if (p.tc) cons.tc_stop();
      }
    }
    asm volatile("bar.sync %0, 128;" ::"r"(10 + (tid >> 7)) : "memory");
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLaunchRegs));
  }
  if constexpr (W) tc_fence_before();
  __syncthreads();
  if constexpr (W) {
    // every tcgen05 operation of the block has completed (each tile waits for its commits)
    if (p.tc && (tid >> 5) == 0) {
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(S.tmem_base), "r"(kTcCols) : "memory");
    }
  }
  // an aborted step may leave copies in flight: let them land before the block exits
  if (tid == 0) {
    #pragma unroll 1
    for (uint32_t c = S.cons_count; c < S.prod_count; ++c) {
      const int s = static_cast<int>(c % kSlots);
      const uint32_t ph = (c / kSlots) & 1u;
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&S.full[s], ph)) {
        if (globaltimer() - t0 > 100000000ull) break;
      }
    }
    __threadfence();
    const uint32_t old = atom_add_acq_rel(p.flags + F_FINISH, 1u);
    S.is_last = (old + 1u == gridDim.x) ? 1 : 0;
  }
  __syncthreads();
  if (S.is_last) {
    #pragma unroll 1
    for (uint32_t i = tid; i < kStepFlags; i += kThreads) p.flags[i] = 0u;
    // Greedy selection, second level: every other block has finished (their partials are
    // ordered before their arrivals on the finish counter, which this block acquired); a warp
    // per row of the batch merges the blocks' partials, read through L2.
    if (p.next_token != nullptr && !aborted(p)) {
      const int warp = tid >> 5, lane = tid & 31;
      #pragma unroll 1
      for (int b = warp; b < p.B; b += kThreads / 32) {
        Top2 t{-INFINITY, -INFINITY, 0x7fffffff};
        #pragma unroll 1
        for (int j = lane; j < static_cast<int>(gridDim.x); j += 32) {
          // (blocks with no LM-head rows -- the host's split of the vocabulary -- wrote nothing)
          const uint64_t V = static_cast<uint64_t>(p.V), N = gridDim.x;
          if (V * (j + 1) / N == V * j / N) continue;
          const float* a = p.argp + (static_cast<size_t>(j) * p.max_batch + b) * 4;
          const Top2 o{__ldcg(a), __ldcg(a + 1), __float_as_int(__ldcg(a + 2))};
          top2_merge(t, o);
        }
        top2_warp(t);
        if (lane == 0) {
          p.next_token[b] = t.i1;
          if (p.margin != nullptr) p.margin[b] = t.m1 - t.m2;
        }
      }
    }
  }
}

template <int TB, int D, bool Q8, bool W, bool SM>
cudaError_t configure_t(size_t smem) {
  return cudaFuncSetAttribute(step_kernel<TB, D, Q8, W, SM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(smem));
}

// One block per SM, all resident at once (a cooperative launch: blocks wait on one another's
// data).  Launched through cudaLaunchKernelEx so that stream capture records it in a graph.
template <int TB, int D, bool Q8, bool W, bool SM>
cudaError_t launch_t(const Params& p, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_kernel<TB, D, Q8, W, SM>, p);
}

template <int D, bool Q8>
cudaError_t configure_all(size_t smem) {
  cudaError_t e;
  if ((e = configure_t<1, D, Q8, false, true>(smem)) != cudaSuccess) return e;
  if ((e = configure_t<2, D, Q8, false, true>(smem)) != cudaSuccess) return e;
  if ((e = configure_t<1, D, Q8, false, false>(smem)) != cudaSuccess) return e;
  if ((e = configure_t<2, D, Q8, false, false>(smem)) != cudaSuccess) return e;
  if ((e = configure_t<4, D, Q8, false, false>(smem)) != cudaSuccess) return e;
  return configure_t<4, D, Q8, true, false>(smem);
}

// kind: 1 or 2 rows per register group with the small-batch MoE path; 11 or 12: the same
// without it (the general MoE path); 4: 3-4 rows; 5: the tcgen05 instantiation
template <int D, bool Q8>
cudaError_t launch_any(const Params& p, int kind, size_t smem, cudaStream_t s) {
  switch (kind) {
    case 1: return launch_t<1, D, Q8, false, true>(p, smem, s);
    case 2: return launch_t<2, D, Q8, false, true>(p, smem, s);
    case 11: return launch_t<1, D, Q8, false, false>(p, smem, s);
    case 12: return launch_t<2, D, Q8, false, false>(p, smem, s);
    case 4: return launch_t<4, D, Q8, false, false>(p, smem, s);
    default: return launch_t<4, D, Q8, true, false>(p, smem, s);
  }
}

template <int D, bool Q8>
cudaError_t occupancy_d(int* blocks, size_t smem) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, step_kernel<1, D, Q8, false, true>, kThreads, smem);
}

}  // namespace
}  // namespace mk
