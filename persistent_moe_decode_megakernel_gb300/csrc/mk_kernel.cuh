// mk_kernel.cuh -- the persistent decode-step kernel for GB300 (sm_103a).
//
// One thread block per SM stays resident for the whole step ("Inside the
// megakernel serving engine for North Mini Code", section "What is a
// Megakernel?").  Each block walks its own host-built task list; dependencies
// between tiles are counters in global memory that a finished tile increments
// (release) and a consumer spins on (acquire), bounded by a watchdog.
//
// Block layout: 8 consumer warps + 1 producer warp.  The producer streams the
// operand each tile reads from HBM -- weight rows, KV pages -- into a ring of
// shared-memory slots with 1-D bulk async copies (cp.async.bulk, completion on
// an mbarrier, L2 evict-first).  Weights never depend on activations and the
// cached KV never depends on this step, so the producer runs ahead across
// every dependency wait: while consumers wait for the previous phase, the ring
// fills with the next phase's operands.  The only producer-side wait is on
// routing, because expert weights are chosen by it.
//
// Consumers do the arithmetic on CUDA cores in fp32: GEMV rows against the
// input vector held in registers (RMSNorm fused into the load), paged GQA
// attention with an online softmax per split, SwiGLU, and the combines.
//
// Work kinds (task list entries, see mk_debug.h):
//   EMBED   residual stream <- embedding rows (a column range)
//   QKV     RMSNorm + fused QKV rows                          wait: layer input complete
//   ATTN    this block's split items of the step's plan        wait: all QKV tiles
//           last split of a (row, KV head) merges the splits -> attention output
//   OPROJ   O-proj rows + residual                             wait: all (row, KV head) pairs merged
//   ROUTER  RMSNorm + router rows; the last router tile routes: top-k, weights,
//           per-expert row lists, active-expert list -> publishes the MoE queue
//   MOE     drain the MoE queue (shared by all blocks, claimed with atomics):
//           gate/up items (expert, 16 FFN rows)  then  down items (expert, 64
//           hidden rows); the last down item of a row tile adds the k slots
//           into the residual in rank order
//   HEAD    final RMSNorm + LM-head rows
// The last block to finish resets every counter for the next step.

#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
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
// two floats -> bf16x2 (first in the low half), and the bf16x2 of what rounding left over
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 r = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// --------------------------------------------------------------------------- shared memory
enum : uint8_t { R_EMBED = 1, R_GEMV = 2, R_ATTN = 3, R_GU = 4, R_DOWN = 5, R_END = 6 };
// GEMV stream kinds beyond the task ops (MK_OP_QKV / OPROJ / ROUTER / HEAD)
enum : int { R_OP_GU = 100, R_OP_DOWN = 101 };

struct Meta {
  uint8_t kind, op, first, last;
  uint16_t layer, n;     // rows (GEMV/GU/DOWN) or pages (ATTN) in this chunk
  uint32_t row0;         // first row / FFN row / hidden row / page index of the chunk
  uint32_t idx;          // task index (GEMV/EMBED) / item index (ATTN) / active expert (GU/DOWN)
  uint32_t e;            // expert id (GU/DOWN)
  uint32_t aux;          // row tile (DOWN)
  uint32_t wait_ctr, wait_target, signal_ctr;
  uint32_t lo, hi;       // tile range
  uint32_t pad[5];
};
static_assert(sizeof(Meta) == 64, "meta size");

constexpr int kAttnScratch = 4 * kMaxG * (128 + 2);

struct __align__(128) Smem {
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
  int32_t moe_layer;                      // layer whose routing rcache holds, or -1
  int32_t ykey;                           // layer whose normalised MoE input scr.attn holds, or -1
  uint32_t prod_count, cons_count;
  int32_t flag;
  int32_t is_last;
};

// --------------------------------------------------------------------------- errors / waits
__device__ void record_error(const Params& p, int code, int op, int layer, uint32_t ctr, uint32_t observed,
                             uint32_t target, int detail, bool abort) {
  if (atomicCAS(&p.status->code, 0, code) == 0) {
    p.status->op = op;
    p.status->layer = layer;
    p.status->cta = blockIdx.x;
    p.status->counter = ctr;
    p.status->observed = observed;
    p.status->target = target;
    p.status->detail = detail;
    __threadfence();
  }
  if (abort) atomicExch(&p.ctr[C_ABORT], 1u);
}

__device__ __forceinline__ bool aborted(const Params& p) {
  return *reinterpret_cast<const volatile uint32_t*>(&p.ctr[C_ABORT]) != 0u;
}

// Spin until counter[idx] >= target (acquire).  Bounded by the watchdog; gives up
// early if another block aborted the step.
__device__ bool wait_counter(const Params& p, uint32_t idx, uint32_t target, int op, int layer) {
  const uint32_t* c = p.ctr + idx;
  uint32_t v = ld_acquire(c);
  if (v >= target) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    v = ld_acquire(c);
    if (v >= target) return true;
    if ((it & 15u) == 0u) {
      if (aborted(p)) return false;
      if (globaltimer() - t0 > p.watchdog_ns) {
        record_error(p, MK_ERR_TIMEOUT, op, layer, idx, v, target, -1, true);
        return false;
      }
    }
    if (it > 64) __nanosleep(64);
  }
}

// one warp: wait until record c has landed in its slot.  Warps consume records
// independently; false (warp-uniform) if the step was aborted meanwhile.
__device__ bool warp_wait_record(const Params& p, Smem& S, uint32_t c) {
  const int s = static_cast<int>(c % kSlots);
  const uint32_t ph = (c / kSlots) & 1u;
  bool ok = mbar_try_wait(&S.full[s], ph);
  if (!ok) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(&S.full[s], ph)) { ok = true; break; }
      if ((it & 63u) == 0u) {
        if (aborted(p)) break;
        if (globaltimer() - t0 > p.watchdog_ns) {
          if ((threadIdx.x & 31) == 0) record_error(p, MK_ERR_TIMEOUT, 0, -1, MK_NO_COUNTER, c, 0, -1, true);
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

// consumer-side dependency wait: thread 0 spins, everyone learns the outcome
__device__ bool consumer_wait(const Params& p, uint32_t idx, uint32_t target, int op, int layer) {
  bool ok = true;
  if (threadIdx.x == 0) ok = wait_counter(p, idx, target, op, layer);
  return cbar_and(ok);
}

// consumer-side signal: all consumer writes of the tile are done -> release-increment
__device__ void consumer_signal(const Params& p, uint32_t idx) {
  cbar();
  if (threadIdx.x == 0 && idx != MK_NO_COUNTER) {
    red_release_add(p.ctr + idx, 1u);
  }
}

// consumer-side arrival with "am I last" (acq_rel), broadcast to every consumer thread
__device__ bool consumer_arrive_last(const Params& p, Smem& S, uint32_t idx, uint32_t total) {
  cbar();
  if (threadIdx.x == 0) {
    const uint32_t old = atom_add_acq_rel(p.ctr + idx, 1u);
    S.flag = (old + 1u == total) ? 1 : 0;
  }
  cbar();
  const bool last = S.flag != 0;
  return last;
}

// --------------------------------------------------------------------------- producer
struct Producer {
  const Params& p;
  Smem& S;
  uint32_t c = 0;
  uint32_t pev = 0;   // producer trace events (written from the end of the block's trace area)
  uint64_t pol;
  __device__ Producer(const Params& p_, Smem& S_) : p(p_), S(S_) { pol = policy_evict_first(); }

  // wait for the slot of record c to be free; false if the step was aborted
  __device__ bool acquire() {
    const int s = static_cast<int>(c % kSlots);
    const uint32_t ph = ((c / kSlots) & 1u) ^ 1u;
    if (mbar_try_wait(&S.empty[s], ph)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(&S.empty[s], ph)) return true;
      if ((it & 63u) == 0u) {
        if (aborted(p)) return false;
        if (globaltimer() - t0 > p.watchdog_ns) {
          record_error(p, MK_ERR_TIMEOUT, 0, -1, MK_NO_COUNTER, c, 0, -1, true);
          return false;
        }
      }
    }
  }
  __device__ Meta& meta() {
    Meta& m = S.meta[c % kSlots];
    if (p.trace) {
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
    m.wait_ctr = t.wait_ctr; m.wait_target = t.wait_base + t.wait_per_b * static_cast<uint32_t>(p.B);
    m.signal_ctr = t.signal_ctr; m.lo = t.lo; m.hi = t.hi;
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
    const int rpc = gemv_rows_per_chunk(K);
    for (uint32_t r0 = t.lo; r0 < t.hi; r0 += rpc) {
      const uint32_t n = min(static_cast<uint32_t>(rpc), t.hi - r0);
      if (!acquire()) return false;
      Meta& m = meta();
      m.kind = R_GEMV; m.op = static_cast<uint8_t>(t.op); m.first = (r0 == t.lo); m.last = (r0 + n >= t.hi);
      m.layer = t.layer; m.n = static_cast<uint16_t>(n); m.row0 = r0; m.idx = ti; m.e = 0; m.aux = 0;
      m.wait_ctr = t.wait_ctr; m.wait_target = t.wait_base + t.wait_per_b * static_cast<uint32_t>(p.B);
      m.signal_ctr = t.signal_ctr; m.lo = t.lo; m.hi = t.hi;
      const uint32_t bytes = n * static_cast<uint32_t>(K) * 2u;
      mbar_arrive_expect_tx(full(), bytes);
      bulk_g2s(slot(), W + static_cast<size_t>(r0) * K, bytes, full(), pol);
      ++c;
    }
    return true;
  }

  // KV pages of this block's attention items: per page, K then V, each as D/64 boxes of
  // [page_size rows][64 dims] (128-byte swizzle).  Within a slot, K occupies the first half
  // and V the second; each holds [dim half][rows][64 dims], page i at rows i*page_size.
  __device__ bool attn_items(const mk_task& t) {
    const int cta = blockIdx.x;
    const int ppc = pages_per_chunk(p.ps, p.D);
    const int rows_cap = (kSlotBytes / 2) / (p.D * 2);
    const int halves = p.D / 64;
    const uint32_t box = static_cast<uint32_t>(p.ps) * 128u;
    for (int it = p.item_off[cta]; it < p.item_off[cta + 1]; ++it) {
      const mk_attn_item item = p.items[it];
      const int32_t* btrow = p.block_tables + static_cast<size_t>(item.b) * p.maxpg;
      for (uint32_t pg = item.page_lo; pg < item.page_hi; pg += ppc) {
        const uint32_t n = min(static_cast<uint32_t>(ppc), item.page_hi - pg);
        if (!acquire()) return false;
        Meta& m = meta();
        m.kind = R_ATTN; m.op = MK_OP_ATTN; m.first = (pg == item.page_lo); m.last = (pg + n >= item.page_hi);
        m.layer = t.layer; m.n = static_cast<uint16_t>(n); m.row0 = pg; m.idx = static_cast<uint32_t>(it);
        m.e = 0; m.aux = 0; m.wait_ctr = t.wait_ctr;
        m.wait_target = t.wait_base + t.wait_per_b * static_cast<uint32_t>(p.B);
        m.signal_ctr = t.signal_ctr; m.lo = item.page_lo; m.hi = item.page_hi;
        mbar_arrive_expect_tx(full(), 2u * halves * n * box);
        uint8_t* dst = slot();
        for (uint32_t i = 0; i < n; ++i) {
          int32_t page = btrow[pg + i];
          if (page < 0 || page >= p.P) {
            record_error(p, MK_ERR_DEVICE_BOUNDS, MK_OP_ATTN, t.layer, MK_NO_COUNTER, static_cast<uint32_t>(page), 0,
                         static_cast<int>(pg + i), false);
            page = 0;  // keep the byte count of the slot; the result is flagged invalid
          }
          const int rowk = (((t.layer * p.P + page) * 2) * p.Hkv + item.kvh) * p.ps;
          const int rowv = rowk + p.Hkv * p.ps;
          for (int h = 0; h < halves; ++h) {
            uint8_t* kd = dst + h * rows_cap * 128 + i * box;
            tma_load_2d(kd, p.kv_map, 64 * h, rowk, full(), pol);
            tma_load_2d(kd + kSlotBytes / 2, p.kv_map, 64 * h, rowv, full(), pol);
          }
        }
        ++c;
      }
    }
    return true;
  }

  __device__ bool moe_queue(const mk_task& t) {
    const int l = t.layer;
    const uint32_t base = p.cm.layer_base(l);
    const uint64_t t0 = p.trace ? globaltimer() : 0;
    if (!wait_counter(p, base + L_RREADY, 1u, MK_OP_MOE, l)) return false;
    if (p.trace && pev < static_cast<uint32_t>(p.trace_cap) / 2) {
      uint64_t* e = p.trace + (static_cast<size_t>(blockIdx.x) * p.trace_cap + p.trace_cap - 1 - pev) * 4;
      e[0] = t0;
      e[1] = globaltimer();
      e[2] = e[1];
      e[3] = static_cast<uint64_t>(MK_OP_MOE) | (static_cast<uint64_t>(l) << 8) |
             (static_cast<uint64_t>(TR_PRODUCER_ROUTE_WAIT) << 24);
      ++pev;
    }
    const uint32_t nact = static_cast<uint32_t>(__ldcg(p.NACT + l));
    const uint32_t n_gu = nact * static_cast<uint32_t>(p.n_ftiles);
    const uint32_t n_tot = n_gu + nact * static_cast<uint32_t>(p.n_rtiles);
    const LayerW& lw = p.layers[l];
    const int H = p.H, F = p.F;
    const int fpc = gemv_rows_per_chunk(H) / 2;    // gate rows (and as many up rows) per chunk
    const int rpc = gemv_rows_per_chunk(F);        // down rows per chunk
    for (;;) {
      const uint32_t q = atomicAdd(p.ctr + base + L_MOEQ, 1u);
      if (q >= n_tot) break;
      if (q < n_gu) {
        const uint32_t a = q / p.n_ftiles, ft = q % p.n_ftiles;
        const uint32_t e = static_cast<uint32_t>(__ldcg(p.ACT + static_cast<size_t>(l) * p.E + a));
        const uint32_t f0 = ft * kFTile, f1 = min(static_cast<uint32_t>(F), f0 + kFTile);
        const uint16_t* gate = lw.w_gate_up + static_cast<size_t>(e) * 2 * F * H;
        for (uint32_t f = f0; f < f1; f += fpc) {
          const uint32_t n = min(static_cast<uint32_t>(fpc), f1 - f);
          if (!acquire()) return false;
          Meta& m = meta();
          m.kind = R_GU; m.op = MK_OP_MOE; m.first = (f == f0); m.last = (f + n >= f1);
          m.layer = static_cast<uint16_t>(l); m.n = static_cast<uint16_t>(n); m.row0 = f; m.idx = a; m.e = e;
          m.aux = ft; m.wait_ctr = MK_NO_COUNTER; m.wait_target = 0; m.signal_ctr = MK_NO_COUNTER;
          m.lo = f0; m.hi = f1;
          const uint32_t bytes = n * static_cast<uint32_t>(H) * 2u;
          mbar_arrive_expect_tx(full(), 2u * bytes);
          bulk_g2s(slot(), gate + static_cast<size_t>(f) * H, bytes, full(), pol);
          bulk_g2s(slot() + bytes, gate + static_cast<size_t>(F + f) * H, bytes, full(), pol);
          ++c;
        }
      } else {
        const uint32_t qq = q - n_gu;
        const uint32_t a = qq / p.n_rtiles, rt = qq % p.n_rtiles;
        const uint32_t e = static_cast<uint32_t>(__ldcg(p.ACT + static_cast<size_t>(l) * p.E + a));
        const uint32_t r0 = rt * kRTile, r1 = min(static_cast<uint32_t>(H), r0 + kRTile);
        const uint16_t* down = lw.w_down + static_cast<size_t>(e) * H * F;
        for (uint32_t r = r0; r < r1; r += rpc) {
          const uint32_t n = min(static_cast<uint32_t>(rpc), r1 - r);
          if (!acquire()) return false;
          Meta& m = meta();
          m.kind = R_DOWN; m.op = MK_OP_MOE; m.first = (r == r0); m.last = (r + n >= r1);
          m.layer = static_cast<uint16_t>(l); m.n = static_cast<uint16_t>(n); m.row0 = r; m.idx = a; m.e = e;
          m.aux = rt; m.wait_ctr = MK_NO_COUNTER; m.wait_target = 0; m.signal_ctr = MK_NO_COUNTER;
          m.lo = r0; m.hi = r1;
          const uint32_t bytes = n * static_cast<uint32_t>(F) * 2u;
          mbar_arrive_expect_tx(full(), bytes);
          bulk_g2s(slot(), down + static_cast<size_t>(r) * F, bytes, full(), pol);
          ++c;
        }
      }
    }
    return true;
  }

  __device__ void run() {
    const int cta = blockIdx.x;
    for (int ti = p.task_off[cta]; ti < p.task_off[cta + 1]; ++ti) {
      const mk_task t = p.tasks[ti];
      bool ok = true;
      switch (t.op) {
        case MK_OP_EMBED: ok = emit_control(R_EMBED, t, static_cast<uint32_t>(ti)); break;
        case MK_OP_QKV:
        case MK_OP_OPROJ:
        case MK_OP_ROUTER:
        case MK_OP_HEAD: ok = gemv_tile(t, static_cast<uint32_t>(ti)); break;
        case MK_OP_ATTN: ok = attn_items(t); break;
        case MK_OP_MOE: ok = moe_queue(t); break;
        case MK_OP_END: ok = emit_control(R_END, t, static_cast<uint32_t>(ti)); break;
        default: break;
      }
      if (!ok) break;
    }
    S.prod_count = c;
    if (p.trace) p.trace[static_cast<size_t>(blockIdx.x) * p.trace_cap * 4 + 2] = pev;
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

// Sums of squares of residual-stream vector `xidx`, row b, as published per
// tile by its producers: issue every load at once (slots <= 256), then reduce in
// fixed order so every warp gets the same value.
__device__ __forceinline__ void ss_issue(const Params& p, int xidx, int b, float (&v)[8]) {
  const float* ss = p.SS + static_cast<size_t>(xidx) * p.n_ss_slots * p.max_batch + b;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = lane + 32 * k;
    v[k] = i < p.n_ss_slots ? __ldcg(ss + static_cast<size_t>(i) * p.max_batch) : 0.f;
  }
}
__device__ __forceinline__ float ss_rstd(const Params& p, const float (&v)[8]) {
  float t = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) t += v[k];
  t = warp_sum(t);
  return 1.0f / sqrtf(t / static_cast<float>(p.H) + p.eps);
}

// Load this warp's segment of nt input vectors into registers.  src[tb] points
// at vector tb (fp32); with g non-null each vector is RMS-normalised with rstd[tb]
// and the bf16 gain g.  Vectors tb >= nt (or with src null) read as zero.
template <int TB>
__device__ __forceinline__ void load_y(const Seg<TB>& sg, const float* const (&src)[TB], const float (&rstd)[TB],
                                       const uint16_t* g, int nt, float (&y)[8 / TB][8][TB]) {
#pragma unroll
  for (int j = 0; j < Seg<TB>::kUnits; ++j) {
    const int e = sg.unit(j);
    float gv[8];
    if (g != nullptr && e >= 0) {
      unpack8(__ldg(reinterpret_cast<const uint4*>(g + e)), gv);
    }
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (e >= 0 && tb < nt && src[tb] != nullptr) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(src[tb] + e));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(src[tb] + e + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        if (g != nullptr) {
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] = (v[q] * rstd[tb]) * gv[q];
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) y[j][q][tb] = v[q];
    }
  }
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

// per-row-of-the-batch sums of one value per thread (thread's row tb, or tb < 0
// for none) over all consumer threads, in fixed order -> out[0..nt)
template <int TB>
__device__ void block_token_sums(Smem& S, int my_tb, float v, int nt, float* out, size_t out_stride) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) {
    const float w = warp_sum(my_tb == tb ? v : 0.f);
    if (lane == 0) S.ssred[warp][tb] = w;
  }
  cbar();
  if (threadIdx.x < nt) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += S.ssred[w][threadIdx.x];
    out[threadIdx.x * out_stride] = tot;
  }
  cbar();
}

// --------------------------------------------------------------------------- consumer
// Warps consume ring records independently (each waits for and releases every
// record of a tile); block-wide barriers are taken only at tile boundaries --
// the dependency wait at a tile's start and the signal at its end -- and, where
// S warps split a row, over those S warps only.
template <int TB, int D>
struct Consumer {
  const Params& p;
  Smem& S;
  uint32_t c = 0;       // this warp's current record
  bool wok = true;      // this warp has not seen the step abort
  uint32_t nev = 1;     // trace events written (event 0 is the header)
  uint64_t twait = 0;   // when the current tile's dependency was met

  __device__ Consumer(const Params& p_, Smem& S_) : p(p_), S(S_) {}

  __device__ void trace_event(uint32_t kind, const Meta& m, uint64_t t0) {
    if (p.trace == nullptr || threadIdx.x != 0) return;
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
  __device__ void trace_mark(uint32_t id, int layer) {
    if (p.trace == nullptr || threadIdx.x != 0) return;
    if (nev < static_cast<uint32_t>(p.trace_cap) / 2) {
      const uint64_t t = globaltimer();
      uint64_t* ev = p.trace + (static_cast<size_t>(blockIdx.x) * p.trace_cap + nev) * 4;
      ev[0] = t; ev[1] = t; ev[2] = t;
      ev[3] = static_cast<uint64_t>(id) | (static_cast<uint64_t>(layer) << 8) | (static_cast<uint64_t>(TR_MARK) << 24);
      ++nev;
    }
  }

  __device__ const Meta& meta() const { return S.meta[c % kSlots]; }
  __device__ const uint8_t* slot() const { return S.ring[c % kSlots]; }

  // chunk timeline (tracing only): issue time, when warp 0 saw the data, when it released the slot
  uint64_t tchunk = 0;
  __device__ void trace_chunk_seen() {
    if (p.trace && threadIdx.x == 0) tchunk = globaltimer();
  }
  __device__ void trace_chunk_done() {
    if (p.trace == nullptr || threadIdx.x != 0) return;
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
  __device__ __forceinline__ const float* xrow(int xidx, int b) const {
    return p.X + (static_cast<size_t>(xidx) * p.max_batch + b) * p.H;
  }

  // Load the GEMV input of `kind` for rows rb[0..nt) into y (this warp's segment).
  // kinds: 0 attention input (x_in, attn_norm), 1 O-proj input (attention output),
  //        2 MoE input (x_mid, ffn_norm), 3 head input (x_final, final_norm)
  __device__ __forceinline__ void load_input(const Seg<TB>& sg, int kind, int l, const int (&rb)[TB], int nt,
                                             float (&y)[8 / TB][8][TB]) {
    const float* src[TB];
    const uint16_t* g = nullptr;
    int xidx = 0;
    if (kind == 0) { g = p.layers[l].attn_norm; xidx = 2 * l; }
    else if (kind == 2) { g = p.layers[l].ffn_norm; xidx = 2 * l + 1; }
    else if (kind == 3) { g = p.final_norm; xidx = 2 * p.L; }
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      const int b = tb < nt ? rb[tb] : rb[0];
      src[tb] = kind == 1 ? p.ATT + (static_cast<size_t>(l) * p.max_batch + b) * (p.Hq * p.D) : xrow(xidx, b);
    }
    float one[TB];
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) one[tb] = 1.f;
    load_y<TB>(sg, src, one, nullptr, nt, y);   // raw values; the loads below overlap with these
    if (g == nullptr) return;
    uint4 gw[Seg<TB>::kUnits];
#pragma unroll
    for (int j = 0; j < Seg<TB>::kUnits; ++j) {
      const int e = sg.unit(j);
      gw[j] = e >= 0 ? __ldg(reinterpret_cast<const uint4*>(g + e)) : make_uint4(0, 0, 0, 0);
    }
    float ssv[TB][8];
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) ss_issue(p, xidx, tb < nt ? rb[tb] : rb[0], ssv[tb]);
    float rs[TB];
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) rs[tb] = ss_rstd(p, ssv[tb]);
#pragma unroll
    for (int j = 0; j < Seg<TB>::kUnits; ++j) {
      float gv[8];
      unpack8(gw[j], gv);
#pragma unroll
      for (int tb = 0; tb < TB; ++tb)
#pragma unroll
        for (int q = 0; q < 8; ++q) y[j][q][tb] = (y[j][q][tb] * rs[tb]) * gv[q];
    }
  }

  // ------------------------------------------------------------------ EMBED
  __device__ bool embed() {
    const Meta m = meta();
    const int H = p.H;
    float* ssout = p.SS + static_cast<size_t>(blockIdx.x) * p.max_batch;   // vector 0, slot = this block
    for (int b = 0; b < p.B; ++b) {
      int tok = __ldg(p.tokens + b);
      if (tok < 0 || tok >= p.V) {
        if (threadIdx.x == 0)
          record_error(p, MK_ERR_DEVICE_BOUNDS, MK_OP_EMBED, -1, MK_NO_COUNTER, static_cast<uint32_t>(tok), 0, b,
                       false);
        tok = 0;
      }
      const uint16_t* row = p.embed + static_cast<size_t>(tok) * H;
      float* x = p.X + static_cast<size_t>(b) * H;
      float ss = 0.f;
      for (uint32_t col = m.lo + threadIdx.x; col < m.hi; col += kConsumerThreads) {
        const float v = bf1(row[col]);
        x[col] = v;
        ss += v * v;
      }
      ss = warp_sum(ss);
      if ((threadIdx.x & 31) == 0) S.ssred[threadIdx.x >> 5][0] = ss;
      cbar();
      if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) tot += S.ssred[w][0];
        ssout[b] = tot;
      }
      cbar();
    }
    consumer_signal(p, m.signal_ctr);
    return true;
  }

  // ------------------------------------------------------------------ GEMV streams
  // One loop serves every weight-streaming record: QKV / O-proj / router / head
  // tiles and the expert gate/up and down items.  Only the input, the
  // dependency and where the results go differ.  Gate/up chunks hold nf gate
  // rows then the nf matching up rows; the row groups are sized so that gate
  // row f and up row f land in the same group (one SwiGLU per pair).
  struct OutMap {
    float* base;          // output of (row 0 of the batch, slot 0, matrix row 0)
    size_t sb, sj;        // strides per batch row and per routing slot
    const float* resid;   // O-proj: residual input (same layout as base), else null
    const float* bias;    // router bias by matrix row, or null
  };

  __device__ __forceinline__ OutMap out_map(int op, int l) const {
    const size_t MB = p.max_batch, xs = MB * p.H;
    OutMap o{nullptr, 0, 0, nullptr, nullptr};
    switch (op) {
      case MK_OP_QKV: o.base = p.QKV + l * MB * p.nqkv; o.sb = p.nqkv; break;
      case MK_OP_OPROJ: o.base = p.X + (2 * l + 1) * xs; o.sb = p.H; o.resid = p.X + 2 * l * xs; break;
      case MK_OP_ROUTER: o.base = p.RLOG + l * MB * p.E; o.sb = p.E; o.bias = p.layers[l].router_bias; break;
      case MK_OP_HEAD: o.base = p.logits; o.sb = p.V; break;
      case R_OP_GU: o.base = p.HB + l * MB * p.K * p.F; o.sb = static_cast<size_t>(p.K) * p.F; o.sj = p.F; break;
      default: o.base = p.PART + l * MB * p.K * p.H; o.sb = static_cast<size_t>(p.K) * p.H; o.sj = p.H; break;
    }
    return o;
  }

  // result v (v2: the matching up row for gate/up) of matrix row `row` for batch row b, slot j;
  // rv: the residual input of that element when the caller already loaded it (O-proj), else NAN
  __device__ __forceinline__ void put(const OutMap& o, bool gu, uint32_t row, int b, int j, float v, float v2,
                                      float& my_ss, float rv = NAN) {
    if (j < 0) return;
    const size_t off = static_cast<size_t>(b) * o.sb + static_cast<size_t>(j) * o.sj + row;
    if (gu) v = (v / (1.0f + expf(-v))) * v2;
    if (o.resid != nullptr) {
      v += isnan(rv) ? __ldcg(o.resid + off) : rv;
      my_ss += v * v;
    }
    if (o.bias != nullptr) v += __ldg(o.bias + row);
    o.base[off] = v;
  }

  __device__ __forceinline__ void stream_load(const Seg<TB>& sg, bool moe, int kind, int l, int e, int b0, int nt,
                                              int (&rb)[TB], int (&rj)[TB], float (&y)[8 / TB][8][TB]) {
    if (moe) {
      expert_rows(l, e, b0, nt, rb, rj);
    } else {
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) { rb[tb] = b0 + tb; rj[tb] = 0; }
    }
    if (kind == 4) load_h(sg, l, rb, rj, nt, y);
    else load_input(sg, kind, l, rb, nt, y);
  }

  __device__ bool stream_gemv(int op) {
    constexpr bool kGroups = TB == 4;   // only the widest instantiation sees batches wider than its registers
    const int l = meta().layer;
    const uint32_t sig = meta().signal_ctr, lo = meta().lo, hi = meta().hi;
    const int e = static_cast<int>(meta().e), a = static_cast<int>(meta().idx);
    const uint32_t rt = meta().aux;
    const int nf0 = meta().n;
    const uint32_t base = p.cm.layer_base(l < p.L ? l : 0);
    const bool moe = op == R_OP_GU || op == R_OP_DOWN;
    const bool gu = op == R_OP_GU;
    bool ok;
    if (gu) ok = consumer_wait(p, base + L_RREADY, 1u, MK_OP_MOE, l);
    else if (op == R_OP_DOWN) ok = consumer_wait(p, base + p.cm.gu_off + a, static_cast<uint32_t>(p.n_ftiles), MK_OP_MOE, l);
    else ok = meta().wait_ctr == MK_NO_COUNTER || consumer_wait(p, meta().wait_ctr, meta().wait_target, op, l);
    if (!ok) return false;
    twait = globaltimer();
    const int B = p.B;
    const int lane = threadIdx.x & 31;
    const int K = op == MK_OP_OPROJ ? p.Hq * p.D : op == R_OP_DOWN ? p.F : p.H;
    const Seg<TB> sg(K, gu ? (nf0 >= kConsumerWarps ? 1 : kConsumerWarps / nf0) : 1);
    // GEMV input: 0 x_in/attn_norm, 1 attention output, 2 x_mid/ffn_norm, 3 x_final/final_norm, 4 SwiGLU h
    const int kind = op == MK_OP_QKV ? 0 : op == MK_OP_OPROJ ? 1 : (op == MK_OP_ROUTER || gu) ? 2
                   : op == MK_OP_HEAD ? 3 : 4;
    trace_mark(10 + (op == MK_OP_ROUTER ? 0 : moe ? 20 : 40), l);
    if (moe) slots_for_expert(l, e);
    const int cnt = (!moe || B <= TB) ? B : __ldcg(p.CNT + static_cast<size_t>(l) * p.E + e);
    const int ngroups = kGroups ? (cnt + TB - 1) / TB : 1;
    const OutMap om = out_map(op, l);
    float my_ss = 0.f;    // O-proj: sum of squares of the residual values this lane wrote
    int rb[TB], rj[TB];
    float y[8 / TB][8][TB];
    const bool cached = gu && B <= TB && B * p.H <= kAttnScratch;
    if (cached) {
      ensure_ffn_input(l);
      expert_rows(l, e, 0, B, rb, rj);
      load_y_smem(sg, B, y);
    } else {
      stream_load(sg, moe, kind, l, e, 0, min(cnt, TB), rb, rj, y);
    }
    trace_mark(11 + (op == MK_OP_ROUTER ? 0 : moe ? 20 : 40), l);
    for (;;) {
      const int n = meta().n;
      const uint32_t row0 = meta().row0;
      const bool last = meta().last;
      const uint8_t* wsm = slot();
      const int par = c & 1;
      ok = true;
      for (int g = 0; g < ngroups && ok; ++g) {
        const int b0 = g * TB;
        const int nt = min(TB, cnt - b0);
        if (kGroups && ngroups > 1) stream_load(sg, moe, kind, l, e, b0, nt, rb, rj, y);
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
                  pick<TB>(acc2, lane), my_ss);
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
              if (r < n) rv[i] = __ldcg(om.resid + static_cast<size_t>(pick_i<TB>(rb, lane)) * om.sb + row0 + r);
            }
          }
          ok = group_bar_and(true, sg.S);
          if (ok && sg.s == 0 && lane < nt) {
            int i = 0;
            for (int r = sg.rg; r < n; r += sg.RPG, ++i) {
              float v = 0.f, v2 = 0.f;
              for (int q = 0; q < sg.S; ++q) {
                v += S.scr.seg[par][r][q][lane];
                if (gu) v2 += S.scr.seg[par][kMaxRowsPerChunk / 2 + r][q][lane];
              }
              put(om, gu, row0 + r, pick_i<TB>(rb, lane), pick_i<TB>(rj, lane), v, v2, my_ss,
                  i == 0 ? rv[0] : i == 1 ? rv[1] : i == 2 ? rv[2] : i == 3 ? rv[3] : NAN);
            }
          }
          if (kGroups && ngroups > 1) ok = group_bar_and(ok, sg.S);   // seg is reused by the next group
        }
      }
      if (!ok) { wok = false; break; }
      if (last) break;
      if (!next_rec()) break;
    }
    if (!cbar_and(wok)) return false;
    switch (op) {
      case MK_OP_OPROJ: {
        // publish this tile's share of sum(x_mid^2) for the RMSNorm of the MoE input
        float* out = p.SS + (static_cast<size_t>(2 * l + 1) * p.n_ss_slots + blockIdx.x) * p.max_batch;
        if (B <= TB) block_token_sums<TB>(S, lane < B ? lane : -1, my_ss, B, out, 1);
        else oproj_ss_wide(l, lo, hi, out);
        consumer_signal(p, sig);
        break;
      }
      case MK_OP_ROUTER:
        trace_mark(12, l);
        if (consumer_arrive_last(p, S, base + L_RARR, static_cast<uint32_t>(p.n_router_tiles))) {
          trace_mark(13, l);
          route(l);
          trace_mark(14, l);
        }
        break;
      case R_OP_GU: consumer_signal(p, base + p.cm.gu_off + a); break;
      case R_OP_DOWN: {
        // the last item of this row tile adds every slot into the residual, in rank order
        const uint32_t nact = static_cast<uint32_t>(__ldcg(p.NACT + l));
        if (consumer_arrive_last(p, S, base + p.cm.down_off + rt, nact)) down_combine(l, rt);
        break;
      }
      default: consumer_signal(p, sig); break;
    }
    return true;
  }

  // x_out = x_mid + sum_j w_j * down_j over rows of row tile rt, rank order; publishes sum(x_out^2)
  __device__ void down_combine(int l, uint32_t rt) {
    const int B = p.B, H = p.H, K = p.K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t xs = static_cast<size_t>(p.max_batch) * H;
    const int r0 = static_cast<int>(rt) * kRTile, r1 = min(H, r0 + kRTile);
    float* ssout = p.SS + (static_cast<size_t>(2 * l + 2) * p.n_ss_slots + rt) * p.max_batch;
    for (int b = warp; b < B; b += kConsumerWarps) {
      const size_t lb = static_cast<size_t>(l) * p.max_batch + b;
      float ss = 0.f;
      for (int r = r0 + lane; r < r1; r += 32) {
        float acc = 0.f;
        for (int j = 0; j < K; ++j) acc += __ldcg(p.RW + lb * K + j) * __ldcg(p.PART + (lb * K + j) * H + r);
        const size_t off = static_cast<size_t>(b) * H + r;
        const float xv = __ldcg(p.X + (2 * static_cast<size_t>(l) + 1) * xs + off) + acc;
        p.X[(2 * static_cast<size_t>(l) + 2) * xs + off] = xv;
        ss += xv * xv;
      }
      ss = warp_sum(ss);
      if (lane == 0) ssout[b] = ss;
    }
    consumer_signal(p, p.cm.layer_base(l) + L_MOE);
  }

  // sums of squares of this O-proj tile's rows for every batch row (batches wider than TB)
  __device__ void oproj_ss_wide(int l, uint32_t lo, uint32_t hi, float* out) {
    const size_t xs = static_cast<size_t>(p.max_batch) * p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int b = warp; b < p.B; b += kConsumerWarps) {
      float ss = 0.f;
      for (uint32_t r = lo + lane; r < hi; r += 32) {
        const float v = __ldcg(p.X + (2 * static_cast<size_t>(l) + 1) * xs + static_cast<size_t>(b) * p.H + r);
        ss += v * v;
      }
      ss = warp_sum(ss);
      if (lane == 0) out[b] = ss;
    }
    cbar();
  }

  // SwiGLU activations of (row, slot) pairs as the down projection's input
  __device__ __forceinline__ void load_h(const Seg<TB>& sg, int l, const int (&rb)[TB], const int (&rj)[TB], int nt,
                                         float (&y)[8 / TB][8][TB]) {
    const float* src[TB];
    float one[TB];
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      one[tb] = 1.f;
      src[tb] = (tb < nt && rj[tb] >= 0) ? p.HB + ((static_cast<size_t>(l) * p.max_batch + rb[tb]) * p.K + rj[tb]) * p.F
                                         : nullptr;
    }
    load_y<TB>(sg, src, one, nullptr, nt, y);
  }

  // ------------------------------------------------------------------ routing (last router tile)
  // Top-k by logit, ties to the lower expert index: an expert's rank is the number
  // of experts with a larger logit plus those with an equal logit and a lower
  // index; every (row, expert) pair counts its own rank against the row's logits
  // staged in shared memory, so no serial selection rounds are needed.  Weights:
  // exp(r - max) over the chosen experts, renormalised over them (or over all
  // experts when norm_topk == 0).  Then the per-expert row lists and the list of
  // active experts, and the MoE queue is published.
  __device__ void route(int l) {
    const int B = p.B, E = p.E, K = p.K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t lb = static_cast<size_t>(l) * p.max_batch;
    float* lg = S.scr.attn;
    if (threadIdx.x == 0) S.ykey = -1;
    const int rpp = kAttnScratch / E;   // rows of logits staged per pass
    for (int b0 = 0; b0 < B; b0 += rpp) {
      const int nb = min(rpp, B - b0);
      for (int i = threadIdx.x; i < nb * E; i += kConsumerThreads) lg[i] = __ldcg(p.RLOG + (lb + b0) * E + i);
      cbar();
      trace_mark(15, l);
      for (int b = warp; b < nb; b += kConsumerWarps) {
        float mx = -INFINITY;
        for (int e = lane; e < E; e += 32) mx = fmaxf(mx, lg[b * E + e]);
        mx = warp_max(mx);
        float z = 0.f;
        for (int e = lane; e < E; e += 32) z += expf(lg[b * E + e] - mx);
        z = warp_sum(z);
        if (lane == 0) { S.rmax[b0 + b] = mx; S.rz[b0 + b] = z; }
      }
      for (int i = threadIdx.x; i < nb * E; i += kConsumerThreads) {
        const int b = i / E, e = i - b * E;
        const float* row = lg + b * E;
        const float v = row[e];
        int rank = 0;
        int e2 = 0;
        if ((E & 3) == 0) {
#pragma unroll 4
          for (; e2 < E; e2 += 4) {
            const float4 w = *reinterpret_cast<const float4*>(row + e2);
            rank += (w.x > v) || (w.x == v && e2 < e);
            rank += (w.y > v) || (w.y == v && e2 + 1 < e);
            rank += (w.z > v) || (w.z == v && e2 + 2 < e);
            rank += (w.w > v) || (w.w == v && e2 + 3 < e);
          }
        }
        for (; e2 < E; ++e2) {
          const float v2 = row[e2];
          rank += (v2 > v) || (v2 == v && e2 < e);
        }
        if (rank < K) {
          S.rids[(b0 + b) * K + rank] = e;
          S.rval[(b0 + b) * K + rank] = v;
        }
      }
      cbar();
      trace_mark(16, l);
    }
    for (int b = threadIdx.x; b < B; b += kConsumerThreads) {
      float sum = 0.f;
      for (int j = 0; j < K; ++j) sum += expf(S.rval[b * K + j] - S.rmax[b]);
      S.rsum[b] = sum;
    }
    cbar();
    for (int i = threadIdx.x; i < B * K; i += kConsumerThreads) {
      const int b = i / K;
      const float ex = expf(S.rval[i] - S.rmax[b]);
      p.RIDS[lb * K + i] = S.rids[i];
      p.RW[lb * K + i] = p.norm_topk ? ex / S.rsum[b] : ex / S.rz[b];
    }
    trace_mark(17, l);
    // rows routed to each expert, ascending row
    const size_t le = static_cast<size_t>(l) * E;
    for (int e = threadIdx.x; e < E; e += kConsumerThreads) {
      int cnt = 0;
      for (int b = 0; b < B; ++b)
        for (int j = 0; j < K; ++j)
          if (S.rids[b * K + j] == e) p.TOK[(le + e) * p.max_batch + cnt++] = (b << 8) | j;
      p.CNT[le + e] = cnt;
      S.ecnt[e] = cnt;
    }
    cbar();
    if (warp == 0) {
      int nact = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool on = e < E && S.ecnt[e] > 0;
        const uint32_t ball = __ballot_sync(0xffffffffu, on);
        if (on) p.ACT[le + nact + __popc(ball & ((1u << lane) - 1u))] = e;
        nact += __popc(ball);
      }
      if (lane == 0) p.NACT[l] = nact;
    }
    trace_mark(18, l);
    consumer_signal(p, p.cm.layer_base(l) + L_RREADY);
  }

  // which slot (rank) expert e has in row b's choice, or -1
  __device__ void slots_for_expert(int l, int e) {
    const int K = p.K;
    if (S.moe_layer != l) {   // first MoE item of this layer in this block: cache the routing
      for (int i = threadIdx.x; i < p.B * K; i += kConsumerThreads)
        S.rcache[i] = __ldcg(p.RIDS + static_cast<size_t>(l) * p.max_batch * K + i);
      cbar();
      if (threadIdx.x == 0) S.moe_layer = l;
    }
    if (threadIdx.x < p.B) {
      int s = -1;
      for (int j = 0; j < K; ++j)
        if (S.rcache[threadIdx.x * K + j] == e) s = j;
      S.slot_of[threadIdx.x] = s;
    }
    cbar();
  }

  // the normalised MoE input of every row (B <= TB), staged once per layer in shared memory
  __device__ void ensure_ffn_input(int l) {
    if (S.ykey == l) return;
    const int B = p.B, H = p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int xidx = 2 * l + 1;
    if (warp < B) {
      float v[8];
      ss_issue(p, xidx, warp, v);
      const float r = ss_rstd(p, v);
      if (lane == 0) S.rstd[warp] = r;
    }
    cbar();
    const uint16_t* g = p.layers[l].ffn_norm;
    float* yc = S.scr.attn;
    for (int i = threadIdx.x * 4; i < B * H; i += kConsumerThreads * 4) {
      const int b = i / H, k = i - b * H;
      const float4 x = __ldcg(reinterpret_cast<const float4*>(xrow(xidx, b) + k));
      const uint2 gw = __ldg(reinterpret_cast<const uint2*>(g + k));
      const float r = S.rstd[b];
      yc[i] = (x.x * r) * bf_lo(gw.x);
      yc[i + 1] = (x.y * r) * bf_hi(gw.x);
      yc[i + 2] = (x.z * r) * bf_lo(gw.y);
      yc[i + 3] = (x.w * r) * bf_hi(gw.y);
    }
    cbar();
    if (threadIdx.x == 0) S.ykey = l;
  }

  __device__ __forceinline__ void load_y_smem(const Seg<TB>& sg, int nt, float (&y)[8 / TB][8][TB]) {
    const float* yc = S.scr.attn;
#pragma unroll
    for (int j = 0; j < Seg<TB>::kUnits; ++j) {
      const int e = sg.unit(j);
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (e >= 0 && tb < nt) {
          a = *reinterpret_cast<const float4*>(yc + tb * p.H + e);
          b = *reinterpret_cast<const float4*>(yc + tb * p.H + e + 4);
        }
        y[j][0][tb] = a.x; y[j][1][tb] = a.y; y[j][2][tb] = a.z; y[j][3][tb] = a.w;
        y[j][4][tb] = b.x; y[j][5][tb] = b.y; y[j][6][tb] = b.z; y[j][7][tb] = b.w;
      }
    }
  }

  // rows of the batch routed to expert e, in groups of TB: (row, slot); slot -1 = not routed
  __device__ __forceinline__ void expert_rows(int l, int e, int b0, int nt, int (&rb)[TB], int (&rj)[TB]) {
    const int32_t* tok = p.TOK + (static_cast<size_t>(l) * p.E + e) * p.max_batch;
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      if (p.B <= TB) {
        rb[tb] = tb;
        rj[tb] = tb < nt ? S.slot_of[tb] : -1;
      } else {
        const int ent = tb < nt ? __ldcg(tok + b0 + tb) : 0;
        rb[tb] = ent >> 8;
        rj[tb] = tb < nt ? (ent & 0xff) : -1;
      }
    }
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
  __device__ __forceinline__ uint32_t swz(int r, int d, int rows_cap) const {
    return static_cast<uint32_t>((d >> 6) * rows_cap * 128 + r * 128 + ((((d & 63) >> 3) ^ (r & 7)) << 4) + (d & 7) * 2);
  }

  __device__ __noinline__ bool attn_item() {
    constexpr int KS = D / 16;                              // k-steps over head dims (Q K^T)
    constexpr int MT = D / 16;                              // 16-dim tiles of the output (P V)
    constexpr int ROWS = (kSlotBytes / 2) / (D * 2);        // positions a chunk's K (or V) region holds
    const Meta m0 = meta();
    const int l = m0.layer;
    if (!consumer_wait(p, m0.wait_ctr, m0.wait_target, MK_OP_ATTN, l)) return false;
    twait = globaltimer();
    const mk_attn_item item = p.items[m0.idx];
    const int b = item.b, kvh = item.kvh, Gq = p.G;
    const int Lc = p.seq_lens[b];
    const int pos = Lc - 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    // Q^T as the B operand of S^T = K Q^T, one 16-byte fragment per (k-step, lane):
    // lane (g, t) holds head g at dims 16s + 2t (+1) and 16s + 2t + 8 (+1), hi then lo parts
    // of the rotated, scaled q (zero for heads at or above G); then this token's bf16 k and v
    uint4* qf = reinterpret_cast<uint4*>(S.scr.attn);                     // [KS][32]
    uint16_t* kvcur = reinterpret_cast<uint16_t*>(S.scr.attn + KS * 32 * 4);  // [2][D]
    if (threadIdx.x == 0) S.ykey = -1;                                // the MoE input cache shares this storage
    const float* qkv = p.QKV + (static_cast<size_t>(l) * p.max_batch + b) * p.nqkv;
    const float* cs = p.rope_cos + static_cast<size_t>(b) * (D / 2);
    const float* sn = p.rope_sin + static_cast<size_t>(b) * (D / 2);
    for (int i = threadIdx.x; i < KS * 32; i += kConsumerThreads) {
      const int s2 = i >> 5, gg = (i >> 2) & 7, tt = i & 3;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (gg < Gq) {
        const float* qh = qkv + (kvh * Gq + gg) * D;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int d = 16 * s2 + 2 * tt + 8 * (j >> 1) + (j & 1);
          const int dh = d % (D / 2);
          const float raw = __ldcg(qh + d), other = __ldcg(qh + (d < D / 2 ? d + D / 2 : d - D / 2));
          const float c = __ldg(cs + dh), sv = __ldg(sn + dh);
          v[j] = (d < D / 2 ? raw * c - other * sv : raw * c + other * sv) * p.scale;
        }
      }
      uint4 f;
      split_bf16x2(v[0], v[1], f.x, f.z);
      split_bf16x2(v[2], v[3], f.y, f.w);
      qf[i] = f;
    }
    for (int d = threadIdx.x; d < D; d += kConsumerThreads) {
      const float* kh = qkv + (p.Hq + kvh) * D;
      const float raw = __ldcg(kh + d), other = __ldcg(kh + (d < D / 2 ? d + D / 2 : d - D / 2));
      const float c = __ldg(cs + (d % (D / 2))), sv = __ldg(sn + (d % (D / 2)));
      kvcur[d] = to_bf16_bits(d < D / 2 ? raw * c - other * sv : raw * c + other * sv);
      kvcur[D + d] = to_bf16_bits(__ldcg(qkv + (p.Hq + p.Hkv + kvh) * D + d));
    }
    cbar();
    if (item.split == 0) {
      // append this token's k and v to the cache
      const int pg = pos / p.ps, sl = pos % p.ps;
      const int32_t page = __ldg(p.block_tables + static_cast<size_t>(b) * p.maxpg + pg);
      if (page >= 0 && page < p.P) {
        const size_t kb = (((static_cast<size_t>(l) * p.P + page) * 2 * p.Hkv + kvh) * p.ps + sl) * D;
        const size_t vb = kb + static_cast<size_t>(p.Hkv) * p.ps * D;
        for (int d = threadIdx.x; d < D; d += kConsumerThreads) {
          p.kv[kb + d] = kvcur[d];
          p.kv[vb + d] = kvcur[D + d];
        }
      } else if (threadIdx.x == 0) {
        record_error(p, MK_ERR_DEVICE_BOUNDS, MK_OP_ATTN, l, MK_NO_COUNTER, static_cast<uint32_t>(page), 0, pg,
                     false);
      }
    }
    trace_mark(61, l);
    float o[MT][4];
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) o[mm][0] = o[mm][1] = o[mm][2] = o[mm][3] = 0.f;
    float mx[2] = {-INFINITY, -INFINITY}, ls[2] = {0.f, 0.f};   // heads 2t, 2t+1 (ls: this lane's share)

    for (;;) {
      const int p0 = static_cast<int>(meta().row0) * p.ps;            // first position of the chunk
      const int npos = min(static_cast<int>(meta().n) * p.ps, Lc - p0);
      const bool last = meta().last;
      const uint32_t Kb = smem_u32(slot());
      const uint32_t Vb = Kb + kSlotBytes / 2;
      for (int tile = warp; tile * 16 < npos; tile += kConsumerWarps) {
        const int r0 = tile * 16;
        bool patched = false;
        if (pos >= p0 + r0 && pos < p0 + r0 + 16) {
          // this token's k and v are not in the copied page yet: put them in its rows
          const int rr = pos - p0;
          for (int cidx = lane; cidx < 2 * (D / 8); cidx += 32) {
            const int which = cidx / (D / 8), d = (cidx - which * (D / 8)) * 8;
            const uint4 v = *reinterpret_cast<const uint4*>(kvcur + which * D + d);
            const uint32_t a = (which ? Vb : Kb) + swz(rr, d, ROWS);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          }
          patched = true;
        }
        if (r0 + 16 > npos) {
          // rows past the sequence: zero them so that 0-probability rows cannot carry NaN into P V
          for (int cidx = lane; cidx < 16 * 2 * (D / 8); cidx += 32) {
            const int rr = r0 + cidx / (2 * (D / 8));
            const int rem = cidx % (2 * (D / 8));
            const int which = rem / (D / 8), d = (rem - which * (D / 8)) * 8;
            if (rr >= npos) {
              const uint32_t a = (which ? Vb : Kb) + swz(rr, d, ROWS);
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
#pragma unroll
        for (int s2 = 0; s2 < KS; ++s2) {
          uint32_t a[4];
          ldsm_x4(Kb + swz(r0 + (lane & 7) + ((lane >> 3) & 1) * 8, 16 * s2 + (lane >> 4) * 8, ROWS), a);
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
          ldsm_x4_t(Vb + swz(r0 + (lane & 7) + (lane >> 4) * 8, 16 * mm + ((lane >> 3) & 1) * 8, ROWS), a);
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
    // merge the warps' states: a tree through shared memory, layout [head][dim] + max[8] + sum[8]
    constexpr int kStride = kMaxG * D + 2 * kMaxG;
    for (int half = kConsumerWarps / 2; half >= 1; half >>= 1) {
      cbar();
      if (warp >= half && warp < 2 * half) {
        float* dst = S.scr.attn + (warp - half) * kStride;
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) {
          dst[(2 * t) * D + 16 * mm + g] = o[mm][0];
          dst[(2 * t + 1) * D + 16 * mm + g] = o[mm][1];
          dst[(2 * t) * D + 16 * mm + g + 8] = o[mm][2];
          dst[(2 * t + 1) * D + 16 * mm + g + 8] = o[mm][3];
        }
        if (g == 0) {
          dst[kMaxG * D + 2 * t] = mx[0];
          dst[kMaxG * D + 2 * t + 1] = mx[1];
          dst[kMaxG * D + kMaxG + 2 * t] = ls[0];
          dst[kMaxG * D + kMaxG + 2 * t + 1] = ls[1];
        }
      }
      cbar();
      if (warp < half) {
        const float* src = S.scr.attn + warp * kStride;
        float fa[2], fb[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float mo = src[kMaxG * D + 2 * t + j], lo = src[kMaxG * D + kMaxG + 2 * t + j];
          const float M = fmaxf(mx[j], mo);
          fa[j] = mx[j] == -INFINITY ? 0.f : __expf(mx[j] - M);
          fb[j] = mo == -INFINITY ? 0.f : __expf(mo - M);
          ls[j] = ls[j] * fa[j] + lo * fb[j];
          mx[j] = M;
        }
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) {
          o[mm][0] = o[mm][0] * fa[0] + src[(2 * t) * D + 16 * mm + g] * fb[0];
          o[mm][1] = o[mm][1] * fa[1] + src[(2 * t + 1) * D + 16 * mm + g] * fb[1];
          o[mm][2] = o[mm][2] * fa[0] + src[(2 * t) * D + 16 * mm + g + 8] * fb[0];
          o[mm][3] = o[mm][3] * fa[1] + src[(2 * t + 1) * D + 16 * mm + g + 8] * fb[1];
        }
      }
    }
    if (warp == 0) {
      float* po = p.PO + static_cast<size_t>(m0.idx) * Gq * D;
      float* pml = p.PML + static_cast<size_t>(m0.idx) * Gq * 2;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = 2 * t + j;
        if (h < Gq) {
#pragma unroll
          for (int mm = 0; mm < MT; ++mm) {
            po[h * D + 16 * mm + g] = o[mm][j];
            po[h * D + 16 * mm + g + 8] = o[mm][j + 2];
          }
          if (g == 0) {
            pml[2 * h] = mx[j];
            pml[2 * h + 1] = ls[j];
          }
        }
      }
    }
    trace_mark(63, l);
    // the last split of (b, kvh) merges every split in split order.  Thread i owns 4 output
    // dims of one head and folds the splits in with a running (max, sum, output); the loads of
    // 16 splits are issued together so that the merge costs a few round trips, not one per split.
    const uint32_t base = p.cm.layer_base(l);
    const int pair = b * p.Hkv + kvh;
    if (consumer_arrive_last(p, S, base + L_PAIR + pair, item.nsplit)) {
      trace_mark(64, l);
      const int first = p.pair_first[pair];
      const int ns = item.nsplit;
      const int q4 = threadIdx.x;                 // float4 index into [Gq][D]
      if (q4 * 4 < Gq * D) {
        const int h = (q4 * 4) / D;
        const float4* po = reinterpret_cast<const float4*>(p.PO) + static_cast<size_t>(first) * (Gq * D / 4) + q4;
        const float2* pml = reinterpret_cast<const float2*>(p.PML) + static_cast<size_t>(first) * Gq + h;
        float M = -INFINITY, Ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        constexpr int kBatch = 16;
        for (int s0 = 0; s0 < ns; s0 += kBatch) {
          float2 ml[kBatch];
          float4 ov[kBatch];
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int s2 = s0 + j;
            ml[j] = s2 < ns ? __ldcg(pml + static_cast<size_t>(s2) * Gq) : make_float2(-INFINITY, 0.f);
            ov[j] = s2 < ns ? __ldcg(po + static_cast<size_t>(s2) * (Gq * D / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            if (ml[j].x == -INFINITY) continue;
            const float Mn = fmaxf(M, ml[j].x);
            const float fa = M == -INFINITY ? 0.f : __expf(M - Mn);
            const float fb = __expf(ml[j].x - Mn);
            Ls = Ls * fa + ml[j].y * fb;
            acc.x = acc.x * fa + ov[j].x * fb;
            acc.y = acc.y * fa + ov[j].y * fb;
            acc.z = acc.z * fa + ov[j].z * fb;
            acc.w = acc.w * fa + ov[j].w * fb;
            M = Mn;
          }
        }
        const float inv = 1.f / Ls;
        float4* dst = reinterpret_cast<float4*>(p.ATT + (static_cast<size_t>(l) * p.max_batch + b) * (p.Hq * D) +
                                                static_cast<size_t>(kvh) * Gq * D) + q4;
        *dst = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      }
      consumer_signal(p, base + L_ATTN);
      trace_mark(65, l);
    }
    return true;
  }

  // ------------------------------------------------------------------ main loop
  __device__ void run() {
    for (;;) {
      bool ok = warp_wait_record(p, S, c);
      trace_chunk_seen();
      if (!cbar_and(ok)) break;   // every warp starts a tile together
      const Meta m0 = meta();
      const uint64_t t0 = p.trace ? globaltimer() : 0;
      twait = 0;
      wok = true;
      switch (m0.kind) {
        case R_EMBED: ok = embed(); break;
        case R_GEMV: ok = stream_gemv(m0.op); break;
        case R_ATTN: ok = attn_item(); break;
        case R_GU: ok = stream_gemv(R_OP_GU); break;
        case R_DOWN: ok = stream_gemv(R_OP_DOWN); break;
        default: break;
      }
      if (!ok) break;
      if (m0.kind != R_END) trace_event(m0.kind == R_ATTN || m0.kind == R_GU || m0.kind == R_DOWN ? TR_ITEM : TR_TILE,
                                        m0, t0);
      trace_chunk_done();
      warp_release_record(S, c);
      ++c;
      if (m0.kind == R_END) break;
    }
    if ((threadIdx.x & 31) == 0) atomicMin(&S.cons_count, c);
    if (threadIdx.x == 0 && p.trace) {
      uint64_t* h = p.trace + static_cast<size_t>(blockIdx.x) * p.trace_cap * 4;
      h[0] = nev;
    }
  }
};

// --------------------------------------------------------------------------- the kernel
template <int TB, int D>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the ring holds 128-byte-swizzled TMA tiles, whose pattern repeats every 1024 bytes
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + pad);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    S.prod_count = 0;
    S.cons_count = 0xffffffffu;
    S.moe_layer = -1;
    S.ykey = -1;
    if (p.trace) p.trace[static_cast<size_t>(blockIdx.x) * p.trace_cap * 4 + 1] = globaltimer();
    fence_mbar_init();
  }
  __syncthreads();
  if (tid >= kConsumerThreads) {
    if (tid == kConsumerThreads) {
      Producer prod(p, S);
      prod.run();
    }
    __syncwarp();
  } else {
    Consumer<TB, D> cons(p, S);
    cons.run();
  }
  __syncthreads();
  // an aborted step may leave copies in flight: let them land before the block exits
  if (tid == 0) {
    for (uint32_t c = S.cons_count; c < S.prod_count; ++c) {
      const int s = static_cast<int>(c % kSlots);
      const uint32_t ph = (c / kSlots) & 1u;
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&S.full[s], ph)) {
        if (globaltimer() - t0 > 100000000ull) break;
      }
    }
    __threadfence();
    const uint32_t old = atom_add_acq_rel(p.ctr + C_FINISH, 1u);
    S.is_last = (old + 1u == gridDim.x) ? 1 : 0;
  }
  __syncthreads();
  if (S.is_last) {
    for (uint32_t i = tid; i < p.cm.total; i += kThreads) p.ctr[i] = 0u;
  }
}

template <int TB, int D>
cudaError_t configure_t(size_t smem) {
  return cudaFuncSetAttribute(step_kernel<TB, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

template <int TB, int D>
cudaError_t launch_t(const Params& p, size_t smem, cudaStream_t s) {
  void* args[] = {const_cast<Params*>(&p)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(step_kernel<TB, D>), dim3(p.n_ctas),
                                     dim3(kThreads), args, smem, s);
}

template <int D>
cudaError_t configure_all(size_t smem) {
  cudaError_t e;
  if ((e = configure_t<1, D>(smem)) != cudaSuccess) return e;
  if ((e = configure_t<2, D>(smem)) != cudaSuccess) return e;
  return configure_t<4, D>(smem);
}

template <int D>
cudaError_t launch_any(const Params& p, int tb, size_t smem, cudaStream_t s) {
  if (tb == 1) return launch_t<1, D>(p, smem, s);
  if (tb == 2) return launch_t<2, D>(p, smem, s);
  return launch_t<4, D>(p, smem, s);
}

template <int D>
cudaError_t occupancy_d(int* blocks, size_t smem) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, step_kernel<1, D>, kThreads, smem);
}

}  // namespace
}  // namespace mk
