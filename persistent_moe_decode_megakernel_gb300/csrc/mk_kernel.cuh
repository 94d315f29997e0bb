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
    float red[kConsumerWarps][kMaxRowsPerChunk][4];
    float attn[kAttnScratch];
  } scr;
  float rstd[kMaxBatch];
  float ssred[kConsumerWarps][4];
  int32_t slot_of[kMaxBatch];
  int32_t rids[kMaxBatch * kMaxTopK];
  int32_t ecnt[kMaxExperts];
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

// all consumer threads: wait until record c has landed in its slot
__device__ bool wait_record(const Params& p, Smem& S, uint32_t c) {
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
          record_error(p, MK_ERR_TIMEOUT, 0, -1, MK_NO_COUNTER, c, 0, -1, true);
          break;
        }
      }
    }
  }
  return cbar_and(ok);
}

__device__ __forceinline__ void release_record(Smem& S, uint32_t c) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&S.empty[c % kSlots]);
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
    __threadfence();
    red_release_add(p.ctr + idx, 1u);
  }
}

// consumer-side arrival with "am I last" (acq_rel), broadcast to every consumer thread
__device__ bool consumer_arrive_last(const Params& p, Smem& S, uint32_t idx, uint32_t total) {
  cbar();
  if (threadIdx.x == 0) {
    __threadfence();
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
  __device__ Meta& meta() { return S.meta[c % kSlots]; }
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

  __device__ bool attn_items(const mk_task& t) {
    const int cta = blockIdx.x;
    const int ppc = pages_per_chunk(p.ps, p.D);
    const uint32_t pb = static_cast<uint32_t>(p.ps * p.D * 2);
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
        mbar_arrive_expect_tx(full(), 2u * n * pb);
        uint8_t* dst = slot();
        for (uint32_t i = 0; i < n; ++i) {
          int32_t page = btrow[pg + i];
          if (page < 0 || page >= p.P) {
            record_error(p, MK_ERR_DEVICE_BOUNDS, MK_OP_ATTN, t.layer, MK_NO_COUNTER, static_cast<uint32_t>(page), 0,
                         static_cast<int>(pg + i), false);
            page = 0;  // keep the byte count of the slot; the result is flagged invalid
          }
          const size_t kbase = ((static_cast<size_t>(t.layer) * p.P + page) * 2 * p.Hkv + item.kvh) *
                               static_cast<size_t>(p.ps) * p.D;
          const size_t vbase = kbase + static_cast<size_t>(p.Hkv) * p.ps * p.D;
          bulk_g2s(dst + i * pb, p.kv + kbase, pb, full(), pol);
          bulk_g2s(dst + kSlotBytes / 2 + i * pb, p.kv + vbase, pb, full(), pol);
        }
        ++c;
      }
    }
    return true;
  }

  __device__ bool moe_queue(const mk_task& t) {
    const int l = t.layer;
    const uint32_t base = p.cm.layer_base(l);
    if (!wait_counter(p, base + L_RREADY, 1u, MK_OP_MOE, l)) return false;
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
  }
};

// --------------------------------------------------------------------------- GEMV pieces
// A chunk holds `n` rows of length K (bf16).  Thread t covers the 16-byte units
// u = ut + NTG*i of every row its group handles; groups split the rows when a
// row has fewer than 256 units.
struct Geom {
  int K, U, NTG, P, UPT, g, ut;
  __device__ Geom(int K_) : K(K_) {
    U = K >> 3;
    NTG = U >= kConsumerThreads ? kConsumerThreads : ((U + 31) & ~31);
    P = kConsumerThreads / NTG;
    UPT = (U + NTG - 1) / NTG;
    const int t = threadIdx.x;
    g = t / NTG;
    ut = t - g * NTG;
  }
  __device__ bool unit_ok(int i) const { return g < P && i < UPT && (ut + NTG * i) < U; }
  __device__ int unit(int i) const { return ut + NTG * i; }
};

// Load this thread's slice of the GEMV input for `nt` rows.  src(b) points at row
// b's fp32 vector (length K).  If g is non-null the slice is RMS-normalised with
// S.rstd[b] and the bf16 gain g.
template <int TB>
__device__ __forceinline__ void load_slice(const Geom& G, const float* const* src, int nt, const float* rstd,
                                           const uint16_t* g, float (&y)[2][8][TB]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool ok = G.unit_ok(i);
    const int u = ok ? G.unit(i) : 0;
    float gv[8];
    if (g != nullptr && ok) {
      const uint4 gw = __ldg(reinterpret_cast<const uint4*>(g + u * 8));
      gv[0] = bf_lo(gw.x); gv[1] = bf_hi(gw.x); gv[2] = bf_lo(gw.y); gv[3] = bf_hi(gw.y);
      gv[4] = bf_lo(gw.z); gv[5] = bf_hi(gw.z); gv[6] = bf_lo(gw.w); gv[7] = bf_hi(gw.w);
    }
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (ok && tb < nt) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(src[tb] + u * 8));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(src[tb] + u * 8 + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        if (g != nullptr) {
          const float r = rstd[tb];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = (v[j] * r) * gv[j];
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) y[i][j][tb] = v[j];
    }
  }
}

// Sum of squares of rows src(0..nt-1) (length K, all threads of the consumer
// group cooperate) -> rstd[tb] in shared memory.
template <int TB>
__device__ __forceinline__ void block_rstd(const Params& p, Smem& S, const Geom& G, const float* const* src, int nt, int K,
                           float* rstd_out) {
  float ss[TB];
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) ss[tb] = 0.f;
  if (G.g == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (!G.unit_ok(i)) continue;
      const int u = G.unit(i);
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) {
        if (tb >= nt) continue;
        const float4 a = __ldcg(reinterpret_cast<const float4*>(src[tb] + u * 8));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(src[tb] + u * 8 + 4));
        ss[tb] += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
      }
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int tb = 0; tb < TB; ++tb) {
    const float v = warp_sum(ss[tb]);
    if (lane == 0) S.ssred[warp][tb] = v;
  }
  cbar();
  if (threadIdx.x < nt) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += S.ssred[w][threadIdx.x];
    rstd_out[threadIdx.x] = 1.0f / sqrtf(tot / static_cast<float>(K) + p.eps);
  }
  cbar();
}

// Dot products of the chunk's rows with the input slices; warp-reduced partials
// land in S.scr.red; returns after the barrier that makes them visible.
template <int TB>
__device__ __forceinline__ void gemv_chunk(Smem& S, const Geom& G, const uint8_t* wsm, int n,
                                           const float (&y)[2][8][TB]) {
  float acc[kMaxRowsPerChunk][TB];
#pragma unroll
  for (int r = 0; r < kMaxRowsPerChunk; ++r)
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) acc[r][tb] = 0.f;
  if (G.g < G.P) {
#pragma unroll
    for (int ri = 0; ri < kMaxRowsPerChunk; ++ri) {
      const int r = G.g + G.P * ri;
      if (r < n) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (G.unit_ok(i)) {
            const uint4 w = *reinterpret_cast<const uint4*>(wsm + (static_cast<size_t>(r) * G.K + G.unit(i) * 8) * 2);
            const float wf[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y),
                                 bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
            for (int tb = 0; tb < TB; ++tb)
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[ri][tb] = fmaf(wf[j], y[i][j][tb], acc[ri][tb]);
          }
        }
      }
    }
  }
  const int RG = (n + G.P - 1) / G.P;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int ri = 0; ri < kMaxRowsPerChunk; ++ri) {
    if (ri < RG) {
#pragma unroll
      for (int tb = 0; tb < TB; ++tb) acc[ri][tb] = warp_sum(acc[ri][tb]);
    }
  }
  cbar();  // previous chunk's readers of S.scr are done
  if (lane == 0) {
#pragma unroll
    for (int ri = 0; ri < kMaxRowsPerChunk; ++ri)
      if (ri < RG)
#pragma unroll
        for (int tb = 0; tb < TB; ++tb) S.scr.red[warp][ri][tb] = acc[ri][tb];
  }
  cbar();
}

// Final value of row r (chunk-local) for input tb: the group's warps in order.
template <int TB>
__device__ __forceinline__ float gemv_result(const Smem& S, const Geom& G, int r, int tb) {
  const int grp = r % G.P, ri = r / G.P;
  const int w0 = grp * (G.NTG >> 5), nw = G.NTG >> 5;
  float s = 0.f;
  for (int w = 0; w < nw; ++w) s += S.scr.red[w0 + w][ri][tb];
  return s;
}

// --------------------------------------------------------------------------- consumer
template <int TB, int D>
struct Consumer {
  const Params& p;
  Smem& S;
  uint32_t c = 0;
  float y[2][8][TB];
  int ykey = -1;   // which input the y slices hold (layer*4 + input kind), when B <= TB

  __device__ Consumer(const Params& p_, Smem& S_) : p(p_), S(S_) {}

  __device__ const Meta& meta() const { return S.meta[c % kSlots]; }
  __device__ const uint8_t* slot() const { return S.ring[c % kSlots]; }

  // advance to the next record of a multi-chunk tile
  __device__ bool next() {
    release_record(S, c);
    ++c;
    return wait_record(p, S, c);
  }

  // ------------------------------------------------------------------ inputs
  // input kinds: 0 attention input (x_in, attn_norm), 1 O-proj input (attention output),
  //              2 MoE input (x_mid, ffn_norm), 3 head input (x_final, final_norm)
  __device__ __forceinline__ void input_rows(int kind, int l, int b0, int nt, const float** src, const uint16_t** g, int* K) {
    const size_t xs = static_cast<size_t>(p.max_batch) * p.H;
    for (int tb = 0; tb < TB; ++tb) {
      const int b = b0 + (tb < nt ? tb : 0);
      switch (kind) {
        case 0: src[tb] = p.X + (2 * static_cast<size_t>(l)) * xs + static_cast<size_t>(b) * p.H; break;
        case 1: src[tb] = p.ATT + (static_cast<size_t>(l) * p.max_batch + b) * (p.Hq * p.D); break;
        case 2: src[tb] = p.X + (2 * static_cast<size_t>(l) + 1) * xs + static_cast<size_t>(b) * p.H; break;
        default: src[tb] = p.X + (2 * static_cast<size_t>(p.L)) * xs + static_cast<size_t>(b) * p.H; break;
      }
    }
    switch (kind) {
      case 0: *g = p.layers[l].attn_norm; *K = p.H; break;
      case 1: *g = nullptr; *K = p.Hq * p.D; break;
      case 2: *g = p.layers[l].ffn_norm; *K = p.H; break;
      default: *g = p.final_norm; *K = p.H; break;
    }
  }

  // load (and normalise) input rows b0..b0+nt-1 into y
  __device__ __forceinline__ void load_input(int kind, int l, int b0, int nt) {
    const float* src[TB];
    const uint16_t* g;
    int K;
    input_rows(kind, l, b0, nt, src, &g, &K);
    Geom G(K);
    if (g != nullptr) block_rstd<TB>(p, S, G, src, nt, K, S.rstd);
    load_slice<TB>(G, src, nt, S.rstd, g, y);
  }

  // ------------------------------------------------------------------ EMBED
  __device__ bool embed() {
    const Meta m = meta();
    const int H = p.H;
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
      for (uint32_t col = m.lo + threadIdx.x; col < m.hi; col += kConsumerThreads) x[col] = bf1(row[col]);
    }
    consumer_signal(p, m.signal_ctr);
    return true;
  }

  // ------------------------------------------------------------------ GEMV tiles (QKV / O / router / head)
  __device__ bool gemv_tile() {
    const Meta m0 = meta();
    const int op = m0.op, l = m0.layer;
    const int kind = op == MK_OP_QKV ? 0 : op == MK_OP_OPROJ ? 1 : op == MK_OP_ROUTER ? 2 : 3;
    if (m0.wait_ctr != MK_NO_COUNTER && !consumer_wait(p, m0.wait_ctr, m0.wait_target, op, l)) return false;
    const int B = p.B;
    const float* src[TB];
    const uint16_t* g;
    int K;
    input_rows(kind, op == MK_OP_HEAD ? p.L : l, 0, 1, src, &g, &K);
    Geom G(K);
    const int key = (op == MK_OP_HEAD ? p.L : l) * 4 + kind;
    if (B <= TB && ykey != key) {
      load_input(kind, l, 0, B);
      ykey = key;
    }
    const size_t xs = static_cast<size_t>(p.max_batch) * p.H;
    for (;;) {
      const Meta m = meta();
      const uint8_t* wsm = slot();
      for (int b0 = 0; b0 < B; b0 += TB) {
        const int nt = min(TB, B - b0);
        if (B > TB) {
          load_input(kind, l, b0, nt);
          ykey = -1;
        }
        gemv_chunk<TB>(S, G, wsm, m.n, y);
        const int t = threadIdx.x;
        if (t < m.n * TB) {
          const int r = t / TB, tb = t % TB;
          if (tb < nt) {
            const float v = gemv_result<TB>(S, G, r, tb);
            const int b = b0 + tb;
            const uint32_t row = m.row0 + r;
            switch (op) {
              case MK_OP_QKV:
                p.QKV[(static_cast<size_t>(l) * p.max_batch + b) * p.nqkv + row] = v;
                break;
              case MK_OP_OPROJ: {
                const size_t off = static_cast<size_t>(b) * p.H + row;
                p.X[(2 * static_cast<size_t>(l) + 1) * xs + off] = __ldcg(p.X + 2 * static_cast<size_t>(l) * xs + off) + v;
                break;
              }
              case MK_OP_ROUTER: {
                const float* bias = p.layers[l].router_bias;
                p.RLOG[(static_cast<size_t>(l) * p.max_batch + b) * p.E + row] = bias ? v + __ldg(bias + row) : v;
                break;
              }
              default:
                p.logits[static_cast<size_t>(b) * p.V + row] = v;
                break;
            }
          }
        }
      }
      if (m.last) break;
      if (!next()) return false;
    }
    if (op == MK_OP_ROUTER) {
      const uint32_t base = p.cm.layer_base(l);
      if (consumer_arrive_last(p, S, base + L_RARR, static_cast<uint32_t>(p.n_router_tiles))) route(l);
      return true;
    }
    consumer_signal(p, m0.signal_ctr);
    return true;
  }

  // ------------------------------------------------------------------ routing (last router tile)
  __device__ void route(int l) {
    const int B = p.B, E = p.E, K = p.K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t lb = static_cast<size_t>(l) * p.max_batch;
    for (int b = warp; b < B; b += kConsumerWarps) {
      const float* r = p.RLOG + (lb + b) * E;
      float v[kMaxExperts / 32];
      uint32_t taken = 0;
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldcg(r + e) : -INFINITY;
        mx = fmaxf(mx, v[i]);
      }
      mx = warp_max(mx);
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i) {
        const int e = lane + 32 * i;
        if (e < E) z += expf(v[i] - mx);
      }
      z = warp_sum(z);
      float psel[kMaxTopK];
      int isel[kMaxTopK];
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        psel[j] = 0.f;
        isel[j] = 0;
        if (j >= K) continue;
        // local best among untaken: larger value, then lower index
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i) {
          const int e = lane + 32 * i;
          if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) { bv = v[i]; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        isel[j] = bi;
        psel[j] = expf(bv - mx) / z;
        psum += psel[j];
      }
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
          if (j >= K) continue;
          const float w = p.norm_topk ? psel[j] / psum : psel[j];
          p.RIDS[(lb + b) * K + j] = isel[j];
          p.RW[(lb + b) * K + j] = w;
          S.rids[b * K + j] = isel[j];
        }
      }
    }
    cbar();
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
    consumer_signal(p, p.cm.layer_base(l) + L_RREADY);
  }

  // which slot (rank) expert e has in row b's choice, or -1
  __device__ void slots_for_expert(int l, int e) {
    const int K = p.K;
    if (threadIdx.x < p.B) {
      const int32_t* ids = p.RIDS + (static_cast<size_t>(l) * p.max_batch + threadIdx.x) * K;
      int s = -1;
      for (int j = 0; j < K; ++j)
        if (__ldcg(ids + j) == e) s = j;
      S.slot_of[threadIdx.x] = s;
    }
    cbar();
  }

  // ------------------------------------------------------------------ MoE gate/up item
  __device__ bool gate_up_item() {
    const Meta m0 = meta();
    const int l = m0.layer, e = static_cast<int>(m0.e), a = static_cast<int>(m0.idx);
    const uint32_t base = p.cm.layer_base(l);
    if (!consumer_wait(p, base + L_RREADY, 1u, MK_OP_MOE, l)) return false;
    const int B = p.B, H = p.H, F = p.F, K = p.K;
    Geom G(H);
    slots_for_expert(l, e);
    const int key = l * 4 + 2;
    if (B <= TB && ykey != key) {
      load_input(2, l, 0, B);
      ykey = key;
    }
    const int cnt = B <= TB ? B : __ldcg(p.CNT + static_cast<size_t>(l) * p.E + e);
    const int32_t* tok = p.TOK + (static_cast<size_t>(l) * p.E + e) * p.max_batch;
    for (;;) {
      const Meta m = meta();
      const int nf = m.n;
      for (int b0 = 0; b0 < cnt; b0 += TB) {
        const int nt = min(TB, cnt - b0);
        int rowb[TB], rowj[TB];
        for (int tb = 0; tb < TB; ++tb) {
          if (B <= TB) { rowb[tb] = b0 + tb; rowj[tb] = tb < nt ? S.slot_of[b0 + tb] : -1; }
          else {
            const int ent = tb < nt ? __ldcg(tok + b0 + tb) : 0;
            rowb[tb] = ent >> 8; rowj[tb] = tb < nt ? (ent & 0xff) : -1;
          }
        }
        if (B > TB) {
          const float* src[TB];
          const size_t xs = static_cast<size_t>(p.max_batch) * p.H;
          for (int tb = 0; tb < TB; ++tb)
            src[tb] = p.X + (2 * static_cast<size_t>(l) + 1) * xs + static_cast<size_t>(rowb[tb]) * H;
          block_rstd<TB>(p, S, G, src, nt, H, S.rstd);
          load_slice<TB>(G, src, nt, S.rstd, p.layers[l].ffn_norm, y);
          ykey = -1;
        }
        gemv_chunk<TB>(S, G, slot(), 2 * nf, y);
        const int t = threadIdx.x;
        if (t < nf * TB) {
          const int f = t / TB, tb = t % TB;
          if (tb < nt && rowj[tb] >= 0) {
            const float gate = gemv_result<TB>(S, G, f, tb);
            const float up = gemv_result<TB>(S, G, nf + f, tb);
            const float h = (gate / (1.0f + expf(-gate))) * up;
            p.HB[((static_cast<size_t>(l) * p.max_batch + rowb[tb]) * K + rowj[tb]) * F + m.row0 + f] = h;
          }
        }
      }
      if (m.last) break;
      if (!next()) return false;
    }
    consumer_signal(p, base + p.cm.gu_off + a);
    return true;
  }

  // ------------------------------------------------------------------ MoE down item
  __device__ bool down_item() {
    const Meta m0 = meta();
    const int l = m0.layer, e = static_cast<int>(m0.e), a = static_cast<int>(m0.idx);
    const uint32_t base = p.cm.layer_base(l);
    if (!consumer_wait(p, base + p.cm.gu_off + a, static_cast<uint32_t>(p.n_ftiles), MK_OP_MOE, l)) return false;
    const int B = p.B, H = p.H, F = p.F, K = p.K;
    Geom G(F);
    slots_for_expert(l, e);
    const int cnt = B <= TB ? B : __ldcg(p.CNT + static_cast<size_t>(l) * p.E + e);
    const int32_t* tok = p.TOK + (static_cast<size_t>(l) * p.E + e) * p.max_batch;
    bool loaded = false;
    for (;;) {
      const Meta m = meta();
      for (int b0 = 0; b0 < cnt; b0 += TB) {
        const int nt = min(TB, cnt - b0);
        int rowb[TB], rowj[TB];
        for (int tb = 0; tb < TB; ++tb) {
          if (B <= TB) { rowb[tb] = b0 + tb; rowj[tb] = tb < nt ? S.slot_of[b0 + tb] : -1; }
          else {
            const int ent = tb < nt ? __ldcg(tok + b0 + tb) : 0;
            rowb[tb] = ent >> 8; rowj[tb] = tb < nt ? (ent & 0xff) : -1;
          }
        }
        if (B > TB || !loaded) {
          const float* src[TB];
          for (int tb = 0; tb < TB; ++tb) {
            const int j = rowj[tb] >= 0 ? rowj[tb] : 0;
            src[tb] = p.HB + ((static_cast<size_t>(l) * p.max_batch + rowb[tb]) * K + j) * F;
          }
          int ntl = nt;
          load_slice<TB>(G, src, ntl, nullptr, nullptr, y);
          // rows of other experts contribute nothing
#pragma unroll
          for (int tb = 0; tb < TB; ++tb)
            if (rowj[tb] < 0)
#pragma unroll
              for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) y[i][j][tb] = 0.f;
          loaded = true;
          ykey = -1;
        }
        gemv_chunk<TB>(S, G, slot(), m.n, y);
        const int t = threadIdx.x;
        if (t < m.n * TB) {
          const int r = t / TB, tb = t % TB;
          if (tb < nt && rowj[tb] >= 0) {
            const float v = gemv_result<TB>(S, G, r, tb);
            p.PART[((static_cast<size_t>(l) * p.max_batch + rowb[tb]) * K + rowj[tb]) * H + m.row0 + r] = v;
          }
        }
      }
      if (m.last) break;
      if (!next()) return false;
    }
    // the last item of this row tile adds every slot into the residual, in rank order
    const uint32_t rt = m0.aux;
    const uint32_t nact = static_cast<uint32_t>(__ldcg(p.NACT + l));
    if (consumer_arrive_last(p, S, base + p.cm.down_off + rt, nact)) {
      const size_t xs = static_cast<size_t>(p.max_batch) * H;
      const int r0 = static_cast<int>(rt) * kRTile, r1 = min(H, r0 + kRTile);
      const int nr = r1 - r0;
      for (int idx = threadIdx.x; idx < B * nr; idx += kConsumerThreads) {
        const int b = idx / nr, r = r0 + idx % nr;
        const size_t lb = static_cast<size_t>(l) * p.max_batch + b;
        float acc = 0.f;
        for (int j = 0; j < K; ++j) acc += __ldcg(p.RW + lb * K + j) * __ldcg(p.PART + (lb * K + j) * H + r);
        const size_t off = static_cast<size_t>(b) * H + r;
        p.X[(2 * static_cast<size_t>(l) + 2) * xs + off] = __ldcg(p.X + (2 * static_cast<size_t>(l) + 1) * xs + off) + acc;
      }
      consumer_signal(p, base + L_MOE);
    }
    return true;
  }

  // ------------------------------------------------------------------ attention split item
  __device__ bool attn_item() {
    constexpr int DL = D / 32;   // dims per lane
    const Meta m0 = meta();
    const int l = m0.layer;
    if (!consumer_wait(p, m0.wait_ctr, m0.wait_target, MK_OP_ATTN, l)) return false;
    const mk_attn_item item = p.items[m0.idx];
    const int b = item.b, kvh = item.kvh, Gq = p.G;
    const int Lc = p.seq_lens[b];
    const int pos = Lc - 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* qkv = p.QKV + (static_cast<size_t>(l) * p.max_batch + b) * p.nqkv;
    const float* cs = p.rope_cos + static_cast<size_t>(b) * (D / 2);
    const float* sn = p.rope_sin + static_cast<size_t>(b) * (D / 2);
    // q (rotated, scaled) for the group's heads; k and v of this token, bf16-rounded
    float q[kMaxG][DL], kc[DL], vc[DL];
    const int d0 = lane * DL;
    float cv[DL], sv[DL];
#pragma unroll
    for (int d = 0; d < DL; ++d) {
      const int i = (d0 + d) % (D / 2);
      cv[d] = __ldg(cs + i);
      sv[d] = __ldg(sn + i);
    }
    const bool lowhalf = lane < 16;
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
#pragma unroll
      for (int d = 0; d < DL; ++d) {
        const float raw = h < Gq ? __ldcg(qkv + (kvh * Gq + h) * D + d0 + d) : 0.f;
        const float other = __shfl_xor_sync(0xffffffffu, raw, 16);
        const float rot = lowhalf ? raw * cv[d] - other * sv[d] : raw * cv[d] + other * sv[d];
        q[h][d] = rot * p.scale;
      }
    }
#pragma unroll
    for (int d = 0; d < DL; ++d) {
      const float raw = __ldcg(qkv + (p.Hq + kvh) * D + d0 + d);
      const float other = __shfl_xor_sync(0xffffffffu, raw, 16);
      kc[d] = round_bf16(lowhalf ? raw * cv[d] - other * sv[d] : raw * cv[d] + other * sv[d]);
      vc[d] = round_bf16(__ldcg(qkv + (p.Hq + p.Hkv + kvh) * D + d0 + d));
    }
    if (item.split == 0 && warp == 0) {
      // append this token's k and v to the cache
      const int pg = pos / p.ps, sl = pos % p.ps;
      const int32_t page = __ldg(p.block_tables + static_cast<size_t>(b) * p.maxpg + pg);
      if (page >= 0 && page < p.P) {
        const size_t kb = (((static_cast<size_t>(l) * p.P + page) * 2 * p.Hkv + kvh) * p.ps + sl) * D + d0;
        const size_t vb = kb + static_cast<size_t>(p.Hkv) * p.ps * D;
#pragma unroll
        for (int d = 0; d < DL; ++d) {
          p.kv[kb + d] = to_bf16_bits(kc[d]);
          p.kv[vb + d] = to_bf16_bits(vc[d]);
        }
      } else if (lane == 0) {
        record_error(p, MK_ERR_DEVICE_BOUNDS, MK_OP_ATTN, l, MK_NO_COUNTER, static_cast<uint32_t>(page), 0, pg,
                     false);
      }
    }
    float mrun = -INFINITY, lrun = 0.f;   // for head hl
    float o[kMaxG][DL];
#pragma unroll
    for (int h = 0; h < kMaxG; ++h)
#pragma unroll
      for (int d = 0; d < DL; ++d) o[h][d] = 0.f;

    for (;;) {
      const Meta m = meta();
      const int p0 = static_cast<int>(m.row0) * p.ps;            // first position of the chunk
      const int npos = min(static_cast<int>(m.n) * p.ps, Lc - p0);
      const uint16_t* Ks = reinterpret_cast<const uint16_t*>(slot());
      const uint16_t* Vs = reinterpret_cast<const uint16_t*>(slot() + kSlotBytes / 2);
      const int nmine = npos > warp ? (npos - warp + kConsumerWarps - 1) / kConsumerWarps : 0;
      for (int i0 = 0; i0 < nmine; i0 += 8) {
        float sc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int pl = warp + kConsumerWarps * (i0 + i);
          const bool valid = (i0 + i) < nmine;
          float kf[DL];
          if (valid && p0 + pl == pos) {
#pragma unroll
            for (int d = 0; d < DL; ++d) kf[d] = kc[d];
          } else if (valid) {
            unpack_row<DL>(Ks + static_cast<size_t>(pl) * D + d0, kf);
          } else {
#pragma unroll
            for (int d = 0; d < DL; ++d) kf[d] = 0.f;
          }
          float v[kMaxG];
#pragma unroll
          for (int h = 0; h < kMaxG; ++h) {
            float s = 0.f;
#pragma unroll
            for (int d = 0; d < DL; ++d) s = fmaf(q[h][d], kf[d], s);
            v[h] = s;
          }
          // reduce-scatter over the 8 head values: lane ends with head (lane>>2)&7
          {
            const bool b4 = lane & 16;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float send = b4 ? v[k] : v[k + 4];
              const float keep = b4 ? v[k + 4] : v[k];
              v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
            const bool b3 = lane & 8;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const float send = b3 ? v[k] : v[k + 2];
              const float keep = b3 ? v[k + 2] : v[k];
              v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
            const bool b2 = lane & 4;
            const float send = b2 ? v[0] : v[1];
            const float keep = b2 ? v[1] : v[0];
            v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
          }
          sc[i] = valid ? v[0] : -INFINITY;
        }
        // online softmax for head hl over these (up to 8) positions
        float mx = mrun;
#pragma unroll
        for (int i = 0; i < 8; ++i) mx = fmaxf(mx, sc[i]);
        const float corr = (mrun == -INFINITY) ? 0.f : __expf(mrun - mx);
        float pr[8];
        float ls = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          pr[i] = sc[i] == -INFINITY ? 0.f : __expf(sc[i] - mx);
          ls += pr[i];
        }
        lrun = lrun * corr + ls;
        mrun = mx;
        // o[h] = o[h]*corr_h + sum_i p_h[i] v_i
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
          const float ch = __shfl_sync(0xffffffffu, corr, h * 4);
#pragma unroll
          for (int d = 0; d < DL; ++d) o[h][d] *= ch;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if ((i0 + i) >= nmine) break;
          const int pl = warp + kConsumerWarps * (i0 + i);
          float vf[DL];
          if (p0 + pl == pos) {
#pragma unroll
            for (int d = 0; d < DL; ++d) vf[d] = vc[d];
          } else {
            unpack_row<DL>(Vs + static_cast<size_t>(pl) * D + d0, vf);
          }
#pragma unroll
          for (int h = 0; h < kMaxG; ++h) {
            const float ph = __shfl_sync(0xffffffffu, pr[i], h * 4);
#pragma unroll
            for (int d = 0; d < DL; ++d) o[h][d] = fmaf(ph, vf[d], o[h][d]);
          }
        }
      }
      if (m.last) break;
      if (!next()) return false;
    }

    // gather each head's (m, l) on every lane, then merge the 8 warps' states
    float mh[kMaxG], lh[kMaxG];
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
      mh[h] = __shfl_sync(0xffffffffu, mrun, h * 4);
      lh[h] = __shfl_sync(0xffffffffu, lrun, h * 4);
    }
    constexpr int kStride = kMaxG * (128 + 2);
    for (int half = kConsumerWarps / 2; half >= 1; half >>= 1) {
      cbar();
      if (warp >= half && warp < 2 * half) {
        float* dst = S.scr.attn + (warp - half) * kStride;
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
#pragma unroll
          for (int d = 0; d < DL; ++d) dst[h * D + d0 + d] = o[h][d];
        }
        if (lane < kMaxG) {
          dst[kMaxG * D + 2 * lane] = mh[lane];
          dst[kMaxG * D + 2 * lane + 1] = lh[lane];
        }
      }
      cbar();
      if (warp < half) {
        const float* src = S.scr.attn + warp * kStride;
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
          const float mo = src[kMaxG * D + 2 * h], lo = src[kMaxG * D + 2 * h + 1];
          const float M = fmaxf(mh[h], mo);
          const float fa = mh[h] == -INFINITY ? 0.f : __expf(mh[h] - M);
          const float fb = mo == -INFINITY ? 0.f : __expf(mo - M);
#pragma unroll
          for (int d = 0; d < DL; ++d) o[h][d] = o[h][d] * fa + src[h * D + d0 + d] * fb;
          lh[h] = lh[h] * fa + lo * fb;
          mh[h] = M;
        }
      }
    }
    if (warp == 0) {
      float* po = p.PO + static_cast<size_t>(m0.idx) * Gq * D;
      float* pml = p.PML + static_cast<size_t>(m0.idx) * Gq * 2;
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h < Gq) {
#pragma unroll
          for (int d = 0; d < DL; ++d) po[h * D + d0 + d] = o[h][d];
        }
      }
      if (lane < Gq) {
        pml[2 * lane] = mh[lane];
        pml[2 * lane + 1] = lh[lane];
      }
    }
    // the last split of (b, kvh) merges every split in split order
    const uint32_t base = p.cm.layer_base(l);
    const int pair = b * p.Hkv + kvh;
    if (consumer_arrive_last(p, S, base + L_PAIR + pair, item.nsplit)) {
      const int first = p.pair_first[pair];
      const int ns = item.nsplit;
      if (warp < Gq) {
        const int h = warp;
        float mloc = -INFINITY;
        for (int s = lane; s < ns; s += 32) mloc = fmaxf(mloc, __ldcg(p.PML + (static_cast<size_t>(first + s) * Gq + h) * 2));
        const float M = warp_max(mloc);
        float lloc = 0.f;
        for (int s = lane; s < ns; s += 32) {
          const float ms = __ldcg(p.PML + (static_cast<size_t>(first + s) * Gq + h) * 2);
          const float ls = __ldcg(p.PML + (static_cast<size_t>(first + s) * Gq + h) * 2 + 1);
          if (ms != -INFINITY) lloc += __expf(ms - M) * ls;
        }
        const float Lsum = warp_sum(lloc);
        float acc[DL];
#pragma unroll
        for (int d = 0; d < DL; ++d) acc[d] = 0.f;
        for (int s = 0; s < ns; ++s) {
          const float ms = __ldcg(p.PML + (static_cast<size_t>(first + s) * Gq + h) * 2);
          const float f = ms == -INFINITY ? 0.f : __expf(ms - M);
          const float* src = p.PO + (static_cast<size_t>(first + s) * Gq + h) * D + d0;
#pragma unroll
          for (int d = 0; d < DL; ++d) acc[d] = fmaf(f, __ldcg(src + d), acc[d]);
        }
        float* dst = p.ATT + (static_cast<size_t>(l) * p.max_batch + b) * (p.Hq * D) + (kvh * Gq + h) * D + d0;
#pragma unroll
        for (int d = 0; d < DL; ++d) dst[d] = acc[d] / Lsum;
      }
      consumer_signal(p, base + L_ATTN);
    }
    return true;
  }

  // ------------------------------------------------------------------ main loop
  __device__ void run() {
    for (;;) {
      if (!wait_record(p, S, c)) break;
      const uint8_t kind = meta().kind;
      bool ok = true;
      switch (kind) {
        case R_EMBED: ok = embed(); break;
        case R_GEMV: ok = gemv_tile(); break;
        case R_ATTN: ok = attn_item(); break;
        case R_GU: ok = gate_up_item(); break;
        case R_DOWN: ok = down_item(); break;
        default: break;
      }
      release_record(S, c);
      ++c;
      if (kind == R_END || !ok) break;
    }
    if (threadIdx.x == 0) S.cons_count = c;
  }
};

// --------------------------------------------------------------------------- the kernel
template <int TB, int D>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    S.prod_count = 0;
    S.cons_count = 0;
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
