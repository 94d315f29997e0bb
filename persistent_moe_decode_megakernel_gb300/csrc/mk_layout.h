// mk_layout.h -- layout shared by the host library and the persistent kernel:
// geometry of the shared-memory ring, tile sizes, the counter map and the
// kernel's parameter block.  Plain C++ (no CUDA types) so both g++ and nvcc
// compile it.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "mk_debug.h"

#ifdef __CUDACC__
#define MK_HD __host__ __device__ __forceinline__
#else
#define MK_HD inline
#endif

namespace mk {

// ---- thread block shape: 8 consumer warps + 1 producer warp ---------------
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;

// ---- shared-memory ring of weight / KV tiles --------------------------------
constexpr int kSlots = 3;
constexpr int kSlotBytes = 65536;

// ---- build limits --------------------------------------------------------------
constexpr int kMaxBatch = 64;
constexpr int kMaxTopK = 8;
constexpr int kMaxG = 8;          // query heads per KV head
constexpr int kMaxExperts = 256;
constexpr int kMaxK = 4096;       // GEMV input length (two 16-byte units per thread)
constexpr int kMaxRowsPerChunk = 32;

// ---- MoE work-queue tiles --------------------------------------------------------
constexpr int kFTile = 16;        // expert FFN rows (gate+up pairs) per gate/up item
constexpr int kRTile = 64;        // hidden rows per down item
constexpr int kRouterRows = 8;    // router (expert) rows per router tile

MK_HD int gemv_rows_per_chunk(int K) {
  int r = kSlotBytes / (2 * K);
  return r > kMaxRowsPerChunk ? kMaxRowsPerChunk : r;
}
// pages of K (and as many of V) per attention chunk: K fills the slot's first half, V the second
MK_HD int pages_per_chunk(int page_size, int head_dim) { return (kSlotBytes / 2) / (page_size * head_dim * 2); }

// ---- counters --------------------------------------------------------------------
// global
enum : uint32_t { C_EMBED = 0, C_FINISH = 1, C_ABORT = 2, C_NEVER = 3, C_GLOBAL = 8 };
// per layer, at layer_base(l) + ...
enum : uint32_t {
  L_QKV = 0,     // QKV tiles done
  L_ATTN = 1,    // (row, kv head) attention pairs combined
  L_O = 2,       // O-proj tiles done
  L_RARR = 3,    // router tiles arrived
  L_RREADY = 4,  // routing published (0/1)
  L_MOEQ = 5,    // MoE queue head (claims)
  L_MOE = 6,     // down row-tiles combined into the residual
  L_PAIR = 8     // [max_batch * Hkv] attention split arrivals, then GU_DONE[E], then DOWN_ARRIVE[n_rtiles]
};

struct CounterMap {
  uint32_t layer_stride;
  uint32_t gu_off;     // offset of GU_DONE[active expert] inside a layer block
  uint32_t down_off;   // offset of DOWN_ARRIVE[row tile]
  uint32_t total;
  MK_HD uint32_t layer_base(int l) const { return C_GLOBAL + (uint32_t)l * layer_stride; }
};

inline CounterMap counter_map(int layers, int max_batch, int n_kv, int n_exp, int n_rtiles) {
  CounterMap m;
  m.gu_off = L_PAIR + (uint32_t)(max_batch * n_kv);
  m.down_off = m.gu_off + (uint32_t)n_exp;
  m.layer_stride = (m.down_off + (uint32_t)n_rtiles + 7u) & ~7u;
  m.total = C_GLOBAL + (uint32_t)layers * m.layer_stride;
  return m;
}

// ---- kernel parameters -------------------------------------------------------------
struct LayerW {
  const uint16_t* attn_norm;
  const uint16_t* w_qkv;
  const uint16_t* w_o;
  const uint16_t* ffn_norm;
  const uint16_t* w_router;
  const float* router_bias;
  const uint16_t* w_gate_up;
  const uint16_t* w_down;
};

struct alignas(64) Params {
  // TMA descriptor (CUtensorMap, 128 bytes) of the KV pool as a 2-D bf16 tensor
  // [L*num_pages*2*Hkv*page_size rows][head_dim], boxes of 64 elements x page_size rows, 128-byte swizzle
  alignas(64) uint64_t kv_map[16];
  // shape
  int32_t L, H, Hq, Hkv, D, G, E, K, F, V, ps, P, maxpg;
  int32_t nqkv;          // (Hq + 2Hkv) * D
  int32_t norm_topk;
  float eps, scale;      // RMSNorm epsilon, 1/sqrt(D)
  int32_t B, max_batch, n_ctas;
  // static plan
  int32_t n_qkv_tiles, n_o_tiles, n_router_tiles, n_ftiles, n_rtiles;
  CounterMap cm;
  uint64_t watchdog_ns;
  const mk_task* tasks;
  const int32_t* task_off;      // [n_ctas + 1]
  // weights
  const LayerW* layers;         // device [L]
  const uint16_t* embed;
  const uint16_t* final_norm;
  const uint16_t* lm_head;
  // step inputs / outputs
  const int32_t* tokens;
  const int32_t* block_tables;
  uint16_t* kv;
  float* logits;
  // per-step plan (device copy of the host-built step buffer)
  const int32_t* seq_lens;      // [B]
  const float* rope_cos;        // [B][D/2]
  const float* rope_sin;        // [B][D/2]
  const mk_attn_item* items;    // [n_items]
  const int32_t* item_off;      // [n_ctas + 1]
  const int32_t* pair_first;    // [B * Hkv] first item of each (row, kv head)
  // workspace
  float* X;        // [2L+1][max_batch][H] residual stream: layer input at 2l, after attention at 2l+1
  float* QKV;      // [L][max_batch][nqkv]
  float* ATT;      // [L][max_batch][Hq*D]
  float* PO;       // [max_items][G][D]   attention split partial outputs (reused by every layer)
  float* PML;      // [max_items][G][2]   their (max, sum)
  float* RLOG;     // [L][max_batch][E]
  int32_t* RIDS;   // [L][max_batch][K]
  float* RW;       // [L][max_batch][K]
  int32_t* ACT;    // [L][E]  active experts in ascending id
  int32_t* NACT;   // [L]
  int32_t* TOK;    // [L][E][max_batch]  (row << 8 | slot) of the rows routed to each expert
  int32_t* CNT;    // [L][E]
  float* HB;       // [L][max_batch][K][F] SwiGLU activations per (row, slot)
  float* PART;     // [L][max_batch][K][H] down-projection output per (row, slot)
  float* SS;       // [2L+1][n_ss_slots][max_batch] per-tile sums of squares of the residual stream
  int32_t n_ss_slots;
  uint32_t* ctr;   // [cm.total]
  mk_status* status;
  // optional timeline: per block `trace_cap` events of 4 x u64 (start, dependency met, end, tag);
  // event 0 of each block holds (consumer events, kernel start, producer events, 0)
  uint64_t* trace;
  int32_t trace_cap;
};

// trace tags: op | layer << 8 | kind << 24 | (uint64)idx << 32
enum : uint32_t { TR_TILE = 1, TR_ITEM = 2, TR_PRODUCER_ROUTE_WAIT = 3, TR_CHUNK = 4, TR_MARK = 5 };

}  // namespace mk
