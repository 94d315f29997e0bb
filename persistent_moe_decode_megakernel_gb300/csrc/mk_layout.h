// mk_layout.h -- layout shared by the host library and the persistent kernel:
// geometry of the shared-memory ring, tile sizes, the MoE work split, the step
// flags and the kernel's parameter block.  Plain C++ (no CUDA types) so both g++ and nvcc
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

// Builds with MK_TRACE=1 record the per-tile timeline of mk_debug_trace; the default build
// compiles it out of the step kernel.
#ifndef MK_TRACE
#define MK_TRACE 0
#endif

namespace mk {

constexpr bool kTrace = MK_TRACE != 0;

// ---- thread block shape: two consumer warpgroups + one producer warpgroup -------
// (one producer thread issues the copies; the producer warpgroup hands most of its
// registers to the consumers: 256 x kConsumerRegs + 128 x kProducerRegs = 384 x 168.  72 for
// the producer: with 56 its MoE task loops spilled in the tcgen05 instantiation and the
// narrow ones spilled too; 216 keeps the consumers of every instantiation but the 4-row one
// free of spills)
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 128;
constexpr int kLaunchRegs = 168;
constexpr int kConsumerRegs = 216;
constexpr int kProducerRegs = 72;
static_assert(kConsumerThreads * kConsumerRegs + 128 * kProducerRegs == kThreads * kLaunchRegs,
              "register hand-over must add up to the launch allocation");

// ---- shared-memory ring of weight / KV tiles --------------------------------
constexpr int kSlots = 2;
constexpr int kSlotBytes = 69632;

// ---- build limits --------------------------------------------------------------
constexpr int kMaxBatch = 64;
constexpr int kMaxTopK = 8;
constexpr int kMaxG = 8;          // query heads per KV head
constexpr int kMaxExperts = 256;
constexpr int kMaxK = 4096;       // GEMV input length (two 16-byte units per thread)
constexpr int kMaxRowsPerChunk = 32;
constexpr int kMaxCtas = 256;     // thread blocks (SMs) a step may use
constexpr int kMoeScratch = 12288;  // floats of shared memory for the down projection of one block

constexpr int kRouterRows = 8;    // router (expert) rows per router tile
// Router rows per tile: kRouterRows, or for engines sized for batches of 8 or more (where a
// tile's cost grows with the batch) as few as spreads the experts over every block.
MK_HD int router_tile_rows(int E, int n_ctas, int max_batch) {
  return max_batch >= 8 ? (E + n_ctas - 1) / n_ctas : kRouterRows;
}

// Rows of the batch per register group in the widest GEMV instantiation: four, or as many
// rows of length K as the input staging area holds (three at K = 4096), so that every
// group's input is staged once in shared memory.
MK_HD int wide_group_rows(int K) { return 4 * K <= kMoeScratch ? 4 : kMoeScratch / K; }
constexpr int kAttnScratch = 4 * kMaxG * (128 + 2);   // floats: attention prologue / cached MoE input

// ---- small-batch MoE path ----------------------------------------------------------
// For batches of at most kSmallMaxB rows whose MoE input fits the input cache, each block
// runs its gate/up units end to end: gate/up rows, then the same FFN rows of the transposed
// down projection (w_down_t, [E][F][H]), accumulated into an on-chip [B][H] partial output;
// the blocks' partials are then summed per hidden row by the row's owner block.
constexpr int kSmallMaxB = 2;
constexpr int kMaxUnits = 256;    // gate/up units of one block whose SwiGLU outputs stay on chip
// (a warp's register slice covers 2048/TB input values, TB the rows of a register group: the
// gate/up rows must fit one warp whole, or split rows would reuse the input cache's storage)
MK_HD bool small_moe_batch(int B, int H) {
  const int tb = B <= 1 ? 1 : 2;
  return B <= kSmallMaxB && tb * H <= 8 * kConsumerThreads && B * H <= kAttnScratch;
}

// ---- wide batches on tcgen05 ------------------------------------------------------
// Batches of kTcMinBatch rows or more run the dense GEMV tiles (QKV, O-proj, router, LM head) on
// the 5th-generation tensor cores: the weight tile is the A operand (M-blocks of 64 or 128 rows,
// K-major, 128-byte swizzle, loaded by TMA in 64-column slices), the whole batch the B operand
// (N = the batch rounded up to 16, staged by the consumers one 64-column slice at a time as bf16
// terms of the fp32 input), the accumulators in tensor memory.
constexpr int kTcMinBatch = 5;
constexpr int kTcUnitBytes128 = 128 * 128;   // one 64-column slice of a 128-row M-block
constexpr int kTcChunkBytes = 65536;          // A units of one ring record
constexpr int kTcXBufs = 3;                   // input slices in flight (fewer when three terms do not fit)
constexpr int kTcReqs = 4;                    // MMA requests in flight from the consumers to the issuing warp
constexpr int kTcCols = 512;                  // tensor-memory columns (all of them: one block per SM)
MK_HD int tc_mblock(int rows) { return rows <= 64 ? 64 : 128; }
MK_HD int tc_batch_cols(int B) { return (B + 15) & ~15; }
// bf16 terms of the fp32 input (one accumulator each: the tensor cores align a sum to its largest
// addend, so a small term summed into a large accumulator would lose its low bits): three keep the
// input whole for the QKV projection (the step rounds its k and v to bf16 for the cache), two
// (~16 bits) elsewhere
MK_HD int tc_terms(int op) { return op == MK_OP_QKV ? 3 : 2; }
// Accumulators of the high term: the QKV projection spreads its 64-column slices over several
// (slice s into accumulator s mod G), summed in fp32 at the end, so that each takes fewer tensor-core
// roundings of a large running sum; one elsewhere.  Accumulators per M-block: G + terms - 1.
MK_HD int tc_hi_groups(int op, int B, int K) {
  if (op != MK_OP_QKV) return 1;
  const int ns = (K + 63) / 64, fit = kTcCols / tc_batch_cols(B) - (tc_terms(op) - 1);
  int g = fit < 8 ? fit : 8;
  g = g < ns ? g : ns;
  return g > 1 ? g : 1;
}
MK_HD int tc_accs(int op, int B, int K) { return tc_hi_groups(op, B, K) + tc_terms(op) - 1; }
// Split-K of the dense tcgen05 tiles: every block reads its tile's whole input from L2, so the
// QKV projection (2), the O-proj and the router (8) run in groups of consecutive blocks that
// share the group's rows, each over a 1/KS share of K; each block publishes its partial sums and
// sums of squares, then finalises its own rows from the group's partials in block order.  Only
// where the groups tile the blocks (and the router tiles) evenly, every block holds rows (rows:
// the QKV width for the QKV projection, the hidden size for the O-proj) and every block gets at
// least one 64-column slice of K.  (QKV stays at 2: a group of 4 would hold two 128-row M-blocks,
// and its accumulators would not fit the tensor memory in one pass.)
MK_HD int tc_ksplit(int op, int n_ctas, int n_router_tiles, int rows, int K) {
  const int ks = op == MK_OP_QKV ? 2 : (op == MK_OP_OPROJ || op == MK_OP_ROUTER) ? 8 : 1;
  if (ks == 1 || n_ctas % ks != 0 || (op == MK_OP_ROUTER && n_router_tiles % ks != 0)) return 1;
  if (op != MK_OP_ROUTER && rows < n_ctas) return 1;
  if ((K + 63) / 64 < ks) return 1;
  return ks;
}
MK_HD int tc_split_slot(int op) { return op == MK_OP_QKV ? 0 : op == MK_OP_OPROJ ? 1 : 2; }
// the tile kind of the experts' down projections (a record op beside the MK_OP_* of mk_debug.h)
constexpr int kTcOpDown = 16;
// hidden rows per down-projection unit (one 128-row M-block of one expert)
constexpr int kTcDownRows = 128;
// tensor map of a weight matrix: QKV of layer l, O-proj, router, the LM head, the experts' gate/up
// rows of layer l ([E * 2F rows][H]), then their down projections ([E * H rows][F])
MK_HD int tc_map_index(int op, int layer, int L) {
  return op == MK_OP_QKV ? layer : op == MK_OP_OPROJ ? L + layer : op == MK_OP_ROUTER ? 2 * L + layer
       : op == MK_OP_MOE ? 3 * L + 1 + layer : op == kTcOpDown ? 4 * L + 1 + layer : 3 * L;
}
constexpr int tc_map_count(int L) { return 5 * L + 1; }

MK_HD int gemv_rows_per_chunk(int K) {
  int r = kSlotBytes / (2 * K);
  return r > kMaxRowsPerChunk ? kMaxRowsPerChunk : r;
}
// bf16 cache: pages per attention chunk, each page's K rows then its V rows (page_size rows of
// head_dim bf16 each), rounded down so that the chunk's positions are whole 16-row tiles (the
// consumers' unit of work); 0 when a single page cannot be held that way
MK_HD int pages_per_chunk(int page_size, int head_dim) {
  int n = kSlotBytes / (2 * page_size * head_dim * 2);
  while (n > 0 && (n * page_size) % 16 != 0) --n;
  return n;
}
// q8_0 cache: pages per chunk, each page's K and V codes (page_size rows of head_dim bytes) and
// their f16 scales (head_dim/32 per row); the slot holds [K codes][V codes][K scales][V scales]
MK_HD int pages_per_chunk_q8(int page_size, int head_dim) {
  return kSlotBytes / (page_size * (2 * head_dim + 2 * (head_dim / 32) * 2));
}

// ---- MoE work split ---------------------------------------------------------------
// Gate/up work of a layer is a list of units, one per FFN row f of each active expert a
// (unit index a * F + f, active experts in ascending id).  A unit costs its weight
// bytes plus the batch rows it serves: max(4, rows routed to the expert), so at small
// batch every unit weighs the same and at large batch crowded experts count for more.
// Block j takes the units whose cost prefix starts in [C*j/N, C*(j+1)/N), C the total.
// (On the tcgen05 path of wide batches the routed rows are the N columns of the MMAs: a unit
// costs its weight bytes plus a share that grows with its rows' 16-column groups, the MMA time.
// The down projection's (expert, row block) units are dealt by the same per-expert cost.)
constexpr int kTcUnitBase = 4;
MK_HD int32_t moe_unit_cost(int routed_rows, bool tc) {
  return tc ? kTcUnitBase + (routed_rows + 15) / 16 : (routed_rows > 4 ? routed_rows : 4);
}

// first unit of block j of N, with F units per expert; cum[a] = cost of the units of experts
// 0..a-1 (cum[nact] = C, at most 256 experts x 1024 units x 64 = 2^24), cost[a] = cost of one
// unit of expert a.  With 0 < j < N <= 256, C * j < 2^32: the arithmetic stays in 32 bits.
// The cost prefix of F units per expert also serves nb units per expert when scaled by nb / F
// (cum[a] is a multiple of F): scale = {nb, F}, {1, 1} for the prefix as it is.
template <class I>
MK_HD int32_t moe_gu_start(int j, int N, const I* cum, const I* cost, int nact, int F, int sn = 1, int sd = 1) {
  if (j <= 0 || nact <= 0) return 0;
  if (j >= N) return nact * F;
  const uint32_t T = static_cast<uint32_t>(cum[nact] / sd * sn) * static_cast<uint32_t>(j) / static_cast<uint32_t>(N);
  int lo = 0, hi = nact - 1;   // last a with cum[a] <= T
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<uint32_t>(cum[mid] / sd * sn) <= T) lo = mid; else hi = mid - 1;
  }
  const uint32_t c = static_cast<uint32_t>(cost[lo]);
  const uint32_t f = (T - static_cast<uint32_t>(cum[lo] / sd * sn) + c - 1u) / c;
  return f >= static_cast<uint32_t>(F) ? (lo + 1) * F : lo * F + static_cast<int32_t>(f);
}

// ---- step flags ------------------------------------------------------------------
// The only words of the step that are not tagged data: the abort flag (set by the block that
// records an error, polled by every wait) and the count of blocks that have finished (the
// last one clears both for the next step and merges the greedy selection).
enum : uint32_t { F_FINISH = 1, F_ABORT = 2, kStepFlags = 8 };

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
  const uint16_t* w_down_t;   // [E][F][H] copy of w_down (small-batch MoE path), or null
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
  int32_t B, max_batch, n_ctas, max_items;
  // static plan
  int32_t n_qkv_tiles, n_o_tiles, n_router_tiles;
  int32_t tc;                   // this step runs the dense GEMV tiles on tcgen05 (wide batch)
  const uint64_t* wmaps;        // [4L + 1][16] TMA descriptors of the weights (box 64 x 16, 128-byte swizzle)
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
  uint16_t* kv;           // the KV pool (bf16 elements, or the bytes of the q8_0 layout)
  int32_t kv_q8;          // the pool holds q8_0 blocks (MK_FLAG_KV_Q8)
  uint64_t kv_layer_bytes; // q8_0: bytes of one layer (codes, then scales)
  uint64_t kv_code_bytes;  // q8_0: bytes of one layer's code plane
  float* logits;
  // per-step plan (device copy of the host-built step buffer)
  const int32_t* seq_lens;      // [B]
  const float* rope_cos;        // [B][D/2]
  const float* rope_sin;        // [B][D/2]
  const mk_attn_item* items;    // [n_items]
  const int32_t* item_off;      // [n_ctas + 1]
  const int32_t* pair_first;    // [B * Hkv] first item of each (row, kv head)
  // workspace.  Every value one block writes and another reads is a tagged 8-byte word:
  // the fp32 (or int32) value in the low half and the step's tag in the high half, written
  // with one 64-bit store.  A reader that sees the current tag has the value of this step;
  // no fence is needed between writer and reader.
  const uint32_t* step_tag;  // this step's tag (never 0), in the uploaded step data so that a
                             // replayed launch of a captured graph reads a fresh one
  int32_t stall_layer; // test hook: the O-proj of this layer waits for a tag that never comes (-1: off)
  uint64_t* X;     // [2L+1][max_batch][H] residual stream: layer input at 2l, after attention at 2l+1
  uint64_t* QKV;   // [L][max_batch][nqkv]
  uint64_t* ATT;   // [L][max_batch][Hq*D]
  uint64_t* PO;    // [L][max_items][G][D]   attention split partial outputs
  uint64_t* PML;   // [L][max_items][G][2]   their (max, sum)
  uint64_t* RLOG;  // [L][max_batch][E] router logits (+ bias)
  uint64_t* HB;    // [L][max_batch][K][F] SwiGLU activations per (row, slot)
  uint64_t* YD;    // [L][max_batch][K][H] weighted down-projection output per (row, slot) (wide batches)
  uint64_t* PSK;   // [L][3][n_ctas][psk_cap] split-K partial sums of the QKV, O-proj, router tiles (wide)
  uint64_t* PSQ;   // [L][3][n_ctas][max_batch] their blocks' partial sums of squares of the input rows
  int32_t psk_cap; // words of one block's partial: its group's rows x max_batch
  int32_t small_moe;    // this step runs the small-batch MoE path
  uint64_t* PT;         // [L][n_ctas][kSmallMaxB][H] per-block partial MoE outputs (small-batch path)
  int32_t* next_token;  // greedy selection: [B] argmax of the logits, or null (not requested)
  float* margin;        // [B] top-1 minus top-2 logit, or null
  float* argp;          // [n_ctas][max_batch][4] per-block (max, second, index bits) of its LM-head rows
  int32_t* RIDS;   // [L][max_batch][K] routing ids (copy kept by block 0 for inspection)
  float* RW;       // [L][max_batch][K] combine weights (same)
  uint32_t* flags; // [kStepFlags] abort flag, finish count
  mk_status* status;
  // optional timeline: per block `trace_cap` events of 4 x u64 (start, dependency met, end, tag);
  // event 0 of each block holds (consumer events, kernel start, producer events, 0)
  uint64_t* trace;
  int32_t trace_cap;
};

// trace tags: op | layer << 8 | kind << 24 | (uint64)idx << 32
enum : uint32_t { TR_TILE = 1, TR_ITEM = 2, TR_PRODUCER_ROUTE_WAIT = 3, TR_CHUNK = 4, TR_MARK = 5 };

}  // namespace mk
