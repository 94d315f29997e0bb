/*
 * mk_debug.h -- host-side planning, simulation and inspection entry points of
 * the megakernel library.  Nothing here is needed to run a decode step; these
 * calls exist so that the scheduler can be tested without a GPU and so that
 * intermediate results of a step can be compared with a reference.
 *
 * Scheduling model ("Inside the megakernel serving engine for North Mini
 * Code", section "What is a Megakernel?" and the "Image 2" paragraph): the
 * host splits the step into tasks of one tile of one operation each and deals
 * them over the SMs, one task list per SM in global memory.  A task needs only
 * the data it reads: every value one SM hands to another is a tagged word (the
 * value and the step's tag), and the reading SM polls exactly the words it
 * needs until they carry this step's tag.  Attention and MoE work depend on
 * live lengths and on routing: the attention split plan is rebuilt on the host
 * every step from the host-side seq_lens, and every SM routes the batch itself
 * from the router logits and takes a cost-balanced share of the MoE work.
 */
#ifndef MK_DEBUG_H
#define MK_DEBUG_H

#include "mk.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Task kinds (mk_task.op) and the data each one waits for. */
#define MK_OP_EMBED 1  /* copy embedding rows into the residual stream (a column range of every row); no wait */
#define MK_OP_QKV 2    /* RMSNorm + fused QKV GEMV, a range of output rows; waits for the whole layer input */
#define MK_OP_ATTN 3   /* this SM's attention split items of the layer (from the per-step plan); each item waits
                          for q, k, v of its (row, KV head); after its last item the SM merges a slice of every
                          pair it holds a split of, waiting for all of that pair's split partials */
#define MK_OP_OPROJ 4  /* O-proj GEMV + residual, a range of output rows; waits for the whole attention output */
#define MK_OP_ROUTER 5 /* RMSNorm + router GEMV, a range of experts; waits for the whole post-attention residual */
#define MK_OP_MOE 6    /* route the batch from all router logits (every SM), then this SM's share of the
                          experts; the down projection's combine waits for every SM's share */
#define MK_OP_HEAD 7   /* final RMSNorm + LM head GEMV, a range of vocab rows; waits for the last layer's output */
#define MK_OP_END 8    /* end of this SM's list */

/* One task of an SM's list (16 bytes): an operation, its layer and its row range. */
typedef struct mk_task {
  uint16_t op;
  uint16_t layer;
  uint32_t lo, hi; /* row (or column) range [lo, hi) */
  uint32_t reserved;
} mk_task;

/* One attention split item (16 bytes): row b, KV head kvh, the block-table
 * entries [page_lo, page_hi) of that row; split index and the number of splits
 * of (b, kvh).  Items of one (b, kvh) are consecutive in the plan. */
typedef struct mk_attn_item {
  uint16_t b, kvh, split, nsplit;
  uint32_t page_lo, page_hi;
} mk_attn_item;

/* Sizes of the static plan for a shape and a number of SMs. */
typedef struct mk_plan_info {
  int32_t n_ctas;
  int32_t n_tasks;        /* total tasks over all lists */
  int32_t n_qkv_tiles, n_o_tiles, n_router_tiles, n_head_tiles, n_embed_tiles;
  int32_t n_down_ranges;    /* blocks that own hidden rows of the down projection */
  int32_t reserved[3];
  int32_t n_flags;          /* words of step flags (abort flag, finish count); all other exchange is tagged data */
  int32_t max_items;        /* attention items a step can produce for max_batch */
} mk_plan_info;

/* Static task lists for `n_ctas` SMs.  Fills `info`; if `tasks` is non-NULL it
 * receives info->n_tasks tasks and `cta_offsets` ([n_ctas+1]) the start of
 * each SM's list.  Host only; no GPU needed. */
int mk_plan_static(const mk_config* cfg, int32_t n_ctas, mk_plan_info* info, mk_task* tasks, int32_t* cta_offsets);

/* Attention split plan of one step (host only).  seq_lens: host [batch].
 * Writes at most `max_items` items and `cta_offsets` ([n_ctas+1]); returns the
 * item count through n_items. */
int mk_plan_attention(const mk_config* cfg, int32_t n_ctas, int32_t batch, const int32_t* seq_lens,
                      mk_attn_item* items, int32_t max_items, int32_t* cta_offsets, int32_t* n_items);

/* Result of mk_simulate. */
typedef struct mk_sim_result {
  int32_t finished;        /* 1 if every list reached its end */
  int32_t deadlocked;      /* 1 if no SM could make progress before the end */
  int64_t events;          /* scheduling events simulated */
  int32_t tiles_run[9];    /* tiles / items executed, indexed by op */
  int32_t writes_ok;       /* 1 if every tile that writes data another SM reads ran exactly once */
  int32_t moe_units_ok;    /* 1 if every gate/up unit and every (expert, hidden row) of the down
                              projection was assigned to exactly one block */
} mk_sim_result;

/* Run the step's task graph on the CPU with `n_ctas` virtual SMs under a seeded
 * random interleaving.  Each virtual SM has a producer that runs at most
 * `producer_lead` records ahead of its consumer (routing is handed from the
 * consumer to its own producer before the MoE records exist, and the MoE work
 * is split with the same rule as the device) and a consumer whose every record
 * waits for exactly the writer tiles of the data the device reads there: an
 * attention item for the QKV tiles holding its (row, KV head)'s q, k and v,
 * the split merge for all splits of its pairs, O-proj for every merge slice
 * and its own residual rows, a router tile for every O-proj tile, routing for
 * every router tile, the MoE combine for every SM's share, QKV and the LM head
 * for every writer of their input.
 * routing_ids: host [num_layers][batch][top_k] expert ids the router is taken to
 * choose. */
int mk_simulate(const mk_config* cfg, int32_t n_ctas, int32_t batch, const int32_t* seq_lens,
                const int32_t* routing_ids, uint64_t seed, int32_t producer_lead, mk_sim_result* out);

/* Intermediate buffers of the last step, for per-operation checks. */
#define MK_DBG_X 1           /* fp32 [2L+1][batch][hidden]: layer l input at 2l, after attention at 2l+1 */
#define MK_DBG_QKV 2         /* fp32 [batch][(Hq+2Hkv)D] of `layer`, before RoPE */
#define MK_DBG_ATTN 3        /* fp32 [batch][Hq*D] attention output of `layer` */
#define MK_DBG_ROUTER 4      /* fp32 [batch][E] router logits (+bias) of `layer` */
#define MK_DBG_ROUTE_IDS 5   /* int32 [batch][k] chosen experts of `layer`, rank order */
#define MK_DBG_ROUTE_W 6     /* fp32 [batch][k] their combine weights */
#define MK_DBG_H 7           /* fp32 [batch][k][F] SwiGLU activations of `layer` */

/* Copy an intermediate of the last completed step of `layer` into host memory.
 * Synchronises the device.  `bytes` must equal the buffer size for the last
 * step's batch. */
int mk_debug_read(mk_ctx* ctx, int32_t what, int32_t layer, void* host_dst, size_t bytes);

/* Test hook: the O-proj tasks of `layer` in the next step wait for a tag that
 * no SM writes, so the watchdog must end the step with MK_ERR_TIMEOUT after
 * `watchdog_ms` (0 keeps the context's budget).  layer < 0 disarms. */
int mk_debug_inject_stall(mk_ctx* ctx, int32_t layer, uint32_t watchdog_ms);

/* Timeline of later steps.  enable != 0 allocates a device buffer of
 * n_ctas * events_per_cta events (4 x uint64 each: time the tile's first
 * operand landed, time its dependency was met, time it finished, tag =
 * op | layer<<8 | kind<<24 | index<<32; globaltimer ns) and records every
 * later step into it (each step overwrites the previous one); enable == 0
 * frees it.  Event 0 of each block is a header (consumer events, kernel start,
 * producer events); producer events fill the block's area from its end. */
int mk_debug_trace(mk_ctx* ctx, int32_t enable, int32_t events_per_cta);

/* Copy the timeline of the last step to host memory (synchronises). */
int mk_debug_trace_read(mk_ctx* ctx, void* host_dst, size_t bytes);

/* Number of SMs (persistent thread blocks) a step of this context launches. */
int mk_num_ctas(mk_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* MK_DEBUG_H */
