/*
 * mk.h -- C ABI of the persistent MoE decode megakernel for GB300 (sm_103a).
 *
 * One call of mk_decode_step runs one decode step of a mixture-of-experts
 * transformer for a batch of sequences as a single persistent kernel: one
 * thread block per SM stays resident for the whole step, walks a task list
 * prepared on the host, and waits only for the data each task reads -- values
 * other SMs wrote as words tagged with the step -- rather than for whole
 * phases ("Inside the megakernel serving engine for North Mini Code", section
 * "What is a Megakernel?" and the "Image 2" paragraph).  The step covers RMSNorm,
 * fused QKV, RoPE, paged GQA decode attention over ragged lengths with block
 * tables, O-proj + residual, router softmax/top-k, SwiGLU experts, the
 * weighted combine, the final norm and the LM head.
 *
 * The calls follow the page's statement of the problem (serving paragraph:
 * "continuous batching, paged attention, and ragged sequence lengths"):
 * every call may use a different batch and different lengths; the caller owns
 * the paged KV cache and its block tables.
 *
 * Conventions
 *   - All weights are bf16, row-major [out, in]; accumulation is fp32.
 *   - Pointers marked "device" are CUDA device pointers of the current device;
 *     "host" pointers are ordinary host memory read during the call.
 *   - Every pointer passed to the library must be 16-byte aligned.
 *   - The library never takes ownership of caller memory.  Weights must stay
 *     valid until mk_destroy; step arguments until the step has completed on
 *     its stream.
 *   - Functions return MK_OK (0) or a negative MK_ERR_* code; mk_last_error()
 *     then gives a text for the calling thread.  Arguments are checked before
 *     anything is launched: out-of-range calls are rejected, never clamped.
 *   - Errors found on the device (a wait that ran out, a page id or token out
 *     of range) cannot be returned by the asynchronous step call; they are
 *     recorded and read with mk_get_status.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_OK 0
#define MK_ERR_INVALID_ARG (-1)   /* bad argument; nothing was launched */
#define MK_ERR_CUDA (-2)          /* a CUDA runtime call failed */
#define MK_ERR_OOM (-3)           /* device or pinned allocation failed */
#define MK_ERR_UNSUPPORTED (-4)   /* not an sm_103 device, no cooperative launch, shape outside the compiled limits */
#define MK_ERR_TIMEOUT (-5)       /* device: a wait exceeded the watchdog budget (mk_get_status) */
#define MK_ERR_DEVICE_BOUNDS (-6) /* device: a token id or block-table page id was out of range (mk_get_status) */

/* CUDA stream handle; ABI-identical to cudaStream_t (NULL = legacy default stream). */
typedef struct CUstream_st* mk_stream_t;

/*
 * Model and cache shape.  All sizes must be > 0.  Limits of this build
 * (mk_create returns MK_ERR_UNSUPPORTED outside them):
 *   head_dim in {64, 128}; num_q_heads % num_kv_heads == 0 with at most 8 query
 *   heads per KV head; hidden, num_q_heads*head_dim and expert_ffn multiples of 8
 *   and <= 4096, expert_ffn <= 1024; num_experts <= 256; top_k <= min(8, num_experts);
 *   page_size*head_dim*2 <= 34816 bytes, page_size a multiple of 8; max_batch <= 64;
 *   max_batch*(top_k+1)*ceil(hidden/SMs) <= 12288; max_batch*num_experts <= 12288.
 */
/*
 * mk_config.flags.  By default mk_create keeps a transposed device copy of every layer's
 * w_down ([num_experts, expert_ffn, hidden], num_layers*num_experts*expert_ffn*hidden*2 bytes)
 * so that steps of 1-2 rows run each expert's gate/up and down rows together on one SM
 * (no exchange of SwiGLU activations between SMs).  MK_FLAG_NO_DOWN_COPY skips the copy;
 * every batch then takes the general MoE path.  Results agree within rounding either way.
 */
#define MK_FLAG_NO_DOWN_COPY 1
/*
 * MK_FLAG_KV_Q8: the KV pool holds q8_0 blocks instead of bf16 ("Kinetic" pages: a quantized
 * cache keeps keys and values as blocks of 32 int8 values with one f16 scale, 34 bytes where
 * bf16 takes 64; outputs are close to, not equal to, the bf16 cache's).  Layout, per layer,
 * one layer after the other (layer_bytes = num_pages*2*Hkv*page_size*head_dim*17/16):
 *   int8 codes   [num_pages][2 (K,V)][Hkv][page_size][head_dim]
 *   f16 scales   [num_pages][2 (K,V)][Hkv][page_size][head_dim/32]
 * A cached value is code * scale.  The step quantizes this token's k (after RoPE) and v from
 * their fp32 values: per block of 32, scale = max|x|/127 (stored rounded to f16), code =
 * x*(1/scale) rounded to nearest, ties away from zero.  Requires head_dim 128.
 */
#define MK_FLAG_KV_Q8 2

typedef struct mk_config {
  int32_t num_layers;
  int32_t hidden;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t num_experts;
  int32_t top_k;
  int32_t expert_ffn;
  int32_t vocab;
  float rope_theta;          /* RoPE base; angles pos*theta^(-2i/D) are evaluated in fp64 on the host */
  float rms_eps;             /* RMSNorm epsilon */
  int32_t page_size;         /* tokens per KV page */
  int32_t num_pages;         /* pages per layer in the caller's KV pool */
  int32_t max_batch;         /* largest batch a step may use */
  int32_t max_pages_per_seq; /* row length of the block table */
  int32_t norm_topk;         /* 1: router weights renormalised over the k chosen experts; 0: raw softmax probs */
  int32_t flags;             /* 0 or MK_FLAG_NO_DOWN_COPY | MK_FLAG_KV_Q8 */
  uint32_t watchdog_ms;      /* per-wait device budget in ms; 0 selects the default (1000 ms) */
} mk_config;

/* One layer's weights (device pointers, bf16 unless noted).  Borrowed. */
typedef struct mk_layer_weights {
  const void* attn_norm;    /* [hidden] RMSNorm gain before attention */
  const void* w_qkv;        /* [(Hq + 2*Hkv)*D, hidden]: rows are q heads, then k heads, then v heads */
  const void* w_o;          /* [hidden, Hq*D] */
  const void* ffn_norm;     /* [hidden] RMSNorm gain before the MoE block */
  const void* w_router;     /* [num_experts, hidden] */
  const float* router_bias; /* [num_experts] fp32 added to the router logits, or NULL */
  const void* w_gate_up;    /* [num_experts, 2*expert_ffn, hidden]: gate rows, then up rows */
  const void* w_down;       /* [num_experts, hidden, expert_ffn] */
} mk_layer_weights;

typedef struct mk_weights {
  const void* embed;              /* [vocab, hidden] */
  const void* final_norm;         /* [hidden] */
  const void* lm_head;            /* [vocab, hidden] (untied from embed) */
  const mk_layer_weights* layers; /* host array [num_layers]; copied by mk_create */
} mk_weights;

/* What a wait that ran out was waiting for (mk_status.wait). */
#define MK_WAIT_DATA 1   /* words another SM writes (they did not carry the step's tag in time) */
#define MK_WAIT_RING 2   /* a shared-memory ring slot of the SM (its copy did not land, or was not released) */
#define MK_WAIT_ROUTE 3  /* the SM's own routing of the layer, which its expert stream waits for */

/* Device-side error record of the last failing step (see mk_get_status). */
typedef struct mk_status {
  int32_t code;      /* MK_OK, MK_ERR_TIMEOUT or MK_ERR_DEVICE_BOUNDS */
  int32_t op;        /* task kind that failed (1 embed, 2 qkv, 3 attention, 4 o-proj, 5 router, 6 moe, 7 head; 0 ring) */
  int32_t layer;     /* its layer, or -1 */
  int32_t cta;       /* thread block that recorded the error */
  uint32_t wait;     /* timeout: MK_WAIT_*; bounds error: 0 */
  uint32_t observed; /* timeout on the ring: the record index; bounds error: the bad token or page id */
  uint32_t tag;      /* timeout on data: the step tag the words had to carry */
  int32_t detail;    /* row / page slot involved, or -1 */
} mk_status;

typedef struct mk_ctx mk_ctx;

/*
 * Create a context on the current CUDA device.
 *   cfg, weights: host structs, read during the call; weight tensors are device
 *                 pointers that must outlive the context.
 *   out:          receives the new context.
 * Allocates the library's workspace (per-layer tagged activations, step flags,
 * task lists, pinned staging) and, unless cfg->flags has MK_FLAG_NO_DOWN_COPY, the
 * transposed copy of the down projections, filled on the device before return.  Errors: MK_ERR_INVALID_ARG (null or non-positive or
 * misaligned argument), MK_ERR_UNSUPPORTED (device or shape outside the
 * build's limits), MK_ERR_OOM, MK_ERR_CUDA.
 */
int mk_create(const mk_config* cfg, const mk_weights* weights, mk_ctx** out);

/*
 * Enqueue one decode step on `stream` and return without waiting.
 *   batch:        number of rows, 1..max_batch.
 *   token_ids:    device int32 [batch], the token decoded by each row.
 *   seq_lens:     HOST int32 [batch], each row's length including this token
 *                 (its position is seq_len-1), 1..max_pages_per_seq*page_size.
 *                 The host splits attention work from these lengths.
 *   block_tables: device int32 [batch, max_pages_per_seq]; entry p of row b is
 *                 the pool page holding positions p*page_size..; entries past
 *                 ceil(seq_len/page_size) are not read.
 *   kv_pages:     device bf16 [num_layers][num_pages][2 (K,V)][num_kv_heads]
 *                 [page_size][head_dim] (or the q8_0 layout of MK_FLAG_KV_Q8).
 *                 K is stored after RoPE.  The step writes this token's K and V
 *                 at position seq_len-1 of every layer and reads positions
 *                 0..seq_len-2.
 *   logits_out:   device fp32 [batch, vocab].
 * Re-running a step with the same arguments is idempotent.  Steps on one
 * context must not run concurrently (the workspace is shared).
 */
int mk_decode_step(mk_ctx* ctx, int32_t batch, const int32_t* token_ids, const int32_t* seq_lens,
                   const int32_t* block_tables, void* kv_pages, float* logits_out, mk_stream_t stream);

/*
 * mk_decode_step plus greedy selection in the same launch: for every row b,
 *   next_token[b] = the index of the largest logit (the lowest index among equal maxima),
 *   margin[b]     = that logit minus the largest logit at any other index (0 at a tie),
 * both computed on the device from the fp32 logits the step writes to logits_out (so they
 * agree exactly with an argmax of logits_out).  next_token: device int32 [batch];
 * margin: device fp32 [batch], or NULL.  Each SM reduces its own LM-head rows; the last SM
 * to finish merges the SMs' (max, index, second) per row.  Other arguments, ownership and
 * errors as mk_decode_step (MK_ERR_INVALID_ARG also for a NULL or misaligned next_token).
 */
int mk_decode_step_greedy(mk_ctx* ctx, int32_t batch, const int32_t* token_ids, const int32_t* seq_lens,
                          const int32_t* block_tables, void* kv_pages, float* logits_out, int32_t* next_token,
                          float* margin, mk_stream_t stream);

/*
 * A decode step captured as a CUDA graph, for callers that decode the same batch shape many
 * times: the host builds step n+1's data (tag, lengths, RoPE rows, attention split plan) into
 * one of two pinned staging buffers while step n runs, and the launch is one graph replay
 * (an upload node and the step kernel).  The plan's NEXT-2 ("Image 2" paragraph: the host
 * schedules the step; per-step task counts follow the live lengths).
 *   mk_graph_create: capture a step of `batch` rows over fixed device buffers token_ids,
 *     block_tables, kv_pages and logits_out (meaning and layout as mk_decode_step).  Their
 *     CONTENTS may change between launches; their addresses may not.  Captures on a private
 *     stream; allocates two pinned and two device staging buffers and two graphs.  Errors:
 *     MK_ERR_INVALID_ARG, MK_ERR_CUDA (e.g. a driver that cannot capture the launch), MK_ERR_OOM.
 *   mk_graph_launch: this step's seq_lens (HOST int32 [batch], as mk_decode_step) and one
 *     replay on `stream` (not the legacy default stream while another stream captures);
 *     asynchronous; device errors through mk_get_status.  Steps of one context, captured or not,
 *     must not overlap on the GPU.
 *   mk_graph_destroy: waits for the graph's launches and frees it (NULL is ignored); the
 *     context stays valid.
 */
typedef struct mk_graph mk_graph;
int mk_graph_create(mk_ctx* ctx, int32_t batch, const int32_t* token_ids, const int32_t* block_tables, void* kv_pages,
                    float* logits_out, mk_graph** out);
int mk_graph_launch(mk_graph* graph, const int32_t* seq_lens, mk_stream_t stream);
void mk_graph_destroy(mk_graph* graph);

/*
 * Wait for the last enqueued step and report device-side errors.  Fills `out`
 * and returns out->code (MK_OK when the step ran clean).  Reading clears the
 * record.  After an error the context stays usable.
 */
int mk_get_status(mk_ctx* ctx, mk_status* out);

/* Text of the last error of the calling thread ("" if none).  Valid until the thread's next call. */
const char* mk_last_error(void);

/* Free everything the library allocated.  NULL is ignored.  Does not touch caller memory. */
void mk_destroy(mk_ctx* ctx);

/*
 * Paged GQA decode attention with no device allocation (the paper has no
 * counterpart; it serves callers that cannot call cudaMalloc -- code running
 * under another framework's allocator or memory-pool hooks, or a plug-in that
 * is only handed pre-allocated buffers -- and therefore cannot create a
 * context).  It computes, for every row b and query head h, the softmax
 * attention of q[b][h] (already rotated; it is scaled by 1/sqrt(head_dim)
 * here) over positions 0..seq_len[b]-1 of the row's pages, exactly the
 * attention of one layer of mk_decode_step, and writes out[b][h*head_dim + d].
 *   q:            device fp32 [batch][num_q_heads][head_dim]
 *   seq_lens:     HOST int32 [batch], 1..max_pages_per_seq*page_size
 *   block_tables: device int32 [batch][max_pages_per_seq]
 *   kv_layer:     device bf16 pages of ONE layer: [num_pages][2 (K,V)][num_kv_heads][page_size][head_dim]
 *   out:          device fp32 [batch][num_q_heads*head_dim]
 *   status_out:   device int32 [1] or NULL; receives MK_OK, or MK_ERR_DEVICE_BOUNDS if a
 *                 block-table entry was outside 0..num_pages-1.  Such pages are skipped (never
 *                 read): the row attends over its other positions, and a row none of whose
 *                 pages is in range gets zeros in out.  status_out is the only report of a bad
 *                 entry; with status_out NULL the call still returns MK_OK.
 * Limits: batch <= 64, head_dim 64 or 128, at most 8 query heads per KV head,
 * max_pages_per_seq*page_size <= 2^30 (MK_ERR_UNSUPPORTED beyond).
 * Its only scratch is one fixed 4 MiB __device__ array inside the library,
 * which every GPU that loads the library keeps until the process exits:
 * batch * num_kv_heads * (num_q_heads/num_kv_heads) * (head_dim+2) * 4 bytes
 * must fit in it (about 4 MiB), otherwise the call returns MK_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Asynchronous on `stream`; allocates nothing.  Every call uses the
 * same array, so calls whose work overlaps on the GPU (other streams, other
 * threads) race and must be serialised by the caller.
 */
int mk_paged_attention_noalloc(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t page_size, int32_t num_pages, int32_t max_pages_per_seq, const float* q,
                               const int32_t* seq_lens, const int32_t* block_tables, const void* kv_layer,
                               float* out, int32_t* status_out, mk_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MK_H */
