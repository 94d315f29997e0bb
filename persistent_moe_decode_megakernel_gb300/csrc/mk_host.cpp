// mk_host.cpp -- host side of the megakernel library: argument checks, the
// static task lists, the per-step attention split plan, the workspace, the
// cooperative launch, status readback, debug reads and a CPU simulator of the
// step's data dependencies.
//
// Scheduling follows "Inside the megakernel serving engine for North Mini
// Code" ("Image 2" paragraph): the step is split into tasks of one tile of one
// operation, dealt over the SMs, one list per SM in global memory; attention
// and MoE work depend on live lengths and routing.  Here the static lists (all
// GEMV tiles, one attention task and one MoE task per layer) are built once per
// context; the attention split plan is rebuilt on the host each step from the
// host-side lengths; the MoE work is split on the device by every SM from its
// own routing of the batch.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <queue>
#include <random>
#include <string>
#include <queue>
#include <vector>

#include "mk.h"
#include "mk_debug.h"
#include "mk_layout.h"

namespace mk {
cudaError_t launch_step(const Params& p, cudaStream_t s);
int tb_for_batch(int B);
cudaError_t transpose_down(const uint16_t* in, uint16_t* out, int E, int H, int F, cudaStream_t s);
cudaError_t configure_kernels(int D, bool kv_q8);
cudaError_t occupancy(int D, bool kv_q8, int* blocks);
size_t smem_bytes();
}  // namespace mk

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? MK_ERR_OOM : MK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace mk {
// lets other translation units of the library set the text mk_last_error() returns
void set_last_error(int, const char* text) { g_err = text; }
}  // namespace mk

namespace {

// ---------------------------------------------------------------- config checks
int check_config(const mk_config* c) {
  if (!c) return fail(MK_ERR_INVALID_ARG, "config is NULL");
  const struct { const char* n; int32_t v; } pos[] = {
      {"num_layers", c->num_layers}, {"hidden", c->hidden}, {"num_q_heads", c->num_q_heads},
      {"num_kv_heads", c->num_kv_heads}, {"head_dim", c->head_dim}, {"num_experts", c->num_experts},
      {"top_k", c->top_k}, {"expert_ffn", c->expert_ffn}, {"vocab", c->vocab}, {"page_size", c->page_size},
      {"num_pages", c->num_pages}, {"max_batch", c->max_batch}, {"max_pages_per_seq", c->max_pages_per_seq}};
  for (const auto& f : pos)
    if (f.v <= 0) return fail(MK_ERR_INVALID_ARG, "config.%s must be > 0 (got %d)", f.n, f.v);
  if (!(c->rope_theta > 0.f) || !(c->rms_eps >= 0.f)) return fail(MK_ERR_INVALID_ARG, "rope_theta must be > 0, rms_eps >= 0");
  if (c->norm_topk != 0 && c->norm_topk != 1) return fail(MK_ERR_INVALID_ARG, "norm_topk must be 0 or 1");
  if (c->flags & ~(MK_FLAG_NO_DOWN_COPY | MK_FLAG_KV_Q8)) return fail(MK_ERR_INVALID_ARG, "unknown bits in flags");
  if (c->num_q_heads % c->num_kv_heads) return fail(MK_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  if (c->top_k > c->num_experts) return fail(MK_ERR_INVALID_ARG, "top_k > num_experts");
  // limits of this build
  if (c->head_dim != 64 && c->head_dim != 128) return fail(MK_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c->num_q_heads / c->num_kv_heads > mk::kMaxG) return fail(MK_ERR_UNSUPPORTED, "more than 8 query heads per KV head");
  const int32_t ks[3] = {c->hidden, c->num_q_heads * c->head_dim, c->expert_ffn};
  for (int32_t k : ks)
    if (k % 8 || k > mk::kMaxK) return fail(MK_ERR_UNSUPPORTED, "GEMV input lengths must be multiples of 8 and <= 4096");
  if (c->num_experts > mk::kMaxExperts) return fail(MK_ERR_UNSUPPORTED, "num_experts > 256");
  if (c->expert_ffn > 1024) return fail(MK_ERR_UNSUPPORTED, "expert_ffn > 1024");
  if (c->top_k > mk::kMaxTopK) return fail(MK_ERR_UNSUPPORTED, "top_k > 8");
  if (c->page_size * c->head_dim * 2 > mk::kSlotBytes / 2)
    return fail(MK_ERR_UNSUPPORTED, "page_size*head_dim*2 > %d", mk::kSlotBytes / 2);
  if (!(c->flags & MK_FLAG_KV_Q8) && mk::pages_per_chunk(c->page_size, c->head_dim) < 1)
    return fail(MK_ERR_UNSUPPORTED, "page_size %d: no whole 16-row tiles of KV pages fit one ring slot", c->page_size);
  if (c->page_size % 8) return fail(MK_ERR_UNSUPPORTED, "page_size must be a multiple of 8");
  if ((c->flags & MK_FLAG_KV_Q8) && c->head_dim != 128)
    return fail(MK_ERR_UNSUPPORTED, "the q8_0 KV cache needs head_dim 128");
  if ((c->flags & MK_FLAG_KV_Q8) && mk::pages_per_chunk_q8(c->page_size, c->head_dim) < 1)
    return fail(MK_ERR_UNSUPPORTED, "a q8_0 page does not fit one ring slot");
  if ((int64_t)c->num_layers * c->num_pages * 2 * c->num_kv_heads * c->page_size >= ((int64_t)1 << 31))
    return fail(MK_ERR_UNSUPPORTED, "KV pool has 2^31 or more rows");
  if (c->max_batch > mk::kMaxBatch) return fail(MK_ERR_UNSUPPORTED, "max_batch > 64");
  if ((int64_t)c->max_pages_per_seq * c->page_size > (int64_t)1 << 30) return fail(MK_ERR_UNSUPPORTED, "sequence too long");
  return MK_OK;
}

// Whether a context on n_ctas SMs can run the small-batch MoE path at all: the SwiGLU
// outputs of one block's gate/up units stay on chip (with at most kSmallMaxB rows every
// unit costs the same, so a block gets at most units/n_ctas + 2 of them), and the partial
// outputs of every block for the block's own hidden rows fit the reduction scratch.
bool small_moe_fits(const mk_config& c, int n_ctas) {
  if (c.flags & MK_FLAG_NO_DOWN_COPY) return false;
  const int64_t act = std::min<int64_t>(c.num_experts, (int64_t)mk::kSmallMaxB * c.top_k);
  if (act * c.expert_ffn / n_ctas + 2 > mk::kMaxUnits) return false;
  const int64_t nr = (c.hidden + n_ctas - 1) / n_ctas;
  return (int64_t)mk::kSmallMaxB * n_ctas * nr <= mk::kMoeScratch;
}

// the MoE path of one step: small-batch when the context has the transposed down copy and
// the batch's MoE input fits the on-chip input cache
bool small_moe_step(const mk_config& c, int n_ctas, int B) {
  return small_moe_fits(c, n_ctas) && mk::small_moe_batch(B, c.hidden);
}

// ---------------------------------------------------------------- static plan
struct Plan {
  std::vector<mk_task> tasks;
  std::vector<int32_t> off;
  mk_plan_info info;
};

void split_range(uint32_t n, int parts, int i, uint32_t* lo, uint32_t* hi) {
  *lo = (uint32_t)((uint64_t)n * i / parts);
  *hi = (uint32_t)((uint64_t)n * (i + 1) / parts);
}

void build_static_plan(const mk_config& c, int n_ctas, Plan& plan) {
  mk_plan_info& in = plan.info;
  std::memset(&in, 0, sizeof in);
  const int L = c.num_layers, H = c.hidden, E = c.num_experts, V = c.vocab;
  const int nqkv = (c.num_q_heads + 2 * c.num_kv_heads) * c.head_dim;
  in.n_ctas = n_ctas;
  in.n_flags = (int32_t)mk::kStepFlags;
  in.max_items = n_ctas + c.max_batch * c.num_kv_heads;
  auto count = [&](uint32_t rows) {
    int n = 0;
    for (int i = 0; i < n_ctas; ++i) {
      uint32_t lo, hi;
      split_range(rows, n_ctas, i, &lo, &hi);
      n += hi > lo;
    }
    return n;
  };
  in.n_embed_tiles = count((uint32_t)H);
  in.n_qkv_tiles = count((uint32_t)nqkv);
  in.n_o_tiles = count((uint32_t)H);
  const int rr = mk::router_tile_rows(E, n_ctas, c.max_batch);
  in.n_router_tiles = (E + rr - 1) / rr;
  in.n_head_tiles = count((uint32_t)V);
  in.n_down_ranges = count((uint32_t)H);
  plan.tasks.clear();
  plan.off.assign(n_ctas + 1, 0);
  auto push = [&](uint16_t op, int layer, uint32_t lo, uint32_t hi) {
    mk_task t;
    t.op = op; t.layer = (uint16_t)layer; t.lo = lo; t.hi = hi; t.reserved = 0;
    plan.tasks.push_back(t);
  };
  // Every list runs the layers in order and, within a layer, the phases in data order; a
  // task waits on the device for exactly the tagged words it reads (see mk_debug.h).
  for (int i = 0; i < n_ctas; ++i) {
    plan.off[i] = (int32_t)plan.tasks.size();
    uint32_t lo, hi;
    split_range((uint32_t)H, n_ctas, i, &lo, &hi);
    if (hi > lo) push(MK_OP_EMBED, 0, lo, hi);
    for (int l = 0; l < L; ++l) {
      split_range((uint32_t)nqkv, n_ctas, i, &lo, &hi);
      if (hi > lo) push(MK_OP_QKV, l, lo, hi);
      push(MK_OP_ATTN, l, 0, 0);
      split_range((uint32_t)H, n_ctas, i, &lo, &hi);
      if (hi > lo) push(MK_OP_OPROJ, l, lo, hi);
      for (int t = i; t < in.n_router_tiles; t += n_ctas)
        push(MK_OP_ROUTER, l, (uint32_t)(t * rr), (uint32_t)std::min(E, (t + 1) * rr));
      push(MK_OP_MOE, l, 0, 0);
    }
    split_range((uint32_t)V, n_ctas, i, &lo, &hi);
    if (hi > lo) push(MK_OP_HEAD, L, lo, hi);
    push(MK_OP_END, 0, 0, 0);
  }
  plan.off[n_ctas] = (int32_t)plan.tasks.size();
  in.n_tasks = (int32_t)plan.tasks.size();
}

// ---------------------------------------------------------------- per-step attention plan
// Pages of every (row, KV head) pair are dealt over the SMs in order, each SM
// taking an equal share of pages; a pair cut at an SM boundary becomes several
// splits whose partial softmax states the last one merges.
int build_attention_plan(const mk_config& c, int n_ctas, int B, const int32_t* seq_lens, std::vector<mk_attn_item>& items,
                         std::vector<int32_t>& off, std::vector<int32_t>& pair_first) {
  const int Hkv = c.num_kv_heads, ps = c.page_size;
  int64_t total = 0;
  for (int b = 0; b < B; ++b) total += (int64_t)Hkv * ((seq_lens[b] + ps - 1) / ps);
  items.clear();
  std::vector<int32_t> cta_of;
  pair_first.assign((size_t)B * Hkv, 0);
  const int npairs = B * Hkv;
  if (npairs <= n_ctas) {
    // one item per block: every (row, KV head) pair gets splits in proportion to its pages
    // (at least one, at most one per page), handed out greedily to the pair whose splits are
    // currently the longest; each pair's pages are then cut into near-equal contiguous ranges
    std::vector<int32_t> ns((size_t)npairs, 1);
    std::vector<int64_t> np((size_t)npairs);
    for (int b = 0; b < B; ++b)
      for (int kvh = 0; kvh < Hkv; ++kvh) np[(size_t)b * Hkv + kvh] = (seq_lens[b] + ps - 1) / ps;
    using E = std::pair<double, int>;
    std::priority_queue<E> pq;
    for (int i = 0; i < npairs; ++i) pq.push(E((double)np[i], i));
    for (int left = n_ctas - npairs; left > 0 && !pq.empty(); --left) {
      const int i = pq.top().second;
      pq.pop();
      if (ns[i] >= np[i]) { ++left; continue; }
      ++ns[i];
      if (ns[i] < np[i]) pq.push(E((double)np[i] / ns[i], i));
    }
    int cta = 0;
    for (int i = 0; i < npairs; ++i) {
      pair_first[i] = (int32_t)items.size();
      for (int k = 0; k < ns[i]; ++k) {
        mk_attn_item it;
        it.b = (uint16_t)(i / Hkv); it.kvh = (uint16_t)(i % Hkv); it.split = (uint16_t)k; it.nsplit = (uint16_t)ns[i];
        it.page_lo = (uint32_t)(np[i] * k / ns[i]);
        it.page_hi = (uint32_t)(np[i] * (k + 1) / ns[i]);
        items.push_back(it);
        cta_of.push_back(cta++);
      }
    }
    off.assign(n_ctas + 1, 0);
    for (size_t i = 0; i < items.size(); ++i) off[cta_of[i] + 1]++;
    for (int i = 0; i < n_ctas; ++i) off[i + 1] += off[i];
    return MK_OK;
  }
  const int64_t quota = std::max<int64_t>(1, (total + n_ctas - 1) / n_ctas);
  int cta = 0;
  int64_t room = quota;
  for (int b = 0; b < B; ++b) {
    const uint32_t np = (uint32_t)((seq_lens[b] + ps - 1) / ps);
    for (int kvh = 0; kvh < Hkv; ++kvh) {
      const size_t first = items.size();
      pair_first[(size_t)b * Hkv + kvh] = (int32_t)first;
      uint32_t lo = 0;
      uint16_t split = 0;
      while (lo < np) {
        const uint32_t take = (uint32_t)std::min<int64_t>(room, np - lo);
        mk_attn_item it;
        it.b = (uint16_t)b; it.kvh = (uint16_t)kvh; it.split = split++; it.nsplit = 0;
        it.page_lo = lo; it.page_hi = lo + take;
        items.push_back(it);
        cta_of.push_back(cta);
        lo += take;
        room -= take;
        if (room == 0) { ++cta; room = quota; }
      }
      for (size_t i = first; i < items.size(); ++i) items[i].nsplit = split;
    }
  }
  off.assign(n_ctas + 1, 0);
  for (size_t i = 0; i < items.size(); ++i) off[cta_of[i] + 1]++;
  for (int i = 0; i < n_ctas; ++i) off[i + 1] += off[i];
  return MK_OK;
}

}  // namespace

// ==================================================================== context
struct mk_ctx {
  mk_config cfg;
  int device = 0;
  int n_ctas = 0;
  Plan plan;
  mk::LayerW* d_layers = nullptr;
  mk_task* d_tasks = nullptr;
  int32_t* d_task_off = nullptr;
  const uint16_t* embed = nullptr;
  const uint16_t* final_norm = nullptr;
  const uint16_t* lm_head = nullptr;
  // workspace
  uint8_t* ws = nullptr;
  // tagged 8-byte words (value | step tag << 32)
  uint64_t *X = nullptr, *QKV = nullptr, *ATT = nullptr, *PO = nullptr, *PML = nullptr, *RLOG = nullptr,
           *HB = nullptr, *PT = nullptr, *YD = nullptr, *PSK = nullptr, *PSQ = nullptr;
  int32_t psk_cap = 0;
  uint16_t* wdt = nullptr;   // transposed down projections [L][E][F][H] (small-batch MoE path), or null
  float* argp = nullptr;     // greedy selection: per-block (max, second, index) of its LM-head rows
  bool small_ok = false;
  float* RW = nullptr;
  int32_t* RIDS = nullptr;
  uint32_t tag = 0;        // tag of the last step (0: none yet)
  size_t tagged_bytes = 0; // bytes of the tagged buffers (cleared when the tag wraps)
  uint32_t* flags = nullptr;   // [kStepFlags] abort flag, finish count
  mk_status* d_status = nullptr;
  // per-step staging (double-buffered)
  size_t step_bytes = 0;
  size_t off_tag = 0, off_lens = 0, off_cos = 0, off_sin = 0, off_items = 0, off_item_off = 0, off_pair = 0;
  uint8_t* h_step[2] = {nullptr, nullptr};
  uint8_t* d_step[2] = {nullptr, nullptr};
  cudaEvent_t ev_step[2] = {nullptr, nullptr};
  cudaEvent_t ev_done = nullptr;
  int cur = 0;
  bool stepped = false;
  int last_B = 0;
  std::vector<double> inv_freq;
  // TMA descriptor of the caller's KV pool (re-encoded when the pool pointer changes)
  alignas(64) CUtensorMap kv_map;
  const void* kv_map_ptr = nullptr;
  // TMA descriptors of the weights for wide batches on tcgen05 ([4L + 1] maps), or null
  uint64_t* d_wmaps = nullptr;
  // timeline
  uint64_t* trace = nullptr;
  int32_t trace_cap = 0;
  // test hook
  int stall_layer = -1;
  uint32_t stall_ms = 0;
};

namespace {

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Bytes of one layer of the q8_0 KV pool (code plane, then scale plane), and of its code plane.
size_t kv_q8_code_bytes(const mk_config& cf) {
  return (size_t)cf.num_pages * 2 * cf.num_kv_heads * cf.page_size * cf.head_dim;
}
size_t kv_q8_layer_bytes(const mk_config& cf) { return kv_q8_code_bytes(cf) / 16 * 17; }

// Describe the KV pool to TMA: the bf16 pool [L][P][2][Hkv][ps][D] as 4-D (innermost first)
// {64 dims, Hkv*ps positions, D/64 dim halves, L*P*2 K/V blocks}, positions 2*D bytes apart and
// dim halves 128, so that one box {64, ps, D/64, 2} at position kvh*ps is the K and the V of
// one page and KV head, landing as [K, V][dim half][position][64 dims]: the 8 consecutive
// positions an ldmatrix reads sit on 8 distinct swizzle phases.  (One box per page: a 4-D box
// costs the producer about what one 2-D box does, a 5-D box several times more.)  The q8_0
// pool's code planes as 3-D [layer][row][D bytes],
// rows of one layer contiguous, layers layer_bytes apart (boxes of D bytes x page_size rows).
// Both with the 128-byte swizzle.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

int encode_kv_map(const mk_config& cf, void* kv, CUtensorMap* out) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (cf.flags & MK_FLAG_KV_Q8) {
    const cuuint64_t rows = (cuuint64_t)cf.num_pages * 2 * cf.num_kv_heads * cf.page_size;
    const cuuint64_t dims[3] = {(cuuint64_t)cf.head_dim, rows, (cuuint64_t)cf.num_layers};
    const cuuint64_t strides[2] = {(cuuint64_t)cf.head_dim, (cuuint64_t)kv_q8_layer_bytes(cf)};
    const cuuint32_t box[3] = {(cuuint32_t)cf.head_dim, (cuuint32_t)cf.page_size, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, kv, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled (q8_0 codes) failed (%d)", (int)r);
    return MK_OK;
  }
  const cuuint64_t row = (cuuint64_t)cf.head_dim * 2;   // bytes of one position
  const cuuint64_t dims[4] = {64, (cuuint64_t)cf.page_size * cf.num_kv_heads, (cuuint64_t)cf.head_dim / 64,
                              (cuuint64_t)cf.num_layers * cf.num_pages * 2};
  const cuuint64_t strides[3] = {row, 128, row * cf.page_size * cf.num_kv_heads};
  const cuuint32_t box[4] = {64, (cuuint32_t)cf.page_size, (cuuint32_t)cf.head_dim / 64, 2};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, kv, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MK_OK;
}

// Describe a dense weight matrix [rows][K] (bf16, row-major) to TMA for the tcgen05 tiles: boxes
// of 64 columns x 16 rows with the 128-byte swizzle (the K-major operand layout of tcgen05.mma);
// rows past the matrix read as zeros.
int encode_weight_map(const void* w, int rows, int K, CUtensorMap* out) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled (weights) failed (%d)", (int)r);
  return MK_OK;
}

void free_ctx(mk_ctx* c) {
  if (!c) return;
  cudaFree(c->d_wmaps);
  cudaFree(c->d_layers);
  cudaFree(c->d_tasks);
  cudaFree(c->d_task_off);
  cudaFree(c->ws);
  cudaFree(c->wdt);
  cudaFree(c->trace);
  for (int i = 0; i < 2; ++i) {
    if (c->h_step[i]) cudaFreeHost(c->h_step[i]);
    cudaFree(c->d_step[i]);
    if (c->ev_step[i]) cudaEventDestroy(c->ev_step[i]);
  }
  if (c->ev_done) cudaEventDestroy(c->ev_done);
  delete c;
}

}  // namespace

extern "C" {

const char* mk_last_error(void) { return g_err.c_str(); }

int mk_create(const mk_config* cfg, const mk_weights* w, mk_ctx** out) {
  g_err.clear();
  if (!out) return fail(MK_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!w || !w->layers || !w->embed || !w->final_norm || !w->lm_head)
    return fail(MK_ERR_INVALID_ARG, "weights: a required pointer is NULL");
  if (!aligned16(w->embed) || !aligned16(w->final_norm) || !aligned16(w->lm_head))
    return fail(MK_ERR_INVALID_ARG, "weights: pointers must be 16-byte aligned");
  for (int l = 0; l < cfg->num_layers; ++l) {
    const mk_layer_weights& lw = w->layers[l];
    const void* req[7] = {lw.attn_norm, lw.w_qkv, lw.w_o, lw.ffn_norm, lw.w_router, lw.w_gate_up, lw.w_down};
    for (const void* p : req) {
      if (!p) return fail(MK_ERR_INVALID_ARG, "weights: layer %d has a NULL tensor", l);
      if (!aligned16(p)) return fail(MK_ERR_INVALID_ARG, "weights: layer %d tensor not 16-byte aligned", l);
    }
    if (lw.router_bias && (reinterpret_cast<uintptr_t>(lw.router_bias) & 3u))
      return fail(MK_ERR_INVALID_ARG, "weights: layer %d router_bias misaligned", l);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaDeviceProp prop;
  if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (prop.major * 10 + prop.minor != 103)
    return fail(MK_ERR_UNSUPPORTED, "device %s is sm_%d%d; this build is for sm_103", prop.name, prop.major, prop.minor);
  if (!prop.cooperativeLaunch) return fail(MK_ERR_UNSUPPORTED, "device has no cooperative launch");
  const size_t smem = mk::smem_bytes();
  if (prop.sharedMemPerBlockOptin < smem)
    return fail(MK_ERR_UNSUPPORTED, "needs %zu bytes of shared memory per block, device offers %zu", smem,
                (size_t)prop.sharedMemPerBlockOptin);
  if ((e = mk::configure_kernels(cfg->head_dim, (cfg->flags & MK_FLAG_KV_Q8) != 0)) != cudaSuccess)
    return cuda_fail(e, "cudaFuncSetAttribute");
  int blocks = 0;
  if ((e = mk::occupancy(cfg->head_dim, (cfg->flags & MK_FLAG_KV_Q8) != 0, &blocks)) != cudaSuccess)
    return cuda_fail(e, "occupancy");
  if (blocks < 1) return fail(MK_ERR_UNSUPPORTED, "the step kernel does not fit on an SM");

  if (prop.multiProcessorCount > mk::kMaxCtas) return fail(MK_ERR_UNSUPPORTED, "more than 256 SMs");
  {
    // per block: the down projection keeps (row, slot) products and x_mid of its hidden rows on chip
    const int64_t nr = (cfg->hidden + prop.multiProcessorCount - 1) / prop.multiProcessorCount;
    if ((int64_t)cfg->max_batch * (cfg->top_k + 1) * nr > mk::kMoeScratch)
      return fail(MK_ERR_UNSUPPORTED, "max_batch*(top_k+1)*ceil(hidden/SMs) exceeds the down-projection scratch");
    if ((int64_t)cfg->max_batch * cfg->num_experts > mk::kMoeScratch)
      return fail(MK_ERR_UNSUPPORTED, "max_batch*num_experts exceeds the routing scratch");
  }
  mk_ctx* c = new mk_ctx();
  c->cfg = *cfg;
  if (c->cfg.watchdog_ms == 0) c->cfg.watchdog_ms = 1000;
  c->device = dev;
  c->n_ctas = prop.multiProcessorCount;
  build_static_plan(c->cfg, c->n_ctas, c->plan);
  const mk_plan_info& in = c->plan.info;
  const int L = cfg->num_layers, H = cfg->hidden, D = cfg->head_dim, Hq = cfg->num_q_heads, Hkv = cfg->num_kv_heads;
  const int G = Hq / Hkv, E = cfg->num_experts, K = cfg->top_k, F = cfg->expert_ffn, MB = cfg->max_batch;
  const int nqkv = (Hq + 2 * Hkv) * D;
  c->embed = static_cast<const uint16_t*>(w->embed);
  c->final_norm = static_cast<const uint16_t*>(w->final_norm);
  c->lm_head = static_cast<const uint16_t*>(w->lm_head);
  c->inv_freq.resize(D / 2);
  for (int i = 0; i < D / 2; ++i) c->inv_freq[i] = std::pow((double)cfg->rope_theta, -2.0 * i / D);

  c->small_ok = small_moe_fits(c->cfg, c->n_ctas);
  const size_t dt_layer = (size_t)E * F * H;   // elements of one layer's down projections
  if (c->small_ok) {
    if ((e = cudaMalloc(&c->wdt, dt_layer * L * sizeof(uint16_t))) != cudaSuccess) {
      free_ctx(c);
      return cuda_fail(e, "transposed down projections");
    }
    for (int l = 0; l < L && e == cudaSuccess; ++l)
      e = mk::transpose_down(static_cast<const uint16_t*>(w->layers[l].w_down), c->wdt + dt_layer * l, E, H, F, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { free_ctx(c); return cuda_fail(e, "down projection transpose"); }
  }
  std::vector<mk::LayerW> lws(L);
  for (int l = 0; l < L; ++l) {
    const mk_layer_weights& s = w->layers[l];
    lws[l] = {static_cast<const uint16_t*>(s.attn_norm), static_cast<const uint16_t*>(s.w_qkv),
              static_cast<const uint16_t*>(s.w_o), static_cast<const uint16_t*>(s.ffn_norm),
              static_cast<const uint16_t*>(s.w_router), s.router_bias, static_cast<const uint16_t*>(s.w_gate_up),
              static_cast<const uint16_t*>(s.w_down), c->wdt ? c->wdt + dt_layer * l : nullptr};
  }
  // split-K partials of the dense tcgen05 tiles: one block's group rows x max_batch words
  {
    int rows = 0;
    const int nrt = c->plan.info.n_router_tiles, rr = mk::router_tile_rows(E, c->n_ctas, MB);
    for (int op : {MK_OP_QKV, MK_OP_OPROJ, MK_OP_ROUTER}) {
      const int ks = mk::tc_ksplit(op, c->n_ctas, nrt, op == MK_OP_QKV ? nqkv : H, op == MK_OP_OPROJ ? Hq * D : H);
      if (ks == 1) continue;
      for (int g = 0; g + ks <= (op == MK_OP_ROUTER ? nrt : c->n_ctas); g += ks) {
        uint32_t lo, hi, lo2, hi2;
        if (op == MK_OP_ROUTER) {
          lo = (uint32_t)(g * rr); hi = (uint32_t)std::min(E, (g + ks) * rr);
        } else {
          const uint32_t n = op == MK_OP_QKV ? (uint32_t)nqkv : (uint32_t)H;
          split_range(n, c->n_ctas, g, &lo, &hi2);
          split_range(n, c->n_ctas, g + ks - 1, &lo2, &hi);
        }
        rows = std::max(rows, (int)(hi - lo));
      }
      // a block's finalisation gathers the group's partials of its own rows into the scratch
      const int own = op == MK_OP_ROUTER ? rr : ((op == MK_OP_QKV ? nqkv : H) + c->n_ctas - 1) / c->n_ctas;
      if ((int64_t)ks * (own + 1) * MB > mk::kMoeScratch) {
        free_ctx(c);
        return fail(MK_ERR_UNSUPPORTED, "split-K partials of %d rows x %d exceed the scratch", own, MB);
      }
    }
    c->psk_cap = rows * MB;
  }
  // workspace
  struct Part { void** ptr; size_t bytes; };
  const size_t f4 = sizeof(float), i4 = sizeof(int32_t), w8 = sizeof(uint64_t);
  const Part parts[] = {
      {(void**)&c->X, (size_t)(2 * L + 1) * MB * H * w8},
      {(void**)&c->QKV, (size_t)L * MB * nqkv * w8},
      {(void**)&c->ATT, (size_t)L * MB * Hq * D * w8},
      {(void**)&c->PO, (size_t)L * in.max_items * mk::kMaxG * D * w8},
      {(void**)&c->PML, (size_t)L * in.max_items * mk::kMaxG * 2 * w8},
      {(void**)&c->RLOG, (size_t)L * MB * E * w8},
      {(void**)&c->HB, (size_t)L * MB * K * F * w8},
      {(void**)&c->PT, c->small_ok ? (size_t)L * c->n_ctas * mk::kSmallMaxB * H * w8 : 0},
      {(void**)&c->YD, MB >= mk::kTcMinBatch ? (size_t)L * MB * K * H * w8 : 0},
      {(void**)&c->PSK, MB >= mk::kTcMinBatch ? (size_t)L * 3 * c->n_ctas * c->psk_cap * w8 : 0},
      {(void**)&c->PSQ, MB >= mk::kTcMinBatch ? (size_t)L * 3 * c->n_ctas * MB * w8 : 0},
      {(void**)&c->RIDS, (size_t)L * MB * K * i4},
      {(void**)&c->argp, (size_t)c->n_ctas * MB * 4 * f4},
      {(void**)&c->RW, (size_t)L * MB * K * f4},
      {(void**)&c->flags, (size_t)mk::kStepFlags * 4},
      {(void**)&c->d_status, sizeof(mk_status)},
  };
  size_t total = 0;
  for (const Part& p : parts) total += align256(p.bytes);
  if ((e = cudaMalloc(&c->ws, total)) != cudaSuccess) { free_ctx(c); return cuda_fail(e, "workspace"); }
  size_t o = 0;
  for (const Part& p : parts) { *p.ptr = c->ws + o; o += align256(p.bytes); }
  if ((e = cudaMemset(c->ws, 0, total)) != cudaSuccess) { free_ctx(c); return cuda_fail(e, "workspace memset"); }
  c->tagged_bytes = (size_t)(reinterpret_cast<uint8_t*>(c->RIDS) - reinterpret_cast<uint8_t*>(c->X));
  // static plan + layer table
  if ((e = cudaMalloc(&c->d_layers, sizeof(mk::LayerW) * L)) != cudaSuccess ||
      (e = cudaMalloc(&c->d_tasks, sizeof(mk_task) * c->plan.tasks.size())) != cudaSuccess ||
      (e = cudaMalloc(&c->d_task_off, sizeof(int32_t) * c->plan.off.size())) != cudaSuccess) {
    free_ctx(c);
    return cuda_fail(e, "plan buffers");
  }
  if ((e = cudaMemcpy(c->d_layers, lws.data(), sizeof(mk::LayerW) * L, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(c->d_tasks, c->plan.tasks.data(), sizeof(mk_task) * c->plan.tasks.size(),
                      cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(c->d_task_off, c->plan.off.data(), sizeof(int32_t) * c->plan.off.size(),
                      cudaMemcpyHostToDevice)) != cudaSuccess) {
    free_ctx(c);
    return cuda_fail(e, "plan upload");
  }
  // tensor maps of the weights, for the tcgen05 tiles of wide batches
  if (cfg->max_batch >= mk::kTcMinBatch) {
    std::vector<CUtensorMap> maps(mk::tc_map_count(L));
    for (int l = 0; l < L && rc == MK_OK; ++l) {
      const mk_layer_weights& s = w->layers[l];
      rc = encode_weight_map(s.w_qkv, nqkv, H, &maps[mk::tc_map_index(MK_OP_QKV, l, L)]);
      if (rc == MK_OK) rc = encode_weight_map(s.w_o, H, Hq * D, &maps[mk::tc_map_index(MK_OP_OPROJ, l, L)]);
      if (rc == MK_OK) rc = encode_weight_map(s.w_router, E, H, &maps[mk::tc_map_index(MK_OP_ROUTER, l, L)]);
      if (rc == MK_OK)
        rc = encode_weight_map(s.w_gate_up, E * 2 * F, H, &maps[mk::tc_map_index(MK_OP_MOE, l, L)]);
      if (rc == MK_OK) rc = encode_weight_map(s.w_down, E * H, F, &maps[mk::tc_map_index(mk::kTcOpDown, l, L)]);
    }
    if (rc == MK_OK) rc = encode_weight_map(w->lm_head, cfg->vocab, H, &maps[mk::tc_map_index(MK_OP_HEAD, L, L)]);
    if (rc) { free_ctx(c); return rc; }
    static_assert(sizeof(CUtensorMap) == 128, "tensor map size");
    if ((e = cudaMalloc(&c->d_wmaps, maps.size() * sizeof(CUtensorMap))) != cudaSuccess ||
        (e = cudaMemcpy(c->d_wmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice)) !=
            cudaSuccess) {
      free_ctx(c);
      return cuda_fail(e, "weight tensor maps");
    }
  }
  // per-step buffer layout
  size_t so = 0;
  auto take = [&](size_t bytes) { size_t r = so; so += (bytes + 15) & ~(size_t)15; return r; };
  c->off_tag = take(16);
  c->off_lens = take((size_t)MB * i4);
  c->off_cos = take((size_t)MB * (D / 2) * f4);
  c->off_sin = take((size_t)MB * (D / 2) * f4);
  c->off_items = take((size_t)in.max_items * sizeof(mk_attn_item));
  c->off_item_off = take((size_t)(c->n_ctas + 1) * i4);
  c->off_pair = take((size_t)MB * Hkv * i4);
  c->step_bytes = so;
  for (int i = 0; i < 2; ++i) {
    if ((e = cudaHostAlloc((void**)&c->h_step[i], so, cudaHostAllocDefault)) != cudaSuccess ||
        (e = cudaMalloc(&c->d_step[i], so)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->ev_step[i], cudaEventDisableTiming)) != cudaSuccess) {
      free_ctx(c);
      return cuda_fail(e, "step staging");
    }
  }
  if ((e = cudaEventCreateWithFlags(&c->ev_done, cudaEventDisableTiming)) != cudaSuccess) {
    free_ctx(c);
    return cuda_fail(e, "event");
  }
  *out = c;
  return MK_OK;
}

static int decode_step(mk_ctx* c, int32_t batch, const int32_t* token_ids, const int32_t* seq_lens,
                       const int32_t* block_tables, void* kv_pages, float* logits_out, int32_t* next_token,
                       float* margin, mk_stream_t stream);

int mk_decode_step(mk_ctx* c, int32_t batch, const int32_t* token_ids, const int32_t* seq_lens,
                   const int32_t* block_tables, void* kv_pages, float* logits_out, mk_stream_t stream) {
  return decode_step(c, batch, token_ids, seq_lens, block_tables, kv_pages, logits_out, nullptr, nullptr, stream);
}

int mk_decode_step_greedy(mk_ctx* c, int32_t batch, const int32_t* token_ids, const int32_t* seq_lens,
                          const int32_t* block_tables, void* kv_pages, float* logits_out, int32_t* next_token,
                          float* margin, mk_stream_t stream) {
  g_err.clear();
  if (!next_token) return fail(MK_ERR_INVALID_ARG, "next_token is NULL");
  if ((reinterpret_cast<uintptr_t>(next_token) | reinterpret_cast<uintptr_t>(margin)) & 3u)
    return fail(MK_ERR_INVALID_ARG, "next_token and margin must be 4-byte aligned");
  return decode_step(c, batch, token_ids, seq_lens, block_tables, kv_pages, logits_out, next_token, margin, stream);
}

// Checks of one step's arguments shared by the plain and the captured step.
static int check_step(mk_ctx* c, int32_t batch, const int32_t* token_ids, const int32_t* seq_lens,
                      const int32_t* block_tables, void* kv_pages, float* logits_out) {
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  const mk_config& cf = c->cfg;
  if (batch < 1 || batch > cf.max_batch) return fail(MK_ERR_INVALID_ARG, "batch %d outside 1..%d", batch, cf.max_batch);
  if (!token_ids || !block_tables || !kv_pages || !logits_out)
    return fail(MK_ERR_INVALID_ARG, "a step pointer is NULL");
  if (!aligned16(kv_pages)) return fail(MK_ERR_INVALID_ARG, "kv_pages must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(token_ids) | reinterpret_cast<uintptr_t>(block_tables) |
       reinterpret_cast<uintptr_t>(logits_out)) & 3u)
    return fail(MK_ERR_INVALID_ARG, "token_ids, block_tables and logits_out must be 4-byte aligned");
  if (seq_lens) {
    const int64_t max_len = (int64_t)cf.max_pages_per_seq * cf.page_size;
    for (int b = 0; b < batch; ++b)
      if (seq_lens[b] < 1 || seq_lens[b] > max_len)
        return fail(MK_ERR_INVALID_ARG, "seq_lens[%d]=%d outside 1..%lld", b, seq_lens[b], (long long)max_len);
  }
  return MK_OK;
}

// The next step tag (never 0).  Tagged words of an earlier step never match it; when the tag
// wraps, the tagged buffers are cleared on `s` first, so that no word from 2^32 steps ago can.
static int next_tag(mk_ctx* c, cudaStream_t s, uint32_t* tag) {
  if (++c->tag == 0) {
    cudaError_t e = cudaMemsetAsync(c->X, 0, c->tagged_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "tag wrap clear");
    c->tag = 1;
  }
  *tag = c->tag;
  return MK_OK;
}

// Host-built data of one step into staging buffer h (the layout the kernel reads from the
// device copy): tag, lengths, RoPE rows (angles in fp64), attention split plan.
static int fill_step(mk_ctx* c, uint8_t* h, int32_t batch, const int32_t* seq_lens, uint32_t tag) {
  const mk_config& cf = c->cfg;
  std::vector<mk_attn_item> items;
  std::vector<int32_t> item_off, pair_first;
  build_attention_plan(cf, c->n_ctas, batch, seq_lens, items, item_off, pair_first);
  if ((int)items.size() > c->plan.info.max_items) return fail(MK_ERR_INVALID_ARG, "attention plan overflow");
  const int D = cf.head_dim;
  std::memcpy(h + c->off_tag, &tag, sizeof tag);
  std::memcpy(h + c->off_lens, seq_lens, sizeof(int32_t) * batch);
  float* cs = reinterpret_cast<float*>(h + c->off_cos);
  float* sn = reinterpret_cast<float*>(h + c->off_sin);
  for (int b = 0; b < batch; ++b) {
    const double pos = (double)(seq_lens[b] - 1);
    for (int i = 0; i < D / 2; ++i) {
      const double ang = pos * c->inv_freq[i];
      cs[b * (D / 2) + i] = (float)std::cos(ang);
      sn[b * (D / 2) + i] = (float)std::sin(ang);
    }
  }
  std::memcpy(h + c->off_items, items.data(), sizeof(mk_attn_item) * items.size());
  std::memcpy(h + c->off_item_off, item_off.data(), sizeof(int32_t) * item_off.size());
  std::memcpy(h + c->off_pair, pair_first.data(), sizeof(int32_t) * pair_first.size());
  return MK_OK;
}

// Launch parameters of a step whose device step data is at d.
static int make_params(mk_ctx* c, mk::Params& p, int32_t batch, const uint8_t* d, const int32_t* token_ids,
                       const int32_t* block_tables, void* kv_pages, float* logits_out, int32_t* next_token,
                       float* margin) {
  const mk_config& cf = c->cfg;
  const int D = cf.head_dim;
  std::memset(&p, 0, sizeof p);
  p.L = cf.num_layers; p.H = cf.hidden; p.Hq = cf.num_q_heads; p.Hkv = cf.num_kv_heads; p.D = D;
  p.G = cf.num_q_heads / cf.num_kv_heads; p.E = cf.num_experts; p.K = cf.top_k; p.F = cf.expert_ffn;
  p.V = cf.vocab; p.ps = cf.page_size; p.P = cf.num_pages; p.maxpg = cf.max_pages_per_seq;
  p.nqkv = (cf.num_q_heads + 2 * cf.num_kv_heads) * D;
  p.norm_topk = cf.norm_topk;
  p.eps = cf.rms_eps;
  p.scale = (float)(1.0 / std::sqrt((double)D));
  p.B = batch; p.max_batch = cf.max_batch; p.n_ctas = c->n_ctas;
  const mk_plan_info& in = c->plan.info;
  p.n_qkv_tiles = in.n_qkv_tiles; p.n_o_tiles = in.n_o_tiles; p.n_router_tiles = in.n_router_tiles;
  p.wmaps = c->d_wmaps;
  p.tc = (c->d_wmaps != nullptr && batch >= mk::kTcMinBatch) ? 1 : 0;
  p.tasks = c->d_tasks; p.task_off = c->d_task_off;
  p.layers = c->d_layers; p.embed = c->embed; p.final_norm = c->final_norm; p.lm_head = c->lm_head;
  p.tokens = token_ids; p.block_tables = block_tables; p.kv = static_cast<uint16_t*>(kv_pages); p.logits = logits_out;
  p.kv_q8 = (cf.flags & MK_FLAG_KV_Q8) ? 1 : 0;
  p.kv_layer_bytes = p.kv_q8 ? kv_q8_layer_bytes(cf) : 0;
  p.kv_code_bytes = p.kv_q8 ? kv_q8_code_bytes(cf) : 0;
  p.step_tag = reinterpret_cast<const uint32_t*>(d + c->off_tag);
  p.seq_lens = reinterpret_cast<const int32_t*>(d + c->off_lens);
  p.rope_cos = reinterpret_cast<const float*>(d + c->off_cos);
  p.rope_sin = reinterpret_cast<const float*>(d + c->off_sin);
  p.items = reinterpret_cast<const mk_attn_item*>(d + c->off_items);
  p.item_off = reinterpret_cast<const int32_t*>(d + c->off_item_off);
  p.pair_first = reinterpret_cast<const int32_t*>(d + c->off_pair);
  p.X = c->X; p.QKV = c->QKV; p.ATT = c->ATT; p.PO = c->PO; p.PML = c->PML; p.RLOG = c->RLOG; p.RIDS = c->RIDS;
  p.RW = c->RW; p.HB = c->HB; p.YD = c->YD; p.PSK = c->PSK; p.PSQ = c->PSQ; p.psk_cap = c->psk_cap;
  p.small_moe = c->small_ok && mk::small_moe_batch(batch, cf.hidden) ? 1 : 0;
  p.PT = c->PT;
  p.next_token = next_token; p.margin = margin; p.argp = c->argp;
  p.max_items = c->plan.info.max_items;
  p.flags = c->flags; p.status = c->d_status;
  p.trace = c->trace; p.trace_cap = c->trace_cap;
  if (kv_pages != c->kv_map_ptr) {
    int rc2 = encode_kv_map(cf, kv_pages, &c->kv_map);
    if (rc2) return rc2;
    c->kv_map_ptr = kv_pages;
  }
  static_assert(sizeof(CUtensorMap) == sizeof(p.kv_map), "tensor map size");
  std::memcpy(p.kv_map, &c->kv_map, sizeof(p.kv_map));
  p.stall_layer = -1;
  p.watchdog_ns = (uint64_t)cf.watchdog_ms * 1000000ull;
  return MK_OK;
}

static int decode_step(mk_ctx* c, int32_t batch, const int32_t* token_ids, const int32_t* seq_lens,
                       const int32_t* block_tables, void* kv_pages, float* logits_out, int32_t* next_token,
                       float* margin, mk_stream_t stream) {
  g_err.clear();
  if (!seq_lens) return fail(MK_ERR_INVALID_ARG, "a step pointer is NULL");
  int rc = check_step(c, batch, token_ids, seq_lens, block_tables, kv_pages, logits_out);
  if (rc) return rc;
  cudaError_t e;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // host-built per-step data into the staging buffer not used by the previous step
  const int cur = c->cur;
  if ((e = cudaEventSynchronize(c->ev_step[cur])) != cudaSuccess) return cuda_fail(e, "staging event");
  uint32_t tag;
  if ((rc = next_tag(c, s, &tag))) return rc;
  uint8_t* h = c->h_step[cur];
  if ((rc = fill_step(c, h, batch, seq_lens, tag))) return rc;
  uint8_t* d = c->d_step[cur];
  if ((e = cudaMemcpyAsync(d, h, c->step_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "step upload");
  if ((e = cudaEventRecord(c->ev_step[cur], s)) != cudaSuccess) return cuda_fail(e, "event record");
  c->cur ^= 1;
  mk::Params p;
  if ((rc = make_params(c, p, batch, d, token_ids, block_tables, kv_pages, logits_out, next_token, margin))) return rc;
  // test hook: the O-proj tiles of one layer wait for a tag that is never written
  if (c->stall_layer >= 0) {
    p.stall_layer = c->stall_layer;
    if (c->stall_ms) p.watchdog_ns = (uint64_t)c->stall_ms * 1000000ull;
    c->stall_layer = -1;
  }
  if ((e = mk::launch_step(p, s)) != cudaSuccess) return cuda_fail(e, "cooperative launch");
  if ((e = cudaEventRecord(c->ev_done, s)) != cudaSuccess) return cuda_fail(e, "event record");
  c->stepped = true;
  c->last_B = batch;
  return MK_OK;
}

// ---------------------------------------------------------------- captured steps (CUDA graphs)
struct mk_graph {
  mk_ctx* c = nullptr;
  int32_t batch = 0;
  uint8_t* h[2] = {nullptr, nullptr};      // pinned host staging, one per graph
  uint8_t* d[2] = {nullptr, nullptr};      // its device copy, read by the graph's kernel
  cudaEvent_t ev[2] = {nullptr, nullptr};  // the graph's copy has read h (recorded after its launch)
  cudaGraph_t g[2] = {nullptr, nullptr};
  cudaGraphExec_t x[2] = {nullptr, nullptr};
  int cur = 0;
};

void mk_graph_destroy(mk_graph* g) {
  if (!g) return;
  for (int i = 0; i < 2; ++i) {
    if (g->ev[i]) cudaEventSynchronize(g->ev[i]);
    if (g->x[i]) cudaGraphExecDestroy(g->x[i]);
    if (g->g[i]) cudaGraphDestroy(g->g[i]);
    if (g->h[i]) cudaFreeHost(g->h[i]);
    cudaFree(g->d[i]);
    if (g->ev[i]) cudaEventDestroy(g->ev[i]);
  }
  delete g;
}

int mk_graph_create(mk_ctx* c, int32_t batch, const int32_t* token_ids, const int32_t* block_tables, void* kv_pages,
                    float* logits_out, mk_graph** out) {
  g_err.clear();
  if (!out) return fail(MK_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int rc = check_step(c, batch, token_ids, nullptr, block_tables, kv_pages, logits_out);
  if (rc) return rc;
  mk_graph* g = new mk_graph();
  g->c = c;
  g->batch = batch;
  cudaError_t e;
  cudaStream_t cs = nullptr;
  for (int i = 0; i < 2; ++i) {
    if ((e = cudaHostAlloc((void**)&g->h[i], c->step_bytes, cudaHostAllocDefault)) != cudaSuccess ||
        (e = cudaMalloc(&g->d[i], c->step_bytes)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&g->ev[i], cudaEventDisableTiming)) != cudaSuccess) {
      mk_graph_destroy(g);
      return cuda_fail(e, "graph staging");
    }
    std::memset(g->h[i], 0, c->step_bytes);
  }
  if ((e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking)) != cudaSuccess) {
    mk_graph_destroy(g);
    return cuda_fail(e, "capture stream");
  }
  for (int i = 0; i < 2 && rc == MK_OK; ++i) {
    mk::Params p;
    if ((rc = make_params(c, p, batch, g->d[i], token_ids, block_tables, kv_pages, logits_out, nullptr, nullptr)))
      break;
    if ((e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal)) != cudaSuccess) {
      rc = cuda_fail(e, "begin capture");
      break;
    }
    cudaError_t e1 = cudaMemcpyAsync(g->d[i], g->h[i], c->step_bytes, cudaMemcpyHostToDevice, cs);
    cudaError_t e2 = e1 == cudaSuccess ? mk::launch_step(p, cs) : e1;
    e = cudaStreamEndCapture(cs, &g->g[i]);
    if (e2 != cudaSuccess) { rc = cuda_fail(e2, "capture of the step"); break; }
    if (e != cudaSuccess) { rc = cuda_fail(e, "end capture"); break; }
    if ((e = cudaGraphInstantiate(&g->x[i], g->g[i], 0)) != cudaSuccess) { rc = cuda_fail(e, "graph instantiate"); break; }
  }
  cudaStreamDestroy(cs);
  if (rc) {
    mk_graph_destroy(g);
    return rc;
  }
  *out = g;
  return MK_OK;
}

int mk_graph_launch(mk_graph* g, const int32_t* seq_lens, mk_stream_t stream) {
  g_err.clear();
  if (!g || !seq_lens) return fail(MK_ERR_INVALID_ARG, "graph or seq_lens is NULL");
  mk_ctx* c = g->c;
  const mk_config& cf = c->cfg;
  const int64_t max_len = (int64_t)cf.max_pages_per_seq * cf.page_size;
  for (int b = 0; b < g->batch; ++b)
    if (seq_lens[b] < 1 || seq_lens[b] > max_len)
      return fail(MK_ERR_INVALID_ARG, "seq_lens[%d]=%d outside 1..%lld", b, seq_lens[b], (long long)max_len);
  cudaError_t e;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int i = g->cur;
  // the graph that read this staging buffer two launches ago has finished with it
  if ((e = cudaEventSynchronize(g->ev[i])) != cudaSuccess) return cuda_fail(e, "graph staging event");
  uint32_t tag;
  int rc = next_tag(c, s, &tag);
  if (rc) return rc;
  if ((rc = fill_step(c, g->h[i], g->batch, seq_lens, tag))) return rc;
  if ((e = cudaGraphLaunch(g->x[i], s)) != cudaSuccess) return cuda_fail(e, "graph launch");
  if ((e = cudaEventRecord(g->ev[i], s)) != cudaSuccess) return cuda_fail(e, "event record");
  if ((e = cudaEventRecord(c->ev_done, s)) != cudaSuccess) return cuda_fail(e, "event record");
  g->cur ^= 1;
  c->stepped = true;
  c->last_B = g->batch;
  return MK_OK;
}

int mk_get_status(mk_ctx* c, mk_status* out) {
  g_err.clear();
  if (!c || !out) return fail(MK_ERR_INVALID_ARG, "ctx or out is NULL");
  std::memset(out, 0, sizeof *out);
  cudaError_t e;
  if (c->stepped && (e = cudaEventSynchronize(c->ev_done)) != cudaSuccess) return cuda_fail(e, "step");
  if ((e = cudaMemcpy(out, c->d_status, sizeof *out, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "status read");
  if (out->code != MK_OK) {
    if ((e = cudaMemset(c->d_status, 0, sizeof(mk_status))) != cudaSuccess) return cuda_fail(e, "status clear");
    g_err = out->code == MK_ERR_TIMEOUT ? "device: a dependency wait ran out" : "device: index out of range";
  }
  return out->code;
}

void mk_destroy(mk_ctx* c) {
  if (!c) return;
  if (c->stepped) cudaEventSynchronize(c->ev_done);
  free_ctx(c);
}

// ==================================================================== debug / planning
int mk_num_ctas(mk_ctx* c) { return c ? c->n_ctas : 0; }

int mk_debug_inject_stall(mk_ctx* c, int32_t layer, uint32_t watchdog_ms) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if (layer >= c->cfg.num_layers) return fail(MK_ERR_INVALID_ARG, "layer out of range");
  c->stall_layer = layer;
  c->stall_ms = watchdog_ms;
  return MK_OK;
}

int mk_debug_read(mk_ctx* c, int32_t what, int32_t layer, void* dst, size_t bytes) {
  g_err.clear();
  if (!c || !dst) return fail(MK_ERR_INVALID_ARG, "ctx or dst is NULL");
  if (!c->stepped) return fail(MK_ERR_INVALID_ARG, "no step has run");
  const mk_config& cf = c->cfg;
  const int B = c->last_B, MB = cf.max_batch, L = cf.num_layers;
  if (what != MK_DBG_X && (layer < 0 || layer >= L)) return fail(MK_ERR_INVALID_ARG, "layer out of range");
  const void* src = nullptr;
  size_t row = 0, rows = 0, stride = 0;   // copy `rows` rows of `row` bytes, source stride `stride`
  const size_t nqkv = (size_t)(cf.num_q_heads + 2 * cf.num_kv_heads) * cf.head_dim;
  const size_t K = cf.top_k, E = cf.num_experts, H = cf.hidden, F = cf.expert_ffn;
  const size_t QD = (size_t)cf.num_q_heads * cf.head_dim;
  bool tagged = true;   // buffer of tagged 8-byte words: the value is the low half
  switch (what) {
    case MK_DBG_X: src = c->X; row = (size_t)B * H; rows = 2 * L + 1; stride = (size_t)MB * H; break;
    case MK_DBG_QKV: src = c->QKV + (size_t)layer * MB * nqkv; row = (size_t)B * nqkv; rows = 1; break;
    case MK_DBG_ATTN: src = c->ATT + (size_t)layer * MB * QD; row = (size_t)B * QD; rows = 1; break;
    case MK_DBG_ROUTER: src = c->RLOG + (size_t)layer * MB * E; row = (size_t)B * E; rows = 1; break;
    case MK_DBG_ROUTE_IDS: src = c->RIDS + (size_t)layer * MB * K; row = (size_t)B * K; rows = 1; tagged = false; break;
    case MK_DBG_ROUTE_W: src = c->RW + (size_t)layer * MB * K; row = (size_t)B * K; rows = 1; tagged = false; break;
    case MK_DBG_H: src = c->HB + (size_t)layer * MB * K * F; row = (size_t)B * K * F; rows = 1; break;
    default: return fail(MK_ERR_INVALID_ARG, "unknown buffer %d", what);
  }
  if (bytes != row * rows * 4) return fail(MK_ERR_INVALID_ARG, "bytes must be %zu", row * rows * 4);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "sync");
  if (!tagged) {
    e = cudaMemcpy(dst, src, row * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "debug read");
    return MK_OK;
  }
  std::vector<uint64_t> tmp(row);
  uint32_t* out = static_cast<uint32_t*>(dst);
  for (size_t r = 0; r < rows; ++r) {
    e = cudaMemcpy(tmp.data(), static_cast<const uint64_t*>(src) + r * stride, row * 8, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "debug read");
    for (size_t i = 0; i < row; ++i) out[r * row + i] = (uint32_t)tmp[i];
  }
  return MK_OK;
}

int mk_debug_trace(mk_ctx* c, int32_t enable, int32_t events_per_cta) {
  g_err.clear();
  if (!c) return fail(MK_ERR_INVALID_ARG, "ctx is NULL");
  if (!mk::kTrace && enable) return fail(MK_ERR_UNSUPPORTED, "the timeline is compiled out of this build (MK_TRACE=0)");
  cudaError_t e;
  if (c->stepped && (e = cudaEventSynchronize(c->ev_done)) != cudaSuccess) return cuda_fail(e, "step");
  cudaFree(c->trace);
  c->trace = nullptr;
  c->trace_cap = 0;
  if (!enable) return MK_OK;
  if (events_per_cta < 16 || events_per_cta > (1 << 20)) return fail(MK_ERR_INVALID_ARG, "events_per_cta out of range");
  const size_t bytes = (size_t)c->n_ctas * events_per_cta * 32;
  if ((e = cudaMalloc(&c->trace, bytes)) != cudaSuccess) return cuda_fail(e, "trace buffer");
  if ((e = cudaMemset(c->trace, 0, bytes)) != cudaSuccess) return cuda_fail(e, "trace clear");
  c->trace_cap = events_per_cta;
  return MK_OK;
}

int mk_debug_trace_read(mk_ctx* c, void* dst, size_t bytes) {
  g_err.clear();
  if (!c || !dst) return fail(MK_ERR_INVALID_ARG, "ctx or dst is NULL");
  if (!c->trace) return fail(MK_ERR_INVALID_ARG, "tracing is not enabled");
  const size_t want = (size_t)c->n_ctas * c->trace_cap * 32;
  if (bytes != want) return fail(MK_ERR_INVALID_ARG, "bytes must be %zu", want);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "sync");
  if ((e = cudaMemcpy(dst, c->trace, want, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e, "trace read");
  return MK_OK;
}

int mk_plan_static(const mk_config* cfg, int32_t n_ctas, mk_plan_info* info, mk_task* tasks, int32_t* cta_offsets) {
  g_err.clear();
  int rc = check_config(cfg);
  if (rc) return rc;
  if (n_ctas < 1 || !info) return fail(MK_ERR_INVALID_ARG, "n_ctas < 1 or info NULL");
  Plan plan;
  build_static_plan(*cfg, n_ctas, plan);
  *info = plan.info;
  if (tasks) std::memcpy(tasks, plan.tasks.data(), sizeof(mk_task) * plan.tasks.size());
  if (cta_offsets) std::memcpy(cta_offsets, plan.off.data(), sizeof(int32_t) * plan.off.size());
  return MK_OK;
}

int mk_plan_attention(const mk_config* cfg, int32_t n_ctas, int32_t batch, const int32_t* seq_lens,
                      mk_attn_item* items, int32_t max_items, int32_t* cta_offsets, int32_t* n_items) {
  g_err.clear();
  int rc = check_config(cfg);
  if (rc) return rc;
  if (n_ctas < 1 || batch < 1 || batch > cfg->max_batch || !seq_lens || !n_items)
    return fail(MK_ERR_INVALID_ARG, "bad arguments");
  const int64_t max_len = (int64_t)cfg->max_pages_per_seq * cfg->page_size;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] < 1 || seq_lens[b] > max_len) return fail(MK_ERR_INVALID_ARG, "seq_lens[%d] out of range", b);
  std::vector<mk_attn_item> it;
  std::vector<int32_t> off, pf;
  build_attention_plan(*cfg, n_ctas, batch, seq_lens, it, off, pf);
  *n_items = (int32_t)it.size();
  if ((int32_t)it.size() > max_items) return fail(MK_ERR_INVALID_ARG, "max_items too small (%zu needed)", it.size());
  if (items) std::memcpy(items, it.data(), sizeof(mk_attn_item) * it.size());
  if (cta_offsets) std::memcpy(cta_offsets, off.data(), sizeof(int32_t) * off.size());
  return MK_OK;
}

// -------------------------------------------------------------------- CPU simulator
// A model of the device runtime at record granularity: per virtual SM, a producer
// that turns tasks into records (at most `lead` ahead of its consumer; the MoE
// records of a layer only once routing is published, split with the device's
// rule) and a consumer that runs records in order, honours each record's counter
// wait and applies its counter effects (including the "last arrival merges" rules
// of attention splits and routing).
int mk_simulate(const mk_config* cfg, int32_t n_ctas, int32_t B, const int32_t* seq_lens, const int32_t* routing_ids,
                uint64_t seed, int32_t lead, mk_sim_result* out) {
  g_err.clear();
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!out || !seq_lens || !routing_ids || n_ctas < 1 || n_ctas > mk::kMaxCtas || B < 1 || B > cfg->max_batch ||
      lead < 1)
    return fail(MK_ERR_INVALID_ARG, "bad arguments");
  std::memset(out, 0, sizeof *out);
  Plan plan;
  build_static_plan(*cfg, n_ctas, plan);
  std::vector<mk_attn_item> items;
  std::vector<int32_t> ioff, pf;
  build_attention_plan(*cfg, n_ctas, B, seq_lens, items, ioff, pf);
  const mk_plan_info& in = plan.info;
  const int L = cfg->num_layers, E = cfg->num_experts, K = cfg->top_k, Hkv = cfg->num_kv_heads;
  const int F = cfg->expert_ffn, H = cfg->hidden, D = cfg->head_dim, Hq = cfg->num_q_heads, G = Hq / Hkv;
  const uint32_t nqkv = (uint32_t)(Hq + 2 * Hkv) * D;
  const int n_items = (int)items.size();
  // wide batches run the dense tiles and the MoE on tcgen05 (the engine has the weight maps)
  const bool tcs = cfg->max_batch >= mk::kTcMinBatch && B >= mk::kTcMinBatch;
  // per layer: active experts (ascending) and the gate/up unit range of every block
  std::vector<std::vector<int>> act(L), rows_of(L);   // active experts; rows routed to each expert
  std::vector<std::vector<int32_t>> gu_start(L), dn_start(L);
  for (int l = 0; l < L; ++l) {
    std::vector<int>& cnt = rows_of[l];
    cnt.assign(E, 0);
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < K; ++j) {
        const int e = routing_ids[((size_t)l * B + b) * K + j];
        if (e < 0 || e >= E) return fail(MK_ERR_INVALID_ARG, "routing id out of range");
        cnt[e]++;
      }
    std::vector<int64_t> cost, cum(1, 0);
    for (int e = 0; e < E; ++e)
      if (cnt[e]) {
        act[l].push_back(e);
        cost.push_back(mk::moe_unit_cost(cnt[e], tcs));
        cum.push_back(cum.back() + (int64_t)F * cost.back());
      }
    const int nact = (int)act[l].size();
    for (int j = 0; j <= n_ctas; ++j) gu_start[l].push_back(mk::moe_gu_start(j, n_ctas, cum.data(), cost.data(), nact, F));
    // the tcgen05 down projection deals its (expert, row block) units by the same costs
    const int nrb = (H + mk::kTcDownRows - 1) / mk::kTcDownRows;
    for (int j = 0; j <= n_ctas; ++j)
      dn_start[l].push_back(mk::moe_gu_start(j, n_ctas, cum.data(), cost.data(), nact, nrb, nrb, F));
  }
  // coverage of the MoE work: gate/up units and (active expert, hidden row) pairs of the down
  // projection, or on the small-batch path the transposed down row of every unit
  const bool small = small_moe_step(*cfg, n_ctas, B);
  std::vector<std::vector<int>> gu_seen(L), dn_seen(L), dt_seen(L);
  for (int l = 0; l < L; ++l) {
    gu_seen[l].assign(act[l].size() * F, 0);
    dn_seen[l].assign(act[l].size() * H, 0);
    dt_seen[l].assign(act[l].size() * F, 0);
  }

  // ---- what has been written this step, by writer tile (the device polls the tagged words
  // those tiles write; a reader proceeds once every word it reads carries the step's tag)
  std::vector<uint32_t> hlo(n_ctas), hhi(n_ctas), qlo(n_ctas), qhi(n_ctas);
  int n_hrow_blocks = 0;   // blocks owning hidden rows: writers of every residual vector
  for (int i = 0; i < n_ctas; ++i) {
    split_range((uint32_t)H, n_ctas, i, &hlo[i], &hhi[i]);
    split_range(nqkv, n_ctas, i, &qlo[i], &qhi[i]);
    n_hrow_blocks += hhi[i] > hlo[i];
  }
  int n_item_blocks = 0;   // blocks that hold attention items (each merges a slice after its last one)
  for (int i = 0; i < n_ctas; ++i) n_item_blocks += ioff[i + 1] > ioff[i];
  // xout[l][i]: block i wrote its hidden rows of the layer-l input X[2l] (l = 0: the embedding,
  // l = L: the last layer's output); its count per layer
  std::vector<std::vector<char>> xout(L + 1, std::vector<char>(n_ctas, 0));
  std::vector<int> xout_n(L + 1, 0);
  std::vector<std::vector<char>> qkv_done(L, std::vector<char>(n_ctas, 0));
  std::vector<std::vector<char>> item_done(L, std::vector<char>(std::max(1, n_items), 0));
  std::vector<int> merged_n(L, 0), oproj_n(L, 0), router_n(L, 0), moe_share_n(L, 0), down_n(L, 0);
  const int nrb = (H + mk::kTcDownRows - 1) / mk::kTcDownRows;   // tcgen05 down projection: row blocks
  std::vector<std::vector<char>> oproj_done(L, std::vector<char>(n_ctas, 0));
  std::vector<std::vector<char>> routed(n_ctas, std::vector<char>(L, 0));
  int writes_twice = 0;
  auto mark = [&](char& f) { if (f) writes_twice++; f = 1; };
  // QKV tiles holding rows [r0, r1) of the fused output: the device's attention item polls
  // those words (q of the pair's query heads, k and v of its KV head)
  auto qkv_rows_ready = [&](int l, uint32_t r0, uint32_t r1) {
    for (int i = 0; i < n_ctas; ++i)
      if (qhi[i] > qlo[i] && qlo[i] < r1 && qhi[i] > r0 && !qkv_done[l][i]) return false;
    return true;
  };
  // residual rows [r0, r1) of X[2l] (the block's own O-proj residual input)
  auto xrows_ready = [&](int l, uint32_t r0, uint32_t r1) {
    for (int i = 0; i < n_ctas; ++i)
      if (hhi[i] > hlo[i] && hlo[i] < r1 && hhi[i] > r0 && !xout[l][i]) return false;
    return true;
  };
  auto orows_ready = [&](int l, uint32_t r0, uint32_t r1) {
    for (int i = 0; i < n_ctas; ++i)
      if (hhi[i] > hlo[i] && hlo[i] < r1 && hhi[i] > r0 && !oproj_done[l][i]) return false;
    return true;
  };

  // record kinds: a task op (ATTN: one per item), 110 = routing (every block), 100 = gate/up
  // chunk, 101 = down chunk; small-batch path: 105 = gate/up chunk, 102 = transposed down
  // chunk, 104 = publish the partial output, 103 = reduce every block's partials; tcgen05 path:
  // 100 = a gate/up run, 106 = an (expert, row block) down unit, 107 = sum of own rows' slots
  struct Rec { int kind; int task; int layer; uint32_t a; uint32_t x; int flags; };
  enum { F_FIRST = 1, F_LAST = 2, F_LAST_GU = 4, F_EMPTY = 8 };
  struct Sm {
    std::vector<Rec> q; size_t qhead = 0; int ti;
    std::vector<Rec> moe; size_t moe_next = 0; bool moe_open = false; bool route_sent = false;
    bool prod_done = false; bool done = false;
    int merge_layer = -1;   // the split merge the consumer runs after its last attention item
  };
  std::vector<Sm> sm(n_ctas);
  for (int i = 0; i < n_ctas; ++i) sm[i].ti = plan.off[i];
  std::mt19937_64 rng(seed);
  const int fpc = std::max(1, mk::gemv_rows_per_chunk(H) / 2);
  const int rows_fit = std::max(1, mk::kSlotBytes / (F * 2));

  // the MoE records block i produces for layer l (the device producer's loops)
  auto moe_records = [&](int i, int l, int task) {
    std::vector<Rec> r;
    const int nact = (int)act[l].size();
    const int u0 = gu_start[l][i], u1 = gu_start[l][i + 1];
    if (small) {   // the device producer's small-batch loops
      for (int u = u0; u < u1;) {
        const int a = u / F, f0 = u % F, fend = std::min(F, u1 - a * F);
        for (int g0 = f0; g0 < fend; g0 += 2 * fpc) {
          const int gend = std::min(fend, g0 + 2 * fpc);
          for (int f = g0; f < gend; f += fpc) {
            const int n = std::min(fpc, gend - f);
            for (int k = 0; k < n; ++k) gu_seen[l][(size_t)a * F + f + k]++;
            r.push_back({105, task, l, (uint32_t)a, (uint32_t)f, 0});
          }
          for (int f = g0; f < gend; ++f) dt_seen[l][(size_t)a * F + f]++;
          r.push_back({102, task, l, (uint32_t)a, (uint32_t)g0, 0});
        }
        u = a * F + fend;
      }
      r.push_back({104, task, l, 0, 0, 0});
      r.push_back({103, task, l, 0, 0, hhi[i] > hlo[i] ? 0 : F_EMPTY});
      return r;
    }
    if (u0 >= u1) r.push_back({100, task, l, 0, 0, F_FIRST | F_LAST | F_LAST_GU | F_EMPTY});
    if (tcs) {   // the device producer's tcgen05 loops (one record stands for a run's chunks)
      for (int u = u0; u < u1;) {
        const int a = u / F, f0 = u % F, fend = std::min(F, u1 - a * F);
        for (int f = f0; f < fend; ++f) gu_seen[l][(size_t)a * F + f]++;
        r.push_back({100, task, l, (uint32_t)a, (uint32_t)f0, F_FIRST | F_LAST | (a * F + fend >= u1 ? F_LAST_GU : 0)});
        u = a * F + fend;
      }
      const int ua = dn_start[l][i], ub = dn_start[l][i + 1];
      for (int u = ua; u < ub; ++u) {
        const int a = u / nrb, rb = u % nrb;
        for (int x = rb * mk::kTcDownRows; x < std::min(H, (rb + 1) * mk::kTcDownRows); ++x) dn_seen[l][(size_t)a * H + x]++;
        r.push_back({106, task, l, (uint32_t)a, (uint32_t)rb, 0});
      }
      r.push_back({107, task, l, 0, hlo[i], hhi[i] > hlo[i] ? 0 : F_EMPTY});
      return r;
    }
    for (int u = u0; u < u1;) {
      const int a = u / F, f0 = u % F, fend = std::min(F, u1 - a * F);
      // batches of 3 or more: the run is streamed once per register group of its routed rows
      const int ng = B > 2 ? (rows_of[l][act[l][a]] + mk::wide_group_rows(H) - 1) / mk::wide_group_rows(H) : 1;
      for (int g = 0; g < ng; ++g) {
        for (int f = f0; f < fend; f += fpc) {
          const int n = std::min(fpc, fend - f);
          if (g == 0)
            for (int k = 0; k < n; ++k) gu_seen[l][(size_t)a * F + f + k]++;
          r.push_back({100, task, l, (uint32_t)a, (uint32_t)f,
                       (g == 0 && f == f0 ? F_FIRST : 0) | (g == ng - 1 && f + n >= fend ? F_LAST : 0) |
                           (a * F + fend >= u1 ? F_LAST_GU : 0)});
        }
      }
      u = a * F + fend;
    }
    const uint32_t r0 = hlo[i], r1 = hhi[i];
    if (r1 <= r0 || nact == 0) {
      r.push_back({101, task, l, 0, r0, F_FIRST | F_LAST | F_EMPTY});
      return r;
    }
    const int rpc = std::min((int)(r1 - r0), rows_fit);
    bool first = true;
    for (int rb = (int)r0; rb < (int)r1; rb += rpc) {
      const int nrc = std::min(rpc, (int)r1 - rb);
      const int epc = std::max(1, mk::kSlotBytes / (nrc * F * 2));
      for (int a = 0; a < nact; a += epc) {
        const int ne = std::min(epc, nact - a);
        for (int k = 0; k < ne; ++k)
          for (int x = 0; x < nrc; ++x) dn_seen[l][(size_t)(a + k) * H + rb + x]++;
        const bool last = rb + nrc >= (int)r1 && a + ne >= nact;
        r.push_back({101, task, l, (uint32_t)a, (uint32_t)rb, (first ? F_FIRST : 0) | (last ? F_LAST : 0)});
        first = false;
      }
    }
    return r;
  };

  auto produce = [&](int i) -> bool {   // one record; false if blocked or finished
    Sm& s = sm[i];
    if (s.prod_done || (int)(s.q.size() - s.qhead) >= lead) return false;
    const mk_task& t = plan.tasks[s.ti];
    switch (t.op) {
      case MK_OP_ATTN:
        for (int it = ioff[i]; it < ioff[i + 1]; ++it) s.q.push_back({MK_OP_ATTN, s.ti, t.layer, (uint32_t)it, 0, 0});
        break;
      case MK_OP_MOE: {
        const int l = t.layer;
        if (!s.route_sent) {            // the routing record, then wait for this block's routing
          s.q.push_back({110, s.ti, l, 0, 0, 0});
          s.route_sent = true;
          return true;
        }
        if (!s.moe_open) {
          if (!routed[i][l]) return false;
          s.moe = moe_records(i, l, s.ti);
          s.moe_next = 0;
          s.moe_open = true;
        }
        s.q.push_back(s.moe[s.moe_next++]);
        if (s.moe_next < s.moe.size()) return true;   // stay on this task
        s.moe_open = false;
        s.route_sent = false;
        break;
      }
      default: s.q.push_back({t.op, s.ti, t.layer, 0, 0, 0}); break;
    }
    if (t.op == MK_OP_END) s.prod_done = true;
    else s.ti++;
    return true;
  };
  auto consume = [&](int i) -> bool {
    Sm& s = sm[i];
    if (s.done) return false;
    if (s.merge_layer >= 0) {
      // the split merge after the block's last item: every split of each pair it holds a split of
      const int l = s.merge_layer;
      for (int it = ioff[i]; it < ioff[i + 1]; ++it) {
        const int first = pf[items[it].b * Hkv + items[it].kvh];
        for (int k = 0; k < items[it].nsplit; ++k)
          if (!item_done[l][first + k]) return false;
      }
      merged_n[l]++;
      s.merge_layer = -1;
      return true;
    }
    if (s.qhead >= s.q.size()) return false;
    const Rec& r = s.q[s.qhead];
    const mk_task& t = plan.tasks[r.task];
    const int l = r.layer;
    switch (r.kind) {
      case MK_OP_EMBED:
        mark(xout[0][i]);
        xout_n[0]++;
        break;
      case MK_OP_QKV:
        if (xout_n[l] < n_hrow_blocks) return false;
        mark(qkv_done[l][i]);
        break;
      case MK_OP_ATTN: {
        const mk_attn_item& it = items[r.a];
        const uint32_t q0 = (uint32_t)it.kvh * G * D, k0 = (uint32_t)(Hq + it.kvh) * D,
                       v0 = (uint32_t)(Hq + Hkv + it.kvh) * D;
        if (!qkv_rows_ready(l, q0, q0 + (uint32_t)G * D) || !qkv_rows_ready(l, k0, k0 + D) ||
            !qkv_rows_ready(l, v0, v0 + D))
          return false;
        mark(item_done[l][r.a]);
        if ((int)r.a == ioff[i + 1] - 1) s.merge_layer = l;
        break;
      }
      case MK_OP_OPROJ:
        if (merged_n[l] < n_item_blocks || !xrows_ready(l, t.lo, t.hi)) return false;
        mark(oproj_done[l][i]);
        oproj_n[l]++;
        break;
      case MK_OP_ROUTER:
        if (oproj_n[l] < in.n_o_tiles) return false;
        router_n[l]++;
        break;
      case 110:   // routing: every router logit (and the MoE input, x after attention)
        if (router_n[l] < in.n_router_tiles || oproj_n[l] < in.n_o_tiles) return false;
        mark(routed[i][l]);
        break;
      case 100:   // a block's gate/up share is complete after its last run's last chunk
        if ((r.flags & F_LAST_GU) && (r.flags & F_LAST)) moe_share_n[l]++;
        break;
      case 101:   // the down projection reads every block's SwiGLU outputs and its own x rows
        if (!(r.flags & F_EMPTY) && (r.flags & F_FIRST) &&
            (moe_share_n[l] < n_ctas || !orows_ready(l, hlo[i], hhi[i])))
          return false;
        if (!(r.flags & F_EMPTY) && (r.flags & F_LAST)) { mark(xout[l + 1][i]); xout_n[l + 1]++; }
        break;
      case 106:   // a tcgen05 down unit reads the SwiGLU outputs of its expert's pairs
        if (moe_share_n[l] < n_ctas) return false;
        down_n[l]++;
        break;
      case 107:   // the slots of the block's own rows: every down unit, and its own x rows
        if (down_n[l] < (int)act[l].size() * nrb) return false;
        if (!(r.flags & F_EMPTY)) {
          if (!orows_ready(l, hlo[i], hhi[i])) return false;
          mark(xout[l + 1][i]);
          xout_n[l + 1]++;
        }
        break;
      case 102:
      case 105:
        break;
      case 104:   // this block's partial output is published
        moe_share_n[l]++;
        break;
      case 103:   // the reduction reads every block's partial and its own x rows
        if (!(r.flags & F_EMPTY)) {
          if (moe_share_n[l] < n_ctas || !orows_ready(l, hlo[i], hhi[i])) return false;
          mark(xout[l + 1][i]);
          xout_n[l + 1]++;
        }
        break;
      case MK_OP_HEAD:
        if (xout_n[L] < n_hrow_blocks) return false;
        break;
      case MK_OP_END:
        s.done = true;
        break;
      default:
        return false;
    }
    const int op = r.kind == 110 || r.kind >= 100 ? MK_OP_MOE : r.kind;
    out->tiles_run[op]++;
    s.qhead++;
    return true;
  };
  std::vector<int> order(2 * n_ctas);
  for (int i = 0; i < 2 * n_ctas; ++i) order[i] = i;
  int finished = 0;
  while (finished < n_ctas) {
    std::shuffle(order.begin(), order.end(), rng);
    bool progress = false;
    for (int k : order) {
      const int i = k >> 1;
      const bool ok = (k & 1) ? consume(i) : produce(i);
      if (ok) {
        progress = true;
        out->events++;
        if ((k & 1) && sm[i].done) finished++;
        break;
      }
    }
    if (!progress) { out->deadlocked = 1; break; }
  }
  out->finished = finished == n_ctas;
  // every writer ran exactly once
  bool ok = writes_twice == 0 && xout_n[0] == in.n_embed_tiles;
  for (int l = 0; l < L && ok; ++l) {
    int nq = 0, ni = 0;
    for (int i = 0; i < n_ctas; ++i) nq += qkv_done[l][i];
    for (int it = 0; it < n_items; ++it) ni += item_done[l][it];
    ok = nq == in.n_qkv_tiles && ni == n_items && merged_n[l] == n_item_blocks && oproj_n[l] == in.n_o_tiles &&
         router_n[l] == in.n_router_tiles && moe_share_n[l] == n_ctas && xout_n[l + 1] == n_hrow_blocks;
    for (int i = 0; i < n_ctas && ok; ++i) ok = routed[i][l] == 1;
  }
  out->writes_ok = ok;
  bool uok = true;
  for (int l = 0; l < L; ++l) {
    for (int v : gu_seen[l]) uok = uok && v == 1;
    for (int v : (small ? dt_seen[l] : dn_seen[l])) uok = uok && v == 1;
  }
  out->moe_units_ok = uok;
  return MK_OK;
}

}  // extern "C"
