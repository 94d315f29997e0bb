// Oracle: a plain, slow, obviously-correct CPU implementation of one decode
// step of the mixture-of-experts transformer that the persistent megakernel
// computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
// CPU-baseline leg of the benchmark are the only code allowed to load it.  It
// shares no code, header, table or constant with the CUDA path.
//
// What it follows ("Inside the megakernel serving engine for North Mini Code",
// Cohere, Sep 2026):
//   * section "What is a Megakernel?" -- the forward pass is "ordinary tiled
//     GEMMs and ordinary paged attention"; this file is the un-tiled, un-fused
//     definition of that same forward pass;
//   * intro / memory-bound paragraph -- a BF16 MoE model (30B total, 3.3B
//     active) decoded one token per sequence per step; weights are bf16;
//   * the serving-system paragraph -- paged attention over ragged sequence
//     lengths with per-sequence block tables;
//   * the "Image 2" paragraph -- attention work depends on live sequence
//     lengths and MoE work on routing.
// The op list (RMSNorm, fused QKV, RoPE, paged GQA attention, O-proj +
// residual, router softmax + top-k, SwiGLU experts, weighted combine, final
// norm, LM head) and the fp32-accumulation rule come from the problem
// statement the library implements; the pages do not spell them out.
//
// Readings where the pages are silent:
//   RMSNorm y = x * (1/sqrt(mean(x^2)+eps)) * g; NeoX rotate-half RoPE with
//   angles pos*theta^(-2i/D) evaluated in fp64 then cast to fp32; pos =
//   seq_len-1; k and v are rounded to bf16 (round-to-nearest-even) when
//   written to the cache and attention reads every position, the current one
//   included, back from the bf16 cache; GQA head h uses kv head h/(Hq/Hkv);
//   router: softmax over all experts, top-k by logit (ties to the lower expert
//   index; identical to top-k by probability because softmax is monotone),
//   weights renormalised over the k selected experts; silu(a) = a/(1+exp(-a));
//   the combine sums the k slots in rank order.
//
// Reduced-byte KV cache (dims.kv_q8 = 1; the Kinetic engine's pages, the
// --cache-type-k/v option and the paragraph on the quantized cache: keys and
// values kept as blocks of 32 int8 values with one f16 scale, 34 bytes where
// f16 takes 64, outputs close to but not equal to the full-precision cache's).
// The pages give no quantizer; the plain symmetric one is taken: per block of
// 32 consecutive values of one K or V row (along head_dim), d = max|x| / 127
// in fp32, stored rounded to f16 (nearest, ties to even); code q = x * (1/d)
// rounded to the nearest integer, ties away from zero (|q| <= 127); a block of
// zeros has d = 0 and codes 0.  A cached value reads back as q * d (exact in
// fp32).  Per layer the cache is a code plane [pages][2][Hkv][page_size][D]
// int8 followed by a scale plane [pages][2][Hkv][page_size][D/32] f16.
//
// Accumulation: every dot product and sum runs in ascending index order in
// the template type T.  The *_f32 entry points are the parity reference
// (fp32, as fixed by the problem statement); the *_f64 entry points run the
// same steps in double and are used by the self-checks.  Build with
// -ffp-contract=off so that x86 and Arm builds round identically.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

extern "C" {

struct orc_dims {
  int32_t layers, hidden, n_q, n_kv, head_dim, n_exp, top_k, ffn, vocab;
  int32_t page_size, num_pages, max_pages_per_seq, norm_topk, kv_q8;   // kv_q8: 0 bf16 cache, 1 q8_0 cache
  double rope_theta, rms_eps;
};

struct orc_layer {
  const uint16_t* attn_norm;   // [H]
  const uint16_t* w_qkv;       // [(Hq+2Hkv)*D, H]; rows: q heads, k heads, v heads
  const uint16_t* w_o;         // [H, Hq*D]
  const uint16_t* ffn_norm;    // [H]
  const uint16_t* w_router;    // [E, H]
  const float* router_bias;    // [E] or null
  const uint16_t* w_gate_up;   // [E, 2F, H] (gate rows then up rows) or null
  const uint16_t* w_down;      // [E, H, F] or null
};

}  // extern "C"

namespace {

inline float bf16_to_f32(uint16_t u) {
  uint32_t bits = static_cast<uint32_t>(u) << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

// fp32 -> bf16, round to nearest, ties to even (NaN kept quiet).
inline uint16_t f32_to_bf16(float f) {
  uint32_t bits;
  std::memcpy(&bits, &f, 4);
  if ((bits & 0x7f800000u) == 0x7f800000u && (bits & 0x007fffffu)) return static_cast<uint16_t>((bits >> 16) | 0x40);
  uint32_t lsb = (bits >> 16) & 1u;
  bits += 0x7fffu + lsb;
  return static_cast<uint16_t>(bits >> 16);
}

// fp32 -> IEEE binary16, round to nearest, ties to even (subnormals and overflow to inf handled).
inline uint16_t f32_to_f16(float f) {
  uint32_t x;
  std::memcpy(&x, &f, 4);
  const uint32_t sign = (x >> 16) & 0x8000u;
  const uint32_t ax = x & 0x7fffffffu;
  if (ax >= 0x7f800000u) return static_cast<uint16_t>(sign | (ax > 0x7f800000u ? 0x7e00u : 0x7c00u));
  const int e = static_cast<int>(ax >> 23) - 127;     // unbiased exponent
  if (e > 15) return static_cast<uint16_t>(sign | 0x7c00u);
  uint32_t mant = (ax & 0x7fffffu) | 0x800000u;       // 24-bit significand with the hidden bit
  int shift;                                          // bits of the 24-bit significand dropped
  uint32_t base;                                      // exponent field of the result
  if (e >= -14) { shift = 13; base = static_cast<uint32_t>(e + 15) << 10; mant &= 0x7fffffu; mant |= 0x800000u; }
  else {
    if (e < -25) return static_cast<uint16_t>(sign);  // below half the smallest subnormal
    shift = 13 + (-14 - e);
    base = 0;
  }
  uint32_t q = mant >> shift;
  const uint32_t rem = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) ++q;
  // normal: q holds the hidden bit at 2^10; adding base - (1 << 10) keeps a carry into the exponent
  const uint32_t h = e >= -14 ? base + q - 0x400u : q;
  return static_cast<uint16_t>(sign | h);
}

inline float f16_to_f32(uint16_t h) {
  const uint32_t sign = static_cast<uint32_t>(h & 0x8000u) << 16;
  const uint32_t ex = (h >> 10) & 0x1fu, man = h & 0x3ffu;
  float f;
  if (ex == 0) {
    f = std::ldexp(static_cast<float>(man), -24);   // zero or subnormal: man * 2^-24
    uint32_t b;
    std::memcpy(&b, &f, 4);
    b |= sign;
    std::memcpy(&f, &b, 4);
    return f;
  }
  uint32_t b = ex == 31 ? (sign | 0x7f800000u | (man << 13)) : (sign | ((ex + 112u) << 23) | (man << 13));
  std::memcpy(&f, &b, 4);
  return f;
}

// One q8_0 block: 32 fp32 values -> 32 codes and the f16 scale (see the reading above).
inline void q8_quantize_block(const float* x, int8_t* q, uint16_t* d_f16) {
  float amax = 0.f;
  for (int i = 0; i < 32; ++i) amax = std::fabs(x[i]) > amax ? std::fabs(x[i]) : amax;
  const float d = amax / 127.0f;
  const float id = d != 0.f ? 1.0f / d : 0.f;
  for (int i = 0; i < 32; ++i) q[i] = static_cast<int8_t>(std::round(x[i] * id));
  *d_f16 = f32_to_f16(d);
}

template <typename T> inline T texp(T v);
template <> inline float texp<float>(float v) { return std::exp(v); }
template <> inline double texp<double>(double v) { return std::exp(v); }
template <typename T> inline T tsqrt(T v);
template <> inline float tsqrt<float>(float v) { return std::sqrt(v); }
template <> inline double tsqrt<double>(double v) { return std::sqrt(v); }

// y[r] = sum_c W[r,c] * x[c]; W row-major bf16 [rows, cols].
template <typename T>
void gemv(int rows, int cols, const uint16_t* W, const T* x, T* y) {
#pragma omp parallel for schedule(static) if (static_cast<long>(rows) * cols > 65536)
  for (int r = 0; r < rows; ++r) {
    const uint16_t* w = W + static_cast<size_t>(r) * cols;
    T acc = 0;
    for (int c = 0; c < cols; ++c) acc += static_cast<T>(bf16_to_f32(w[c])) * x[c];
    y[r] = acc;
  }
}

template <typename T>
void rmsnorm(int n, const T* x, const uint16_t* g, double eps, T* y) {
  T ss = 0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  T rstd = static_cast<T>(1) / tsqrt<T>(ss / static_cast<T>(n) + static_cast<T>(eps));
  for (int i = 0; i < n; ++i) y[i] = (x[i] * rstd) * static_cast<T>(bf16_to_f32(g[i]));
}

// NeoX rotate-half: pairs (i, i + D/2), angle pos * theta^(-2i/D) in fp64,
// cos/sin rounded to fp32 before use.
template <typename T>
void rope(int D, int pos, double theta, T* v) {
  const int half = D / 2;
  for (int i = 0; i < half; ++i) {
    double ang = static_cast<double>(pos) * std::pow(theta, -2.0 * i / D);
    T c = static_cast<T>(static_cast<float>(std::cos(ang)));
    T s = static_cast<T>(static_cast<float>(std::sin(ang)));
    T a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

template <typename T>
void softmax(int n, const T* r, T* p) {
  T m = r[0];
  for (int i = 1; i < n; ++i) m = r[i] > m ? r[i] : m;
  T z = 0;
  for (int i = 0; i < n; ++i) { p[i] = texp<T>(r[i] - m); z += p[i]; }
  for (int i = 0; i < n; ++i) p[i] = p[i] / z;
}

// Indices of the k largest r, in descending order; equal values -> lower index first.
template <typename T>
void topk(int n, int k, const T* r, int32_t* ids) {
  std::vector<char> taken(n, 0);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int i = 0; i < n; ++i) {
      if (taken[i]) continue;
      if (best < 0 || r[i] > r[best]) best = i;
    }
    taken[best] = 1;
    ids[j] = best;
  }
}

inline size_t kv_offset(const orc_dims& d, int page, int which, int kvh, int slot) {
  // per-layer cache layout [num_pages][2 (K,V)][Hkv][page_size][D] (elements of the bf16 cache,
  // codes of the q8_0 cache)
  return ((((static_cast<size_t>(page) * 2 + which) * d.n_kv + kvh) * d.page_size + slot) * d.head_dim);
}

// Bytes of one layer of the cache.
inline size_t kv_layer_bytes(const orc_dims& d) {
  const size_t n = static_cast<size_t>(d.num_pages) * 2 * d.n_kv * d.page_size * d.head_dim;
  return d.kv_q8 ? n + n / 32 * 2 : n * 2;
}

// One layer of the cache, in either format: rows are written from fp32 values (rounded to bf16,
// or quantized block by block) and read back element by element as fp32.
struct KvLayer {
  const orc_dims& d;
  uint16_t* bf = nullptr;     // bf16 cache
  int8_t* codes = nullptr;    // q8_0 code plane
  uint16_t* scales = nullptr; // q8_0 scale plane (f16 bits)
  KvLayer(const orc_dims& d_, void* base) : d(d_) {
    if (d.kv_q8) {
      codes = static_cast<int8_t*>(base);
      scales = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(base) +
                                           static_cast<size_t>(d.num_pages) * 2 * d.n_kv * d.page_size * d.head_dim);
    } else {
      bf = static_cast<uint16_t*>(base);
    }
  }
  float get(int page, int which, int kvh, int slot, int i) const {
    const size_t o = kv_offset(d, page, which, kvh, slot);
    if (bf) return bf16_to_f32(bf[o + i]);
    return static_cast<float>(codes[o + i]) * f16_to_f32(scales[o / 32 + i / 32]);
  }
  void put(int page, int which, int kvh, int slot, const float* v) {
    const size_t o = kv_offset(d, page, which, kvh, slot);
    if (bf) {
      for (int i = 0; i < d.head_dim; ++i) bf[o + i] = f32_to_bf16(v[i]);
      return;
    }
    for (int b = 0; b < d.head_dim / 32; ++b) q8_quantize_block(v + 32 * b, codes + o + 32 * b, scales + o / 32 + b);
  }
};

// append = false: the cache already holds the current token's k and v at position
// seq_len-1 (codes another implementation wrote); they are read, not recomputed, so a check
// of the attention can use the same bf16 codes as the implementation it checks.
template <typename T>
int attn_block(const orc_dims& d, const orc_layer& w, int B, T* x, const int32_t* seq_lens,
               const int32_t* bt, uint16_t* kv, T* trace_qkv, T* trace_attn, bool append = true) {
  const int H = d.hidden, D = d.head_dim, Hq = d.n_q, Hkv = d.n_kv, G = Hq / Hkv;
  if (d.kv_q8 && D % 32) return -4;
  KvLayer cache(d, kv);
  std::vector<float> row(D);
  const int NQKV = (Hq + 2 * Hkv) * D;
  const T scale = static_cast<T>(1) / tsqrt<T>(static_cast<T>(D));
  std::vector<T> y(H), qkv(NQKV), attn(static_cast<size_t>(Hq) * D), o(H);
  for (int b = 0; b < B; ++b) {
    const int Lc = seq_lens[b];
    if (Lc < 1 || Lc > d.max_pages_per_seq * d.page_size) return -1;
    const int pos = Lc - 1;
    T* xb = x + static_cast<size_t>(b) * H;
    const int32_t* tab = bt + static_cast<size_t>(b) * d.max_pages_per_seq;
    rmsnorm<T>(H, xb, w.attn_norm, d.rms_eps, y.data());
    gemv<T>(NQKV, H, w.w_qkv, y.data(), qkv.data());
    if (trace_qkv) std::memcpy(trace_qkv + static_cast<size_t>(b) * NQKV, qkv.data(), sizeof(T) * NQKV);
    for (int h = 0; h < Hq + Hkv; ++h) rope<T>(D, pos, d.rope_theta, qkv.data() + static_cast<size_t>(h) * D);
    // append the current token's k and v to the cache (rounded to bf16, or quantized to q8_0, from
    // their fp32 values)
    const int page = tab[pos / d.page_size], slot = pos % d.page_size;
    if (page < 0 || page >= d.num_pages) return -2;
    for (int g = 0; g < Hkv && append; ++g) {
      const T* kg = qkv.data() + static_cast<size_t>(Hq + g) * D;
      const T* vg = qkv.data() + static_cast<size_t>(Hq + Hkv + g) * D;
      for (int i = 0; i < D; ++i) row[i] = static_cast<float>(kg[i]);
      cache.put(page, 0, g, slot, row.data());
      for (int i = 0; i < D; ++i) row[i] = static_cast<float>(vg[i]);
      cache.put(page, 1, g, slot, row.data());
    }
    // attention: every q head over positions 0..Lc-1, read from the paged cache
#pragma omp parallel for schedule(static) if (static_cast<long>(Lc) * Hq > 4096)
    for (int h = 0; h < Hq; ++h) {
      const int g = h / G;
      const T* q = qkv.data() + static_cast<size_t>(h) * D;
      std::vector<T> s(Lc), acc(D, static_cast<T>(0));
      for (int t = 0; t < Lc; ++t) {
        const int pg = tab[t / d.page_size], sl = t % d.page_size;
        T dot = 0;
        for (int i = 0; i < D; ++i) dot += q[i] * static_cast<T>(cache.get(pg, 0, g, sl, i));
        s[t] = dot * scale;
      }
      T m = s[0];
      for (int t = 1; t < Lc; ++t) m = s[t] > m ? s[t] : m;
      T l = 0;
      for (int t = 0; t < Lc; ++t) { s[t] = texp<T>(s[t] - m); l += s[t]; }
      for (int t = 0; t < Lc; ++t) {
        const int pg = tab[t / d.page_size], sl = t % d.page_size;
        for (int i = 0; i < D; ++i) acc[i] += s[t] * static_cast<T>(cache.get(pg, 1, g, sl, i));
      }
      for (int i = 0; i < D; ++i) attn[static_cast<size_t>(h) * D + i] = acc[i] / l;
    }
    if (trace_attn) std::memcpy(trace_attn + static_cast<size_t>(b) * Hq * D, attn.data(), sizeof(T) * Hq * D);
    gemv<T>(H, Hq * D, w.w_o, attn.data(), o.data());
    for (int i = 0; i < H; ++i) xb[i] = xb[i] + o[i];
  }
  return 0;
}

template <typename T>
void route(const orc_dims& d, const orc_layer& w, int B, const T* x, T* y_out, T* logits_out,
           int32_t* ids_out, T* w_out) {
  const int H = d.hidden, E = d.n_exp, K = d.top_k;
  std::vector<T> p(E);
  for (int b = 0; b < B; ++b) {
    T* y = y_out + static_cast<size_t>(b) * H;
    T* r = logits_out + static_cast<size_t>(b) * E;
    rmsnorm<T>(H, x + static_cast<size_t>(b) * H, w.ffn_norm, d.rms_eps, y);
    gemv<T>(E, H, w.w_router, y, r);
    if (w.router_bias)
      for (int e = 0; e < E; ++e) r[e] = r[e] + static_cast<T>(w.router_bias[e]);
    softmax<T>(E, r, p.data());
    int32_t* ids = ids_out + static_cast<size_t>(b) * K;
    topk<T>(E, K, r, ids);
    T* wb = w_out + static_cast<size_t>(b) * K;
    T z = 0;
    for (int j = 0; j < K; ++j) z += p[ids[j]];
    for (int j = 0; j < K; ++j) wb[j] = d.norm_topk ? p[ids[j]] / z : p[ids[j]];
  }
}

template <typename T>
void moe(const orc_dims& d, int B, const T* y_in, const int32_t* ids, const T* wts,
         const uint16_t* const* gate_up, const uint16_t* const* down, T* x, T* trace_h, T* trace_out) {
  (void)ids;
  const int H = d.hidden, F = d.ffn, K = d.top_k;
  std::vector<T> gu(2 * static_cast<size_t>(F)), h(F), yj(H), out(H);
  for (int b = 0; b < B; ++b) {
    const T* y = y_in + static_cast<size_t>(b) * H;
    for (int i = 0; i < H; ++i) out[i] = 0;
    for (int j = 0; j < K; ++j) {
      const size_t slot = static_cast<size_t>(b) * K + j;
      gemv<T>(2 * F, H, gate_up[slot], y, gu.data());
      for (int f = 0; f < F; ++f) {
        T a = gu[f];
        T silu = a / (static_cast<T>(1) + texp<T>(-a));
        h[f] = silu * gu[F + f];
      }
      if (trace_h) std::memcpy(trace_h + slot * F, h.data(), sizeof(T) * F);
      gemv<T>(H, F, down[slot], h.data(), yj.data());
      for (int i = 0; i < H; ++i) out[i] += wts[slot] * yj[i];
    }
    if (trace_out) std::memcpy(trace_out + static_cast<size_t>(b) * H, out.data(), sizeof(T) * H);
    T* xb = x + static_cast<size_t>(b) * H;
    for (int i = 0; i < H; ++i) xb[i] = xb[i] + out[i];
  }
}

template <typename T>
void embed(const orc_dims& d, const uint16_t* table, int B, const int32_t* tokens, T* x) {
  for (int b = 0; b < B; ++b) {
    const uint16_t* row = table + static_cast<size_t>(tokens[b]) * d.hidden;
    for (int i = 0; i < d.hidden; ++i) x[static_cast<size_t>(b) * d.hidden + i] = static_cast<T>(bf16_to_f32(row[i]));
  }
}

template <typename T>
void final_head(const orc_dims& d, const uint16_t* final_norm, const uint16_t* lm_head, int B, const T* x, T* logits) {
  std::vector<T> y(d.hidden);
  for (int b = 0; b < B; ++b) {
    rmsnorm<T>(d.hidden, x + static_cast<size_t>(b) * d.hidden, final_norm, d.rms_eps, y.data());
    gemv<T>(d.vocab, d.hidden, lm_head, y.data(), logits + static_cast<size_t>(b) * d.vocab);
  }
}

template <typename T>
int decode_step(const orc_dims& d, const uint16_t* emb, const orc_layer* layers, const uint16_t* final_norm,
                const uint16_t* lm_head, int B, const int32_t* tokens, const int32_t* seq_lens, const int32_t* bt,
                uint16_t* kv, T* logits) {
  const int H = d.hidden, K = d.top_k, F = d.ffn, E = d.n_exp;
  for (int b = 0; b < B; ++b)
    if (tokens[b] < 0 || tokens[b] >= d.vocab) return -3;
  std::vector<T> x(static_cast<size_t>(B) * H), y(static_cast<size_t>(B) * H), r(static_cast<size_t>(B) * E),
      wts(static_cast<size_t>(B) * K);
  std::vector<int32_t> ids(static_cast<size_t>(B) * K);
  std::vector<const uint16_t*> gu(static_cast<size_t>(B) * K), dn(static_cast<size_t>(B) * K);
  embed<T>(d, emb, B, tokens, x.data());
  const size_t layer_bytes = kv_layer_bytes(d);
  for (int l = 0; l < d.layers; ++l) {
    const orc_layer& w = layers[l];
    uint16_t* kvl = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(kv) + l * layer_bytes);
    int rc = attn_block<T>(d, w, B, x.data(), seq_lens, bt, kvl, nullptr, nullptr);
    if (rc) return rc;
    route<T>(d, w, B, x.data(), y.data(), r.data(), ids.data(), wts.data());
    for (size_t s = 0; s < gu.size(); ++s) {
      gu[s] = w.w_gate_up + static_cast<size_t>(ids[s]) * 2 * F * H;
      dn[s] = w.w_down + static_cast<size_t>(ids[s]) * H * F;
    }
    moe<T>(d, B, y.data(), ids.data(), wts.data(), gu.data(), dn.data(), x.data(), nullptr, nullptr);
  }
  final_head<T>(d, final_norm, lm_head, B, x.data(), logits);
  return 0;
}

}  // namespace

extern "C" {

uint16_t orc_f32_to_bf16(float f) { return f32_to_bf16(f); }
float orc_bf16_to_f32(uint16_t u) { return bf16_to_f32(u); }
uint16_t orc_f32_to_f16(float f) { return f32_to_f16(f); }
float orc_f16_to_f32(uint16_t h) { return f16_to_f32(h); }
// n blocks of 32 values -> n * 32 codes and n f16 scales
void orc_q8_quantize(int n, const float* x, int8_t* q, uint16_t* d) {
  for (int b = 0; b < n; ++b) q8_quantize_block(x + 32 * b, q + 32 * b, d + b);
}

#define ORC_EXPORT_ALL(SUF, T)                                                                                     \
  void orc_gemv_##SUF(int rows, int cols, const uint16_t* W, const T* x, T* y) { gemv<T>(rows, cols, W, x, y); }  \
  void orc_rmsnorm_##SUF(int n, const T* x, const uint16_t* g, double eps, T* y) { rmsnorm<T>(n, x, g, eps, y); } \
  void orc_rope_##SUF(int D, int pos, double theta, T* v) { rope<T>(D, pos, theta, v); }                          \
  void orc_softmax_##SUF(int n, const T* r, T* p) { softmax<T>(n, r, p); }                                        \
  void orc_topk_##SUF(int n, int k, const T* r, int32_t* ids) { topk<T>(n, k, r, ids); }                          \
  void orc_embed_##SUF(const orc_dims* d, const uint16_t* table, int B, const int32_t* tok, T* x) {               \
    embed<T>(*d, table, B, tok, x);                                                                               \
  }                                                                                                               \
  int orc_attn_block_##SUF(const orc_dims* d, const orc_layer* w, int B, T* x, const int32_t* seq_lens,           \
                           const int32_t* bt, uint16_t* kv_layer, T* trace_qkv, T* trace_attn, int append) {      \
    return attn_block<T>(*d, *w, B, x, seq_lens, bt, kv_layer, trace_qkv, trace_attn, append != 0);               \
  }                                                                                                               \
  void orc_route_##SUF(const orc_dims* d, const orc_layer* w, int B, const T* x, T* y, T* logits, int32_t* ids,  \
                       T* wts) {                                                                                  \
    route<T>(*d, *w, B, x, y, logits, ids, wts);                                                                  \
  }                                                                                                               \
  void orc_moe_##SUF(const orc_dims* d, int B, const T* y, const int32_t* ids, const T* wts,                      \
                     const uint16_t* const* gate_up, const uint16_t* const* down, T* x, T* trace_h,               \
                     T* trace_out) {                                                                              \
    moe<T>(*d, B, y, ids, wts, gate_up, down, x, trace_h, trace_out);                                             \
  }                                                                                                               \
  void orc_final_##SUF(const orc_dims* d, const uint16_t* fn, const uint16_t* head, int B, const T* x, T* lg) {   \
    final_head<T>(*d, fn, head, B, x, lg);                                                                        \
  }                                                                                                               \
  int orc_decode_step_##SUF(const orc_dims* d, const uint16_t* emb, const orc_layer* layers, const uint16_t* fn, \
                            const uint16_t* head, int B, const int32_t* tok, const int32_t* seq_lens,            \
                            const int32_t* bt, uint16_t* kv, T* logits) {                                         \
    return decode_step<T>(*d, emb, layers, fn, head, B, tok, seq_lens, bt, kv, logits);                           \
  }

ORC_EXPORT_ALL(f32, float)
ORC_EXPORT_ALL(f64, double)

}  // extern "C"
