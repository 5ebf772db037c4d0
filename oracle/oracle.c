/*
 * oracle.c — plain, slow, obviously-correct CPU reference for the batch-1
 * block-quantized Llama decode step.  TEST INFRASTRUCTURE ONLY: the tests,
 * the smoke check and the benchmark's CPU-baseline leg call it; the product
 * path never does.  It shares no code with the CUDA library.
 *
 * Sources (page title, then section):
 *  [P-about]  "Ntransformer" (en.unwiki.net), About — GGUF model format with
 *             Q4_0, Q8_0, Q4_K_M, Q5_K, Q6_K, F16 and F32 quantisation.
 *  [P-feat]   "ntransformer - moteur d'inférence NVMe-to-GPU…" (fr.news.hada.io),
 *             "Fonctionnalités principales" — Llama architecture: RoPE, GQA,
 *             SwiGLU, RMSNorm, KV cache; self-speculative decoding that uses
 *             the VRAM-resident layers as the draft.
 *  [P-code]   same page, "Architecture et structure du code" — cuda/: GEMV,
 *             RMSNorm, RoPE, SwiGLU, softmax kernels; model/: transformer
 *             composition, attention, FFN, normalisation; inference/: sampler.
 *  [P-cache]  same page, "Performances et structure de cache" — layer skip by
 *             cosine similarity, 20 of 80 layers.
 *  [P-road]   "Ntransformer" (en.unwiki.net), roadmap — F16 KV cache.
 *
 * The pages name the block formats but do not define their bytes; the layouts
 * below are the public GGUF block convention (a reading, listed in the design
 * notes).  Closed forms for the element values:
 *   Q8_0  v = d*q                      (32 per block, int8 q)
 *   Q4_0  v = d*(q-8)                  (32 per block, 4-bit q)
 *   Q4_K  v = d*sc*q - dmin*m          (256 per block, 8 sub-blocks of 32)
 *   Q5_K  same as Q4_K with 5-bit q
 *   Q6_K  v = d*sc*(q-32)              (256 per block, 16 sub-blocks of 16)
 *
 * Precision: dequantised weights are produced in fp32 with the operation order
 * below (each product exact, at most one rounding), every other quantity is
 * fp64.  The KV cache is stored as binary16: fp64 -> fp32 -> f16 (RNE).
 *
 * Parity pins for every function live in tests/test_oracle_*.py.  Parity
 * unpinned: that the block layouts match real GGUF files byte for byte (no
 * such file is available; the golden blocks pin the reading, not the files),
 * and the quality of layer skip (the pages give no measure of it).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_Q8_0 = 0, OR_Q4_0 = 1, OR_Q4_K = 2, OR_Q5_K = 3, OR_Q6_K = 4, OR_F16 = 5, OR_F32 = 6 };

int or_block_elems(int fmt) {
  switch (fmt) {
    case OR_Q8_0: case OR_Q4_0: case OR_F16: case OR_F32: return 32;  /* F16/F32: 32 plain values */
    case OR_Q4_K: case OR_Q5_K: case OR_Q6_K: return 256;
    default: return 0;
  }
}

int or_block_bytes(int fmt) {
  switch (fmt) {
    case OR_Q8_0: return 2 + 32;             /* d, qs[32]                      */
    case OR_Q4_0: return 2 + 16;             /* d, qs[16]                      */
    case OR_Q4_K: return 2 + 2 + 12 + 128;   /* d, dmin, scales[12], qs[128]   */
    case OR_Q5_K: return 2 + 2 + 12 + 32 + 128; /* + qh[32]                    */
    case OR_Q6_K: return 128 + 64 + 16 + 2;  /* ql[128], qh[64], sc[16], d     */
    case OR_F16: return 32 * 2;              /* binary16 values                */
    case OR_F32: return 32 * 4;              /* binary32 values                */
    default: return 0;
  }
}

/* ---- binary16 <-> binary64 from the IEEE-754 bit layout ----------------- */
double or_half_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, f = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)f, -24);                       /* subnormal */
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp(1.0 + (double)f / 1024.0, e - 15);
  return s ? -v : v;
}

/* fp32 value -> binary16 bits, round to nearest even (input already fp32) */
uint16_t or_float_to_half(float xf) {
  double x = (double)xf;
  uint16_t s = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x);
  if (isnan(a)) return (uint16_t)(s | 0x7E00u);
  if (a >= 65520.0) return (uint16_t)(s | 0x7C00u);
  if (a < ldexp(1.0, -14)) {                 /* result subnormal (or rounds up to min normal) */
    double k = nearbyint(ldexp(a, 24));
    return (uint16_t)(s | (uint16_t)k);
  }
  int e;
  frexp(a, &e);
  int E = e - 1;
  double f = nearbyint((ldexp(a, -E) - 1.0) * 1024.0);
  if (f >= 1024.0) { f = 0.0; E++; }
  if (E > 15) return (uint16_t)(s | 0x7C00u);
  return (uint16_t)(s | (uint16_t)((E + 15) << 10) | (uint16_t)f);
}

static float half_f(const uint8_t* p) { return (float)or_half_to_double((uint16_t)(p[0] | (p[1] << 8))); }

/* K-quant sub-block j (0..7) scale and min, each 6 bits, from scales[12] */
void or_kquant_scale_min(const uint8_t* s, int j, int* sc, int* m) {
  if (j < 4) {
    *sc = s[j] & 63;
    *m = s[j + 4] & 63;
  } else {
    *sc = (s[j + 4] & 0x0F) | ((s[j - 4] >> 6) << 4);
    *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
  }
}

/* integer quant of element i of one block (for the K formats: 0..15 / 0..31 / 0..63) */
int or_quant_of(int fmt, const uint8_t* b, int i) {
  switch (fmt) {
    case OR_Q8_0: return (int)(int8_t)b[2 + i];
    case OR_Q4_0: return i < 16 ? (b[2 + i] & 0x0F) : (b[2 + i - 16] >> 4);
    case OR_Q4_K: {
      const uint8_t* qs = b + 16;
      int j = i / 32, l = i % 32, c = j / 2;
      return (j & 1) ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 0x0F);
    }
    case OR_Q5_K: {
      const uint8_t* qh = b + 16;
      const uint8_t* qs = b + 48;
      int j = i / 32, l = i % 32, c = j / 2;
      int lo = (j & 1) ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 0x0F);
      int hi = (qh[l] >> j) & 1;
      return lo | (hi << 4);
    }
    case OR_Q6_K: {
      const uint8_t* ql = b;
      const uint8_t* qh = b + 128;
      int h = i / 128, e = i % 128, g = e / 32, l = e % 32;
      const uint8_t* qlh = ql + 64 * h;
      const uint8_t* qhh = qh + 32 * h;
      int lo;
      switch (g) {
        case 0: lo = qlh[l] & 0x0F; break;
        case 1: lo = qlh[l + 32] & 0x0F; break;
        case 2: lo = qlh[l] >> 4; break;
        default: lo = qlh[l + 32] >> 4; break;
      }
      int hi = (qhh[l] >> (2 * g)) & 3;
      return lo | (hi << 4);
    }
    default: return 0;
  }
}

/* Dequantise one block to fp32 (closed forms above, order chosen so that each
 * product is exact in fp32 and at most one rounding happens). */
void or_dequant_block(int fmt, const uint8_t* b, float* out) {
  switch (fmt) {
    case OR_Q8_0: {
      float d = half_f(b);
      for (int i = 0; i < 32; ++i) out[i] = d * (float)or_quant_of(fmt, b, i);
      break;
    }
    case OR_Q4_0: {
      float d = half_f(b);
      for (int i = 0; i < 32; ++i) out[i] = d * (float)(or_quant_of(fmt, b, i) - 8);
      break;
    }
    case OR_Q4_K:
    case OR_Q5_K: {
      float d = half_f(b), dmin = half_f(b + 2);
      for (int i = 0; i < 256; ++i) {
        int sc, m;
        or_kquant_scale_min(b + 4, i / 32, &sc, &m);
        float a = d * (float)sc;       /* exact: 11-bit x 6-bit */
        float bq = a * (float)or_quant_of(fmt, b, i); /* exact: <= 22 bits */
        float c = dmin * (float)m;     /* exact */
        out[i] = bq - c;               /* the one rounding */
      }
      break;
    }
    case OR_Q6_K: {
      float d = half_f(b + 208);
      const int8_t* sc = (const int8_t*)(b + 192);
      for (int i = 0; i < 256; ++i) {
        int s = sc[(i / 128) * 8 + (i % 128) / 16];
        int q = or_quant_of(fmt, b, i) - 32;
        out[i] = d * (float)(s * q);   /* |s*q| <= 4096: exact product */
      }
      break;
    }
    case OR_F16:   /* every binary16 value is exact in fp32 */
      for (int i = 0; i < 32; ++i) out[i] = half_f(b + 2 * i);
      break;
    case OR_F32: { /* little-endian binary32 */
      for (int i = 0; i < 32; ++i) {
        uint32_t u = (uint32_t)b[4 * i] | ((uint32_t)b[4 * i + 1] << 8) | ((uint32_t)b[4 * i + 2] << 16) |
                     ((uint32_t)b[4 * i + 3] << 24);
        memcpy(&out[i], &u, 4);
      }
      break;
    }
    default: break;
  }
}

/* Dequantise `nrows` rows starting at row0 of a rows x cols matrix (fp32). */
int or_dequant_rows(int fmt, const uint8_t* W, int64_t row0, int64_t nrows, int64_t cols, float* out) {
  int be = or_block_elems(fmt), bb = or_block_bytes(fmt);
  if (!be || cols % be) return -1;
  int64_t nb = cols / be;
  for (int64_t r = 0; r < nrows; ++r)
    for (int64_t k = 0; k < nb; ++k)
      or_dequant_block(fmt, W + ((row0 + r) * nb + k) * bb, out + r * cols + k * be);
  return 0;
}

/* y[r] = sum_c w[r,c] * x[c], accumulated in fp64 in column order.
 * [P-code] cuda/ GEMV; [P-about] quantised formats.  residual (nullable) is
 * added after the sum: y = W x + residual. */
int or_gemv(int fmt, const uint8_t* W, const double* x, double* y, int64_t rows, int64_t cols,
            const double* residual) {
  int be = or_block_elems(fmt), bb = or_block_bytes(fmt);
  if (!be || cols % be) return -1;
  int64_t nb = cols / be;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t r = 0; r < rows; ++r) {
    float w[256];
    double acc = 0.0;
    for (int64_t k = 0; k < nb; ++k) {
      or_dequant_block(fmt, W + (r * nb + k) * bb, w);
      for (int i = 0; i < be; ++i) acc += (double)w[i] * x[k * be + i];
    }
    y[r] = acc + (residual ? residual[r] : 0.0);
  }
  return 0;
}

/* y = x / sqrt(mean(x^2) + eps) * g   ([P-feat] RMSNorm) */
void or_rmsnorm(const double* x, const float* g, int64_t n, double eps, double* y) {
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int64_t i = 0; i < n; ++i) y[i] = x[i] * inv * (double)g[i];
}

/* Rotary embedding on adjacent pairs (2i, 2i+1) of every head at position pos:
 * angle_i = pos * theta^(-2i/head_dim)   ([P-feat] RoPE) */
void or_rope(double* v, int n_heads, int head_dim, int64_t pos, double theta) {
  for (int i = 0; i < head_dim / 2; ++i) {
    double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)head_dim);
    double c = cos(ang), s = sin(ang);
    for (int h = 0; h < n_heads; ++h) {
      double* p = v + (int64_t)h * head_dim + 2 * i;
      double a = p[0], b = p[1];
      p[0] = a * c - b * s;
      p[1] = a * s + b * c;
    }
  }
}

/* numerically stable softmax in place: exp(s - max) / sum   ([P-code] softmax) */
void or_softmax(double* s, int64_t n) {
  if (n <= 0) return;
  double m = s[0];
  for (int64_t i = 1; i < n; ++i) m = s[i] > m ? s[i] : m;
  double z = 0.0;
  for (int64_t i = 0; i < n; ++i) { s[i] = exp(s[i] - m); z += s[i]; }
  for (int64_t i = 0; i < n; ++i) s[i] /= z;
}

/* Decode attention with grouped KV heads ([P-feat] GQA, [P-road] F16 KV):
 * q head h reads KV head h / (n_qh / n_kvh); scores q.K_j / sqrt(head_dim)
 * over cached positions j < n_pos; out = softmax(scores) . V.
 * Kc, Vc: binary16 bits laid out [n_kvh][kv_stride][head_dim]. */
int or_attn_decode(const double* q, const uint16_t* Kc, const uint16_t* Vc, double* out, int n_qh, int n_kvh,
                   int head_dim, int64_t n_pos, int64_t kv_stride) {
  if (n_kvh <= 0 || n_qh % n_kvh || n_pos <= 0 || n_pos > kv_stride) return -1;
  int grp = n_qh / n_kvh;
  double* s = (double*)malloc(sizeof(double) * (size_t)n_pos);
  if (!s) return -1;
  double scale = 1.0 / sqrt((double)head_dim);
  for (int h = 0; h < n_qh; ++h) {
    int g = h / grp;
    const uint16_t* K = Kc + (int64_t)g * kv_stride * head_dim;
    const uint16_t* V = Vc + (int64_t)g * kv_stride * head_dim;
    const double* qh = q + (int64_t)h * head_dim;
    for (int64_t j = 0; j < n_pos; ++j) {
      double dot = 0.0;
      for (int d = 0; d < head_dim; ++d) dot += qh[d] * or_half_to_double(K[j * head_dim + d]);
      s[j] = dot * scale;
    }
    or_softmax(s, n_pos);
    for (int d = 0; d < head_dim; ++d) {
      double acc = 0.0;
      for (int64_t j = 0; j < n_pos; ++j) acc += s[j] * or_half_to_double(V[j * head_dim + d]);
      out[(int64_t)h * head_dim + d] = acc;
    }
  }
  free(s);
  return 0;
}

/* silu(z) = z / (1 + e^-z); SwiGLU h = silu(gate) * up   ([P-feat] SwiGLU) */
double or_silu(double z) { return z / (1.0 + exp(-z)); }

void or_swiglu(const double* gate, const double* up, double* h, int64_t n) {
  for (int64_t i = 0; i < n; ++i) h[i] = or_silu(gate[i]) * up[i];
}

/* greedy sampler: index of the largest value, lowest index on ties ([P-code] sampler) */
int64_t or_argmax(const double* v, int64_t n) {
  int64_t best = 0;
  for (int64_t i = 1; i < n; ++i)
    if (v[i] > v[best]) best = i;
  return best;
}

/* ---- non-greedy sampler ([P-code] inference/: sampler) --------------------
 * Reading: temperature softmax followed by nucleus (top-p) truncation, the
 * usual non-greedy decoding of a Llama engine.  Written out as the plain
 * definition:
 *   w_i   = rint(exp((z_i - max z) / T) * 2^40)   (token weights, integers)
 *   order = tokens by logit descending, ties by lower index
 *   N     = the shortest prefix of that order whose weight sum reaches
 *           target = ceil(top_p * sum_i w_i)
 *   pick  = with r = floor(u * sum_{N} w), the token of N, taken in index
 *           order, whose cumulative weight first exceeds r.
 * T <= 0 is greedy (argmax, lowest index).  Integer weights make every sum
 * exact and independent of the order of addition. */

/* SplitMix64 output function (Steele, Lea & Flood, OOPSLA 2014): the state
 * advanced by the golden-ratio increment, then two xor-shift-multiply steps. */
uint64_t or_splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* the sampler's uniform for (seed, counter): the top 24 bits of
 * splitmix64(seed xor 2 counter), as a multiple of 2^-24 in [0, 1) */
double or_sample_uniform(uint64_t seed, uint64_t counter) {
  return (double)(or_splitmix64(seed ^ (counter << 1)) >> 40) * 0x1.0p-24;
}

static const float* g_sort_z;  /* comparison context of the sort below */
static int cmp_desc(const void* a, const void* b) {
  int64_t i = *(const int64_t*)a, j = *(const int64_t*)b;
  float zi = g_sort_z[i], zj = g_sort_z[j];
  if (zi > zj) return -1;
  if (zi < zj) return 1;
  return (i > j) - (i < j);
}

/* the nucleus of the definition above: w[i] = token i's weight, in[i] = 1
 * for the nucleus tokens, *size = their count; returns the nucleus weight
 * sum_{N} w (0 when out of memory) */
static uint64_t nucleus(const float* z, int64_t n, double temperature, double top_p, uint64_t* w, uint8_t* in,
                        int64_t* size) {
  double mx = z[0];
  for (int64_t i = 1; i < n; ++i)
    if (z[i] > mx) mx = z[i];
  int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
  if (!idx) return 0;
  uint64_t Z = 0;
  for (int64_t i = 0; i < n; ++i) {
    w[i] = (uint64_t)nearbyint(exp(((double)z[i] - mx) / temperature) * 0x1.0p40);
    Z += w[i];
    idx[i] = i;
    in[i] = 0;
  }
  double t = ceil(top_p * (double)Z);
  uint64_t target = t < 1.0 ? 1 : (t > (double)Z ? Z : (uint64_t)t);
  g_sort_z = z;
  qsort(idx, (size_t)n, sizeof(int64_t), cmp_desc);
  uint64_t M = 0;
  int64_t k = 0;
  while (k < n && M < target) { M += w[idx[k]]; in[idx[k]] = 1; ++k; }
  free(idx);
  *size = k;
  return M;
}

int64_t or_sample(const float* z, int64_t n, double temperature, double top_p, double u, int64_t* nucleus_out) {
  if (n <= 0) return -1;
  if (temperature <= 0.0) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
      if (z[i] > z[best]) best = i;
    if (nucleus_out) *nucleus_out = 1;
    return best;
  }
  uint64_t* w = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)n);
  uint8_t* in = (uint8_t*)malloc((size_t)n);
  if (!w || !in) { free(w); free(in); return -2; }
  int64_t k = 0;
  const uint64_t M = nucleus(z, n, temperature, top_p, w, in, &k);
  if (!M) { free(w); free(in); return -2; }
  uint64_t r = (uint64_t)floor(u * (double)M);
  uint64_t acc = 0;
  int64_t pick = -1;
  for (int64_t i = 0; i < n; ++i) {
    if (!in[i]) continue;
    acc += w[i];
    if (acc > r) { pick = i; break; }
  }
  if (nucleus_out) *nucleus_out = k;
  free(w); free(in);
  return pick;
}

/* The sampler's distribution as integer weights: w_out[i] = token i's weight
 * when it is in the nucleus, else 0.  Returns the nucleus weight (the sum of
 * w_out), 0 on bad arguments. */
uint64_t or_sample_weights(const float* z, int64_t n, double temperature, double top_p, uint64_t* w_out) {
  if (n <= 0 || !(temperature > 0.0)) return 0;
  uint8_t* in = (uint8_t*)malloc((size_t)n);
  if (!in) return 0;
  int64_t k = 0;
  const uint64_t M = nucleus(z, n, temperature, top_p, w_out, in, &k);
  for (int64_t i = 0; i < n; ++i)
    if (!in[i]) w_out[i] = 0;
  free(in);
  return M;
}

/* ---- speculative sampling with sampled drafts ------------------------------
 * [P-feat] names self-speculative decoding and [P-code] a sampler; the pages
 * say nothing of how a sampled draft is accepted.  Reading: the published
 * speculative sampling rule (Leviathan, Kalman & Matias, ICML 2023, section
 * 2.3; Chen et al. 2023, algorithm 2), which keeps the output distribution
 * exactly the target's.  With q the draft's and p the target's sampler
 * distribution at a position (integer weights wq, wp with sums Wq, Wp):
 *   - draft token d is accepted when u < p(d) / q(d), u uniform;
 *   - otherwise the position's token is drawn from the residual
 *     max(0, p - q), renormalised;
 *   - after k accepted drafts one more token is drawn from p at the next
 *     position.
 * Exactness: with u = k_acc / 2^24 the test is
 *   k_acc * wq(d) * Wp < 2^24 * wp(d) * Wq,
 * and the residual weights R_t = max(0, wp_t * Wq - wq_t * Wp) are integers;
 * the pick is the token, in index order, whose cumulative R first exceeds
 * floor(k_res * sum R / 2^24).  Weights are below 2^40 and their sums below
 * 2^57, so every product fits in 128 bits.
 * The two 24-bit uniforms of a position come from one splitmix64 output,
 * h = splitmix64(seed xor (2 counter + 1)) — the odd counters, disjoint from
 * the sampler's even ones: k_acc = bits 40..63 of h, k_res = bits 16..39. */
typedef unsigned __int128 u128;

void or_spec_uniforms(uint64_t seed, uint64_t counter, uint32_t* k_acc, uint32_t* k_res) {
  const uint64_t h = or_splitmix64(seed ^ ((counter << 1) | 1u));
  *k_acc = (uint32_t)(h >> 40);
  *k_res = (uint32_t)((h >> 16) & 0xFFFFFFu);
}

/* 1 when draft token d (weights wq_d of Wq under the draft, wp_d of Wp under
 * the target) is accepted with uniform k_acc / 2^24 */
int or_spec_accept(uint64_t wq_d, uint64_t Wq, uint64_t wp_d, uint64_t Wp, uint32_t k_acc) {
  return (u128)k_acc * wq_d * Wp < (((u128)wp_d * Wq) << 24);
}

/* the residual draw: index of the token picked from max(0, p - q) with
 * uniform k_res / 2^24; -1 when the residual is empty (p == q) */
int64_t or_spec_residual(const uint64_t* wp, uint64_t Wp, const uint64_t* wq, uint64_t Wq, int64_t n,
                         uint32_t k_res) {
  u128 total = 0;
  for (int64_t t = 0; t < n; ++t) {
    const u128 a = (u128)wp[t] * Wq, b = (u128)wq[t] * Wp;
    if (a > b) total += a - b;
  }
  if (total == 0) return -1;
  /* floor(k_res * total / 2^24), split so that no product exceeds 128 bits */
  const u128 r = (u128)k_res * (total >> 24) + (((u128)k_res * (uint64_t)(total & 0xFFFFFFu)) >> 24);
  u128 acc = 0;
  for (int64_t t = 0; t < n; ++t) {
    const u128 a = (u128)wp[t] * Wq, b = (u128)wq[t] * Wp;
    if (a > b) acc += a - b;
    if (acc > r) return t;
  }
  return -1;
}

/* cosine similarity <a,b> / (|a| |b|)   ([P-cache] layer skip) */
double or_cos_sim(const double* a, const double* b, int64_t n) {
  double ab = 0.0, aa = 0.0, bb = 0.0;
  for (int64_t i = 0; i < n; ++i) { ab += a[i] * b[i]; aa += a[i] * a[i]; bb += b[i] * b[i]; }
  return ab / (sqrt(aa) * sqrt(bb));
}

/* Pick the n_skip layers with the highest cosine (ties: lower index first).
 * mask[l] = 1 for a skipped layer.  ([P-cache] "skips 20 of 80 layers") */
void or_layer_skip_select(const double* cos_l, int n_layers, int n_skip, uint8_t* mask) {
  memset(mask, 0, (size_t)n_layers);
  for (int k = 0; k < n_skip && k < n_layers; ++k) {
    int best = -1;
    for (int l = 0; l < n_layers; ++l) {
      if (mask[l]) continue;
      if (best < 0 || cos_l[l] > cos_l[best]) best = l;
    }
    mask[best] = 1;
  }
}

/* ---- one whole decode step ----------------------------------------------- */
typedef struct {
  int fmt;
  const uint8_t* w;
} or_qt;

typedef struct {
  or_qt wq, wk, wv, wo, wg, wu, wd;
  const float* attn_norm;
  const float* ffn_norm;
} or_layer;

typedef struct {
  int n_layers, d_model, n_qh, n_kvh, head_dim, ffn, vocab;
  double eps, theta;
  int64_t kv_cap;
  or_qt embd, out;
  const float* out_norm;
  const or_layer* layers;
  uint16_t* kcache; /* [n_layers][n_kvh][kv_cap][head_dim] binary16 */
  uint16_t* vcache;
} or_model;

static double* dalloc(int64_t n) { return (double*)calloc((size_t)(n > 0 ? n : 1), sizeof(double)); }

/*
 * Teacher-forced decode of token `token` at position `pos` ([P-code] model/:
 * transformer composition; [P-feat] RoPE, GQA, SwiGLU, RMSNorm, KV cache):
 *   x = embd[token]
 *   per layer l not skipped:
 *     xn = rmsnorm(x, g_attn); q,k,v = Wq xn, Wk xn, Wv xn; rope(q,k,pos)
 *     K[l][:,pos] = f16(k); V[l][:,pos] = f16(v)
 *     x += Wo attn(q, K[l][:, :pos+1], V[l][:, :pos+1])
 *     xn = rmsnorm(x, g_ffn); x += Wd (silu(Wg xn) * (Wu xn))
 *   logits = Wout rmsnorm(x, g_out)
 * skip (nullable) marks layers left out.  cos_out (nullable) receives
 * cos(x before layer, x after layer) for every executed layer.
 */
int or_decode_step(const or_model* m, int32_t token, int64_t pos, const uint8_t* skip, double* logits,
                   double* cos_out) {
  const int d = m->d_model, hd = m->head_dim, H = m->n_qh, G = m->n_kvh, F = m->ffn;
  if (pos < 0 || pos >= m->kv_cap || token < 0 || token >= m->vocab) return -1;
  double *x = dalloc(d), *xn = dalloc(d), *xin = dalloc(d);
  double *q = dalloc((int64_t)H * hd), *k = dalloc((int64_t)G * hd), *v = dalloc((int64_t)G * hd);
  double *o = dalloc((int64_t)H * hd), *gt = dalloc(F), *up = dalloc(F), *hh = dalloc(F);
  float* row = (float*)malloc(sizeof(float) * (size_t)d);
  int rc = 0;
  if (!x || !xn || !xin || !q || !k || !v || !o || !gt || !up || !hh || !row) { rc = -2; goto done; }

  or_dequant_rows(m->embd.fmt, m->embd.w, token, 1, d, row);
  for (int i = 0; i < d; ++i) x[i] = row[i];

  for (int l = 0; l < m->n_layers; ++l) {
    if (skip && skip[l]) continue;
    const or_layer* L = &m->layers[l];
    memcpy(xin, x, sizeof(double) * (size_t)d);
    or_rmsnorm(x, L->attn_norm, d, m->eps, xn);
    or_gemv(L->wq.fmt, L->wq.w, xn, q, (int64_t)H * hd, d, NULL);
    or_gemv(L->wk.fmt, L->wk.w, xn, k, (int64_t)G * hd, d, NULL);
    or_gemv(L->wv.fmt, L->wv.w, xn, v, (int64_t)G * hd, d, NULL);
    or_rope(q, H, hd, pos, m->theta);
    or_rope(k, G, hd, pos, m->theta);
    int64_t lay_off = (int64_t)l * G * m->kv_cap * hd;
    for (int g = 0; g < G; ++g)
      for (int i = 0; i < hd; ++i) {
        int64_t at = lay_off + ((int64_t)g * m->kv_cap + pos) * hd + i;
        m->kcache[at] = or_float_to_half((float)k[g * hd + i]);
        m->vcache[at] = or_float_to_half((float)v[g * hd + i]);
      }
    if (or_attn_decode(q, m->kcache + lay_off, m->vcache + lay_off, o, H, G, hd, pos + 1, m->kv_cap)) {
      rc = -3;
      goto done;
    }
    or_gemv(L->wo.fmt, L->wo.w, o, x, d, (int64_t)H * hd, x);
    or_rmsnorm(x, L->ffn_norm, d, m->eps, xn);
    or_gemv(L->wg.fmt, L->wg.w, xn, gt, F, d, NULL);
    or_gemv(L->wu.fmt, L->wu.w, xn, up, F, d, NULL);
    or_swiglu(gt, up, hh, F);
    or_gemv(L->wd.fmt, L->wd.w, hh, x, d, F, x);
    if (cos_out) cos_out[l] = or_cos_sim(xin, x, d);
  }
  or_rmsnorm(x, m->out_norm, d, m->eps, xn);
  or_gemv(m->out.fmt, m->out.w, xn, logits, m->vocab, d, NULL);
done:
  free(x); free(xn); free(xin); free(q); free(k); free(v); free(o); free(gt); free(up); free(hh); free(row);
  return rc;
}

int or_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void or_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
