// ops.cu — the small kernels around the quant GEMV: RMSNorm, RoPE (+ F16 KV
// append), split-K GQA decode attention with its softmax, SwiGLU, greedy
// argmax and cosine similarity.  Sources: "ntransformer - moteur d'inférence
// NVMe-to-GPU…" (fr.news.hada.io), "Architecture et structure du code"
// (cuda/: RMSNorm, RoPE, SwiGLU, softmax; inference/: sampler) and
// "Fonctionnalités principales" (RoPE, GQA, SwiGLU, RMSNorm, KV cache);
// "Performances et structure de cache" (cosine-similarity layer skip).
#include <cfloat>
#include <mutex>

#include "nt_internal.cuh"
#include "ops.cuh"

namespace nt {
namespace {

template <int NW>
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) t += red[w];
  return t;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int NW>
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = -FLT_MAX;
#pragma unroll
  for (int w = 0; w < NW; ++w) t = fmaxf(t, red[w]);
  return t;
}

// ---- RMSNorm: y = x * rsqrt(mean(x^2) + eps) * g ------------------------------
__global__ void __launch_bounds__(1024) rmsnorm_kernel(const float* x, const float* g, float* y, int64_t n,
                                                       float eps) {
  __shared__ float red[32];
  float ss = 0.f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
  ss = block_sum<32>(ss, red);
  const float inv = rsqrtf(ss / float(n) + eps);
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) y[i] = x[i] * inv * g[i];
}

// ---- RoPE ----------------------------------------------------------------------
// pair i of every head turns by pos * theta^(-2i/head_dim)
__device__ __forceinline__ void rope_table(float* cs, float* sn, int head_dim, int64_t pos, float theta) {
  for (int i = threadIdx.x; i < head_dim / 2; i += blockDim.x) rope_cs(pos, rope_inv_freq(i, head_dim, theta), cs[i], sn[i]);
  __syncthreads();
}

__device__ __forceinline__ void rotate(float* v, int n_heads, int head_dim, const float* cs, const float* sn) {
  const int half = head_dim / 2;
  for (int t = threadIdx.x; t < n_heads * half; t += blockDim.x) {
    const int h = t / half, i = t % half;
    float* p = v + int64_t(h) * head_dim + 2 * i;
    const float a = p[0], b = p[1];
    p[0] = a * cs[i] - b * sn[i];
    p[1] = a * sn[i] + b * cs[i];
  }
}

__global__ void rope_kernel(float* q, float* k, int n_qh, int n_kvh, int head_dim, int64_t pos, float theta) {
  __shared__ float cs[256], sn[256];
  rope_table(cs, sn, head_dim, pos, theta);
  rotate(q, n_qh, head_dim, cs, sn);
  if (k) rotate(k, n_kvh, head_dim, cs, sn);
}

// RoPE q in place; rotate k and append f16(k), f16(v) at cache position pos.
// pos_dev (nullable) overrides pos with a device value (graph replays).
__global__ void rope_append_kernel(float* q, const float* k, const float* v, __half* kc, __half* vc, int n_qh,
                                   int n_kvh, int head_dim, int64_t pos, const int64_t* pos_dev, int64_t kv_stride,
                                   float theta) {
  __shared__ float cs[256], sn[256];
  if (pos_dev) pos = *pos_dev;
  rope_table(cs, sn, head_dim, pos, theta);
  rotate(q, n_qh, head_dim, cs, sn);
  const int half = head_dim / 2;
  for (int t = threadIdx.x; t < n_kvh * half; t += blockDim.x) {
    const int h = t / half, i = t % half;
    const float* p = k + int64_t(h) * head_dim + 2 * i;
    const float a = p[0], b = p[1];
    const int64_t at = (int64_t(h) * kv_stride + pos) * head_dim + 2 * i;
    kc[at] = __float2half_rn(a * cs[i] - b * sn[i]);
    kc[at + 1] = __float2half_rn(a * sn[i] + b * cs[i]);
    vc[at] = __float2half_rn(v[int64_t(h) * head_dim + 2 * i]);
    vc[at + 1] = __float2half_rn(v[int64_t(h) * head_dim + 2 * i + 1]);
  }
}

// ---- split-K GQA decode attention ----------------------------------------------
// grid (n_kvh, S); CTA (g, s) covers positions [s*chunk, (s+1)*chunk) of KV head
// g for its whole group of G q heads, so K and V are read once per group.  The
// chunk of K and of V (contiguous in the cache) arrive by two TMA bulk copies.
// Each of the 4 warps runs an online softmax over 32-position tiles: scores
// with one lane per position (dims visited in a lane-rotated order so the
// shared-memory reads of a warp hit distinct banks), P.V with one lane per 4
// dims and the probabilities broadcast by shuffle.  The warps merge in shared
// memory; partials (m, l, o[128]) go to scratch; the last CTA of a KV head
// combines the S partials.
constexpr int kAttnThreads = 256;
constexpr int kTiles = 4;  // 32-position tiles per chunk (kMaxChunk / 32)
constexpr int kHD = 128;
constexpr int kMaxChunk = 128;

struct AttnArgs {
  const float* q;
  const __half* K;
  const __half* V;
  float* out;
  int n_qh, n_kvh, G, S;
  int64_t n_pos;
  const int64_t* pos_dev;  // nullable: n_pos = *pos_dev + 1
  int64_t kv_stride;
  float* part;             // [nq][n_kvh][S][G][kPS]
  unsigned* err;
  int64_t q_stride;        // floats between the q (and out) vectors of consecutive queries
  int64_t part_stride;     // floats between the partials of consecutive queries
  int stall;               // test hook: issue no bulk copies; the wait gives up after kStallSpin tries
  int nan_on_err;          // the combine writes NaN when *err holds a timed-out wait
};

// a partial row (a warp's in shared memory, a CTA's in scratch): o[128]
// (16-byte aligned), then m, l, 2 pad
constexpr int kWpStride = kHD + 4;
constexpr int kWpM = kHD, kWpL = kHD + 1;
constexpr int kPS = kWpStride;  // floats per (split, head) partial in scratch

// shared memory: K and V chunks, q (scaled), warp partials
__host__ __device__ constexpr size_t attn_smem_bytes(int G) {
  return size_t(2) * kMaxChunk * kHD * 2 + size_t(G) * kHD * 4 + size_t(kTiles) * G * kWpStride * 4 + 16;
}

__device__ __forceinline__ float4 h4(uint2 raw) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <int G>
__global__ void __launch_bounds__(kAttnThreads, (G >= 16 ? 1 : 2)) attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t asmem[];
  __half* Ks = reinterpret_cast<__half*>(asmem);                  // [kMaxChunk][128]
  __half* Vs = Ks + kMaxChunk * kHD;                               // [kMaxChunk][128]
  float* qs = reinterpret_cast<float*>(Vs + kMaxChunk * kHD);      // [G][128], pre-scaled by 1/sqrt(128)
  float* wp = qs + G * kHD;                                        // [warps][G][kWpStride] warp partials
  uint64_t* bar = reinterpret_cast<uint64_t*>(wp + kTiles * G * kWpStride);

  const int g = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // query qi (blockIdx.z) sees one position more than query qi - 1: causal
  // attention of consecutive tokens (the verify pass); one query in decode
  const int qi = blockIdx.z;
  const float* qv = a.q + int64_t(qi) * a.q_stride;
  float* partv = a.part + int64_t(qi) * a.part_stride;
  pdl_trigger();
  // In the decode step (pos_dev set) the cached positions before pos were
  // written by earlier tokens and are stable, so their K/V chunk streams in
  // before waiting for the kernel that writes q and positions pos.. .  Called
  // standalone, everything waits: the caller may have just written the cache.
  if (!a.pos_dev) pdl_wait();
  const int64_t pos0 = a.pos_dev ? __ldcg(a.pos_dev) : 0;  // read before the wait: bypass L1
  int64_t n_pos = (a.pos_dev ? pos0 + 1 : a.n_pos) + qi;
  if (n_pos < 1 || n_pos > a.kv_stride) {
    // a device-side position outside the cache: read nothing beyond it
    if (tid == 0 && s == 0) flag_error(a.err, kErrPosRange);
    n_pos = n_pos < 1 ? 1 : a.kv_stride;
  }
  const int64_t stable = a.pos_dev ? pos0 : n_pos;  // positions written before this step
  const int64_t chunk = (n_pos + a.S - 1) / a.S;
  const int64_t p0 = int64_t(s) * chunk;
  const int64_t p1 = min(n_pos, p0 + chunk);
  const int np = p1 > p0 ? int(p1 - p0) : 0;
  const int np_early = a.pos_dev ? max(0, int(min(p1, stable) - p0)) : np;  // positions safe before the wait
  const __half* Kg = a.K + int64_t(g) * a.kv_stride * kHD;
  const __half* Vg = a.V + int64_t(g) * a.kv_stride * kHD;
  const uint32_t b = smem_u32(bar);

  if (tid == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
    if (np > 0) {
      mbar_arrive_expect_tx(b, uint32_t(np) * kHD * 2 * 2);
      if (np_early > 0 && !a.stall) {
        const uint32_t bytes = uint32_t(np_early) * kHD * 2;
        const uint64_t pol = policy_evict_first();
        bulk_g2s(smem_u32(Ks), Kg + p0 * kHD, bytes, b, pol);
        bulk_g2s(smem_u32(Vs), Vg + p0 * kHD, bytes, b, pol);
      }
    }
  }
  if (a.pos_dev) {
    pdl_wait();
    if (tid == 0 && np > np_early && !a.stall) {
      // the rest (the new position pos) after the producer has finished
      const uint32_t off = uint32_t(np_early) * kHD, bytes = uint32_t(np - np_early) * kHD * 2;
      const uint64_t pol = policy_evict_first();
      bulk_g2s(smem_u32(Ks + off), Kg + (p0 + np_early) * kHD, bytes, b, pol);
      bulk_g2s(smem_u32(Vs + off), Vg + (p0 + np_early) * kHD, bytes, b, pol);
    }
  }
  const float scale = rsqrtf(float(kHD));
  for (int i = tid; i < G * kHD; i += kAttnThreads) qs[i] = qv[int64_t(g) * G * kHD + i] * scale;
  __syncthreads();
  bool ok = true;
  if (np > 0) ok = mbar_wait(b, 0, a.stall ? kStallSpin : kMaxSpin);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) flag_error(a.err, kErrWaitTimeout);
    return;
  }

  // ---- per-warp online softmax over one 32-position tile: warp w takes tile
  // w % 4 of the chunk and half of the group's heads (all of them when G = 1)
  constexpr int NH = G >= 2 ? 2 : 1;  // head halves
  constexpr int HS = G / NH;           // heads per warp
  const int tile = warp % kTiles, hh = warp / kTiles;
  float m[HS], l[HS], o[HS][4];
#pragma unroll
  for (int h = 0; h < HS; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
    o[h][0] = o[h][1] = o[h][2] = o[h][3] = 0.f;
  }
  const float* qh = qs + hh * HS * kHD;
  for (int t0 = 32 * tile; hh < NH && t0 < np; t0 += 32 * kTiles) {
    const int j = t0 + lane;
    const bool valid = j < np;
    float sc[HS];
#pragma unroll
    for (int h = 0; h < HS; ++h) sc[h] = 0.f;
    if (valid) {
      const __half* krow = Ks + j * kHD;
      // four partial sums per head (4-dim chunks c = 4i + r go to sum r): four
      // short dependency chains instead of one of 128 FMAs
      float sp[HS][4];
#pragma unroll
      for (int h = 0; h < HS; ++h) sp[h][0] = sp[h][1] = sp[h][2] = sp[h][3] = 0.f;
#pragma unroll 2
      for (int c4 = 0; c4 < 32; c4 += 4) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int cc = (c4 + r + lane) & 31;  // lane-rotated 4-dim chunk: distinct banks across the warp
          const float4 k = h4(*reinterpret_cast<const uint2*>(krow + 4 * cc));
#pragma unroll
          for (int h = 0; h < HS; ++h) {
            const float4 qv = *reinterpret_cast<const float4*>(qh + h * kHD + 4 * cc);
            sp[h][r] = fmaf(qv.x, k.x, fmaf(qv.y, k.y, fmaf(qv.z, k.z, fmaf(qv.w, k.w, sp[h][r]))));
          }
        }
      }
#pragma unroll
      for (int h = 0; h < HS; ++h) sc[h] = (sp[h][0] + sp[h][1]) + (sp[h][2] + sp[h][3]);
    }
    float pj[HS];
#pragma unroll
    for (int h = 0; h < HS; ++h) {
      const float sv = valid ? sc[h] : -INFINITY;
      const float mn = fmaxf(m[h], warp_max(sv));
      const float corr = m[h] == -INFINITY ? 0.f : __expf(m[h] - mn);
      pj[h] = valid ? __expf(sv - mn) : 0.f;
      l[h] = fmaf(l[h], corr, warp_sum(pj[h]));
      o[h][0] *= corr;
      o[h][1] *= corr;
      o[h][2] *= corr;
      o[h][3] *= corr;
      m[h] = mn;
    }
    const int nt = min(32, np - t0);
#pragma unroll 4
    for (int jj = 0; jj < nt; ++jj) {
      const float4 v = h4(*reinterpret_cast<const uint2*>(Vs + (t0 + jj) * kHD + 4 * lane));
#pragma unroll
      for (int h = 0; h < HS; ++h) {
        const float p = __shfl_sync(0xffffffffu, pj[h], jj);
        o[h][0] = fmaf(p, v.x, o[h][0]);
        o[h][1] = fmaf(p, v.y, o[h][1]);
        o[h][2] = fmaf(p, v.z, o[h][2]);
        o[h][3] = fmaf(p, v.w, o[h][3]);
      }
    }
  }
  // ---- merge the tiles: (m, l, o) of each (tile, head) -> one CTA partial
  if (hh < NH) {
    float* mine = wp + tile * G * kWpStride;
#pragma unroll
    for (int hl = 0; hl < HS; ++hl) {
      const int h = hh * HS + hl;
      if (lane == 0) {
        mine[h * kWpStride + kWpM] = m[hl];
        mine[h * kWpStride + kWpL] = l[hl];
      }
      *reinterpret_cast<float4*>(mine + h * kWpStride + 4 * lane) =
          make_float4(o[hl][0], o[hl][1], o[hl][2], o[hl][3]);
    }
  }
  __syncthreads();
  float* my = partv + (int64_t(g) * a.S + s) * G * kPS;
  for (int i = tid; i < G * (kHD + 1); i += kAttnThreads) {
    const int h = i / (kHD + 1), d = i % (kHD + 1);  // d == kHD: the (m, l) pair
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kTiles; ++w) M = fmaxf(M, wp[(w * G + h) * kWpStride + kWpM]);
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kTiles; ++w) {
      const float* pw = wp + (w * G + h) * kWpStride;
      const float c = pw[kWpM] == -INFINITY ? 0.f : __expf(pw[kWpM] - M);
      acc = fmaf(d < kHD ? pw[d] : pw[kWpL], c, acc);
    }
    if (d < kHD) {
      my[h * kPS + d] = acc;
    } else {
      my[h * kPS + kWpM] = M;
      my[h * kPS + kWpL] = acc;
    }
  }

}

// The split partials of one (KV head g, head h of its group, query qi) into
// the attention output: with the splits' maxima m_t and sums l_t,
// M = max m_t, w_t = e^(m_t - M) / sum_t l_t e^(m_t - M), out = sum_t w_t o_t.
// One CTA of kHD threads, one per output dimension.  Launched right behind
// the attention kernel (a dependent launch: its CTAs wait for that grid to
// finish, which orders the partials' writes before the reads here).
__global__ void __launch_bounds__(kHD) attn_combine_kernel(const AttnArgs a) {
  __shared__ float wts[kMaxChunk];
  __shared__ float red[kHD / 32];
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.x, h = blockIdx.y, qi = blockIdx.z, d = threadIdx.x, lane = d & 31, warp = d >> 5;
  const int G = a.G, S = a.S;
  const float* base = a.part + int64_t(qi) * a.part_stride + (int64_t(g) * S * G + h) * kPS;
  const int64_t stride = int64_t(G) * kPS;  // floats between consecutive splits
  // split d's (max, sum), and this dimension of the first 32 splits, all in flight together
  float mt = -INFINITY, lt = 0.f;
  if (d < S) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(base + d * stride + kWpM));
    mt = ml.x;
    lt = ml.y;
  }
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = j < S ? __ldcg(base + j * stride + d) : 0.f;
  float M = warp_max(mt);
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kHD / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  const float w = (d < S && mt != -INFINITY) ? __expf(mt - M) : 0.f;
  float L = warp_sum(lt * w);
  if (lane == 0) red[warp] = L;
  __syncthreads();
  L = red[0];
#pragma unroll
  for (int k = 1; k < kHD / 32; ++k) L += red[k];
  if (d < S) wts[d] = w * (1.0f / L);
  __syncthreads();
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j < S) acc = fmaf(v[j], wts[j], acc);
  for (int t0 = 32; t0 < S; t0 += 32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = t0 + j < S ? __ldcg(base + (t0 + j) * stride + d) : 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (t0 + j < S) acc = fmaf(v[j], wts[t0 + j], acc);
  }
  // a split whose wait ran out left its partial unwritten: no plausible-looking output
  if (a.nan_on_err && (__ldcg(a.err) & kErrWaitTimeout)) acc = __int_as_float(0x7fc00000);
  a.out[int64_t(qi) * a.q_stride + (int64_t(g) * G + h) * kHD + d] = acc;
}

using AttnKernel = void (*)(AttnArgs);
AttnKernel attn_kernel_for(int G) {
  switch (G) {
    case 1: return attn_kernel<1>;
    case 2: return attn_kernel<2>;
    case 4: return attn_kernel<4>;
    case 8: return attn_kernel<8>;
    case 16: return attn_kernel<16>;
    default: return nullptr;
  }
}

// ---- softmax (standalone) --------------------------------------------------------
__global__ void __launch_bounds__(1024) softmax_kernel(const float* x, float* y, int64_t n) {
  __shared__ float red[32];
  float m = -FLT_MAX;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, x[i]);
  m = block_max<32>(m, red);
  float l = 0.f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) l += __expf(x[i] - m);
  l = block_sum<32>(l, red);
  const float inv = 1.0f / l;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) y[i] = __expf(x[i] - m) * inv;
}

// ---- SwiGLU (standalone) -----------------------------------------------------------
__global__ void swiglu_kernel(const float* gate, const float* up, float* h, int64_t n) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
    h[i] = silu(gate[i]) * up[i];
}

// ---- greedy argmax ------------------------------------------------------------------
// key = (order-preserving bits of v) << 32 | (~index): the largest key is the
// largest value with the lowest index.  NaN never wins.
__device__ __forceinline__ unsigned long long argmax_key(float v, int64_t i) {
  if (v != v) return 0ull;
  const unsigned b = __float_as_uint(v);
  const unsigned o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(o) << 32) | (0xFFFFFFFFu - unsigned(i));
}

__global__ void argmax_kernel(const float* v, int64_t n, unsigned long long* key, unsigned* counter, int32_t* out,
                              int32_t* tok_state, int64_t* pos_state) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned long long wbest[32];
  __shared__ bool last;
  unsigned long long best = 0ull;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const unsigned long long k = argmax_key(v[i], i);
    best = k > best ? k : best;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
    best = t > best ? t : best;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) wbest[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long b = 0ull;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) b = wbest[w] > b ? wbest[w] : b;
    atomicMax(key, b);
    __threadfence();
    last = atomicAdd(counter, 1u) == gridDim.x - 1;
    if (last) {
      __threadfence();
      const unsigned long long k = atomicAdd(key, 0ull);
      const int32_t idx = k ? int32_t(0xFFFFFFFFu - unsigned(k & 0xFFFFFFFFull)) : 0;
      if (out) *out = idx;
      if (tok_state) *tok_state = idx;   // decode loop: next token and position
      if (pos_state) *pos_state += 1;
      *key = 0ull;
      *counter = 0u;
    }
  }
}

// ---- non-greedy sampler: temperature + nucleus (top-p) -------------------------------
// Token weights are integers, w = rint(exp((z - max z) / T) * 2^40), so every
// sum is exact and independent of the order of addition.  The nucleus is the
// shortest prefix of the tokens ordered by logit (descending, ties by lower
// index) whose weight reaches ceil(top_p * sum w), found by a radix select on
// the order-preserving 32-bit key of the logit (digits of 11, 11 and 10
// bits); the token is the one of the nucleus, in index order, whose
// cumulative weight first exceeds floor(u * nucleus weight), u from
// SplitMix64 (Steele, Lea & Flood 2014) of (seed, counter).  T <= 0 is greedy.
//
// Work split: each row (blockIdx.y) is cut into G contiguous CTA ranges of at
// most kSampPer logits, each thread owning a contiguous run.  Six launches:
// max, three histogram rounds, a count of ties and of the weight above the
// threshold key, and the pick.  In every launch the last CTA to finish (an
// arrival counter, no waiting) does the row-wide step: reduce the maxima,
// select the digit, place the pick in a CTA range.  Histograms are summed in
// shared memory as two 32-bit halves of the weight (20 low bits, 21 high
// bits), then added once per non-empty bin into the row's 64-bit histogram.
constexpr int kSampThreads = 256;
constexpr int kSampMaxCtas = 256;
constexpr int64_t kSampPer = 4000;  // logits per CTA at most: 4000 * 2^20 keeps each 32-bit half below 2^32
constexpr int kSampBins = 2048;

struct SampRow {
  unsigned cnt;  // CTAs of the current launch that arrived; the last resets it
  float M;       // largest logit
  int arg;       // lowest index holding it
  uint32_t prefix;
  unsigned long long Z, target, above, wt, j, Mn, r, cbase;
  int cstar, pad;
  unsigned long long hist[kSampBins];
  float part_max[kSampMaxCtas];
  int part_arg[kSampMaxCtas];
  unsigned long long part_ties[kSampMaxCtas], part_mass[kSampMaxCtas], tie0[kSampMaxCtas];
};
static_assert(sizeof(SampRow) <= kSampRowBytes, "sampler state row");

struct SampArgs {
  const float* z;
  int64_t n, per;
  float T, P;
  uint64_t seed;
  const int64_t* ctr_dev;  // per-row counters, or null: ctr + row
  int64_t ctr;
  int32_t* out;             // [rows]
  int32_t* tok_state;       // nullable (one row): the pick also becomes the model's token ...
  int64_t* pos_state;       // ... and its position advances
  unsigned long long* w_out;  // nullable: [rows][n] each token's weight inside the nucleus, else 0
  unsigned long long* W_out;  // nullable: [rows] the nucleus weight
  SampRow* st;              // [rows]
};

__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// order-preserving key of a logit; NaN ranks below everything
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (v != v) return 0u;
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ unsigned long long samp_weight(float v, float M, float T) {
  if (!(v >= -3.0e38f)) return 0ull;  // NaN and -inf weigh nothing
  return __float2ull_rn(expf((v - M) / T) * 1099511627776.0f);  // 2^40
}

// exclusive prefix sum over a block of kSampThreads threads; total in *total
__device__ __forceinline__ unsigned long long samp_scan(unsigned long long v, unsigned long long* total) {
  __shared__ unsigned long long sw[kSampThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sw[warp] = x;
  __syncthreads();
  unsigned long long before = x - v, all = 0;
#pragma unroll
  for (int w = 0; w < kSampThreads / 32; ++w) {
    const unsigned long long t = sw[w];
    if (w < warp) before += t;
    all += t;
  }
  *total = all;
  __syncthreads();
  return before;
}

// the thread's contiguous run of its CTA's range of row `z`
struct SampRange {
  int64_t i0, i1;
  __device__ SampRange(const SampArgs& a) {
    const int64_t lo = int64_t(blockIdx.x) * a.per, hi = min(a.n, lo + a.per);
    const int64_t tper = (a.per + kSampThreads - 1) / kSampThreads;
    i0 = min(hi, lo + int64_t(threadIdx.x) * tper);
    i1 = min(hi, i0 + tper);
  }
};

// true in the last CTA of the launch to arrive (after every other CTA's
// global writes are visible to it); resets the counter for the next launch
__device__ __forceinline__ bool samp_arrive(SampRow* s) {
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&s->cnt, 1u);
    last = prev == gridDim.x - 1;
    if (last) s->cnt = 0;
  }
  __syncthreads();
  if (last) __threadfence();
  return last;
}

__device__ __forceinline__ void samp_finish(const SampArgs& a, int row, int pick, unsigned long long Mn) {
  const int32_t t = pick < 0 ? 0 : pick;
  if (a.out) a.out[row] = t;
  if (a.tok_state) *a.tok_state = t;
  if (a.pos_state) *a.pos_state += 1;
  if (a.W_out) a.W_out[row] = Mn;
}

// (max, lowest index) pairs: the larger value, then the lower index
__device__ __forceinline__ void maxarg_merge(float& m, int64_t& i, float m2, int64_t i2) {
  if (m2 > m || (m2 == m && i2 < i)) {
    m = m2;
    i = i2;
  }
}

__device__ __forceinline__ void block_maxarg(float& m, int64_t& i) {
  __shared__ float sm_m[kSampThreads / 32];
  __shared__ int64_t sm_i[kSampThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) maxarg_merge(m, i, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, i, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sm_m[warp] = m;
    sm_i[warp] = i;
  }
  __syncthreads();
  for (int w = 0; w < kSampThreads / 32; ++w) maxarg_merge(m, i, sm_m[w], sm_i[w]);
  __syncthreads();
}

// launch 1: the row's largest logit and the lowest index holding it; greedy
// rows finish here
__global__ void __launch_bounds__(kSampThreads) samp_max_kernel(SampArgs a) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y;
  SampRow* s = a.st + row;
  const float* z = a.z + int64_t(row) * a.n;
  const SampRange r(a);
  float m = -INFINITY;
  int64_t idx = a.n;
  for (int64_t i = r.i0; i < r.i1; ++i) {
    const float v = z[i];
    if (v > m || (idx == a.n && v == m)) {  // NaN never enters
      m = v;
      idx = i;
    }
  }
  block_maxarg(m, idx);
  if (threadIdx.x == 0) {
    s->part_max[blockIdx.x] = m;
    s->part_arg[blockIdx.x] = int(idx);
  }
  if (!samp_arrive(s)) return;
  m = -INFINITY;
  idx = a.n;
  for (int c = threadIdx.x; c < gridDim.x; c += kSampThreads) maxarg_merge(m, idx, __ldcg(&s->part_max[c]), __ldcg(&s->part_arg[c]));
  block_maxarg(m, idx);
  if (threadIdx.x == 0) {
    s->M = m;
    s->arg = int(idx < a.n ? idx : 0);
    if (!(a.T > 0.f)) samp_finish(a, row, s->arg, 0ull);
  }
}

// add each lane's weight w (when `has`) to bin d of the split histogram:
// lanes holding the same bin are summed first (up to 4 distinct bins per
// call, the usual case when the logits crowd a few bins), the rest add alone
__device__ __forceinline__ void hist_add(uint32_t* hlo, uint32_t* hhi, bool has, uint32_t d, unsigned long long w) {
  const unsigned lane = threadIdx.x & 31;
  const uint32_t lo = uint32_t(w & 0xFFFFFu), hi = uint32_t(w >> 20);
  unsigned todo = __ballot_sync(0xffffffffu, has);
  for (int it = 0; todo && it < 4; ++it) {
    const int leader = __ffs(todo) - 1;
    const uint32_t dl = __shfl_sync(0xffffffffu, d, leader);
    const bool mine = ((todo >> lane) & 1u) && d == dl;
    const uint32_t slo = __reduce_add_sync(0xffffffffu, mine ? lo : 0u);
    const uint32_t shi = __reduce_add_sync(0xffffffffu, mine ? hi : 0u);
    if (int(lane) == leader) {
      atomicAdd(&hlo[dl], slo);
      atomicAdd(&hhi[dl], shi);
    }
    todo &= ~__ballot_sync(0xffffffffu, mine);
  }
  if ((todo >> lane) & 1u) {
    atomicAdd(&hlo[d], lo);
    atomicAdd(&hhi[d], hi);
  }
}

// launches 2-4: histogram of digit `round` (bits 31..21, 20..10, 9..0) of the
// keys that match the digits already selected, weighted; the last CTA selects
// the digit at which the weight, counted from the top, reaches the target
__global__ void __launch_bounds__(kSampThreads) samp_round_kernel(SampArgs a, int round) {
  __shared__ uint32_t hlo[kSampBins], hhi[kSampBins];
  __shared__ int s_d;
  __shared__ unsigned long long s_above, s_h0;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y;
  SampRow* s = a.st + row;
  const float* z = a.z + int64_t(row) * a.n;
  const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
  const int nb = round == 2 ? 1024 : 2048;
  const int sel = shift + (round == 2 ? 10 : 11);  // the bits at and above `sel` are already selected
  for (int b = threadIdx.x; b < nb; b += kSampThreads) hlo[b] = hhi[b] = 0u;
  __syncthreads();
  const float M = s->M;
  const uint32_t prefix = round == 0 ? 0u : s->prefix;
  const SampRange r(a);
  unsigned long long zp = 0;
  const int64_t tper = (a.per + kSampThreads - 1) / kSampThreads;  // the same trip count in every lane
  for (int64_t e = 0; e < tper; ++e) {
    const int64_t i = r.i0 + e;
    const float v = i < r.i1 ? z[i] : -INFINITY;
    const uint32_t k = logit_key(v);
    const bool match = round == 0 || (k >> sel) == (prefix >> sel);
    const unsigned long long w = match ? samp_weight(v, M, a.T) : 0ull;
    zp += w;
    hist_add(hlo, hhi, w != 0ull, (k >> shift) & uint32_t(nb - 1), w);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < nb; b += kSampThreads) {
    const unsigned long long v = (static_cast<unsigned long long>(hhi[b]) << 20) + hlo[b];
    if (v) atomicAdd(&s->hist[b], v);
  }
  if (round == 0) {
    unsigned long long tot;
    samp_scan(zp, &tot);
    if (threadIdx.x == 0 && tot) atomicAdd(&s->Z, tot);
  }
  if (!samp_arrive(s)) return;

  if (round == 0 && threadIdx.x == 0) {
    const unsigned long long Z = __ldcg(&s->Z);
    const double tgt = ceil(double(a.P) * double(Z));
    s->target = tgt < 1.0 ? 1ull : (tgt > double(Z) ? Z : static_cast<unsigned long long>(tgt));
    s->above = 0ull;
    s->Z = 0ull;
  }
  __syncthreads();
  const unsigned long long target = s->target, above = s->above;
  // thread t holds bins nb-1-t*g .. nb-g-t*g, highest first
  const int g = nb / kSampThreads;
  unsigned long long h[kSampBins / kSampThreads], sum = 0;
#pragma unroll
  for (int q = 0; q < kSampBins / kSampThreads; ++q) {
    h[q] = 0ull;
    if (q >= g) continue;
    const int b = nb - 1 - threadIdx.x * g - q;
    h[q] = __ldcg(&s->hist[b]);
    s->hist[b] = 0ull;
    sum += h[q];
    if (b == 0) s_h0 = h[q];
  }
  unsigned long long total;
  unsigned long long cum = above + samp_scan(sum, &total);
  if (threadIdx.x == 0) {
    s_d = -1;
    s_above = 0;
  }
  __syncthreads();
  if (cum < target && cum + sum >= target) {
#pragma unroll
    for (int q = 0; q < kSampBins / kSampThreads; ++q) {
      if (q < g && cum + h[q] >= target) {
        s_d = nb - 1 - threadIdx.x * g - q;
        s_above = cum;
        break;
      }
      cum += h[q];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int d = s_d;
    unsigned long long ab = s_above;
    if (d < 0) {  // the target is not reached above digit 0: take digit 0
      d = 0;
      ab = above + total - s_h0;
    }
    const uint32_t pre = prefix | (uint32_t(d) << shift);
    s->prefix = pre;
    s->above = ab;
    if (round == 2) {
      // pre is the key of the last token the nucleus needs; the nucleus takes
      // the first j of the tokens holding it (index order)
      const unsigned long long wt = samp_weight(key_value(pre), M, a.T);
      const unsigned long long need = target - ab;
      const unsigned long long j = wt ? (need + wt - 1) / wt : 0ull;
      const unsigned long long Mn = ab + j * wt;
      const uint64_t counter = a.ctr_dev ? uint64_t(a.ctr_dev[row]) : uint64_t(a.ctr + row);
      const double u = double(splitmix64(a.seed ^ (counter << 1)) >> 40) * 0x1.0p-24;
      s->wt = wt;
      s->j = j;
      s->Mn = Mn;
      s->r = static_cast<unsigned long long>(u * double(Mn));
    }
  }
}

// launch 5: per CTA, the tokens at the threshold key and the weight above it;
// the last CTA ranks the ties across CTAs and finds the CTA whose nucleus
// weight holds r
__global__ void __launch_bounds__(kSampThreads) samp_count_kernel(SampArgs a) {
  __shared__ int s_c;
  __shared__ unsigned long long s_base;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y;
  SampRow* s = a.st + row;
  const float* z = a.z + int64_t(row) * a.n;
  const float M = s->M;
  const uint32_t tau = s->prefix;
  const SampRange r(a);
  unsigned long long ties = 0, mass = 0;
  for (int64_t i = r.i0; i < r.i1; ++i) {
    const float v = z[i];
    const uint32_t k = logit_key(v);
    if (k > tau) mass += samp_weight(v, M, a.T);
    ties += k == tau;
  }
  unsigned long long tt, tm;
  samp_scan(ties, &tt);
  samp_scan(mass, &tm);
  if (threadIdx.x == 0) {
    s->part_ties[blockIdx.x] = tt;
    s->part_mass[blockIdx.x] = tm;
  }
  if (!samp_arrive(s)) return;
  const int c = threadIdx.x;  // gridDim.x <= kSampThreads
  const bool has = c < int(gridDim.x);
  const unsigned long long t = has ? __ldcg(&s->part_ties[c]) : 0ull, ma = has ? __ldcg(&s->part_mass[c]) : 0ull;
  unsigned long long tot;
  const unsigned long long t0 = samp_scan(t, &tot);
  const unsigned long long j = s->j, wt = s->wt, rr = s->r;
  const unsigned long long take = j > t0 ? (j - t0 < t ? j - t0 : t) : 0ull;
  const unsigned long long nm = ma + take * wt;
  const unsigned long long base = samp_scan(nm, &tot);
  if (threadIdx.x == 0) s_c = -1;
  __syncthreads();
  if (has) s->tie0[c] = t0;
  if (has && nm && base <= rr && rr < base + nm) {
    s_c = c;
    s_base = base;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    s->cstar = s_c;
    s->cbase = s_c >= 0 ? s_base : 0ull;
  }
}

// launch 6: the pick, in the CTA holding r; with w_out every CTA also writes
// its tokens' nucleus weights
__global__ void __launch_bounds__(kSampThreads) samp_pick_kernel(SampArgs a) {
  __shared__ int s_pick;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y;
  SampRow* s = a.st + row;
  const int cstar = s->cstar;
  const bool mine = int(blockIdx.x) == cstar || (cstar < 0 && blockIdx.x == 0);
  if (!mine && !a.w_out) return;
  const float* z = a.z + int64_t(row) * a.n;
  const float M = s->M;
  const uint32_t tau = s->prefix;
  const unsigned long long j = s->j, rr = s->r;
  const SampRange r(a);
  unsigned long long ties = 0;
  for (int64_t i = r.i0; i < r.i1; ++i) ties += logit_key(z[i]) == tau;
  unsigned long long tmp;
  const unsigned long long tie_first = s->tie0[blockIdx.x] + samp_scan(ties, &tmp);
  unsigned long long mass = 0, seen = tie_first;
  unsigned long long* wo = a.w_out ? a.w_out + int64_t(row) * a.n : nullptr;
  for (int64_t i = r.i0; i < r.i1; ++i) {
    const float v = z[i];
    const uint32_t k = logit_key(v);
    const bool in = k > tau || (k == tau && seen < j);
    seen += k == tau;
    const unsigned long long w = in ? samp_weight(v, M, a.T) : 0ull;
    mass += w;
    if (wo) wo[i] = w;
  }
  if (!mine) return;
  const unsigned long long base = s->cbase + samp_scan(mass, &tmp);
  if (threadIdx.x == 0) s_pick = -1;
  __syncthreads();
  if (cstar >= 0 && mass && base <= rr && rr < base + mass) {
    unsigned long long acc = base;
    seen = tie_first;
    for (int64_t i = r.i0; i < r.i1; ++i) {
      const float v = z[i];
      const uint32_t k = logit_key(v);
      const bool in = k > tau || (k == tau && seen < j);
      seen += k == tau;
      if (!in) continue;
      acc += samp_weight(v, M, a.T);
      if (acc > rr) {
        s_pick = int(i);
        break;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) samp_finish(a, row, s_pick, s->Mn);
}

// ---- cosine similarity --------------------------------------------------------------
__global__ void __launch_bounds__(1024) cos_kernel(const float* x, const float* y, int64_t n, float* out) {
  pdl_wait();
  pdl_trigger();
  __shared__ double red[3][32];
  double ab = 0, aa = 0, bb = 0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const double p = x[i], q = y[i];
    ab += p * q;
    aa += p * p;
    bb += q * q;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ab += __shfl_xor_sync(0xffffffffu, ab, o);
    aa += __shfl_xor_sync(0xffffffffu, aa, o);
    bb += __shfl_xor_sync(0xffffffffu, bb, o);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    red[0][warp] = ab;
    red[1][warp] = aa;
    red[2][warp] = bb;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double s0 = 0, s1 = 0, s2 = 0;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) {
      s0 += red[0][w];
      s1 += red[1][w];
      s2 += red[2][w];
    }
    *out = float(s0 / (sqrt(s1) * sqrt(s2)));
  }
}

}  // namespace

// ---------------------------------------------------------------------------------
// launchers (arguments already validated by the C ABI layer)

nt_status launch_rmsnorm(Ctx* c, const float* x, const float* g, float* y, int64_t n, float eps, cudaStream_t st) {
  rmsnorm_kernel<<<1, 1024, 0, st>>>(x, g, y, n, eps);
  return cuda_check(c, cudaGetLastError(), "rmsnorm launch");
}

nt_status launch_rope(Ctx* c, float* q, float* k, int n_qh, int n_kvh, int hd, int64_t pos, float theta,
                      cudaStream_t st) {
  rope_kernel<<<1, 256, 0, st>>>(q, k, n_qh, n_kvh, hd, pos, theta);
  return cuda_check(c, cudaGetLastError(), "rope launch");
}

nt_status launch_rope_append(Ctx* c, float* q, const float* k, const float* v, void* kc, void* vc, int n_qh,
                             int n_kvh, int hd, int64_t pos, const int64_t* pos_dev, int64_t kv_stride, float theta,
                             cudaStream_t st) {
  rope_append_kernel<<<1, 256, 0, st>>>(q, k, v, static_cast<__half*>(kc), static_cast<__half*>(vc), n_qh, n_kvh,
                                        hd, pos, pos_dev, kv_stride, theta);
  return cuda_check(c, cudaGetLastError(), "rope/append launch");
}

// splits per KV head: enough CTAs to cover the SMs, chunks of at most
// kMaxChunk positions, and at most kMaxChunk splits (the combine stages one
// weight per split in a kMaxChunk-long row), so kv_stride <= kMaxChunk^2
int attn_splits(const Ctx* c, int n_kvh, int64_t kv_stride) {
  // chunks of up to kMaxChunk positions keep every warp on a full 32-position
  // tile; with attn_fill, also at least one CTA per SM
  int S = c->attn_fill ? (c->num_sms + n_kvh - 1) / n_kvh : 1;
  const int64_t need = (kv_stride + kMaxChunk - 1) / kMaxChunk;
  if (need > S) S = int(need);
  return S < kMaxChunk ? S : kMaxChunk;
}

int64_t attn_max_stride() { return int64_t(kMaxChunk) * kMaxChunk; }

size_t attn_scratch_bytes(int n_qh, int n_kvh, int S, int nq) {
  return size_t(nq) * size_t(n_kvh) * S * (n_qh / n_kvh) * kPS * sizeof(float) + kAttnCounterBytes;
}

size_t attn_part_floats(int n_qh, int n_kvh, int S) { return size_t(n_kvh) * S * (n_qh / n_kvh) * kPS; }

nt_status launch_attn(Ctx* c, const float* q, const void* K, const void* V, float* out, int n_qh, int n_kvh,
                      int64_t n_pos, const int64_t* pos_dev, int64_t kv_stride, float* part, int S, cudaStream_t st,
                      int nq) {
  if (c->dry) return NT_OK;
  AttnArgs a{};
  a.q_stride = int64_t(n_qh) * kHD;
  a.part_stride = int64_t(attn_part_floats(n_qh, n_kvh, S));
  a.q = q;
  a.K = static_cast<const __half*>(K);
  a.V = static_cast<const __half*>(V);
  a.out = out;
  a.n_qh = n_qh;
  a.n_kvh = n_kvh;
  a.G = n_qh / n_kvh;
  a.S = S;
  a.n_pos = n_pos;
  a.pos_dev = pos_dev;
  a.kv_stride = kv_stride;
  a.part = part;
  a.err = c->err_flag;
  const size_t smem = attn_smem_bytes(a.G);
  AttnKernel k = attn_kernel_for(a.G);
  if (!k) return set_err(c, NT_ERR_INVALID_ARG, "attention: group size %d not in {1,2,4,8,16}", a.G);
  a.stall = take_stall(st);
  nt_status s = cuda_check(c, launch_k(c, k, dim3(n_kvh, S, nq), dim3(kAttnThreads), smem, st, a), "attention launch");
  if (s) return s;
  return cuda_check(c, launch_k(c, attn_combine_kernel, dim3(n_kvh, a.G, nq), dim3(kHD), 0, st, a),
                    "attention combine launch");
}

cudaError_t configure_attn(size_t optin) {
  for (int G : {1, 2, 4, 8, 16}) {
    const size_t smem = attn_smem_bytes(G);
    AttnKernel k = attn_kernel_for(G);
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, k);
    if (e == cudaSuccess && smem + fa.sharedSizeBytes > optin) e = cudaErrorInvalidValue;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

nt_status configure_ops(Ctx* c) {
  return cuda_check(c, configure_attn(c->smem_optin), "attention shared-memory attribute");
}

__global__ void inv_freq_kernel(double* out, int head_dim, float theta) {
  for (int i = threadIdx.x; i < head_dim / 2; i += blockDim.x) out[i] = rope_inv_freq(i, head_dim, theta);
}

nt_status launch_inv_freq(Ctx* c, double* out, int head_dim, float theta, cudaStream_t st) {
  inv_freq_kernel<<<1, 128, 0, st>>>(out, head_dim, theta);
  return cuda_check(c, cudaGetLastError(), "inv_freq launch");
}

nt_status launch_softmax(Ctx* c, const float* x, float* y, int64_t n, cudaStream_t st) {
  softmax_kernel<<<1, 1024, 0, st>>>(x, y, n);
  return cuda_check(c, cudaGetLastError(), "softmax launch");
}

nt_status launch_swiglu(Ctx* c, const float* g, const float* u, float* h, int64_t n, cudaStream_t st) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  swiglu_kernel<<<int(blocks), 256, 0, st>>>(g, u, h, n);
  return cuda_check(c, cudaGetLastError(), "swiglu launch");
}

nt_status launch_argmax(Ctx* c, const float* v, int64_t n, int32_t* out, unsigned long long* key, unsigned* counter,
                        cudaStream_t st, int32_t* tok_state, int64_t* pos_state) {
  if (c->dry) return NT_OK;
  int64_t blocks = (n + 1023) / 1024;
  if (blocks > c->num_sms) blocks = c->num_sms;
  if (blocks < 1) blocks = 1;
  return cuda_check(c, launch_k(c, argmax_kernel, dim3(int(blocks)), dim3(1024), 0, st, v, n, key, counter, out,
                                tok_state, pos_state),
                    "argmax launch");
}

int sample_ctas(int64_t n) {
  const int64_t g = (n + 1023) / 1024;
  return int(g < 1 ? 1 : (g > kSampMaxCtas ? kSampMaxCtas : g));
}

nt_status launch_sample(Ctx* c, const float* z, int64_t n, int rows, float T, float P, uint64_t seed,
                        const int64_t* ctr_dev, int64_t ctr, int32_t* out, void* state, cudaStream_t st,
                        int32_t* tok_state, int64_t* pos_state, unsigned long long* w_out,
                        unsigned long long* W_out) {
  if (c->dry) return NT_OK;
  const int G = sample_ctas(n);
  const int64_t per = (n + G - 1) / G;
  if (per > kSampPer || rows < 1) return set_err(c, NT_ERR_INVALID_ARG, "sampler: n %lld too large", (long long)n);
  const SampArgs a{z, n, per, T, P, seed, ctr_dev, ctr, out, tok_state, pos_state, w_out, W_out,
                   static_cast<SampRow*>(state)};
  const dim3 grid(G, rows), block(kSampThreads);
  nt_status s = cuda_check(c, launch_k(c, samp_max_kernel, grid, block, 0, st, a), "sample launch");
  if (s || !(T > 0.f)) return s;
  for (int round = 0; round < 3 && !s; ++round)
    s = cuda_check(c, launch_k(c, samp_round_kernel, grid, block, 0, st, a, round), "sample launch");
  if (!s) s = cuda_check(c, launch_k(c, samp_count_kernel, grid, block, 0, st, a), "sample launch");
  if (!s) s = cuda_check(c, launch_k(c, samp_pick_kernel, grid, block, 0, st, a), "sample launch");
  return s;
}

nt_status launch_cos(Ctx* c, const float* a, const float* b, int64_t n, float* out, cudaStream_t st) {
  if (c->dry) return NT_OK;
  cos_kernel<<<1, 1024, 0, st>>>(a, b, n, out);
  return cuda_check(c, cudaGetLastError(), "cos launch");
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the decode attention.  Its scratch (split
// partials, error word) is this file-scope array instead
// of context memory, so the entry point needs no nt_ctx and calls neither
// cudaMalloc nor cudaFree.  Every GPU that loads the library holds the array
// until the process exits.
namespace {
constexpr size_t kAttnStaticBytes = size_t(4) << 20;  // 4 MiB
constexpr size_t kAttnStaticErr = 256;                // unsigned error word (bytes 0..255 unused)
constexpr size_t kAttnStaticPart = 512;               // split partials
static __device__ __align__(256) unsigned char g_attn_static_scratch[kAttnStaticBytes];

struct StaticAttnDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_attn_static_scratch
  int num_sms = 0;
};
constexpr int kMaxDevices = 64;
StaticAttnDevice g_static_dev[kMaxDevices];
std::mutex g_static_mu;
}  // namespace

}  // namespace nt

extern "C" nt_status nt_attn_decode_static(const float* q, const void* kc, const void* vc, float* out, int n_qh,
                                           int n_kvh, int head_dim, int64_t n_pos, int64_t kv_stride,
                                           void* stream) {
  using namespace nt;
  if (!q || !kc || !vc || !out) return NT_ERR_INVALID_ARG;
  if (head_dim != kHD) return NT_ERR_INVALID_ARG;
  if (n_kvh <= 0 || n_qh <= 0 || n_qh % n_kvh || n_kvh > 64 || !attn_kernel_for(n_qh / n_kvh)) return NT_ERR_INVALID_ARG;
  if (n_pos < 1 || n_pos > kv_stride) return NT_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(kc, 16) || !aligned(vc, 16)) return NT_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NT_ERR_CUDA;
  StaticAttnDevice* sd = &g_static_dev[dev];
  {
    // once per device, with that device current: the device address of the
    // scratch array, the SM count and the kernel's shared-memory allowance
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!sd->ready) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_attn_static_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return NT_ERR_CUDA;
      }
      int sms = 0, optin = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return NT_ERR_CUDA;
      if (configure_attn(size_t(optin)) != cudaSuccess) return NT_ERR_CUDA;
      sd->scratch = static_cast<unsigned char*>(ptr);
      sd->num_sms = sms;
      sd->ready = true;
    }
  }
  if (kv_stride > int64_t(kMaxChunk) * kMaxChunk) return NT_ERR_INVALID_ARG;
  int S = (sd->num_sms + n_kvh - 1) / n_kvh;
  const int64_t need_s = (kv_stride + kMaxChunk - 1) / kMaxChunk;
  if (need_s > S) S = int(need_s);
  if (S > kMaxChunk) S = kMaxChunk;
  const size_t part_bytes = size_t(n_kvh) * S * (n_qh / n_kvh) * kPS * sizeof(float);
  if (kAttnStaticPart + part_bytes > kAttnStaticBytes) return NT_ERR_INVALID_ARG;  // beyond the fixed scratch
  cudaStream_t st = as_stream(stream);
  AttnArgs a{};
  a.q = q;
  a.K = static_cast<const __half*>(kc);
  a.V = static_cast<const __half*>(vc);
  a.out = out;
  a.n_qh = n_qh;
  a.n_kvh = n_kvh;
  a.G = n_qh / n_kvh;
  a.S = S;
  a.n_pos = n_pos;
  a.pos_dev = nullptr;
  a.kv_stride = kv_stride;
  a.part = reinterpret_cast<float*>(sd->scratch + kAttnStaticPart);
  a.err = reinterpret_cast<unsigned*>(sd->scratch + kAttnStaticErr);
  a.nan_on_err = 1;  // no context to report a timed-out wait: the output says it
  AttnKernel k = attn_kernel_for(a.G);
  if (!k) return NT_ERR_INVALID_ARG;
  a.stall = take_stall(st);
  // the error word starts every call clear (an earlier call may have left it
  // set); each enqueue below returns its own status, so an error left by
  // unrelated earlier work is not reported as this call's
  if (cudaMemsetAsync(a.err, 0, sizeof(unsigned), st) != cudaSuccess) return NT_ERR_CUDA;
  if (launch_k(nullptr, k, dim3(n_kvh, S), dim3(kAttnThreads), attn_smem_bytes(a.G), st, a) != cudaSuccess)
    return NT_ERR_CUDA;
  if (launch_k(nullptr, attn_combine_kernel, dim3(n_kvh, a.G), dim3(kHD), 0, st, a) != cudaSuccess)
    return NT_ERR_CUDA;
  return NT_OK;
}

