// qgemm.cu — the verify GEMM of self-speculative decoding ("ntransformer -
// moteur d'inférence NVMe-to-GPU…" (fr.news.hada.io), "Fonctionnalités
// principales": the VRAM-resident layers draft, the whole model verifies):
// Y[m] = W X[m] for M <= 8 activation vectors, every weight byte read once.
//
// GB300 design.  Two forms.  The integer form (every format) keeps the
// contraction on the integer pipes: the same 24-bit fixed-point x planes and
// dp4a dot products as the M = 1 GEMV, with the weights staged once per CTA
// and reused for all M vectors.  The tensor-core form (below) serves Q8_0,
// Q4_K and Q6_K whenever the part rows meet the bulk-copy alignment.
//  * grid (X, P): the columns are cut into P parts (2048 columns; 1024 /
//    512 for F16 / F32) so that M vectors of x fit in shared memory; CTA
//    (x, p) holds part p of every vector and walks row groups of R = 2 rows.
//  * each warp streams its rows' part through a private ring of TMA bulk
//    copies (mbarrier completion, L2 evict-first), as the GEMV does.
//  * partial sums go to scratch [P][M][rows]; a second kernel adds the P
//    parts in a fixed order (results do not depend on scheduling) and
//    applies the epilogue: residual add, SwiGLU, RoPE at position pos + m,
//    or the f16 KV-cache append at pos + m.
//
// Tensor-core form (Q8_0, Q4_K, Q6_K; qgemm_mma_kernel below).  The dp4a
// form pays 3 byte-plane dp4a per weight for every one of the M vectors; an
// MMA multiplies a 16-row tile of weights by all 8 vector slots at once, so
// each weight is unpacked once and the per-vector cost nearly vanishes:
//  * the quants are small integers, exact in f16 (Q8_0 q, Q4_K q, Q6_K
//    q - 32); they go straight from the staged block bytes into the A
//    fragments of mma.sync m16n8k16 (f16 in, fp32 accumulate);
//  * x is split into two f16 terms, hi = f16(x s) and lo = f16(x s - hi),
//    with a power-of-two s per vector and part, so hi + lo carries x to
//    about 2^-22; two MMAs per k-step, one per term;
//  * the MMA's 16 k-indices are mapped to the physical columns so that
//    each thread's four weights of a row are one contiguous 4-byte word;
//  * block (and sub-block) scales multiply the fp32 accumulator fragment
//    once per block; the K-quant mins subtract dmin m_j sum(x) per
//    sub-block from precomputed sums of x;
//  * each warp owns whole 16-row tiles of its CTA's column part and streams
//    them through a private ring of bulk copies, so no barrier or reduction
//    joins the warps; the parts are narrowed for small matrices (a
//    function of the shape alone) so that every SM has tiles to work on.
#include "nt_internal.cuh"
#include "ops.cuh"
#include "qformats.cuh"

namespace nt {
namespace {

using namespace qf;

constexpr int kGemmWarps = 8;
constexpr int kGemmThreads = kGemmWarps * 32;
constexpr int kGemmStages = 4;  // per warp
constexpr int kGemmR = 2;       // rows per group
// columns per part: 2048 for the quantized formats; the float formats carry
// 2 or 4 bytes per weight, so their parts are narrower (2 KB of each row)
__host__ __device__ constexpr int part_cols(int fmt) { return fmt == NT_F32 ? 512 : fmt == NT_F16 ? 1024 : 2048; }

struct GemmJobDev {
  const uint8_t* W;
  int64_t rows;
  int64_t g0;    // first row group of the job
  int64_t rb;    // first row of the job in the concatenated row space
};

struct GemmArgs {
  GemmJobDev job[3];
  int njobs;
  int64_t total_groups;
  int64_t total_rows;
  const float* X;
  int64_t ldx;
  const float* norm_g;
  float eps;
  int M;
  int cols, nb, cwb, nparts;
  int64_t rowB;
  int segStride;  // bytes between the rows of one stage
  int stb;        // bytes per stage
  int vstride;    // shared bytes per vector (planes, scales, plane sums)
  int tma;
  float* part;    // [nparts][M][total_rows]
  unsigned* err;
};

__device__ __forceinline__ void gemm_locate(const GemmArgs& a, int64_t g, int& j, int64_t& r0, int& nr) {
  j = 0;
  while (j + 1 < a.njobs && g >= a.job[j + 1].g0) ++j;
  r0 = (g - a.job[j].g0) * kGemmR;
  const int64_t left = a.job[j].rows - r0;
  nr = left < kGemmR ? int(left) : kGemmR;
}

template <int FMT>
__global__ void __launch_bounds__(kGemmThreads, 1) qgemm_kernel(const GemmArgs a) {
  using F = Q<FMT>;
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int R = kGemmR, S = kGemmStages;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p = blockIdx.y;
  const int blk_lo = p * a.cwb;
  const int blk_hi = min(a.nb, blk_lo + a.cwb);
  const int ngp = (blk_hi - blk_lo) * F::BE / 32;  // 32-column groups of this part
  const int ngmax = a.cwb * F::BE / 32;
  const int xB = x_bytes<FMT>(a.cwb * F::BE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.M * a.vstride);
  uint8_t* stages = smem + ((a.M * a.vstride + kGemmWarps * S * 8 + 127) / 128) * 128;
  uint8_t* st0 = stages + size_t(warp) * S * a.stb;
  const uint32_t bar0 = smem_u32(bars + warp * S);

  const int64_t nw_total = int64_t(gridDim.x) * kGemmWarps;
  const int64_t wg = int64_t(blockIdx.x) * kGemmWarps + warp;
  const int my_groups = wg < a.total_groups ? int((a.total_groups - wg + nw_total - 1) / nw_total) : 0;
  const int n_items = my_groups;  // a stage holds the whole part of R rows

  if (a.tma) {
    if (lane == 0) {
      for (int s = 0; s < S; ++s) mbar_init(bar0 + 8 * s, 1);
      fence_barrier_init();
    }
    __syncwarp();
  }
  const uint64_t pol = policy_evict_first();

  // ---- issue cursor
  int it_t = 0, it_slot = 0;
  auto fill = [&](int t, int slot) {
    int j, nr;
    int64_t r0;
    gemm_locate(a, wg + int64_t(t) * nw_total, j, r0, nr);
    uint8_t* st = st0 + size_t(slot) * a.stb;
    const uint32_t bytes_row = uint32_t(blk_hi - blk_lo) * F::BB;
    const uint8_t* src = a.job[j].W + r0 * a.rowB + size_t(blk_lo) * F::BB;
    if (a.tma) {
      const uint32_t bar = bar0 + 8 * uint32_t(slot);
      if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(nr) * bytes_row);
      __syncwarp();
      if (lane < nr) bulk_g2s(smem_u32(st + lane * a.segStride), src + lane * a.rowB, bytes_row, bar, pol);
    } else {
      for (int i = 0; i < nr; ++i)
        for (uint32_t b = lane; b < bytes_row; b += 32) st[i * a.segStride + b] = src[i * a.rowB + b];
      __syncwarp();
    }
  };
  auto issue_next = [&]() {
    fill(it_t, it_slot);
    ++it_t;
    if (++it_slot == S) it_slot = 0;
  };
  if (a.tma) {
    const int pre = n_items < S - 1 ? n_items : S - 1;
    for (int k = 0; k < pre; ++k) issue_next();
  }
  pdl_trigger();
  pdl_wait();

  // ---- prologue: the part's columns of every vector -> 24-bit planes
  {
    __shared__ float inv_s[8];
    if (a.norm_g) {
      // RMSNorm needs the whole row of each vector
      for (int m = warp; m < a.M; m += kGemmWarps) {
        const float* xr = a.X + int64_t(m) * a.ldx;
        float ss = 0.f;
        for (int c = 4 * lane; c < a.cols; c += 128) {
          const float4 t = *reinterpret_cast<const float4*>(xr + c);
          ss = fmaf(t.x, t.x, fmaf(t.y, t.y, fmaf(t.z, t.z, fmaf(t.w, t.w, ss))));
        }
        ss = warp_sum(ss);
        if (lane == 0) inv_s[m] = rsqrtf(ss / float(a.cols) + a.eps);
      }
      __syncthreads();
    }
    const int sub = lane & 7;
    const int total = a.M * ngp;
    const int stride = kGemmWarps * 4;
    const int npass = (total - warp * 4 + stride - 1) / stride;  // warp-uniform, may be <= 0
    for (int k = 0; k < npass; ++k) {
      const int idx = warp * 4 + k * stride + (lane >> 3);
      const bool live = idx < total;
      const int m = live ? idx / ngp : 0, gl = live ? idx % ngp : 0;
      float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
      const int col = blk_lo * F::BE + 32 * gl + 4 * sub;
      if (live) {
        x4 = *reinterpret_cast<const float4*>(a.X + int64_t(m) * a.ldx + col);
        if (a.norm_g) {
          const float inv = inv_s[m];
          const float4 g = *reinterpret_cast<const float4*>(a.norm_g + col);
          x4.x = x4.x * inv * g.x;
          x4.y = x4.y * inv * g.y;
          x4.z = x4.z * inv * g.z;
          x4.w = x4.w * inv * g.w;
        }
      }
      uint8_t* xm = smem + m * a.vstride;
      put_x4<FMT>(x4, live, gl, sub, xm, reinterpret_cast<int*>(xm + xB + 4 * ngmax),
                  reinterpret_cast<float*>(xm + xB));
    }
    __syncthreads();
  }
  if (my_groups == 0) return;

  float acc[R][8];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[i][m] = 0.f;

  int cs = 0;
  uint32_t cph = 0;
  bool dead = false;
  const int units = (blk_hi - blk_lo) * F::UPB;
  for (int k = 0; k < n_items; ++k) {
    uint8_t* st = st0 + size_t(cs) * a.stb;
    if (dead) {
    } else if (a.tma) {
      if (k + S - 1 < n_items) issue_next();
      const bool ok = mbar_wait(bar0 + 8 * uint32_t(cs), cph);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) flag_error(a.err, kErrWaitTimeout);
        int q = cs;
        uint32_t ph = cph;
        for (int n = k + 1; n < min(n_items, k + S - 1); ++n) {
          if (++q == S) {
            q = 0;
            ph ^= 1u;
          }
          mbar_wait(bar0 + 8 * uint32_t(q), ph);
        }
        dead = true;
      }
    } else {
      issue_next();
    }
    if (!dead) {
      for (int u = lane; u < units; u += 32) {
        const int b = u / F::UPB, uu = u % F::UPB;
        const int col0 = b * F::BE;  // column within the part
        const uint8_t* bp = st + b * F::BB;
        // the R rows' weights of this unit are unpacked once and serve all M vectors
        typename F::W w[R];
#pragma unroll
        for (int i = 0; i < R; ++i) F::unpack(bp + i * a.segStride, uu, w[i]);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          if (m < a.M) {
            const uint8_t* xm = smem + m * a.vstride;
            const XS xs{xm, reinterpret_cast<const float*>(xm + xB), reinterpret_cast<const int*>(xm + xB + 4 * ngmax)};
            typename F::X x;
            F::load_x(x, xm + goff<FMT>(col0 / 32 + (F::UPB == 4 && FMT != NT_Q6_K ? 2 * uu : 0)), xs, col0, uu);
#pragma unroll
            for (int i = 0; i < R; ++i) acc[i][m] += F::dotw(w[i], uu, x);
          }
        }
      }
    }
    __syncwarp();
    // group done: lane sums, partials to scratch
    {
      int j, nr;
      int64_t r0;
      gemm_locate(a, wg + int64_t(k) * nw_total, j, r0, nr);
      const int64_t row = a.job[j].rb + r0;
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          if (m < a.M) {
            const float v = warp_sum(acc[i][m]);
            if (lane == 0 && i < nr) a.part[(int64_t(p) * a.M + m) * a.total_rows + row + i] = v;
          }
          acc[i][m] = 0.f;
        }
    }
    if (++cs == S) {
      cs = 0;
      cph ^= 1u;
    }
  }
}

// ---- the P parts added in order, then the epilogue of each job
struct EpiJob {
  float* y;           // [M][ldy] outputs (plain, rope)
  const float* res;   // [M][ldy] residual (plain), nullable
  __half* cache;      // cache epilogues: [n_kvh][kv_stride][head_dim]
  int64_t ldy;
  int64_t rows;
  int64_t rb;         // first row in the concatenated row space
  int64_t pb;         // first row pair of the job
  int epi;
};

struct EpiArgs {
  EpiJob job[3];
  int njobs;
  int64_t total_pairs;
  int64_t total_rows;
  int M, nparts;
  int swiglu;         // job 0 = gate rows, job 1 = up rows; output job 0's y
  const float* part;
  RopeArgs rope;
  unsigned* err;
};

__global__ void qgemm_epi_kernel(const EpiArgs e) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.y;
  auto sum_row = [&](int64_t row) {
    float v = 0.f;
#pragma unroll 8
    for (int p = 0; p < e.nparts; ++p) v += __ldcg(e.part + (int64_t(p) * e.M + m) * e.total_rows + row);
    return v;
  };
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  if (e.swiglu) {
    const EpiJob& G = e.job[0];
    const EpiJob& U = e.job[1];
    for (int64_t r = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; r < G.rows; r += stride)
      G.y[m * G.ldy + r] = silu(sum_row(G.rb + r)) * sum_row(U.rb + r);
    return;
  }
  for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < e.total_pairs; t += stride) {
    int j = 0;
    while (j + 1 < e.njobs && t >= e.job[j + 1].pb) ++j;
    const EpiJob& J = e.job[j];
    const int64_t r = 2 * (t - J.pb);
    const bool two = r + 1 < J.rows;
    const float v0 = sum_row(J.rb + r);
    const float v1 = two ? sum_row(J.rb + r + 1) : 0.f;
    if (J.epi == kEpiPlain) {
      float* y = J.y + m * J.ldy;
      const float* rs = J.res ? J.res + m * J.ldy : nullptr;
      y[r] = rs ? v0 + rs[r] : v0;
      if (two) y[r + 1] = rs ? v1 + rs[r + 1] : v1;
      continue;
    }
    // adjacent (even, odd) pairs at position pos + m
    const int hd = e.rope.head_dim;
    const int64_t pos = *e.rope.pos_dev + m;
    const int head = int(r / hd), d = int(r % hd);
    float o0 = v0, o1 = v1;
    if (J.epi != kEpiCache) {
      float cs_, sn;
      rope_cs(pos, e.rope.inv_freq[d >> 1], cs_, sn);
      o0 = fmaf(v0, cs_, -v1 * sn);
      o1 = fmaf(v0, sn, v1 * cs_);
    }
    if (J.epi == kEpiRope) {
      J.y[m * J.ldy + r] = o0;
      J.y[m * J.ldy + r + 1] = o1;
    } else if (pos >= 0 && pos < e.rope.kv_stride) {
      __half* c = J.cache + (int64_t(head) * e.rope.kv_stride + pos) * hd + d;
      c[0] = __float2half_rn(o0);
      c[1] = __float2half_rn(o1);
    } else {
      flag_error(e.err, kErrPosRange);
    }
  }
}

// ---------------------------------------------------------------------------
// Tensor-core form: mma.sync m16n8k16 (f16 x f16 -> f32), 16-row tiles.
constexpr int kMmaWarps = 12;                     // warps per CTA at most (the rings of more do not fit)
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kMmaRows = 16;                      // rows per tile (the MMA's m)

constexpr int kMaxChunksRms = 1024;  // 128-column chunks: vectors of up to 131072 columns

struct MmaArgs {
  GemmJobDev job[3];  // g0: first 16-row tile of the job; rb: first row in the row space
  int njobs;
  int64_t total_tiles;
  int64_t total_rows;
  const float* X;
  int64_t ldx;
  const float* norm_g;
  float eps;
  int M;
  int cols, nb, cwb, nparts;
  int64_t rowB;
  int segB;  // stage bytes per row (the part's blocks, rounded up to 16)
  int SB;    // bytes per stage (16 rows)
  int NS;    // stages
  float* part;
  unsigned* err;
  int stall;
  const float* inv;  // with norm_g: rsqrt(mean x_m^2 + eps) per vector, from rms_inv_kernel
};

// The RMSNorm scalar of each of the M vectors, once per launch instead of in
// every CTA: block m sums x_m^2 per 128-column chunk (one warp per chunk),
// then over the chunks in index order, and writes rsqrt(mean + eps).
__global__ void __launch_bounds__(256) rms_inv_kernel(const float* X, int64_t ldx, int cols, float eps, float* inv) {
  __shared__ float red[kMaxChunksRms];
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const float* xr = X + int64_t(m) * ldx;
  const int nchunk = (cols + 127) / 128;
  for (int ch = warp; ch < nchunk; ch += nwarps) {
    const int c = 128 * ch + 4 * lane;
    float ss = 0.f;
    if (c < cols) {
      const float4 v = *reinterpret_cast<const float4*>(xr + c);
      ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, v.w * v.w)));
    }
    ss = warp_sum(ss);
    if (lane == 0) red[ch] = ss;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int ch = 0; ch < nchunk; ++ch) tot += red[ch];
    inv[m] = rsqrtf(tot / float(cols) + eps);
  }
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// bytes 0,1 (lo) or 2,3 (hi) of w, each an unsigned value u < 1024, as the
// f16 pair (u - bias): f16(1024 + u) is exact, built by placing u in the
// mantissa under the exponent of 1024
__device__ __forceinline__ uint32_t u8lo_f16(uint32_t w, uint32_t bias2) { return hsub2(__byte_perm(w, 0x64646464u, 0x4140), bias2); }
__device__ __forceinline__ uint32_t u8hi_f16(uint32_t w, uint32_t bias2) { return hsub2(__byte_perm(w, 0x64646464u, 0x4342), bias2); }
constexpr uint32_t kBias1024 = 0x64006400u;  // f16 pair (1024, 1024)
constexpr uint32_t kBias1056 = 0x64206420u;  // (1056, 1056): 1024 + the Q6_K offset 32
constexpr uint32_t kBias1152 = 0x64806480u;  // (1152, 1152): 1024 + 128 for sign-flipped int8


template <int FMT>
struct MmaRows;

// The vectors come in N-tiles of 8 (the MMA's n): NT tiles, the x of tile
// nt at xh + nt * xt (and xl + nt * xt), the sums of x of vector n at
// xs[group * 8 NT + n]; acc[nt] holds the fragment of tile nt.

// Q8_0: per block (32 columns, 2 k-steps) the 4-byte words of qs for rows
// g and g + 8, signed -> f16; one scale d per row and block.
template <>
struct MmaRows<NT_Q8_0> {
  // block b of a staged row whose first byte is 4-byte aligned (R0, R1: rows
  // g and g + 8 as words).  Blocks come in pairs of 68 bytes = 17 words: the
  // even block's quants sit 2 bytes off a word boundary (one funnel shift by
  // 16 per word), the odd block's are word-aligned.
  template <int NT>
  __device__ static void block_w(const uint32_t* R0, const uint32_t* R1, int b, int t, int c0, const uint32_t* xh,
                                 const uint32_t* xl, int xt, float (&acc)[NT][4]) {
    const int pw = 17 * (b >> 1);
    float d0, d1;
    uint32_t w[2][2];  // [sub][row]
    if ((b & 1) == 0) {
      d0 = qf::h2f(R0[pw] & 0xFFFFu);
      d1 = qf::h2f(R1[pw] & 0xFFFFu);
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        const int k = pw + 4 * sub + t;
        w[sub][0] = __funnelshift_r(R0[k], R0[k + 1], 16);
        w[sub][1] = __funnelshift_r(R1[k], R1[k + 1], 16);
      }
    } else {
      d0 = qf::h2f(R0[pw + 8] >> 16);
      d1 = qf::h2f(R1[pw + 8] >> 16);
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        const int k = pw + 9 + 4 * sub + t;
        w[sub][0] = R0[k];
        w[sub][1] = R1[k];
      }
    }
    float c[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
    for (int sub = 0; sub < 2; ++sub) {
      const uint32_t w0 = w[sub][0] ^ 0x80808080u, w1 = w[sub][1] ^ 0x80808080u;
      const uint32_t a[4] = {u8lo_f16(w0, kBias1152), u8lo_f16(w1, kBias1152), u8hi_f16(w0, kBias1152),
                             u8hi_f16(w1, kBias1152)};
      const int col = c0 + 16 * sub;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint2 bh = *reinterpret_cast<const uint2*>(xh + nt * xt + col / 2);
        const uint2 bl = *reinterpret_cast<const uint2*>(xl + nt * xt + col / 2);
        mma16816(c[nt], a, bh.x, bh.y);
        mma16816(c[nt], a, bl.x, bl.y);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc[nt][0] = fmaf(d0, c[nt][0], acc[nt][0]);
      acc[nt][1] = fmaf(d0, c[nt][1], acc[nt][1]);
      acc[nt][2] = fmaf(d1, c[nt][2], acc[nt][2]);
      acc[nt][3] = fmaf(d1, c[nt][3], acc[nt][3]);
    }
  }
};

// Q4_K: per block (256 columns): for each pair of sub-blocks (2c, 2c+1) the
// words of qs[32c..32c+31] give both sub-blocks' quants (low / high
// nibbles); scale d sc_j and min dmin m_j per row and sub-block.
template <>
struct MmaRows<NT_Q4_K> {
  // half-block hb: the half `half` (sub-block pairs 2 half, 2 half + 1) of block b = hb / 2
  template <int NT>
  __device__ static void half_block(const uint8_t* r0, const uint8_t* r1, int hb, int nblk, int t,
                                    const uint32_t* xh, const uint32_t* xl, int xt, const float* xs,
                                    float (&acc)[NT][4]) {
    constexpr int MV = 8 * NT;
    const int b = hb >> 1, half = hb & 1;
    if (b >= nblk) return;
    const uint8_t* p0 = r0 + b * 144;
    const uint8_t* p1 = r1 + b * 144;
    const int c0 = b * 256;
    const uint4 h0 = *reinterpret_cast<const uint4*>(p0);
    const uint4 h1 = *reinterpret_cast<const uint4*>(p1);
    const float d0 = qf::h2f(h0.x & 0xFFFFu), dm0 = qf::h2f(h0.x >> 16);
    const float d1 = qf::h2f(h1.x & 0xFFFFu), dm1 = qf::h2f(h1.x >> 16);
    // with two N-tiles the sub-block pairs go one at a time (register room)
#pragma unroll(3 - NT)
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * half + cc;
      float sa0, sb0, ma0, mb0, sa1, sb1, ma1, mb1;
      qf::kq_scales(h0.y, h0.z, h0.w, c, sa0, sb0, ma0, mb0);
      qf::kq_scales(h1.y, h1.z, h1.w, c, sa1, sb1, ma1, mb1);
      float ca[NT][4], cb[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) ca[nt][e] = cb[nt][e] = 0.f;
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(p0 + 16 + 32 * c + 16 * s + 4 * t);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(p1 + 16 + 32 * c + 16 * s + 4 * t);
        const uint32_t l0 = w0 & 0x0F0F0F0Fu, l1 = w1 & 0x0F0F0F0Fu;
        const uint32_t u0 = (w0 >> 4) & 0x0F0F0F0Fu, u1 = (w1 >> 4) & 0x0F0F0F0Fu;
        const uint32_t al[4] = {u8lo_f16(l0, kBias1024), u8lo_f16(l1, kBias1024), u8hi_f16(l0, kBias1024),
                                u8hi_f16(l1, kBias1024)};
        const uint32_t au[4] = {u8lo_f16(u0, kBias1024), u8lo_f16(u1, kBias1024), u8hi_f16(u0, kBias1024),
                                u8hi_f16(u1, kBias1024)};
        const int colA = c0 + 64 * c + 16 * s, colB = colA + 32;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 bha = *reinterpret_cast<const uint2*>(xh + nt * xt + colA / 2);
          const uint2 bla = *reinterpret_cast<const uint2*>(xl + nt * xt + colA / 2);
          const uint2 bhb = *reinterpret_cast<const uint2*>(xh + nt * xt + colB / 2);
          const uint2 blb = *reinterpret_cast<const uint2*>(xl + nt * xt + colB / 2);
          mma16816(ca[nt], al, bha.x, bha.y);
          mma16816(ca[nt], al, bla.x, bla.y);
          mma16816(cb[nt], au, bhb.x, bhb.y);
          mma16816(cb[nt], au, blb.x, blb.y);
        }
      }
      // sums of x over the two sub-blocks for this thread's vectors 8 nt + 2t, 8 nt + 2t + 1
      const int grp = (c0 + 64 * c) / 32;
      const float ka0 = d0 * sa0, kb0 = d0 * sb0, ka1 = d1 * sa1, kb1 = d1 * sb1;
      const float na0 = dm0 * ma0, nb0 = dm0 * mb0, na1 = dm1 * ma1, nb1 = dm1 * mb1;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float2 xa = *reinterpret_cast<const float2*>(xs + grp * MV + 8 * nt + 2 * t);
        const float2 xb = *reinterpret_cast<const float2*>(xs + (grp + 1) * MV + 8 * nt + 2 * t);
        acc[nt][0] += fmaf(ka0, ca[nt][0], fmaf(kb0, cb[nt][0], -fmaf(na0, xa.x, nb0 * xb.x)));
        acc[nt][1] += fmaf(ka0, ca[nt][1], fmaf(kb0, cb[nt][1], -fmaf(na0, xa.y, nb0 * xb.y)));
        acc[nt][2] += fmaf(ka1, ca[nt][2], fmaf(kb1, cb[nt][2], -fmaf(na1, xa.x, nb1 * xb.x)));
        acc[nt][3] += fmaf(ka1, ca[nt][3], fmaf(kb1, cb[nt][3], -fmaf(na1, xa.y, nb1 * xb.y)));
      }
    }
  }
};

// Q6_K: per block (256 columns) and half h, step s: the words of ql (two
// runs) and qh give the 6-bit quants of the four 16-column sub-blocks
// (g = 0..3); q - 32 as f16; scale d sc per row and sub-block.
template <>
struct MmaRows<NT_Q6_K> {
  // half-block hb: the half h = hb & 1 (128 columns) of block hb / 2
  template <int NT>
  __device__ static void half_block(const uint8_t* r0, const uint8_t* r1, int hb, int nblk, int t,
                                    const uint32_t* xh, const uint32_t* xl, int xt, const float*,
                                    float (&acc)[NT][4]) {
    const int b = hb >> 1, h = hb & 1;
    if (b >= nblk) return;
    const uint8_t* p0 = r0 + b * 210;
    const uint8_t* p1 = r1 + b * 210;
    const int c0 = b * 256;
    const float d0 = __half2float(*reinterpret_cast<const __half*>(p0 + 208));
    const float d1 = __half2float(*reinterpret_cast<const __half*>(p1 + 208));
    // a segment's first block starts 4-byte aligned (a multiple of 420 bytes
    // plus the 16-byte-aligned copy's offset, a multiple of 4): block 0 of a
    // pair is word-aligned, block 1 sits 2 bytes off (a funnel shift by 16)
    // (with two N-tiles the runtime-checked form measured faster: register room)
    auto ldw = [&](const uint8_t* p, int off) -> uint32_t {
      if constexpr (NT == 1) {
        if (b % 2 == 0) return *reinterpret_cast<const uint32_t*>(p + off);
        const uint32_t* w = reinterpret_cast<const uint32_t*>(p + off - 2);
        return __funnelshift_r(w[0], w[1], 16);
      } else {
        const uint32_t mis = smem_u32(p + off) & 2u;
        const uint32_t* w = reinterpret_cast<const uint32_t*>(p + off - mis);
        return mis ? __funnelshift_r(w[0], w[1], 16) : w[0];
      }
    };
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int lo = 64 * h + 16 * s + 4 * t, qh = 128 + 32 * h + 16 * s + 4 * t;
      const uint32_t A0 = ldw(p0, lo), B0 = ldw(p0, lo + 32), H0 = ldw(p0, qh);
      const uint32_t A1 = ldw(p1, lo), B1 = ldw(p1, lo + 32), H1 = ldw(p1, qh);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint32_t L0 = (g & 1) ? B0 : A0, L1 = (g & 1) ? B1 : A1;
        const int nib = 4 * (g >> 1);
        const uint32_t q0 = ((L0 >> nib) & 0x0F0F0F0Fu) | (((H0 >> (2 * g)) & 0x03030303u) << 4);
        const uint32_t q1 = ((L1 >> nib) & 0x0F0F0F0Fu) | (((H1 >> (2 * g)) & 0x03030303u) << 4);
        const uint32_t a[4] = {u8lo_f16(q0, kBias1056), u8lo_f16(q1, kBias1056), u8hi_f16(q0, kBias1056),
                               u8hi_f16(q1, kBias1056)};
        const int col = c0 + 128 * h + 32 * g + 16 * s;
        const int j = 8 * h + 2 * g + s;  // sub-block: scales[j]
        const float k0 = d0 * float(*reinterpret_cast<const int8_t*>(p0 + 192 + j));
        const float k1 = d1 * float(*reinterpret_cast<const int8_t*>(p1 + 192 + j));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 bh = *reinterpret_cast<const uint2*>(xh + nt * xt + col / 2);
          const uint2 bl = *reinterpret_cast<const uint2*>(xl + nt * xt + col / 2);
          float c[4] = {0.f, 0.f, 0.f, 0.f};
          mma16816(c, a, bh.x, bh.y);
          mma16816(c, a, bl.x, bl.y);
          acc[nt][0] = fmaf(k0, c[0], acc[nt][0]);
          acc[nt][1] = fmaf(k0, c[1], acc[nt][1]);
          acc[nt][2] = fmaf(k1, c[2], acc[nt][2]);
          acc[nt][3] = fmaf(k1, c[3], acc[nt][3]);
        }
      }
    }
  }
};

__device__ __forceinline__ void mma_locate(const MmaArgs& a, int64_t tile, int& j, int64_t& r0, int& nr) {
  j = 0;
  while (j + 1 < a.njobs && tile >= a.job[j + 1].g0) ++j;
  r0 = (tile - a.job[j].g0) * kMmaRows;
  const int64_t left = a.job[j].rows - r0;
  nr = left < kMmaRows ? int(left) : kMmaRows;
}

// shared layout for MV vector slots, sized by the part's columns pc: x hi
// [MV][pc + 16] f16, x lo [MV][pc + 16] f16 (the extra 32 bytes per vector
// keep the B loads free of bank conflicts), sums of x [pc / 32][MV] f32,
// vector scales [MV], stage barriers [warps][NS], then each warp's ring of NS
// stages of 16 staged rows
struct MmaLayout {
  size_t xl, xs, sc, bar, ring;
};
__host__ __device__ inline MmaLayout mma_layout(int pc, int MV, int warps, int NS) {
  MmaLayout L;
  const size_t pitch = size_t(pc) + 16;
  L.xl = size_t(MV) * pitch * 2;
  L.xs = L.xl + size_t(MV) * pitch * 2;
  L.sc = L.xs + size_t(pc / 32) * MV * 4;
  L.bar = L.sc + size_t(MV) * 4 + 32;
  L.ring = ((L.bar + size_t(warps) * NS * 8 + 127) / 128) * 128;
  return L;
}

// blocks per staged segment of a row: about 512 bytes of weights per row
// (each row copy moves that much; segments half this size measured up to
// 19% slower)
__host__ __device__ constexpr int mma_seg_blocks(int fmt) { return fmt == NT_Q8_0 ? 16 : fmt == NT_Q4_K ? 4 : 2; }

// one segment of 16 rows: the blocks [0, nbk) of the segment, r0 and r1
// pointing at its first byte in the staged rows g and g + 8
template <int FMT, int NT>
__device__ __forceinline__ void mma_segment(const uint8_t* r0, const uint8_t* r1, int nbk, int t, const uint32_t* xh,
                                            const uint32_t* xl, int xt, const float* xs, float (&acc)[NT][4]) {
  constexpr int S = mma_seg_blocks(FMT);
  // a whole segment is straight-line code (every offset a constant); a
  // part's ragged last segment takes the loop
  if constexpr (FMT == NT_Q8_0) {
    // a segment starts at a multiple of 16 blocks (544 bytes) from a 16-byte
    // aligned row start: word-aligned
    const uint32_t* R0 = reinterpret_cast<const uint32_t*>(r0);
    const uint32_t* R1 = reinterpret_cast<const uint32_t*>(r1);
    if (nbk == S) {
#pragma unroll
      for (int b = 0; b < S; ++b) MmaRows<FMT>::template block_w<NT>(R0, R1, b, t, b * 32, xh, xl, xt, acc);
    } else {
#pragma unroll 1
      for (int b = 0; b < nbk; ++b) MmaRows<FMT>::template block_w<NT>(R0, R1, b, t, b * 32, xh, xl, xt, acc);
    }
  } else {
    if (nbk == S) {
#pragma unroll
      for (int h = 0; h < 2 * S; ++h) MmaRows<FMT>::template half_block<NT>(r0, r1, h, S, t, xh, xl, xt, xs, acc);
    } else {
#pragma unroll 1
      for (int h = 0; h < 2 * nbk; ++h)
        MmaRows<FMT>::template half_block<NT>(r0, r1, h, nbk, t, xh, xl, xt, xs, acc);
    }
  }
}

// Each warp owns whole 16-row tiles of its CTA's column part: it walks the
// part in segments through its own ring of bulk copies (16 row copies per
// stage, mbarrier completion), accumulates the MMA results of every segment
// in registers, and writes the tile's partial sums itself.  No two warps
// share a tile, so there is no barrier and no reduction between warps.
template <int FMT, int NT>
__global__ void __launch_bounds__(kMmaThreads, 1) qgemm_mma_kernel(const MmaArgs a) {
  using F = Q<FMT>;
  constexpr int S = mma_seg_blocks(FMT);
  constexpr int MV = 8 * NT;  // vector slots
  extern __shared__ __align__(128) uint8_t smem[];
  const int NS = a.NS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int xpitch = a.cwb * F::BE + 16;  // f16 per staged x vector
  const MmaLayout L = mma_layout(a.cwb * F::BE, MV, nwarps, NS);
  __half* xh = reinterpret_cast<__half*>(smem);
  __half* xl = reinterpret_cast<__half*>(smem + L.xl);
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  float* xsc = reinterpret_cast<float*>(smem + L.sc);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar) + warp * NS;
  uint8_t* ring = smem + L.ring + size_t(warp) * NS * a.SB;
  const int g = lane >> 2, t = lane & 3;
  const int p = blockIdx.y;
  const int blk_lo = p * a.cwb;
  const int blk_hi = min(a.nb, blk_lo + a.cwb);
  const int pcols = (blk_hi - blk_lo) * F::BE;  // columns of this part
  const int nseg = (blk_hi - blk_lo + S - 1) / S;
  // this warp's tiles: ws, ws + stride, ...
  const int64_t ws = int64_t(blockIdx.x) * nwarps + warp, stride = int64_t(gridDim.x) * nwarps;
  const int ntiles = ws < a.total_tiles ? int((a.total_tiles - ws + stride - 1) / stride) : 0;
  const int n_items = ntiles * nseg;
  const uint64_t pol = policy_evict_first();
  const int cap = a.stall ? kStallSpin : kMaxSpin;

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(smem_u32(full + s), 1);
    fence_barrier_init();
  }
  __syncwarp();
  // item i = (tile ws + (i / nseg) stride, segment i % nseg) into stage i % NS.
  // Each row's segment is copied as the 16-byte-aligned range around it
  // (rows start 16-byte aligned, so the range stays inside the row); the
  // segment's bytes start `o` bytes into the staged row.
  auto seg_off = [&](int sg) { return int((int64_t(blk_lo + sg * S) * F::BB) & 15); };
  // issue cursor: tile ordinal, segment, stage slot; the tile's rows cached
  int it_t = 0, it_sg = 0, it_slot = 0, it_nr = 0;
  const uint8_t* it_row = nullptr;  // lane < 16: its row of the issue tile (null past the tile's rows)
  auto issue_next = [&]() {
    if (it_sg == 0) {
      int j;
      int64_t r0;
      mma_locate(a, ws + int64_t(it_t) * stride, j, r0, it_nr);
      it_row = lane < it_nr ? a.job[j].W + (r0 + lane) * a.rowB : nullptr;
    }
    const int b0 = blk_lo + it_sg * S, nbk = min(S, blk_hi - b0);
    const int64_t lo = int64_t(b0) * F::BB, hi = lo + int64_t(nbk) * F::BB;
    const int64_t lo16 = lo & ~int64_t(15), hi16 = (hi + 15) & ~int64_t(15);
    const uint32_t bytes = uint32_t(hi16 - lo16);
    const uint32_t bar = smem_u32(full + it_slot);
    if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(it_nr) * bytes);
    __syncwarp();
    if (it_row && !a.stall)
      bulk_g2s(smem_u32(ring + size_t(it_slot) * a.SB + size_t(lane) * a.segB), it_row + lo16, bytes, bar, pol);
    if (++it_sg == nseg) {
      it_sg = 0;
      ++it_t;
    }
    if (++it_slot == NS) it_slot = 0;
  };
  // weights do not depend on x: start streaming before waiting for its producer
  const int pre = n_items < NS - 1 ? n_items : NS - 1;
  for (int i = 0; i < pre; ++i) issue_next();
  pdl_trigger();
  pdl_wait();

  // ---- prologue: warp w converts vectors w, w + warps, ... < MV (zeros for
  // m >= M): the part's columns, RMS-normalised when asked, scaled by a power
  // of two, split into f16 hi + lo, and the sums of x over each 32 columns
  // (scaled likewise)
  for (int m = warp; m < MV; m += nwarps) {
    float inv = 1.f;
    const float* xr = a.X + int64_t(m) * a.ldx;
    if (m < a.M && a.norm_g) inv = a.inv[m];
    // lane l holds columns 64 l .. 64 l + 63 of the part: 16 float4, loaded
    // together (one memory round trip)
    float4 xv[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int col = 64 * lane + 4 * k;
      float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m < a.M && col < pcols) {
        const int gc = blk_lo * F::BE + col;
        x4 = *reinterpret_cast<const float4*>(xr + gc);
        if (a.norm_g) {
          const float4 gg = *reinterpret_cast<const float4*>(a.norm_g + gc);
          x4.x = x4.x * inv * gg.x;
          x4.y = x4.y * inv * gg.y;
          x4.z = x4.z * inv * gg.z;
          x4.w = x4.w * inv * gg.w;
        }
      }
      xv[k] = x4;
    }
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k)
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(xv[k].x), fabsf(xv[k].y)), fmaxf(fabsf(xv[k].z), fabsf(xv[k].w))));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // scale 2^sh puts the vector's largest |x| in [2^13, 2^14): far inside the f16 range
    int sh = 0;
    if (mx > 0.f) sh = min(100, max(-100, 13 - (int((__float_as_uint(mx) >> 23) & 0xFFu) - 127)));
    const float scl = ldexpf(1.f, sh);
    if (lane == 0) xsc[m] = m < a.M ? ldexpf(1.f, -sh) : 0.f;
    __half* hr = xh + m * xpitch;
    __half* lr = xl + m * xpitch;
    float gs0 = 0.f, gs1 = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float e[4] = {xv[k].x * scl, xv[k].y * scl, xv[k].z * scl, xv[k].w * scl};
      __half hi[4], lo[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        hi[q] = __float2half_rn(e[q]);
        lo[q] = __float2half_rn(e[q] - __half2float(hi[q]));
      }
      const int col = 64 * lane + 4 * k;
      if (col < a.cwb * F::BE) {  // inside the layout's part width
        *reinterpret_cast<uint2*>(hr + col) = make_uint2(
            uint32_t(__half_as_ushort(hi[0])) | (uint32_t(__half_as_ushort(hi[1])) << 16),
            uint32_t(__half_as_ushort(hi[2])) | (uint32_t(__half_as_ushort(hi[3])) << 16));
        *reinterpret_cast<uint2*>(lr + col) = make_uint2(
            uint32_t(__half_as_ushort(lo[0])) | (uint32_t(__half_as_ushort(lo[1])) << 16),
            uint32_t(__half_as_ushort(lo[2])) | (uint32_t(__half_as_ushort(lo[3])) << 16));
      }
      const float s4 = (e[0] + e[1]) + (e[2] + e[3]);
      if (k < 8) gs0 += s4;
      else gs1 += s4;
    }
    if (64 * lane < a.cwb * F::BE) {  // the groups of the layout's part width
      xs[(2 * lane) * MV + m] = gs0;
      xs[(2 * lane + 1) * MV + m] = gs1;
    }
  }
  __syncthreads();
  if (n_items == 0) return;

  const uint32_t* xh32 = reinterpret_cast<const uint32_t*>(xh + g * xpitch) + 2 * t;
  const uint32_t* xl32 = reinterpret_cast<const uint32_t*>(xl + g * xpitch) + 2 * t;
  const int xt = 4 * xpitch;  // uint32 words between the x of N-tiles (8 vectors)
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  bool dead = false;
  // consume cursor: stage slot and phase, segment, tile ordinal
  int cs = 0, csg = 0, ct = 0;
  uint32_t cph = 0;
  for (int i = 0; i < n_items; ++i) {
    if (!dead) {
      if (i + NS - 1 < n_items) issue_next();  // into the stage consumed last
      const bool ok = mbar_wait(smem_u32(full + cs), cph, cap);
      if (!__all_sync(0xffffffffu, ok)) {
        // flag it, wait (bounded) for the copies still in flight, stream no more
        if (lane == 0) flag_error(a.err, kErrWaitTimeout);
        int q = cs;
        uint32_t ph = cph;
        for (int n = i + 1; n < min(n_items, i + NS); ++n) {
          if (++q == NS) {
            q = 0;
            ph ^= 1u;
          }
          mbar_wait(smem_u32(full + q), ph, cap);
        }
        dead = true;
      }
    }
    if (!dead) {
      const int b0 = csg * S, nbk = min(S, blk_hi - blk_lo - b0);
      const uint8_t* stage = ring + size_t(cs) * a.SB + seg_off(csg);
      const int c0 = b0 * F::BE;  // first column of the segment in the part
      mma_segment<FMT, NT>(stage + size_t(g) * a.segB, stage + size_t(g + 8) * a.segB, nbk, t, xh32 + c0 / 2,
                           xl32 + c0 / 2, xt, xs + (c0 / 32) * MV, acc);
    }
    __syncwarp();
    if (++csg == nseg) {
      // the tile's partial sums: rows g, g + 8 and vectors 8 nt + 2t, 8 nt + 2t + 1 of this thread
      csg = 0;
      int j, nr;
      int64_t r0;
      mma_locate(a, ws + int64_t(ct) * stride, j, r0, nr);
      const int64_t rbase = a.job[j].rb + r0;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = g + 8 * (e >> 1), n = 8 * nt + 2 * t + (e & 1);
          if (!dead && row < nr && n < a.M)
            a.part[(int64_t(p) * a.M + n) * a.total_rows + rbase + row] = acc[nt][e] * xsc[n];
          acc[nt][e] = 0.f;
        }
      ++ct;
    }
    if (++cs == NS) {
      cs = 0;
      cph ^= 1u;
    }
  }
}

// bytes between the staged rows: room for a segment's 16-byte-aligned range,
// a multiple of 16 holding an odd number of 16-byte units, so the eight row
// groups of a warp read eight different bank quads
int mma_segB(int fmt) {
  const int sb = mma_seg_blocks(fmt) * block_bytes(fmt);
  // segments of a multiple of 16 bytes start 16-byte aligned; otherwise the
  // range may start up to 14 bytes before the segment
  int u = sb % 16 == 0 ? sb / 16 : (sb + 14 + 15) / 16;
  if (!(u & 1)) ++u;
  return 16 * u;
}

size_t mma_smem(int fmt, int cwb, int MV, int warps, int NS) {
  const int segB = mma_segB(fmt);
  // + 16: the unaligned readers may touch 4 bytes past a row
  return mma_layout(cwb * block_elems(fmt), MV, warps, NS).ring + size_t(warps) * NS * kMmaRows * segB + 16;
}

bool mma_format(int fmt) { return fmt == NT_Q8_0 || fmt == NT_Q4_K || fmt == NT_Q6_K; }

template <int FMT>
cudaError_t gemm_launch_t(const Ctx* c, const GemmArgs& a, dim3 grid, size_t smem, cudaStream_t st) {
  return launch_k(c, qgemm_kernel<FMT>, grid, dim3(kGemmThreads), smem, st, a);
}

template <int FMT>
int gemm_vstride() {
  const int ng = part_cols(FMT) / 32;
  return ((x_bytes<FMT>(part_cols(FMT)) + 12 * ng) + 15) / 16 * 16;
}

int fmt_vstride(int fmt) {
  switch (fmt) {
    case NT_Q8_0: return gemm_vstride<NT_Q8_0>();
    case NT_Q4_0: return gemm_vstride<NT_Q4_0>();
    case NT_Q4_K: return gemm_vstride<NT_Q4_K>();
    case NT_Q5_K: return gemm_vstride<NT_Q5_K>();
    case NT_Q6_K: return gemm_vstride<NT_Q6_K>();
    case NT_F16: return gemm_vstride<NT_F16>();
    default: return gemm_vstride<NT_F32>();
  }
}

size_t gemm_smem(int fmt, int M) {
  const int cwb = part_cols(fmt) / block_elems(fmt);
  const int segStride = ((cwb * block_bytes(fmt) + 15) / 16) * 16;
  const int stb = kGemmR * segStride + 16;  // the unaligned readers may touch 4 bytes past a row
  const size_t head = ((size_t(M) * fmt_vstride(fmt) + kGemmWarps * kGemmStages * 8 + 127) / 128) * 128;
  return head + size_t(kGemmWarps) * kGemmStages * ((stb + 15) / 16 * 16);
}

}  // namespace

int gemm_parts(int fmt, int64_t cols) { return int((cols + part_cols(fmt) - 1) / part_cols(fmt)); }

// Blocks per column part of the tensor-core form: 2048 columns, halved (down
// to one staged segment) while the 16-row tiles times the parts give fewer
// than 4096 warp tasks, so that small matrices still occupy every SM.  A
// function of the shape alone: the parts fix the order of the additions.
// bytes after the partial sums for the M RMSNorm scalars (and alignment)
constexpr size_t kInvBytes = 512;

static int mma_part_blocks(int fmt, int64_t tiles, int64_t nb, int MV) {
  int cwb = (MV > 8 ? 1024 : 2048) / block_elems(fmt);  // the x of 16 vectors fits for 1024 columns
  const int S = mma_seg_blocks(fmt);
  while (cwb > S && tiles * ((nb + cwb - 1) / cwb) < 4096) cwb /= 2;
  return cwb;
}

bool gemm_wide_ok(const Ctx* c, int fmt, int64_t cols) {
  return c->gemm_mma && mma_format(fmt) && cols % block_elems(fmt) == 0 &&
         (cols / block_elems(fmt) * block_bytes(fmt)) % 16 == 0;
}

size_t gemm_scratch_bytes(int fmt, int64_t total_rows, int64_t cols, int M) {
  int64_t parts = gemm_parts(fmt, cols);
  if (mma_format(fmt)) {
    // fewer tiles than ceil(rows / 16) summed per job never occur, and more tiles never ask for more parts
    const int64_t nb = cols / block_elems(fmt);
    const int cwb = mma_part_blocks(fmt, (total_rows + kMmaRows - 1) / kMmaRows, nb, M > 8 ? 16 : 8);
    parts = std::max<int64_t>(parts, (nb + cwb - 1) / cwb);
  }
  // + the RMSNorm scalars of the tensor-core form, after the partials
  return size_t(parts) * size_t(M) * size_t(total_rows) * sizeof(float) + kInvBytes;
}

nt_status configure_gemm(Ctx* c) {
  // dynamic shared memory: the opt-in limit minus each kernel's static part
  const int optin = int(c->smem_optin);
  int st = 0;
  cudaError_t e = cudaSuccess;
  auto allow = [&](auto kernel) {
    if (e != cudaSuccess) return;
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return;
    if (int(fa.sharedSizeBytes) > st) st = int(fa.sharedSizeBytes);
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - int(fa.sharedSizeBytes));
  };
  allow(qgemm_kernel<NT_Q8_0>);
  allow(qgemm_kernel<NT_Q4_0>);
  allow(qgemm_kernel<NT_Q4_K>);
  allow(qgemm_kernel<NT_Q5_K>);
  allow(qgemm_kernel<NT_Q6_K>);
  allow(qgemm_kernel<NT_F16>);
  allow(qgemm_kernel<NT_F32>);
  allow(qgemm_mma_kernel<NT_Q8_0, 1>);
  allow(qgemm_mma_kernel<NT_Q4_K, 1>);
  allow(qgemm_mma_kernel<NT_Q6_K, 1>);
  allow(qgemm_mma_kernel<NT_Q8_0, 2>);
  allow(qgemm_mma_kernel<NT_Q4_K, 2>);
  allow(qgemm_mma_kernel<NT_Q6_K, 2>);
  c->gemm_static_smem = st;
  return cuda_check(c, e, "gemm shared-memory attribute");
}

nt_status launch_gemm(Ctx* c, int fmt, const GemmJobEx* jobs, int njobs, bool swiglu, const float* X, int64_t ldx,
                      int M, const float* norm_g, float eps, int64_t cols, const RopeArgs* rope, float* part,
                      size_t part_bytes, cudaStream_t st) {
  if (c->dry) return NT_OK;
  if (M < 1 || M > kMaxGemmM) return set_err(c, NT_ERR_INVALID_ARG, "gemm: M must be 1..%d", kMaxGemmM);
  const int BB = block_bytes(fmt), BE = block_elems(fmt);
  const int64_t nb = cols / BE;
  const int64_t rowB = nb * BB;
  bool tma = (rowB % 16) == 0;
  for (int j = 0; j < njobs; ++j) tma = tma && aligned(jobs[j].W, 16);

  GemmArgs a{};
  EpiArgs e{};
  int64_t g = 0, rb = 0, pb = 0;
  for (int j = 0; j < njobs; ++j) {
    const GemmJobEx& J = jobs[j];
    a.job[j].W = static_cast<const uint8_t*>(J.W);
    a.job[j].rows = J.rows;
    a.job[j].g0 = g;
    a.job[j].rb = rb;
    e.job[j] = EpiJob{J.y, J.res, static_cast<__half*>(J.cache), J.ldy, J.rows, rb, pb, J.epi};
    g += (J.rows + kGemmR - 1) / kGemmR;
    rb += J.rows;
    pb += (J.rows + 1) / 2;
  }
  if (g == 0) return NT_OK;
  // the tensor-core form: its formats and bulk-copy alignment (rows of a
  // multiple of 16 bytes at 16-byte-aligned addresses)
  const bool mma = c->gemm_mma && mma_format(fmt) && tma;
  if (M > kMaxVerify && !mma)
    return set_err(c, NT_ERR_INVALID_ARG, "gemm: M > %d needs the tensor-core form (Q8_0, Q4_K, Q6_K; aligned rows)",
                   kMaxVerify);
  const int MV = M > 8 ? 16 : 8;  // vector slots: one or two MMA N-tiles
  int64_t tiles = 0;
  for (int j = 0; j < njobs; ++j) tiles += (jobs[j].rows + kMmaRows - 1) / kMmaRows;
  const int cwb = mma ? mma_part_blocks(fmt, tiles, nb, MV) : part_cols(fmt) / BE;
  const int nparts = int((nb + cwb - 1) / cwb);
  const size_t need = size_t(nparts) * M * size_t(rb) * sizeof(float) + (mma && norm_g ? kInvBytes : 0);
  if (need > part_bytes)
    return set_err(c, NT_ERR_OOM, "gemm: %zu scratch bytes needed for the partial sums, %zu available", need,
                   part_bytes);
  if (mma) {
    MmaArgs ma{};
    tiles = 0;
    for (int j = 0; j < njobs; ++j) {
      ma.job[j] = a.job[j];
      ma.job[j].g0 = tiles;
      tiles += (jobs[j].rows + kMmaRows - 1) / kMmaRows;
    }
    ma.njobs = njobs;
    ma.total_tiles = tiles;
    ma.total_rows = rb;
    ma.X = X;
    ma.ldx = ldx;
    ma.norm_g = norm_g;
    ma.eps = eps;
    ma.M = M;
    ma.cols = int(cols);
    ma.nb = int(nb);
    ma.cwb = cwb;
    ma.nparts = nparts;
    ma.rowB = rowB;
    ma.segB = mma_segB(fmt);
    ma.SB = kMmaRows * ma.segB;
    ma.part = part;
    ma.err = c->err_flag;
    ma.stall = take_stall(st);
    if (norm_g) {
      // the M RMSNorm scalars, once, right after the partial sums (256-byte aligned)
      if ((cols + 127) / 128 > kMaxChunksRms)
        return set_err(c, NT_ERR_INVALID_ARG, "gemm: cols=%lld too large for the fused RMSNorm", (long long)cols);
      const size_t off = (size_t(nparts) * M * size_t(rb) * sizeof(float) + 255) / 256 * 256;
      float* inv = reinterpret_cast<float*>(reinterpret_cast<char*>(part) + off);
      nt_status s0 = cuda_check(c, launch_k(c, rms_inv_kernel, dim3(M), dim3(256), 0, st, X, ldx, int(cols), eps, inv),
                                "gemm RMSNorm launch");
      if (s0) return s0;
      ma.inv = inv;
    }
    // warps per CTA and stages per warp: the most warps whose rings of at
    // least two stages fit beside x, then as many stages as fit
    const size_t room = c->smem_optin - size_t(c->gemm_static_smem);
    int warps = std::min(c->gemm_warps, kMmaWarps);
    while (warps > 8 && mma_smem(fmt, cwb, MV, warps, 2) > room) warps -= 4;
    ma.NS = 2;
    while (ma.NS < c->gemm_stages && mma_smem(fmt, cwb, MV, warps, ma.NS + 1) <= room) ++ma.NS;
    const size_t msmem = mma_smem(fmt, cwb, MV, warps, ma.NS);
    if (msmem > room) return set_err(c, NT_ERR_INVALID_ARG, "gemm: no shared-memory plan for the tensor-core form");
    // CTAs side by side over the parts, at most one per SM in all (one wave);
    // no more warps than tiles
    int gx = c->num_sms / nparts;
    if (gx < 1) gx = 1;
    const int64_t need_x = (tiles + warps - 1) / warps;
    if (gx > need_x) gx = int(need_x);
    const dim3 grid(gx, nparts);
    cudaError_t err;
    const dim3 blk(32 * warps);
    if (MV == 8) {
      switch (fmt) {
        case NT_Q8_0: err = launch_k(c, qgemm_mma_kernel<NT_Q8_0, 1>, grid, blk, msmem, st, ma); break;
        case NT_Q4_K: err = launch_k(c, qgemm_mma_kernel<NT_Q4_K, 1>, grid, blk, msmem, st, ma); break;
        default: err = launch_k(c, qgemm_mma_kernel<NT_Q6_K, 1>, grid, blk, msmem, st, ma); break;
      }
    } else {
      switch (fmt) {
        case NT_Q8_0: err = launch_k(c, qgemm_mma_kernel<NT_Q8_0, 2>, grid, blk, msmem, st, ma); break;
        case NT_Q4_K: err = launch_k(c, qgemm_mma_kernel<NT_Q4_K, 2>, grid, blk, msmem, st, ma); break;
        default: err = launch_k(c, qgemm_mma_kernel<NT_Q6_K, 2>, grid, blk, msmem, st, ma); break;
      }
    }
    nt_status s = cuda_check(c, err, "qgemm (tensor-core) launch");
    if (s) return s;
  }
  a.njobs = njobs;
  a.total_groups = g;
  a.total_rows = rb;
  a.X = X;
  a.ldx = ldx;
  a.norm_g = norm_g;
  a.eps = eps;
  a.M = M;
  a.cols = int(cols);
  a.nb = int(nb);
  a.cwb = cwb;
  a.nparts = nparts;
  a.rowB = rowB;
  a.segStride = ((cwb * BB + 15) / 16) * 16;
  a.stb = ((kGemmR * a.segStride + 16) + 15) / 16 * 16;
  a.vstride = fmt_vstride(fmt);
  a.tma = tma;
  a.part = part;
  a.err = c->err_flag;
  if (!mma) {
    const size_t smem = gemm_smem(fmt, M);
    if (smem + size_t(c->gemm_static_smem) > c->smem_optin)
      return set_err(c, NT_ERR_INVALID_ARG, "gemm: no shared-memory plan for M=%d", M);
    // one CTA per SM in all: the parts side by side
    int gx = c->num_sms / nparts;  // one wave
    if (gx < 1) gx = 1;
    const int64_t need_x = (g + kGemmWarps - 1) / kGemmWarps;
    if (gx > need_x) gx = int(need_x);
    const dim3 grid(gx, nparts);
    cudaError_t err;
    switch (fmt) {
      case NT_Q8_0: err = gemm_launch_t<NT_Q8_0>(c, a, grid, smem, st); break;
      case NT_Q4_0: err = gemm_launch_t<NT_Q4_0>(c, a, grid, smem, st); break;
      case NT_Q4_K: err = gemm_launch_t<NT_Q4_K>(c, a, grid, smem, st); break;
      case NT_Q5_K: err = gemm_launch_t<NT_Q5_K>(c, a, grid, smem, st); break;
      case NT_Q6_K: err = gemm_launch_t<NT_Q6_K>(c, a, grid, smem, st); break;
      case NT_F16: err = gemm_launch_t<NT_F16>(c, a, grid, smem, st); break;
      default: err = gemm_launch_t<NT_F32>(c, a, grid, smem, st); break;
    }
    nt_status s = cuda_check(c, err, "qgemm launch");
    if (s) return s;
  }

  e.njobs = njobs;
  e.total_pairs = pb;
  e.total_rows = rb;
  e.M = M;
  e.nparts = nparts;
  e.swiglu = swiglu;
  e.part = part;
  e.err = c->err_flag;
  if (rope) e.rope = *rope;
  const int64_t work = swiglu ? jobs[0].rows : pb;
  int blocks = int((work + 255) / 256);
  if (blocks > 4 * c->num_sms) blocks = 4 * c->num_sms;
  return cuda_check(c, launch_k(c, qgemm_epi_kernel, dim3(blocks, M), dim3(256), 0, st, e), "qgemm epilogue launch");
}

}  // namespace nt
