// qgemv.cu — dequantize-fused GEMV for the GGUF block formats named on
// "Ntransformer" (en.unwiki.net), About (Q8_0, Q4_0, Q4_K_M = Q4_K + Q6_K,
// Q5_K, Q6_K); the GEMV kernel of "Architecture et structure du code"
// (fr.news.hada.io).  y[r] = sum_c deq(W[r,c]) x[c].
//
// GB300 design (HBM-bound, M = 1, one CTA per SM):
//  * Weights stream through a private ring of shared-memory stages per warp,
//    filled by TMA bulk copies (cp.async.bulk + mbarrier complete_tx, L2
//    evict-first).  A warp works on groups of R consecutive rows, so each x
//    value it loads serves R rows; long rows are cut into column segments
//    whose unit count is a multiple of 32 so every lane has work.
//  * x (RMS-normalised in the prologue when asked) is held in shared memory
//    as 24-bit fixed point with one power-of-two scale per 32 columns,
//    split into three byte planes: |x - x24 2^-s| <= 2^-23 max|x over the
//    32 columns|, the order of fp32 rounding.  Quant x plane products are
//    exact integer MACs: dp4a multiplies four (u)int8 pairs and accumulates
//    in int32 — no per-weight int-to-float conversion.  The three plane
//    sums, sub-block scales, mins and the group scale are applied once per
//    16 or 32 elements in fp32.
//  * The plane layout is padded per format so the 16-byte reads of a
//    quarter-warp hit 8 distinct bank groups.
#include "nt_internal.cuh"
#include "ops.cuh"

namespace nt {
namespace {

constexpr int kMaxWarps = 32;

struct JobDev {
  const uint8_t* W;
  const uint8_t* W2;  // up-projection rows for the SwiGLU epilogue
  float* y;
  const float* res;
  __half* cache;      // f16 KV cache for the cache epilogues
  int64_t rows;
  int64_t g0;         // first group index of this job
  int epi;
};

struct GemvArgs {
  JobDev job[3];
  int njobs;
  const float* x;
  const float* norm_g;
  float eps;
  int cols;
  int nb;             // blocks per row
  int64_t rowB;       // bytes per row
  int seg;            // blocks per row in one stage
  int nseg;           // segments per row
  int segStride;      // bytes between the rows of one stage
  int stb;            // bytes per stage
  int nst;            // stages per warp
  int merged;         // one bulk copy per stage (whole consecutive rows)
  int tma;            // bulk-copy path (else plain loads)
  int swiglu;
  int64_t total_groups;
  unsigned* err;
  RopeArgs rope;
  int ks;             // warps sharing a row group, each over a column part
  int pblk[5];        // part p covers blocks [pblk[p], pblk[p+1])
};

// ---------------------------------------------------------------------------
// device helpers

// dp4a: d = c + sum_i a.byte_i * b.byte_i.  Suffixes: signedness of a, then b.
#define NT_DP4A(name, ta, tb)                                                        \
  __device__ __forceinline__ int name(uint32_t a, uint32_t b, int c) {               \
    int d;                                                                           \
    asm("dp4a." ta "." tb " %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));     \
    return d;                                                                        \
  }
NT_DP4A(dp4_su, "s32", "u32")
NT_DP4A(dp4_uu, "u32", "u32")
NT_DP4A(dp4_ss, "s32", "s32")
NT_DP4A(dp4_us, "u32", "s32")
#undef NT_DP4A

// N little-endian words from a 2-byte-aligned shared address (the aligned
// base is formed from p itself so the loads stay shared-memory loads)
template <int N>
__device__ __forceinline__ void lds_a2(const uint8_t* p, uint32_t* w) {
  const uint32_t mis = smem_u32(p) & 3u;
  const uint32_t* b = reinterpret_cast<const uint32_t*>(p - mis);
  const uint32_t sh = mis * 8;
  uint32_t t[N + 1];
#pragma unroll
  for (int i = 0; i <= N; ++i) t[i] = b[i];
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = __funnelshift_r(t[i], t[i + 1], sh);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float h2f(uint32_t bits16) { return __half2float(__ushort_as_half((unsigned short)bits16)); }

__device__ __forceinline__ void ld4(const uint8_t* p, uint32_t* w) {
  const uint4 t = *reinterpret_cast<const uint4*>(p);
  w[0] = t.x;
  w[1] = t.y;
  w[2] = t.z;
  w[3] = t.w;
}

// ---------------------------------------------------------------------------
// Shared x.  Each 32-column group g holds x as 24-bit fixed point,
// x24 = rint(x * 2^sh_g), split into three byte planes
//   x24 = p2 * 2^16 + p1 * 2^8 + p0   (p2 signed, p1 and p0 unsigned)
// stored as [p0: 32 B][p1: 32 B][p2: 32 B][16 B pad] at goff(g), plus
// scale[g] = 2^-sh_g and psum[3 * (col/16) + k] = sum of plane k over 16
// columns (for the constant offsets of Q4_0 and Q6_K).  |x - x24 2^-sh| is
// at most 2^-23 of the group's largest |x|.
struct XS {
  const uint8_t* x;
  const float* scale;
  const int* psum;
};

// sum of the three planes' integer dot products: 65536 a2 + 256 a1 + a0
__device__ __forceinline__ float planes(int a2, int a1, int a0) {
  return fmaf(float(a2), 65536.0f, fmaf(float(a1), 256.0f, float(a0)));
}

template <int FMT>
struct Q;

// Q8_0: d (f16) | qs[32] int8.  value d*q.  unit = one block (one group).
template <>
struct Q<NT_Q8_0> {
  static constexpr int BE = 32, BB = 34, ALIGN = 32, UPB = 1, PB = 0;
  struct X {
    uint32_t v[3][8];
    float s;
  };
  __device__ static void load_x(X& x, const uint8_t* g, const XS& xs, int col0, int) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      ld4(g + 32 * k, x.v[k]);
      ld4(g + 32 * k + 16, x.v[k] + 4);
    }
    x.s = xs.scale[col0 / 32];
  }
  __device__ static float dot(const uint8_t* blk, int, const X& x) {
    uint32_t w[8];
    lds_a2<8>(blk + 2, w);
    int a0 = 0, a1 = 0, a2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a0 = dp4_us(x.v[0][i], w[i], a0);
      a1 = dp4_us(x.v[1][i], w[i], a1);
      a2 = dp4_ss(x.v[2][i], w[i], a2);
    }
    const float d = __half2float(*reinterpret_cast<const __half*>(blk));
    return planes(a2, a1, a0) * (d * x.s);
  }
};

// Q4_0: d | qs[16]; element i<16 = low nibble of qs[i], i+16 = high nibble.
// value d*(q-8).  unit = one block (one group).
template <>
struct Q<NT_Q4_0> {
  static constexpr int BE = 32, BB = 18, ALIGN = 32, UPB = 1, PB = 0;
  struct X {
    uint32_t v[3][8];
    float s;
    int off[3];  // -8 * sum of each plane over the block
  };
  __device__ static void load_x(X& x, const uint8_t* g, const XS& xs, int col0, int) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      ld4(g + 32 * k, x.v[k]);
      ld4(g + 32 * k + 16, x.v[k] + 4);
    }
    x.s = xs.scale[col0 / 32];
    const int* ps = xs.psum + 3 * (col0 / 16);
#pragma unroll
    for (int k = 0; k < 3; ++k) x.off[k] = -8 * (ps[k] + ps[3 + k]);
  }
  __device__ static float dot(const uint8_t* blk, int, const X& x) {
    uint32_t w[4];
    lds_a2<4>(blk + 2, w);
    int a0 = x.off[0], a1 = x.off[1], a2 = x.off[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
      a0 = dp4_uu(x.v[0][4 + i], hi, dp4_uu(x.v[0][i], lo, a0));
      a1 = dp4_uu(x.v[1][4 + i], hi, dp4_uu(x.v[1][i], lo, a1));
      a2 = dp4_su(x.v[2][4 + i], hi, dp4_su(x.v[2][i], lo, a2));
    }
    const float d = __half2float(*reinterpret_cast<const __half*>(blk));
    return planes(a2, a1, a0) * (d * x.s);
  }
};

// K-quant scale/min pairs of the two sub-blocks 2c, 2c+1 from header words
// h1 = scales[0..3], h2 = scales[4..7], h3 = scales[8..11].
__device__ __forceinline__ void kq_scales(uint32_t h1, uint32_t h2, uint32_t h3, int c, float& sc0, float& sc1,
                                          float& m0, float& m1) {
  const int sh = (c & 1) * 16;
  const uint32_t a1 = h1 >> sh, a2 = h2 >> sh, a3 = h3 >> sh;
  uint32_t scp, mp;
  if (c < 2) {
    scp = a1 & 0x3F3Fu;
    mp = a2 & 0x3F3Fu;
  } else {
    scp = (a3 & 0x0F0Fu) | ((a1 >> 2) & 0x3030u);
    mp = ((a3 >> 4) & 0x0F0Fu) | ((a2 >> 2) & 0x3030u);
  }
  sc0 = float(scp & 0xFFu);
  sc1 = float((scp >> 8) & 0xFFu);
  m0 = float(mp & 0xFFu);
  m1 = float((mp >> 8) & 0xFFu);
}

// X of the 4/5-bit K formats: unit c = 64 columns = sub-blocks 2c, 2c+1 =
// groups A (low nibbles) and B (high nibbles).
struct XK {
  uint32_t a[3][8], b[3][8];
  float s0, s1;  // group scales
  float t0, t1;  // sum(x) over each sub-block
};
__device__ __forceinline__ void load_xk(XK& x, const uint8_t* g, const uint8_t* g2, const XS& xs, int col0, int c) {
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    ld4(g + 32 * k, x.a[k]);
    ld4(g + 32 * k + 16, x.a[k] + 4);
    ld4(g2 + 32 * k, x.b[k]);
    ld4(g2 + 32 * k + 16, x.b[k] + 4);
  }
  const int col = col0 + 64 * c;
  x.s0 = xs.scale[col / 32];
  x.s1 = xs.scale[col / 32 + 1];
  const int* ps = xs.psum + 3 * (col / 16);
  x.t0 = planes(ps[2] + ps[5], ps[1] + ps[4], ps[0] + ps[3]) * x.s0;
  x.t1 = planes(ps[8] + ps[11], ps[7] + ps[10], ps[6] + ps[9]) * x.s1;
}

__device__ __forceinline__ float kq_combine(uint4 hdr, int c, float qa, float qb, const XK& x) {
  float sc0, sc1, m0, m1;
  kq_scales(hdr.y, hdr.z, hdr.w, c, sc0, sc1, m0, m1);
  const float d = h2f(hdr.x & 0xFFFFu), dmin = h2f(hdr.x >> 16);
  // sum_j (d sc_j q - dmin m_j) x = d (sc0 s0 qa + sc1 s1 qb) - dmin (m0 t0 + m1 t1)
  return d * fmaf(sc0 * x.s0, qa, sc1 * x.s1 * qb) - dmin * fmaf(m0, x.t0, m1 * x.t1);
}

// nibble bytes lo/hi of one qs word against plane words of groups A and B
#define NT_KQ_MAC(i, lo, hi)                                          \
  do {                                                                \
    A0 = dp4_uu(x.a[0][i], lo, A0);                                   \
    A1 = dp4_uu(x.a[1][i], lo, A1);                                   \
    A2 = dp4_su(x.a[2][i], lo, A2);                                   \
    B0 = dp4_uu(x.b[0][i], hi, B0);                                   \
    B1 = dp4_uu(x.b[1][i], hi, B1);                                   \
    B2 = dp4_su(x.b[2][i], hi, B2);                                   \
  } while (0)

// Q4_K: d | dmin | scales[12] | qs[128].  value d*sc*q - dmin*m.
template <>
struct Q<NT_Q4_K> {
  static constexpr int BE = 256, BB = 144, ALIGN = 8, UPB = 4, PB = 1;
  using X = XK;
  __device__ static void load_x(X& x, const uint8_t* g, const XS& xs, int col0, int c) {
    load_xk(x, g, g + 112, xs, col0, c);
  }
  __device__ static float dot(const uint8_t* blk, int c, const X& x) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint4* qp = reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 q0 = qp[0], q1 = qp[1];
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    int A0 = 0, A1 = 0, A2 = 0, B0 = 0, B1 = 0, B2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
      NT_KQ_MAC(i, lo, hi);
    }
    return kq_combine(hdr, c, planes(A2, A1, A0), planes(B2, B1, B0), x);
  }
};

// Q5_K: d | dmin | scales[12] | qh[32] | qs[128]; the fifth bit of element l
// of sub-block j is bit j of qh[l].
template <>
struct Q<NT_Q5_K> {
  static constexpr int BE = 256, BB = 176, ALIGN = 8, UPB = 4, PB = 1;
  using X = XK;
  __device__ static void load_x(X& x, const uint8_t* g, const XS& xs, int col0, int c) {
    load_xk(x, g, g + 112, xs, col0, c);
  }
  __device__ static float dot(const uint8_t* blk, int c, const X& x) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint4* hp = reinterpret_cast<const uint4*>(blk + 16);
    const uint4 h0 = hp[0], h1 = hp[1];
    const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    const uint4* qp = reinterpret_cast<const uint4*>(blk + 48 + 32 * c);
    const uint4 q0 = qp[0], q1 = qp[1];
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const int b0 = 2 * c;
    int A0 = 0, A1 = 0, A2 = 0, B0 = 0, B1 = 0, B2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = (w[i] & 0x0F0F0F0Fu) | (((hw[i] >> b0) & 0x01010101u) << 4);
      const uint32_t hi = ((w[i] >> 4) & 0x0F0F0F0Fu) | (((hw[i] >> (b0 + 1)) & 0x01010101u) << 4);
      NT_KQ_MAC(i, lo, hi);
    }
    return kq_combine(hdr, c, planes(A2, A1, A0), planes(B2, B1, B0), x);
  }
};
#undef NT_KQ_MAC

// Q6_K: ql[128] | qh[64] | scales[16] int8 | d.  value d*sc*(q-32).
// unit u = (half h = u>>1, s = u&1): chunks g = 0..3 of 16 elements at block
// columns 128h + 32g + 16s + l', l' < 16 (the s-th half of group 4h+g);
// chunk g has scale scales[8h+2g+s].
template <>
struct Q<NT_Q6_K> {
  static constexpr int BE = 256, BB = 210, ALIGN = 8, UPB = 4, PB = 2;
  struct X {
    uint32_t v[4][3][4];  // chunk g, plane k, 4 words (16 columns)
    float s[4];           // group scales
    int off[4][3];        // -32 * plane sums over the chunk
  };
  __device__ static void load_x(X& x, const uint8_t* g0, const XS& xs, int col0, int u) {
    const int h = u >> 1, s = u & 1;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint8_t* p = g0 + 112 * (4 * h + g) + 16 * s;
#pragma unroll
      for (int k = 0; k < 3; ++k) ld4(p + 32 * k, x.v[g][k]);
      const int col = col0 + 128 * h + 32 * g + 16 * s;
      x.s[g] = xs.scale[col / 32];
      const int* ps = xs.psum + 3 * (col / 16);
#pragma unroll
      for (int k = 0; k < 3; ++k) x.off[g][k] = -32 * ps[k];
    }
  }
  __device__ static float dot(const uint8_t* blk, int u, const X& x) {
    const int h = u >> 1, s = u & 1;
    uint32_t A[4], B[4], H[4], S[2];
    lds_a2<4>(blk + 64 * h + 16 * s, A);        // low nibble: chunk 0, high: chunk 2
    lds_a2<4>(blk + 64 * h + 32 + 16 * s, B);   // low nibble: chunk 1, high: chunk 3
    lds_a2<4>(blk + 128 + 32 * h + 16 * s, H);  // bits 2g..2g+1: top bits of chunk g
    lds_a2<2>(blk + 192 + 8 * h, S);            // scales[8h .. 8h+7]
    int a[4][3];
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int k = 0; k < 3; ++k) a[g][k] = x.off[g][k];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t q[4] = {(A[i] & 0x0F0F0F0Fu) | ((H[i] << 4) & 0x30303030u),
                             (B[i] & 0x0F0F0F0Fu) | ((H[i] << 2) & 0x30303030u),
                             ((A[i] >> 4) & 0x0F0F0F0Fu) | (H[i] & 0x30303030u),
                             ((B[i] >> 4) & 0x0F0F0F0Fu) | ((H[i] >> 2) & 0x30303030u)};
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        a[g][0] = dp4_uu(x.v[g][0][i], q[g], a[g][0]);
        a[g][1] = dp4_uu(x.v[g][1][i], q[g], a[g][1]);
        a[g][2] = dp4_su(x.v[g][2][i], q[g], a[g][2]);
      }
    }
    // scale of chunk g: scales[8h + 2g + s] = byte (2g + s) of the 8-byte window
    const float sc0 = float(int8_t(S[0] >> (8 * s)));
    const float sc1 = float(int8_t(S[0] >> (8 * s + 16)));
    const float sc2 = float(int8_t(S[1] >> (8 * s)));
    const float sc3 = float(int8_t(S[1] >> (8 * s + 16)));
    float t = sc0 * x.s[0] * planes(a[0][2], a[0][1], a[0][0]);
    t = fmaf(sc1 * x.s[1], planes(a[1][2], a[1][1], a[1][0]), t);
    t = fmaf(sc2 * x.s[2], planes(a[2][2], a[2][1], a[2][0]), t);
    t = fmaf(sc3 * x.s[3], planes(a[3][2], a[3][1], a[3][0]), t);
    const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
    return d * t;
  }
};

// byte offset of 32-column group g: 112 bytes per group, plus PB*16 bytes
// per 8 groups (one K block), chosen per format so that the 16-byte plane
// reads of a quarter-warp fall into 8 distinct bank groups
template <int FMT>
__host__ __device__ constexpr int goff(int g) {
  return 112 * g + 16 * Q<FMT>::PB * (g / 8);
}

template <int FMT>
__host__ __device__ constexpr int x_bytes(int cols) {
  return ((goff<FMT>(cols / 32 + 1) + 15) / 16) * 16;
}

// ---------------------------------------------------------------------------

__device__ __forceinline__ void locate(const GemvArgs& a, int64_t g, int rpg, int& j, int64_t& r0, int& nr) {
  j = 0;
  while (j + 1 < a.njobs && g >= a.job[j + 1].g0) ++j;
  r0 = (g - a.job[j].g0) * rpg;
  const int64_t left = a.job[j].rows - r0;
  nr = left < rpg ? int(left) : rpg;
}

template <int FMT, int R, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) qgemv_kernel(const GemvArgs a) {
  using F = Q<FMT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int nwarps = blockDim.x >> 5, kStages = a.nst;
  const int xB = x_bytes<FMT>(a.cols);
  const int ng = a.cols / 32;
  uint8_t* xsm = smem;
  float* gscale = reinterpret_cast<float*>(smem + xB);
  int* psum = reinterpret_cast<int*>(smem + xB + 4 * ng);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ((xB + 28 * ng + 7) / 8) * 8);
  uint8_t* stages = smem + ((xB + 28 * ng + 8 + nwarps * kStages * 8 + 127) / 128) * 128;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // warps come in slots of a.ks; the warps of a slot share row groups, warp
  // `part` of a slot covers the blocks [pblk[part], pblk[part+1]) of each row
  const int KS = a.ks, slots = nwarps / KS, slot = warp / KS, part = warp % KS;
  const int pb0 = a.pblk[part], pb1 = a.pblk[part + 1];
  const int nseg = (pb1 - pb0 + a.seg - 1) / a.seg;
  const int64_t total_warps = int64_t(gridDim.x) * slots;  // group stride
  const int64_t wg = int64_t(blockIdx.x) * slots + slot;   // first group
  const int my_groups = wg < a.total_groups ? int((a.total_groups - wg + total_warps - 1) / total_warps) : 0;
  const int n_items = my_groups * nseg;
  __shared__ float xchg[2 * 4 * kMaxWarps];  // [2][slots][KS][R] partial sums of split groups
  uint8_t* st0 = stages + size_t(warp) * kStages * a.stb;
  const uint32_t bar0 = smem_u32(bars + warp * kStages);
  const int rpg = a.swiglu ? R / 2 : R;

  if (a.tma) {
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
      fence_barrier_init();
    }
    __syncwarp();
  }
  const uint64_t pol = policy_evict_first();

  // ---- issue cursor: group ordinal, segment, stage slot; rows of the group cached
  int it_t = 0, it_s = 0, it_slot = 0;
  int g_j = 0, g_nr = 0;
  int64_t g_r0 = 0;
  const uint8_t* my_row = nullptr;  // lane i < R: row i of the current issue group (null past the end)

  auto load_group = [&](int t) {
    locate(a, wg + int64_t(t) * total_warps, rpg, g_j, g_r0, g_nr);
    my_row = nullptr;
    if (lane < R) {
      const JobDev& J = a.job[g_j];
      if (a.swiglu) {
        const int h = R / 2, k = lane < h ? lane : lane - h;
        if (k < g_nr) my_row = (lane < h ? J.W : J.W2) + (g_r0 + k) * a.rowB;
      } else if (lane < g_nr) {
        my_row = J.W + (g_r0 + lane) * a.rowB;
      }
    }
  };

  auto fill = [&](uint8_t* st, uint32_t bar, int s) {
    const int blk0 = pb0 + s * a.seg;
    const int nblk = min(a.seg, pb1 - blk0);
    const uint32_t bytes_row = uint32_t(nblk) * F::BB;
    if (a.tma) {
      if (a.merged) {
        if (lane == 0) {
          const uint32_t tot = uint32_t(g_nr) * uint32_t(a.rowB);
          mbar_arrive_expect_tx(bar, tot);
          bulk_g2s(smem_u32(st), a.job[g_j].W + g_r0 * a.rowB, tot, bar, pol);
        }
      } else {
        const int nvalid = a.swiglu ? 2 * g_nr : g_nr;
        if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(nvalid) * bytes_row);
        __syncwarp();
        if (my_row) bulk_g2s(smem_u32(st + lane * a.segStride), my_row + size_t(blk0) * F::BB, bytes_row, bar, pol);
      }
    } else {
      // plain-load path for weights that break the bulk-copy alignment rules
      for (int i = 0; i < R; ++i) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(
            __shfl_sync(0xffffffffu, static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(my_row)), i));
        if (!src) continue;
        src += size_t(blk0) * F::BB;
        for (int b = lane; b < int(bytes_row); b += 32) st[i * a.segStride + b] = src[b];
      }
      __syncwarp();
    }
  };

  auto issue_next = [&]() {
    if (it_s == 0) load_group(it_t);
    fill(st0 + size_t(it_slot) * a.stb, bar0 + 8 * uint32_t(it_slot), it_s);
    if (++it_s == nseg) {
      it_s = 0;
      ++it_t;
    }
    if (++it_slot == kStages) it_slot = 0;
  };

  // weights do not depend on x: start streaming them before waiting for the
  // kernel that produces x
  if (a.tma) {
    const int pre = n_items < kStages - 1 ? n_items : kStages - 1;
    for (int k = 0; k < pre; ++k) issue_next();
  }
  pdl_trigger();
  pdl_wait();

  // ---- prologue: x (optionally RMS-normalised) -> 24-bit fixed point per 32-column group.
  // 8 lanes per group of 32 columns, 4 columns per lane; a warp covers 4 groups
  // per pass.  All of a lane's x loads are issued first (one memory round
  // trip), the RMSNorm sum of squares comes from the same registers.
  {
    __shared__ float red[kMaxWarps];
    constexpr int kPF = 16;  // passes held in registers
    const int sub = lane & 7;
    const int pass_stride = nwarps * 4;
    const int npass = (ng - warp * 4 + pass_stride - 1) / pass_stride;  // passes of this warp (may be <= 0)
    const bool whole = (ng + pass_stride - 1) / pass_stride <= kPF;      // CTA-uniform: all of x in registers
    float4 v[kPF];
    auto load_passes = [&](int p0) {
#pragma unroll
      for (int k = 0; k < kPF; ++k) {
        const int grp = warp * 4 + (p0 + k) * pass_stride + (lane >> 3);
        v[k] = (p0 + k < npass && grp < ng) ? *reinterpret_cast<const float4*>(a.x + 32 * grp + 4 * sub)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    if (whole) load_passes(0);
    float inv = 1.f;
    if (a.norm_g) {
      float ss = 0.f;
      if (whole) {
#pragma unroll
        for (int k = 0; k < kPF; ++k)
          ss = fmaf(v[k].x, v[k].x, fmaf(v[k].y, v[k].y, fmaf(v[k].z, v[k].z, fmaf(v[k].w, v[k].w, ss))));
      } else {
        for (int i = tid * 4; i < a.cols; i += blockDim.x * 4) {
          const float4 t = *reinterpret_cast<const float4*>(a.x + i);
          ss = fmaf(t.x, t.x, fmaf(t.y, t.y, fmaf(t.z, t.z, fmaf(t.w, t.w, ss))));
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      float tot = 0.f;
      for (int w = 0; w < nwarps; ++w) tot += red[w];
      inv = rsqrtf(tot / float(a.cols) + a.eps);
    }
    for (int p0 = 0; p0 < npass; p0 += kPF) {
      if (!whole) load_passes(p0);
#pragma unroll
      for (int k = 0; k < kPF; ++k) {
        if (p0 + k >= npass) break;  // warp-uniform
        const int grp = warp * 4 + (p0 + k) * pass_stride + (lane >> 3);
        const bool live = grp < ng;
        const int col = 32 * grp + 4 * sub;
        float4 x4 = v[k];
        if (a.norm_g && live) {
          const float4 g = *reinterpret_cast<const float4*>(a.norm_g + col);
          x4.x = x4.x * inv * g.x;
          x4.y = x4.y * inv * g.y;
          x4.z = x4.z * inv * g.z;
          x4.w = x4.w * inv * g.w;
        }
        float m = fmaxf(fmaxf(fabsf(x4.x), fabsf(x4.y)), fmaxf(fabsf(x4.z), fabsf(x4.w)));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        // m = f * 2^e with f in [0.5, 1): e from the exponent field; scale = 2^(23 - e)
        const int e = int((__float_as_uint(m) >> 23) & 0xFFu) - 126;
        const int sh = min(126, max(-126, 23 - e));
        const float scl = __uint_as_float(uint32_t(127 + sh) << 23);
        constexpr int kLim = (1 << 23) - 1;
        const int q0 = max(-kLim, min(kLim, __float2int_rn(x4.x * scl)));
        const int q1 = max(-kLim, min(kLim, __float2int_rn(x4.y * scl)));
        const int q2 = max(-kLim, min(kLim, __float2int_rn(x4.z * scl)));
        const int q3 = max(-kLim, min(kLim, __float2int_rn(x4.w * scl)));
        // byte planes: plane k holds byte k of the four 24-bit values
        const uint32_t lo01 = __byte_perm(q0, q1, 0x5410), lo23 = __byte_perm(q2, q3, 0x5410);  // bytes 0,1 of each
        const uint32_t hi01 = __byte_perm(q0, q1, 0x7632), hi23 = __byte_perm(q2, q3, 0x7632);  // bytes 2,3 of each
        const uint32_t pw0 = __byte_perm(lo01, lo23, 0x6420);
        const uint32_t pw1 = __byte_perm(lo01, lo23, 0x7531);
        const uint32_t pw2 = __byte_perm(hi01, hi23, 0x6420);
        int ps0 = __dp4a(pw0, 0x01010101u, 0u), ps1 = __dp4a(pw1, 0x01010101u, 0u);
        int ps2 = __dp4a(int(pw2), 0x01010101, 0);  // plane 2 is signed
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
        ps2 += __shfl_xor_sync(0xffffffffu, ps2, 1);
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
        ps2 += __shfl_xor_sync(0xffffffffu, ps2, 2);
        if (live) {
          uint8_t* gp = xsm + goff<FMT>(grp) + 4 * sub;
          *reinterpret_cast<uint32_t*>(gp) = pw0;
          *reinterpret_cast<uint32_t*>(gp + 32) = pw1;
          *reinterpret_cast<uint32_t*>(gp + 64) = pw2;
          if ((sub & 3) == 0) {
            int* dst = psum + 3 * (2 * grp + (sub >> 2));
            dst[0] = ps0;
            dst[1] = ps1;
            dst[2] = ps2;
          }
          if (sub == 0) gscale[grp] = __uint_as_float(uint32_t(127 - sh) << 23);
        }
      }
    }
    __syncthreads();
  }
  if (my_groups == 0) return;
  const XS xs{xsm, gscale, psum};

  float acc[R];
#pragma unroll
  for (int i = 0; i < R; ++i) acc[i] = 0.f;

  // ---- consume cursor
  int cs = 0, ct = 0, cseg = 0;
  uint32_t cph = 0;
  bool dead = false;  // a copy never landed: stop streaming, keep the group barriers
  for (int k = 0; k < n_items; ++k) {
    uint8_t* st = st0 + size_t(cs) * a.stb;
    if (dead) {
    } else if (a.tma) {
      if (k + kStages - 1 < n_items) issue_next();
      const bool ok = mbar_wait(bar0 + 8 * uint32_t(cs), cph);
      if (!__all_sync(0xffffffffu, ok)) {
        // flag it, wait (bounded) for the copies still in flight, stream no more
        if (lane == 0) flag_error(a.err, kErrWaitTimeout);
        int q = cs;
        uint32_t ph = cph;
        for (int n = k + 1; n < min(n_items, k + kStages - 1); ++n) {
          if (++q == kStages) {
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
      const int blk0 = pb0 + cseg * a.seg;
      const int nblk = min(a.seg, pb1 - blk0);
      const int units = nblk * F::UPB;
      for (int u = lane; u < units; u += 32) {
        const int b = u / F::UPB, uu = u % F::UPB;
        typename F::X x;
        const int col0 = (blk0 + b) * F::BE;
        F::load_x(x, xsm + goff<FMT>(col0 / 32 + (F::UPB == 4 && FMT != NT_Q6_K ? 2 * uu : 0)), xs, col0, uu);
        const uint8_t* bp = st + b * F::BB;
#pragma unroll
        for (int i = 0; i < R; ++i) acc[i] += F::dot(bp + i * a.segStride, uu, x);
      }
    }
    __syncwarp();
    if (cseg == nseg - 1) {
      // group done: reduce across lanes, lane i holds row i
      float mine = 0.f;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const float v = warp_sum(acc[i]);
        if (lane == i) mine = v;
        acc[i] = 0.f;
      }
      if (KS > 1) {
        // the parts of a split group meet in shared memory (double-buffered by group parity)
        float* xb = xchg + ((ct & 1) * slots + slot) * KS * R;
        if (part > 0 && lane < R) xb[part * R + lane] = mine;
        named_sync(1 + slot, 32 * KS);
        if (part == 0 && lane < R)
          for (int p = 1; p < KS; ++p) mine += xb[p * R + lane];
      }
      if (part == 0) {
        const float other = __shfl_down_sync(0xffffffffu, mine, R / 2);  // lane i: row i + R/2
        int j, nr;
        int64_t r0;
        locate(a, wg + int64_t(ct) * total_warps, rpg, j, r0, nr);
        const JobDev& J = a.job[j];
        if (a.swiglu) {
          if (lane < nr) J.y[r0 + lane] = silu(mine) * other;
        } else if (J.epi == kEpiPlain) {
          if (lane < nr) J.y[r0 + lane] = J.res ? mine + J.res[r0 + lane] : mine;
        } else {
          // rows come in adjacent (even, odd) pairs: lane i^1 holds the partner
          const float partner = __shfl_xor_sync(0xffffffffu, mine, 1);
          if (lane < nr) {
            const int64_t r = r0 + lane;
            const int hd = a.rope.head_dim;
            const int64_t pos = *a.rope.pos_dev;
            const int head = int(r / hd), d = int(r % hd);
            float out = mine;
            if (J.epi != kEpiCache) {
              float cs_, sn;
              rope_cs(pos, a.rope.inv_freq[d >> 1], cs_, sn);
              out = (d & 1) ? fmaf(partner, sn, mine * cs_) : fmaf(mine, cs_, -partner * sn);
            }
            if (J.epi == kEpiRope)
              J.y[r] = out;
            else
              J.cache[(int64_t(head) * a.rope.kv_stride + pos) * hd + d] = __float2half_rn(out);
          }
        }
      }
    }
    if (++cs == kStages) {
      cs = 0;
      cph ^= 1u;
    }
    if (++cseg == nseg) {
      cseg = 0;
      ++ct;
    }
  }
}

// ---------------------------------------------------------------------------
// host side

template <int FMT, int R>
cudaError_t launch_t(const Ctx* c, const GemvArgs& a, int warps, int grid, size_t smem, cudaStream_t st) {
  if (warps > 8) return launch_k(c, qgemv_kernel<FMT, R, 512>, dim3(grid), dim3(warps * 32), smem, st, a);
  return launch_k(c, qgemv_kernel<FMT, R, 256>, dim3(grid), dim3(warps * 32), smem, st, a);
}

// dynamic shared memory a kernel may use: the opt-in limit minus its static
// part; the largest static part is remembered for the launch plans
template <typename K>
cudaError_t allow_smem(K kernel, int optin, int* max_static) {
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  if (int(fa.sharedSizeBytes) > *max_static) *max_static = int(fa.sharedSizeBytes);
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - int(fa.sharedSizeBytes));
}

template <int FMT>
cudaError_t configure_fmt(int smem, int* st) {
  cudaError_t e = allow_smem(qgemv_kernel<FMT, 4, 256>, smem, st);
  if (e == cudaSuccess) e = allow_smem(qgemv_kernel<FMT, 2, 256>, smem, st);
  if (e == cudaSuccess) e = allow_smem(qgemv_kernel<FMT, 4, 512>, smem, st);
  if (e == cudaSuccess) e = allow_smem(qgemv_kernel<FMT, 2, 512>, smem, st);
  return e;
}

template <int FMT>
cudaError_t dispatch_r(const Ctx* c, int R, const GemvArgs& a, int warps, int grid, size_t smem, cudaStream_t st) {
  return R == 4 ? launch_t<FMT, 4>(c, a, warps, grid, smem, st) : launch_t<FMT, 2>(c, a, warps, grid, smem, st);
}

struct FmtInfo {
  int align;   // blocks per segment unit: 16-byte aligned and a multiple of 32 lane units
  int xbytes;  // shared bytes of x
};

FmtInfo fmt_info(int fmt, int cols) {
  switch (fmt) {
    case NT_Q8_0: return {Q<NT_Q8_0>::ALIGN, x_bytes<NT_Q8_0>(cols)};
    case NT_Q4_0: return {Q<NT_Q4_0>::ALIGN, x_bytes<NT_Q4_0>(cols)};
    case NT_Q4_K: return {Q<NT_Q4_K>::ALIGN, x_bytes<NT_Q4_K>(cols)};
    case NT_Q5_K: return {Q<NT_Q5_K>::ALIGN, x_bytes<NT_Q5_K>(cols)};
    default: return {Q<NT_Q6_K>::ALIGN, x_bytes<NT_Q6_K>(cols)};
  }
}

}  // namespace

// Allow every GEMV instantiation the opt-in shared memory once, at context
// creation (never during a stream capture).
nt_status configure_gemv(Ctx* c) {
  const int smem = int(c->smem_optin);
  int st = 0;
  cudaError_t e = configure_fmt<NT_Q8_0>(smem, &st);
  if (e == cudaSuccess) e = configure_fmt<NT_Q4_0>(smem, &st);
  if (e == cudaSuccess) e = configure_fmt<NT_Q4_K>(smem, &st);
  if (e == cudaSuccess) e = configure_fmt<NT_Q5_K>(smem, &st);
  if (e == cudaSuccess) e = configure_fmt<NT_Q6_K>(smem, &st);
  c->gemv_static_smem = st;
  return cuda_check(c, e, "gemv shared-memory attribute");
}

nt_status launch_gemv(Ctx* c, int fmt, const nt_gemv_job* jobs, int njobs, const void* W2, const float* x,
                      const float* norm_g, float eps, int64_t cols, bool swiglu, cudaStream_t st) {
  GemvJobEx ex[3];
  for (int j = 0; j < njobs && j < 3; ++j) ex[j] = GemvJobEx{jobs[j], kEpiPlain, nullptr};
  return launch_gemv_ex(c, fmt, ex, njobs, W2, x, norm_g, eps, cols, swiglu, nullptr, st);
}

nt_status launch_gemv_ex(Ctx* c, int fmt, const GemvJobEx* jobsx, int njobs, const void* W2, const float* x,
                         const float* norm_g, float eps, int64_t cols, bool swiglu, const RopeArgs* rope,
                         cudaStream_t st) {
  const int BB = block_bytes(fmt);
  const int64_t nb = cols / block_elems(fmt);
  const int64_t rowB = nb * BB;
  bool tma = (rowB % 16) == 0;
  for (int j = 0; j < njobs; ++j) tma = tma && aligned(jobsx[j].j.W_dev, 16);
  if (swiglu) tma = tma && aligned(W2, 16);

  const FmtInfo fi = fmt_info(fmt, int(cols));
  const int ng = int(cols / 32);
  const int pad = 16;  // the unaligned readers may touch 4 bytes past a stage
  GemvArgs a{};
  int R = 0, kStages = 0, kWarps = 0, head = 0, stb = 0;
  const int al = fi.align;
  // the configured warps and stages; fewer when x leaves too little shared memory
  for (int nw = c->gemv_warps; nw >= 4 && R == 0; nw /= 2) {
    for (int ns = c->gemv_stages; ns >= 2 && R == 0; --ns) {
      head = ((fi.xbytes + 28 * ng + 8 + nw * ns * 8 + 127) / 128) * 128;
      const long avail = long(c->smem_optin) - head - pad - c->gemv_static_smem;
      stb = int(avail / (nw * ns)) / 16 * 16;
      if (stb > c->gemv_stage_max) stb = c->gemv_stage_max;
      if (stb < 256) continue;
      for (int r : {4, 2}) {
        // whole rows when R of them fit a stage
        if (int64_t(r) * (tma ? rowB : ((rowB + 15) / 16) * 16) <= stb) {
          R = r;
          a.seg = int(nb);
          a.nseg = 1;
          a.merged = tma && !swiglu;
          a.segStride = int(a.merged ? rowB : ((rowB + 15) / 16) * 16);
          break;
        }
        int seg = int(stb / (int64_t(r) * BB)) / al * al;
        while (seg >= al && int64_t(r) * (((seg * BB + 15) / 16) * 16) > stb) seg -= al;
        if (seg >= al) {
          R = r;
          a.seg = seg;
          a.nseg = int((nb + seg - 1) / seg);
          a.merged = 0;
          a.segStride = ((seg * BB + 15) / 16) * 16;
          break;
        }
      }
      if (R) {
        kStages = ns;
        kWarps = nw;
      }
    }
  }
  if (R == 0)
    return set_err(c, NT_ERR_INVALID_ARG, "gemv: cols=%lld too large for the shared-memory plan", (long long)cols);

  const int rpg = swiglu ? R / 2 : R;
  int64_t g = 0;
  for (int j = 0; j < njobs; ++j) {
    const nt_gemv_job& jb = jobsx[j].j;
    a.job[j].W = static_cast<const uint8_t*>(jb.W_dev);
    a.job[j].W2 = static_cast<const uint8_t*>(W2);
    a.job[j].y = jb.y_dev;
    a.job[j].res = jb.residual_dev;
    a.job[j].rows = jb.rows;
    a.job[j].g0 = g;
    a.job[j].epi = jobsx[j].epi;
    a.job[j].cache = static_cast<__half*>(jobsx[j].cache);
    g += (jb.rows + rpg - 1) / rpg;
  }
  if (rope) a.rope = *rope;
  if (g == 0) return NT_OK;

  // split row groups over KS warps (column parts) when there are too few
  // groups to give every warp of every SM the same amount of work
  int ks = 1;
  {
    const int64_t T = int64_t(c->num_sms) * kWarps;
    double best = 0.0;
    const int units = int(nb / al);  // ALIGN-block units per row
    for (int cand : {1, 2, 4}) {
      if (kWarps % cand || (cand > 1 && units < cand)) continue;
      const int64_t u = g * cand;
      const int64_t per = (u + T - 1) / T;
      const double eff = double(u) / double(T * per);
      if (eff > best + 0.02) {
        best = eff;
        ks = cand;
      }
    }
  }
  a.ks = ks;
  if (ks == 1) {
    a.pblk[0] = 0;
    a.pblk[1] = int(nb);
  } else {
    const int units = int(nb / al);
    for (int p = 0; p <= ks; ++p) a.pblk[p] = (p * units / ks) * al;
    a.pblk[ks] = int(nb);
    const int plen = a.pblk[1] - a.pblk[0];
    if (a.seg > plen) a.seg = plen;  // a part fits one stage
    a.merged = 0;
    a.segStride = ((a.seg * BB + 15) / 16) * 16;
  }
  a.nseg = 0;  // per part, computed in the kernel
  a.njobs = njobs;
  a.x = x;
  a.norm_g = norm_g;
  a.eps = eps;
  a.cols = int(cols);
  a.nb = int(nb);
  a.rowB = rowB;
  a.stb = stb;
  a.nst = kStages;
  a.tma = tma;
  a.swiglu = swiglu;
  a.total_groups = g;
  a.err = c->err_flag;

  // every SM gets a CTA (fewer only when there are fewer groups than warps);
  // groups go round-robin, so warps differ by at most one group
  const int slots = kWarps / ks;
  int64_t grid64 = (g + slots - 1) / slots;
  if (grid64 > c->num_sms) grid64 = c->num_sms;
  const int grid = int(grid64);
  const size_t smem = size_t(head) + size_t(kWarps) * kStages * stb + pad;

  cudaError_t e;
  switch (fmt) {
    case NT_Q8_0: e = dispatch_r<NT_Q8_0>(c, R, a, kWarps, grid, smem, st); break;
    case NT_Q4_0: e = dispatch_r<NT_Q4_0>(c, R, a, kWarps, grid, smem, st); break;
    case NT_Q4_K: e = dispatch_r<NT_Q4_K>(c, R, a, kWarps, grid, smem, st); break;
    case NT_Q5_K: e = dispatch_r<NT_Q5_K>(c, R, a, kWarps, grid, smem, st); break;
    default: e = dispatch_r<NT_Q6_K>(c, R, a, kWarps, grid, smem, st); break;
  }
  return cuda_check(c, e, "qgemv launch");
}

}  // namespace nt
