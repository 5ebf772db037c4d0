// qformats.cuh — the GGUF block formats as seen by the quant-GEMV kernels:
// per-format dot products of one block unit against x held in shared memory
// as fixed point in byte planes (24-bit in three planes by default, 16-bit
// in two with NT_X_PLANES=2), and the x prologue that builds those planes.  Formats and element values ("Ntransformer" (en.unwiki.net),
// About; GGUF layouts): Q8_0 d*q; Q4_0 d*(q-8); Q4_K/Q5_K d*sc*q - dmin*m;
// Q6_K d*sc*(q-32).
#pragma once
#include "nt_internal.cuh"

namespace nt {
namespace qf {

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

__device__ __forceinline__ float h2f(uint32_t bits16) { return __half2float(__ushort_as_half((unsigned short)bits16)); }

__device__ __forceinline__ void ld4(const uint8_t* p, uint32_t* w) {
  const uint4 t = *reinterpret_cast<const uint4*>(p);
  w[0] = t.x;
  w[1] = t.y;
  w[2] = t.z;
  w[3] = t.w;
}

// ---------------------------------------------------------------------------
// Shared x.  Each 32-column group g holds x as B-bit fixed point (B = 8 *
// kPlanes: 24 by default, 16 with NT_X_PLANES=2), xq = rint(x * 2^sh_g),
// split into kPlanes byte planes
//   xq = sum_k p_k 256^k   (the top plane signed, the others unsigned)
// stored as [p0: 32 B][p1: 32 B]([p2: 32 B])[16 B pad] at goff(g), plus
// scale[g] = 2^-sh_g and psum[col/16] = sum of xq over 16 columns (for the
// constant offsets of Q4_0 and Q6_K and the mins of the K formats; at most
// 2^(B+4) in magnitude).  sh_g puts the group's largest |x| just below
// 2^(B-1), so |x - xq 2^-sh| is at most 2^-B of it: 2^-24 with three planes,
// the order of fp32 rounding.  Two planes (2^-16) save a third of the dp4a
// work — 12-15% faster on the ALU-bound K formats — but a dot product that
// cancels (|y| far below sum |w x|) can then miss a 1e-3 relative bound, so
// the library is built with three.
#ifndef NT_X_PLANES
#define NT_X_PLANES 3
#endif
constexpr int kPlanes = NT_X_PLANES;
static_assert(kPlanes == 2 || kPlanes == 3, "x is held in two or three byte planes");
constexpr int kXBits = 8 * kPlanes;
constexpr int kGroupPitch = 32 * kPlanes + 16;  // shared bytes per 32-column group (planes + pad)

struct XS {
  const uint8_t* x;
  const float* scale;
  const int* psum;
};

// sum of the planes' integer dot products: sum_k 256^k a[k].  256 a1 + a0 is
// formed in int32 (every format keeps |a1|, |a0| below 2^22, so it cannot
// overflow), then one fp32 rounding per step.
__device__ __forceinline__ float planes(const int (&a)[kPlanes]) {
  if constexpr (kPlanes == 3) return fmaf(float(a[2]), 65536.0f, float(a[1] * 256 + a[0]));
  else return float(a[1] * 256 + a[0]);
}

// -c * S split over the planes (S = sum_k 256^k s_k, the top digit signed),
// so the constant offset folds exactly into the integer sums
__device__ __forceinline__ void plane_offsets(int S, int c, int (&off)[kPlanes]) {
  off[0] = -c * (S & 255);
  if constexpr (kPlanes == 3) {
    off[1] = -c * ((S >> 8) & 255);
    off[2] = -c * (S >> 16);
  } else {
    off[1] = -c * (S >> 8);
  }
}

// a + (x plane word xw) . (weight word w): plane `top` is the signed plane;
// WS: the weight bytes are signed
template <bool WS>
__device__ __forceinline__ int dp(bool top, uint32_t xw, uint32_t w, int a) {
  if (WS) return top ? dp4_ss(xw, w, a) : dp4_us(xw, w, a);
  return top ? dp4_su(xw, w, a) : dp4_uu(xw, w, a);
}

template <int FMT>
struct Q;

// Q8_0: d (f16) | qs[32] int8.  value d*q.  unit = one block (one group).
template <>
struct Q<NT_Q8_0> {
  static constexpr int BE = 32, BB = 34, ALIGN = 32, UPB = 1, PB = 0;
  static constexpr bool FLOATX = false;  // x as fixed-point byte planes
  struct X {
    uint32_t v[kPlanes][8];
    float s;
  };
  __device__ static void load_x(X& x, const uint8_t* g, const XS& xs, int col0, int) {
#pragma unroll
    for (int k = 0; k < kPlanes; ++k) {
      ld4(g + 32 * k, x.v[k]);
      ld4(g + 32 * k + 16, x.v[k] + 4);
    }
    x.s = xs.scale[col0 / 32];
  }
  // one unit of one row, unpacked: quants and scale
  struct W {
    uint32_t q[8];
    float d;
  };
  __device__ static void unpack(const uint8_t* blk, int, W& w) {
    lds_a2<8>(blk + 2, w.q);
    w.d = __half2float(*reinterpret_cast<const __half*>(blk));
  }
  __device__ static float dotw(const W& w, int, const X& x) {
    int a[kPlanes] = {};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int k = 0; k < kPlanes; ++k) a[k] = dp<true>(k == kPlanes - 1, x.v[k][i], w.q[i], a[k]);
    return planes(a) * (w.d * x.s);
  }
  __device__ static float dot(const uint8_t* blk, int u, const X& x) {
    W w;
    unpack(blk, u, w);
    return dotw(w, u, x);
  }
};

// Q4_0: d | qs[16]; element i<16 = low nibble of qs[i], i+16 = high nibble.
// value d*(q-8).  unit = one block (one group).
template <>
struct Q<NT_Q4_0> {
  static constexpr int BE = 32, BB = 18, ALIGN = 32, UPB = 1, PB = 0;
  static constexpr bool FLOATX = false;  // x as fixed-point byte planes
  struct X {
    uint32_t v[kPlanes][8];
    float s;
    int off[kPlanes];  // -8 * sum(xq) over the block, split over the planes
  };
  __device__ static void load_x(X& x, const uint8_t* g, const XS& xs, int col0, int) {
#pragma unroll
    for (int k = 0; k < kPlanes; ++k) {
      ld4(g + 32 * k, x.v[k]);
      ld4(g + 32 * k + 16, x.v[k] + 4);
    }
    x.s = xs.scale[col0 / 32];
    const int* ps = xs.psum + col0 / 16;
    plane_offsets(ps[0] + ps[1], 8, x.off);
  }
  struct W {
    uint32_t lo[4], hi[4];
    float d;
  };
  __device__ static void unpack(const uint8_t* blk, int, W& w) {
    uint32_t q[4];
    lds_a2<4>(blk + 2, q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w.lo[i] = q[i] & 0x0F0F0F0Fu;
      w.hi[i] = (q[i] >> 4) & 0x0F0F0F0Fu;
    }
    w.d = __half2float(*reinterpret_cast<const __half*>(blk));
  }
  __device__ static float dotw(const W& w, int, const X& x) {
    int a[kPlanes];
#pragma unroll
    for (int k = 0; k < kPlanes; ++k) a[k] = x.off[k];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < kPlanes; ++k) {
        const bool top = k == kPlanes - 1;
        a[k] = dp<false>(top, x.v[k][4 + i], w.hi[i], dp<false>(top, x.v[k][i], w.lo[i], a[k]));
      }
    return planes(a) * (w.d * x.s);
  }
  __device__ static float dot(const uint8_t* blk, int u, const X& x) {
    W w;
    unpack(blk, u, w);
    return dotw(w, u, x);
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
  uint32_t a[kPlanes][8], b[kPlanes][8];
  float s0, s1;  // group scales
  float t0, t1;  // sum(x) over each sub-block
};
__device__ __forceinline__ void load_xk(XK& x, const uint8_t* g, const uint8_t* g2, const XS& xs, int col0, int c) {
#pragma unroll
  for (int k = 0; k < kPlanes; ++k) {
    ld4(g + 32 * k, x.a[k]);
    ld4(g + 32 * k + 16, x.a[k] + 4);
    ld4(g2 + 32 * k, x.b[k]);
    ld4(g2 + 32 * k + 16, x.b[k] + 4);
  }
  const int col = col0 + 64 * c;
  x.s0 = xs.scale[col / 32];
  x.s1 = xs.scale[col / 32 + 1];
  const int* ps = xs.psum + col / 16;
  x.t0 = float(ps[0] + ps[1]) * x.s0;
  x.t1 = float(ps[2] + ps[3]) * x.s1;
}

// one unit of one row of a 4/5-bit K format, unpacked: the quants of
// sub-blocks 2c (lo) and 2c+1 (hi) as bytes, their scales and mins, d, dmin
struct WK {
  uint32_t lo[8], hi[8];
  float sc0, sc1, m0, m1, d, dmin;
};
__device__ __forceinline__ void kq_header(const uint8_t* blk, int c, WK& w) {
  const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
  kq_scales(hdr.y, hdr.z, hdr.w, c, w.sc0, w.sc1, w.m0, w.m1);
  w.d = h2f(hdr.x & 0xFFFFu);
  w.dmin = h2f(hdr.x >> 16);
}

// the quant bytes lo (sub-block 2c) and hi (2c+1) against the plane words
// of groups A and B
__device__ __forceinline__ float kq_dotw(const WK& w, const XK& x) {
  int A[kPlanes] = {}, B[kPlanes] = {};
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int k = 0; k < kPlanes; ++k) {
      A[k] = dp<false>(k == kPlanes - 1, x.a[k][i], w.lo[i], A[k]);
      B[k] = dp<false>(k == kPlanes - 1, x.b[k][i], w.hi[i], B[k]);
    }
  const float qa = planes(A), qb = planes(B);
  // sum_j (d sc_j q - dmin m_j) x = d (sc0 s0 qa + sc1 s1 qb) - dmin (m0 t0 + m1 t1)
  return w.d * fmaf(w.sc0 * x.s0, qa, w.sc1 * x.s1 * qb) - w.dmin * fmaf(w.m0, x.t0, w.m1 * x.t1);
}

// Q4_K: d | dmin | scales[12] | qs[128].  value d*sc*q - dmin*m.
template <>
struct Q<NT_Q4_K> {
  static constexpr int BE = 256, BB = 144, ALIGN = 8, UPB = 4, PB = 1;
  static constexpr bool FLOATX = false;  // x as fixed-point byte planes
  using X = XK;
  __device__ static void load_x(X& x, const uint8_t* g, const XS& xs, int col0, int c) {
    load_xk(x, g, g + kGroupPitch, xs, col0, c);
  }
  using W = WK;
  __device__ static void unpack(const uint8_t* blk, int c, W& w) {
    kq_header(blk, c, w);
    const uint4* qp = reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 q0 = qp[0], q1 = qp[1];
    const uint32_t q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      w.lo[i] = q[i] & 0x0F0F0F0Fu;
      w.hi[i] = q[i] & 0xF0F0F0F0u;  // 16 x the high nibble: no shift; 1/16 in the combine
    }
    w.sc1 *= 0.0625f;
  }
  __device__ static float dotw(const W& w, int, const X& x) { return kq_dotw(w, x); }
  __device__ static float dot(const uint8_t* blk, int c, const X& x) {
    W w;
    unpack(blk, c, w);
    return dotw(w, c, x);
  }
};

// Q5_K: d | dmin | scales[12] | qh[32] | qs[128]; the fifth bit of element l
// of sub-block j is bit j of qh[l].
template <>
struct Q<NT_Q5_K> {
  static constexpr int BE = 256, BB = 176, ALIGN = 8, UPB = 4, PB = 1;
  static constexpr bool FLOATX = false;  // x as fixed-point byte planes
  using X = XK;
  __device__ static void load_x(X& x, const uint8_t* g, const XS& xs, int col0, int c) {
    load_xk(x, g, g + kGroupPitch, xs, col0, c);
  }
  using W = WK;
  __device__ static void unpack(const uint8_t* blk, int c, W& w) {
    kq_header(blk, c, w);
    const uint4* hp = reinterpret_cast<const uint4*>(blk + 16);
    const uint4 h0 = hp[0], h1 = hp[1];
    const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    const uint4* qp = reinterpret_cast<const uint4*>(blk + 48 + 32 * c);
    const uint4 q0 = qp[0], q1 = qp[1];
    const uint32_t q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const int b0 = 2 * c;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      w.lo[i] = (q[i] & 0x0F0F0F0Fu) | (((hw[i] >> b0) & 0x01010101u) << 4);
      w.hi[i] = ((q[i] >> 4) & 0x0F0F0F0Fu) | (((hw[i] >> (b0 + 1)) & 0x01010101u) << 4);
    }
  }
  __device__ static float dotw(const W& w, int, const X& x) { return kq_dotw(w, x); }
  __device__ static float dot(const uint8_t* blk, int c, const X& x) {
    W w;
    unpack(blk, c, w);
    return dotw(w, c, x);
  }
};
// Q6_K: ql[128] | qh[64] | scales[16] int8 | d.  value d*sc*(q-32).
// unit u = (half h = u>>1, s = u&1): chunks g = 0..3 of 16 elements at block
// columns 128h + 32g + 16s + l', l' < 16 (the s-th half of group 4h+g);
// chunk g has scale scales[8h+2g+s].
template <>
struct Q<NT_Q6_K> {
  static constexpr int BE = 256, BB = 210, ALIGN = 8, UPB = 4, PB = 2;
  static constexpr bool FLOATX = false;  // x as fixed-point byte planes
  struct X {
    uint32_t v[4][kPlanes][4];  // chunk g, plane k, 4 words (16 columns)
    float s[4];                 // group scales
    int off[4][kPlanes];        // -32 * sum(xq) over the chunk, split over the planes
  };
  __device__ static void load_x(X& x, const uint8_t* g0, const XS& xs, int col0, int u) {
    const int h = u >> 1, s = u & 1;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint8_t* p = g0 + kGroupPitch * (4 * h + g) + 16 * s;
#pragma unroll
      for (int k = 0; k < kPlanes; ++k) ld4(p + 32 * k, x.v[g][k]);
      const int col = col0 + 128 * h + 32 * g + 16 * s;
      x.s[g] = xs.scale[col / 32];
      plane_offsets(xs.psum[col / 16], 32, x.off[g]);
    }
  }
  // one unit of one row, unpacked: the 6-bit quants of chunks 0..3 (4 words
  // each, as bytes), their scales, d
  struct W {
    uint32_t q[4][4];  // word i of chunk g: q[i][g]
    float sc[4];
    float d;
  };
  __device__ static void unpack(const uint8_t* blk, int u, W& w) {
    const int h = u >> 1, s = u & 1;
    uint32_t A[4], B[4], H[4], S[2];
    lds_a2<4>(blk + 64 * h + 16 * s, A);        // low nibble: chunk 0, high: chunk 2
    lds_a2<4>(blk + 64 * h + 32 + 16 * s, B);   // low nibble: chunk 1, high: chunk 3
    lds_a2<4>(blk + 128 + 32 * h + 16 * s, H);  // bits 2g..2g+1: top bits of chunk g
    lds_a2<2>(blk + 192 + 8 * h, S);            // scales[8h .. 8h+7]
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w.q[i][0] = (A[i] & 0x0F0F0F0Fu) | ((H[i] << 4) & 0x30303030u);
      w.q[i][1] = (B[i] & 0x0F0F0F0Fu) | ((H[i] << 2) & 0x30303030u);
      w.q[i][2] = ((A[i] >> 4) & 0x0F0F0F0Fu) | (H[i] & 0x30303030u);
      w.q[i][3] = ((B[i] >> 4) & 0x0F0F0F0Fu) | ((H[i] >> 2) & 0x30303030u);
    }
    // scale of chunk g: scales[8h + 2g + s] = byte (2g + s) of the 8-byte window
    w.sc[0] = float(int8_t(S[0] >> (8 * s)));
    w.sc[1] = float(int8_t(S[0] >> (8 * s + 16)));
    w.sc[2] = float(int8_t(S[1] >> (8 * s)));
    w.sc[3] = float(int8_t(S[1] >> (8 * s + 16)));
    w.d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
  }
  __device__ static float dotw(const W& w, int, const X& x) {
    int a[4][kPlanes];
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int k = 0; k < kPlanes; ++k) a[g][k] = x.off[g][k];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int k = 0; k < kPlanes; ++k) a[g][k] = dp<false>(k == kPlanes - 1, x.v[g][k][i], w.q[i][g], a[g][k]);
    float t = w.sc[0] * x.s[0] * planes(a[0]);
    t = fmaf(w.sc[1] * x.s[1], planes(a[1]), t);
    t = fmaf(w.sc[2] * x.s[2], planes(a[2]), t);
    t = fmaf(w.sc[3] * x.s[3], planes(a[3]), t);
    return w.d * t;
  }
  __device__ static float dot(const uint8_t* blk, int u, const X& x) {
    W w;
    unpack(blk, u, w);
    return dotw(w, u, x);
  }
};

// F16 / F32: plain weights, so x stays fp32 in shared memory (32 floats per
// 32-column group at a 144-byte pitch: a quarter-warp's 16-byte reads of
// consecutive groups fall into 8 distinct bank groups) and the dot product
// is fp32 FMA.  unit = 32 values of one row.
struct XF {
  float v[32];
};

template <>
struct Q<NT_F16> {
  static constexpr int BE = 32, BB = 64, ALIGN = 8, UPB = 1, PB = 0;
  static constexpr bool FLOATX = true;
  using X = XF;
  __device__ static void load_x(X& x, const uint8_t* g, const XS&, int, int) {
#pragma unroll
    for (int k = 0; k < 8; ++k) *reinterpret_cast<float4*>(x.v + 4 * k) = *reinterpret_cast<const float4*>(g + 16 * k);
  }
  struct W {
    uint32_t h[16];  // 32 binary16 values, two per word
  };
  __device__ static void unpack(const uint8_t* blk, int, W& w) {
#pragma unroll
    for (int k = 0; k < 4; ++k) ld4(blk + 16 * k, w.h + 4 * k);
  }
  __device__ static float dotw(const W& w, int, const X& x) {
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w.h[i]));
      a = fmaf(f.x, x.v[2 * i], a);
      b = fmaf(f.y, x.v[2 * i + 1], b);
    }
    return a + b;
  }
  __device__ static float dot(const uint8_t* blk, int u, const X& x) {
    W w;
    unpack(blk, u, w);
    return dotw(w, u, x);
  }
};

template <>
struct Q<NT_F32> {
  static constexpr int BE = 32, BB = 128, ALIGN = 8, UPB = 1, PB = 0;
  static constexpr bool FLOATX = true;
  using X = XF;
  __device__ static void load_x(X& x, const uint8_t* g, const XS&, int, int) { Q<NT_F16>::load_x(x, g, XS{}, 0, 0); }
  struct W {
    float f[32];
  };
  __device__ static void unpack(const uint8_t* blk, int, W& w) {
#pragma unroll
    for (int k = 0; k < 8; ++k) *reinterpret_cast<float4*>(w.f + 4 * k) = *reinterpret_cast<const float4*>(blk + 16 * k);
  }
  __device__ static float dotw(const W& w, int, const X& x) {
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      a = fmaf(w.f[2 * i], x.v[2 * i], a);
      b = fmaf(w.f[2 * i + 1], x.v[2 * i + 1], b);
    }
    return a + b;
  }
  __device__ static float dot(const uint8_t* blk, int u, const X& x) {
    W w;
    unpack(blk, u, w);
    return dotw(w, u, x);
  }
};

// byte offset of 32-column group g: kGroupPitch bytes per group (80 with two
// planes, 112 with three), plus PB*16 bytes per 8 groups (one K block),
// chosen per format so that the 16-byte plane reads of a quarter-warp fall
// into 8 distinct bank groups; 144 bytes per group for fp32 x
template <int FMT>
__host__ __device__ constexpr int goff(int g) {
  return Q<FMT>::FLOATX ? 144 * g : kGroupPitch * g + 16 * Q<FMT>::PB * (g / 8);
}

template <int FMT>
__host__ __device__ constexpr int x_bytes(int cols) {
  return ((goff<FMT>(cols / 32 + 1) + 15) / 16) * 16;
}


// One pass of the x prologue for one warp: 8 lanes per 32-column group, 4
// columns (x4) per lane, lane `sub` = lane & 7 of group `grp`.  Converts the
// group to kXBits-bit fixed point with scale 2^-sh (sh from the exponent of
// the group's largest |x|), writes its byte planes, the sum of xq over each
// 16 columns and the scale.  Every lane of the warp must call it (shuffles);
// `live` = grp is a real group.
template <int FMT>
__device__ __forceinline__ void put_x4(float4 x4, bool live, int grp, int sub, uint8_t* xsm, int* psum,
                                       float* gscale) {
  if constexpr (Q<FMT>::FLOATX) {
    if (live) *reinterpret_cast<float4*>(xsm + goff<FMT>(grp) + 16 * sub) = x4;
    return;
  }
  float m = fmaxf(fmaxf(fabsf(x4.x), fabsf(x4.y)), fmaxf(fabsf(x4.z), fabsf(x4.w)));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  // m = f * 2^e with f in [0.5, 1): e from the exponent field; scale = 2^(kXBits - 1 - e)
  const int e = int((__float_as_uint(m) >> 23) & 0xFFu) - 126;
  const int sh = min(126, max(-126, kXBits - 1 - e));
  const float scl = __uint_as_float(uint32_t(127 + sh) << 23);
  constexpr int kLim = (1 << (kXBits - 1)) - 1;
  const int q0 = max(-kLim, min(kLim, __float2int_rn(x4.x * scl)));
  const int q1 = max(-kLim, min(kLim, __float2int_rn(x4.y * scl)));
  const int q2 = max(-kLim, min(kLim, __float2int_rn(x4.z * scl)));
  const int q3 = max(-kLim, min(kLim, __float2int_rn(x4.w * scl)));
  // byte planes: plane k holds byte k of the four values (the top one signed)
  const uint32_t lo01 = __byte_perm(q0, q1, 0x5410), lo23 = __byte_perm(q2, q3, 0x5410);  // bytes 0,1 of each
  const uint32_t pw0 = __byte_perm(lo01, lo23, 0x6420);
  const uint32_t pw1 = __byte_perm(lo01, lo23, 0x7531);
  // sum of xq over the 16 columns of this lane's quarter-group (4 lanes)
  int ps = (q0 + q1) + (q2 + q3);
  ps += __shfl_xor_sync(0xffffffffu, ps, 1);
  ps += __shfl_xor_sync(0xffffffffu, ps, 2);
  if (live) {
    uint8_t* gp = xsm + goff<FMT>(grp) + 4 * sub;
    *reinterpret_cast<uint32_t*>(gp) = pw0;
    *reinterpret_cast<uint32_t*>(gp + 32) = pw1;
    if constexpr (kPlanes == 3) {
      const uint32_t hi01 = __byte_perm(q0, q1, 0x7632), hi23 = __byte_perm(q2, q3, 0x7632);  // bytes 2,3 of each
      *reinterpret_cast<uint32_t*>(gp + 64) = __byte_perm(hi01, hi23, 0x6420);
    }
    if ((sub & 3) == 0) psum[2 * grp + (sub >> 2)] = ps;
    if (sub == 0) gscale[grp] = __uint_as_float(uint32_t(127 - sh) << 23);
  }
}

}  // namespace qf
}  // namespace nt
