// qgemv.cu — dequantize-fused GEMV for the GGUF block formats named on
// "Ntransformer" (en.unwiki.net), About (Q8_0, Q4_0, Q4_K_M = Q4_K + Q6_K,
// Q5_K, Q6_K); the GEMV kernel of "Architecture et structure du code"
// (fr.news.hada.io).  y[r] = sum_c deq(W[r,c]) x[c], fp32 accumulate.
//
// GB300 design (HBM-bound, M = 1):
//  * x (optionally RMS-normalised in the prologue) lives in shared memory as
//    fp32, with a table of 16-column partial sums used by the offset terms.
//  * Every warp owns a private ring of NST shared-memory stages fed by TMA
//    bulk copies (cp.async.bulk + mbarrier complete_tx, L2 evict-first) and
//    works on groups of R consecutive rows, so each x value read from shared
//    memory serves R rows.  Long rows are cut into column segments.
//  * Quants become floats without the int->float converter: a byte or nibble
//    is placed into the mantissa of a constant with PRMT, giving exactly
//    2^23 + b (8-bit, then one subtract) or 0.5 + q/256 (4..6-bit; the 0.5
//    offset is removed once per sub-block through the partial sums of x).
//    Products use packed fp32x2 FMAs.
//  * K-quant sub-block scale and min are applied once per 32 (16 for Q6_K)
//    elements: sum (d sc q - dmin m) x = d sc sum(q x) - dmin m sum(x).
#include "nt_internal.cuh"
#include "ops.cuh"

namespace nt {
namespace {

constexpr int kMaxWarps = 32;  // warps per CTA: a launch parameter (one CTA per SM)

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
};

// ---------------------------------------------------------------------------
// small device helpers

// 16 bytes from a 2-byte-aligned shared address, as 4 little-endian words.
__device__ __forceinline__ void lds16_a2(const uint8_t* p, uint32_t w[4]) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* b = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  const uint32_t sh = uint32_t(a & 3) * 8;
  const uint32_t t0 = b[0], t1 = b[1], t2 = b[2], t3 = b[3], t4 = b[4];
  w[0] = __funnelshift_r(t0, t1, sh);
  w[1] = __funnelshift_r(t1, t2, sh);
  w[2] = __funnelshift_r(t2, t3, sh);
  w[3] = __funnelshift_r(t3, t4, sh);
}

// 8 bytes from a 2-byte-aligned shared address.
__device__ __forceinline__ void lds8_a2(const uint8_t* p, uint32_t w[2]) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* b = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  const uint32_t sh = uint32_t(a & 3) * 8;
  const uint32_t t0 = b[0], t1 = b[1], t2 = b[2];
  w[0] = __funnelshift_r(t0, t1, sh);
  w[1] = __funnelshift_r(t1, t2, sh);
}

// byte k of v as the float 2^23 + byte (exact)
template <int K>
__device__ __forceinline__ float big(uint32_t v) {
  return __int_as_float(__byte_perm(v, 0x4B000000u, 0x7650 | K));
}
// byte k of v (< 128) as the float 0.5 + byte/256 (exact)
template <int K>
__device__ __forceinline__ float half_q(uint32_t v) {
  return __int_as_float(__byte_perm(v, 0x3F000000u, 0x7054 | (K << 8)));
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// acc += (0.5 + q_k/256) * x_k for the four bytes of v against x pair p0, p1
__device__ __forceinline__ float2 fma4(uint32_t v, float2 p0, float2 p1, float2 acc) {
  acc = __ffma2_rn(f2(half_q<0>(v), half_q<1>(v)), p0, acc);
  acc = __ffma2_rn(f2(half_q<2>(v), half_q<3>(v)), p1, acc);
  return acc;
}

__device__ __forceinline__ void ld_x4(const float* p, float2& a, float2& b) {
  const float4 t = *reinterpret_cast<const float4*>(p);
  a = f2(t.x, t.y);
  b = f2(t.z, t.w);
}

__device__ __forceinline__ float h2f(uint32_t bits16) { return __half2float(__ushort_as_half((unsigned short)bits16)); }

// ---------------------------------------------------------------------------
// per-format traits.  A "unit" is one lane's share of one block; X holds the
// unit's x values (and offset terms), loaded once and reused for R rows.

template <int FMT>
struct Q;

// x lives in shared memory with 4 pad floats after every PADC columns, PADC
// matched to the lane-to-column mapping of each format, so the float4 reads
// of the 8 lanes of a quarter-warp land in 8 different bank groups.
template <int PADC>
__device__ __forceinline__ int xidx(int col) {
  return col + 4 * (col / PADC);
}

// Q8_0: d (f16) | qs[32] int8.  value d*q.  unit = 16 quants, 2 per block.
template <>
struct Q<NT_Q8_0> {
  static constexpr int BE = 32, BB = 34, ALIGN = 8, UPB = 2, PADC = 16;
  struct X {
    float2 v[8];
  };
  __device__ static void load_x(X& x, const float* xs, const float*, int col0, int uu) {
    const float* p = xs + xidx<PADC>(col0 + 16 * uu);
#pragma unroll
    for (int k = 0; k < 4; ++k) ld_x4(p + 4 * k, x.v[2 * k], x.v[2 * k + 1]);
  }
  __device__ static float dot(const uint8_t* blk, int uu, const X& x) {
    uint32_t w[4];
    lds16_a2(blk + 2 + 16 * uu, w);
    const float d = __half2float(*reinterpret_cast<const __half*>(blk));
    const float2 c = f2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
    float2 a = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = w[i] ^ 0x80808080u;  // q + 128 as an unsigned byte
      const float2 q01 = __fadd2_rn(f2(big<0>(v), big<1>(v)), c);
      const float2 q23 = __fadd2_rn(f2(big<2>(v), big<3>(v)), c);
      a = __ffma2_rn(q01, x.v[2 * i], a);
      a = __ffma2_rn(q23, x.v[2 * i + 1], a);
    }
    return d * (a.x + a.y);
  }
};

// Q4_0: d | qs[16]; element i<16 = low nibble of qs[i], i+16 = high nibble.
// value d*(q-8).  unit = one block.
template <>
struct Q<NT_Q4_0> {
  static constexpr int BE = 32, BB = 18, ALIGN = 8, UPB = 1, PADC = 32;
  struct X {
    float2 v[16];
    float k;  // -136 * sum(x over the block): removes the 0.5 offset and the -8
  };
  __device__ static void load_x(X& x, const float* xs, const float* sx16, int col0, int) {
    const float* p = xs + xidx<PADC>(col0);
#pragma unroll
    for (int k = 0; k < 8; ++k) ld_x4(p + 4 * k, x.v[2 * k], x.v[2 * k + 1]);
    x.k = -136.0f * (sx16[col0 / 16] + sx16[col0 / 16 + 1]);
  }
  __device__ static float dot(const uint8_t* blk, int, const X& x) {
    uint32_t w[4];
    lds16_a2(blk + 2, w);
    const float d = __half2float(*reinterpret_cast<const __half*>(blk));
    float2 a = f2(0.f, 0.f), b = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
      a = fma4(lo, x.v[2 * i], x.v[2 * i + 1], a);
      b = fma4(hi, x.v[8 + 2 * i], x.v[8 + 2 * i + 1], b);
    }
    // sum (q-8) x = 256 * sum((0.5 + q/256) x) - 136 * sum(x)
    return d * fmaf(256.0f, (a.x + a.y) + (b.x + b.y), x.k);
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

// Shared X of the 4/5-bit K formats: unit c = 64 columns (sub-blocks 2c, 2c+1).
struct XK {
  float2 v[32];
  float s0, s1;  // sum(x) over each sub-block
};
__device__ __forceinline__ void load_xk(XK& x, const float* xs, const float* sx16, int col0, int c) {
  const float* p = xs + xidx<64>(col0 + 64 * c);
#pragma unroll
  for (int k = 0; k < 16; ++k) ld_x4(p + 4 * k, x.v[2 * k], x.v[2 * k + 1]);
  const float* s = sx16 + (col0 + 64 * c) / 16;
  x.s0 = s[0] + s[1];
  x.s1 = s[2] + s[3];
}

__device__ __forceinline__ float kq_combine(uint4 hdr, int c, float2 a0, float2 a1, const XK& x) {
  float sc0, sc1, m0, m1;
  kq_scales(hdr.y, hdr.z, hdr.w, c, sc0, sc1, m0, m1);
  const float d = h2f(hdr.x & 0xFFFFu), dmin = h2f(hdr.x >> 16);
  const float t0 = fmaf(256.0f, a0.x + a0.y, -128.0f * x.s0);  // sum q x, sub-block 2c
  const float t1 = fmaf(256.0f, a1.x + a1.y, -128.0f * x.s1);  // sum q x, sub-block 2c+1
  return d * fmaf(sc0, t0, sc1 * t1) - dmin * fmaf(m0, x.s0, m1 * x.s1);
}

// Q4_K: d | dmin | scales[12] | qs[128].  value d*sc*q - dmin*m.
template <>
struct Q<NT_Q4_K> {
  static constexpr int BE = 256, BB = 144, ALIGN = 1, UPB = 4, PADC = 64;
  using X = XK;
  __device__ static void load_x(X& x, const float* xs, const float* sx16, int col0, int c) {
    load_xk(x, xs, sx16, col0, c);
  }
  __device__ static float dot(const uint8_t* blk, int c, const X& x) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint4* qp = reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 q0 = qp[0], q1 = qp[1];
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float2 a0 = f2(0.f, 0.f), a1 = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a0 = fma4(w[i] & 0x0F0F0F0Fu, x.v[2 * i], x.v[2 * i + 1], a0);
      a1 = fma4((w[i] >> 4) & 0x0F0F0F0Fu, x.v[16 + 2 * i], x.v[16 + 2 * i + 1], a1);
    }
    return kq_combine(hdr, c, a0, a1, x);
  }
};

// Q5_K: d | dmin | scales[12] | qh[32] | qs[128]; fifth bit of element l of
// sub-block j is bit j of qh[l].
template <>
struct Q<NT_Q5_K> {
  static constexpr int BE = 256, BB = 176, ALIGN = 1, UPB = 4, PADC = 64;
  using X = XK;
  __device__ static void load_x(X& x, const float* xs, const float* sx16, int col0, int c) {
    load_xk(x, xs, sx16, col0, c);
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
    float2 a0 = f2(0.f, 0.f), a1 = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = (w[i] & 0x0F0F0F0Fu) | (((hw[i] >> b0) & 0x01010101u) << 4);
      const uint32_t hi = ((w[i] >> 4) & 0x0F0F0F0Fu) | (((hw[i] >> (b0 + 1)) & 0x01010101u) << 4);
      a0 = fma4(lo, x.v[2 * i], x.v[2 * i + 1], a0);
      a1 = fma4(hi, x.v[16 + 2 * i], x.v[16 + 2 * i + 1], a1);
    }
    return kq_combine(hdr, c, a0, a1, x);
  }
};

// Q6_K: ql[128] | qh[64] | scales[16] int8 | d.  value d*sc*(q-32).
// unit u = (half h = u>>1, s = u&1): elements 128h + 32g + 16s + l', g, l' < 16.
template <>
struct Q<NT_Q6_K> {
  static constexpr int BE = 256, BB = 210, ALIGN = 8, UPB = 4, PADC = 128;
  struct X {
    float2 v[32];  // v[8g + i]: the 16 columns of group g
    float k[4];    // -160 * sum(x) over group g: removes the 0.5 offset and the -32
  };
  __device__ static void load_x(X& x, const float* xs, const float* sx16, int col0, int u) {
    const int h = u >> 1, s = u & 1;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int c = col0 + 128 * h + 32 * g + 16 * s;
      const float* p = xs + xidx<PADC>(c);
#pragma unroll
      for (int k = 0; k < 4; ++k) ld_x4(p + 4 * k, x.v[8 * g + 2 * k], x.v[8 * g + 2 * k + 1]);
      x.k[g] = -160.0f * sx16[c / 16];
    }
  }
  __device__ static float dot(const uint8_t* blk, int u, const X& x) {
    const int h = u >> 1, s = u & 1;
    uint32_t A[4], B[4], H[4], S[2];
    lds16_a2(blk + 64 * h + 16 * s, A);       // low nibble: group 0, high: group 2
    lds16_a2(blk + 64 * h + 32 + 16 * s, B);  // low nibble: group 1, high: group 3
    lds16_a2(blk + 128 + 32 * h + 16 * s, H); // bits 2g..2g+1: top bits of group g
    lds8_a2(blk + 192 + 8 * h, S);            // scales[8h .. 8h+7]
    const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
    float2 a[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) a[g] = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t q0 = (A[i] & 0x0F0F0F0Fu) | ((H[i] << 4) & 0x30303030u);
      const uint32_t q1 = (B[i] & 0x0F0F0F0Fu) | ((H[i] << 2) & 0x30303030u);
      const uint32_t q2 = ((A[i] >> 4) & 0x0F0F0F0Fu) | (H[i] & 0x30303030u);
      const uint32_t q3 = ((B[i] >> 4) & 0x0F0F0F0Fu) | ((H[i] >> 2) & 0x30303030u);
      a[0] = fma4(q0, x.v[2 * i], x.v[2 * i + 1], a[0]);
      a[1] = fma4(q1, x.v[8 + 2 * i], x.v[8 + 2 * i + 1], a[1]);
      a[2] = fma4(q2, x.v[16 + 2 * i], x.v[16 + 2 * i + 1], a[2]);
      a[3] = fma4(q3, x.v[24 + 2 * i], x.v[24 + 2 * i + 1], a[3]);
    }
    // scale of group g: scales[8h + 2g + s] = byte (2g + s) of the 8-byte window
    const float sc0 = float(int8_t(S[0] >> (8 * s)));
    const float sc1 = float(int8_t(S[0] >> (8 * s + 16)));
    const float sc2 = float(int8_t(S[1] >> (8 * s)));
    const float sc3 = float(int8_t(S[1] >> (8 * s + 16)));
    float t = sc0 * fmaf(256.0f, a[0].x + a[0].y, x.k[0]);
    t = fmaf(sc1, fmaf(256.0f, a[1].x + a[1].y, x.k[1]), t);
    t = fmaf(sc2, fmaf(256.0f, a[2].x + a[2].y, x.k[2]), t);
    t = fmaf(sc3, fmaf(256.0f, a[3].x + a[3].y, x.k[3]), t);
    return d * t;
  }
};

// ---------------------------------------------------------------------------

__device__ __forceinline__ void locate(const GemvArgs& a, int64_t g, int rpg, int& j, int64_t& r0, int& nr) {
  j = 0;
  while (j + 1 < a.njobs && g >= a.job[j + 1].g0) ++j;
  r0 = (g - a.job[j].g0) * rpg;
  const int64_t left = a.job[j].rows - r0;
  nr = left < rpg ? int(left) : rpg;
}

__host__ __device__ constexpr int xs_bytes(int cols, int padc) {
  return (((cols + 4 * ((cols + padc - 1) / padc)) * 4 + 15) / 16) * 16;
}

template <int FMT, int R>
__global__ void __launch_bounds__(256, 1) qgemv_kernel(const GemvArgs a) {
  using F = Q<FMT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int nwarps = blockDim.x >> 5, kStages = a.nst;
  float* xs = reinterpret_cast<float*>(smem);
  const int xsB = xs_bytes(a.cols, F::PADC);
  float* sx16 = reinterpret_cast<float*>(smem + xsB);
  const int sxB = ((a.cols / 16 * 4 + 15) / 16) * 16;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + xsB + sxB);
  uint8_t* stages = smem + ((xsB + sxB + nwarps * kStages * 8 + 127) / 128) * 128;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- per-warp pipeline
  const int64_t total_warps = int64_t(gridDim.x) * nwarps;
  const int64_t wg = int64_t(blockIdx.x) * nwarps + warp;
  const int64_t my_groups = wg < a.total_groups ? (a.total_groups - wg + total_warps - 1) / total_warps : 0;
  const int64_t n_items = my_groups * a.nseg;
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

  // row pointer of local row i of a group (nullptr when the row is past the end)
  auto row_ptr = [&](int j, int64_t r0, int nr, int i) -> const uint8_t* {
    if (a.swiglu) {
      const int h = R / 2;
      const int k = i < h ? i : i - h;
      if (k >= nr) return nullptr;
      return (i < h ? a.job[j].W : a.job[j].W2) + (r0 + k) * a.rowB;
    }
    if (i >= nr) return nullptr;
    return a.job[j].W + (r0 + i) * a.rowB;
  };

  auto issue = [&](int64_t k) {
    const int64_t gi = wg + (k / a.nseg) * total_warps;
    const int s = int(k % a.nseg);
    int j, nr;
    int64_t r0;
    locate(a, gi, rpg, j, r0, nr);
    const int blk0 = s * a.seg;
    const int nblk = min(a.seg, a.nb - blk0);
    const uint32_t bytes_row = uint32_t(nblk) * F::BB;
    uint8_t* st = st0 + size_t(k % kStages) * a.stb;
    const uint32_t bar = bar0 + 8 * uint32_t(k % kStages);
    if (a.merged) {
      if (lane == 0) {
        const uint32_t tot = uint32_t(nr) * uint32_t(a.rowB);
        mbar_arrive_expect_tx(bar, tot);
        bulk_g2s(smem_u32(st), a.job[j].W + r0 * a.rowB, tot, bar, pol);
      }
    } else {
      const int nvalid = a.swiglu ? 2 * nr : nr;
      if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(nvalid) * bytes_row);
      __syncwarp();
      if (lane < R) {
        const uint8_t* src = row_ptr(j, r0, nr, lane);
        if (src) bulk_g2s(smem_u32(st + lane * a.segStride), src + size_t(blk0) * F::BB, bytes_row, bar, pol);
      }
    }
  };

  // plain-load path for weights that break the bulk-copy alignment rules
  auto fill_plain = [&](int64_t k, uint8_t* st) {
    const int64_t gi = wg + (k / a.nseg) * total_warps;
    const int s = int(k % a.nseg);
    int j, nr;
    int64_t r0;
    locate(a, gi, rpg, j, r0, nr);
    const int blk0 = s * a.seg;
    const int nblk = min(a.seg, a.nb - blk0);
    const int bytes_row = nblk * F::BB;
    for (int i = 0; i < R; ++i) {
      const uint8_t* src = row_ptr(j, r0, nr, i);
      if (!src) continue;
      src += size_t(blk0) * F::BB;
      for (int b = lane; b < bytes_row; b += 32) st[i * a.segStride + b] = src[b];
    }
    __syncwarp();
  };

  // weights do not depend on x: start streaming them before waiting for the
  // kernel that produces x
  if (a.tma) {
    const int64_t pre = n_items < kStages - 1 ? n_items : kStages - 1;
    for (int64_t k = 0; k < pre; ++k) issue(k);
  }
  pdl_trigger();
  pdl_wait();

  // ---- prologue: x (optionally RMS-normalised, padded layout) and 16-column partial sums
  {
    __shared__ float red[kMaxWarps];
    float ss = 0.f;
    for (int i = tid * 4; i < a.cols; i += blockDim.x * 4) {
      const float4 v = *reinterpret_cast<const float4*>(a.x + i);
      *reinterpret_cast<float4*>(xs + xidx<F::PADC>(i)) = v;
      ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    }
    if (a.norm_g) {
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      float tot = 0.f;
      for (int w = 0; w < nwarps; ++w) tot += red[w];
      const float inv = rsqrtf(tot / float(a.cols) + a.eps);
      for (int i = tid * 4; i < a.cols; i += blockDim.x * 4) {
        float4* px = reinterpret_cast<float4*>(xs + xidx<F::PADC>(i));
        float4 v = *px;
        const float4 g = *reinterpret_cast<const float4*>(a.norm_g + i);
        v.x = v.x * inv * g.x;
        v.y = v.y * inv * g.y;
        v.z = v.z * inv * g.z;
        v.w = v.w * inv * g.w;
        *px = v;
      }
    }
    __syncthreads();
    for (int i = tid; i < a.cols / 16; i += blockDim.x) {
      const float* p = xs + xidx<F::PADC>(16 * i);
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) s += p[k];
      sx16[i] = s;
    }
    __syncthreads();
  }

  if (my_groups == 0) return;

  float acc[R];
#pragma unroll
  for (int i = 0; i < R; ++i) acc[i] = 0.f;

  for (int64_t k = 0; k < n_items; ++k) {
    uint8_t* st = st0 + size_t(k % kStages) * a.stb;
    if (a.tma) {
      if (k + kStages - 1 < n_items) issue(k + kStages - 1);
      const bool ok = mbar_wait(bar0 + 8 * uint32_t(k % kStages), uint32_t((k / kStages) & 1));
      if (!__all_sync(0xffffffffu, ok)) {
        // a copy never landed: flag it, wait (bounded) for what is in flight, stop
        if (lane == 0) flag_error(a.err, kErrWaitTimeout);
        const int64_t last = min(n_items, k + kStages - 1);
        for (int64_t q = k + 1; q < last; ++q) mbar_wait(bar0 + 8 * uint32_t(q % kStages), uint32_t((q / kStages) & 1));
        return;
      }
    } else {
      fill_plain(k, st);
    }
    const int s = int(k % a.nseg);
    const int blk0 = s * a.seg;
    const int nblk = min(a.seg, a.nb - blk0);
    const int units = nblk * F::UPB;
    for (int u = lane; u < units; u += 32) {
      const int b = u / F::UPB, uu = u % F::UPB;
      typename F::X x;
      F::load_x(x, xs, sx16, (blk0 + b) * F::BE, uu);
      const uint8_t* bp = st + b * F::BB;
#pragma unroll
      for (int i = 0; i < R; ++i) acc[i] += F::dot(bp + i * a.segStride, uu, x);
    }
    __syncwarp();
    if (s == a.nseg - 1) {
      // group done: reduce across lanes, lane i writes row i
      float mine = 0.f, other = 0.f;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const float v = warp_sum(acc[i]);
        if (lane == i) mine = v;
        if (a.swiglu && lane + R / 2 == i) other = v;
        acc[i] = 0.f;
      }
      const int64_t gi = wg + (k / a.nseg) * total_warps;
      int j, nr;
      int64_t r0;
      locate(a, gi, rpg, j, r0, nr);
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
            float cs, sn;
            rope_cs(pos, a.rope.inv_freq[d >> 1], cs, sn);
            out = (d & 1) ? fmaf(partner, sn, mine * cs) : fmaf(mine, cs, -partner * sn);
          }
          if (J.epi == kEpiRope)
            J.y[r] = out;
          else
            J.cache[(int64_t(head) * a.rope.kv_stride + pos) * hd + d] = __float2half_rn(out);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host side

template <int FMT, int R>
cudaError_t launch_t(const Ctx* c, const GemvArgs& a, int grid, size_t smem, cudaStream_t st) {
  return launch_k(c, qgemv_kernel<FMT, R>, dim3(grid), dim3(c->gemv_warps * 32), smem, st, a);
}

// dynamic shared memory a kernel may use: the opt-in limit minus its static part
template <typename K>
cudaError_t allow_smem(K kernel, int optin) {
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - int(fa.sharedSizeBytes));
}

template <int FMT>
cudaError_t configure_fmt(int smem) {
  cudaError_t e = allow_smem(qgemv_kernel<FMT, 4>, smem);
  if (e == cudaSuccess) e = allow_smem(qgemv_kernel<FMT, 2>, smem);
  return e;
}

template <int FMT>
cudaError_t dispatch_r(const Ctx* c, int R, const GemvArgs& a, int grid, size_t smem, cudaStream_t st) {
  return R == 4 ? launch_t<FMT, 4>(c, a, grid, smem, st) : launch_t<FMT, 2>(c, a, grid, smem, st);
}

constexpr int align_of(int fmt) { return (fmt == NT_Q4_K || fmt == NT_Q5_K) ? 1 : 8; }

}  // namespace

// Allow every GEMV instantiation the opt-in shared memory once, at context
// creation (never during a stream capture).
nt_status configure_gemv(Ctx* c) {
  const int smem = int(c->smem_optin);
  cudaError_t e = configure_fmt<NT_Q8_0>(smem);
  if (e == cudaSuccess) e = configure_fmt<NT_Q4_0>(smem);
  if (e == cudaSuccess) e = configure_fmt<NT_Q4_K>(smem);
  if (e == cudaSuccess) e = configure_fmt<NT_Q5_K>(smem);
  if (e == cudaSuccess) e = configure_fmt<NT_Q6_K>(smem);
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
  const int BE = block_elems(fmt), BB = block_bytes(fmt);
  const int64_t nb = cols / BE;
  const int64_t rowB = nb * BB;
  bool tma = (rowB % 16) == 0;
  for (int j = 0; j < njobs; ++j) tma = tma && aligned(jobsx[j].j.W_dev, 16);
  if (swiglu) tma = tma && aligned(W2, 16);

  static const int padc_of[5] = {16, 32, 64, 64, 128};
  const int kWarps = c->gemv_warps, kStages = c->gemv_stages;
  const int xsB = xs_bytes(int(cols), padc_of[fmt]);
  const int sxB = int(((cols / 16 * 4 + 15) / 16) * 16);
  const int head = ((xsB + sxB + kWarps * kStages * 8 + 127) / 128) * 128;
  const int pad = 16;  // the unaligned 16-byte reader may touch 4 bytes past a stage
  const long avail = long(c->smem_optin) - head - pad - 256;  // 256: static shared memory
  int stb = int(avail / (kWarps * kStages)) / 16 * 16;
  if (stb > c->gemv_stage_max) stb = c->gemv_stage_max;

  GemvArgs a{};
  int R = 0;
  const int al = align_of(fmt);
  for (int r : {4, 2}) {
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
  if (R == 0 || stb < 256)
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
  int64_t grid64 = (g + kWarps - 1) / kWarps;
  if (grid64 > c->num_sms) grid64 = c->num_sms;
  const int grid = int(grid64);
  const size_t smem = size_t(head) + size_t(kWarps) * kStages * stb + pad;

  cudaError_t e;
  switch (fmt) {
    case NT_Q8_0: e = dispatch_r<NT_Q8_0>(c, R, a, grid, smem, st); break;
    case NT_Q4_0: e = dispatch_r<NT_Q4_0>(c, R, a, grid, smem, st); break;
    case NT_Q4_K: e = dispatch_r<NT_Q4_K>(c, R, a, grid, smem, st); break;
    case NT_Q5_K: e = dispatch_r<NT_Q5_K>(c, R, a, grid, smem, st); break;
    default: e = dispatch_r<NT_Q6_K>(c, R, a, grid, smem, st); break;
  }
  return cuda_check(c, e, "qgemv launch");
}

// ---------------------------------------------------------------------------
// dequantisation of whole rows (embedding lookup; bit-exact parity checks)

namespace {

__device__ __forceinline__ int quant_of(int fmt, const uint8_t* b, int i) {
  switch (fmt) {
    case NT_Q8_0: return int(int8_t(b[2 + i]));
    case NT_Q4_0: return i < 16 ? (b[2 + i] & 15) : (b[2 + i - 16] >> 4);
    case NT_Q4_K: {
      const int j = i >> 5, l = i & 31, c = j >> 1;
      const uint8_t v = b[16 + 32 * c + l];
      return (j & 1) ? (v >> 4) : (v & 15);
    }
    case NT_Q5_K: {
      const int j = i >> 5, l = i & 31, c = j >> 1;
      const uint8_t v = b[48 + 32 * c + l];
      return ((j & 1) ? (v >> 4) : (v & 15)) | (((b[16 + l] >> j) & 1) << 4);
    }
    default: {
      const int h = i >> 7, e = i & 127, g = e >> 5, l = e & 31;
      const uint8_t* ql = b + 64 * h;
      const uint8_t lo = (g & 1) ? ql[l + 32] : ql[l];
      const int q4 = (g >= 2) ? (lo >> 4) : (lo & 15);
      return q4 | (((b[128 + 32 * h + l] >> (2 * g)) & 3) << 4);
    }
  }
}

__device__ __forceinline__ void kq_sm(const uint8_t* s, int j, int& sc, int& m) {
  if (j < 4) {
    sc = s[j] & 63;
    m = s[j + 4] & 63;
  } else {
    sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
    m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
  }
}

__global__ void dequant_kernel(int fmt, const uint8_t* W, int64_t row0, int64_t nrows, int64_t cols, float* out) {
  const int BE = block_elems(fmt), BB = block_bytes(fmt);
  const int64_t nb = cols / BE;
  const int64_t total = nrows * cols;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = e / cols, col = e % cols;
    const uint8_t* b = W + ((row0 + r) * nb + col / BE) * BB;
    const int i = int(col % BE);
    float v;
    switch (fmt) {
      case NT_Q8_0: v = __fmul_rn(__half2float(*reinterpret_cast<const __half*>(b)), float(quant_of(fmt, b, i))); break;
      case NT_Q4_0:
        v = __fmul_rn(__half2float(*reinterpret_cast<const __half*>(b)), float(quant_of(fmt, b, i) - 8));
        break;
      case NT_Q4_K:
      case NT_Q5_K: {
        int sc, m;
        kq_sm(b + 4, i >> 5, sc, m);
        const float d = __half2float(*reinterpret_cast<const __half*>(b));
        const float dm = __half2float(*reinterpret_cast<const __half*>(b + 2));
        v = __fsub_rn(__fmul_rn(__fmul_rn(d, float(sc)), float(quant_of(fmt, b, i))), __fmul_rn(dm, float(m)));
        break;
      }
      default: {
        const int s = int(int8_t(b[192 + (i >> 7) * 8 + ((i & 127) >> 4)]));
        v = __fmul_rn(__half2float(*reinterpret_cast<const __half*>(b + 208)), float(s * (quant_of(fmt, b, i) - 32)));
        break;
      }
    }
    out[e] = v;
  }
}

// row *token_dev of an embedding table, dequantised (token read on the device)
__global__ void embed_kernel(int fmt, const uint8_t* W, int64_t cols, const int32_t* token_dev, float* out) {
  pdl_wait();
  pdl_trigger();
  const int64_t row = *token_dev;
  const int BE = block_elems(fmt), BB = block_bytes(fmt);
  const int64_t nb = cols / BE;
  for (int64_t col = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; col < cols; col += int64_t(gridDim.x) * blockDim.x) {
    const uint8_t* b = W + (row * nb + col / BE) * BB;
    const int i = int(col % BE);
    float v;
    switch (fmt) {
      case NT_Q8_0: v = __fmul_rn(__half2float(*reinterpret_cast<const __half*>(b)), float(quant_of(fmt, b, i))); break;
      case NT_Q4_0:
        v = __fmul_rn(__half2float(*reinterpret_cast<const __half*>(b)), float(quant_of(fmt, b, i) - 8));
        break;
      case NT_Q4_K:
      case NT_Q5_K: {
        int sc, m;
        kq_sm(b + 4, i >> 5, sc, m);
        const float d = __half2float(*reinterpret_cast<const __half*>(b));
        const float dm = __half2float(*reinterpret_cast<const __half*>(b + 2));
        v = __fsub_rn(__fmul_rn(__fmul_rn(d, float(sc)), float(quant_of(fmt, b, i))), __fmul_rn(dm, float(m)));
        break;
      }
      default: {
        const int s = int(int8_t(b[192 + (i >> 7) * 8 + ((i & 127) >> 4)]));
        v = __fmul_rn(__half2float(*reinterpret_cast<const __half*>(b + 208)), float(s * (quant_of(fmt, b, i) - 32)));
        break;
      }
    }
    out[col] = v;
  }
}

}  // namespace

nt_status launch_embed(Ctx* c, int fmt, const void* W, int64_t cols, const int32_t* token_dev, float* out,
                       cudaStream_t st) {
  const int blocks = int((cols + 255) / 256);
  return cuda_check(c, launch_k(c, embed_kernel, dim3(blocks), dim3(256), 0, st, fmt, static_cast<const uint8_t*>(W),
                                cols, token_dev, out),
                    "embed launch");
}

nt_status launch_dequant(Ctx* c, int fmt, const void* W, int64_t row0, int64_t nrows, int64_t cols, float* out,
                         cudaStream_t st) {
  const int64_t total = nrows * cols;
  if (total == 0) return NT_OK;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = int64_t(c->num_sms) * 8;
  if (blocks > cap) blocks = cap;
  dequant_kernel<<<int(blocks), 256, 0, st>>>(fmt, static_cast<const uint8_t*>(W), row0, nrows, cols, out);
  return cuda_check(c, cudaGetLastError(), "dequant launch");
}

}  // namespace nt
