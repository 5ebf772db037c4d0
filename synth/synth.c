/*
 * synth.c — seeded, counter-based synthetic inputs for the block-quantized
 * decode path.  This module draws random bytes and normals; it holds none of
 * the method's arithmetic (no dequantisation, no dot products).  Both the CUDA
 * path and the CPU oracle read the bytes it writes.
 *
 * Generator: the SplitMix64 output function (Steele, Lea & Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014) applied to a
 * 64-bit key  (seed << 56) ^ (stream << 40) ^ counter , so every element is a
 * pure function of (seed, stream, counter) and can be generated in parallel.
 * Normals: Box & Muller (1958), z = sqrt(-2 ln u1) cos(2 pi u2).
 *
 * Block byte layouts follow the GGUF-style formats named on the pages
 * ("Ntransformer", en.unwiki.net — About: Q4_0, Q8_0, Q4_K_M, Q5_K, Q6_K, F16,
 * F32; the float formats are handled as "blocks" of 32 plain values);
 * this file only needs to know where the fp16 scale fields sit and which
 * bytes carry quants, because every other byte is drawn uniformly.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* format ids — kept identical to the numbering of the public C ABI */
enum { SY_Q8_0 = 0, SY_Q4_0 = 1, SY_Q4_K = 2, SY_Q5_K = 3, SY_Q6_K = 4, SY_F16 = 5, SY_F32 = 6 };

static inline uint64_t sm64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t seed, uint64_t stream, uint64_t ctr) {
  return sm64((seed << 56) ^ (stream << 40) ^ (ctr & 0xFFFFFFFFFFull));
}

/* u in (0, 1] from the top 53 bits */
static inline double unit_open0(uint64_t h) { return ((double)(h >> 11) + 1.0) * 0x1.0p-53; }
static inline double unit_closed0(uint64_t h) { return (double)(h >> 11) * 0x1.0p-53; }

static inline double box_muller(uint64_t h1, uint64_t h2) {
  const double two_pi = 6.283185307179586476925286766559;
  return sqrt(-2.0 * log(unit_open0(h1))) * cos(two_pi * unit_closed0(h2));
}

/* double -> IEEE-754 binary16 bits, round to nearest, ties to even */
static uint16_t to_half_bits(double v) {
  uint16_t sign = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (isnan(a)) return (uint16_t)(sign | 0x7E00u);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u); /* rounds to infinity */
  int e;
  (void)frexp(a, &e);          /* a = m * 2^e, m in [0.5, 1) */
  int E = e - 1;               /* a = (1 + f) * 2^E */
  if (a == 0.0 || E < -14) {   /* subnormal range: a = k * 2^-24 */
    double k = nearbyint(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)k); /* k == 1024 is the smallest normal */
  }
  double f = nearbyint((ldexp(a, -E) - 1.0) * 1024.0);
  if (f >= 1024.0) { f = 0.0; E += 1; }
  if (E > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)f);
}

static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }

/* fill n bytes with uniform random bytes taken 8 at a time from counters c0.. */
static void rand_bytes(uint8_t* p, int n, uint64_t seed, uint64_t stream, uint64_t c0) {
  for (int i = 0; i < n; i += 8) {
    uint64_t h = draw(seed, stream, c0 + (uint64_t)(i >> 3));
    for (int k = 0; k < 8 && i + k < n; ++k) p[i + k] = (uint8_t)(h >> (8 * k));
  }
}

int sy_block_elems(int fmt) {
  switch (fmt) {
    case SY_Q8_0: case SY_Q4_0: case SY_F16: case SY_F32: return 32;
    case SY_Q4_K: case SY_Q5_K: case SY_Q6_K: return 256;
    default: return 0;
  }
}
int sy_block_bytes(int fmt) {
  switch (fmt) {
    case SY_Q8_0: return 34;
    case SY_Q4_0: return 18;
    case SY_Q4_K: return 144;
    case SY_Q5_K: return 176;
    case SY_Q6_K: return 210;
    case SY_F16: return 64;   /* 32 binary16 values, no scale */
    case SY_F32: return 128;  /* 32 binary32 values */
    default: return 0;
  }
}

/*
 * One block j of tensor `stream`.  Counters j*64 + k (k < 64) belong to block
 * j: k = 0,1 feed the normal of the first fp16 scale, k = 2,3 the second,
 * k >= 4 the uniform bytes.  Scales are f16(|N(0,1)| * scale_std).
 * Q8_0 quants are uniform over -127..127; every other quant, sub-scale and
 * high-bit byte is a uniform random byte, which makes every packed bit field
 * uniform over its own range.
 */
static void fill_block(int fmt, uint8_t* b, uint64_t seed, uint64_t stream, uint64_t j, double scale_std) {
  const uint64_t c = j * 64u;
  double n0 = fabs(box_muller(draw(seed, stream, c + 0), draw(seed, stream, c + 1))) * scale_std;
  double n1 = fabs(box_muller(draw(seed, stream, c + 2), draw(seed, stream, c + 3))) * scale_std;
  switch (fmt) {
    case SY_Q8_0: {
      put_u16(b, to_half_bits(n0));
      for (int i = 0; i < 32; i += 2) {
        uint64_t h = draw(seed, stream, c + 4 + (uint64_t)(i >> 1));
        uint32_t lo = (uint32_t)h, hi = (uint32_t)(h >> 32);
        b[2 + i] = (uint8_t)(int8_t)((int)(((uint64_t)lo * 255u) >> 32) - 127);
        b[3 + i] = (uint8_t)(int8_t)((int)(((uint64_t)hi * 255u) >> 32) - 127);
      }
      break;
    }
    case SY_Q4_0:
      put_u16(b, to_half_bits(n0));
      rand_bytes(b + 2, 16, seed, stream, c + 4);
      break;
    case SY_Q4_K:
      put_u16(b, to_half_bits(n0));
      put_u16(b + 2, to_half_bits(n1));
      rand_bytes(b + 4, 140, seed, stream, c + 4);
      break;
    case SY_Q5_K:
      put_u16(b, to_half_bits(n0));
      put_u16(b + 2, to_half_bits(n1));
      rand_bytes(b + 4, 172, seed, stream, c + 4);
      break;
    case SY_Q6_K:
      rand_bytes(b, 208, seed, stream, c + 4);
      put_u16(b + 208, to_half_bits(n0));
      break;
    case SY_F16:
    case SY_F32:
      /* plain weights N(0, scale_std^2): element i from counters c + 2i, c + 2i + 1 */
      for (int i = 0; i < 32; ++i) {
        double v = box_muller(draw(seed, stream, c + 2u * (uint64_t)i), draw(seed, stream, c + 2u * (uint64_t)i + 1u)) *
                   scale_std;
        if (fmt == SY_F16) {
          put_u16(b + 2 * i, to_half_bits(v));
        } else {
          float f = (float)v;
          memcpy(b + 4 * i, &f, 4);  /* little-endian on every supported host */
        }
      }
      break;
    default: break;
  }
}

/* rows x cols matrix of blocks, row-major, cols/block_elems blocks per row.
 * Returns 0 on success, -1 on a bad format or a ragged column count. */
int sy_fill_quant(int fmt, uint8_t* out, int64_t rows, int64_t cols, uint64_t seed, uint32_t stream,
                  double scale_std) {
  int be = sy_block_elems(fmt), bb = sy_block_bytes(fmt);
  if (be == 0 || cols % be != 0 || rows < 0) return -1;
  int64_t nblk = rows * (cols / be);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nblk; ++j) fill_block(fmt, out + j * bb, seed, stream, (uint64_t)j, scale_std);
  return 0;
}

/* n fp32 values mean + std * N(0,1); element i uses counters 2i, 2i+1 */
void sy_fill_normal_f32(float* out, int64_t n, double mean, double std, uint64_t seed, uint32_t stream) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double z = box_muller(draw(seed, stream, 2u * (uint64_t)i), draw(seed, stream, 2u * (uint64_t)i + 1u));
    out[i] = (float)(mean + std * z);
  }
}

/* n binary16 values f16(std * N(0,1)) */
void sy_fill_normal_f16(uint16_t* out, int64_t n, double std, uint64_t seed, uint32_t stream) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double z = box_muller(draw(seed, stream, 2u * (uint64_t)i), draw(seed, stream, 2u * (uint64_t)i + 1u));
    out[i] = to_half_bits(std * z);
  }
}

/* n uniform bytes (used by edge-case tests that want arbitrary block bytes) */
void sy_fill_bytes(uint8_t* out, int64_t n, uint64_t seed, uint32_t stream) {
  int64_t nw = (n + 7) / 8;
#pragma omp parallel for schedule(static)
  for (int64_t w = 0; w < nw; ++w) {
    uint64_t h = draw(seed, stream, (uint64_t)w);
    for (int k = 0; k < 8 && w * 8 + k < n; ++k) out[w * 8 + k] = (uint8_t)(h >> (8 * k));
  }
}

int sy_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
