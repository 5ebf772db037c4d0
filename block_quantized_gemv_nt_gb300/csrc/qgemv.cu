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
#include <algorithm>
#include <string>
#include <vector>

#include "nt_internal.cuh"
#include "ops.cuh"
#include "qformats.cuh"

namespace nt {
namespace {

using namespace qf;

constexpr int kMaxWarps = 32;
constexpr int kMaxChunks = 512;  // 128-column chunks of a normalised x (cols <= 65536)

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
  int stall;          // test hook: issue no bulk copies; waits give up after kStallSpin tries
};

// the R per-lane partial sums of a row group, summed over the warp: lane
// i < R returns row i.  A butterfly that halves the rows each lane carries
// before the plain tree: 7 shuffles for R = 4 and 6 for R = 2, against 5 per
// row for R separate warp sums.
__device__ __forceinline__ float rows_reduce(float (&a)[4], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8;
  float k0 = b4 ? a[2] : a[0], k1 = b4 ? a[3] : a[1];  // rows 2*b4 and 2*b4 + 1 stay
  k0 += __shfl_xor_sync(0xffffffffu, b4 ? a[0] : a[2], 16);
  k1 += __shfl_xor_sync(0xffffffffu, b4 ? a[1] : a[3], 16);
  float k = b3 ? k1 : k0;                               // row 2*b4 + b3 stays
  k += __shfl_xor_sync(0xffffffffu, b3 ? k0 : k1, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return __shfl_sync(0xffffffffu, k, (lane & 3) * 8);  // row r lives on lane 8r
}
__device__ __forceinline__ float rows_reduce(float (&a)[2], int lane) {
  const bool b4 = lane & 16;
  float k = b4 ? a[1] : a[0];
  k += __shfl_xor_sync(0xffffffffu, b4 ? a[0] : a[1], 16);
  k += __shfl_xor_sync(0xffffffffu, k, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return __shfl_sync(0xffffffffu, k, (lane & 1) * 16);  // row r lives on lane 16r
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
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
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ((xB + 12 * ng + 7) / 8) * 8);
  uint8_t* stages = smem + ((xB + 12 * ng + 8 + nwarps * kStages * 8 + 127) / 128) * 128;

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
          if (!a.stall) bulk_g2s(smem_u32(st), a.job[g_j].W + g_r0 * a.rowB, tot, bar, pol);
        }
      } else {
        const int nvalid = a.swiglu ? 2 * g_nr : g_nr;
        if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(nvalid) * bytes_row);
        __syncwarp();
        if (my_row && !a.stall)
          bulk_g2s(smem_u32(st + lane * a.segStride), my_row + size_t(blk0) * F::BB, bytes_row, bar, pol);
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

  // ---- prologue: x (times the RMSNorm gain when asked) -> 24-bit fixed point
  // per 32-column group.  8 lanes per group of 32 columns, 4 columns per lane;
  // a warp covers 4 groups per pass.  All of a lane's x loads are issued first
  // (one memory round trip); the RMSNorm sum of squares comes from the same
  // registers, and its scalar rsqrt(mean x^2 + eps) multiplies the row sums in
  // the epilogue, so the quantization waits for no CTA-wide reduction.
  float inv = 1.f;
  {
    // sum of squares of x per 128-column chunk, then over the chunks in
    // index order: the same additions whatever the warp count
    __shared__ float red[kMaxChunks];
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
    const int nchunk = (ng + 3) / 4;  // a warp's pass covers chunk warp + pass * nwarps
    if (a.norm_g) {
      if (whole) {
#pragma unroll
        for (int k = 0; k < kPF; ++k) {
          if (k >= npass) break;  // warp-uniform
          float ss = fmaf(v[k].x, v[k].x, fmaf(v[k].y, v[k].y, fmaf(v[k].z, v[k].z, v[k].w * v[k].w)));
          ss = warp_sum(ss);
          if (lane == 0) red[warp + k * nwarps] = ss;
        }
      } else {
        for (int ch = warp; ch < nchunk; ch += nwarps) {
          const int grp = 4 * ch + (lane >> 3);
          float ss = 0.f;
          if (grp < ng) {
            const float4 t = *reinterpret_cast<const float4*>(a.x + 32 * grp + 4 * sub);
            ss = fmaf(t.x, t.x, fmaf(t.y, t.y, fmaf(t.z, t.z, t.w * t.w)));
          }
          ss = warp_sum(ss);
          if (lane == 0) red[ch] = ss;
        }
      }
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
          x4.x *= g.x;
          x4.y *= g.y;
          x4.z *= g.z;
          x4.w *= g.w;
        }
        put_x4<FMT>(x4, live, grp, sub, xsm, psum, gscale);
      }
    }
    __syncthreads();
    if (a.norm_g) {
      float tot = 0.f;
      for (int ch = 0; ch < nchunk; ++ch) tot += red[ch];
      inv = rsqrtf(tot / float(a.cols) + a.eps);
    }
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
      const int cap = a.stall ? kStallSpin : kMaxSpin;
      const bool ok = mbar_wait(bar0 + 8 * uint32_t(cs), cph, cap);
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
          mbar_wait(bar0 + 8 * uint32_t(q), ph, cap);
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
      float mine = rows_reduce(acc, lane);
#pragma unroll
      for (int i = 0; i < R; ++i) acc[i] = 0.f;
      if (KS > 1) {
        // the parts of a split group meet in shared memory (double-buffered by group parity)
        float* xb = xchg + ((ct & 1) * slots + slot) * KS * R;
        if (part > 0 && lane < R) xb[part * R + lane] = mine;
        named_sync(1 + slot, 32 * KS);
        if (part == 0 && lane < R)
          for (int p = 1; p < KS; ++p) mine += xb[p * R + lane];
      }
      if (part == 0) {
        mine *= inv;  // the RMSNorm scalar (1 without a norm)
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
            else if (pos >= 0 && pos < a.rope.kv_stride)
              J.cache[(int64_t(head) * a.rope.kv_stride + pos) * hd + d] = __float2half_rn(out);
            else
              flag_error(a.err, kErrPosRange);
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
    case NT_Q6_K: return {Q<NT_Q6_K>::ALIGN, x_bytes<NT_Q6_K>(cols)};
    case NT_F16: return {Q<NT_F16>::ALIGN, x_bytes<NT_F16>(cols)};
    default: return {Q<NT_F32>::ALIGN, x_bytes<NT_F32>(cols)};
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
  if (e == cudaSuccess) e = configure_fmt<NT_F16>(smem, &st);
  if (e == cudaSuccess) e = configure_fmt<NT_F32>(smem, &st);
  c->gemv_static_smem = st;
  return cuda_check(c, e, "gemv shared-memory attribute");
}

nt_status launch_gemv(Ctx* c, int fmt, const nt_gemv_job* jobs, int njobs, const void* W2, const float* x,
                      const float* norm_g, float eps, int64_t cols, bool swiglu, cudaStream_t st) {
  GemvJobEx ex[3];
  for (int j = 0; j < njobs && j < 3; ++j) ex[j] = GemvJobEx{jobs[j], kEpiPlain, nullptr};
  return launch_gemv_ex(c, fmt, ex, njobs, W2, x, norm_g, eps, cols, swiglu, nullptr, st);
}

namespace {

// one launch configuration of the GEMV
struct Plan {
  GemvArgs a{};
  int R = 0, warps = 0, grid = 0;
  size_t smem = 0;
};

// blocks per segment granule: a multiple of the format's alignment unit that
// also holds a multiple of 32 lane units, so that lane l always takes the
// units l, l + 32, ... of a row part, in that order, whatever the segment size
int seg_granule(int fmt, int align) { return (fmt == NT_F16 || fmt == NT_F32) ? 32 : align; }

// The arithmetic of a launch shape: rows per lane group R and column parts
// KS.  Together with the granule above they fix every addition a row's sum
// goes through, so they are a function of the shape (and the device's SM
// count and shared memory) alone: the plans the tuner times differ only in
// warps per CTA and stage size, and never change a result bit.
struct Arith {
  int R, ks;
};
Arith arith_plan(const Ctx* c, int fmt, const GemvJobEx* jobsx, int njobs, int64_t cols, bool swiglu) {
  const int BB = block_bytes(fmt);
  const int64_t nb = cols / block_elems(fmt);
  const int64_t rowB = nb * BB;
  const FmtInfo fi = fmt_info(fmt, int(cols));
  const int al = seg_granule(fmt, fi.align);
  const int ng = int(cols / 32);
  const int nw = 16, ns = 2;  // the default launch
  const int head = ((fi.xbytes + 12 * ng + 8 + nw * ns * 8 + 127) / 128) * 128;
  const long avail = long(c->smem_optin) - head - 16 - c->gemv_static_smem;
  long stb = avail / (nw * ns) / 16 * 16;
  if (stb > 12288) stb = 12288;
  Arith r{4, 1};
  if (!(4 * rowB <= stb || 4L * al * BB <= stb)) r.R = 2;
  const int rpg = swiglu ? r.R / 2 : r.R;
  int64_t g = 0;
  for (int j = 0; j < njobs; ++j) g += (jobsx[j].j.rows + rpg - 1) / rpg;
  // split a row over KS warps when there are too few row groups to give every
  // warp of every SM the same amount of work
  const int units = int(nb / al);
  const int64_t T = int64_t(c->num_sms) * nw;
  double best = 0.0;
  for (int cand : {1, 2, 4}) {
    if (cand > 1 && units < cand) continue;
    const int64_t u = g * cand;
    const int64_t per = (u + T - 1) / T;
    const double eff = double(u) / double(T * per);
    if (eff > best + 0.02) {
      best = eff;
      r.ks = cand;
    }
  }
  return r;
}

// the launch plan for `pc` (warps, stage size cap, split-K: 0 = by balance);
// false when x leaves no shared-memory room for it
bool make_plan(const Ctx* c, int fmt, const GemvJobEx* jobsx, int njobs, const void* W2, const float* x,
               const float* norm_g, float eps, int64_t cols, bool swiglu, const RopeArgs* rope, PlanChoice pc,
               Plan& P) {
  const int BB = block_bytes(fmt);
  const int64_t nb = cols / block_elems(fmt);
  const int64_t rowB = nb * BB;
  bool tma = (rowB % 16) == 0;
  for (int j = 0; j < njobs; ++j) tma = tma && aligned(jobsx[j].j.W_dev, 16);
  if (swiglu) tma = tma && aligned(W2, 16);

  const FmtInfo fi = fmt_info(fmt, int(cols));
  const int ng = int(cols / 32);
  const int pad = 16;  // the unaligned readers may touch 4 bytes past a stage
  if (norm_g && (ng + 3) / 4 > kMaxChunks) return false;
  GemvArgs& a = P.a;
  a = GemvArgs{};
  int R = 0, kStages = 0, kWarps = 0, head = 0, stb = 0;
  const int al = seg_granule(fmt, fi.align);
  const int nw = pc.warps;
  const Arith ar = arith_plan(c, fmt, jobsx, njobs, cols, swiglu);
  for (int ns = c->gemv_stages; ns >= 2 && R == 0; --ns) {
    head = ((fi.xbytes + 12 * ng + 8 + nw * ns * 8 + 127) / 128) * 128;
    const long avail = long(c->smem_optin) - head - pad - c->gemv_static_smem;
    stb = int(avail / (nw * ns)) / 16 * 16;
    if (stb > pc.stage_max) stb = pc.stage_max;
    if (stb < 256) continue;
    for (int r : {ar.R}) {
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
  if (R == 0) return false;

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

  // the column parts of the shape's arithmetic (arith_plan)
  const int ks = ar.ks;
  const int units = int(nb / al);  // granule units per row
  if (kWarps % ks || (ks > 1 && units < ks)) return false;
  a.ks = ks;
  if (ks == 1) {
    a.pblk[0] = 0;
    a.pblk[1] = int(nb);
  } else {
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
  P.R = R;
  P.warps = kWarps;
  P.grid = int(grid64 > 0 ? grid64 : 1);
  P.smem = size_t(head) + size_t(kWarps) * kStages * stb + pad;
  return true;
}

cudaError_t launch_plan(const Ctx* c, int fmt, const Plan& P, cudaStream_t st) {
  switch (fmt) {
    case NT_Q8_0: return dispatch_r<NT_Q8_0>(c, P.R, P.a, P.warps, P.grid, P.smem, st);
    case NT_Q4_0: return dispatch_r<NT_Q4_0>(c, P.R, P.a, P.warps, P.grid, P.smem, st);
    case NT_Q4_K: return dispatch_r<NT_Q4_K>(c, P.R, P.a, P.warps, P.grid, P.smem, st);
    case NT_Q5_K: return dispatch_r<NT_Q5_K>(c, P.R, P.a, P.warps, P.grid, P.smem, st);
    case NT_Q6_K: return dispatch_r<NT_Q6_K>(c, P.R, P.a, P.warps, P.grid, P.smem, st);
    case NT_F16: return dispatch_r<NT_F16>(c, P.R, P.a, P.warps, P.grid, P.smem, st);
    default: return dispatch_r<NT_F32>(c, P.R, P.a, P.warps, P.grid, P.smem, st);
  }
}

// the shape of a launch: what the plan depends on
std::string plan_key(int fmt, const GemvJobEx* jobsx, int njobs, const void* W2, int64_t cols, bool swiglu) {
  char buf[160];
  bool tma = true;
  for (int j = 0; j < njobs; ++j) tma = tma && aligned(jobsx[j].j.W_dev, 16);
  if (swiglu) tma = tma && aligned(W2, 16);
  snprintf(buf, sizeof buf, "%d/%lld/%d/%d/%lld/%lld/%lld", fmt, (long long)cols, int(swiglu), int(tma),
           (long long)jobsx[0].j.rows, (long long)(njobs > 1 ? jobsx[1].j.rows : -1),
           (long long)(njobs > 2 ? jobsx[2].j.rows : -1));
  return buf;
}

// reads a buffer larger than L2, evicting what the previous launch left there
// (reads: no dirty lines to write back during the next timing)
__global__ void l2_flush_kernel(const int4* p, int64_t n, int* sink) {
  int acc = 0;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const int4 v = __ldcg(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x7fffffff && sink) *sink = acc;  // keeps the loads; practically never taken
}

// time the candidate plans of one launch shape on `st` (outputs to scratch,
// plain epilogue, no residual) and remember the fastest: each candidate is
// launched once to warm up, then timed alone 7 times, each time after L2 has
// been flushed (its weights come from HBM as in a decode step); the median
// decides
nt_status tune(Ctx* c, const std::string& key, int fmt, const GemvJobEx* jobsx, int njobs, const void* W2,
               const float* x, const float* norm_g, float eps, int64_t cols, bool swiglu, cudaStream_t st) {
  GemvJobEx tj[3];
  size_t off = 0;
  for (int j = 0; j < njobs; ++j) {
    tj[j] = jobsx[j];
    tj[j].j.y_dev = reinterpret_cast<float*>(c->scratch + kScratchTune + off);
    tj[j].j.residual_dev = nullptr;
    tj[j].epi = kEpiPlain;
    tj[j].cache = nullptr;
    off += (size_t(jobsx[j].j.rows) * 4 + 255) / 256 * 256;
  }
  if (kScratchTune + off > kScratchGemm || kScratchGemm > c->scratch_bytes) {
    const Arith ar = arith_plan(c, fmt, jobsx, njobs, cols, swiglu);
    std::lock_guard<std::mutex> lk(c->mu);  // no room to tune: keep the default
    c->gemv_plans[key] = PlanChoice{c->gemv_warps, c->gemv_stage_max, ar.ks, ar.R};
    return NT_OK;
  }
  const PlanChoice cands[] = {{c->gemv_warps, c->gemv_stage_max, 0}, {12, 16384, 0}, {8, 24576, 0}, {12, 12288, 0},
                              {16, 16384, 0}, {8, 16384, 0}, {16, 8192, 0}};
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t ce = cudaEventCreate(&e0);
  if (ce == cudaSuccess) ce = cudaEventCreate(&e1);
  if (ce == cudaSuccess && !c->flush) {
    int l2 = 0;
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, c->device);
    const size_t fb = (size_t(l2 > 0 ? l2 : (128 << 20)) * 5 / 4 + 4095) / 4096 * 4096;
    if (cudaMalloc(&c->flush, fb) == cudaSuccess) {
      c->flush_bytes = fb;
      ce = cudaMemsetAsync(c->flush, 0, fb, st);
    } else {
      cudaGetLastError();
      c->flush = nullptr;  // no room: time without flushing
    }
  }
  auto flush_l2 = [&]() -> cudaError_t {
    if (!c->flush) return cudaSuccess;
    l2_flush_kernel<<<c->num_sms * 4, 256, 0, st>>>(reinterpret_cast<const int4*>(c->flush),
                                                     int64_t(c->flush_bytes / 16), nullptr);
    return cudaGetLastError();
  };
  float best_ms = 1e30f;
  PlanChoice best = cands[0];
  std::vector<std::string> seen;
  for (const PlanChoice& pc : cands) {
    if (ce != cudaSuccess) break;
    if (pc.warps > 16 || pc.warps < 4) continue;
    Plan P;
    if (!make_plan(c, fmt, tj, njobs, W2, x, norm_g, eps, cols, swiglu, nullptr, pc, P)) continue;
    char sig[96];
    snprintf(sig, sizeof sig, "%d/%d/%d/%d/%d/%d", P.R, P.warps, P.a.seg, P.a.ks, P.a.stb, P.a.nst);
    if (std::find(seen.begin(), seen.end(), std::string(sig)) != seen.end()) continue;
    seen.push_back(sig);
    if (ce == cudaSuccess) ce = launch_plan(c, fmt, P, st);  // warm-up
    float t[7];
    for (int r = 0; r < 7 && ce == cudaSuccess; ++r) {
      ce = flush_l2();
      if (ce == cudaSuccess) ce = cudaEventRecord(e0, st);
      if (ce == cudaSuccess) ce = launch_plan(c, fmt, P, st);
      if (ce == cudaSuccess) ce = cudaEventRecord(e1, st);
      if (ce == cudaSuccess) ce = cudaEventSynchronize(e1);
      if (ce == cudaSuccess) ce = cudaEventElapsedTime(&t[r], e0, e1);
    }
    if (ce != cudaSuccess) break;
    std::sort(t, t + 7);
    const float ms = t[3];
    if (ms < best_ms) {
      best_ms = ms;
      best = pc;
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (ce != cudaSuccess) return cuda_check(c, ce, "gemv plan tuning");
  const Arith ar = arith_plan(c, fmt, jobsx, njobs, cols, swiglu);
  best.R = ar.R;
  best.ks = ar.ks;
  std::lock_guard<std::mutex> lk(c->mu);
  c->gemv_plans[key] = best;
  return NT_OK;
}

}  // namespace

nt_status launch_gemv_ex(Ctx* c, int fmt, const GemvJobEx* jobsx, int njobs, const void* W2, const float* x,
                         const float* norm_g, float eps, int64_t cols, bool swiglu, const RopeArgs* rope,
                         cudaStream_t st) {
  int64_t rows = 0;
  for (int j = 0; j < njobs; ++j) rows += jobsx[j].j.rows;
  if (rows == 0) return NT_OK;
  const std::string key = plan_key(fmt, jobsx, njobs, W2, cols, swiglu);
  PlanChoice pc{c->gemv_warps, c->gemv_stage_max, 0};
  bool known = false;
  {
    std::lock_guard<std::mutex> lk(c->mu);
    auto it = c->gemv_plans.find(key);
    if (it != c->gemv_plans.end()) {
      pc = it->second;
      known = true;
    }
  }
  if (!known && c->gemv_tune) {
    // tune on the first eager call of a shape (never inside a stream capture)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone) {
      nt_status s = tune(c, key, fmt, jobsx, njobs, W2, x, norm_g, eps, cols, swiglu, st);
      if (s) return s;
      std::lock_guard<std::mutex> lk(c->mu);
      pc = c->gemv_plans[key];
    }
    cudaGetLastError();
  }
  if (!known && !c->gemv_tune) {
    const Arith ar = arith_plan(c, fmt, jobsx, njobs, cols, swiglu);
    std::lock_guard<std::mutex> lk(c->mu);
    c->gemv_plans[key] = PlanChoice{pc.warps, pc.stage_max, ar.ks, ar.R};
  }
  if (c->dry) return NT_OK;
  // the chosen plan, else fewer warps when x leaves too little shared memory
  Plan P;
  bool ok = make_plan(c, fmt, jobsx, njobs, W2, x, norm_g, eps, cols, swiglu, rope, pc, P);
  for (int nw : {12, 8, 4})
    if (!ok && nw < pc.warps)
      ok = make_plan(c, fmt, jobsx, njobs, W2, x, norm_g, eps, cols, swiglu, rope, PlanChoice{nw, pc.stage_max, 0}, P);
  if (!ok)
    return set_err(c, NT_ERR_INVALID_ARG, "gemv: cols=%lld too large for the shared-memory plan", (long long)cols);
  P.a.stall = P.a.tma && take_stall(st);
  return cuda_check(c, launch_plan(c, fmt, P, st), "qgemv launch");
}

}  // namespace nt
