// qgemm.cu — the verify GEMM of self-speculative decoding ("ntransformer -
// moteur d'inférence NVMe-to-GPU…" (fr.news.hada.io), "Fonctionnalités
// principales": the VRAM-resident layers draft, the whole model verifies):
// Y[m] = W X[m] for M <= 8 activation vectors, every weight byte read once.
//
// GB300 design.  M = 5 is still far from a tensor-core shape (an MMA tile is
// 64 or 128 rows of one operand), and the block formats carry one scale per
// 16 or 32 weights, so the contraction stays on the integer pipes: the same
// 24-bit fixed-point x planes and dp4a dot products as the M = 1 GEMV, with
// the weights staged once per CTA and reused for all M vectors.
//  * grid (X, P): the columns are cut into P parts (2048 columns; 1024 /
//    512 for F16 / F32) so that M vectors of x fit in shared memory; CTA
//    (x, p) holds part p of every vector and walks row groups of R = 2 rows.
//  * each warp streams its rows' part through a private ring of TMA bulk
//    copies (mbarrier completion, L2 evict-first), as the GEMV does.
//  * partial sums go to scratch [P][M][rows]; a second kernel adds the P
//    parts in a fixed order (results do not depend on scheduling) and
//    applies the epilogue: residual add, SwiGLU, RoPE at position pos + m,
//    or the f16 KV-cache append at pos + m.
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

size_t gemm_scratch_bytes(int fmt, int64_t total_rows, int64_t cols, int M) {
  return size_t(gemm_parts(fmt, cols)) * size_t(M) * size_t(total_rows) * sizeof(float);
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
  c->gemm_static_smem = st;
  return cuda_check(c, e, "gemm shared-memory attribute");
}

nt_status launch_gemm(Ctx* c, int fmt, const GemmJobEx* jobs, int njobs, bool swiglu, const float* X, int64_t ldx,
                      int M, const float* norm_g, float eps, int64_t cols, const RopeArgs* rope, float* part,
                      size_t part_bytes, cudaStream_t st) {
  if (c->dry) return NT_OK;
  if (M < 1 || M > kMaxVerify) return set_err(c, NT_ERR_INVALID_ARG, "gemm: M must be 1..%d", kMaxVerify);
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
  const int cwb = part_cols(fmt) / BE;
  const int nparts = int((nb + cwb - 1) / cwb);
  const size_t need = size_t(nparts) * M * size_t(rb) * sizeof(float);
  if (need > part_bytes)
    return set_err(c, NT_ERR_OOM, "gemm: %zu scratch bytes needed for the partial sums, %zu available", need,
                   part_bytes);
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
  const size_t smem = gemm_smem(fmt, M);
  if (smem + size_t(c->gemm_static_smem) > c->smem_optin)
    return set_err(c, NT_ERR_INVALID_ARG, "gemm: no shared-memory plan for M=%d", M);
  // one CTA per SM in all: the parts side by side
  int gx = (c->num_sms + nparts - 1) / nparts;
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
