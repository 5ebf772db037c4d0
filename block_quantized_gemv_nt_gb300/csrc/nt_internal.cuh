// nt_internal.cuh — shared internals of libnt.so: the context, status
// helpers, and the inline-PTX wrappers for mbarriers and TMA bulk copies.
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "../../include/nt.h"

namespace nt {

constexpr int kMaxSpin = 1 << 16;   // iteration cap of every device-side wait
constexpr int kStallSpin = 8;       // the cap of a launch armed by nt_debug_stall_waits
constexpr unsigned kWaitHintNs = 50000;  // each try_wait may sleep this long (cap ~3 s in all)
constexpr unsigned kErrWaitTimeout = 1u;
constexpr unsigned kErrPosRange = 2u;  // a device-side position fell outside the KV cache: nothing written there

// a GEMV launch configuration: warps per CTA and stage-size cap (what the
// tuner chooses), and, for the record, the shape's arithmetic: column parts
// KS and rows per lane group R (fixed by the shape alone)
struct PlanChoice {
  int warps, stage_max, ks;
  int R = 0;
};

struct Ctx {
  int device = 0;
  int num_sms = 0;
  size_t smem_optin = 0;
  char* scratch = nullptr;      // device scratch owned by the context
  size_t scratch_bytes = 0;
  unsigned* err_flag = nullptr; // device word, set by kernels whose bounded wait ran out
  bool pdl = true;               // launch with programmatic stream serialization
  mutable bool pdl_hold = false; // the next launch waits for everything before it (set after an event wait)
  int copy_fail_in = -1;         // fault injection: the copy_fail_in-th following layer copy fails (-1: none)
  int gemv_warps = 16;           // quant-GEMV launch shape (tuning knobs, env NT_GEMV_*)
  int gemv_stages = 2;
  int gemv_stage_max = 12288;
  int gemv_static_smem = 2048;   // largest static shared memory of the GEMV kernels
  int gemm_static_smem = 1024;   // same for the verify-GEMM kernels
  bool gemm_mma = true;
  int gemm_warps = 12;           // tensor-core verify GEMM: warps per CTA, stages per warp at most
  int gemm_stages = 4;          // verify GEMM: the tensor-core form for Q8_0 / Q4_K / Q6_K
  std::string last_error;
  std::mutex mu;
  bool attn_fill = true;         // attention splits: also one CTA per SM (else by positions only)
  bool gemv_tune = true;         // time candidate plans on a shape's first eager launch
  bool dry = false;              // enqueue nothing: launchers only tune (a dry pass before a capture)
  std::map<std::string, PlanChoice> gemv_plans;  // tuned plan per launch shape
  char* flush = nullptr;         // read before each timed tuning launch so its weights come from HBM
  size_t flush_bytes = 0;
};

// an NVTX range over a host-side call (visible in a profiler timeline; next to
// free when no tool is attached)
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// host-side status helpers ----------------------------------------------------
nt_status set_err(Ctx* c, nt_status s, const char* fmt, ...);
// Test hook (nt_debug_stall_waits): true when the launch about to be made on
// st takes one of the armed stalls (never while st is being captured).  An
// armed launch issues no bulk copies, so its waits run out after kStallSpin
// tries and take the kernel's timeout path.
bool take_stall(cudaStream_t st);
nt_status cuda_check(Ctx* c, cudaError_t e, const char* what);
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// scratch layout (bytes from ctx->scratch) ------------------------------------
constexpr size_t kScratchErr = 0;            // unsigned err flag (also ctx->err_flag)
constexpr size_t kScratchArgmax = 256;       // unsigned long long key + unsigned counter
constexpr size_t kScratchAttn = 4096;        // attention: a reserved head (kAttnCounterBytes), then partials
constexpr size_t kAttnCounterBytes = 2048;
constexpr size_t kScratchSample = size_t(20) << 20;  // sampler state (one row of kSampRowBytes)
constexpr size_t kSampRowBytes = 32768;             // sampler state per logits row
constexpr int64_t kSampMaxN = 256 * 4000;           // longest row the sampler takes
constexpr size_t kScratchTune = size_t(24) << 20;  // GEMV plan tuning outputs (8 MiB)
constexpr size_t kScratchGemm = size_t(32) << 20;  // verify-GEMM partial sums, to the end of the scratch

// format geometry ---------------------------------------------------------------
__host__ __device__ constexpr int block_elems(int fmt) {
  return (fmt == NT_Q4_K || fmt == NT_Q5_K || fmt == NT_Q6_K) ? 256 : 32;
}
__host__ __device__ constexpr int block_bytes(int fmt) {
  return fmt == NT_Q8_0   ? 34
         : fmt == NT_Q4_0 ? 18
         : fmt == NT_Q4_K ? 144
         : fmt == NT_Q5_K ? 176
         : fmt == NT_Q6_K ? 210
         : fmt == NT_F16  ? 64
                          : 128;
}
inline bool fmt_ok(int fmt) { return fmt >= NT_Q8_0 && fmt <= NT_F32; }

// device helpers -----------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Bounded wait on phase `parity` of an mbarrier; false if the cap ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int max_spin = kMaxSpin) {
  for (int i = 0; i < max_spin; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kWaitHintNs)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// TMA bulk copy global -> shared, completion counted on mbarrier `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Programmatic dependent launch: a kernel may start before its predecessor on
// the stream has finished; pdl_wait() blocks until the predecessor grid has
// completed and its writes are visible (a no-op without the launch attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void flag_error(unsigned* err, unsigned code) {
  if (err) atomicOr(err, code);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

// cos and sin of pos * inv_freq: the angle and its reduction modulo 2*pi in
// fp64 (angles reach thousands of radians), the trigonometry in fp32 on
// the reduced angle.
__device__ __forceinline__ void rope_cs(int64_t pos, double inv_freq, float& c, float& s) {
  const double ang = double(pos) * inv_freq;
  const double k = rint(ang * 0.15915494309189533577);    // 1 / (2 pi)
  double r = fma(-k, 6.283185307179586232, ang);          // 2 pi, high part
  r = fma(-k, 2.4492935982947064e-16, r);                 // 2 pi, low part
  sincosf(float(r), &s, &c);
}

__device__ __forceinline__ double rope_inv_freq(int pair, int head_dim, float theta) {
  return pow(double(theta), -2.0 * double(pair) / double(head_dim));
}

// kernel launch with the programmatic-serialization attribute when enabled
template <typename... KArgs, typename... Args>
cudaError_t launch_k(const Ctx* c, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // a launch that follows a cross-stream event wait is not programmatic: its
  // early part (weight prefetch) must not run before the awaited work
  cfg.numAttrs = (c && c->pdl && !c->pdl_hold) ? 1 : 0;
  if (c) c->pdl_hold = false;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch helpers (defined in the op files) -----------------------------------------
// epilogue of one GEMV job
enum Epi : int {
  kEpiPlain = 0,      // y = Wx (+ residual)
  kEpiRope = 1,       // y = rope(Wx) on adjacent row pairs (fp32 q)
  kEpiRopeCache = 2,  // cache[head][pos][d] = f16(rope(Wx))       (k)
  kEpiCache = 3,      // cache[head][pos][d] = f16(Wx)              (v)
};

struct RopeArgs {
  const int64_t* pos_dev;   // device position (decode step state)
  const double* inv_freq;   // [head_dim/2]
  int head_dim;
  int64_t kv_stride;
};

struct GemvJobEx {
  nt_gemv_job j;
  int epi;
  void* cache;  // f16 cache of one layer [n_kvh][kv_stride][head_dim] for kEpi*Cache
};

// one job of the M-vector verify GEMM: Y[m] = W X[m], with the epilogue applied
// per vector m (RoPE and the cache append at position pos + m)
constexpr int kMaxVerify = 8;  // vectors per verify GEMM (draft length + 1)
constexpr int kMaxGemmM = 16;  // vectors per GEMM in the tensor-core form (prompt chunks)
struct GemmJobEx {
  const void* W;
  int64_t rows;
  float* y;            // [M][ldy]
  int64_t ldy;
  const float* res;    // [M][ldy] residual, nullable (kEpiPlain)
  void* cache;         // f16 cache of one layer for kEpi*Cache
  int epi;
};

nt_status launch_gemv(Ctx* c, int fmt, const nt_gemv_job* jobs, int njobs, const void* W2, const float* x,
                      const float* norm_g, float eps, int64_t cols, bool swiglu, cudaStream_t st);
nt_status launch_gemv_ex(Ctx* c, int fmt, const GemvJobEx* jobs, int njobs, const void* W2, const float* x,
                         const float* norm_g, float eps, int64_t cols, bool swiglu, const RopeArgs* rope,
                         cudaStream_t st);

}  // namespace nt

struct nt_ctx : nt::Ctx {};
