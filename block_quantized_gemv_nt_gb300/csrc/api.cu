// api.cu — the extern "C" boundary of libnt.so (declared in include/nt.h):
// context management and argument checking of every single-op entry point.
// Nothing is launched until every check has passed.
#include <cstdlib>
#include <cstring>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <thread>

#include "nt_internal.cuh"
#include "ops.cuh"

namespace nt {

nt_status set_err(Ctx* c, nt_status s, const char* fmt, ...) {
  if (c) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    c->last_error = buf;
  }
  return s;
}

nt_status cuda_check(Ctx* c, cudaError_t e, const char* what) {
  if (e == cudaSuccess) return NT_OK;
  return set_err(c, e == cudaErrorMemoryAllocation ? NT_ERR_OOM : NT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// failures of nt_ctx_create have no context to hold their message
thread_local std::string g_create_error;

// launches still to be armed by nt_debug_stall_waits (process-wide)
std::atomic<int> g_stall_waits{0};

bool take_stall(cudaStream_t st) {
  if (g_stall_waits.load(std::memory_order_relaxed) <= 0) return false;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return false;  // a captured launch would stall at every replay
  }
  int n = g_stall_waits.load();
  while (n > 0 && !g_stall_waits.compare_exchange_weak(n, n - 1)) {
  }
  return n > 0;
}

}  // namespace nt

using namespace nt;

namespace {

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    cudaGetDevice(&cur);
    if (prev >= 0 && cur != prev) cudaSetDevice(prev);
  }
};

#define NT_REQUIRE(cond, code, ...)                         \
  do {                                                      \
    if (!(cond)) return set_err(ctx, code, __VA_ARGS__);    \
  } while (0)

nt_status check_fmt_cols(nt_ctx* ctx, int fmt, int64_t cols) {
  NT_REQUIRE(fmt_ok(fmt), NT_ERR_UNSUPPORTED_FMT, "unknown format id %d", fmt);
  NT_REQUIRE(cols > 0 && cols % block_elems(fmt) == 0, NT_ERR_INVALID_ARG,
             "cols=%lld is not a positive multiple of the block size %d", (long long)cols, block_elems(fmt));
  NT_REQUIRE(cols <= (int64_t(1) << 30), NT_ERR_INVALID_ARG, "cols=%lld too large", (long long)cols);
  return NT_OK;
}

nt_status check_vec(nt_ctx* ctx, const void* p, const char* name) {
  NT_REQUIRE(p != nullptr, NT_ERR_INVALID_ARG, "%s is NULL", name);
  NT_REQUIRE(aligned(p, 16), NT_ERR_ALIGNMENT, "%s must be 16-byte aligned", name);
  return NT_OK;
}

// every entry point's first check: a context is required (device error flags
// are read by nt_ctx_sync / nt_stream_sync, after the work that sets them)
nt_status pre_call(nt_ctx* ctx) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  return NT_OK;
}

}  // namespace

#define NT_TRY(expr)                  \
  do {                                \
    nt_status s_ = (expr);            \
    if (s_ != NT_OK) return s_;       \
  } while (0)

extern "C" {

int nt_block_bytes(int fmt) { return fmt_ok(fmt) ? block_bytes(fmt) : 0; }
int nt_block_elems(int fmt) { return fmt_ok(fmt) ? block_elems(fmt) : 0; }

nt_status nt_ctx_create(nt_ctx** out, int device, size_t scratch_bytes) {
  if (!out) return NT_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  cudaError_t ce = cudaGetDeviceCount(&ndev);
  if (ce != cudaSuccess || device < 0 || device >= ndev) {
    g_create_error = ce != cudaSuccess ? std::string("cudaGetDeviceCount: ") + cudaGetErrorString(ce)
                                       : "device " + std::to_string(device) + " not present";
    cudaGetLastError();
    return NT_ERR_CUDA;
  }
  DeviceGuard g(device);
  nt_ctx* c = new (std::nothrow) nt_ctx();
  if (!c) return NT_ERR_OOM;
  c->device = device;
  int v = 0;
  cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device);
  c->num_sms = v;
  cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  c->smem_optin = size_t(v);
  auto env_int = [](const char* name, int lo, int hi, int dflt) {
    const char* v = getenv(name);
    if (!v) return dflt;
    const int x = atoi(v);
    return (x >= lo && x <= hi) ? x : dflt;
  };
  c->gemv_warps = env_int("NT_GEMV_WARPS", 4, 16, 16);
  c->gemv_stages = env_int("NT_GEMV_STAGES", 2, 8, 2);
  c->gemv_stage_max = env_int("NT_GEMV_STAGE_MAX", 1024, 65536, 12288) / 16 * 16;
  c->pdl = env_int("NT_PDL", 0, 1, 1) != 0;
  // timing candidate launch shapes picks the fastest alone, which is not
  // always the fastest inside a decode step: off unless asked for
  c->gemv_tune = env_int("NT_GEMV_TUNE", 0, 1, 0) != 0;
  c->attn_fill = env_int("NT_ATTN_FILL", 0, 1, 1) != 0;
  c->gemm_mma = env_int("NT_GEMM_MMA", 0, 1, 1) != 0;
  c->gemm_warps = env_int("NT_GEMM_WARPS", 8, 12, 12) / 4 * 4;
  c->gemm_stages = env_int("NT_GEMM_STAGES", 2, 8, 4);
  c->scratch_bytes = scratch_bytes ? scratch_bytes : (size_t(64) << 20);
  if (c->scratch_bytes < (size_t(1) << 20)) c->scratch_bytes = size_t(1) << 20;
  if (cudaMalloc(&c->scratch, c->scratch_bytes) != cudaSuccess) {
    cudaGetLastError();
    g_create_error = "scratch allocation failed";
    delete c;
    return NT_ERR_OOM;
  }
  if (cudaMemset(c->scratch, 0, c->scratch_bytes) != cudaSuccess) {
    g_create_error = "scratch memset failed";
    cudaFree(c->scratch);
    delete c;
    return NT_ERR_CUDA;
  }
  c->err_flag = reinterpret_cast<unsigned*>(c->scratch + kScratchErr);
  if (configure_gemv(c) != NT_OK || configure_ops(c) != NT_OK || configure_gemm(c) != NT_OK) {
    g_create_error = c->last_error;
    cudaFree(c->scratch);
    delete c;
    return NT_ERR_CUDA;
  }
  *out = c;
  return NT_OK;
}

nt_status nt_ctx_destroy(nt_ctx* ctx) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  {
    DeviceGuard g(ctx->device);
    cudaDeviceSynchronize();
    cudaFree(ctx->scratch);
    if (ctx->flush) cudaFree(ctx->flush);
  }
  delete ctx;
  return NT_OK;
}

// the device error flag, read and cleared after the work that may set it has finished
static nt_status take_device_flag(nt_ctx* ctx) {
  unsigned flag = 0;
  cudaError_t e = cudaMemcpy(&flag, ctx->err_flag, sizeof flag, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_check(ctx, e, "read device error flag");
  if (flag) {
    cudaMemset(ctx->err_flag, 0, sizeof(unsigned));
    if (flag & kErrWaitTimeout)
      return set_err(ctx, NT_ERR_TIMEOUT, "a device-side bounded wait ran out (flag 0x%x)", flag);
    return set_err(ctx, NT_ERR_INVALID_ARG, "a device-side position ran past the KV cache (flag 0x%x)", flag);
  }
  return NT_OK;
}

nt_status nt_ctx_sync(nt_ctx* ctx) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_check(ctx, e, "device synchronize");
  return take_device_flag(ctx);
}

nt_status nt_stream_sync(nt_ctx* ctx, void* stream, int64_t timeout_us) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(timeout_us >= 0, NT_ERR_INVALID_ARG, "negative timeout");
  DeviceGuard g(ctx->device);
  const cudaStream_t st = as_stream(stream);
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t e = cudaStreamQuery(st);
    if (e == cudaSuccess) break;
    if (e != cudaErrorNotReady) return cuda_check(ctx, e, "stream query");
    const auto us = std::chrono::duration_cast<std::chrono::microseconds>(std::chrono::steady_clock::now() - t0);
    if (us.count() >= timeout_us) {
      cudaGetLastError();
      return set_err(ctx, NT_ERR_TIMEOUT, "stream still busy after %lld us", (long long)timeout_us);
    }
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  return take_device_flag(ctx);
}

nt_status nt_debug_fail_copy(nt_ctx* ctx, int nth) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(nth >= -1, NT_ERR_INVALID_ARG, "nth must be -1 (off) or >= 0");
  ctx->copy_fail_in = nth;
  return NT_OK;
}

nt_status nt_debug_stall_waits(int n) {
  if (n < 0 || n > 1000) return NT_ERR_INVALID_ARG;
  g_stall_waits.store(n);
  return NT_OK;
}

static void CUDART_CB host_delay_fn(void* us) {
  std::this_thread::sleep_for(std::chrono::microseconds(reinterpret_cast<intptr_t>(us)));
}

nt_status nt_debug_host_delay(nt_ctx* ctx, void* stream, int64_t us) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(us >= 0 && us <= 10000000, NT_ERR_INVALID_ARG, "delay outside 0..10 s");
  DeviceGuard g(ctx->device);
  return cuda_check(ctx, cudaLaunchHostFunc(as_stream(stream), host_delay_fn, reinterpret_cast<void*>(intptr_t(us))),
                    "host delay");
}

nt_status nt_ctx_gemv_plans(nt_ctx* ctx, char* out, size_t cap, size_t* len) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(len && (out || cap == 0), NT_ERR_INVALID_ARG, "null length or buffer");
  std::string text;
  {
    std::lock_guard<std::mutex> lk(ctx->mu);
    for (const auto& kv : ctx->gemv_plans) {
      // key: fmt/cols/swiglu/tma/rows0/rows1/rows2
      char line[256];
      snprintf(line, sizeof line, "%s -> warps=%d stage_max=%d R=%d ks=%d\n", kv.first.c_str(), kv.second.warps,
               kv.second.stage_max, kv.second.R, kv.second.ks);
      text += line;
    }
  }
  *len = text.size() + 1;
  if (cap) {
    const size_t n = std::min(cap - 1, text.size());
    std::memcpy(out, text.data(), n);
    out[n] = 0;
  }
  return NT_OK;
}

const char* nt_last_error(const nt_ctx* ctx) { return ctx ? ctx->last_error.c_str() : g_create_error.c_str(); }

nt_status nt_dequant_rows(nt_ctx* ctx, int fmt, const void* W, int64_t row0, int64_t nrows, int64_t cols,
                          float* out, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_TRY(check_fmt_cols(ctx, fmt, cols));
  NT_REQUIRE(W && out, NT_ERR_INVALID_ARG, "null pointer");
  NT_REQUIRE(row0 >= 0 && nrows >= 0, NT_ERR_INVALID_ARG, "negative row range");
  NT_REQUIRE(aligned(W, fmt == NT_F32 ? 4 : 2), NT_ERR_ALIGNMENT, "W must be %d-byte aligned",
             fmt == NT_F32 ? 4 : 2);
  NT_REQUIRE(aligned(out, 4), NT_ERR_ALIGNMENT, "out must be 4-byte aligned");
  DeviceGuard g(ctx->device);
  return launch_dequant(ctx, fmt, W, row0, nrows, cols, out, as_stream(stream));
}

nt_status nt_gemv_q_multi(nt_ctx* ctx, int fmt, const nt_gemv_job* jobs, int njobs, const float* x,
                          const float* norm_g, float eps, int64_t cols, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_TRY(check_fmt_cols(ctx, fmt, cols));
  NT_REQUIRE(jobs && njobs >= 1 && njobs <= 3, NT_ERR_INVALID_ARG, "njobs must be 1..3");
  NT_TRY(check_vec(ctx, x, "x"));
  if (norm_g) NT_TRY(check_vec(ctx, norm_g, "norm_g"));
  for (int j = 0; j < njobs; ++j) {
    NT_REQUIRE(jobs[j].rows >= 0, NT_ERR_INVALID_ARG, "job %d: negative rows", j);
    if (jobs[j].rows == 0) continue;
    NT_REQUIRE(jobs[j].W_dev && jobs[j].y_dev, NT_ERR_INVALID_ARG, "job %d: null W or y", j);
    NT_REQUIRE(aligned(jobs[j].W_dev, 2), NT_ERR_ALIGNMENT, "job %d: W must be 2-byte aligned", j);
    NT_REQUIRE(aligned(jobs[j].y_dev, 4), NT_ERR_ALIGNMENT, "job %d: y must be 4-byte aligned", j);
    NT_REQUIRE(!jobs[j].residual_dev || aligned(jobs[j].residual_dev, 4), NT_ERR_ALIGNMENT,
               "job %d: residual must be 4-byte aligned", j);
  }
  DeviceGuard g(ctx->device);
  return launch_gemv(ctx, fmt, jobs, njobs, nullptr, x, norm_g, eps, cols, false, as_stream(stream));
}

nt_status nt_gemv_q(nt_ctx* ctx, int fmt, const void* W, const float* x, float* y, int64_t rows, int64_t cols,
                    const float* residual, void* stream) {
  NvtxRange nvtx_range("nt_gemv_q");
  nt_gemv_job j{W, y, residual, rows};
  return nt_gemv_q_multi(ctx, fmt, &j, 1, x, nullptr, 0.f, cols, stream);
}

nt_status nt_gemm_q(nt_ctx* ctx, int fmt, const void* W, const float* X, float* Y, int64_t rows, int64_t cols, int M,
                    const float* residual, const float* norm_g, float eps, void* stream) {
  NvtxRange nvtx_range("nt_gemm_q");
  NT_TRY(pre_call(ctx));
  NT_TRY(check_fmt_cols(ctx, fmt, cols));
  NT_REQUIRE(M >= 1 && M <= kMaxGemmM, NT_ERR_INVALID_ARG, "M must be 1..%d", kMaxGemmM);
  NT_REQUIRE(rows >= 0, NT_ERR_INVALID_ARG, "negative rows");
  if (rows == 0) return NT_OK;
  NT_REQUIRE(W && Y, NT_ERR_INVALID_ARG, "null W or Y");
  NT_REQUIRE(aligned(W, 2), NT_ERR_ALIGNMENT, "W must be 2-byte aligned");
  NT_TRY(check_vec(ctx, X, "X"));
  NT_REQUIRE(cols % 4 == 0, NT_ERR_INVALID_ARG, "cols must be a multiple of 4");
  NT_REQUIRE(aligned(Y, 4) && (!residual || aligned(residual, 4)), NT_ERR_ALIGNMENT,
             "Y and residual must be 4-byte aligned");
  if (norm_g) NT_TRY(check_vec(ctx, norm_g, "norm_g"));
  NT_REQUIRE(ctx->scratch_bytes > kScratchGemm, NT_ERR_OOM, "the context scratch has no room for partial sums");
  const GemmJobEx job{W, rows, Y, rows, residual, nullptr, kEpiPlain};
  DeviceGuard g(ctx->device);
  return launch_gemm(ctx, fmt, &job, 1, false, X, cols, M, norm_g, eps, cols, nullptr,
                     reinterpret_cast<float*>(ctx->scratch + kScratchGemm), ctx->scratch_bytes - kScratchGemm,
                     as_stream(stream));
}

nt_status nt_gemv_q_swiglu(nt_ctx* ctx, int fmt, const void* Wg, const void* Wu, const float* x, const float* norm_g,
                           float eps, float* h, int64_t rows, int64_t cols, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_TRY(check_fmt_cols(ctx, fmt, cols));
  NT_TRY(check_vec(ctx, x, "x"));
  if (norm_g) NT_TRY(check_vec(ctx, norm_g, "norm_g"));
  NT_REQUIRE(rows >= 0, NT_ERR_INVALID_ARG, "negative rows");
  if (rows == 0) return NT_OK;
  NT_REQUIRE(Wg && Wu && h, NT_ERR_INVALID_ARG, "null pointer");
  NT_REQUIRE(aligned(Wg, 2) && aligned(Wu, 2), NT_ERR_ALIGNMENT, "weights must be 2-byte aligned");
  NT_REQUIRE(aligned(h, 4), NT_ERR_ALIGNMENT, "h must be 4-byte aligned");
  nt_gemv_job j{Wg, h, nullptr, rows};
  DeviceGuard g(ctx->device);
  return launch_gemv(ctx, fmt, &j, 1, Wu, x, norm_g, eps, cols, true, as_stream(stream));
}

nt_status nt_rmsnorm(nt_ctx* ctx, const float* x, const float* g, float* y, int64_t n, float eps, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(x && g && y && n > 0, NT_ERR_INVALID_ARG, "null pointer or n <= 0");
  NT_REQUIRE(aligned(x, 4) && aligned(g, 4) && aligned(y, 4), NT_ERR_ALIGNMENT, "vectors must be 4-byte aligned");
  NT_REQUIRE(eps >= 0.f, NT_ERR_INVALID_ARG, "eps must be >= 0");
  DeviceGuard gd(ctx->device);
  return launch_rmsnorm(ctx, x, g, y, n, eps, as_stream(stream));
}

nt_status nt_rope(nt_ctx* ctx, float* q, float* k, int n_qh, int n_kvh, int head_dim, int64_t pos, float theta,
                  void* stream) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(q && n_qh > 0 && (!k || n_kvh > 0), NT_ERR_INVALID_ARG, "bad q/k or head counts");
  NT_REQUIRE(head_dim > 0 && head_dim % 2 == 0 && head_dim <= 512, NT_ERR_INVALID_ARG, "head_dim must be even, <= 512");
  NT_REQUIRE(pos >= 0 && theta > 0.f, NT_ERR_INVALID_ARG, "pos must be >= 0 and theta > 0");
  NT_REQUIRE(aligned(q, 4) && aligned(k, 4), NT_ERR_ALIGNMENT, "q and k must be 4-byte aligned");
  DeviceGuard g(ctx->device);
  return launch_rope(ctx, q, k, n_qh, n_kvh, head_dim, pos, theta, as_stream(stream));
}

nt_status nt_rope_kv_append(nt_ctx* ctx, float* q, const float* k, const float* v, void* kc, void* vc, int n_qh,
                            int n_kvh, int head_dim, int64_t pos, int64_t kv_stride, float theta, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(q && k && v && kc && vc, NT_ERR_INVALID_ARG, "null pointer");
  NT_REQUIRE(n_qh > 0 && n_kvh > 0, NT_ERR_INVALID_ARG, "bad head counts");
  NT_REQUIRE(head_dim > 0 && head_dim % 2 == 0 && head_dim <= 512, NT_ERR_INVALID_ARG, "head_dim must be even, <= 512");
  NT_REQUIRE(pos >= 0 && pos < kv_stride, NT_ERR_INVALID_ARG, "pos=%lld outside the cache (stride %lld)",
             (long long)pos, (long long)kv_stride);
  NT_REQUIRE(aligned(kc, 2) && aligned(vc, 2), NT_ERR_ALIGNMENT, "caches must be 2-byte aligned");
  NT_REQUIRE(aligned(q, 4) && aligned(k, 4) && aligned(v, 4), NT_ERR_ALIGNMENT, "q, k and v must be 4-byte aligned");
  DeviceGuard g(ctx->device);
  return launch_rope_append(ctx, q, k, v, kc, vc, n_qh, n_kvh, head_dim, pos, nullptr, kv_stride, theta,
                            as_stream(stream));
}

namespace {
nt_status attn_entry(nt_ctx* ctx, const float* q, const void* kc, const void* vc, float* out, int n_qh, int n_kvh,
                     int head_dim, int64_t n_pos, int nq, int64_t kv_stride, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(q && kc && vc && out, NT_ERR_INVALID_ARG, "null pointer");
  NT_REQUIRE(nq >= 1 && nq <= kMaxVerify, NT_ERR_INVALID_ARG, "n_query must be 1..%d", kMaxVerify);
  NT_REQUIRE(head_dim == 128, NT_ERR_INVALID_ARG, "head_dim must be 128");
  NT_REQUIRE(n_kvh > 0 && n_qh > 0 && n_qh % n_kvh == 0 && n_kvh <= 64, NT_ERR_INVALID_ARG,
             "n_qh must be a multiple of n_kvh, n_kvh <= 64");
  {
    const int grp = n_qh / n_kvh;
    NT_REQUIRE(grp == 1 || grp == 2 || grp == 4 || grp == 8 || grp == 16, NT_ERR_INVALID_ARG,
               "n_qh / n_kvh must be 1, 2, 4, 8 or 16");
  }
  NT_REQUIRE(n_pos >= 1 && n_pos + nq - 1 <= kv_stride, NT_ERR_INVALID_ARG,
             "need 1 <= n_pos and n_pos + n_query - 1 <= kv_stride");
  NT_REQUIRE(kv_stride <= attn_max_stride(), NT_ERR_INVALID_ARG, "kv_stride above %lld", (long long)attn_max_stride());
  NT_TRY(check_vec(ctx, q, "q"));
  NT_TRY(check_vec(ctx, out, "out"));
  NT_REQUIRE(aligned(kc, 16) && aligned(vc, 16), NT_ERR_ALIGNMENT, "caches must be 16-byte aligned");
  const int S = attn_splits(ctx, n_kvh, kv_stride);
  const size_t need = attn_scratch_bytes(n_qh, n_kvh, S, nq);
  NT_REQUIRE(kScratchAttn + need <= kScratchSample && kScratchAttn + need <= ctx->scratch_bytes, NT_ERR_OOM,
             "attention needs %zu scratch bytes", need);
  float* part = reinterpret_cast<float*>(ctx->scratch + kScratchAttn + kAttnCounterBytes);
  DeviceGuard g(ctx->device);
  return launch_attn(ctx, q, kc, vc, out, n_qh, n_kvh, n_pos, nullptr, kv_stride, part, S,
                     as_stream(stream), nq);
}
}  // namespace

nt_status nt_attn_decode(nt_ctx* ctx, const float* q, const void* kc, const void* vc, float* out, int n_qh,
                         int n_kvh, int head_dim, int64_t n_pos, int64_t kv_stride, void* stream) {
  NvtxRange nvtx_range("nt_attn_decode");
  return attn_entry(ctx, q, kc, vc, out, n_qh, n_kvh, head_dim, n_pos, 1, kv_stride, stream);
}

nt_status nt_attn_verify(nt_ctx* ctx, const float* q, const void* kc, const void* vc, float* out, int n_qh,
                         int n_kvh, int head_dim, int64_t n_pos0, int n_query, int64_t kv_stride, void* stream) {
  return attn_entry(ctx, q, kc, vc, out, n_qh, n_kvh, head_dim, n_pos0, n_query, kv_stride, stream);
}

nt_status nt_softmax(nt_ctx* ctx, const float* x, float* y, int64_t n, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(x && y && n > 0, NT_ERR_INVALID_ARG, "null pointer or n <= 0");
  NT_REQUIRE(aligned(x, 4) && aligned(y, 4), NT_ERR_ALIGNMENT, "vectors must be 4-byte aligned");
  DeviceGuard g(ctx->device);
  return launch_softmax(ctx, x, y, n, as_stream(stream));
}

nt_status nt_swiglu(nt_ctx* ctx, const float* gate, const float* up, float* h, int64_t n, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(gate && up && h && n >= 0, NT_ERR_INVALID_ARG, "null pointer or n < 0");
  NT_REQUIRE(aligned(gate, 4) && aligned(up, 4) && aligned(h, 4), NT_ERR_ALIGNMENT, "vectors must be 4-byte aligned");
  if (n == 0) return NT_OK;
  DeviceGuard g(ctx->device);
  return launch_swiglu(ctx, gate, up, h, n, as_stream(stream));
}

nt_status nt_argmax(nt_ctx* ctx, const float* v, int64_t n, int32_t* out, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(v && out && n > 0 && n < (int64_t(1) << 31), NT_ERR_INVALID_ARG, "null pointer or bad n");
  auto* key = reinterpret_cast<unsigned long long*>(ctx->scratch + kScratchArgmax);
  auto* counter = reinterpret_cast<unsigned*>(ctx->scratch + kScratchArgmax + 8);
  DeviceGuard g(ctx->device);
  return launch_argmax(ctx, v, n, out, key, counter, as_stream(stream));
}

nt_status nt_sample(nt_ctx* ctx, const float* z, int64_t n, float T, float P, uint64_t seed, uint64_t counter,
                    int32_t* out, void* stream) {
  NvtxRange nvtx_range("nt_sample");
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(z && out && n >= 1 && n <= kSampMaxN, NT_ERR_INVALID_ARG, "null pointer or n outside 1..%lld",
             (long long)kSampMaxN);
  NT_REQUIRE(aligned(z, 4) && aligned(out, 4), NT_ERR_ALIGNMENT, "logits and out must be 4-byte aligned");
  NT_REQUIRE(P > 0.f && P <= 1.f && !(T != T) && T < 3.0e38f, NT_ERR_INVALID_ARG, "top_p in (0, 1], finite temperature");
  NT_REQUIRE(ctx->scratch_bytes >= kScratchSample + kSampRowBytes, NT_ERR_OOM, "the context scratch has no room for the sampler");
  DeviceGuard g(ctx->device);
  return launch_sample(ctx, z, n, 1, T, P, seed, nullptr, int64_t(counter), out, ctx->scratch + kScratchSample,
                       as_stream(stream));
}

nt_status nt_host_register(nt_ctx* ctx, const void* p, size_t bytes, int read_only) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(p && bytes, NT_ERR_INVALID_ARG, "null pointer or zero bytes");
  NT_REQUIRE(aligned(p, 4096) && bytes % 4096 == 0, NT_ERR_ALIGNMENT, "pointer and size must be multiples of 4096");
  DeviceGuard g(ctx->device);
  unsigned flags = cudaHostRegisterPortable | cudaHostRegisterMapped;
  if (read_only) flags |= cudaHostRegisterReadOnly;
  const cudaError_t e = cudaHostRegister(const_cast<void*>(p), bytes, flags);
  if (e != cudaSuccess) cudaGetLastError();  // a refused registration leaves no error behind for later calls
  return cuda_check(ctx, e, "host register");
}

nt_status nt_host_unregister(nt_ctx* ctx, const void* p) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(p, NT_ERR_INVALID_ARG, "null pointer");
  DeviceGuard g(ctx->device);
  const cudaError_t e = cudaHostUnregister(const_cast<void*>(p));
  if (e != cudaSuccess) cudaGetLastError();
  return cuda_check(ctx, e, "host unregister");
}

nt_status nt_cos_sim(nt_ctx* ctx, const float* a, const float* b, int64_t n, float* out, void* stream) {
  NT_TRY(pre_call(ctx));
  NT_REQUIRE(a && b && out && n > 0, NT_ERR_INVALID_ARG, "null pointer or n <= 0");
  NT_REQUIRE(aligned(a, 4) && aligned(b, 4) && aligned(out, 4), NT_ERR_ALIGNMENT, "vectors must be 4-byte aligned");
  DeviceGuard g(ctx->device);
  return launch_cos(ctx, a, b, n, out, as_stream(stream));
}

}  // extern "C"
