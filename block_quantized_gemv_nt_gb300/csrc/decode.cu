// decode.cu — the batch-1 decode step of a Llama-architecture model with
// block-quantized weights ("ntransformer - moteur d'inférence NVMe-to-GPU…",
// fr.news.hada.io: "Architecture et structure du code" — model/ transformer
// composition, inference/ engine and sampler; "Fonctionnalités principales" —
// RoPE, GQA, SwiGLU, RMSNorm, KV cache), and layer-skip calibration by cosine
// similarity ("Performances et structure de cache").
//
// GB300 shape of the step: per layer four quant-GEMV launches (Q/K/V with the
// attention RMSNorm fused in front and RoPE plus the f16 KV append fused
// behind; a second launch for V when its format differs, as in Q4_K_M; O with
// the residual add; gate/up with the FFN RMSNorm in front and SwiGLU behind;
// down with the residual add) and one split attention kernel; then the LM
// head (final RMSNorm fused) and the argmax, which also advances the
// device-side (token, pos) state.  The whole sequence is captured once into a CUDA graph
// per skip mask and replayed, so a token costs one graph launch and no host
// round trip.
#include <algorithm>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "nt_internal.cuh"
#include "ops.cuh"

struct nt_model {
  nt_model_desc d{};
  std::vector<nt_layer_ptrs> layers;
  const void* embd = nullptr;
  const void* out = nullptr;
  const float* out_norm = nullptr;
  char* buf = nullptr;           // one device allocation for everything below
  float *x = nullptr, *q = nullptr, *k = nullptr, *v = nullptr, *ao = nullptr, *h = nullptr, *xin = nullptr;
  float* cos = nullptr;
  double* inv_freq = nullptr;    // RoPE frequencies theta^(-2i/head_dim), fp64
  int32_t* tok = nullptr;        // device step state
  int64_t* pos = nullptr;
  unsigned long long* amax_key = nullptr;
  unsigned* amax_cnt = nullptr;
  float* attn_part = nullptr;
  unsigned* attn_cnt = nullptr;
  int S = 0;
  cudaStream_t cap = nullptr;
  std::map<std::string, cudaGraphExec_t> graphs;
};

namespace nt {
namespace {

__global__ void set_state_kernel(int32_t* tok, int64_t* pos, int32_t t, int64_t p) {
  pdl_wait();
  *tok = t;
  *pos = p;
}

size_t up256(size_t n) { return (n + 255) / 256 * 256; }

struct Launch {
  Ctx* c;
  nt_model* m;
  cudaStream_t st;
};

// all kernels of one decode step, enqueued on st
nt_status enqueue_step(Ctx* c, nt_model* m, const uint8_t* skip, float* logits, int32_t* next_tok, cudaStream_t st,
                       bool want_cos) {
  const nt_model_desc& d = m->d;
  const int hd = d.head_dim;
  const int64_t nq = int64_t(d.n_qh) * hd, nkv = int64_t(d.n_kvh) * hd;
  nt_status s = launch_embed(c, d.fmt_embd, m->embd, d.d_model, m->tok, m->x, st);
  if (s) return s;
  for (int l = 0; l < d.n_layers; ++l) {
    if (skip && skip[l]) continue;
    const nt_layer_ptrs& L = m->layers[l];
    if (want_cos) {
      s = cuda_check(c, cudaMemcpyAsync(m->xin, m->x, sizeof(float) * d.d_model, cudaMemcpyDeviceToDevice, st),
                     "copy x");
      if (s) return s;
    }
    // Q, K, V: one launch per distinct format; attention RMSNorm fused in
    // front, RoPE and the f16 KV append fused behind
    {
      const RopeArgs ra{m->pos, m->inv_freq, hd, d.kv_cap};
      const GemvJobEx J[3] = {GemvJobEx{nt_gemv_job{L.wq, m->q, nullptr, nq}, kEpiRope, nullptr},
                              GemvJobEx{nt_gemv_job{L.wk, nullptr, nullptr, nkv}, kEpiRopeCache, L.kcache},
                              GemvJobEx{nt_gemv_job{L.wv, nullptr, nullptr, nkv}, kEpiCache, L.vcache}};
      const int F[3] = {d.fmt_q, d.fmt_k, d.fmt_v};
      bool done[3] = {false, false, false};
      for (int i = 0; i < 3; ++i) {
        if (done[i]) continue;
        GemvJobEx jobs[3];
        int nj = 0;
        for (int j = i; j < 3; ++j)
          if (!done[j] && F[j] == F[i]) {
            jobs[nj++] = J[j];
            done[j] = true;
          }
        s = launch_gemv_ex(c, F[i], jobs, nj, nullptr, m->x, L.attn_norm, d.eps, d.d_model, false, &ra, st);
        if (s) return s;
      }
    }
    s = launch_attn(c, m->q, L.kcache, L.vcache, m->ao, d.n_qh, d.n_kvh, 0, m->pos, d.kv_cap, m->attn_part,
                    m->attn_cnt, m->S, st);
    if (s) return s;
    {
      nt_gemv_job j{L.wo, m->x, m->x, d.d_model};
      s = launch_gemv(c, d.fmt_o, &j, 1, nullptr, m->ao, nullptr, 0.f, nq, false, st);
      if (s) return s;
    }
    {
      nt_gemv_job j{L.wg, m->h, nullptr, d.ffn};
      s = launch_gemv(c, d.fmt_gate, &j, 1, L.wu, m->x, L.ffn_norm, d.eps, d.d_model, true, st);
      if (s) return s;
    }
    {
      nt_gemv_job j{L.wd, m->x, m->x, d.d_model};
      s = launch_gemv(c, d.fmt_down, &j, 1, nullptr, m->h, nullptr, 0.f, d.ffn, false, st);
      if (s) return s;
    }
    if (want_cos) {
      s = launch_cos(c, m->xin, m->x, d.d_model, m->cos + l, st);
      if (s) return s;
    }
  }
  {
    nt_gemv_job j{m->out, logits, nullptr, d.vocab};
    s = launch_gemv(c, d.fmt_out, &j, 1, nullptr, m->x, m->out_norm, d.eps, d.d_model, false, st);
    if (s) return s;
  }
  return launch_argmax(c, logits, d.vocab, next_tok, m->amax_key, m->amax_cnt, st, m->tok, m->pos);
}

std::string graph_key(const nt_model* m, const uint8_t* skip, const float* logits, const int32_t* next_tok) {
  std::string k(reinterpret_cast<const char*>(&logits), sizeof logits);
  k.append(reinterpret_cast<const char*>(&next_tok), sizeof next_tok);
  for (int l = 0; l < m->d.n_layers; ++l) k.push_back(skip && skip[l] ? '1' : '0');
  return k;
}

}  // namespace
}  // namespace nt

using namespace nt;

#define NT_REQUIRE(cond, code, ...)                         \
  do {                                                      \
    if (!(cond)) return set_err(ctx, code, __VA_ARGS__);    \
  } while (0)

extern "C" {

nt_status nt_model_init(nt_ctx* ctx, const nt_model_desc* desc, const nt_layer_ptrs* layers, const void* embd,
                        const void* out, const float* out_norm, nt_model** res) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(desc && layers && embd && out && out_norm && res, NT_ERR_INVALID_ARG, "null pointer");
  const nt_model_desc& d = *desc;
  NT_REQUIRE(d.n_layers > 0 && d.d_model > 0 && d.ffn > 0 && d.vocab > 0, NT_ERR_INVALID_ARG, "bad dims");
  NT_REQUIRE(d.head_dim == 128, NT_ERR_INVALID_ARG, "head_dim must be 128");
  NT_REQUIRE(d.n_kvh > 0 && d.n_qh % d.n_kvh == 0 && d.n_kvh <= 64, NT_ERR_INVALID_ARG, "bad head counts");
  {
    const int grp = d.n_qh / d.n_kvh;
    NT_REQUIRE(grp == 1 || grp == 2 || grp == 4 || grp == 8 || grp == 16, NT_ERR_INVALID_ARG,
               "n_qh / n_kvh must be 1, 2, 4, 8 or 16");
  }
  NT_REQUIRE(d.kv_cap > 0 && d.eps >= 0.f && d.theta > 0.f, NT_ERR_INVALID_ARG, "bad kv_cap/eps/theta");
  NT_REQUIRE(d.kv_cap <= attn_max_stride(), NT_ERR_INVALID_ARG, "kv_cap above %lld", (long long)attn_max_stride());
  const int fm[9] = {d.fmt_q, d.fmt_k, d.fmt_v, d.fmt_o, d.fmt_gate, d.fmt_up, d.fmt_down, d.fmt_embd, d.fmt_out};
  for (int f : fm) NT_REQUIRE(fmt_ok(f), NT_ERR_UNSUPPORTED_FMT, "unknown format id %d", f);
  NT_REQUIRE(d.fmt_gate == d.fmt_up, NT_ERR_INVALID_ARG, "gate and up must share a format");
  const int64_t nq = int64_t(d.n_qh) * d.head_dim;
  NT_REQUIRE(d.d_model % block_elems(d.fmt_q) == 0 && d.d_model % block_elems(d.fmt_k) == 0 &&
                 d.d_model % block_elems(d.fmt_v) == 0 && d.d_model % block_elems(d.fmt_gate) == 0 &&
                 d.d_model % block_elems(d.fmt_embd) == 0 && d.d_model % block_elems(d.fmt_out) == 0 &&
                 nq % block_elems(d.fmt_o) == 0 && d.ffn % block_elems(d.fmt_down) == 0,
             NT_ERR_INVALID_ARG, "a matrix width is not a multiple of its block size");
  for (int l = 0; l < d.n_layers; ++l) {
    const nt_layer_ptrs& L = layers[l];
    NT_REQUIRE(L.attn_norm && L.ffn_norm && L.kcache && L.vcache, NT_ERR_INVALID_ARG, "layer %d: null norm/cache", l);
    NT_REQUIRE(aligned(L.kcache, 16) && aligned(L.vcache, 16) && aligned(L.attn_norm, 16) && aligned(L.ffn_norm, 16),
               NT_ERR_ALIGNMENT, "layer %d: caches and norms must be 16-byte aligned", l);
  }
  NT_REQUIRE(aligned(out_norm, 16), NT_ERR_ALIGNMENT, "out_norm must be 16-byte aligned");

  nt_model* m = new (std::nothrow) nt_model();
  if (!m) return NT_ERR_OOM;
  m->d = d;
  m->layers.assign(layers, layers + d.n_layers);
  m->embd = embd;
  m->out = out;
  m->out_norm = out_norm;
  m->S = attn_splits(ctx, d.n_kvh, d.kv_cap);
  const size_t fl = sizeof(float);
  const size_t nx = up256(fl * d.d_model), nqb = up256(fl * nq), nkb = up256(fl * d.n_kvh * d.head_dim),
               nh = up256(fl * d.ffn), ncos = up256(fl * d.n_layers), nst = 256, nfreq = up256(8 * d.head_dim),
               npart = up256(attn_scratch_bytes(d.n_qh, d.n_kvh, m->S));
  const size_t total = 2 * nx + nqb * 2 + nkb * 2 + nh + ncos + nst + npart + nfreq;
  int dev_prev = 0;
  cudaGetDevice(&dev_prev);
  cudaSetDevice(ctx->device);
  cudaError_t e = cudaMalloc(&m->buf, total);
  if (e == cudaSuccess) e = cudaMemset(m->buf, 0, total);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&m->cap, cudaStreamNonBlocking);
  cudaSetDevice(dev_prev);
  if (e != cudaSuccess) {
    if (m->buf) cudaFree(m->buf);
    delete m;
    return cuda_check(ctx, e, "model allocation");
  }
  char* p = m->buf;
  auto take = [&](size_t n) {
    char* r = p;
    p += n;
    return r;
  };
  m->x = reinterpret_cast<float*>(take(nx));
  m->xin = reinterpret_cast<float*>(take(nx));
  m->q = reinterpret_cast<float*>(take(nqb));
  m->ao = reinterpret_cast<float*>(take(nqb));
  m->k = reinterpret_cast<float*>(take(nkb));
  m->v = reinterpret_cast<float*>(take(nkb));
  m->h = reinterpret_cast<float*>(take(nh));
  m->cos = reinterpret_cast<float*>(take(ncos));
  char* stt = take(nst);
  m->tok = reinterpret_cast<int32_t*>(stt);
  m->pos = reinterpret_cast<int64_t*>(stt + 8);
  m->amax_key = reinterpret_cast<unsigned long long*>(stt + 16);
  m->amax_cnt = reinterpret_cast<unsigned*>(stt + 24);
  m->inv_freq = reinterpret_cast<double*>(take(nfreq));
  char* part = take(npart);
  m->attn_cnt = reinterpret_cast<unsigned*>(part);
  m->attn_part = reinterpret_cast<float*>(part + 64 * sizeof(unsigned));
  cudaSetDevice(ctx->device);
  nt_status st = launch_inv_freq(ctx, m->inv_freq, d.head_dim, d.theta, nullptr);
  if (!st) st = cuda_check(ctx, cudaDeviceSynchronize(), "model init");
  cudaSetDevice(dev_prev);
  if (st) {
    nt_model_destroy(ctx, m);
    return st;
  }
  *res = m;
  return NT_OK;
}

nt_status nt_model_destroy(nt_ctx* ctx, nt_model* m) {
  if (!ctx || !m) return NT_ERR_INVALID_ARG;
  int dev_prev = 0;
  cudaGetDevice(&dev_prev);
  cudaSetDevice(ctx->device);
  cudaDeviceSynchronize();
  for (auto& kv : m->graphs) cudaGraphExecDestroy(kv.second);
  if (m->cap) cudaStreamDestroy(m->cap);
  cudaFree(m->buf);
  cudaSetDevice(dev_prev);
  delete m;
  return NT_OK;
}

nt_status nt_decode_step(nt_ctx* ctx, nt_model* m, int32_t token, int64_t pos, const uint8_t* skip, float* logits,
                         int32_t* next_tok, void* stream) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m && logits, NT_ERR_INVALID_ARG, "null model or logits");
  NT_REQUIRE(aligned(logits, 16), NT_ERR_ALIGNMENT, "logits must be 16-byte aligned");
  if (token >= 0) {
    NT_REQUIRE(token < m->d.vocab, NT_ERR_INVALID_ARG, "token %d outside the vocabulary", token);
    NT_REQUIRE(pos >= 0 && pos < m->d.kv_cap, NT_ERR_INVALID_ARG, "pos %lld outside the KV cache",
               (long long)pos);
  }
  for (int l = 0; l < m->d.n_layers; ++l) {
    if (skip && skip[l]) continue;
    const nt_layer_ptrs& L = m->layers[l];
    NT_REQUIRE(L.wq && L.wk && L.wv && L.wo && L.wg && L.wu && L.wd, NT_ERR_INVALID_ARG,
               "layer %d has no weights bound", l);
  }
  int dev_prev = 0;
  cudaGetDevice(&dev_prev);
  if (dev_prev != ctx->device) cudaSetDevice(ctx->device);
  cudaStream_t st = as_stream(stream);
  nt_status s = NT_OK;
  if (token >= 0) {
    set_state_kernel<<<1, 1, 0, st>>>(m->tok, m->pos, token, pos);
    s = cuda_check(ctx, cudaGetLastError(), "set step state");
  }
  if (!s) {
    const std::string key = graph_key(m, skip, logits, next_tok);
    auto it = m->graphs.find(key);
    if (it == m->graphs.end()) {
      cudaGraph_t g = nullptr;
      cudaGraphExec_t ge = nullptr;
      s = cuda_check(ctx, cudaStreamBeginCapture(m->cap, cudaStreamCaptureModeThreadLocal), "begin capture");
      if (!s) {
        nt_status s2 = enqueue_step(ctx, m, skip, logits, next_tok, m->cap, false);
        cudaError_t e = cudaStreamEndCapture(m->cap, &g);
        s = s2 ? s2 : cuda_check(ctx, e, "end capture");
      }
      if (!s) s = cuda_check(ctx, cudaGraphInstantiate(&ge, g, 0), "graph instantiate");
      if (g) cudaGraphDestroy(g);
      if (!s) it = m->graphs.emplace(key, ge).first;
    }
    if (!s) s = cuda_check(ctx, cudaGraphLaunch(it->second, st), "graph launch");
  }
  if (dev_prev != ctx->device) cudaSetDevice(dev_prev);
  return s;
}

nt_status nt_layer_skip_calibrate(nt_ctx* ctx, nt_model* m, int32_t token, int64_t pos, int n_skip, uint8_t* mask,
                                  float* cos_host, float* logits, int32_t* next_tok, void* stream) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m && mask && logits, NT_ERR_INVALID_ARG, "null pointer");
  NT_REQUIRE(n_skip >= 0 && n_skip <= m->d.n_layers, NT_ERR_INVALID_ARG, "n_skip outside 0..n_layers");
  NT_REQUIRE(token >= 0 && token < m->d.vocab && pos >= 0 && pos < m->d.kv_cap, NT_ERR_INVALID_ARG,
             "bad token/pos");
  int dev_prev = 0;
  cudaGetDevice(&dev_prev);
  if (dev_prev != ctx->device) cudaSetDevice(ctx->device);
  cudaStream_t st = as_stream(stream);
  std::vector<float> cs(m->d.n_layers, 0.f);
  set_state_kernel<<<1, 1, 0, st>>>(m->tok, m->pos, token, pos);
  nt_status s = cuda_check(ctx, cudaGetLastError(), "set step state");
  if (!s) s = enqueue_step(ctx, m, nullptr, logits, next_tok, st, true);
  if (!s)
    s = cuda_check(ctx, cudaMemcpyAsync(cs.data(), m->cos, sizeof(float) * cs.size(), cudaMemcpyDeviceToHost, st),
                   "read cosines");
  if (!s) s = cuda_check(ctx, cudaStreamSynchronize(st), "calibration sync");
  if (dev_prev != ctx->device) cudaSetDevice(dev_prev);
  if (s) return s;
  // the n_skip largest cosines, ties to the lower layer index
  std::vector<int> idx(m->d.n_layers);
  for (int l = 0; l < m->d.n_layers; ++l) idx[l] = l;
  std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return cs[a] > cs[b]; });
  std::memset(mask, 0, size_t(m->d.n_layers));
  for (int i = 0; i < n_skip; ++i) mask[idx[i]] = 1;
  if (cos_host) std::memcpy(cos_host, cs.data(), sizeof(float) * cs.size());
  return NT_OK;
}

}  // extern "C"
