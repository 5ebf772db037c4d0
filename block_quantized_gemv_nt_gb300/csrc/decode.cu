// decode.cu — the batch-1 decode step of a Llama-architecture model with
// block-quantized weights ("ntransformer - moteur d'inférence NVMe-to-GPU…",
// fr.news.hada.io: "Architecture et structure du code" — model/ transformer
// composition, inference/ engine and sampler, memory/ layer streaming;
// "Fonctionnalités principales" — RoPE, GQA, SwiGLU, RMSNorm, KV cache, SLEP
// double-buffered streaming, self-speculative decoding), and layer-skip
// calibration by cosine similarity ("Performances et structure de cache").
//
// GB300 shape of the step: per layer four quant-GEMV launches (Q/K/V with the
// attention RMSNorm fused in front and RoPE plus the f16 KV append fused
// behind; a second launch for V when its format differs, as in Q4_K_M; O with
// the residual add; gate/up with the FFN RMSNorm in front and SwiGLU behind;
// down with the residual add) and one split attention kernel; then the LM
// head (final RMSNorm fused) and the argmax, which also advances the
// device-side (token, pos) state.  The whole sequence is captured once into
// a CUDA graph per skip mask and replayed, so a token costs one graph launch
// and no host round trip.
//
// Streamed layers (weights in page-locked host memory) are copied into HBM
// slots on a side stream inside the same graph, each copy overlapping the
// compute of earlier layers.  The self-speculative step drafts k tokens with
// the first layers, then verifies the k + 1 tokens in one pass of all layers
// (M = k + 1 GEMMs, causal multi-query attention) and keeps the longest
// agreeing prefix plus one token — all on the device, one graph per step.
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
  int S = 0;
  cudaStream_t cap = nullptr;
  // captured steps, keyed on what changes their kernels (skip mask, sampler,
  // draft shape), never on the caller's output pointers: each graph writes
  // its outputs into the model's own buffers and ends with copy nodes to the
  // caller's, re-pointed on the executable graph when they change
  struct OutCopy {
    const void* src;
    size_t bytes;
    void* dst;
    cudaGraphNode_t node;
  };
  struct Graph {
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ge = nullptr;
    std::vector<OutCopy> outs;
  };
  std::map<std::string, Graph> graphs;
  float* out_logits = nullptr;   // [2 kMaxVerify - 1][vocab]: the step's logits before the copy out
  int32_t* out_tok = nullptr;    // [kMaxVerify]: next token / emitted tokens
  int32_t* out_n = nullptr;      // emitted-token count of a speculative step
  // streaming: layers whose weights stay in page-locked host memory
  std::vector<const void*> host_blob;  // per layer; null = resident
  int n_slots = 0;
  size_t blob_bytes = 0, blob_off[7] = {};
  char* slots = nullptr;               // n_slots HBM slots of blob_bytes
  std::vector<int> slot_layer;         // last layer copied into each slot
  cudaStream_t copy_st = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  cudaEvent_t ev_ready[8] = {}, ev_free[8] = {};
  // self-speculative verify: up to kMaxVerify tokens per pass
  int32_t* spec_tok = nullptr;         // [kMaxVerify]: the step's token, then the drafts
  int64_t* spec_pos = nullptr;         // [kMaxVerify]: pos + i
  int32_t* vtok = nullptr;             // [kMaxVerify]: argmax of each verify row
  int32_t* prompt = nullptr;           // [kv_cap]: prefill tokens
  std::vector<int32_t> prompt_host;    // the host side of the prompt upload (see nt_prefill)
  cudaEvent_t ev_prompt = nullptr;     // recorded after that upload
  unsigned long long* vkey = nullptr;  // [kMaxVerify] argmax keys and counters
  unsigned* vcnt = nullptr;
  float *xv = nullptr, *qv = nullptr, *aov = nullptr, *hv = nullptr, *lv = nullptr, *dlogits = nullptr;
  float* gpart = nullptr;              // verify-GEMM partial sums
  size_t gpart_bytes = 0;
  float temperature = 0.f, top_p = 1.f;  // decode-step sampler (temperature <= 0: greedy)
  uint64_t seed = 0;
  char* samp = nullptr;                  // sampler state, kMaxVerify rows of kSampRowBytes
  // speculative sampling: nucleus weights of the draft rows and of the verify rows
  unsigned long long *sw_q = nullptr, *sW_q = nullptr;  // [kMaxVerify - 1][vocab], [kMaxVerify]
  unsigned long long *sw_p = nullptr, *sW_p = nullptr;  // [kMaxVerify][vocab], [kMaxVerify]
};

namespace nt {
namespace {

__global__ void set_state_kernel(int32_t* tok, int64_t* pos, int32_t t, int64_t p) {
  pdl_wait();
  *tok = t;
  *pos = p;
}

size_t up256(size_t n) { return (n + 255) / 256 * 256; }

constexpr int kMaxSlots = 8;

// rows x cols of the seven layer matrices, in blob order wq wk wv wo wg wu wd
void layer_shapes(const nt_model_desc& d, int64_t rows[7], int64_t cols[7], int fmt[7]) {
  const int64_t nq = int64_t(d.n_qh) * d.head_dim, nkv = int64_t(d.n_kvh) * d.head_dim;
  const int64_t r[7] = {nq, nkv, nkv, d.d_model, d.ffn, d.ffn, d.d_model};
  const int64_t c[7] = {d.d_model, d.d_model, d.d_model, nq, d.d_model, d.d_model, d.ffn};
  const int f[7] = {d.fmt_q, d.fmt_k, d.fmt_v, d.fmt_o, d.fmt_gate, d.fmt_up, d.fmt_down};
  for (int i = 0; i < 7; ++i) {
    rows[i] = r[i];
    cols[i] = c[i];
    fmt[i] = f[i];
  }
}

void blob_layout(const nt_model_desc& d, size_t off[7], size_t* total) {
  int64_t rows[7], cols[7];
  int fmt[7];
  layer_shapes(d, rows, cols, fmt);
  size_t o = 0;
  for (int i = 0; i < 7; ++i) {
    off[i] = o;
    o += up256(size_t(rows[i]) * size_t(cols[i] / block_elems(fmt[i])) * size_t(block_bytes(fmt[i])));
  }
  *total = o;
}

char* slot_ptr(const nt_model* m, int slot) { return m->slots + size_t(slot) * m->blob_bytes; }

// the layer's weight pointers when its blob sits in `slot`
void bind_slot(const nt_model* m, int slot, nt_layer_ptrs& L) {
  const char* b = slot_ptr(m, slot);
  const void** w[7] = {&L.wq, &L.wk, &L.wv, &L.wo, &L.wg, &L.wu, &L.wd};
  for (int i = 0; i < 7; ++i) *w[i] = b + m->blob_off[i];
}

// the copy step of the streaming engine: layer blob host -> HBM slot on st
nt_status copy_layer(Ctx* c, nt_model* m, int layer, const void* src, int slot, cudaStream_t st) {
  if (c->copy_fail_in >= 0 && c->copy_fail_in-- == 0)  // fault injection (host side): nothing is enqueued
    return set_err(c, NT_ERR_CUDA, "layer %d copy into slot %d: injected failure", layer, slot);
  nt_status s = cuda_check(c, cudaMemcpyAsync(slot_ptr(m, slot), src, m->blob_bytes, cudaMemcpyHostToDevice, st),
                           "stream layer copy");
  if (!s) m->slot_layer[slot] = layer;
  return s;
}

// Streaming schedule of one pass over the layers: the executed streamed
// layers, in order, go through slot i % n_slots on the copy stream; the
// first n_slots copies start with the pass, each later copy waits for the
// compute of the layer that last used its slot, and each streamed layer's
// compute waits for its copy.  Works eagerly and under stream capture (the
// copy stream joins the capture through the fork event).
struct Streamer {
  Ctx* c;
  nt_model* m;
  cudaStream_t st;
  std::vector<int> sl;
  int si = 0;           // ordinal of the next streamed layer
  bool forked = false;  // the copy stream waits on st and must be joined back

  // a pass cut short by an error still joins the copy stream, so a stream
  // capture in progress ends cleanly
  ~Streamer() {
    if (forked) {
      cudaEventRecord(m->ev_join, m->copy_st);
      cudaStreamWaitEvent(st, m->ev_join, 0);
    }
  }

  nt_status copy(int i) {
    if (c->dry) return NT_OK;
    const int NS = m->n_slots, slot = i % NS;
    nt_status r = NT_OK;
    if (i >= NS) r = cuda_check(c, cudaStreamWaitEvent(m->copy_st, m->ev_free[slot], 0), "copy waits for its slot");
    if (!r) r = copy_layer(c, m, sl[i], m->host_blob[sl[i]], slot, m->copy_st);
    if (!r) r = cuda_check(c, cudaEventRecord(m->ev_ready[slot], m->copy_st), "slot ready");
    return r;
  }
  nt_status begin(const uint8_t* skip) {
    for (int l = 0; l < m->d.n_layers; ++l)
      if (!(skip && skip[l]) && m->host_blob[l]) sl.push_back(l);
    if (sl.empty() || c->dry) return NT_OK;
    nt_status s = cuda_check(c, cudaEventRecord(m->ev_fork, st), "fork copy stream");
    if (!s) s = cuda_check(c, cudaStreamWaitEvent(m->copy_st, m->ev_fork, 0), "fork copy stream");
    forked = !s;
    for (int i = 0; i < m->n_slots && i < int(sl.size()) && !s; ++i) s = copy(i);
    return s;
  }
  // layer l's pointers (bound to its slot when streamed); slot = -1 when resident
  nt_status before(int l, nt_layer_ptrs& L, int& slot) {
    L = m->layers[l];
    slot = -1;
    if (!m->host_blob[l]) return NT_OK;
    slot = si % m->n_slots;
    bind_slot(m, slot, L);
    if (c->dry) return NT_OK;
    c->pdl_hold = true;  // the layer's first kernel must not prefetch the slot before the copy lands
    return cuda_check(c, cudaStreamWaitEvent(st, m->ev_ready[slot], 0), "compute waits for its layer copy");
  }
  nt_status after(int slot) {
    if (slot < 0) return NT_OK;
    if (c->dry) {
      ++si;
      return NT_OK;
    }
    // the slot is free once this layer's kernels are done: the copy that reuses it may start
    nt_status s = cuda_check(c, cudaEventRecord(m->ev_free[slot], st), "slot free");
    if (!s && si + m->n_slots < int(sl.size())) s = copy(si + m->n_slots);
    ++si;
    return s;
  }
  nt_status end() {
    if (sl.empty() || c->dry) return NT_OK;
    forked = false;
    nt_status s = cuda_check(c, cudaEventRecord(m->ev_join, m->copy_st), "join copy stream");
    if (!s) s = cuda_check(c, cudaStreamWaitEvent(st, m->ev_join, 0), "join copy stream");
    return s;
  }
};

// where one decode pass reads its token and position and puts its result
struct StepIO {
  const int32_t* tok;  // device token
  const int64_t* pos;  // device position
  float* logits;
  int32_t* next_tok;   // nullable: receives the argmax
  bool advance;        // the argmax also moves the model state: tok = argmax, pos += 1
  // sampled drafts (model sampler set): the draft row's nucleus weights and their sum
  unsigned long long* w_out = nullptr;
  unsigned long long* W_out = nullptr;
};

// all kernels of one decode step, enqueued on st
nt_status enqueue_step(Ctx* c, nt_model* m, const uint8_t* skip, const StepIO& io, cudaStream_t st, bool want_cos) {
  const nt_model_desc& d = m->d;
  const int hd = d.head_dim;
  const int64_t nq = int64_t(d.n_qh) * hd, nkv = int64_t(d.n_kvh) * hd;
  Streamer sm{c, m, st};
  nt_status s = sm.begin(skip);
  if (s) return s;
  s = launch_embed(c, d.fmt_embd, m->embd, d.d_model, io.tok, m->x, st);
  if (s) return s;
  char lname[24];
  for (int l = 0; l < d.n_layers; ++l) {
    if (skip && skip[l]) continue;
    snprintf(lname, sizeof lname, "layer %d", l);
    NvtxRange layer_range(lname);
    nt_layer_ptrs L;
    int slot;
    s = sm.before(l, L, slot);
    if (s) return s;
    if (want_cos && !c->dry) {
      s = cuda_check(c, cudaMemcpyAsync(m->xin, m->x, sizeof(float) * d.d_model, cudaMemcpyDeviceToDevice, st),
                     "copy x");
      if (s) return s;
    }
    // Q, K, V: one launch per distinct format; attention RMSNorm fused in
    // front, RoPE and the f16 KV append fused behind
    {
      const RopeArgs ra{io.pos, m->inv_freq, hd, d.kv_cap};
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
    s = launch_attn(c, m->q, L.kcache, L.vcache, m->ao, d.n_qh, d.n_kvh, 0, io.pos, d.kv_cap, m->attn_part,
                    m->S, st);
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
    s = sm.after(slot);
    if (s) return s;
  }
  s = sm.end();
  if (s) return s;
  {
    nt_gemv_job j{m->out, io.logits, nullptr, d.vocab};
    s = launch_gemv(c, d.fmt_out, &j, 1, nullptr, m->x, m->out_norm, d.eps, d.d_model, false, st);
    if (s) return s;
  }
  if ((io.advance || io.w_out) && m->temperature > 0.f)  // counter: the position of this step's input token
    return launch_sample(c, io.logits, d.vocab, 1, m->temperature, m->top_p, m->seed, io.pos, 0, io.next_tok, m->samp,
                         st, io.advance ? m->tok : nullptr, io.advance ? m->pos : nullptr, io.w_out, io.W_out);
  return launch_argmax(c, io.logits, d.vocab, io.next_tok, m->amax_key, m->amax_cnt, st,
                       io.advance ? m->tok : nullptr, io.advance ? m->pos : nullptr);
}

// the verify pass: tokens spec_tok[0..M) at positions spec_pos[0] + i
// through every layer (M-vector GEMMs, causal M-query attention), logits
// [M][vocab], row argmaxes into vtok
// the M tokens tok_dev[0..M) at positions pos_dev[0] + i; sm: the pass's
// streaming schedule, begun by the caller (its first copies may overlap the
// drafts); logits == nullptr: no LM head (a prefill chunk before the last)
nt_status enqueue_multi(Ctx* c, nt_model* m, int M, const int32_t* tok_dev, const int64_t* pos_dev, float* logits,
                        bool argmax, Streamer& sm, cudaStream_t st) {
  const nt_model_desc& d = m->d;
  const int hd = d.head_dim;
  const int64_t nq = int64_t(d.n_qh) * hd, nkv = int64_t(d.n_kvh) * hd;
  nt_status s = launch_embed(c, d.fmt_embd, m->embd, d.d_model, tok_dev, m->xv, st, M);
  if (s) return s;
  const RopeArgs ra{pos_dev, m->inv_freq, hd, d.kv_cap};
  for (int l = 0; l < d.n_layers; ++l) {
    nt_layer_ptrs L;
    int slot;
    s = sm.before(l, L, slot);
    if (s) return s;
    {
      const GemmJobEx J[3] = {GemmJobEx{L.wq, nq, m->qv, nq, nullptr, nullptr, kEpiRope},
                              GemmJobEx{L.wk, nkv, nullptr, 0, nullptr, L.kcache, kEpiRopeCache},
                              GemmJobEx{L.wv, nkv, nullptr, 0, nullptr, L.vcache, kEpiCache}};
      const int F[3] = {d.fmt_q, d.fmt_k, d.fmt_v};
      bool done[3] = {false, false, false};
      for (int i = 0; i < 3; ++i) {
        if (done[i]) continue;
        GemmJobEx jobs[3];
        int nj = 0;
        for (int j = i; j < 3; ++j)
          if (!done[j] && F[j] == F[i]) {
            jobs[nj++] = J[j];
            done[j] = true;
          }
        s = launch_gemm(c, F[i], jobs, nj, false, m->xv, d.d_model, M, L.attn_norm, d.eps, d.d_model, &ra,
                        m->gpart, m->gpart_bytes, st);
        if (s) return s;
      }
    }
    s = launch_attn(c, m->qv, L.kcache, L.vcache, m->aov, d.n_qh, d.n_kvh, 0, pos_dev, d.kv_cap, m->attn_part,
                    m->S, st, M);
    if (s) return s;
    {
      const GemmJobEx j{L.wo, d.d_model, m->xv, d.d_model, m->xv, nullptr, kEpiPlain};
      s = launch_gemm(c, d.fmt_o, &j, 1, false, m->aov, nq, M, nullptr, 0.f, nq, nullptr, m->gpart, m->gpart_bytes,
                      st);
      if (s) return s;
    }
    {
      const GemmJobEx j[2] = {GemmJobEx{L.wg, d.ffn, m->hv, d.ffn, nullptr, nullptr, kEpiPlain},
                              GemmJobEx{L.wu, d.ffn, nullptr, 0, nullptr, nullptr, kEpiPlain}};
      s = launch_gemm(c, d.fmt_gate, j, 2, true, m->xv, d.d_model, M, L.ffn_norm, d.eps, d.d_model, nullptr,
                      m->gpart, m->gpart_bytes, st);
      if (s) return s;
    }
    {
      const GemmJobEx j{L.wd, d.d_model, m->xv, d.d_model, m->xv, nullptr, kEpiPlain};
      s = launch_gemm(c, d.fmt_down, &j, 1, false, m->hv, d.ffn, M, nullptr, 0.f, d.ffn, nullptr, m->gpart,
                      m->gpart_bytes, st);
      if (s) return s;
    }
    s = sm.after(slot);
    if (s) return s;
  }
  s = sm.end();
  if (s || !logits) return s;
  {
    const GemmJobEx j{m->out, d.vocab, logits, d.vocab, nullptr, nullptr, kEpiPlain};
    s = launch_gemm(c, d.fmt_out, &j, 1, false, m->xv, d.d_model, M, m->out_norm, d.eps, d.d_model, nullptr,
                    m->gpart, m->gpart_bytes, st);
    if (s) return s;
  }
  for (int i = 0; argmax && i < M && !s; ++i)
    s = launch_argmax(c, logits + int64_t(i) * d.vocab, d.vocab, m->vtok + i, m->vkey + i, m->vcnt + i, st);
  return s;
}

// one prefill chunk: tokens prompt[0..M) at positions base + i
__global__ void prefill_setup_kernel(const int32_t* prompt, int64_t base, int32_t* tok, int64_t* pos, int M) {
  pdl_wait();
  pdl_trigger();
  if (int(threadIdx.x) < M) {
    tok[threadIdx.x] = prompt[threadIdx.x];
    pos[threadIdx.x] = base + threadIdx.x;
  }
}

// start of a speculative step: the step's token and the positions of the
// verify rows, from the model state
__global__ void spec_setup_kernel(const int32_t* tok, const int64_t* pos, int32_t* spec_tok, int64_t* spec_pos,
                                  int M) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) spec_tok[0] = *tok;
  if (int(threadIdx.x) < M) spec_pos[threadIdx.x] = *pos + threadIdx.x;
}

// end of a speculative step: draft i + 1 is kept while it equals the verify
// argmax of row i; the kept drafts plus the verify argmax after them are the
// step's tokens, and the model state moves past them
__global__ void spec_accept_kernel(const int32_t* spec_tok, const int32_t* vtok, int k, int32_t* out, int32_t* n_out,
                                   int32_t* tok, int64_t* pos, const int64_t* spec_pos) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x != 0) return;
  int n = 0;
  while (n < k && spec_tok[n + 1] == vtok[n]) ++n;
  for (int i = 0; i <= n; ++i) out[i] = vtok[i];
  *n_out = n + 1;
  *tok = vtok[n];
  *pos = spec_pos[0] + n + 1;
}

// end of a sampled speculative step (speculative sampling: Leviathan, Kalman
// & Matias 2023, section 2.3): draft i + 1, drawn from the draft's nucleus
// distribution q_i, is kept when u < p_i(d) / q_i(d), p_i the target's
// (verify row i); at the first rejection the step's last token is drawn from
// max(0, p_i - q_i) renormalised; with every draft kept, the last token is the
// sampler's pick from verify row k.  All in integers: weights below 2^40,
// sums below 2^57, products in 128 bits.  Uniforms: h = splitmix64(seed xor
// (2 (pos + i) + 1)), u = bits 40..63 of h / 2^24 for the test, bits 16..39
// for the residual draw.  One CTA.
typedef unsigned __int128 u128;
constexpr int kAccThreads = 1024;

__device__ __forceinline__ uint64_t spec_splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// exclusive prefix sum of 128-bit values over the block; total in *total
__device__ u128 scan128(u128 v, u128* total) {
  __shared__ unsigned long long slo[kAccThreads / 32], shi[kAccThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  u128 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long lo = __shfl_up_sync(0xffffffffu, static_cast<unsigned long long>(x), o);
    const unsigned long long hi = __shfl_up_sync(0xffffffffu, static_cast<unsigned long long>(x >> 64), o);
    if (lane >= o) x += (u128(hi) << 64) | lo;
  }
  if (lane == 31) {
    slo[warp] = static_cast<unsigned long long>(x);
    shi[warp] = static_cast<unsigned long long>(x >> 64);
  }
  __syncthreads();
  u128 before = x - v, all = 0;
  for (int w = 0; w < kAccThreads / 32; ++w) {
    const u128 t = (u128(shi[w]) << 64) | slo[w];
    if (w < warp) before += t;
    all += t;
  }
  *total = all;
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kAccThreads)
    spec_accept_sampled_kernel(const int32_t* spec_tok, const int32_t* vtok, int k, int64_t n,
                               const unsigned long long* wq, const unsigned long long* Wq,
                               const unsigned long long* wp, const unsigned long long* Wp, uint64_t seed,
                               int32_t* out, int32_t* n_out, int32_t* tok, int64_t* pos, const int64_t* spec_pos) {
  __shared__ int s_pick;
  pdl_wait();
  pdl_trigger();
  const int64_t per = (n + kAccThreads - 1) / kAccThreads;
  const int64_t i0 = min(n, int64_t(threadIdx.x) * per), i1 = min(n, i0 + per);
  int e = k + 1;  // tokens the step emits
  for (int i = 0; i < k; ++i) {
    const int32_t d = spec_tok[i + 1];
    const unsigned long long* q = wq + int64_t(i) * n;
    const unsigned long long* p = wp + int64_t(i) * n;
    const unsigned long long Wqi = Wq[i], Wpi = Wp[i];
    const uint64_t h = spec_splitmix64(seed ^ ((uint64_t(spec_pos[i]) << 1) | 1u));
    const uint32_t kacc = uint32_t(h >> 40), kres = uint32_t((h >> 16) & 0xFFFFFFu);
    if (u128(kacc) * q[d] * Wpi < ((u128(p[d]) * Wqi) << 24)) {
      if (threadIdx.x == 0) out[i] = d;
      continue;
    }
    // rejected: the residual draw, R_t = max(0, p_t Wq - q_t Wp), pick at floor(kres * sum R / 2^24)
    u128 mass = 0;
    for (int64_t t = i0; t < i1; ++t) {
      const u128 a = u128(p[t]) * Wqi, b = u128(q[t]) * Wpi;
      if (a > b) mass += a - b;
    }
    u128 total;
    const u128 base = scan128(mass, &total);
    const u128 r = u128(kres) * (total >> 24) + ((u128(kres) * static_cast<unsigned long long>(total & 0xFFFFFFu)) >> 24);
    if (threadIdx.x == 0) s_pick = -1;
    __syncthreads();
    if (mass && base <= r && r < base + mass) {
      u128 acc = base;
      for (int64_t t = i0; t < i1; ++t) {
        const u128 a = u128(p[t]) * Wqi, b = u128(q[t]) * Wpi;
        if (a > b) acc += a - b;
        if (acc > r) {
          s_pick = int(t);
          break;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) out[i] = s_pick >= 0 ? s_pick : vtok[i];  // the residual is never empty after a rejection
    e = i + 1;
    break;
  }
  if (threadIdx.x == 0) {
    if (e == k + 1) out[k] = vtok[k];
    *n_out = e;
    *tok = out[e - 1];
    *pos = spec_pos[0] + e;
  }
}

// draft layers: [0, n_draft) when n_draft > 0, else every resident layer
std::vector<uint8_t> draft_mask(const nt_model* m, int n_draft) {
  std::vector<uint8_t> mask(m->d.n_layers, 0);
  for (int l = 0; l < m->d.n_layers; ++l) mask[l] = n_draft > 0 ? (l >= n_draft) : (m->host_blob[l] != nullptr);
  return mask;
}

nt_status enqueue_spec(Ctx* c, nt_model* m, int k, int n_draft, int32_t* out, int32_t* n_out, float* logits,
                       cudaStream_t st) {
  const int M = k + 1;
  nt_status s = c->dry ? NT_OK
                       : cuda_check(c, launch_k(c, spec_setup_kernel, dim3(1), dim3(32), 0, st, m->tok, m->pos,
                                                m->spec_tok, m->spec_pos, M),
                                    "spec setup launch");
  if (s) return s;
  const std::vector<uint8_t> mask = draft_mask(m, n_draft);
  // the verify pass's first layer copies start now and overlap the drafts
  // (drafts that run streamed layers stream them themselves, so then the
  // verify's copies start after the drafts)
  bool drafts_stream = false;
  for (int l = 0; l < m->d.n_layers; ++l) drafts_stream = drafts_stream || (!mask[l] && m->host_blob[l]);
  Streamer sm{c, m, st};
  const bool sampled = m->temperature > 0.f;
  const int64_t V = m->d.vocab;
  if (!drafts_stream) s = sm.begin(nullptr);
  for (int i = 0; i < k && !s; ++i) {
    StepIO io{m->spec_tok + i, m->spec_pos + i, m->dlogits, m->spec_tok + i + 1, false};
    if (sampled) {  // drafts drawn by the sampler, their distributions kept for the acceptance test
      if (logits) io.logits = logits + (M + i) * V;
      io.w_out = m->sw_q + i * V;
      io.W_out = m->sW_q + i;
    }
    s = enqueue_step(c, m, mask.data(), io, st, false);
  }
  if (!s && drafts_stream) s = sm.begin(nullptr);
  float* vl = logits ? logits : m->lv;
  if (!s) s = enqueue_multi(c, m, M, m->spec_tok, m->spec_pos, vl, !sampled, sm, st);
  if (!s && sampled)
    s = launch_sample(c, vl, V, M, m->temperature, m->top_p, m->seed, m->spec_pos, 0, m->vtok, m->samp, st, nullptr,
                      nullptr, m->sw_p, m->sW_p);
  if (!s && !c->dry)
    s = sampled ? cuda_check(c, launch_k(c, spec_accept_sampled_kernel, dim3(1), dim3(kAccThreads), 0, st,
                                         static_cast<const int32_t*>(m->spec_tok), static_cast<const int32_t*>(m->vtok),
                                         k, V, static_cast<const unsigned long long*>(m->sw_q),
                                         static_cast<const unsigned long long*>(m->sW_q),
                                         static_cast<const unsigned long long*>(m->sw_p),
                                         static_cast<const unsigned long long*>(m->sW_p), m->seed, out, n_out, m->tok,
                                         m->pos, static_cast<const int64_t*>(m->spec_pos)),
                             "spec accept launch")
                : cuda_check(c, launch_k(c, spec_accept_kernel, dim3(1), dim3(32), 0, st, m->spec_tok, m->vtok, k, out,
                                         n_out, m->tok, m->pos, m->spec_pos),
                             "spec accept launch");
  return s;
}

template <typename T>
void key_append(std::string& k, const T& v) {
  k.append(reinterpret_cast<const char*>(&v), sizeof v);
}

std::string graph_key(const nt_model* m, const uint8_t* skip, const int32_t* next_tok) {
  std::string k("d");
  key_append(k, next_tok != nullptr);
  key_append(k, m->temperature);
  key_append(k, m->top_p);
  key_append(k, m->seed);
  for (int l = 0; l < m->d.n_layers; ++l) k.push_back(skip && skip[l] ? '1' : '0');
  return k;
}

// one output of a step: the model buffer the step writes, its size, and
// the caller's buffer it is copied to at the end of the graph
struct Out {
  const void* src;
  size_t bytes;
  void* dst;
};

// replay the graph under `key`, capturing it first with `enqueue` on the
// model's capture stream, followed by the copies `outs`
template <typename F>
nt_status run_graph(Ctx* c, nt_model* m, const std::string& key, cudaStream_t st, const std::vector<Out>& outs,
                    F enqueue) {
  auto it = m->graphs.find(key);
  nt_status s = NT_OK;
  if (it == m->graphs.end()) {
    if (c->gemv_tune) {
      // a dry pass first: every GEMV shape of the sequence gets its plan
      // tuned eagerly on st, so the captured graph holds tuned launches
      c->dry = true;
      s = enqueue(st);
      c->dry = false;
      if (s) return s;
    }
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ge = nullptr;
    const std::vector<int> slots_before = m->slot_layer;  // a failed capture copies nothing
    s = cuda_check(c, cudaStreamBeginCapture(m->cap, cudaStreamCaptureModeThreadLocal), "begin capture");
    if (!s) {
      nt_status s2 = enqueue(m->cap);
      for (const Out& o : outs)
        if (!s2)
          s2 = cuda_check(c, cudaMemcpyAsync(o.dst, o.src, o.bytes, cudaMemcpyDeviceToDevice, m->cap), "copy out");
      cudaError_t e = cudaStreamEndCapture(m->cap, &g);
      if (s2 && e != cudaSuccess) cudaGetLastError();  // the first error is the one reported
      s = s2 ? s2 : cuda_check(c, e, "end capture");
    }
    nt_model::Graph gr;
    gr.g = g;
    if (!s) {
      // the copy-out nodes, found by their source buffers
      size_t n = 0;
      s = cuda_check(c, cudaGraphGetNodes(g, nullptr, &n), "graph nodes");
      std::vector<cudaGraphNode_t> nodes(n);
      if (!s && n) s = cuda_check(c, cudaGraphGetNodes(g, nodes.data(), &n), "graph nodes");
      for (const Out& o : outs) {
        nt_model::OutCopy oc{o.src, o.bytes, o.dst, nullptr};
        for (size_t i = 0; i < n && !s && !oc.node; ++i) {
          cudaGraphNodeType t;
          if (cudaGraphNodeGetType(nodes[i], &t) != cudaSuccess || t != cudaGraphNodeTypeMemcpy) continue;
          cudaMemcpy3DParms p{};
          if (cudaGraphMemcpyNodeGetParams(nodes[i], &p) == cudaSuccess && p.srcPtr.ptr == o.src) oc.node = nodes[i];
        }
        if (!s && !oc.node) s = set_err(c, NT_ERR_CUDA, "copy-out node not found in the captured step");
        gr.outs.push_back(oc);
      }
    }
    if (!s) s = cuda_check(c, cudaGraphInstantiate(&ge, g, 0), "graph instantiate");
    if (s) {
      if (g) cudaGraphDestroy(g);
      cudaGetLastError();
      m->slot_layer = slots_before;
      return s;
    }
    gr.ge = ge;
    it = m->graphs.emplace(key, gr).first;
  }
  // point the copy-out nodes at this call's buffers
  nt_model::Graph& gr = it->second;
  for (size_t i = 0; i < gr.outs.size() && i < outs.size() && !s; ++i) {
    nt_model::OutCopy& oc = gr.outs[i];
    if (oc.dst == outs[i].dst) continue;
    s = cuda_check(c, cudaGraphExecMemcpyNodeSetParams1D(gr.ge, oc.node, outs[i].dst, oc.src, oc.bytes,
                                                         cudaMemcpyDeviceToDevice),
                   "re-point the step's output copy");
    if (!s) oc.dst = outs[i].dst;
  }
  if (s) return s;
  return cuda_check(c, cudaGraphLaunch(gr.ge, st), "graph launch");
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
  NvtxRange nvtx_range("nt_model_init");
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
  const int n_slots = d.stream_slots == 0 ? 2 : d.stream_slots;
  NT_REQUIRE(n_slots >= 1 && n_slots <= kMaxSlots, NT_ERR_INVALID_ARG, "stream_slots must be 0..%d", kMaxSlots);
  int n_streamed = 0;
  for (int l = 0; l < d.n_layers; ++l) {
    const nt_layer_ptrs& L = layers[l];
    NT_REQUIRE(L.attn_norm && L.ffn_norm && L.kcache && L.vcache, NT_ERR_INVALID_ARG, "layer %d: null norm/cache", l);
    NT_REQUIRE(aligned(L.kcache, 16) && aligned(L.vcache, 16) && aligned(L.attn_norm, 16) && aligned(L.ffn_norm, 16),
               NT_ERR_ALIGNMENT, "layer %d: caches and norms must be 16-byte aligned", l);
    const void* w[7] = {L.wq, L.wk, L.wv, L.wo, L.wg, L.wu, L.wd};
    int nw = 0;
    for (const void* p : w) nw += p != nullptr;
    if (nw == 7) {
      NT_REQUIRE(!L.host_blob, NT_ERR_INVALID_ARG, "layer %d: resident weights and a host blob", l);
    } else {
      NT_REQUIRE(nw == 0 && L.host_blob, NT_ERR_INVALID_ARG,
                 "layer %d: set all seven weight pointers, or none and a host blob", l);
      cudaPointerAttributes pa{};
      const cudaError_t pe = cudaPointerGetAttributes(&pa, L.host_blob);
      if (pe != cudaSuccess) cudaGetLastError();  // a refused query leaves no error behind for later launches
      NT_REQUIRE(pe == cudaSuccess && pa.type == cudaMemoryTypeHost, NT_ERR_INVALID_ARG,
                 "layer %d: host_blob must be page-locked host memory", l);
      ++n_streamed;
    }
  }
  NT_REQUIRE(aligned(out_norm, 16), NT_ERR_ALIGNMENT, "out_norm must be 16-byte aligned");
  NT_REQUIRE(aligned(embd, d.fmt_embd == NT_F32 ? 4 : 2), NT_ERR_ALIGNMENT, "embd is misaligned for its format");
  // an embedding table in page-locked host memory is read through its device alias
  {
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, embd) == cudaSuccess && pa.type == cudaMemoryTypeHost) {
      NT_REQUIRE(pa.devicePointer, NT_ERR_INVALID_ARG, "embd: host memory without a device mapping");
      embd = pa.devicePointer;
    }
    cudaGetLastError();
  }

  nt_model* m = new (std::nothrow) nt_model();
  if (!m) return NT_ERR_OOM;
  m->d = d;
  m->layers.assign(layers, layers + d.n_layers);
  m->host_blob.resize(d.n_layers);
  for (int l = 0; l < d.n_layers; ++l) m->host_blob[l] = layers[l].host_blob;
  blob_layout(d, m->blob_off, &m->blob_bytes);
  m->n_slots = n_streamed ? n_slots : 0;
  m->slot_layer.assign(m->n_slots, -1);
  m->embd = embd;
  m->out = out;
  m->out_norm = out_norm;
  m->S = attn_splits(ctx, d.n_kvh, d.kv_cap);
  const size_t fl = sizeof(float);
  const size_t nx = up256(fl * d.d_model), nqb = up256(fl * nq), nkb = up256(fl * d.n_kvh * d.head_dim),
               nh = up256(fl * d.ffn), ncos = up256(fl * d.n_layers), nst = 256, nfreq = up256(8 * d.head_dim),
               npart = up256(attn_scratch_bytes(d.n_qh, d.n_kvh, m->S, kMaxGemmM)), nspec = 1024,
               nvx = up256(fl * kMaxGemmM * d.d_model), nvq = up256(fl * kMaxGemmM * nq),
               nvh = up256(fl * kMaxGemmM * d.ffn), nvl = up256(fl * kMaxGemmM * d.vocab), ndl = up256(fl * d.vocab),
               nprompt = up256(sizeof(int32_t) * size_t(d.kv_cap)), nsamp = kSampRowBytes * kMaxVerify,
               nsw = up256(8 * size_t(d.vocab)), nsW = up256(8 * kMaxVerify),
               nout = up256(fl * size_t(2 * kMaxVerify - 1) * size_t(d.vocab)), nouttok = 256;
  {
    // partial sums of the largest verify GEMM
    const int64_t nkv = int64_t(d.n_kvh) * d.head_dim;
    const int64_t rc[7][3] = {{nq + 2 * nkv, d.d_model, d.fmt_q}, {nq + 2 * nkv, d.d_model, d.fmt_k},
                              {nq + 2 * nkv, d.d_model, d.fmt_v}, {d.d_model, nq, d.fmt_o},
                              {2 * int64_t(d.ffn), d.d_model, d.fmt_gate}, {d.d_model, d.ffn, d.fmt_down},
                              {d.vocab, d.d_model, d.fmt_out}};
    for (auto& x : rc)
      m->gpart_bytes = std::max(m->gpart_bytes, gemm_scratch_bytes(int(x[2]), x[0], x[1], kMaxGemmM));
    m->gpart_bytes = up256(m->gpart_bytes);
  }
  const size_t total = 2 * nx + nqb * 2 + nkb * 2 + nh + ncos + nst + npart + nfreq + nspec + nvx + 2 * nvq + nvh +
                       nvl + ndl + nprompt + m->gpart_bytes + nsamp + nsw * (2 * kMaxVerify - 1) + 2 * nsW + nout +
                       nouttok;
  int dev_prev = 0;
  cudaGetDevice(&dev_prev);
  cudaSetDevice(ctx->device);
  cudaError_t e = cudaMalloc(&m->buf, total);
  if (e == cudaSuccess) e = cudaMemset(m->buf, 0, total);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&m->cap, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_prompt, cudaEventDisableTiming);
  if (e == cudaSuccess && m->n_slots) {
    e = cudaMalloc(&m->slots, size_t(m->n_slots) * m->blob_bytes);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&m->copy_st, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_join, cudaEventDisableTiming);
    for (int i = 0; i < m->n_slots && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&m->ev_ready[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_free[i], cudaEventDisableTiming);
    }
  }
  cudaSetDevice(dev_prev);
  if (e != cudaSuccess) {
    const nt_status st = cuda_check(ctx, e, "model allocation");
    nt_model_destroy(ctx, m);
    return e == cudaErrorMemoryAllocation ? set_err(ctx, NT_ERR_OOM, "model allocation: out of device memory") : st;
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
  m->attn_part = reinterpret_cast<float*>(part + kAttnCounterBytes);
  char* sp = take(nspec);
  m->spec_tok = reinterpret_cast<int32_t*>(sp);         // [kMaxGemmM]
  m->spec_pos = reinterpret_cast<int64_t*>(sp + 64);     // [kMaxGemmM]
  m->vtok = reinterpret_cast<int32_t*>(sp + 192);        // [kMaxVerify]
  m->vkey = reinterpret_cast<unsigned long long*>(sp + 256);
  m->vcnt = reinterpret_cast<unsigned*>(sp + 320);
  m->xv = reinterpret_cast<float*>(take(nvx));
  m->qv = reinterpret_cast<float*>(take(nvq));
  m->aov = reinterpret_cast<float*>(take(nvq));
  m->hv = reinterpret_cast<float*>(take(nvh));
  m->lv = reinterpret_cast<float*>(take(nvl));
  m->dlogits = reinterpret_cast<float*>(take(ndl));
  m->prompt = reinterpret_cast<int32_t*>(take(nprompt));
  m->gpart = reinterpret_cast<float*>(take(m->gpart_bytes));
  m->samp = take(nsamp);
  m->sw_q = reinterpret_cast<unsigned long long*>(take(nsw * (kMaxVerify - 1)));
  m->sw_p = reinterpret_cast<unsigned long long*>(take(nsw * kMaxVerify));
  m->out_logits = reinterpret_cast<float*>(take(nout));
  {
    char* ot = take(nouttok);
    m->out_tok = reinterpret_cast<int32_t*>(ot);
    m->out_n = reinterpret_cast<int32_t*>(ot + 64);
  }
  m->sW_q = reinterpret_cast<unsigned long long*>(take(nsW));
  m->sW_p = reinterpret_cast<unsigned long long*>(take(nsW));
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
  for (auto& kv : m->graphs) {
    cudaGraphExecDestroy(kv.second.ge);
    cudaGraphDestroy(kv.second.g);
  }
  if (m->cap) cudaStreamDestroy(m->cap);
  if (m->copy_st) cudaStreamDestroy(m->copy_st);
  for (cudaEvent_t ev : {m->ev_fork, m->ev_join, m->ev_prompt})
    if (ev) cudaEventDestroy(ev);
  for (int i = 0; i < kMaxSlots; ++i) {
    if (m->ev_ready[i]) cudaEventDestroy(m->ev_ready[i]);
    if (m->ev_free[i]) cudaEventDestroy(m->ev_free[i]);
  }
  if (m->slots) cudaFree(m->slots);
  if (m->buf) cudaFree(m->buf);
  cudaSetDevice(dev_prev);
  delete m;
  return NT_OK;
}

nt_status nt_decode_step(nt_ctx* ctx, nt_model* m, int32_t token, int64_t pos, const uint8_t* skip, float* logits,
                         int32_t* next_tok, void* stream) {
  NvtxRange nvtx_range("nt_decode_step");
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m && logits, NT_ERR_INVALID_ARG, "null model or logits");
  NT_REQUIRE(aligned(logits, 16), NT_ERR_ALIGNMENT, "logits must be 16-byte aligned");
  if (token >= 0) {
    NT_REQUIRE(token < m->d.vocab, NT_ERR_INVALID_ARG, "token %d outside the vocabulary", token);
    NT_REQUIRE(pos >= 0 && pos < m->d.kv_cap, NT_ERR_INVALID_ARG, "pos %lld outside the KV cache",
               (long long)pos);
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
    const StepIO io{m->tok, m->pos, m->out_logits, next_tok ? m->out_tok : nullptr, true};
    std::vector<Out> outs{{m->out_logits, sizeof(float) * size_t(m->d.vocab), logits}};
    if (next_tok) outs.push_back({m->out_tok, sizeof(int32_t), next_tok});
    s = run_graph(ctx, m, graph_key(m, skip, next_tok), st, outs,
                  [&](cudaStream_t cs) { return enqueue_step(ctx, m, skip, io, cs, false); });
  }
  if (dev_prev != ctx->device) cudaSetDevice(dev_prev);
  return s;
}

nt_status nt_layer_skip_calibrate(nt_ctx* ctx, nt_model* m, int32_t token, int64_t pos, int n_skip, uint8_t* mask,
                                  float* cos_host, float* logits, int32_t* next_tok, void* stream) {
  NvtxRange nvtx_range("nt_layer_skip_calibrate");
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
  if (!s) s = enqueue_step(ctx, m, nullptr, StepIO{m->tok, m->pos, logits, next_tok, true}, st, true);
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

nt_status nt_spec_step(nt_ctx* ctx, nt_model* m, int32_t token, int64_t pos, int k, int n_draft_layers,
                       int32_t* tokens_out, int32_t* n_out, float* logits, void* stream) {
  NvtxRange nvtx_range("nt_spec_step");
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m && tokens_out && n_out, NT_ERR_INVALID_ARG, "null model or outputs");
  NT_REQUIRE(k >= 1 && k < kMaxVerify, NT_ERR_INVALID_ARG, "k must be 1..%d", kMaxVerify - 1);
  NT_REQUIRE(n_draft_layers >= 0 && n_draft_layers <= m->d.n_layers, NT_ERR_INVALID_ARG,
             "n_draft_layers outside 0..n_layers");
  NT_REQUIRE(aligned(tokens_out, 4) && aligned(n_out, 4), NT_ERR_ALIGNMENT, "outputs must be 4-byte aligned");
  NT_REQUIRE(!logits || aligned(logits, 16), NT_ERR_ALIGNMENT, "logits must be 16-byte aligned");
  if (token >= 0) {
    NT_REQUIRE(token < m->d.vocab, NT_ERR_INVALID_ARG, "token %d outside the vocabulary", token);
    NT_REQUIRE(pos >= 0 && pos + k < m->d.kv_cap, NT_ERR_INVALID_ARG, "pos %lld: pos + k outside the KV cache",
               (long long)pos);
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
    std::string key("s");
    key_append(key, k);
    key_append(key, n_draft_layers);
    key_append(key, logits != nullptr);
    key_append(key, m->temperature);
    key_append(key, m->top_p);
    key_append(key, m->seed);
    std::vector<Out> outs{{m->out_tok, sizeof(int32_t) * size_t(k + 1), tokens_out},
                          {m->out_n, sizeof(int32_t), n_out}};
    if (logits) outs.push_back({m->out_logits, sizeof(float) * size_t(2 * k + 1) * size_t(m->d.vocab), logits});
    float* own_logits = logits ? m->out_logits : nullptr;
    s = run_graph(ctx, m, key, st, outs, [&](cudaStream_t cs) {
      return enqueue_spec(ctx, m, k, n_draft_layers, m->out_tok, m->out_n, own_logits, cs);
    });
  }
  if (dev_prev != ctx->device) cudaSetDevice(dev_prev);
  return s;
}

nt_status nt_model_graph_count(nt_ctx* ctx, nt_model* m, int* n) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m && n, NT_ERR_INVALID_ARG, "null model or output");
  *n = int(m->graphs.size());
  return NT_OK;
}

nt_status nt_layer_blob_layout(const nt_model_desc* d, size_t* off, size_t* bytes) {
  if (!d || !off || !bytes) return NT_ERR_INVALID_ARG;
  const int fm[7] = {d->fmt_q, d->fmt_k, d->fmt_v, d->fmt_o, d->fmt_gate, d->fmt_up, d->fmt_down};
  for (int f : fm)
    if (!fmt_ok(f)) return NT_ERR_UNSUPPORTED_FMT;
  if (d->d_model <= 0 || d->n_qh <= 0 || d->n_kvh <= 0 || d->head_dim <= 0 || d->ffn <= 0) return NT_ERR_INVALID_ARG;
  blob_layout(*d, off, bytes);
  return NT_OK;
}

// prompt tokens per prefill pass: 16 when every GEMM of the step takes the
// tensor-core form (formats, row widths, 16-byte-aligned resident weights;
// streamed weights sit in aligned slots), else the verify size
static int prefill_chunk(const Ctx* c, const nt_model* m) {
  const nt_model_desc& d = m->d;
  const int64_t nq = int64_t(d.n_qh) * d.head_dim;
  const bool fmts = gemm_wide_ok(c, d.fmt_q, d.d_model) && gemm_wide_ok(c, d.fmt_k, d.d_model) &&
                    gemm_wide_ok(c, d.fmt_v, d.d_model) && gemm_wide_ok(c, d.fmt_o, nq) &&
                    gemm_wide_ok(c, d.fmt_gate, d.d_model) && gemm_wide_ok(c, d.fmt_down, d.ffn) &&
                    gemm_wide_ok(c, d.fmt_out, d.d_model);
  if (!fmts || !aligned(m->out, 16)) return kMaxVerify;
  for (const nt_layer_ptrs& L : m->layers)
    for (const void* w : {L.wq, L.wk, L.wv, L.wo, L.wg, L.wu, L.wd})
      if (w && !aligned(w, 16)) return kMaxVerify;
  return kMaxGemmM;
}

nt_status nt_model_prefill_chunk(nt_ctx* ctx, nt_model* m, int* chunk) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m && chunk, NT_ERR_INVALID_ARG, "null model or chunk");
  *chunk = prefill_chunk(ctx, m);
  return NT_OK;
}

nt_status nt_prefill(nt_ctx* ctx, nt_model* m, const int32_t* tokens_host, int64_t n, int64_t pos0, float* logits,
                     int32_t* next_tok, void* stream) {
  NvtxRange nvtx_range("nt_prefill");
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m && tokens_host && logits, NT_ERR_INVALID_ARG, "null model, tokens or logits");
  NT_REQUIRE(aligned(logits, 16), NT_ERR_ALIGNMENT, "logits must be 16-byte aligned");
  NT_REQUIRE(n >= 1 && pos0 >= 0 && pos0 + n <= m->d.kv_cap, NT_ERR_INVALID_ARG,
             "need n >= 1 and pos0 + n <= kv_cap (%lld)", (long long)m->d.kv_cap);
  for (int64_t i = 0; i < n; ++i)
    NT_REQUIRE(tokens_host[i] >= 0 && tokens_host[i] < m->d.vocab, NT_ERR_INVALID_ARG,
               "token %lld outside the vocabulary", (long long)i);
  int dev_prev = 0;
  cudaGetDevice(&dev_prev);
  if (dev_prev != ctx->device) cudaSetDevice(ctx->device);
  cudaStream_t st = as_stream(stream);
  // the upload reads the model's own host copy of the tokens, so the caller's array is free once this call
  // returns; that copy is rewritten only after the previous upload from it has completed
  nt_status s = cuda_check(ctx, cudaEventSynchronize(m->ev_prompt), "previous prompt upload");
  if (!s) {
    m->prompt_host.assign(tokens_host, tokens_host + n);
    s = cuda_check(ctx, cudaMemcpyAsync(m->prompt, m->prompt_host.data(), sizeof(int32_t) * size_t(n),
                                        cudaMemcpyHostToDevice, st),
                   "prompt upload");
  }
  if (!s) s = cuda_check(ctx, cudaEventRecord(m->ev_prompt, st), "prompt upload event");
  // chunks of 16 prompt tokens when every GEMM of the model takes the
  // tensor-core form (its time hardly depends on the vector count, so each
  // weight pass serves twice the tokens); 8 otherwise
  const int chunk = prefill_chunk(ctx, m);
  for (int64_t base = 0; base < n && !s; base += chunk) {
    const int M = int(std::min<int64_t>(chunk, n - base));
    const bool last = base + M == n;
    s = cuda_check(ctx, launch_k(ctx, prefill_setup_kernel, dim3(1), dim3(32), 0, st, m->prompt + base, pos0 + base,
                                 m->spec_tok, m->spec_pos, M),
                   "prefill chunk setup");
    Streamer sm{ctx, m, st};
    if (!s) s = sm.begin(nullptr);
    if (!s) s = enqueue_multi(ctx, m, M, m->spec_tok, m->spec_pos, last ? m->lv : nullptr, false, sm, st);
    if (!s && last) {
      // the last token's logits; greedy next token and the device state for decoding on
      s = cuda_check(ctx, cudaMemcpyAsync(logits, m->lv + int64_t(M - 1) * m->d.vocab, sizeof(float) * m->d.vocab,
                                          cudaMemcpyDeviceToDevice, st),
                     "prefill logits");
      if (!s) {
        set_state_kernel<<<1, 1, 0, st>>>(m->tok, m->pos, 0, pos0 + n - 1);
        s = cuda_check(ctx, cudaGetLastError(), "prefill state");
      }
      if (!s)
        s = launch_argmax(ctx, logits, m->d.vocab, next_tok, m->amax_key, m->amax_cnt, st, m->tok, m->pos);
    }
  }
  if (dev_prev != ctx->device) cudaSetDevice(dev_prev);
  return s;
}

nt_status nt_model_set_sampler(nt_ctx* ctx, nt_model* m, float T, float P, uint64_t seed) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m, NT_ERR_INVALID_ARG, "null model");
  NT_REQUIRE(P > 0.f && P <= 1.f && !(T != T) && T < 3.0e38f, NT_ERR_INVALID_ARG, "top_p in (0, 1], finite temperature");
  NT_REQUIRE(!(T > 0.f) || m->d.vocab <= kSampMaxN, NT_ERR_INVALID_ARG, "the sampler takes at most %lld logits",
             (long long)kSampMaxN);
  m->temperature = T > 0.f ? T : 0.f;
  m->top_p = P;
  m->seed = seed;
  return NT_OK;
}

nt_status nt_plan_residency(const nt_model_desc* d, size_t budget, int embd_in_hbm, nt_residency_plan* out) {
  if (!d || !out) return NT_ERR_INVALID_ARG;
  const int fm[9] = {d->fmt_q, d->fmt_k, d->fmt_v, d->fmt_o, d->fmt_gate, d->fmt_up, d->fmt_down, d->fmt_embd,
                     d->fmt_out};
  for (int f : fm)
    if (!fmt_ok(f)) return NT_ERR_UNSUPPORTED_FMT;
  if (d->n_layers <= 0 || d->d_model <= 0 || d->vocab <= 0 || d->d_model % block_elems(d->fmt_out) ||
      d->d_model % block_elems(d->fmt_embd) || d->stream_slots < 0 || d->stream_slots > kMaxSlots)
    return NT_ERR_INVALID_ARG;
  size_t off[7], layer = 0;
  blob_layout(*d, off, &layer);
  const auto mat = [&](int fmt) {
    return size_t(d->vocab) * size_t(d->d_model / block_elems(fmt)) * size_t(block_bytes(fmt));
  };
  const size_t fixed = mat(d->fmt_out) + (embd_in_hbm ? mat(d->fmt_embd) : 0);
  const int slots = d->stream_slots ? d->stream_slots : 2;
  nt_residency_plan p{};
  p.layer_bytes = layer;
  p.fixed_bytes = fixed;
  if (fixed + size_t(d->n_layers) * layer <= budget) {
    p.n_resident = d->n_layers;  // everything fits: nothing streams
    p.stream_slots = 0;
  } else {
    const size_t need = fixed + size_t(slots) * layer;
    const size_t room = budget > need ? budget - need : 0;
    p.n_resident = int(std::min<size_t>(room / layer, size_t(d->n_layers - 1)));
    p.stream_slots = slots;
  }
  p.total_bytes = fixed + size_t(p.n_resident) * layer + size_t(p.stream_slots) * layer;
  *out = p;
  return NT_OK;
}

nt_status nt_stream_layer(nt_ctx* ctx, nt_model* m, int layer, const void* src, size_t bytes, int slot,
                          void* copy_stream) {
  NvtxRange nvtx_range("nt_stream_layer");
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m && src, NT_ERR_INVALID_ARG, "null model or source");
  NT_REQUIRE(m->n_slots > 0, NT_ERR_INVALID_ARG, "the model streams no layer");
  NT_REQUIRE(layer >= 0 && layer < m->d.n_layers && m->host_blob[layer], NT_ERR_INVALID_ARG,
             "layer %d is not a streamed layer", layer);
  NT_REQUIRE(slot >= 0 && slot < m->n_slots, NT_ERR_INVALID_ARG, "slot %d outside 0..%d", slot, m->n_slots - 1);
  NT_REQUIRE(bytes == m->blob_bytes, NT_ERR_INVALID_ARG, "bytes %zu, the layer blob is %zu", bytes, m->blob_bytes);
  cudaPointerAttributes pa{};
  const cudaError_t pe = cudaPointerGetAttributes(&pa, src);
  cudaGetLastError();
  NT_REQUIRE(pe == cudaSuccess && pa.type == cudaMemoryTypeHost, NT_ERR_INVALID_ARG,
             "the source must be page-locked host memory");
  int dev_prev = 0;
  cudaGetDevice(&dev_prev);
  if (dev_prev != ctx->device) cudaSetDevice(ctx->device);
  const nt_status s = copy_layer(ctx, m, layer, src, slot, as_stream(copy_stream));
  if (dev_prev != ctx->device) cudaSetDevice(dev_prev);
  return s;
}

nt_status nt_model_slot(nt_ctx* ctx, nt_model* m, int slot, void** dev, size_t* bytes, int* layer) {
  if (!ctx) return NT_ERR_INVALID_ARG;
  NT_REQUIRE(m, NT_ERR_INVALID_ARG, "null model");
  NT_REQUIRE(m->n_slots > 0, NT_ERR_INVALID_ARG, "the model streams no layer");
  NT_REQUIRE(slot >= 0 && slot < m->n_slots, NT_ERR_INVALID_ARG, "slot %d outside 0..%d", slot, m->n_slots - 1);
  if (dev) *dev = slot_ptr(m, slot);
  if (bytes) *bytes = m->blob_bytes;
  if (layer) *layer = m->slot_layer[slot];
  return NT_OK;
}

}  // extern "C"
