/*
 * nt.h — C ABI of libnt.so: batch-1 decode of a Llama-architecture
 * transformer whose linear weights are GGUF-style block-quantized, on one
 * GB300 (sm_103a).
 *
 * Passages the operations come from (page title, then section):
 *  [about]  "Ntransformer" (en.unwiki.net), About — GGUF formats Q4_0, Q8_0,
 *           Q4_K_M, Q5_K, Q6_K.
 *  [code]   "ntransformer - moteur d'inférence NVMe-to-GPU…" (fr.news.hada.io),
 *           "Architecture et structure du code" — cuda/: GEMV, RMSNorm, RoPE,
 *           SwiGLU and softmax kernels; model/: transformer composition,
 *           attention, FFN, normalisation; inference/: sampler, engine;
 *           memory/: layer streaming engine.
 *  [feat]   same page, "Fonctionnalités principales" — RoPE, GQA, SwiGLU,
 *           RMSNorm, KV cache; SLEP double-buffered streaming; self-speculative
 *           decoding with the VRAM-resident layers as the draft.
 *  [cache]  same page, "Performances et structure de cache" — layer skip by
 *           cosine similarity (20 of 80 layers); VRAM-resident layers and
 *           pinned-RAM H2D tiers.
 *  [road]   "Ntransformer" (en.unwiki.net), roadmap — F16 KV cache; public C
 *           API planned.
 *
 * Conventions shared by every entry point:
 *  - Every call returns nt_status.  Arguments are checked on the host first;
 *    a call that fails its checks launches nothing and leaves outputs as they
 *    were.  nt_last_error(ctx) then holds a one-line reason.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls only enqueue work.  The device error flag (a bounded
 *    wait inside a kernel that ran out, a device-held position past the KV
 *    cache) is read and cleared by nt_ctx_sync() and nt_stream_sync(); a
 *    CUDA fault also fails the next launch on the context.
 *  - Pointers named *_dev are device (HBM) pointers; pointers named *_host
 *    are host pointers.  The caller owns every weight, activation, KV-cache
 *    and output buffer; the context owns only its scratch, events, side
 *    streams and captured graphs.
 *  - A context, and every model made on it, is used from one host thread at
 *    a time (its tuning state, scratch and per-call settings are shared);
 *    separate contexts are independent.  Work from calls on one context that
 *    share scratch (the standalone kernels, the sampler) must not overlap
 *    on the GPU: keep it on one stream or order the streams.
 *  - Block-quantized matrices are row-major: row r is cols/block_elems
 *    consecutive blocks.  cols must be a multiple of the format's block size
 *    (32 for Q8_0/Q4_0/F16/F32, 256 for Q4_K/Q5_K/Q6_K).  Block bytes: Q8_0
 *    34, Q4_0 18, Q4_K 144, Q5_K 176, Q6_K 210, F16 64, F32 128; layouts are
 *    the GGUF ones.
 *  - Weight pointers must be 2-byte aligned.  When the weight pointer is
 *    16-byte aligned and each row is a multiple of 16 bytes, weights stream
 *    through TMA bulk copies; otherwise a slower plain-load path runs.
 *  - fp32 vectors must be 4-byte aligned; the GEMV / GEMM inputs (x, X),
 *    the norm gains and the attention q and out 16-byte aligned.
 */
#ifndef NT_H
#define NT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NT_OK = 0,
  NT_ERR_INVALID_ARG = 1,     /* null pointer, bad size, ragged cols, ... */
  NT_ERR_UNSUPPORTED_FMT = 2, /* format id outside nt_fmt */
  NT_ERR_ALIGNMENT = 3,       /* pointer alignment rule broken */
  NT_ERR_CUDA = 4,            /* a CUDA runtime call failed */
  NT_ERR_OOM = 5,             /* device or pinned allocation failed */
  NT_ERR_TIMEOUT = 6,         /* a host-side or device-side bounded wait ran out */
} nt_status;

/* Weight formats [about].  The quantized ones are GGUF blocks (block bytes
 * below); F16 / F32 rows are plain little-endian binary16 / binary32 values,
 * handled in units of 32 (their "block": 32 values, 64 / 128 bytes). */
typedef enum { NT_Q8_0 = 0, NT_Q4_0 = 1, NT_Q4_K = 2, NT_Q5_K = 3, NT_Q6_K = 4, NT_F16 = 5, NT_F32 = 6 } nt_fmt;

typedef struct nt_ctx nt_ctx;
typedef struct nt_model nt_model;

/* ---- context ------------------------------------------------------------ */

/* Context [road] (the planned public C API): create one on CUDA device
 * `device`.  scratch_bytes = 0 picks the default (64 MiB).  The context
 * allocates its scratch on the device. */
nt_status nt_ctx_create(nt_ctx** out, int device, size_t scratch_bytes);
nt_status nt_ctx_destroy(nt_ctx* ctx);
/* nt_last_error(NULL) describes this thread's last failed nt_ctx_create,
 * nt_file_open or nt_file_close (the calls made without a context). */
/* [road] Wait for all work of this context's device, then report any asynchronous
 * CUDA error or device-side flag and clear the flag: NT_ERR_TIMEOUT when a
 * bounded wait inside a kernel ran out; NT_ERR_INVALID_ARG when a position
 * held on the device (a decode step continued with token < 0) ran past the
 * KV cache — the kernels then wrote nothing outside the caches. */
nt_status nt_ctx_sync(nt_ctx* ctx);
/* [road] Wait at most timeout_us for the work enqueued on `stream` to finish (a
 * host-side poll with a deadline), then report like nt_ctx_sync:
 * NT_ERR_TIMEOUT when the deadline passes first (the work is not
 * cancelled; call again to keep waiting), else the device-side error flag
 * (bounded-wait timeout or position out of range), cleared when read. */
nt_status nt_stream_sync(nt_ctx* ctx, void* stream, int64_t timeout_us);
/* Fault injection for the streaming engine's tests ([feat] SLEP streaming;
 * host side only; nothing is ever made to fail on the GPU): the nth following
 * request to copy a layer blob into an HBM slot (nth = 0: the next one;
 * counted over nt_stream_layer and the copies a decode step enqueues) returns
 * NT_ERR_CUDA with nothing enqueued.  A decode step whose capture hits it
 * returns the error, keeps no graph and leaves the slot bookkeeping as it
 * was; the next call captures again.  nth = -1 disarms it. */
nt_status nt_debug_fail_copy(nt_ctx* ctx, int nth);
/* [road] Test hook for the device-side bounded waits (failure detection; no
 * GPU is made to fault or hang): the next n eager launches in this process
 * of the kernels that wait on bulk copies — the quant GEMV (nt_gemv_q,
 * nt_gemv_q_multi, nt_gemv_swiglu), nt_attn_decode and
 * nt_attn_decode_static — issue no copies, so their waits run out after a
 * few tries and take the timeout path: the context flag that nt_ctx_sync
 * reports as NT_ERR_TIMEOUT, or NaN output from nt_attn_decode_static.
 * Launches on a stream being captured are never armed.  n = 0 disarms;
 * n outside 0..1000 is NT_ERR_INVALID_ARG. */
nt_status nt_debug_stall_waits(int n);
/* [road] Test helper: a host callback on `stream` that sleeps `us` microseconds
 * (0..10 s), so that the stream stays busy without any GPU work. */
nt_status nt_debug_host_delay(nt_ctx* ctx, void* stream, int64_t us);
/* [road] The quant-GEMV launch plans this context has chosen, one line per
 * launch shape: "fmt/cols/swiglu/tma/rows0/rows1/rows2 -> warps=W
 * stage_max=B R=r ks=k".  A shape's arithmetic (R rows per lane group, ks
 * column parts, the segment granule) is fixed by the shape and the device's
 * SM count and shared memory alone; the first eager launch of a shape times
 * only launch shapes (warps, stage size) that leave every addition
 * unchanged, so results are bit-identical across processes and runs on the
 * same kind of GPU whichever plan the timing picks.  Writes at most cap
 * bytes (NUL-terminated) to out and the full size, NUL included, to *len;
 * out may be NULL when cap is 0. */
nt_status nt_ctx_gemv_plans(nt_ctx* ctx, char* out, size_t cap, size_t* len);
const char* nt_last_error(const nt_ctx* ctx);
/* [about] Bytes per block / elements per block of a format (0 for an unknown id). */
int nt_block_bytes(int fmt);
int nt_block_elems(int fmt);

/* ---- single ops ------------------------------------------------------------ */

/* Dequantise rows [row0, row0+nrows) of a rows x cols matrix into fp32
 * out_dev[nrows][cols].  Element values [about], GGUF reading:
 *   Q8_0 d*q;  Q4_0 d*(q-8);  Q4_K/Q5_K (d*sc)*q - dmin*m;  Q6_K d*(sc*(q-32)).
 * Each product is exact in fp32, so results are bit-identical to any
 * implementation that rounds the same single subtraction. */
nt_status nt_dequant_rows(nt_ctx* ctx, int fmt, const void* W_dev, int64_t row0, int64_t nrows, int64_t cols,
                          float* out_dev, void* stream);

/* Quant GEMV [code] cuda/ GEMV:  y[r] = sum_c deq(W[r,c]) * x[c]  (+ residual[r]),
 * r < rows, fp32 accumulation.  residual_dev may be NULL or equal y_dev.
 * Launch plans (warps per CTA, stage size, split of each row over warps)
 * are tuned per launch shape: the first call of a shape on a stream that is
 * not being captured times a few plans, writing only context scratch, then
 * synchronizes the stream and keeps the fastest.  Later calls, captured or
 * not, use that plan; a shape first seen inside a capture uses the default
 * plan.  The plan changes only the summation order (fp32 rounding). */
nt_status nt_gemv_q(nt_ctx* ctx, int fmt, const void* W_dev, const float* x_dev, float* y_dev, int64_t rows,
                    int64_t cols, const float* residual_dev, void* stream);

/* Gate/up GEMV with the SwiGLU epilogue [feat] SwiGLU:
 *   h[r] = silu(Wg[r,:] . x') * (Wu[r,:] . x'),  silu(z) = z / (1 + e^-z),
 * x' = x, or x / sqrt(mean(x^2) + eps) * g when norm_g_dev != NULL (the FFN
 * RMSNorm fused in front).  Wg and Wu share format and shape. */
nt_status nt_gemv_q_swiglu(nt_ctx* ctx, int fmt, const void* Wg_dev, const void* Wu_dev, const float* x_dev,
                           const float* norm_g_dev, float eps, float* h_dev, int64_t rows, int64_t cols,
                           void* stream);

/* One launch of several GEMVs sharing x (e.g. Q, K and V), optionally with the
 * RMSNorm of x fused in front:  x' = x / sqrt(mean(x^2) + eps) * g  when
 * norm_g_dev != NULL.  Up to 3 jobs, all of format fmt and width cols. */
typedef struct {
  const void* W_dev;
  float* y_dev;
  const float* residual_dev; /* nullable; may equal y_dev */
  int64_t rows;
} nt_gemv_job;
nt_status nt_gemv_q_multi(nt_ctx* ctx, int fmt, const nt_gemv_job* jobs, int njobs, const float* x_dev,
                          const float* norm_g_dev, float eps, int64_t cols, void* stream);

/* RMSNorm [feat]:  y = x / sqrt(mean(x^2) + eps) * g, fp32, n elements. */
nt_status nt_rmsnorm(nt_ctx* ctx, const float* x_dev, const float* g_dev, float* y_dev, int64_t n, float eps,
                     void* stream);

/* RoPE [feat] in place on q [n_qh][head_dim] and k [n_kvh][head_dim] (k may be
 * NULL): adjacent pairs (2i, 2i+1) turn by pos * theta^(-2i/head_dim). */
nt_status nt_rope(nt_ctx* ctx, float* q_dev, float* k_dev, int n_qh, int n_kvh, int head_dim, int64_t pos,
                  float theta, void* stream);

/* RoPE on q and k, then append k and v (fp32 -> binary16, round to nearest
 * even) to the F16 KV cache [road] at position pos.  Caches are laid out
 * [n_kvh][kv_stride][head_dim] (one layer). */
nt_status nt_rope_kv_append(nt_ctx* ctx, float* q_dev, const float* k_dev, const float* v_dev, void* kcache_dev,
                            void* vcache_dev, int n_qh, int n_kvh, int head_dim, int64_t pos, int64_t kv_stride,
                            float theta, void* stream);

/* Decode attention with grouped KV heads [feat] GQA over the F16 KV cache:
 * for q head h, KV head g = h / (n_qh / n_kvh):
 *   out_h = softmax_j(q_h . K_g[j] / sqrt(head_dim)) . V_g[j],  j < n_pos.
 * Split over positions (flash-decoding): one launch writes each split's
 * partial (max, sum, unnormalised output) to context scratch, a second
 * combines them.  head_dim must be 128, n_qh / n_kvh one of 1, 2, 4, 8, 16,
 * kv_stride at most 16384 positions. */
nt_status nt_attn_decode(nt_ctx* ctx, const float* q_dev, const void* kcache_dev, const void* vcache_dev,
                         float* out_dev, int n_qh, int n_kvh, int head_dim, int64_t n_pos, int64_t kv_stride,
                         void* stream);

/* Causal multi-query decode attention, the attention of the verify pass of
 * self-speculative decoding [feat]: n_query consecutive tokens whose K/V
 * are already in the caches; query i (0 <= i < n_query) attends to
 * positions 0 .. n_pos0 - 1 + i.  q_dev, out_dev fp32 [n_query][n_qh][128];
 * other arguments as nt_attn_decode; n_query 1..8, n_pos0 + n_query - 1 <=
 * kv_stride.  n_query = 1 is nt_attn_decode. */
nt_status nt_attn_verify(nt_ctx* ctx, const float* q_dev, const void* kcache_dev, const void* vcache_dev,
                         float* out_dev, int n_qh, int n_kvh, int head_dim, int64_t n_pos0, int n_query,
                         int64_t kv_stride, void* stream);

/* Softmax [code]: y = exp(x - max x) / sum, fp32, n elements (standalone). */
nt_status nt_softmax(nt_ctx* ctx, const float* x_dev, float* y_dev, int64_t n, void* stream);

/* SwiGLU [feat]: h = silu(gate) * up, fp32, n elements (standalone). */
nt_status nt_swiglu(nt_ctx* ctx, const float* gate_dev, const float* up_dev, float* h_dev, int64_t n,
                    void* stream);

/* Verify GEMM of self-speculative decoding [feat] (M = draft length + 1
 * tokens through one layer's weights at once): for m < M,
 *   Y_dev[m][r] = sum_c deq(W[r, c]) * xn_m[c] (+ residual_dev[m][r]),
 * xn_m = rmsnorm(X_dev[m], norm_g_dev, eps) when norm_g_dev is non-NULL,
 * else X_dev[m].  X_dev fp32 [M][cols] (16-byte aligned, cols a multiple of
 * 4), Y_dev and residual_dev fp32 [M][rows] (residual may equal Y).  Every
 * weight byte is read once for all M vectors.  Precision and layout rules
 * as nt_gemv_q.  M 1..8 for every format; M 1..16 for Q8_0, Q4_K and Q6_K
 * with rows of a multiple of 16 bytes at a 16-byte-aligned W_dev (the
 * tensor-core form; NT_ERR_INVALID_ARG otherwise, and under NT_GEMM_MMA=0).
 * Uses the context scratch beyond its first 32 MiB for partial sums:
 * NT_ERR_OOM when 4 * M * rows * P bytes do not fit, P the column parts
 * (ceil(cols / 2048) for the integer form, 1024 for F16, 512 for F32; the
 * tensor-core form narrows its parts for small matrices, at most to one
 * staged segment: 512 columns for Q8_0 and Q6_K, 1024 for Q4_K). */
nt_status nt_gemm_q(nt_ctx* ctx, int fmt, const void* W_dev, const float* X_dev, float* Y_dev, int64_t rows,
                    int64_t cols, int M, const float* residual_dev, const float* norm_g_dev, float eps,
                    void* stream);

/* Greedy sampler [code] inference/: index of the largest of v[0..n), lowest
 * index on ties (NaN never wins), written as int32 to out_dev. */
nt_status nt_argmax(nt_ctx* ctx, const float* v_dev, int64_t n, int32_t* out_dev, void* stream);

/* Non-greedy sampler [code] inference/ (sampler): temperature and nucleus
 * (top-p) sampling of logits_dev[0..n) into *out_dev.  Definition:
 * w_i = rint(exp((z_i - max z) / temperature) * 2^40) (integer weights);
 * the nucleus is the shortest prefix of the tokens ordered by logit
 * (descending, ties by lower index) whose weight reaches
 * ceil(top_p * sum w); with u = (splitmix64(seed ^ (counter << 1)) >> 40) *
 * 2^-24 (SplitMix64 output function: Steele, Lea & Flood 2014) and
 * r = floor(u * nucleus weight), the pick is the nucleus token, in index
 * order, whose cumulative weight first exceeds r.  temperature <= 0 is
 * greedy (nt_argmax).  top_p in (0, 1]; n 1..1,024,000.  Six launches over
 * up to 256 CTAs (one for greedy); the state between them lives in context
 * scratch at 20 MiB, so calls on one context must not overlap on the GPU. */
nt_status nt_sample(nt_ctx* ctx, const float* logits_dev, int64_t n, float temperature, float top_p, uint64_t seed,
                    uint64_t counter, int32_t* out_dev, void* stream);

/* Cosine similarity [cache] of a and b: <a,b> / (|a| |b|), fp32 result. */
nt_status nt_cos_sim(nt_ctx* ctx, const float* a_dev, const float* b_dev, int64_t n, float* out_dev,
                     void* stream);


/* ---- whole decode step ------------------------------------------------------ */

/* Shapes and per-tensor formats of a Llama-architecture model [feat]
 * (Q4_K_M = attn_v and ffn_down in Q6_K, the rest in Q4_K [about]). */
typedef struct {
  int n_layers, d_model, n_qh, n_kvh, head_dim, ffn, vocab;
  float eps, theta;
  int64_t kv_cap;                       /* positions per (layer, KV head) in the caches, <= 16384 */
  int fmt_q, fmt_k, fmt_v, fmt_o, fmt_gate, fmt_up, fmt_down, fmt_embd, fmt_out;
  int stream_slots;                     /* HBM slots for streamed layers: 0 = 2 (double buffering), max 8 */
} nt_model_desc;

/* Pointers of one layer.  Weights: row-major block matrices
 * wq [n_qh*hd x d], wk/wv [n_kvh*hd x d], wo [d x n_qh*hd], wg/wu [ffn x d],
 * wd [d x ffn]; norms fp32 [d]; caches binary16 [n_kvh][kv_cap][head_dim];
 * norms and caches always in HBM.
 * A resident layer sets all seven weight pointers (HBM) and host_blob NULL.
 * A streamed layer [feat] (pinned-RAM tier [cache]) sets the seven weight
 * pointers NULL and host_blob to page-locked host memory holding its weights
 * in the blob layout of nt_layer_blob_layout; every decode step copies it
 * into one of the model's HBM slots while earlier layers compute. */
typedef struct {
  const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;
  const float *attn_norm, *ffn_norm;
  void *kcache, *vcache;
  const void* host_blob;
} nt_layer_ptrs;

/* [feat] (SLEP layer streaming) Byte layout of one layer's weights as one
 * contiguous blob (the unit the streaming engine copies): offsets_out[0..6] =
 * offsets of wq, wk, wv, wo, wg, wu, wd, each a multiple of 256;
 * *blob_bytes_out = total size (a multiple of 256).  Pure host computation
 * from the descriptor. */
nt_status nt_layer_blob_layout(const nt_model_desc* desc, size_t offsets_out[7], size_t* blob_bytes_out);

/* [code] (model/: transformer composition) Bind a model: copies the
 * descriptor and the pointer table (the buffers stay the caller's) and
 * allocates the model's activations and step state on the device, plus, when
 * a layer is streamed, desc->stream_slots HBM slots of one blob each, a copy
 * stream and its events.  embd [vocab x d] and out [vocab x d] are block
 * matrices, out_norm fp32 [d].  embd may live in page-locked host memory: the
 * step reads one row of it per token. */
nt_status nt_model_init(nt_ctx* ctx, const nt_model_desc* desc, const nt_layer_ptrs* layers, const void* embd_dev,
                        const void* out_dev, const float* out_norm_dev, nt_model** out);
nt_status nt_model_destroy(nt_ctx* ctx, nt_model* model);

/* One batch-1 decode step [code] model/ + inference/ + memory/:
 *   x = embd[token];  per layer l with skip_mask_host[l] == 0:
 *     q,k,v = W{q,k,v} rmsnorm(x, g_attn); rope(q, k, pos); K/V[l][:,pos] = f16(k, v)
 *     x += Wo attn(q, K/V[l][:, :pos+1]);  x += Wd (silu(Wg xn) * (Wu xn)), xn = rmsnorm(x, g_ffn)
 *   logits_dev = Wout rmsnorm(x, g_out);  next = argmax(logits) (lowest index on ties)
 * token >= 0: start from (token, pos).  token < 0: continue on the device
 * from the previous step (token = its argmax, pos = its pos + 1) with no host
 * round trip.  next_token_dev (nullable) receives the argmax.  Each distinct
 * (skip mask, sampler setting, next_token given or not) is captured once
 * into a CUDA graph and replayed; the graph computes into the model's own
 * buffers and ends by copying the logits (and the token) to the caller's,
 * so fresh logits_dev / next_token_dev pointers on every call re-point those
 * copies and capture nothing new (nt_model_graph_count stays constant).
 * skip_mask_host is n_layers bytes or NULL.  Before the first
 * capture of a graph, a dry pass tunes the GEMV plans of its shapes on
 * `stream` (see nt_gemv_q), which synchronizes that stream once.
 * Streamed layers: inside the same graph, executed streamed layer i (in layer
 * order) is copied into slot i mod stream_slots on the model's copy stream;
 * the first stream_slots copies start with the step and overlap the
 * resident layers, every later copy waits for the compute of the layer that
 * last occupied its slot, and each streamed layer's compute waits for its
 * copy (double buffering with 2 slots).  Skipped layers are not copied. */
nt_status nt_decode_step(nt_ctx* ctx, nt_model* model, int32_t token, int64_t pos, const uint8_t* skip_mask_host,
                         float* logits_dev, int32_t* next_token_dev, void* stream);
/* [road] The number of step graphs the model holds (decode and speculative
 * steps): one per distinct skip mask, sampler setting and output shape. */
nt_status nt_model_graph_count(nt_ctx* ctx, nt_model* model, int* n);

/* [code] (inference/: sampler) Sampling for the model's decode steps
 * (nt_decode_step, nt_prefill's next token stays greedy): every later step
 * draws its next token with nt_sample's definition, counter = the position of
 * the step's input token, so a sequence is reproducible from (seed, start).
 * temperature <= 0 restores greedy decoding.  nt_spec_step then samples too
 * (speculative sampling). With temperature > 0 the vocabulary must be at most
 * 1,024,000. */
nt_status nt_model_set_sampler(nt_ctx* ctx, nt_model* model, float temperature, float top_p, uint64_t seed);

/* Layer-skip calibration [cache]: one full decode step (all layers) at
 * (token, pos) that also measures cos(x before layer l, x after layer l) for
 * every layer; marks the n_skip layers with the highest cosine (ties: lower
 * index) in skip_mask_host[n_layers].  cos_host (nullable) gets the cosines.
 * Synchronous on `stream`. */
nt_status nt_layer_skip_calibrate(nt_ctx* ctx, nt_model* model, int32_t token, int64_t pos, int n_skip,
                                  uint8_t* skip_mask_host, float* cos_host, float* logits_dev,
                                  int32_t* next_token_dev, void* stream);

/* Prompt prefill [feat] (KV cache): run tokens_host[0..n) at positions
 * pos0 .. pos0 + n - 1 through every layer, writing their K/V into the
 * caches, in chunks of up to 16 tokens (8 when a GEMM of the model cannot
 * take the tensor-core form: a format other than Q8_0 / Q4_K / Q6_K, rows
 * not a multiple of 16 bytes, or a resident weight not 16-byte aligned) —
 * each chunk one pass of the M-vector GEMMs and the causal multi-query
 * attention of the verify step (weights read once per chunk).  logits_dev receives the logits after the last
 * token, next_token_dev (nullable) their argmax, and the device state
 * becomes (that argmax, pos0 + n): nt_decode_step with token < 0 continues
 * from there.  Runs eagerly on `stream` (no graph); streamed layers stream
 * once per chunk.  tokens_host is read before the call returns. */
nt_status nt_prefill(nt_ctx* ctx, nt_model* model, const int32_t* tokens_host, int64_t n, int64_t pos0,
                     float* logits_dev, int32_t* next_token_dev, void* stream);

/* Prompt tokens per nt_prefill pass [feat] (KV cache): 16 when every GEMM of
 * the model's step takes the tensor-core form, else 8 (the rule above).
 * Writes it to *chunk; NT_ERR_INVALID_ARG for a NULL model or chunk. */
nt_status nt_model_prefill_chunk(nt_ctx* ctx, nt_model* model, int* chunk);

/* Resident-layer planner [about] (3-tier adaptive caching: VRAM-resident
 * layers first, the rest from pinned RAM) [cache] (the format decides how
 * many layers fit: "36 vs 26" for Q4_K_M vs Q6_K on the pages' card): how
 * many leading layers keep their weights in HBM when the weights may use
 * at most hbm_weight_budget bytes — the LM head, the embedding table when
 * embd_in_hbm, the resident layers and, if any layer is streamed,
 * stream_slots (0 = 2) slots of one layer blob.  KV caches and activations
 * are outside this budget.  Pure host arithmetic from the descriptor. */
typedef struct {
  int n_resident;      /* layers 0..n_resident-1 resident, the rest streamed */
  int stream_slots;    /* slots the plan reserves (0 when nothing streams) */
  size_t layer_bytes;  /* one layer's weights: the blob of nt_layer_blob_layout */
  size_t fixed_bytes;  /* LM head (+ embedding table) */
  size_t total_bytes;  /* fixed + resident layers + slots, <= the budget unless nothing fits */
} nt_residency_plan;
nt_status nt_plan_residency(const nt_model_desc* desc, size_t hbm_weight_budget, int embd_in_hbm,
                            nt_residency_plan* plan_out);

/* Host-file tier [about] (3-tier adaptive caching: NVMe/mmap fallback;
 * "mmap pinned" data path): page-lock bytes [host_ptr, host_ptr + bytes) of
 * host memory — typically a read-only mmap of a model file — so streamed
 * layers (nt_layer_ptrs.host_blob) and the embedding table can point into
 * it and copy like pinned RAM.  host_ptr and bytes must be multiples of 4096;
 * read_only != 0 registers read-only (what a PROT_READ mapping needs).
 * nt_host_unregister releases it; the caller unregisters before unmapping. */
nt_status nt_host_register(nt_ctx* ctx, const void* host_ptr, size_t bytes, int read_only);
nt_status nt_host_unregister(nt_ctx* ctx, const void* host_ptr);

/* ---- host-file tier: model files ----------------------------------------- */

/* A model file [about] (3-tier adaptive caching: NVMe/mmap fallback), the
 * GGUF-style container of one model's weights:
 *   offset 0   "NTQF", u32 version (1), u64 header length H (little-endian)
 *   offset 16  H bytes of JSON: {"spec": {n_layers, d_model, n_qh, n_kvh,
 *              head_dim, ffn, vocab, eps, theta, fmt: {wq, wk, wv, wo, wg,
 *              wu, wd, embd, out: nt_fmt ids}, ...}, "blob_offsets": [7],
 *              "blob_bytes": N, "entries": {name: [offset, bytes], ...}}
 *   data       from the first multiple of 4096 after the header, entries at
 *              4096-aligned offsets (relative to it): "embd", "out",
 *              "out_norm" (fp32 [d]), and per layer l "blob.l" (its seven
 *              weight matrices in the layout of nt_layer_blob_layout, so a
 *              streamed layer is one contiguous range), "attn_norm.l",
 *              "ffn_norm.l" (fp32 [d]).
 * The KV cache is runtime state, not part of the file.  An nt_file, like a
 * context, is used from one host thread at a time. */
typedef struct nt_file nt_file;

/* Rungs of nt_file_lock, in the pages' order of preference
 * [feat] ("mmap pinned > CPU memcpy"). */
enum { NT_FILE_MMAP_PINNED = 0, NT_FILE_MMAP_PINNED_PRIVATE = 1, NT_FILE_CPU_MEMCPY = 2 };

/* [about] (NVMe/mmap fallback) Open a model file: map it read-only (shared)
 * and check it before anything is handed out — the preamble, the header's
 * JSON, every field the descriptor needs, the blob layout against this
 * library's, and every entry a model needs, with the size its shape gives,
 * 4096-aligned and (rounded up to 4096 bytes) inside the file.  A file that
 * fails a check is refused with NT_ERR_INVALID_ARG; nt_last_error(NULL) then
 * holds the reason on the calling thread.  Host-only: needs no GPU and no
 * context.  The caller owns *out and closes it with nt_file_close. */
nt_status nt_file_open(const char* path, nt_file** out);
/* [about] (NVMe/mmap fallback) Unmap and free.  Refused (NT_ERR_INVALID_ARG, reason in nt_last_error(NULL))
 * while an entry is still page-locked: nt_file_unlock each first. */
nt_status nt_file_close(nt_file* f);
/* [about] The descriptor stored in the file; kv_cap and stream_slots are 0 (runtime
 * choices the caller sets before nt_model_init). */
nt_status nt_file_desc(const nt_file* f, nt_model_desc* desc);
/* [about] The header's JSON text (NUL-terminated, owned by f, valid until
 * nt_file_close); *len (nullable) gets its length. */
nt_status nt_file_header(const nt_file* f, const char** text, size_t* len);
/* [about] Entry `name`: its address in the read-only mapping (*host_ptr; reading it
 * faults the pages in from the file), its offset from the start of the file
 * and its size.  Each output is nullable.  NT_ERR_INVALID_ARG for an unknown
 * name.  Resident weights are uploaded from here by the caller. */
nt_status nt_file_entry(const nt_file* f, const char* name, const void** host_ptr, uint64_t* offset,
                        size_t* bytes);
/* [feat] ("mmap pinned" data path) Page-lock entry `name` (its size rounded
 * up to 4096 bytes) for streaming, taking the first rung the operating
 * system and driver accept:
 *   NT_FILE_MMAP_PINNED          the read-only mapping itself, registered read-only;
 *   NT_FILE_MMAP_PINNED_PRIVATE  a private, writable, pre-faulted mapping of the
 *                                range (copy-on-write: the file is never written),
 *                                registered without the read-only flag;
 *   NT_FILE_CPU_MEMCPY           (only when allow_copy) one CPU copy into
 *                                page-locked memory (tail bytes zero).
 * *pinned_out gets the page-locked address to stream from (a layer's
 * nt_layer_ptrs.host_blob, the embedding table of nt_model_init), *rung_out
 * (nullable) the rung.  Locking a locked entry returns the same address.
 * NT_ERR_CUDA when neither mapping can be locked and allow_copy is 0;
 * NT_ERR_OOM when the copy cannot be allocated. */
nt_status nt_file_lock(nt_ctx* ctx, nt_file* f, const char* name, int allow_copy, const void** pinned_out,
                       int* rung_out);
/* [feat] ("mmap pinned" data path) Release what nt_file_lock took for `name` (unregister, unmap the private
 * mapping or free the copy).  Call it with the context the entry was locked
 * with, before destroying that context, once no stream still copies from it. */
nt_status nt_file_unlock(nt_ctx* ctx, nt_file* f, const char* name);
/* [feat] ("mmap pinned > CPU memcpy") Test hook for the rung order, host
 * side only: on = 1 makes every following nt_file_lock in this process treat
 * both in-place rungs as refused, so it takes NT_FILE_CPU_MEMCPY (or fails
 * with NT_ERR_CUDA when the copy is not allowed); on = 0 restores the order.
 * Any other value is NT_ERR_INVALID_ARG. */
nt_status nt_debug_file_refuse_in_place(int on);

/* Streaming-engine copy step [feat] (SLEP double buffering), [cache]
 * (pinned-RAM H2D tier): enqueue on copy_stream the host-to-HBM copy of one
 * layer blob of `bytes` (= the model's blob size) from page-locked
 * host_pinned_src into HBM slot `slot`.  `layer` must be a streamed layer of
 * the model; it is recorded as the slot's occupant.  Ordering is the
 * caller's: copy_stream must already wait for every kernel still reading the
 * slot.  nt_decode_step runs this copy itself for each streamed layer; the
 * call is for staging a layer outside a step (read the slot through
 * nt_model_slot). */
nt_status nt_stream_layer(nt_ctx* ctx, nt_model* model, int layer, const void* host_pinned_src, size_t bytes,
                          int slot, void* copy_stream);

/* [feat] (SLEP double buffering) HBM address and size of streaming slot
 * `slot`, and the layer last copied into it (-1: none yet).
 * NT_ERR_INVALID_ARG when the model streams no layer or slot is out of range. */
nt_status nt_model_slot(nt_ctx* ctx, nt_model* model, int slot, void** slot_dev_out, size_t* bytes_out,
                        int* layer_out);

/* Self-speculative decoding step [feat] (the VRAM-resident layers are the
 * draft model): from (token, pos) — or, token < 0, from the device state
 * left by the previous step — draft k tokens greedily with layers
 * [0, n_draft_layers) (n_draft_layers = 0: every resident, i.e. not
 * streamed, layer) followed by the final norm, LM head and argmax; then
 * verify [token, d_1 .. d_k] at positions pos .. pos + k in one pass of all
 * layers (M = k + 1 GEMMs, causal attention among the k + 1 queries).  With
 * v_i the argmax of verify row i, d_{i+1} is accepted while d_{i+1} == v_i;
 * with n accepted, tokens_out_dev[0..n] = v_0 .. v_n (the greedy tokens) and
 * *n_out_dev = n + 1, and the device state moves to (v_n, pos + n + 1).  The
 * KV entries written past the accepted ones are overwritten by later steps.
 * logits_dev (nullable) receives the verify logits [k + 1][vocab].  k is
 * 1..7; pos + k < kv_cap.  Streamed layers stream in the verify pass as in
 * nt_decode_step.  One CUDA graph per (k, n_draft_layers, logits given or
 * not, sampler); the outputs are copied to the caller's buffers at the end
 * of the graph, so new output pointers capture nothing new.
 *
 * With the model's sampler set (nt_model_set_sampler, temperature > 0) the
 * step is speculative sampling (Leviathan, Kalman & Matias 2023, section
 * 2.3), whose output follows the target model's sampler distribution:
 *  - draft d_{i+1} is nt_sample's pick from the draft logits at position
 *    pos + i (counter pos + i); q_i, p_i are the nucleus distributions of the
 *    draft row and of verify row i, as integer weights w and their sum W;
 *  - d_{i+1} is accepted when k_acc * wq(d) * Wp < 2^24 * wp(d) * Wq, i.e.
 *    u < p_i(d) / q_i(d); at the first rejection the step's last token is the
 *    index-order pick at floor(k_res * sum R / 2^24) of the residual
 *    R_t = max(0, wp_t * Wq - wq_t * Wp); with all k accepted it is
 *    nt_sample's pick from verify row k (counter pos + k);
 *  - k_acc = bits 40..63 and k_res = bits 16..39 of
 *    splitmix64(seed ^ (2 (pos + i) + 1)).
 * tokens_out_dev gets the accepted drafts then that last token, *n_out_dev
 * their count, and logits_dev (when given) must hold 2k + 1 rows: the k + 1
 * verify rows, then the k draft rows. */
nt_status nt_spec_step(nt_ctx* ctx, nt_model* model, int32_t token, int64_t pos, int k, int n_draft_layers,
                       int32_t* tokens_out_dev, int32_t* n_out_dev, float* logits_dev, void* stream);

/* ---- allocation-free attention ------------------------------------------------ */

/* nt_attn_decode without a context and without any device allocation.  The
 * pages have no counterpart for this form; it exists for callers that cannot
 * call cudaMalloc — code running while a stream is captured into a CUDA graph
 * in a mode that forbids allocation, and hosts whose device memory is handed
 * out only by their own pool (an nt_ctx allocates its scratch, so such
 * callers cannot create one).
 *
 * Same operation, arguments and result as nt_attn_decode, on the calling
 * thread's current device.  The split partials and the error word live in
 * one fixed 4 MiB array compiled into the library
 * (every GPU that loads the library holds it until the process exits);
 * n_kvh * S * (n_qh / n_kvh) * 132 * 4 + 512 bytes must fit in it, where
 * S = min(128, max(ceil(SMs / n_kvh), ceil(kv_stride / 128))) — e.g. 64 q
 * heads over 8 KV heads fit for kv_stride up to 15,872 positions.  Larger
 * shapes return NT_ERR_INVALID_ARG before any launch.
 *  - The first call on a device looks up the array's device address and sets
 *    the kernel's shared-memory limit; make that first call before any stream
 *    capture.
 *  - Each device has its own copy of the array, shared by every call on that
 *    device: calls whose work overlaps on one device (different streams, or
 *    threads sharing the device) race on it — serialize them.  Calls on
 *    different devices do not interact.
 *  - Returns NT_OK once the work is enqueued (each enqueue's own status, not
 *    an error left by earlier unrelated work).  There is no context to carry
 *    an asynchronous error: a device-side wait that runs out makes this
 *    call's output NaN.  The array's error word is cleared at the start of
 *    every call, so a later call is unaffected. */
nt_status nt_attn_decode_static(const float* q_dev, const void* kcache_dev, const void* vcache_dev, float* out_dev,
                                int n_qh, int n_kvh, int head_dim, int64_t n_pos, int64_t kv_stride, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NT_H */
