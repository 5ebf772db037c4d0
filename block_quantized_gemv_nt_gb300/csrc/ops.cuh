// ops.cuh — launchers of the kernels in qgemv.cu and ops.cu (arguments are
// validated by the C ABI layer before any of these runs).
#pragma once
#include "nt_internal.cuh"

namespace nt {

nt_status launch_dequant(Ctx* c, int fmt, const void* W, int64_t row0, int64_t nrows, int64_t cols, float* out,
                         cudaStream_t st);
// out[m][cols] = dequantised row token_dev[m], m < M
nt_status launch_embed(Ctx* c, int fmt, const void* W, int64_t cols, const int32_t* token_dev, float* out,
                       cudaStream_t st, int M = 1);
nt_status launch_rmsnorm(Ctx* c, const float* x, const float* g, float* y, int64_t n, float eps, cudaStream_t st);
nt_status launch_rope(Ctx* c, float* q, float* k, int n_qh, int n_kvh, int hd, int64_t pos, float theta,
                      cudaStream_t st);
nt_status launch_rope_append(Ctx* c, float* q, const float* k, const float* v, void* kc, void* vc, int n_qh,
                             int n_kvh, int hd, int64_t pos, const int64_t* pos_dev, int64_t kv_stride, float theta,
                             cudaStream_t st);
int attn_splits(const Ctx* c, int n_kvh, int64_t kv_stride);
int64_t attn_max_stride();
// a reserved head of kAttnCounterBytes (unused since the combine became its own
// launch) followed by the partials of nq queries
size_t attn_scratch_bytes(int n_qh, int n_kvh, int S, int nq = 1);
size_t attn_part_floats(int n_qh, int n_kvh, int S);
// nq queries: query i sees n_pos + i positions (pos_dev set: *pos_dev + 1 + i);
// q, out [nq][n_qh * 128]; part [nq][attn_part_floats].  Two launches: the
// split kernel, then the combine of its partials.
nt_status launch_attn(Ctx* c, const float* q, const void* K, const void* V, float* out, int n_qh, int n_kvh,
                      int64_t n_pos, const int64_t* pos_dev, int64_t kv_stride, float* part, int S, cudaStream_t st,
                      int nq = 1);
nt_status launch_softmax(Ctx* c, const float* x, float* y, int64_t n, cudaStream_t st);
nt_status launch_swiglu(Ctx* c, const float* g, const float* u, float* h, int64_t n, cudaStream_t st);
nt_status launch_argmax(Ctx* c, const float* v, int64_t n, int32_t* out, unsigned long long* key, unsigned* counter,
                        cudaStream_t st, int32_t* tok_state = nullptr, int64_t* pos_state = nullptr);
// nucleus sample of rows z[row][0..n), row < rows: temperature T (<= 0:
// greedy), top-p P, uniform from (seed, counter), counter = ctr_dev[row] when
// ctr_dev is set, else ctr + row; state: rows x kSampRowBytes, zero at rest
// (the launches leave it so).  tok_state / pos_state (one row): the pick also
// becomes the model's token and its position advances.  w_out [rows][n] /
// W_out [rows] (nullable, T > 0): each token's weight inside the nucleus
// (else 0) and the nucleus weight.
nt_status launch_sample(Ctx* c, const float* z, int64_t n, int rows, float T, float P, uint64_t seed,
                        const int64_t* ctr_dev, int64_t ctr, int32_t* out, void* state, cudaStream_t st,
                        int32_t* tok_state = nullptr, int64_t* pos_state = nullptr,
                        unsigned long long* w_out = nullptr, unsigned long long* W_out = nullptr);
nt_status configure_gemv(Ctx* c);
nt_status configure_gemm(Ctx* c);
int gemm_parts(int fmt, int64_t cols);
size_t gemm_scratch_bytes(int fmt, int64_t total_rows, int64_t cols, int M);
// whether launch_gemm takes more than kMaxVerify vectors for this format and
// width (the tensor-core form, with rows at 16-byte-aligned addresses)
bool gemm_wide_ok(const Ctx* c, int fmt, int64_t cols);
nt_status launch_gemm(Ctx* c, int fmt, const GemmJobEx* jobs, int njobs, bool swiglu, const float* X, int64_t ldx,
                      int M, const float* norm_g, float eps, int64_t cols, const RopeArgs* rope, float* part,
                      size_t part_bytes, cudaStream_t st);
nt_status launch_inv_freq(Ctx* c, double* out, int head_dim, float theta, cudaStream_t st);
nt_status configure_ops(Ctx* c);
nt_status launch_cos(Ctx* c, const float* a, const float* b, int64_t n, float* out, cudaStream_t st);

}  // namespace nt
