// dequant.cu — dequantisation of whole rows of the weight formats named on
// "Ntransformer" (en.unwiki.net), About: the embedding-row lookup of the
// decode step and the bit-exact dequantisation entry point.  Element values
// (GGUF reading): Q8_0 d*q; Q4_0 d*(q-8); Q4_K/Q5_K (d*sc)*q - dmin*m;
// Q6_K d*(sc*(q-32)); F16 / F32 the value itself.  Every product is exact in
// fp32, only the K-quant subtraction rounds.
#include "nt_internal.cuh"
#include "ops.cuh"

namespace nt {
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

// element i of block b, exactly as the formats define it (every product exact
// in fp32; only the K-quant subtraction rounds)
__device__ __forceinline__ float elem_value(int fmt, const uint8_t* b, int i) {
  switch (fmt) {
    case NT_Q8_0: return __fmul_rn(__half2float(*reinterpret_cast<const __half*>(b)), float(quant_of(fmt, b, i)));
    case NT_Q4_0:
      return __fmul_rn(__half2float(*reinterpret_cast<const __half*>(b)), float(quant_of(fmt, b, i) - 8));
    case NT_Q4_K:
    case NT_Q5_K: {
      int sc, m;
      kq_sm(b + 4, i >> 5, sc, m);
      const float d = __half2float(*reinterpret_cast<const __half*>(b));
      const float dm = __half2float(*reinterpret_cast<const __half*>(b + 2));
      return __fsub_rn(__fmul_rn(__fmul_rn(d, float(sc)), float(quant_of(fmt, b, i))), __fmul_rn(dm, float(m)));
    }
    case NT_Q6_K: {
      const int s = int(int8_t(b[192 + (i >> 7) * 8 + ((i & 127) >> 4)]));
      return __fmul_rn(__half2float(*reinterpret_cast<const __half*>(b + 208)), float(s * (quant_of(fmt, b, i) - 32)));
    }
    case NT_F16: return __half2float(*reinterpret_cast<const __half*>(b + 2 * i));
    default: return *reinterpret_cast<const float*>(b + 4 * i);
  }
}

__global__ void dequant_kernel(int fmt, const uint8_t* W, int64_t row0, int64_t nrows, int64_t cols, float* out) {
  const int BE = block_elems(fmt), BB = block_bytes(fmt);
  const int64_t nb = cols / BE;
  const int64_t total = nrows * cols;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = e / cols, col = e % cols;
    out[e] = elem_value(fmt, W + ((row0 + r) * nb + col / BE) * BB, int(col % BE));
  }
}

// rows token_dev[m] of an embedding table, dequantised into out[m][cols]
// (m = blockIdx.y; tokens read on the device)
__global__ void embed_kernel(int fmt, const uint8_t* W, int64_t cols, const int32_t* token_dev, float* out) {
  pdl_wait();
  pdl_trigger();
  const int64_t row = token_dev[blockIdx.y];
  out += int64_t(blockIdx.y) * cols;
  const int BE = block_elems(fmt), BB = block_bytes(fmt);
  const int64_t nb = cols / BE;
  for (int64_t col = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; col < cols; col += int64_t(gridDim.x) * blockDim.x)
    out[col] = elem_value(fmt, W + (row * nb + col / BE) * BB, int(col % BE));
}

}  // namespace

nt_status launch_embed(Ctx* c, int fmt, const void* W, int64_t cols, const int32_t* token_dev, float* out,
                       cudaStream_t st, int M) {
  if (c->dry) return NT_OK;
  const int blocks = int((cols + 255) / 256);
  return cuda_check(c, launch_k(c, embed_kernel, dim3(blocks, M), dim3(256), 0, st, fmt, static_cast<const uint8_t*>(W),
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
