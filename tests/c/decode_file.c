/*
 * decode_file.c — a C caller of libnt.so, with no Python anywhere: the
 * public C API ("Ntransformer" (en.unwiki.net), roadmap: a public C API)
 * driving the host-file tier ("Ntransformer", About: NVMe/mmap fallback)
 * end to end.
 *
 *   decode_file MODEL_FILE N_RESIDENT KV_CAP N_DECODE OUT_FILE TOKEN...
 *
 * Opens the model file, uploads layers 0..N_RESIDENT-1 (and the LM head) to
 * HBM from the file's read-only mapping, page-locks the other layers' blobs
 * (and the embedding table) in place for streaming, binds the model with
 * zeroed KV caches of KV_CAP positions, prefills the prompt TOKEN... from
 * position 0, then decodes N_DECODE greedy steps on the device.  OUT_FILE
 * receives 1 + N_DECODE rows of vocab float32 logits: after the prompt,
 * then after each step.  Exit status 0 on success; on any failure the
 * call, its status and nt_last_error go to stderr and the status is 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "nt.h"

static nt_ctx* g_ctx;

#define NT(call)                                                                                     \
  do {                                                                                               \
    nt_status s_ = (call);                                                                           \
    if (s_ != NT_OK) {                                                                               \
      fprintf(stderr, "%s:%d: %s -> %d: %s\n", __FILE__, __LINE__, #call, (int)s_, nt_last_error(g_ctx)); \
      exit(1);                                                                                       \
    }                                                                                                \
  } while (0)

#define CU(call)                                                                                     \
  do {                                                                                               \
    cudaError_t e_ = (call);                                                                         \
    if (e_ != cudaSuccess) {                                                                         \
      fprintf(stderr, "%s:%d: %s: %s\n", __FILE__, __LINE__, #call, cudaGetErrorString(e_));         \
      exit(1);                                                                                       \
    }                                                                                                \
  } while (0)

/* a device copy of entry `name` of the file */
static void* upload(const nt_file* f, const char* name) {
  const void* host = NULL;
  size_t n = 0;
  void* dev = NULL;
  NT(nt_file_entry(f, name, &host, NULL, &n));
  CU(cudaMalloc(&dev, n));
  CU(cudaMemcpy(dev, host, n, cudaMemcpyHostToDevice));
  return dev;
}

int main(int argc, char** argv) {
  if (argc < 7) {
    fprintf(stderr, "usage: %s MODEL_FILE N_RESIDENT KV_CAP N_DECODE OUT_FILE TOKEN...\n", argv[0]);
    return 2;
  }
  const char* path = argv[1];
  const int n_resident = atoi(argv[2]);
  const int64_t kv_cap = atoll(argv[3]);
  const int n_decode = atoi(argv[4]);
  const char* out_path = argv[5];
  const int n_prompt = argc - 6;
  int32_t* prompt = malloc(sizeof(int32_t) * (size_t)n_prompt);
  for (int i = 0; i < n_prompt; ++i) prompt[i] = (int32_t)atoi(argv[6 + i]);

  NT(nt_ctx_create(&g_ctx, 0, 0));
  nt_file* f = NULL;
  NT(nt_file_open(path, &f));
  nt_model_desc d;
  NT(nt_file_desc(f, &d));
  d.kv_cap = kv_cap;  /* runtime choices: the file holds weights only */
  d.stream_slots = 0;
  size_t offs[7], blob_bytes = 0;
  NT(nt_layer_blob_layout(&d, offs, &blob_bytes));

  const int L = d.n_layers;
  nt_layer_ptrs* layers = calloc((size_t)L, sizeof *layers);
  void** owned = calloc((size_t)(4 * L + 3), sizeof *owned);  /* device buffers to free */
  int n_owned = 0;
  const size_t kv_bytes = (size_t)d.n_kvh * (size_t)kv_cap * (size_t)d.head_dim * 2;  /* binary16 */
  char name[64];
  for (int l = 0; l < L; ++l) {
    nt_layer_ptrs* p = &layers[l];
    snprintf(name, sizeof name, "blob.%d", l);
    if (l < n_resident) {
      uint8_t* b = upload(f, name);  /* the seven matrices, in the blob layout */
      owned[n_owned++] = b;
      p->wq = b + offs[0], p->wk = b + offs[1], p->wv = b + offs[2], p->wo = b + offs[3];
      p->wg = b + offs[4], p->wu = b + offs[5], p->wd = b + offs[6];
    } else {
      int rung = -1;
      NT(nt_file_lock(g_ctx, f, name, 1, &p->host_blob, &rung));
      printf("layer %d streamed from the file, rung %d\n", l, rung);
    }
    snprintf(name, sizeof name, "attn_norm.%d", l);
    owned[n_owned++] = (void*)(p->attn_norm = upload(f, name));
    snprintf(name, sizeof name, "ffn_norm.%d", l);
    owned[n_owned++] = (void*)(p->ffn_norm = upload(f, name));
    CU(cudaMalloc(&p->kcache, kv_bytes));
    CU(cudaMalloc(&p->vcache, kv_bytes));
    CU(cudaMemset(p->kcache, 0, kv_bytes));
    CU(cudaMemset(p->vcache, 0, kv_bytes));
  }
  const void* embd = NULL;
  if (n_resident < L) {
    NT(nt_file_lock(g_ctx, f, "embd", 1, &embd, NULL));  /* one row per token, read from host memory */
  } else {
    embd = owned[n_owned++] = upload(f, "embd");
  }
  void* out = owned[n_owned++] = upload(f, "out");
  float* out_norm = owned[n_owned++] = upload(f, "out_norm");

  nt_model* m = NULL;
  NT(nt_model_init(g_ctx, &d, layers, embd, out, out_norm, &m));
  float* logits = NULL;
  int32_t* next = NULL;
  CU(cudaMalloc((void**)&logits, sizeof(float) * (size_t)d.vocab));
  CU(cudaMalloc((void**)&next, sizeof(int32_t)));
  float* host = malloc(sizeof(float) * (size_t)d.vocab);
  FILE* fo = fopen(out_path, "wb");
  if (!fo) {
    perror(out_path);
    return 1;
  }
  NT(nt_prefill(g_ctx, m, prompt, n_prompt, 0, logits, next, NULL));
  for (int i = 0; i <= n_decode; ++i) {
    if (i > 0) NT(nt_decode_step(g_ctx, m, -1, n_prompt + i - 1, NULL, logits, next, NULL));
    NT(nt_ctx_sync(g_ctx));
    CU(cudaMemcpy(host, logits, sizeof(float) * (size_t)d.vocab, cudaMemcpyDeviceToHost));
    if (fwrite(host, sizeof(float), (size_t)d.vocab, fo) != (size_t)d.vocab) {
      perror(out_path);
      return 1;
    }
  }
  fclose(fo);

  NT(nt_model_destroy(g_ctx, m));
  for (int l = n_resident; l < L; ++l) {
    snprintf(name, sizeof name, "blob.%d", l);
    NT(nt_file_unlock(g_ctx, f, name));
  }
  if (n_resident < L) NT(nt_file_unlock(g_ctx, f, "embd"));
  NT(nt_file_close(f));
  for (int l = 0; l < L; ++l) {
    CU(cudaFree(layers[l].kcache));
    CU(cudaFree(layers[l].vcache));
  }
  for (int i = 0; i < n_owned; ++i) CU(cudaFree(owned[i]));
  CU(cudaFree(logits));
  CU(cudaFree(next));
  NT(nt_ctx_destroy(g_ctx));
  free(host);
  free(owned);
  free(layers);
  free(prompt);
  printf("decoded %d steps after a %d-token prompt\n", n_decode, n_prompt);
  return 0;
}
