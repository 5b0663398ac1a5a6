/*
 * One decode step through the C ABI alone (no Python, no PyTorch): quantize new K/V tokens
 * into an int8 side-tensor slot pool with qkv_write_int8, then run the top-k gather attention
 * with qsa_gather_attn, unsplit and split (qsa_splitk_merge). Device memory comes from the CUDA
 * runtime; the library allocates nothing.
 *
 * usage: decode_step <dir>
 *   <dir>/meta.txt   "T S R K Hq D": tokens, slots, rows, top-k, query heads (one KV head), head dim
 *   <dir>/k.bin      bf16 bits uint16 [T, 1, D]      <dir>/v.bin  the same for V
 *   <dir>/slots.bin  int64 [T]                        <dir>/q.bin  bf16 bits uint16 [R, Hq, D]
 *   <dir>/idx.bin    int32 [R, K], -1 = padding
 * writes <dir>/out.bin, out_split.bin (fp32 [R, Hq, D]), lse.bin (fp32 [R, Hq]) and
 * <dir>/status.txt (the device status words). Exits non-zero on any error status.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "qkv.h"

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) { fprintf(stderr, "cannot open %s\n", path); exit(2); }
  void* p = malloc(bytes ? bytes : 1);
  if (fread(p, 1, bytes, f) != bytes) { fprintf(stderr, "short read %s\n", path); exit(2); }
  fclose(f);
  return p;
}

static void write_file(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(p, 1, bytes, f) != bytes) { fprintf(stderr, "cannot write %s\n", path); exit(2); }
  fclose(f);
}

static void* dev_copy(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) { fprintf(stderr, "cudaMalloc failed\n"); exit(3); }
  if (host && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) { fprintf(stderr, "h2d failed\n"); exit(3); }
  if (!host && cudaMemset(d, 0, bytes ? bytes : 16) != cudaSuccess) { fprintf(stderr, "memset failed\n"); exit(3); }
  return d;
}

#define CHECK(call)                                                                 \
  do {                                                                              \
    qkv_status s_ = (call);                                                         \
    if (s_ != QKV_OK) { fprintf(stderr, "%s: %s\n", #call, qkv_status_str(s_)); return 4; } \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 2) { fprintf(stderr, "usage: decode_step <dir>\n"); return 1; }
  const char* dir = argv[1];
  long long T, S, R, K, Hq, D;
  {
    char path[4096];
    snprintf(path, sizeof path, "%s/meta.txt", dir);
    FILE* f = fopen(path, "r");
    if (!f || fscanf(f, "%lld %lld %lld %lld %lld %lld", &T, &S, &R, &K, &Hq, &D) != 6) { fprintf(stderr, "bad meta\n"); return 1; }
    fclose(f);
  }
  const size_t tok = (size_t)T * D * 2, qb = (size_t)R * Hq * D * 2, ob = (size_t)R * Hq * D * 4;
  void* k = dev_copy(read_file(dir, "k.bin", tok), tok);
  void* v = dev_copy(read_file(dir, "v.bin", tok), tok);
  void* slots = dev_copy(read_file(dir, "slots.bin", (size_t)T * 8), (size_t)T * 8);
  void* q = dev_copy(read_file(dir, "q.bin", qb), qb);
  void* idx = dev_copy(read_file(dir, "idx.bin", (size_t)R * K * 4), (size_t)R * K * 4);
  void* kc = dev_copy(NULL, (size_t)S * D);
  void* vc = dev_copy(NULL, (size_t)S * D);
  float* ks = (float*)dev_copy(NULL, (size_t)S * 4);
  float* vs = (float*)dev_copy(NULL, (size_t)S * 4);
  float* out = (float*)dev_copy(NULL, ob);
  float* lse = (float*)dev_copy(NULL, (size_t)R * Hq * 4);
  const int P = 3;
  float* o_part = (float*)dev_copy(NULL, ob * P);
  float* lse_part = (float*)dev_copy(NULL, (size_t)R * P * Hq * 4);
  float* out_split = (float*)dev_copy(NULL, ob);
  uint32_t* status = (uint32_t*)dev_copy(NULL, 8);

  cudaStream_t stream;
  if (cudaStreamCreate(&stream) != cudaSuccess) return 3;
  CHECK(qkv_write_int8(k, v, T, 1, (int)D, D, (const int64_t*)slots, QKV_INT8_SIDE, kc, vc, ks, vs, S,
                       status, stream));
  const float scale = 1.0f / 16.0f;
  CHECK(qsa_gather_attn(q, R, (int)Hq, 1, (int)D, QKV_INT8_SIDE, kc, vc, ks, vs, 1.0f, 1.0f, S,
                        (const int32_t*)idx, (int)K, scale, 1, out, lse, NULL, NULL, status + 1, stream));
  CHECK(qsa_gather_attn(q, R, (int)Hq, 1, (int)D, QKV_INT8_SIDE, kc, vc, ks, vs, 1.0f, 1.0f, S,
                        (const int32_t*)idx, (int)K, scale, P, NULL, NULL, o_part, lse_part, status + 1, stream));
  CHECK(qsa_splitk_merge(o_part, lse_part, R, (int)Hq, (int)D, P, 1.0f, out_split, NULL, stream));
  if (cudaStreamSynchronize(stream) != cudaSuccess) { fprintf(stderr, "stream failed\n"); return 3; }

  float* h = (float*)malloc(ob);
  cudaMemcpy(h, out, ob, cudaMemcpyDeviceToHost);
  write_file(dir, "out.bin", h, ob);
  cudaMemcpy(h, out_split, ob, cudaMemcpyDeviceToHost);
  write_file(dir, "out_split.bin", h, ob);
  cudaMemcpy(h, lse, (size_t)R * Hq * 4, cudaMemcpyDeviceToHost);
  write_file(dir, "lse.bin", h, (size_t)R * Hq * 4);
  uint32_t st[2];
  cudaMemcpy(st, status, 8, cudaMemcpyDeviceToHost);
  char path[4096];
  snprintf(path, sizeof path, "%s/status.txt", dir);
  FILE* f = fopen(path, "w");
  if (!f) return 2;
  fprintf(f, "%u %u\n", st[0], st[1]);
  fclose(f);
  return 0;
}
