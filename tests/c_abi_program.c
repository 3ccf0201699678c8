/*
 * A plain C caller of libgqa_attn.so, for tests/test_c_abi_program_gpu.py.
 *
 * It uses nothing but the C ABI of include/gqa_attn.h and the CUDA runtime:
 * device buffers from cudaMalloc, one decode (gqa_attn_decode with a workspace
 * of the size the library reports) and one causal prefill
 * (gqa_attn_prefill_causal), the device status word, and copies back.  Inputs
 * and outputs are raw little-endian files in the directory given as argv[1]:
 *   shapes.txt          "B H_q H_kv S_max T_q S_kv q_offset scale"
 *   q.bin k.bin v.bin   decode q [B,H_q,128], K/V [B,H_kv,S_max,128] (bf16 bits)
 *   seqlens.bin         int32 [B]
 *   pq.bin pk.bin pv.bin  prefill q [1,H_q,T_q,128], K/V [1,H_kv,S_kv,128]
 * and it writes o.bin, lse.bin (decode) and po.bin, plse.bin (prefill).
 * Exit status 0 when every call returned GQA_OK.
 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>

#include "gqa_attn.h"

static void *read_file(const char *dir, const char *name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (!f) return NULL;
  void *buf = malloc(bytes);
  size_t got = buf ? fread(buf, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

static int write_file(const char *dir, const char *name, const void *buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "wb");
  if (!f) return 0;
  size_t put = fwrite(buf, 1, bytes, f);
  fclose(f);
  return put == bytes;
}

/* host buffer -> new device buffer */
static void *to_device(const void *host, size_t bytes) {
  void *dev = NULL;
  if (cudaMalloc(&dev, bytes) != cudaSuccess) return NULL;
  if (cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return dev;
}

#define CHECK(cond, what)                    \
  do {                                       \
    if (!(cond)) {                           \
      fprintf(stderr, "failed: %s\n", what); \
      return 1;                              \
    }                                        \
  } while (0)

int main(int argc, char **argv) {
  CHECK(argc == 2, "usage: c_abi_program <dir>");
  const char *dir = argv[1];
  char path[4096];
  snprintf(path, sizeof path, "%s/shapes.txt", dir);
  FILE *sf = fopen(path, "r");
  CHECK(sf != NULL, "shapes.txt");
  int B, H_q, H_kv, S_max, T_q, S_kv, q_offset;
  float scale;
  CHECK(fscanf(sf, "%d %d %d %d %d %d %d %f", &B, &H_q, &H_kv, &S_max, &T_q, &S_kv, &q_offset,
               &scale) == 8,
        "shapes");
  fclose(sf);
  const int d = 128;
  int num_sms = 0;
  CHECK(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, 0) == cudaSuccess,
        "SM count");

  /* ---- decode ---- */
  const size_t q_bytes = (size_t)B * H_q * d * 2, kv_bytes = (size_t)B * H_kv * S_max * d * 2;
  void *q_h = read_file(dir, "q.bin", q_bytes), *k_h = read_file(dir, "k.bin", kv_bytes);
  void *v_h = read_file(dir, "v.bin", kv_bytes);
  void *sl_h = read_file(dir, "seqlens.bin", (size_t)B * 4);
  CHECK(q_h && k_h && v_h && sl_h, "decode inputs");
  void *q = to_device(q_h, q_bytes), *k = to_device(k_h, kv_bytes), *v = to_device(v_h, kv_bytes);
  void *sl = to_device(sl_h, (size_t)B * 4);
  void *o = NULL, *lse = NULL, *ws = NULL;
  CHECK(q && k && v && sl, "decode device buffers");
  CHECK(cudaMalloc(&o, q_bytes) == cudaSuccess && cudaMalloc(&lse, (size_t)B * H_q * 4) ==
                                                      cudaSuccess,
        "decode outputs");
  const size_t ws_bytes = gqa_attn_decode_workspace_size(B, H_q, H_kv, S_max, d, num_sms, 0);
  CHECK(ws_bytes > 0 && cudaMalloc(&ws, ws_bytes) == cudaSuccess, "decode workspace");
  int rc = gqa_attn_decode((const gqa_bf16_t *)q, (const gqa_bf16_t *)k, (const gqa_bf16_t *)v,
                           (const int32_t *)sl, B, H_q, H_kv, S_max, d, scale, 0,
                           (gqa_bf16_t *)o, (float *)lse, ws, ws_bytes, NULL);
  if (rc != GQA_OK) fprintf(stderr, "gqa_attn_decode: %s\n", gqa_status_string(rc));
  CHECK(rc == GQA_OK, "gqa_attn_decode");

  /* ---- causal prefill ---- */
  const size_t pq_bytes = (size_t)H_q * T_q * d * 2, pkv_bytes = (size_t)H_kv * S_kv * d * 2;
  void *pq_h = read_file(dir, "pq.bin", pq_bytes), *pk_h = read_file(dir, "pk.bin", pkv_bytes);
  void *pv_h = read_file(dir, "pv.bin", pkv_bytes);
  CHECK(pq_h && pk_h && pv_h, "prefill inputs");
  void *pq = to_device(pq_h, pq_bytes), *pk = to_device(pk_h, pkv_bytes);
  void *pv = to_device(pv_h, pkv_bytes), *po = NULL, *plse = NULL;
  CHECK(pq && pk && pv, "prefill device buffers");
  CHECK(cudaMalloc(&po, pq_bytes) == cudaSuccess &&
            cudaMalloc(&plse, (size_t)H_q * T_q * 4) == cudaSuccess,
        "prefill outputs");
  rc = gqa_attn_prefill_causal((const gqa_bf16_t *)pq, (const gqa_bf16_t *)pk,
                               (const gqa_bf16_t *)pv, 1, H_q, H_kv, T_q, S_kv, d, q_offset,
                               scale, (gqa_bf16_t *)po, (float *)plse, NULL);
  if (rc != GQA_OK) fprintf(stderr, "gqa_attn_prefill_causal: %s\n", gqa_status_string(rc));
  CHECK(rc == GQA_OK, "gqa_attn_prefill_causal");

  /* the bounded device-side waits all finished; the status word is clear */
  int status = -1;
  CHECK(gqa_attn_device_status(NULL, &status) == GQA_OK && status == GQA_OK, "device status");

  void *o_h = malloc(q_bytes), *lse_h = malloc((size_t)B * H_q * 4);
  void *po_h = malloc(pq_bytes), *plse_h = malloc((size_t)H_q * T_q * 4);
  CHECK(o_h && lse_h && po_h && plse_h, "host outputs");
  CHECK(cudaMemcpy(o_h, o, q_bytes, cudaMemcpyDeviceToHost) == cudaSuccess &&
            cudaMemcpy(lse_h, lse, (size_t)B * H_q * 4, cudaMemcpyDeviceToHost) == cudaSuccess &&
            cudaMemcpy(po_h, po, pq_bytes, cudaMemcpyDeviceToHost) == cudaSuccess &&
            cudaMemcpy(plse_h, plse, (size_t)H_q * T_q * 4, cudaMemcpyDeviceToHost) ==
                cudaSuccess,
        "copies back");
  CHECK(write_file(dir, "o.bin", o_h, q_bytes) && write_file(dir, "lse.bin", lse_h, (size_t)B * H_q * 4) &&
            write_file(dir, "po.bin", po_h, pq_bytes) &&
            write_file(dir, "plse.bin", plse_h, (size_t)H_q * T_q * 4),
        "output files");
  printf("c abi program ok: %d SMs, decode workspace %zu bytes\n", num_sms, ws_bytes);
  return 0;
}
