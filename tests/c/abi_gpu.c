/* The decode path driven from plain C through the C ABI, on a GPU: device
 * buffers from the CUDA runtime, pa_kv_append, pa_plan, pa_plan_upload and
 * pa_decode_attention on one stream, then pa_append_decode_attention_fp8
 * over an FP8 (E4M3) cache with the same plan.  Every sequence holds one
 * token (the one appended), so each query head's softmax is a single weight
 * 1 and its output must be exactly the new V row of its KV head (a closed
 * form; the values are exact in fp16, and for the FP8 cache the V rows are
 * E4M3 values times 2^-7 with largest magnitude 448 * 2^-7, so the row's
 * scale is 2^-7 and its codes dequantise exactly).  Exit status 0 on
 * success. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "pagedattn.h"

/* binary16 bits of a float that fp16 holds exactly (small multiples of 2^-6) */
static uint16_t half_bits(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  const uint32_t sign = (x >> 16) & 0x8000u;
  const int exp = (int)((x >> 23) & 0xff) - 127 + 15;
  const uint32_t man = (x >> 13) & 0x3ffu;
  if ((x & 0x7fffffffu) == 0) return (uint16_t)sign;
  return (uint16_t)(sign | ((uint32_t)exp << 10) | man);
}

#define CUDA_OK(e)                                                       \
  do {                                                                   \
    cudaError_t err_ = (e);                                              \
    if (err_ != cudaSuccess) {                                           \
      fprintf(stderr, "CUDA error %s at line %d\n", cudaGetErrorString(err_), __LINE__); \
      return 2;                                                          \
    }                                                                    \
  } while (0)

enum { B = 2, HQ = 4, HKV = 2, D = 64, S = 16, MAXP = 4, P = 8 };

int main(void) {
  pa_shape_t s;
  memset(&s, 0, sizeof(s));
  s.batch = B;
  s.num_q_heads = HQ;
  s.num_kv_heads = HKV;
  s.head_dim = D;
  s.page_size = S;
  s.max_pages_per_seq = MAXP;
  s.num_pages = P;
  s.dtype = PA_DTYPE_F16;

  static uint16_t q[B][HQ][D], kn[B][HKV][D], vn[B][HKV][D], out[B][HQ][D];
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < HKV; ++h)
      for (int d = 0; d < D; ++d) {
        kn[b][h][d] = half_bits(0.25f * (float)(d % 4) - 0.5f);
        vn[b][h][d] = half_bits((float)(b * HKV + h + 1) + (float)d / 64.0f);
      }
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < HQ; ++h)
      for (int d = 0; d < D; ++d) q[b][h][d] = half_bits((float)((b + h + d) % 5) - 2.0f);
  const int32_t bt[B][MAXP] = {{3, -1, -1, -1}, {6, -1, -1, -1}};
  const int32_t lens[B] = {1, 1};

  void *dq, *dkn, *dvn, *dk, *dv, *dout, *dbt, *dsl, *dst, *ws;
  const size_t pool = (size_t)P * HKV * S * D * 2;
  CUDA_OK(cudaMalloc(&dq, sizeof(q)));
  CUDA_OK(cudaMalloc(&dkn, sizeof(kn)));
  CUDA_OK(cudaMalloc(&dvn, sizeof(vn)));
  CUDA_OK(cudaMalloc(&dk, pool));
  CUDA_OK(cudaMalloc(&dv, pool));
  CUDA_OK(cudaMalloc(&dout, sizeof(out)));
  CUDA_OK(cudaMalloc(&dbt, sizeof(bt)));
  CUDA_OK(cudaMalloc(&dsl, sizeof(lens)));
  CUDA_OK(cudaMalloc(&dst, 4));
  CUDA_OK(cudaMemset(dk, 0, pool));
  CUDA_OK(cudaMemset(dv, 0, pool));
  CUDA_OK(cudaMemset(dst, 0, 4));
  CUDA_OK(cudaMemcpy(dq, q, sizeof(q), cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dkn, kn, sizeof(kn), cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dvn, vn, sizeof(vn), cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dbt, bt, sizeof(bt), cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(dsl, lens, sizeof(lens), cudaMemcpyHostToDevice));
  cudaStream_t st;
  CUDA_OK(cudaStreamCreate(&st));

  int sms = 0;
  CUDA_OK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  pa_plan_t plan;
  if (pa_plan(&s, lens, sms, 0, &plan) != PA_OK) return 3;
  CUDA_OK(cudaMalloc(&ws, plan.workspace_bytes));
  int rc = 0;
  rc |= pa_kv_append(&s, dkn, dvn, dk, dv, dbt, dsl, dst, st) != PA_OK;
  rc |= pa_plan_upload(&plan, ws, plan.workspace_bytes, st) != PA_OK;
  rc |= pa_decode_attention(&s, &plan, dq, dk, dv, dbt, dsl, 0.125f, dout, ws,
                            plan.workspace_bytes, dst, st) != PA_OK;
  if (rc) {
    fprintf(stderr, "a call returned an error\n");
    return 4;
  }
  CUDA_OK(cudaStreamSynchronize(st));
  int32_t status = -1;
  CUDA_OK(cudaMemcpy(&status, dst, 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(out, dout, sizeof(out), cudaMemcpyDeviceToHost));
  int bad = status != 0;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < HQ; ++h)
      for (int d = 0; d < D; ++d)
        if (out[b][h][d] != vn[b][h / (HQ / HKV)][d]) ++bad;

  /* FP8 cache: V rows (256 + 32 * (d % 7)) / 128, i.e. E4M3 values 256..448
   * times 2^-7, so max|v| / 448 = 2^-7 exactly and every code is exact */
  static uint16_t vn8[B][HKV][D];
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < HKV; ++h)
      for (int d = 0; d < D; ++d) vn8[b][h][d] = half_bits((float)(256 + 32 * (d % 7)) / 128.0f);
  void *dvn8, *dkc, *dvc, *dks, *dvs;
  const size_t codes = (size_t)P * HKV * S * D, scales = (size_t)P * HKV * S * 4;
  CUDA_OK(cudaMalloc(&dvn8, sizeof(vn8)));
  CUDA_OK(cudaMalloc(&dkc, codes));
  CUDA_OK(cudaMalloc(&dvc, codes));
  CUDA_OK(cudaMalloc(&dks, scales));
  CUDA_OK(cudaMalloc(&dvs, scales));
  CUDA_OK(cudaMemset(dkc, 0, codes));
  CUDA_OK(cudaMemset(dvc, 0, codes));
  CUDA_OK(cudaMemset(dks, 0, scales));
  CUDA_OK(cudaMemset(dvs, 0, scales));
  CUDA_OK(cudaMemcpy(dvn8, vn8, sizeof(vn8), cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemset(dout, 0, sizeof(out)));
  if (pa_append_decode_attention_fp8(&s, &plan, dq, dkn, dvn8, dkc, dvc, (float*)dks, (float*)dvs,
                                     dbt, dsl, 0.125f, dout, ws, plan.workspace_bytes, dst,
                                     st) != PA_OK) {
    fprintf(stderr, "the FP8 call returned an error\n");
    return 4;
  }
  CUDA_OK(cudaStreamSynchronize(st));
  int32_t status8 = -1;
  CUDA_OK(cudaMemcpy(&status8, dst, 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(out, dout, sizeof(out), cudaMemcpyDeviceToHost));
  int bad8 = status8 != 0;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < HQ; ++h)
      for (int d = 0; d < D; ++d)
        if (out[b][h][d] != vn8[b][h / (HQ / HKV)][d]) ++bad8;
  cudaFree(dvn8);
  cudaFree(dkc);
  cudaFree(dvc);
  cudaFree(dks);
  cudaFree(dvs);
  if (bad8) {
    fprintf(stderr, "FP8 cache: status %d, %d outputs differ from their V rows\n", (int)status8,
            bad8);
    return 1;
  }
  pa_plan_free(&plan);
  cudaFree(ws);
  cudaFree(dq);
  cudaFree(dkn);
  cudaFree(dvn);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(dout);
  cudaFree(dbt);
  cudaFree(dsl);
  cudaFree(dst);
  cudaStreamDestroy(st);
  if (bad) {
    fprintf(stderr, "status %d, %d outputs differ from their V rows\n", (int)status, bad);
    return 1;
  }
  printf("decode from C ok (fp16 and FP8 caches)\n");
  return 0;
}
