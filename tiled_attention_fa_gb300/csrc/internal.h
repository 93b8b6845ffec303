// Internal (C++) entry points between the C ABI and the kernel units.
#pragma once

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace fa {

fa_status run_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Lq,
                  int Lk, int H, int Hkv, int D, int causal, int dtype, cudaStream_t s);
fa_status run_fwd_fp8(const void* Q8, const void* K8, const void* V8, float q_scale, float k_scale,
                      float v_scale, void* O, float* LSE, int B, int Lq, int Lk, int H, int Hkv,
                      int causal, int out_dtype, cudaStream_t s);
unsigned int fwd_read_error(cudaStream_t s);
fa_status run_selftest_wait(unsigned long long limit_ns, cudaStream_t s);

fa_status run_bwd_prep(const void* O, const void* dO, float* Delta, float* dq_accum, int B, int L,
                       int H, int D, int dtype, cudaStream_t s);
fa_status run_bwd(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                  const float* Delta, void* dQ, void* dK, void* dV, float* dq_accum,
                  int zero_accum, int B, int Lq, int Lk, int H, int Hkv, int D, int causal,
                  int dtype, cudaStream_t s);
fa_status run_bwd_main(const void* Q, const void* K, const void* V, const void* dO,
                       const float* LSE, const float* Delta, void* dK, void* dV, float* dq_accum,
                       int zero_accum, int B, int Lq, int Lk, int H, int Hkv, int D, int causal,
                       int dtype, cudaStream_t s);
fa_status run_bwd_post(const float* dq_accum, void* dQ, int B, int L, int H, int D, int dtype,
                       cudaStream_t s);
unsigned int bwd_read_error(cudaStream_t s);
fa_status run_bwd_noalloc(const void* Q, const void* K, const void* V, const void* dO,
                          const float* LSE, const float* Delta, void* dQ, void* dK, void* dV,
                          int B, int L, int H, int Hkv, int D, int causal, int dtype,
                          cudaStream_t s);

// Split-KV decoding (decode.cu).
struct DecodePlan {
  int nsplit;  // key slices per (batch, K/V head)
  int tps;     // 128-key tiles per slice
  int n_kv;    // 128-key tiles in all
};
DecodePlan decode_plan(int B, int Lq, int Lk, int H, int Hkv, int sms);
size_t decode_workspace_size(int B, int Lq, int Lk, int H, int Hkv, int D);
fa_status run_decode(const void* Q, const void* K, const void* V, void* O, float* LSE, void* ws,
                     size_t ws_bytes, int B, int Lq, int Lk, int H, int Hkv, int D, int causal,
                     int dtype, cudaStream_t s);
fa_status run_decode_slices(const void* Q, const void* K, const void* V, void* ws, size_t ws_bytes,
                            int B, int Lq, int Lk, int H, int Hkv, int D, int causal, int dtype,
                            cudaStream_t s);
fa_status run_decode_merge(const void* ws, size_t ws_bytes, void* O, float* LSE, int B, int Lq,
                           int Lk, int H, int Hkv, int D, int dtype, cudaStream_t s);
unsigned int decode_read_error(cudaStream_t s);

inline int padded_len(int L) { return (L + 127) / 128 * 128; }

}  // namespace fa
