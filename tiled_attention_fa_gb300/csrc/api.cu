// C ABI: argument validation and dispatch to the kernel units.
#include <cmath>
#include <cstdint>

#include "../../include/fa.h"
#include "internal.h"

namespace {

unsigned int g_last_site = 0;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ptr_ok(const void* p) { return p != nullptr && aligned16(p); }

// Lq query rows, Lk key rows (equal for the square entry points).
fa_status check_shape(int B, int Lq, int Lk, int H, int Hkv, int D, int dtype) {
  if (B < 1 || Lq < 1 || Lk < 1 || H < 1 || Hkv < 1) return FA_ERR_INVALID_ARG;
  if (Lq > (1 << 30) || Lk > (1 << 30) || H > (1 << 20) || B > (1 << 20)) return FA_ERR_INVALID_ARG;
  if (H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  // Work-item and element counts must fit the kernels' integer arithmetic.
  const int Lmax = Lq > Lk ? Lq : Lk;
  const long long items = static_cast<long long>(B) * H * ((Lmax + 127) / 128);
  const long long elems = static_cast<long long>(B) * fa::padded_len(Lmax) * H * D;
  if (items >= (1ll << 31) || elems >= (1ll << 40)) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * fa::padded_len(Lmax) >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status check_shape(int B, int L, int H, int Hkv, int D, int dtype) {
  return check_shape(B, L, L, H, Hkv, D, dtype);
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int L,
                 int H, int Hkv, int D, int causal, int dtype, void* stream) {
  fa_status st = check_shape(B, L, H, Hkv, D, dtype);
  if (st != FA_OK) return st;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(O) || !ptr_ok(LSE))
    return FA_ERR_INVALID_ARG;
  return fa::run_fwd(Q, K, V, O, LSE, B, L, L, H, Hkv, D, causal, dtype,
                     static_cast<cudaStream_t>(stream));
}

fa_status fa_fwd_kv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Lq,
                    int Lk, int H, int Hkv, int D, int causal, int dtype, void* stream) {
  fa_status st = check_shape(B, Lq, Lk, H, Hkv, D, dtype);
  if (st != FA_OK) return st;
  if (causal && Lk < Lq) return FA_ERR_INVALID_ARG;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(O) || !ptr_ok(LSE))
    return FA_ERR_INVALID_ARG;
  return fa::run_fwd(Q, K, V, O, LSE, B, Lq, Lk, H, Hkv, D, causal, dtype,
                     static_cast<cudaStream_t>(stream));
}

fa_status fa_fwd_fp8(const void* Q8, const void* K8, const void* V8, float q_scale,
                     float k_scale, float v_scale, void* O, float* LSE, int B, int Lq, int Lk,
                     int H, int Hkv, int D, int causal, int out_dtype, void* stream) {
  fa_status st = check_shape(B, Lq, Lk, H, Hkv, D, out_dtype);
  if (st != FA_OK) return st;
  if (D != 128) return FA_ERR_UNSUPPORTED;
  if (causal && Lk < Lq) return FA_ERR_INVALID_ARG;
  for (float sc : {q_scale, k_scale, v_scale})
    if (!(sc > 0.f) || !std::isfinite(sc)) return FA_ERR_INVALID_ARG;
  if (!ptr_ok(Q8) || !ptr_ok(K8) || !ptr_ok(V8) || !ptr_ok(O) || !ptr_ok(LSE))
    return FA_ERR_INVALID_ARG;
  return fa::run_fwd_fp8(Q8, K8, V8, q_scale, k_scale, v_scale, O, LSE, B, Lq, Lk, H, Hkv, causal,
                         out_dtype, static_cast<cudaStream_t>(stream));
}

fa_status fa_bwd_preprocess(const void* O, const void* dO, float* Delta, float* dq_accum, int B,
                            int L, int H, int D, int dtype, void* stream) {
  fa_status st = check_shape(B, L, H, H, D, dtype);
  if (st != FA_OK) return st;
  if (!ptr_ok(O) || !ptr_ok(dO) || !ptr_ok(Delta)) return FA_ERR_INVALID_ARG;
  if (dq_accum != nullptr && !aligned16(dq_accum)) return FA_ERR_INVALID_ARG;
  return fa::run_bwd_prep(O, dO, Delta, dq_accum, B, L, H, D, dtype,
                          static_cast<cudaStream_t>(stream));
}

size_t fa_bwd_workspace_size(int B, int L, int H, int D) {
  if (B < 1 || L < 1 || H < 1 || D < 1) return 0;
  return static_cast<size_t>(B) * H * fa::padded_len(L) * D * sizeof(float);
}

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, const float* Delta, void* dQ, void* dK, void* dV,
                 float* dq_accum, int zero_accum, int B, int L, int H, int Hkv, int D, int causal,
                 int dtype, void* stream) {
  (void)O;
  fa_status st = check_shape(B, L, H, Hkv, D, dtype);
  if (st != FA_OK) return st;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(dO) || !ptr_ok(LSE) || !ptr_ok(Delta) ||
      !ptr_ok(dQ) || !ptr_ok(dK) || !ptr_ok(dV) || !ptr_ok(dq_accum))
    return FA_ERR_INVALID_ARG;
  return fa::run_bwd(Q, K, V, dO, LSE, Delta, dQ, dK, dV, dq_accum, zero_accum, B, L, L, H, Hkv, D,
                     causal, dtype, static_cast<cudaStream_t>(stream));
}

fa_status fa_bwd_kv(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* LSE, const float* Delta, void* dQ, void* dK, void* dV,
                    float* dq_accum, int zero_accum, int B, int Lq, int Lk, int H, int Hkv, int D,
                    int causal, int dtype, void* stream) {
  (void)O;
  fa_status st = check_shape(B, Lq, Lk, H, Hkv, D, dtype);
  if (st != FA_OK) return st;
  if (causal && Lk < Lq) return FA_ERR_INVALID_ARG;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(dO) || !ptr_ok(LSE) || !ptr_ok(Delta) ||
      !ptr_ok(dQ) || !ptr_ok(dK) || !ptr_ok(dV) || !ptr_ok(dq_accum))
    return FA_ERR_INVALID_ARG;
  return fa::run_bwd(Q, K, V, dO, LSE, Delta, dQ, dK, dV, dq_accum, zero_accum, B, Lq, Lk, H, Hkv,
                     D, causal, dtype, static_cast<cudaStream_t>(stream));
}

fa_status fa_bwd_main(const void* Q, const void* K, const void* V, const void* dO,
                      const float* LSE, const float* Delta, void* dK, void* dV, float* dq_accum,
                      int zero_accum, int B, int L, int H, int Hkv, int D, int causal, int dtype,
                      void* stream) {
  fa_status st = check_shape(B, L, H, Hkv, D, dtype);
  if (st != FA_OK) return st;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(dO) || !ptr_ok(LSE) || !ptr_ok(Delta) ||
      !ptr_ok(dK) || !ptr_ok(dV) || !ptr_ok(dq_accum))
    return FA_ERR_INVALID_ARG;
  return fa::run_bwd_main(Q, K, V, dO, LSE, Delta, dK, dV, dq_accum, zero_accum, B, L, L, H, Hkv, D,
                          causal, dtype, static_cast<cudaStream_t>(stream));
}

fa_status fa_bwd_postprocess(const float* dq_accum, void* dQ, int B, int L, int H, int D,
                             int dtype, void* stream) {
  fa_status st = check_shape(B, L, H, H, D, dtype);
  if (st != FA_OK) return st;
  if (!ptr_ok(dq_accum) || !ptr_ok(dQ)) return FA_ERR_INVALID_ARG;
  return fa::run_bwd_post(dq_accum, dQ, B, L, H, D, dtype, static_cast<cudaStream_t>(stream));
}

fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* LSE, const float* Delta, void* dQ,
                         void* dK, void* dV, int B, int L, int H, int Hkv, int D, int causal,
                         int dtype, void* stream) {
  (void)O;
  fa_status st = check_shape(B, L, H, Hkv, D, dtype);
  if (st != FA_OK) return st;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(dO) || !ptr_ok(LSE) || !ptr_ok(Delta) ||
      !ptr_ok(dQ) || !ptr_ok(dK) || !ptr_ok(dV))
    return FA_ERR_INVALID_ARG;
  return fa::run_bwd_noalloc(Q, K, V, dO, LSE, Delta, dQ, dK, dV, B, L, H, Hkv, D, causal, dtype,
                             static_cast<cudaStream_t>(stream));
}

size_t fa_decode_workspace_size(int B, int Lq, int Lk, int H, int Hkv, int D) {
  if (B < 1 || Lq < 1 || Lk < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || (D != 64 && D != 128))
    return 0;
  return fa::decode_workspace_size(B, Lq, Lk, H, Hkv, D);
}

namespace {
fa_status check_decode(int B, int Lq, int Lk, int H, int Hkv, int D, int causal, int dtype) {
  fa_status st = check_shape(B, Lq, Lk, H, Hkv, D, dtype);
  if (st != FA_OK) return st;
  if (causal && Lk < Lq) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(H / Hkv) * Lq > 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}
}  // namespace

fa_status fa_decode(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    void* workspace, size_t workspace_bytes, int B, int Lq, int Lk, int H, int Hkv,
                    int D, int causal, int dtype, void* stream) {
  const fa_status st = check_decode(B, Lq, Lk, H, Hkv, D, causal, dtype);
  if (st != FA_OK) return st;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(O) || !ptr_ok(LSE) || !ptr_ok(workspace))
    return FA_ERR_INVALID_ARG;
  return fa::run_decode(Q, K, V, O, LSE, workspace, workspace_bytes, B, Lq, Lk, H, Hkv, D, causal,
                        dtype, static_cast<cudaStream_t>(stream));
}

fa_status fa_decode_slices(const void* Q, const void* K, const void* V, void* workspace,
                           size_t workspace_bytes, int B, int Lq, int Lk, int H, int Hkv, int D,
                           int causal, int dtype, void* stream) {
  const fa_status st = check_decode(B, Lq, Lk, H, Hkv, D, causal, dtype);
  if (st != FA_OK) return st;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(workspace)) return FA_ERR_INVALID_ARG;
  return fa::run_decode_slices(Q, K, V, workspace, workspace_bytes, B, Lq, Lk, H, Hkv, D, causal,
                               dtype, static_cast<cudaStream_t>(stream));
}

fa_status fa_decode_merge(const void* workspace, size_t workspace_bytes, void* O, float* LSE, int B,
                          int Lq, int Lk, int H, int Hkv, int D, int dtype, void* stream) {
  const fa_status st = check_decode(B, Lq, Lk, H, Hkv, D, 0, dtype);
  if (st != FA_OK) return st;
  if (!ptr_ok(workspace) || !ptr_ok(O) || !ptr_ok(LSE)) return FA_ERR_INVALID_ARG;
  return fa::run_decode_merge(workspace, workspace_bytes, O, LSE, B, Lq, Lk, H, Hkv, D, dtype,
                              static_cast<cudaStream_t>(stream));
}

fa_status fa_check_device_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned int words[3] = {fa::fwd_read_error(s), fa::bwd_read_error(s),
                                 fa::decode_read_error(s)};
  unsigned int site = 0;
  for (unsigned int w : words) {
    if (w == 0xFFFFFFFFu) return FA_ERR_CUDA;
    if (w && !site) site = w;
  }
  if (site) {
    g_last_site = site;
    return FA_ERR_DEVICE_TIMEOUT;
  }
  return FA_OK;
}

fa_status fa_selftest_bounded_wait(unsigned long long limit_ns, void* stream) {
  if (limit_ns < 1000000ull) limit_ns = 1000000ull;
  if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
  return fa::run_selftest_wait(limit_ns, static_cast<cudaStream_t>(stream));
}

unsigned int fa_last_error_site(void) { return g_last_site; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or dtype";
    case FA_ERR_CUDA: return "CUDA runtime or launch error";
    case FA_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case FA_ERR_SCRATCH_TOO_SMALL:
      return "scratch too small: the problem needs more than fa_bwd_noalloc's fixed array or "
             "the fa_decode workspace given";
  }
  return "unknown status";
}

const char* fa_version(void) { return "tiled_attention_fa_gb300 0.1 (sm_103a)"; }

}  // extern "C"
