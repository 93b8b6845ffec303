// Host launcher of the forward kernel.
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "fwd.cuh"
#include "internal.h"

namespace fa {

// FP8: Q, K, V are E4M3 codes with per-tensor scales qs, ks, vs; BF16 then
// selects the output type.
template <int D, bool BF16, bool FP8 = false>
static fa_status launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                        int Lq, int Lk, int H, int Hkv, int causal, cudaStream_t s, float qs = 1.f,
                        float ks = 1.f, float vs = 1.f) {
  using Ly = FwdLayout<D, FP8>;
  CUtensorMap tq, tk, tv;
  if constexpr (FP8) {
    if (!make_bshd_map_e4m3(&tq, Q, B, Lq, H, D) || !make_bshd_map_e4m3(&tk, K, B, Lk, Hkv, D) ||
        !make_bshd_map_e4m3(&tv, V, B, Lk, Hkv, D))
      return FA_ERR_CUDA;
  } else {
    if (!make_bshd_map(&tq, Q, B, Lq, H, D, BF16) || !make_bshd_map(&tk, K, B, Lk, Hkv, D, BF16) ||
        !make_bshd_map(&tv, V, B, Lk, Hkv, D, BF16))
      return FA_ERR_CUDA;
  }
  FwdParams p;
  p.O = O;
  p.LSE = LSE;
  p.B = B;
  p.Lq = Lq;
  p.Lk = Lk;
  p.past = Lk - Lq;
  p.H = H;
  p.Hkv = Hkv;
  p.causal = causal ? 1 : 0;
  p.n_kv = (Lk + 127) / 128;
  p.n_qpairs = (Lq + 255) / 256;
  p.n_items = B * H * p.n_qpairs;
  // Scores carry q_scale * k_scale (1 for 16-bit inputs); v_scale is applied
  // with 1 / l at the store.
  p.sl2 = FP8 ? static_cast<float>(1.4426950408889634 * static_cast<double>(qs) *
                                   static_cast<double>(ks) / std::sqrt(static_cast<double>(D)))
              : 1.4426950408889634f / sqrtf(static_cast<float>(D));
  p.o_scale = vs;
  // Causal problems of a few rounds of items leave much of the last round
  // idle in head-major order; ordered by decreasing work across all heads
  // the alternating rounds balance them.  That order runs all heads at once,
  // so it is taken only while every head's K and V take at most 1.2 x L2
  // (the CTAs of one head stream the same K/V tiles nearly in step).
  // Measured, fp16 causal forward, B1 H32 D128: L4096 0.128 -> 0.113-0.116
  // ms, L8192 (128 MiB of K, V) 0.401 -> 0.373-0.378; forced on B8 H32 L4096
  // (512 MiB, 54 rounds) it lost 12%, and at D = 64 (B8 H32 L1024, B4 H32/8
  // L1024) it was neutral to 5% slower, so D = 128 only.
  p.sorted = 0;
  {
    const int sm = sm_count();
    int dev = 0, l2 = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    const double kv_bytes = 2.0 * B * Hkv * static_cast<double>(Lk) * D * (FP8 ? 1 : 2);
    if (D == 128 && causal && p.n_items >= sm && p.n_items <= 8 * sm && kv_bytes <= 1.2 * l2)
      p.sorted = 1;
  }
  auto kern = fa_fwd_kernel<D, BF16, FP8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM_ALLOC) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  const int grid = p.n_items < sm_count() ? p.n_items : sm_count();
  kern<<<grid, Ly::NTHREADS, Ly::SMEM_ALLOC, s>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status run_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Lq,
                  int Lk, int H, int Hkv, int D, int causal, int dtype, cudaStream_t s) {
  const bool bf16 = dtype == FA_BF16;
  if (D == 64) {
    return bf16 ? launch<64, true>(Q, K, V, O, LSE, B, Lq, Lk, H, Hkv, causal, s)
                : launch<64, false>(Q, K, V, O, LSE, B, Lq, Lk, H, Hkv, causal, s);
  }
  return bf16 ? launch<128, true>(Q, K, V, O, LSE, B, Lq, Lk, H, Hkv, causal, s)
              : launch<128, false>(Q, K, V, O, LSE, B, Lq, Lk, H, Hkv, causal, s);
}

fa_status run_fwd_fp8(const void* Q8, const void* K8, const void* V8, float q_scale, float k_scale,
                      float v_scale, void* O, float* LSE, int B, int Lq, int Lk, int H, int Hkv,
                      int causal, int out_dtype, cudaStream_t s) {
  return out_dtype == FA_BF16
             ? launch<128, true, true>(Q8, K8, V8, O, LSE, B, Lq, Lk, H, Hkv, causal, s, q_scale,
                                       k_scale, v_scale)
             : launch<128, false, true>(Q8, K8, V8, O, LSE, B, Lq, Lk, H, Hkv, causal, s, q_scale,
                                        k_scale, v_scale);
}

unsigned int fwd_read_error(cudaStream_t s) { return read_and_clear_error(s); }

// One thread waits on an mbarrier that is initialised for one arrival and
// never receives it.  The bounded wait gives up after `limit_ns`, records
// kSelftestSite in the error word and the kernel returns normally.
constexpr unsigned int kSelftestSite = 900;
__global__ void fa_selftest_wait_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ AbortState ab;
  const uint32_t bar = smem_u32(&bar_storage);
  mbar_init(bar, 1);
  ab.flag = 0;
  fence_barrier_init();
  mbar_wait_limit(bar, 0, &ab, device_error_word(), kSelftestSite, limit_ns);
}

fa_status run_selftest_wait(unsigned long long limit_ns, cudaStream_t s) {
  fa_selftest_wait_kernel<<<1, 1, 0, s>>>(limit_ns);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
