// Host launcher of the forward kernel.
#include <type_traits>

#include "common.cuh"
#include "fwd.cuh"
#include "internal.h"

namespace fa {

template <int D, bool BF16>
static fa_status launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                        int Lq, int Lk, int H, int Hkv, int causal, cudaStream_t s) {
  using Ly = FwdLayout<D>;
  CUtensorMap tq, tk, tv;
  if (!make_bshd_map(&tq, Q, B, Lq, H, D, BF16) || !make_bshd_map(&tk, K, B, Lk, Hkv, D, BF16) ||
      !make_bshd_map(&tv, V, B, Lk, Hkv, D, BF16))
    return FA_ERR_CUDA;
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
  p.sl2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  auto kern = fa_fwd_kernel<D, BF16>;
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
