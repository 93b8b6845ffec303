// Host launchers of the backward kernels (preprocess, main pass, dQ post-process).
#include <mutex>
#include <type_traits>

#include "bwd.cuh"
#include "common.cuh"
#include "internal.h"

namespace fa {

template <int D, bool BF16>
static fa_status launch_prep(const void* O, const void* dO, float* Delta, float* dq_accum, int B,
                             int L, int H, cudaStream_t s) {
  const int Lpad = padded_len(L);
  // Heads per CTA: all of them when (batch, chunk) pairs alone fill the GPU
  // twice over, else fewer (halving) until they do.
  const long long pairs = static_cast<long long>(B) * (Lpad / 32);
  int hg = H;
  while (hg > 1 && pairs * ((H + hg - 1) / hg) < 2LL * sm_count()) hg = (hg + 1) / 2;
  const long long grid = pairs * ((H + hg - 1) / hg);
  if (grid > 0x7FFFFFFFLL) return FA_ERR_UNSUPPORTED;
  const size_t smem = static_cast<size_t>(hg) * 32 * sizeof(float);
  auto kern = fa_bwd_prep_kernel<D, BF16>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return FA_ERR_UNSUPPORTED;
  kern<<<static_cast<unsigned>(grid), 256, smem, s>>>(O, dO, Delta, dq_accum, B, L, H, Lpad, hg);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status run_bwd_prep(const void* O, const void* dO, float* Delta, float* dq_accum, int B, int L,
                       int H, int D, int dtype, cudaStream_t s) {
  const bool bf16 = dtype == FA_BF16;
  if (static_cast<size_t>(H) * 32 * sizeof(float) > 200 * 1024) return FA_ERR_UNSUPPORTED;
  if (D == 64)
    return bf16 ? launch_prep<64, true>(O, dO, Delta, dq_accum, B, L, H, s)
                : launch_prep<64, false>(O, dO, Delta, dq_accum, B, L, H, s);
  return bf16 ? launch_prep<128, true>(O, dO, Delta, dq_accum, B, L, H, s)
              : launch_prep<128, false>(O, dO, Delta, dq_accum, B, L, H, s);
}

// L2 size of the current device (cached per device).
static double l2_bytes() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev);
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

template <int D, bool BF16>
static fa_status launch_bwd(const void* Q, const void* K, const void* V, const void* dO,
                            const float* LSE, const float* Delta, void* dK, void* dV,
                            float* dq_accum, int zero_accum, int B, int Lq, int Lk, int H,
                            int Hkv, int causal, cudaStream_t s) {
  using Ly = BwdLayout<D>;
  const int Lpad = padded_len(Lq);
  if (zero_accum &&
      cudaMemsetAsync(dq_accum, 0, static_cast<size_t>(B) * H * Lpad * D * sizeof(float), s) !=
          cudaSuccess)
    return FA_ERR_CUDA;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_bshd_map(&tq, Q, B, Lq, H, D, BF16) || !make_bshd_map(&tk, K, B, Lk, Hkv, D, BF16) ||
      !make_bshd_map(&tv, V, B, Lk, Hkv, D, BF16) || !make_bshd_map(&tdo, dO, B, Lq, H, D, BF16))
    return FA_ERR_CUDA;
  BwdParams p;
  p.LSE = LSE;
  p.Delta = Delta;
  p.dq_accum = dq_accum;
  p.dK = dK;
  p.dV = dV;
  p.B = B;
  p.Lq = Lq;
  p.Lk = Lk;
  p.past = Lk - Lq;
  p.H = H;
  p.Hkv = Hkv;
  p.causal = causal ? 1 : 0;
  p.n_kv = (Lk + 127) / 128;
  p.n_q = Lpad / 128;
  p.Lpad = Lpad;
  p.n_items = B * Hkv * p.n_kv;
  p.ipu = p.causal ? 2 : 1;
  p.n_units = p.causal ? B * Hkv * ((p.n_kv + 1) / 2) : p.n_items;
  p.snake = 0;
  {
    // Causal problems of at most four rounds of pair units leave much of the
    // last round idle, so deal single tiles in snake order instead -- when
    // every head's Q and dO fit in 0.6 of L2 together (the snake order runs
    // all heads at once; the pair order a few heads at a time).  Measured,
    // fp16 causal: B1 H32 D128 L1024 0.0446 -> 0.0436 ms, L4096 (64 MiB of
    // Q, dO; 512 pair units) 0.371 -> 0.335 ms; L8192 (128 MiB) 1.184 ->
    // 1.257 ms and B8 H32 L1024 D64 (1,024 pair units) 0.162 -> 0.184 ms
    // with it, hence the limits.
    const int sm = sm_count();
    const double qdo_bytes = 4.0 * B * H * static_cast<double>(Lq) * D;  // Q and dO, 16-bit
    if (p.causal && p.n_items >= sm && p.n_units <= 4 * sm && qdo_bytes <= 0.6 * l2_bytes()) {
      p.snake = 1;
      p.ipu = 1;
      p.n_units = (p.n_items + sm - 1) / sm * sm;
    }
  }
  p.scale = 1.f / sqrtf(static_cast<float>(D));
  p.sl2 = 1.4426950408889634f * p.scale;
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (optin < static_cast<int>(Ly::SMEM_ALLOC)) return FA_ERR_UNSUPPORTED;
  auto kern = fa_bwd_kernel<D, BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM_ALLOC) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  {
    // The kernel re-balances registers between its warpgroups (setmaxnreg:
    // Ly::REGS_COMPUTE twice, REGS_DRAIN, REGS_OTHER per thread); the budgets
    // add up only when every thread starts with NTHREADS_REGS.  Any other
    // allocation would leave an increase waiting for registers that never
    // come back, so refuse to launch instead.
    static int num_regs = -1;
    static std::once_flag once;
    std::call_once(once, [&] {
      cudaFuncAttributes a;
      if (cudaFuncGetAttributes(&a, kern) == cudaSuccess) num_regs = a.numRegs;
    });
    if (num_regs != Ly::NTHREADS_REGS) return FA_ERR_UNSUPPORTED;
  }
  const int grid = p.n_units < sm_count() ? p.n_units : sm_count();  // persistent CTAs
  kern<<<grid, Ly::NTHREADS, Ly::SMEM_ALLOC, s>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, bool BF16>
static fa_status launch_post(const float* dq_accum, void* dQ, int B, int L, int H, cudaStream_t s) {
  const int Lpad = padded_len(L);
  auto kern = fa_dq_convert_kernel<D, BF16>;
  constexpr size_t smem = conv_smem_bytes<D>();
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return FA_ERR_CUDA;
  kern<<<B * H * (Lpad / kConvRows), kConvThreads, smem, s>>>(
      dq_accum, dQ, B, L, H, Lpad, 1.f / sqrtf(static_cast<float>(D)));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status run_bwd_main(const void* Q, const void* K, const void* V, const void* dO,
                       const float* LSE, const float* Delta, void* dK, void* dV, float* dq_accum,
                       int zero_accum, int B, int Lq, int Lk, int H, int Hkv, int D, int causal,
                       int dtype, cudaStream_t s) {
  const bool bf16 = dtype == FA_BF16;
  if (D == 64)
    return bf16 ? launch_bwd<64, true>(Q, K, V, dO, LSE, Delta, dK, dV, dq_accum, zero_accum, B,
                                       Lq, Lk, H, Hkv, causal, s)
                : launch_bwd<64, false>(Q, K, V, dO, LSE, Delta, dK, dV, dq_accum, zero_accum, B,
                                        Lq, Lk, H, Hkv, causal, s);
  return bf16 ? launch_bwd<128, true>(Q, K, V, dO, LSE, Delta, dK, dV, dq_accum, zero_accum, B,
                                      Lq, Lk, H, Hkv, causal, s)
              : launch_bwd<128, false>(Q, K, V, dO, LSE, Delta, dK, dV, dq_accum, zero_accum, B,
                                       Lq, Lk, H, Hkv, causal, s);
}

fa_status run_bwd_post(const float* dq_accum, void* dQ, int B, int L, int H, int D, int dtype,
                       cudaStream_t s) {
  const bool bf16 = dtype == FA_BF16;
  if (D == 64)
    return bf16 ? launch_post<64, true>(dq_accum, dQ, B, L, H, s)
                : launch_post<64, false>(dq_accum, dQ, B, L, H, s);
  return bf16 ? launch_post<128, true>(dq_accum, dQ, B, L, H, s)
              : launch_post<128, false>(dq_accum, dQ, B, L, H, s);
}

fa_status run_bwd(const void* Q, const void* K, const void* V, const void* dO, const float* LSE,
                  const float* Delta, void* dQ, void* dK, void* dV, float* dq_accum,
                  int zero_accum, int B, int Lq, int Lk, int H, int Hkv, int D, int causal,
                  int dtype, cudaStream_t s) {
  fa_status st = run_bwd_main(Q, K, V, dO, LSE, Delta, dK, dV, dq_accum, zero_accum, B, Lq, Lk, H,
                              Hkv, D, causal, dtype, s);
  if (st != FA_OK) return st;
  return run_bwd_post(dq_accum, dQ, B, Lq, H, D, dtype, s);
}

unsigned int bwd_read_error(cudaStream_t s) { return read_and_clear_error(s); }

// ---------------------------------------------------------------- no-allocation variant
// Scratch for fa_bwd_noalloc's fp32 dQ accumulator.  It is part of this
// module's device image, so every GPU that loads the library holds these
// FA_NOALLOC_SCRATCH_BYTES until the process exits; all calls share it.
static __device__ __align__(256) float g_noalloc_dq_accum[FA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with the device current.  It is looked up again on every call whose stream
// is not being captured (a device reset reloads the module, possibly at
// another address) and remembered per device for calls made during a
// capture, where the lookup is not attempted.
fa_status noalloc_scratch(cudaStream_t s, float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_dq_accum) != cudaSuccess || ptr == nullptr)
      return FA_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(ptr);
  } else if (g_noalloc_ptr[dev] == nullptr) {
    return FA_ERR_CUDA;  // first call on this device made during a capture
  }
  *out = g_noalloc_ptr[dev];
  return FA_OK;
}
}  // namespace

fa_status run_bwd_noalloc(const void* Q, const void* K, const void* V, const void* dO,
                          const float* LSE, const float* Delta, void* dQ, void* dK, void* dV,
                          int B, int L, int H, int Hkv, int D, int causal, int dtype,
                          cudaStream_t s) {
  const size_t need = static_cast<size_t>(B) * H * padded_len(L) * D * sizeof(float);
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_TOO_SMALL;
  float* acc = nullptr;
  fa_status st = noalloc_scratch(s, &acc);
  if (st != FA_OK) return st;
  // The array keeps the previous call's sums: clear the part this call uses.
  if (cudaMemsetAsync(acc, 0, need, s) != cudaSuccess) return FA_ERR_CUDA;
  return run_bwd(Q, K, V, dO, LSE, Delta, dQ, dK, dV, acc, 0, B, L, L, H, Hkv, D, causal, dtype,
                 s);
}

}  // namespace fa
