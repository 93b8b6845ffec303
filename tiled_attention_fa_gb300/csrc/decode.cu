// Host side of split-KV decoding: the slice plan, the workspace layout and
// the two launches (per-slice kernel, then the merge).
#include <type_traits>

#include "common.cuh"
#include "decode.cuh"
#include "internal.h"

namespace fa {

namespace {

// Packed-Q tensor map: dims {D, H, Lq, B}, box {64, g, Lq, 1}, so one load
// brings a K/V head's g query heads for all Lq queries, row = query * g + head.
bool make_group_map(CUtensorMap* map, const void* Q, int B, int Lq, int H, int g, int D, bool bf16) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)Lq, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)Lq * H * D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)g, (cuuint32_t)Lq, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  4, const_cast<void*>(Q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

DecodePlan decode_plan(int B, int Lq, int Lk, int H, int Hkv, int sms) {
  // Choose the number of equal key slices per (batch, K/V head) that
  // minimises the modelled time: waves of one CTA per SM, each slice costing
  // its tiles plus about two tiles of fixed work (Q load, pipeline fill,
  // epilogue), plus the merge's read and write of the fp32 partials in the
  // same units (one tile = 128 keys of K and V = 512 * D bytes).
  DecodePlan best{1, 1, 0};
  const int n_kv = (Lk + 127) / 128;
  const long long pairs = static_cast<long long>(B) * Hkv;
  const long long rows = static_cast<long long>(H / Hkv) * Lq;
  if (sms < 1) sms = 1;
  double best_cost = 0.0;
  bool have = false;
  for (int ns = 1; ns <= n_kv; ++ns) {
    const int tps = (n_kv + ns - 1) / ns;
    if ((n_kv + tps - 1) / tps != ns) continue;  // same slices as a smaller count
    const long long ctas = pairs * ns;
    const long long waves = (ctas + sms - 1) / sms;
    const double cost = static_cast<double>(waves) * (tps + 2.0) +
                        static_cast<double>(pairs) * ns * rows / (64.0 * sms);
    if (!have || cost < best_cost - 1e-9) {
      have = true;
      best_cost = cost;
      best.nsplit = ns;
      best.tps = tps;
    }
  }
  best.n_kv = n_kv;
  return best;
}

size_t decode_workspace_bytes(const DecodePlan& pl, int B, int Lq, int H, int D) {
  const size_t rows = static_cast<size_t>(pl.nsplit) * B * H * Lq;
  return align256(rows * D * sizeof(float)) + align256(rows * sizeof(float));
}

namespace {

struct WsView {
  float* part_o;
  float* part_lse;
};

WsView ws_view(void* ws, const DecodePlan& pl, int B, int Lq, int H, int D) {
  const size_t rows_all = static_cast<size_t>(pl.nsplit) * B * H * Lq;
  return {static_cast<float*>(ws),
          reinterpret_cast<float*>(static_cast<char*>(ws) + align256(rows_all * D * sizeof(float)))};
}

template <int D, bool BF16>
fa_status launch_slices(const void* Q, const void* K, const void* V, void* ws, size_t ws_bytes,
                        int B, int Lq, int Lk, int H, int Hkv, int causal, cudaStream_t s) {
  using Ly = DecLayout<D>;
  const DecodePlan pl = decode_plan(B, Lq, Lk, H, Hkv, sm_count());
  if (ws_bytes < decode_workspace_bytes(pl, B, Lq, H, D)) return FA_ERR_SCRATCH_TOO_SMALL;
  const int g = H / Hkv;
  CUtensorMap tq, tk, tv;
  if (!make_group_map(&tq, Q, B, Lq, H, g, D, BF16) || !make_bshd_map(&tk, K, B, Lk, Hkv, D, BF16) ||
      !make_bshd_map(&tv, V, B, Lk, Hkv, D, BF16))
    return FA_ERR_CUDA;
  const WsView w = ws_view(ws, pl, B, Lq, H, D);
  DecParams p;
  p.part_o = w.part_o;
  p.part_lse = w.part_lse;
  p.B = B;
  p.Lq = Lq;
  p.Lk = Lk;
  p.H = H;
  p.Hkv = Hkv;
  p.g = g;
  p.rows = g * Lq;
  p.causal = causal ? 1 : 0;
  p.past = Lk - Lq;
  p.n_kv = pl.n_kv;
  p.tps = pl.tps;
  p.nsplit = pl.nsplit;
  p.sl2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  auto kern = fa_decode_kernel<D, BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::SMEM_ALLOC) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  const long long grid = static_cast<long long>(B) * Hkv * pl.nsplit;
  kern<<<static_cast<unsigned>(grid), Ly::NTHREADS, Ly::SMEM_ALLOC, s>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, bool BF16>
fa_status launch_merge(const void* ws, size_t ws_bytes, void* O, float* LSE, int B, int Lq, int Lk,
                       int H, int Hkv, cudaStream_t s) {
  const DecodePlan pl = decode_plan(B, Lq, Lk, H, Hkv, sm_count());
  if (ws_bytes < decode_workspace_bytes(pl, B, Lq, H, D)) return FA_ERR_SCRATCH_TOO_SMALL;
  const WsView w = ws_view(const_cast<void*>(ws), pl, B, Lq, H, D);
  const int nrows = B * H * Lq;
  fa_decode_combine_kernel<D, BF16><<<(nrows + 7) / 8, 256, 0, s>>>(w.part_o, w.part_lse, O, LSE, B,
                                                                    Lq, H, pl.nsplit);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status run_decode_slices(const void* Q, const void* K, const void* V, void* ws, size_t ws_bytes,
                            int B, int Lq, int Lk, int H, int Hkv, int D, int causal, int dtype,
                            cudaStream_t s) {
  const bool bf16 = dtype == FA_BF16;
  if (D == 64)
    return bf16 ? launch_slices<64, true>(Q, K, V, ws, ws_bytes, B, Lq, Lk, H, Hkv, causal, s)
                : launch_slices<64, false>(Q, K, V, ws, ws_bytes, B, Lq, Lk, H, Hkv, causal, s);
  return bf16 ? launch_slices<128, true>(Q, K, V, ws, ws_bytes, B, Lq, Lk, H, Hkv, causal, s)
              : launch_slices<128, false>(Q, K, V, ws, ws_bytes, B, Lq, Lk, H, Hkv, causal, s);
}

fa_status run_decode_merge(const void* ws, size_t ws_bytes, void* O, float* LSE, int B, int Lq,
                           int Lk, int H, int Hkv, int D, int dtype, cudaStream_t s) {
  const bool bf16 = dtype == FA_BF16;
  if (D == 64)
    return bf16 ? launch_merge<64, true>(ws, ws_bytes, O, LSE, B, Lq, Lk, H, Hkv, s)
                : launch_merge<64, false>(ws, ws_bytes, O, LSE, B, Lq, Lk, H, Hkv, s);
  return bf16 ? launch_merge<128, true>(ws, ws_bytes, O, LSE, B, Lq, Lk, H, Hkv, s)
              : launch_merge<128, false>(ws, ws_bytes, O, LSE, B, Lq, Lk, H, Hkv, s);
}

fa_status run_decode(const void* Q, const void* K, const void* V, void* O, float* LSE, void* ws,
                     size_t ws_bytes, int B, int Lq, int Lk, int H, int Hkv, int D, int causal,
                     int dtype, cudaStream_t s) {
  const fa_status st =
      run_decode_slices(Q, K, V, ws, ws_bytes, B, Lq, Lk, H, Hkv, D, causal, dtype, s);
  if (st != FA_OK) return st;
  return run_decode_merge(ws, ws_bytes, O, LSE, B, Lq, Lk, H, Hkv, D, dtype, s);
}

size_t decode_workspace_size(int B, int Lq, int Lk, int H, int Hkv, int D) {
  return decode_workspace_bytes(decode_plan(B, Lq, Lk, H, Hkv, sm_count()), B, Lq, H, D);
}

unsigned int decode_read_error(cudaStream_t s) { return read_and_clear_error(s); }

}  // namespace fa
