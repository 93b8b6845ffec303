// Split-KV decoding: a few queries (Lq small) against a long key/value
// sequence, forward only.
//
// Method: the online-softmax forward of page "使用 TileLang 在 AMD GPU 上快速开发
// 高性能 Flash Attention" (section "K/V Tile 遍历与核心计算"), run over one slice
// of the keys per CTA, after which the slices' partial results are merged by
// their log-sum-exp.  Page "TileLang性能分析报告：H100上FlashAttention吞吐量达
// 1.2PFlops" (section "生产环境部署建议", item 2) only names flash_decoding for
// inference; the slicing and the merge are the plain reading of that name, and
// the merged result equals the forward over all keys up to rounding.  Causal
// masking follows the past_len rule of the same page's causal-mask section,
// with past_len = Lk - Lq (the queries are the last Lq positions).
//
// GB300 design: one CTA per (batch, K/V head, key slice), 192 threads.  The
// group's g query heads x Lq queries are packed into the rows of one 128-row
// tile (row r = query r / g, head r % g of the group; one 4-D TMA box of
// head-dim x g heads x Lq queries), so every K/V tile loaded feeds all of them
// and K/V are read once per (batch, K/V head).
//   warps 0-3  softmax (thread = packed row = TMEM lane) and epilogue; warps
//              whose 32 rows are all padding sit the loop out
//   warp  4    TMA producer: packed Q once, then K_0, and K_{j+1}, V_j per tile
//   warp  5    TMEM allocator and tcgen05.mma issuer
// S is double-buffered in TMEM: S(j+1) = Q K_{j+1}^T runs while tile j is
// exponentiated.  P overwrites its S buffer as 16-bit values and is the A
// operand of O += P V_j.  Padding rows of Q are zero, so their S and P are
// zero and their O rows stay zero (never stored).  Each slice writes
// O_s = (sum_j P_j V_j) / l_s and LSE_s (natural log) in fp32 to the caller's
// workspace; fa_decode_combine_kernel merges the slices.  The work is bound by
// HBM reads of K and V: two 128 x D tiles per 128 keys.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "fwd.cuh"  // pack2
#include "ptx.cuh"

namespace fa {

struct DecParams {
  float* part_o;    // [nsplit, B, H, Lq, D] fp32
  float* part_lse;  // [nsplit, B, H, Lq] fp32
  int B, Lq, Lk, H, Hkv;
  int g;          // H / Hkv
  int rows;       // g * Lq <= 128 packed rows
  int causal, past;
  int n_kv;       // ceil(Lk / 128)
  int tps;        // K/V tiles per slice
  int nsplit;     // slices per (b, kv head); every slice has >= 1 tile
  float sl2;      // log2(e) / sqrt(D)
};

template <int D>
struct DecLayout {
  static constexpr int KCH = D / 64;
  static constexpr uint32_t CHUNK = 128u * 128u;  // 128 rows x 64 columns x 2 B
  static constexpr uint32_t TILE = KCH * CHUNK;
  static constexpr int STAGES = (D == 128) ? 6 : 12;
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t RING_OFF = TILE;
  static constexpr uint32_t BAR_OFF = RING_OFF + STAGES * TILE;
  static constexpr int B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = 1 + STAGES, B_SFULL = 1 + 2 * STAGES,
                       B_PFULL = B_SFULL + 2, B_PVDONE = B_PFULL + 2, B_OFULL = B_PVDONE + 2,
                       B_DONE = B_OFULL + 1, NBAR = B_DONE + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr uint32_t SMEM_USED = MISC_OFF + 16;
  static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int NTHREADS = 192;
  static_assert(SMEM_ALLOC <= 232448, "shared memory");
};

template <int D, bool BF16>
__global__ void __launch_bounds__(192, 1)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const DecParams p) {
  using Ly = DecLayout<D>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr uint32_t IDESC_S = idesc_f16(BF16, 128, 128, false, false);
  constexpr uint32_t IDESC_PV = idesc_f16(BF16, 128, D, false, true);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + Ly::BAR_OFF + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Ly::MISC_OFF);
  AbortState* ab = reinterpret_cast<AbortState*>(gbase + Ly::MISC_OFF + 8);
  unsigned int* err = device_error_word();
  const uint32_t warp = warp_id(), lane = lane_id();

  const int s_idx = blockIdx.x % p.nsplit;
  const int bh = blockIdx.x / p.nsplit;
  const int b = bh / p.Hkv, hkv = bh - (bh / p.Hkv) * p.Hkv;
  const int j0 = s_idx * p.tps;
  const int n = min(p.n_kv, j0 + p.tps) - j0;  // K/V tiles of this slice (>= 1)
  const int live_warps = (p.rows + 31) >> 5;

  // Padding rows [rows, 128) of the Q tile are zero; TMA fills rows [0, rows).
  for (uint32_t i = threadIdx.x; i < Ly::KCH * 128u * 8u; i += blockDim.x) {
    const uint32_t c = i / 1024u, rem = i % 1024u, r = rem / 8u, u = rem % 8u;
    if (r >= static_cast<uint32_t>(p.rows))
      reinterpret_cast<uint4*>(gbase + Ly::Q_OFF + c * Ly::CHUNK + r * 128u)[u] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_QFULL), 1);
    for (int s = 0; s < Ly::STAGES; ++s) {
      mbar_init(bar(Ly::B_KVFULL + s), 1);
      mbar_init(bar(Ly::B_KVEMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(Ly::B_SFULL + i), 1);
      mbar_init(bar(Ly::B_PFULL + i), 32 * live_warps);
      mbar_init(bar(Ly::B_PVDONE + i), 1);
    }
    mbar_init(bar(Ly::B_OFULL), 1);
    mbar_init(bar(Ly::B_DONE), 1);
    ab->flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(base + Ly::MISC_OFF, Ly::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // Ring order matches the issuer's consumption: K_0, then K_{j+1}, V_j.
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued[Ly::STAGES];
      for (int s = 0; s < Ly::STAGES; ++s) issued[s] = 0;
      mbar_arrive_expect_tx(bar(Ly::B_QFULL), Ly::KCH * p.rows * 128u);
      for (int c = 0; c < Ly::KCH; ++c)
        tma_load_4d(base + Ly::Q_OFF + c * Ly::CHUNK, &tmQ, bar(Ly::B_QFULL), c * 64, hkv * p.g, 0, b);
      auto load = [&](const CUtensorMap* map, int tile) -> bool {
        if (!mbar_wait(bar(Ly::B_KVEMPTY + stage), phase ^ 1u, ab, err, 801)) return false;
        mbar_arrive_expect_tx(bar(Ly::B_KVFULL + stage), Ly::TILE);
        for (int c = 0; c < Ly::KCH; ++c)
          tma_load_4d(base + Ly::RING_OFF + stage * Ly::TILE + c * Ly::CHUNK, map,
                      bar(Ly::B_KVFULL + stage), c * 64, hkv, tile * 128, b);
        ++issued[stage];
        if (++stage == Ly::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        return true;
      };
      bool ok = load(&tmK, j0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n && !load(&tmK, j0 + j + 1)) { ok = false; break; }
        if (!load(&tmV, j0 + j)) ok = false;
      }
      mbar_wait_drain(bar(Ly::B_QFULL), 0);
      if (!ok)
        for (int s = 0; s < Ly::STAGES; ++s)
          if (issued[s] > 0) mbar_wait_drain(bar(Ly::B_KVFULL + s), (issued[s] - 1) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, p_cnt[2] = {0, 0};
      bool ok = mbar_wait(bar(Ly::B_QFULL), 0, ab, err, 802);
      tc_fence_after();
      auto take = [&](uint32_t& slot, unsigned int site) -> bool {
        slot = stage;
        if (!mbar_wait(bar(Ly::B_KVFULL + stage), phase, ab, err, site)) return false;
        if (++stage == Ly::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        tc_fence_after();
        return true;
      };
      auto issue_s = [&](int buf, uint32_t kslot) {
        const uint32_t qa = base + Ly::Q_OFF, ka = base + Ly::RING_OFF + kslot * Ly::TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * Ly::CHUNK + (k & 3) * 32u;
          mma_ss(tmem + (buf ? Ly::TM_S1 : Ly::TM_S0), sdesc_sw128(qa + off, 16, 1024),
                 sdesc_sw128(ka + off, 16, 1024), IDESC_S, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(Ly::B_SFULL + buf));
        tc_commit(bar(Ly::B_KVEMPTY + kslot));
      };
      uint32_t ks = 0;
      if (ok && take(ks, 803))
        issue_s(0, ks);
      else
        ok = false;
      for (int j = 0; ok && j < n; ++j) {
        const int buf = j & 1;
        if (j + 1 < n) {
          // Buffer buf^1 held P(j-1); PV(j-1) was issued earlier by this
          // thread and tcgen05 MMAs execute in issue order.
          if (!take(ks, 804)) { ok = false; break; }
          issue_s(buf ^ 1, ks);
        }
        uint32_t vs;
        if (!take(vs, 805)) { ok = false; break; }
        if (!mbar_wait(bar(Ly::B_PFULL + buf), p_cnt[buf] & 1, ab, err, 806)) { ok = false; break; }
        ++p_cnt[buf];
        tc_fence_after();
        const uint32_t va = base + Ly::RING_OFF + vs * Ly::TILE;
        const uint32_t tP = tmem + (buf ? Ly::TM_S1 : Ly::TM_S0);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + Ly::TM_O, tP + 8u * k, sdesc_sw128(va + 2048u * k, Ly::CHUNK, 1024),
                 IDESC_PV, (j > 0 || k > 0) ? 1u : 0u);
        tc_commit(bar(Ly::B_PVDONE + buf));
        tc_commit(bar(Ly::B_KVEMPTY + vs));
        if (j == n - 1) tc_commit(bar(Ly::B_OFULL));
      }
      tc_commit(bar(Ly::B_DONE));
      mbar_wait_drain(bar(Ly::B_DONE), 0);
    }
  } else if (static_cast<int>(warp) < live_warps) {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = threadIdx.x;  // packed row == TMEM lane
    const uint32_t lane_off = ((warp & 3u) * 32u) << 16;
    const int ql = r / p.g, hh = r - ql * p.g;  // query, head within the group
    const float sl2 = p.sl2;
    const int lim = p.causal ? min(ql + p.past + 1, p.Lk) : p.Lk;  // keys [0, lim) visible
    float m = -INFINITY, l = 0.f;
    uint32_t s_cnt[2] = {0, 0};
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int buf = j & 1;
      if (!mbar_wait_warp(bar(Ly::B_SFULL + buf), s_cnt[buf] & 1, ab, err, 807)) { ok = false; break; }
      ++s_cnt[buf];
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + (buf ? Ly::TM_S1 : Ly::TM_S0);
      uint32_t sr[128];
      tmem_ld32(tS + 0, sr);
      tmem_ld32(tS + 32, sr + 32);
      tmem_ld32(tS + 64, sr + 64);
      tmem_ld32(tS + 96, sr + 96);
      tmem_ld_wait32(sr);
      tmem_ld_wait32(sr + 32);
      tmem_ld_wait32(sr + 64);
      tmem_ld_wait32(sr + 96);
      const int k0 = (j0 + j) * 128;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        if (k0 + c >= lim) sr[c] = __float_as_uint(-INFINITY);
        mx = fmaxf(mx, __uint_as_float(sr[c]));
      }
      const float m_new = fmaxf(m, mx);
      // A row with no visible key yet (m = -inf) has accumulated nothing and
      // takes the new max directly.  Otherwise the max is moved only when it
      // grew by more than 2^8 (exp2 units) somewhere in the warp, and O is
      // rescaled then; the stale max is used for l and O alike.
      const bool fresh = (m == -INFINITY);
      const bool grow = !fresh && (m_new - m) * sl2 > 8.0f;
      float alpha = 1.f;
      const bool rescale = __any_sync(0xffffffffu, grow);
      if (rescale && !fresh) alpha = ex2((m - m_new) * sl2);
      if (rescale || fresh) m = m_new;
      const float mb = (m == -INFINITY) ? 0.f : m * sl2;
      float rs = 0.f;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[32 * q4 + 2 * i]), sl2, -mb));
          const float p1 = ex2(fmaf(__uint_as_float(sr[32 * q4 + 2 * i + 1]), sl2, -mb));
          rs += p0 + p1;
          pk[i] = pack2<T>(p0, p1);
        }
        tmem_st16(tS + 16 * q4, pk);
      }
      if (rescale) {
        // O must hold PV(j-1) before it is scaled.  PV products of odd and
        // even tiles signal separate barriers; on the one of tile j-1, the
        // product two tiles earlier completed long ago (before S(j)) and the
        // one two tiles later cannot start before this warp arrives, so the
        // parity names the phase of PV(j-1) exactly.
        if (!mbar_wait_warp(bar(Ly::B_PVDONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, ab, err, 808)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + Ly::TM_O + 32 * cc, o);
          tmem_ld_wait32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_off + Ly::TM_O + 32 * cc, o);
        }
      }
      l = l * alpha + rs;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Ly::B_PFULL + buf));
    }
    if (ok && mbar_wait_warp(bar(Ly::B_OFULL), 0, ab, err, 809)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool valid = r < p.rows;
      const int h = hkv * p.g + hh;
      const size_t row_idx = ((static_cast<size_t>(s_idx) * p.B + b) * p.H + h) * p.Lq + ql;
      float* dst = p.part_o + row_idx * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + Ly::TM_O + 32 * cc, o);
        tmem_ld_wait32(o);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(dst + 32 * cc)[i] =
                make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                            __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
        }
      }
      if (valid)
        p.part_lse[row_idx] = l > 0.f ? (m * sl2 + __log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Ly::TMEM_COLS);
  }
}

// Merge the slices of every (b, h, query): LSE = ln sum_s exp(LSE_s) and
// O = sum_s exp(LSE_s - LSE) O_s.  One warp per row; lanes split the head dim.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
    fa_decode_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                             void* __restrict__ O, float* __restrict__ LSE, int B, int Lq, int H,
                             int nsplit) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);  // (b, h, l) flattened, l fastest
  const int lane = threadIdx.x & 31;
  const int nrows = B * H * Lq;
  if (row >= nrows) return;
  const size_t slab = static_cast<size_t>(nrows);
  float mx = -INFINITY;
  for (int s = 0; s < nsplit; ++s) mx = fmaxf(mx, part_lse[s * slab + row]);
  float den = 0.f;
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float w = __expf(part_lse[s * slab + row] - mx);
      den += w;
      const float* src = part_o + (s * slab + row) * D;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, src[lane + 32 * e], acc[e]);
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const int l = row % Lq, bh = row / Lq;
  const int h = bh % H, b = bh / H;
  T* dst = reinterpret_cast<T*>(O) + ((static_cast<size_t>(b) * Lq + l) * H + h) * D;
#pragma unroll
  for (int e = 0; e < PER; ++e) dst[lane + 32 * e] = static_cast<T>(acc[e] * inv);
  if (lane == 0) LSE[row] = den > 0.f ? mx + __logf(den) : -INFINITY;
}

}  // namespace fa
