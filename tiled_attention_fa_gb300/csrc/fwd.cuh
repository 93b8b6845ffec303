// Forward tiled online-softmax attention for sm_103a.
//
// Method (page "使用 TileLang 在 AMD GPU 上快速开发高性能 Flash Attention",
// sections "Q Tile 处理与缓存初始化", "K/V Tile 遍历与核心计算" and
// "最终输出写回与Q tile 迭代"): each 128-row Q tile streams its K/V tiles,
// keeps a running row max m and row sum l in fp32, rescales the output
// accumulator when the max moves, turns scores into probabilities with the
// scale folded into the exponent, down-casts P to the input type before the PV
// product, and divides by l at the end.  Causal tiles past the diagonal are
// never visited; K/V heads are shared by groups of query heads.
//
// GB300 design (not the page's): one persistent CTA per SM, 320 threads.
//   warps 0-3  softmax warpgroup for Q tile 0 (thread i owns row i)
//   warps 4-7  softmax warpgroup for Q tile 1
//   warp  8    TMA producer: Q pair, then (V_{j-1}, K_j) tile pairs into a ring
//   warp  9    TMEM allocator and MMA issuer (the warp runs the schedule,
//              one elected lane issues the MMAs and their commits)
// Registers are not re-balanced between warps (no setmaxnreg): the softmax
// fits the uniform budget of 168 per thread.  (The backward does move
// registers between warpgroups; its launcher checks the launch allocation the
// split relies on.)
// A work item is (batch, head, pair of 128-row Q tiles).  S_t = Q_t K_j^T and
// O_t += P_t V_j accumulate in tensor memory; P_t overwrites S_t in TMEM as
// 16-bit values and is read from there by the PV MMA.  While warpgroup 0
// turns S_0 into P_0 the tensor cores compute S_1 (and the reverse), so the
// exponentials overlap the MMAs.  O is rescaled only when a row max grows by
// more than 2^8 (in exp2 units); the stale max is used consistently for l and
// O, so the final O / l is exact up to rounding.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace fa {

struct FwdParams {
  void* O;      // [B, Lq, H, D] fp16/bf16
  float* LSE;   // [B, H, Lq] fp32, natural log
  int B, Lq, Lk, H, Hkv, causal;
  int past;      // Lk - Lq: causal offset (query i sees keys j <= i + past)
  int n_kv;      // ceil(Lk / 128)
  int n_qpairs;  // ceil(Lq / 256)
  int n_items;   // B * H * n_qpairs
  float sl2;     // log2(e) / sqrt(D) (times q_scale * k_scale for E4M3 inputs)
  float o_scale; // factor on O / l at the store: 1, or v_scale for E4M3 inputs
  int sorted;    // 1: items ordered by decreasing work across all heads (else head-major)
};

// FP8: Q, K, V are E4M3 codes (one byte per element; D = 128 only).
template <int D, bool FP8 = false>
struct FwdLayout {
  static constexpr int EB = FP8 ? 1 : 2;          // bytes per input element
  static constexpr int KCH = D * EB / 128;        // 128-byte column chunks per row
  static constexpr uint32_t CHUNK = 128u * 128u;  // 128 rows x 128 B
  static constexpr uint32_t TILE = KCH * CHUNK;   // one 128 x D tile
  // Ring stages, each holding a pair of tiles: (V_{j-1}, K_j), the tiles one
  // step of the MMA schedule consumes (V_{j-1} for P V, K_j for the next S).
  static constexpr int STAGES = FP8 ? 5 : ((D == 128) ? 2 : 4);
  static constexpr int KS_S = D * EB / 32;        // MMA steps of S = Q K^T (32 bytes of K each)
  static constexpr int KS_PV = 4 * EB;            // MMA steps of O += P V (32 / EB keys each)
  static constexpr uint32_t V_STEP = (32 / EB) * 128u;  // V bytes per PV step
  static_assert(!FP8 || D == 128, "E4M3 inputs need D = 128");
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t RING_OFF = 2 * TILE;
  static constexpr uint32_t BAR_OFF = RING_OFF + STAGES * 2 * TILE;
  // barrier slots
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KVFULL = 2, B_KVEMPTY = 2 + STAGES,
                       B_SFULL = 2 + 2 * STAGES, B_PFULL = B_SFULL + 2, B_OFULL = B_PFULL + 4,
                       B_OEMPTY = B_OFULL + 2, B_DONE = B_OEMPTY + 2, NBAR = B_DONE + 1;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr uint32_t SMEM_USED = MISC_OFF + 16;
  static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 256 + D;
  // At D = 64 (16-bit inputs) the Q tiles also live in TMEM (32 columns of
  // 16-bit pairs each), copied there once per item, so S = Q K^T reads only
  // K from shared memory.
  static constexpr bool Q_TMEM = (D == 64 && !FP8);
  static constexpr uint32_t TM_Q0 = 256 + 2 * D, TM_Q1 = TM_Q0 + D / 2;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(TM_O1 + D <= TMEM_COLS, "TMEM regions overflow");
  static_assert(!Q_TMEM || TM_Q1 + D / 2 <= TMEM_COLS, "TMEM copies of Q overflow");
  static_assert(SMEM_ALLOC <= 232448, "shared memory beyond the 227 KB per-block limit");
  static constexpr int NTHREADS = 320;
};

struct FwdItem {
  int b, h, hkv, q0;
  int n[2];  // KV tiles visited by Q tile 0 / 1 (0 = tile lies past L)
};

__device__ __forceinline__ FwdItem fwd_decode(int item, const FwdParams& p) {
  FwdItem it;
  int bh, qp;
  if (p.sorted) {
    // Pair index falling (work falling under causal masking), all heads of
    // one pair index together.
    const int nbh = p.n_items / p.n_qpairs;
    const int r = item / nbh;
    bh = item - r * nbh;
    qp = p.n_qpairs - 1 - r;
  } else {
    // Head-major; within a head, pairs run from the last (longest under
    // causal) to the first.
    bh = item / p.n_qpairs;
    qp = p.n_qpairs - 1 - (item - bh * p.n_qpairs);
  }
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  it.hkv = it.h / (p.H / p.Hkv);
  it.q0 = qp * 256;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int lo = it.q0 + 128 * t;
    if (lo >= p.Lq) it.n[t] = 0;
    else it.n[t] = p.causal ? min((lo + 127 + p.past) / 128 + 1, p.n_kv) : p.n_kv;
  }
  return it;
}

// Items are handed out in rounds of gridDim.x, alternating direction each
// round (CTA c takes position c, then G-1-c, ...).  Within a head the pairs
// run longest-first, so under causal masking every CTA gets a mix of long
// and short items; consecutive items still share a head's K/V in L2.
__device__ __forceinline__ int fwd_item_of(int round) {
  const int G = static_cast<int>(gridDim.x);
  const int pos = (round & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  return round * G + pos;
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int D, bool BF16, bool FP8 = false>
__global__ void __launch_bounds__(320, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using Ly = FwdLayout<D, FP8>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  // Operand formats: F16 = 0 / BF16 = 1 for 16-bit inputs; E4M3 = 0 under
  // .kind::f8f6f4 (BF16 then only selects the output type).
  constexpr uint32_t IDESC_S = idesc_f16(BF16 && !FP8, 128, 128, false, false);
  constexpr uint32_t IDESC_PV = idesc_f16(BF16 && !FP8, 128, D, false, true);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + Ly::BAR_OFF + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Ly::MISC_OFF);
  AbortState* ab = reinterpret_cast<AbortState*>(gbase + Ly::MISC_OFF + 8);
  unsigned int* err = fwd_error_word();

  const uint32_t warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::B_QFULL), 1);
    mbar_init(bar(Ly::B_QEMPTY), 1);
    for (int s = 0; s < Ly::STAGES; ++s) {
      mbar_init(bar(Ly::B_KVFULL + s), 1);
      mbar_init(bar(Ly::B_KVEMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(Ly::B_SFULL + t), 1);
      // P of tile t in two halves (keys 0-63, 64-127): one arrival per warp
      mbar_init(bar(Ly::B_PFULL + 2 * t), 4);
      mbar_init(bar(Ly::B_PFULL + 2 * t + 1), 4);
      mbar_init(bar(Ly::B_OFULL + t), 1);
      mbar_init(bar(Ly::B_OEMPTY + t), 4);
    }
    mbar_init(bar(Ly::B_DONE), 1);
    ab->flag = 0;
    fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 9) {
    tmem_alloc(base + Ly::MISC_OFF, Ly::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, q_uses = 0;
      uint32_t issued[Ly::STAGES];
      for (int s = 0; s < Ly::STAGES; ++s) issued[s] = 0;
      const uint64_t keep = policy_evict_last();
      bool ok = true;
      for (int round = 0; ok && round * static_cast<int>(gridDim.x) < p.n_items; ++round) {
        const int item = fwd_item_of(round);
        if (item >= p.n_items) continue;
        const FwdItem it = fwd_decode(item, p);
        if (q_uses > 0 && !mbar_wait(bar(Ly::B_QEMPTY), (q_uses - 1) & 1, ab, err, 101)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(Ly::B_QFULL), 2 * Ly::TILE);
        for (int t = 0; t < 2; ++t)
          for (int c = 0; c < Ly::KCH; ++c)
            tma_load_4d(base + Ly::Q_OFF + t * Ly::TILE + c * Ly::CHUNK, &tmQ, bar(Ly::B_QFULL),
                        c * (128 / Ly::EB), it.h, it.q0 + 128 * t, it.b);
        ++q_uses;
        const int nmax = max(it.n[0], it.n[1]);
        // Pair j = (V_{j-1}, K_j): the first has no V, the last no K.
        for (int j = 0; ok && j <= nmax; ++j) {
          if (!mbar_wait(bar(Ly::B_KVEMPTY + stage), phase ^ 1u, ab, err, 102)) {
            ok = false;
            break;
          }
          const uint32_t slot = base + Ly::RING_OFF + stage * 2 * Ly::TILE;
          mbar_arrive_expect_tx(bar(Ly::B_KVFULL + stage),
                                ((j > 0 ? 1u : 0u) + (j < nmax ? 1u : 0u)) * Ly::TILE);
          for (int c = 0; c < Ly::KCH; ++c) {
            if (j > 0)
              tma_load_4d_hint(slot + c * Ly::CHUNK, &tmV, bar(Ly::B_KVFULL + stage),
                               c * (128 / Ly::EB), it.hkv, (j - 1) * 128, it.b, keep);
            if (j < nmax)
              tma_load_4d_hint(slot + Ly::TILE + c * Ly::CHUNK, &tmK, bar(Ly::B_KVFULL + stage),
                               c * (128 / Ly::EB), it.hkv, j * 128, it.b, keep);
          }
          ++issued[stage];
          if (++stage == Ly::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Unwinding: let copies already in flight land before the CTA exits.
        if (q_uses > 0) mbar_wait_drain(bar(Ly::B_QFULL), (q_uses - 1) & 1);
        for (int s = 0; s < Ly::STAGES; ++s)
          if (issued[s] > 0) mbar_wait_drain(bar(Ly::B_KVFULL + s), (issued[s] - 1) & 1);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule, so loop state and operand descriptors
    // are warp-uniform values; one elected lane issues each MMA group and the
    // commits that track it.
    {
      uint32_t stage = 0, phase = 0, q_cnt = 0;
      // Per-tile counters of P hand-offs and O uses, kept in registers.
      uint32_t p_cnt0 = 0, p_cnt1 = 0, o_uses0 = 0, o_uses1 = 0;
      bool ok = true;
      auto tS = [&](int t) { return tmem + Ly::TM_S0 + (Ly::TM_S1 - Ly::TM_S0) * t; };
      auto tO = [&](int t) { return tmem + Ly::TM_O0 + (Ly::TM_O1 - Ly::TM_O0) * t; };
      auto commit = [&](int b) {
        if (elect_one()) tc_commit(bar(b));
        __syncwarp();
      };

      // Descriptors of the first K step; later steps add their byte offset
      // (>> 4) to the start-address field, which stays below 2^14.
      // K of pair `ps` is its second tile, V its first.
      auto issue_s = [&](int t, uint32_t ps) {
        const uint64_t qd = sdesc_sw128(base + Ly::Q_OFF + t * Ly::TILE, 16, 1024);
        const uint64_t kd =
            sdesc_sw128(base + Ly::RING_OFF + (2 * ps + 1) * Ly::TILE, 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < Ly::KS_S; ++k) {
            const uint64_t off = ((k >> 2) * Ly::CHUNK + (k & 3) * 32u) >> 4;
            if constexpr (FP8)
              mma_ss_f8(tS(t), qd + off, kd + off, IDESC_S, k > 0 ? 1u : 0u);
            else if constexpr (Ly::Q_TMEM)
              mma_ts(tS(t), tmem + (t ? Ly::TM_Q1 : Ly::TM_Q0) + 8u * k, kd + off, IDESC_S,
                     k > 0 ? 1u : 0u);
            else
              mma_ss(tS(t), qd + off, kd + off, IDESC_S, k > 0 ? 1u : 0u);
          }
        }
        __syncwarp();
      };
      // PV over the keys of K steps [k_lo, k_hi) of the tile.
      auto issue_pv = [&](int t, uint32_t ps, bool acc, int k_lo, int k_hi) {
        const uint64_t vd = sdesc_sw128(base + Ly::RING_OFF + 2 * ps * Ly::TILE, Ly::CHUNK, 1024);
        if (elect_one()) {
#pragma unroll
          for (int k = k_lo; k < k_hi; ++k) {
            // P: 8 TMEM columns (16 or 32 keys) per step; V read MN-major.
            const uint64_t off = (Ly::V_STEP * k) >> 4;
            if constexpr (FP8)
              mma_ts_f8(tO(t), tS(t) + 8u * k, vd + off, IDESC_PV, (acc || k > 0) ? 1u : 0u);
            else
              mma_ts(tO(t), tS(t) + 8u * k, vd + off, IDESC_PV, (acc || k > 0) ? 1u : 0u);
          }
        }
        __syncwarp();
      };
      auto take = [&](uint32_t& slot, unsigned int site) -> bool {
        slot = stage;
        if (!mbar_wait_warp(bar(Ly::B_KVFULL + stage), phase, ab, err, site)) return false;
        if (++stage == Ly::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        tc_fence_after();
        return true;
      };

      for (int round = 0; ok && round * static_cast<int>(gridDim.x) < p.n_items; ++round) {
        const int item = fwd_item_of(round);
        if (item >= p.n_items) continue;
        const FwdItem it = fwd_decode(item, p);
        const int nmax = max(it.n[0], it.n[1]);
        if (!mbar_wait_warp(bar(Ly::B_QFULL), q_cnt & 1, ab, err, 201)) { ok = false; break; }
        ++q_cnt;
        tc_fence_after();
        if constexpr (Ly::Q_TMEM) {
          // Both Q tiles into TMEM (after the previous item's S MMAs, which
          // read these columns and were issued before).
          if (elect_one()) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const uint64_t qd = sdesc_sw128(base + Ly::Q_OFF + t * Ly::TILE, 16, 1024);
#pragma unroll
              for (int k = 0; k < Ly::KS_S; ++k)
                tmem_cp_128x256b(tmem + (t ? Ly::TM_Q1 : Ly::TM_Q0) + 8u * k,
                                 qd + (((k >> 2) * Ly::CHUNK + (k & 3) * 32u) >> 4));
            }
          }
          __syncwarp();
          // The copies are the only readers of the Q tiles in shared memory:
          // the next item's Q may load as soon as they complete.
          commit(Ly::B_QEMPTY);
        }
        // Pair 0 holds K_0: the first S of both tiles.
        uint32_t ps;
        if (!take(ps, 202)) { ok = false; break; }
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (it.n[t] > 0) {
            issue_s(t, ps);
            commit(Ly::B_SFULL + t);
          }
        commit(Ly::B_KVEMPTY + ps);
        for (int j = 0; ok && j < nmax; ++j) {
          // Pair j+1 holds V_j and K_{j+1}.
          if (!take(ps, 203)) { ok = false; break; }
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            uint32_t& p_cnt = t ? p_cnt1 : p_cnt0;
            uint32_t& o_uses = t ? o_uses1 : o_uses0;
            if (j < it.n[t]) {
              if (j == 0 && o_uses > 0 &&
                  !mbar_wait_warp(bar(Ly::B_OEMPTY + t), (o_uses - 1) & 1, ab, err, 204)) {
                ok = false;
                break;
              }
              // PV on the first half of P while the softmax finishes the second.
              if (!mbar_wait_warp(bar(Ly::B_PFULL + 2 * t), p_cnt & 1, ab, err, 205)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_pv(t, ps, j > 0, 0, Ly::KS_PV / 2);
              if (!mbar_wait_warp(bar(Ly::B_PFULL + 2 * t + 1), p_cnt & 1, ab, err, 207)) {
                ok = false;
                break;
              }
              ++p_cnt;
              tc_fence_after();
              issue_pv(t, ps, true, Ly::KS_PV / 2, Ly::KS_PV);
              if (j == it.n[t] - 1) {
                commit(Ly::B_OFULL + t);
                ++o_uses;
              }
            }
            if (j + 1 < it.n[t]) {
              issue_s(t, ps);
              commit(Ly::B_SFULL + t);
            }
          }
          if (!ok) break;
          commit(Ly::B_KVEMPTY + ps);
        }
        if (!ok) break;
        if constexpr (!Ly::Q_TMEM) commit(Ly::B_QEMPTY);
      }
      // Every MMA issued by the elected lane completes before TMEM is released.
      commit(Ly::B_DONE);
      mbar_wait_drain(bar(Ly::B_DONE), 0);
    }
  }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;                       // Q tile of this warpgroup
    const int r = threadIdx.x & 127;               // row within the tile == TMEM lane
    const uint32_t lane_off = ((warp & 3u) * 32u) << 16;
    const uint32_t tS = tmem + lane_off + (t ? Ly::TM_S1 : Ly::TM_S0);
    const uint32_t tO = tmem + lane_off + (t ? Ly::TM_O1 : Ly::TM_O0);
    const float sl2 = p.sl2;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    for (int round = 0; ok && round * static_cast<int>(gridDim.x) < p.n_items; ++round) {
        const int item = fwd_item_of(round);
        if (item >= p.n_items) continue;
      const FwdItem it = fwd_decode(item, p);
      const int n = it.n[t];
      if (n == 0) continue;
      const int tile_lo = it.q0 + 128 * t;
      const int q = tile_lo + r;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        if (!mbar_wait_warp(bar(Ly::B_SFULL + t), s_cnt & 1, ab, err, 301)) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld32(tS + 0, sr);
        tmem_ld32(tS + 32, sr + 32);
        tmem_ld32(tS + 64, sr + 64);
        tmem_ld32(tS + 96, sr + 96);
        tmem_ld_wait32(sr);
        tmem_ld_wait32(sr + 32);
        tmem_ld_wait32(sr + 64);
        tmem_ld_wait32(sr + 96);
        const int k0 = j * 128;
        const bool need_mask = (k0 + 128 > p.Lk) || (p.causal && k0 + 127 > tile_lo + p.past);
        if (need_mask) {
          const int lim = p.causal ? min(q + p.past + 1, p.Lk) : p.Lk;  // keys [0, lim) visible
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (k0 + c >= lim) sr[c] = __float_as_uint(-INFINITY);
        }
        // The row max runs as eight independent chains of three-input max
        // operations (key 8w+u in chain u, 16 keys each) instead of 128
        // dependent ones, then combines the chains.
        float mx8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          mx8[u] = fmax3(__uint_as_float(sr[u]), __uint_as_float(sr[8 + u]), __uint_as_float(sr[16 + u]));
#pragma unroll
          for (int w = 3; w < 15; w += 2)
            mx8[u] = fmax3(mx8[u], __uint_as_float(sr[8 * w + u]), __uint_as_float(sr[8 * w + 8 + u]));
          mx8[u] = fmaxf(mx8[u], __uint_as_float(sr[120 + u]));
        }
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        const float m_new = fmaxf(m, mx);
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m = m_new;
        } else if (__any_sync(0xffffffffu, (m_new - m) * sl2 > 8.0f)) {
          // The running max grew by more than 2^8 somewhere in this warp:
          // rescale this warp's rows (others get alpha = 1).
          alpha = ex2((m - m_new) * sl2);
          m = m_new;
          rescale = true;
        }
        // Half h of P is in TMEM: this thread's stores complete, then one
        // lane per warp signals the MMA warp.  Before the first half, O of
        // this row is scaled by alpha if the max moved (this tile's PV
        // accumulates into it next; the previous PV has completed, as the
        // commit that signalled this tile's S covers it).  That happens once
        // the first half's scores are spent, so their registers hold O.
        auto p_ready = [&](int h) {
          if (h == 0 && rescale) {
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32(tO + 32 * cc, o);
              tmem_ld_wait32(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO + 32 * cc, o);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(Ly::B_PFULL + 2 * t + h));
        };
        const float mb = m * sl2;
        float rs = 0.f;
        if constexpr (FP8) {
          // Exponent arguments and the row sum on paired fp32 instructions
          // (two keys per FMA / ADD), the sum over four independent pairs.
          const uint64_t sl2x2 = f2_pack(sl2, sl2), nmb2 = f2_pack(-mb, -mb);
          uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int c = 64 * h2 + 4 * i;
              float a0, a1, a2, a3;
              f2_unpack(ffma2(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2, nmb2), a0, a1);
              f2_unpack(ffma2(f2_pack(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), sl2x2, nmb2), a2, a3);
              const float p0 = ex2(a0), p1 = ex2(a1), p2 = ex2(a2), p3 = ex2(a3);
              acc[2 * (i & 1)] = fadd2(acc[2 * (i & 1)], f2_pack(p0, p1));
              acc[2 * (i & 1) + 1] = fadd2(acc[2 * (i & 1) + 1], f2_pack(p2, p3));
              pk[i] = pack4_e4m3(p0, p1, p2, p3);
            }
            tmem_st16(tS + 16 * h2, pk);
            p_ready(h2);
          }
          float rs4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float lo, hi;
            f2_unpack(acc[u], lo, hi);
            rs4[u] = lo + hi;
          }
          rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        } else {
          // Exponent arguments and the row sum on paired fp32 instructions
          // (two keys per FMA / ADD), the sum over four independent pairs.
          const uint64_t sl2x2 = f2_pack(sl2, sl2), nmb2 = f2_pack(-mb, -mb);
          uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int c = 32 * q4 + 2 * i;
              float a0, a1;
              f2_unpack(ffma2(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2, nmb2), a0, a1);
              const float p0 = ex2(a0), p1 = ex2(a1);
              acc[i & 3] = fadd2(acc[i & 3], f2_pack(p0, p1));
              pk[i] = pack2<T>(p0, p1);
            }
            tmem_st16(tS + 16 * q4, pk);
            if (q4 & 1) p_ready(q4 >> 1);
          }
          float rs4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float lo, hi;
            f2_unpack(acc[u], lo, hi);
            rs4[u] = lo + hi;
          }
          rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        }
        l = l * alpha + rs;
      }
      if (!ok) break;
      // ---- epilogue: O / l, LSE
      if (!mbar_wait_warp(bar(Ly::B_OFULL + t), o_cnt & 1, ab, err, 302)) { ok = false; break; }
      ++o_cnt;
      tc_fence_after();
      const float inv = l > 0.f ? p.o_scale / l : 0.f;
      T* orow = reinterpret_cast<T*>(p.O) + ((static_cast<size_t>(it.b) * p.Lq + q) * p.H + it.h) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * cc, o);
        tmem_ld_wait32(o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<T>(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        if (q < p.Lq) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cc);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (q < p.Lq)
        p.LSE[(static_cast<size_t>(it.b) * p.H + it.h) * p.Lq + q] =
            (m * sl2 + __log2f(l)) * 0.6931471805599453f;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::B_OEMPTY + t));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Ly::TMEM_COLS);
  }
}

}  // namespace fa
