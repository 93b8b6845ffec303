// Backward attention kernels for sm_103a.
//
// Method (page "TileLang与机器学习训练：反向传播算子优化案例", sections
// 算子拆分与流水线设计 and 内存布局优化): three stages --
//   1. preprocess: Delta_i = sum_d O_id dO_id per query row;
//   2. main pass: one CTA per K/V tile that loops over the Q tiles,
//      recomputes the transposed scores, accumulates dV from the transposed
//      probabilities (and, completing the elided steps with the analytic
//      gradient, dK from dS^T Q), and adds each dQ partial into an fp32
//      accumulator with atomics laid out to match the accumulator fragments;
//   3. post-process: scale and convert the dQ accumulator back to BSHD.
//
// GB300 design of the main pass (512 threads, one persistent CTA per SM; a
// work unit is one or two 128-key K/V tiles of one head, see bwd_unit_item):
//   warps 0-7  compute warps: each query half of a tile (columns 0-63, then
//              64-127) is split over all eight, warp w taking 32 columns
//              of key rows 32*(w%4).. (its TMEM lanes); a thread owns one
//              key row and forms P^T = exp2(S^T*c - LSE*log2e) for both
//              halves as soon as S^T lands, then dS^T = P^T o (dP^T - Delta)
//              for both once dP^T does; both go back to TMEM over the
//              chunk's S^T columns (A operands of dV += P^T dO and
//              dK += dS^T Q) and dS^T also to a swizzled smem tile (read
//              MN-major as the A operand of dQ = dS K).  At the end warps
//              0-3 write dK and warps 4-7 dV.
//   warps 8-11 dQ drain: thread r owns query row r; takes the whole dQ row
//              from TMEM, releases the columns, then adds it into the fp32
//              accumulator with paced 16-byte vector reductions.
//   warp  12   TMA producer: K_j, V_j once per K/V tile (two slots at D = 64,
//              so the next tile's load overlaps the current one); then dO_i
//              and Q_i (with LSE_i, Delta_i) through a two-slot ring whose dO
//              and Q halves are released separately (after their last
//              readers, dV and dK).
//   warp  13   TMEM allocator and MMA issuer (the warp runs the schedule,
//              one elected lane issues the MMAs and their commits).
//   warps 14-15 idle (they only lower their register budget with 12-13).
// The S^T and dP^T tiles alternate between two TMEM regions with the tile
// counter, so the next tile's S^T is issued as soon as the compute warps have
// consumed this tile's dP^T, ahead of this tile's last dK and its dQ.
// An MMA with both operands in shared memory reads them at the shared-memory
// rate (128 B per clock: an M=128 N=128 K=16 step, 8 KB, takes its 64 tensor
// cycles in reads alone), so the schedule keeps every operand it can in TMEM:
// per tile S^T and dP^T (both operands in shared memory, N = 128 queries;
// at D = 64 K_j and V_j are copied into spare TMEM columns once per K/V tile
// and these read only Q / dO), dV and dK (A from TMEM), dQ (both in shared
// memory): 40 MMAs, 256 KB of operand reads at D = 128.  dK and dV stay in
// TMEM for a whole K/V tile; for grouped-query attention the CTA loops over
// every query head of its K/V head, so dK/dV need no atomics.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "fwd.cuh"  // pack2
#include "ptx.cuh"

// Pacing of the dQ drain's reductions: a pause of FA_BWD_PACE_NS after every
// FA_BWD_PACE_EVERY reductions at D = 128, and at D = 64 unless
// FA_BWD_PACE_D64 is 0 (see the drain).
#ifndef FA_BWD_PACE_NS
#define FA_BWD_PACE_NS 100
#endif
#ifndef FA_BWD_PACE_EVERY
#define FA_BWD_PACE_EVERY 2
#endif
#ifndef FA_BWD_PACE_D64
#define FA_BWD_PACE_D64 1
#endif



namespace fa {

struct BwdParams {
  const float* LSE;    // [B, H, Lq]
  const float* Delta;  // [B, H, Lq]
  float* dq_accum;     // [B, H, D/4, Lpad, 4], Lpad = n_q * 128
  void* dK;            // [B, Lk, Hkv, D]
  void* dV;            // [B, Lk, Hkv, D]
  int B, Lq, Lk, H, Hkv, causal;
  int past;     // Lk - Lq: query i sees keys j <= i + past under causal masking
  int n_kv;     // ceil(Lk / 128) K/V tiles
  int n_q;      // ceil(Lq / 128) Q tiles
  int Lpad;     // n_q * 128
  int n_items;  // B * Hkv * n_kv
  int n_units;  // work units of the persistent CTAs (see bwd_unit_item)
  int ipu;      // K/V tiles per unit: 2 under causal masking, else 1
  int snake;    // 1: units are single tiles in decreasing-work order, dealt out in snake order
  float sl2;    // log2(e) / sqrt(D)
  float scale;  // 1 / sqrt(D)
};

template <int D>
struct BwdLayout {
  static constexpr int KCH = D / 64;
  static constexpr uint32_t CHUNK = 128u * 128u;
  static constexpr uint32_t TILE = KCH * CHUNK;
  static constexpr int STAGES = 2;
  // K/V slots: at D = 64 shared memory has room for a second (K, V) pair, so
  // the next K/V tile loads while the current one is in use.
  static constexpr int KVS = (D == 64) ? 2 : 1;
  // Small region first (barriers, TMEM address, abort flag, LSE/Delta slots),
  // then the 1024-byte aligned operand tiles.
  static constexpr int B_KVFULL = 0, B_QFULL = KVS, B_QEMPTY = KVS + STAGES,
                       B_SFULL = KVS + 2 * STAGES,
                       B_DPFULL = B_SFULL + 1, B_PFULL = B_DPFULL + 1, B_DSFULL = B_PFULL + 2,
                       B_DQFULL = B_DSFULL + 2, B_DQEMPTY = B_DQFULL + 1,
                       B_DKVFULL = B_DQEMPTY + 1, B_DONE = B_DKVFULL + 1, B_KVEMPTY = B_DONE + 1,
                       B_DOFULL = B_KVEMPTY + KVS, B_DOEMPTY = B_DOFULL + STAGES,
                       NBAR = B_DOEMPTY + STAGES;
  static constexpr uint32_t BAR_OFF = 0;
  static constexpr uint32_t MISC_OFF = BAR_OFF + NBAR * 8;              // tmem slot, abort flag
  static constexpr uint32_t STAT_OFF = (MISC_OFF + 16 + 15) / 16 * 16;  // [STAGES][2][128] f32
  static constexpr uint32_t SMALL_END = STAT_OFF + STAGES * 2 * 128 * 4;
  static constexpr uint32_t TILE_BASE = (SMALL_END + 1023) / 1024 * 1024;
  static constexpr uint32_t KV_OFF = TILE_BASE;                 // [KVS] (K, V) tile pairs
  __host__ __device__ static constexpr uint32_t k_off(int slot) { return KV_OFF + 2u * slot * TILE; }
  __host__ __device__ static constexpr uint32_t v_off(int slot) { return k_off(slot) + TILE; }
  static constexpr uint32_t Q_OFF = KV_OFF + 2 * KVS * TILE;   // [STAGES] tiles
  static constexpr uint32_t DO_OFF = Q_OFF + STAGES * TILE;   // [STAGES] tiles
  static constexpr uint32_t DS_OFF = DO_OFF + STAGES * TILE;  // 2 chunks (128 keys x 128 queries)
  static constexpr uint32_t SMEM_ALLOC = DS_OFF + 2 * CHUNK;
  // TMEM columns: dK | dV | R0 | R1, two 128-column regions that alternate
  // with the CTA's tile counter g: S^T(g) goes into R[g % 2] and dP^T(g) into
  // the other.  The compute warps overwrite each 32-query chunk of S^T with
  // P^T (16 columns of 16-bit pairs) and dS^T (the next 16), the A operands
  // of the dV and dK products; dQ(g) (N = D) then goes into R[g % 2] as well,
  // and dP^T(g+1) into R[g % 2] once the drain holds dQ(g) in registers.  So
  // S^T(g+1) needs only dP^T(g) consumed, and is issued before dK and dQ of
  // tile g.
  static constexpr uint32_t TM_DK = 0, TM_DV = D, TM_R0 = 2 * D, TM_R1 = 2 * D + 128;
  __host__ __device__ static constexpr uint32_t tm_region(uint32_t g) { return (g & 1u) ? TM_R1 : TM_R0; }
  // At D = 64 K_j and V_j also live in TMEM (32 columns of 16-bit pairs each),
  // copied there once per K/V tile, so S^T and dP^T read only Q / dO from
  // shared memory (at D = 128 the columns are all taken).
  static constexpr bool KV_TMEM = (D == 64);
  static constexpr uint32_t TM_K = 2 * D + 256, TM_V = TM_K + D / 2;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int NTHREADS = 512;
  // Registers per thread at launch (65,536 / NTHREADS); the D = 128 register
  // split between warpgroups assumes exactly this many.
  static constexpr int NTHREADS_REGS = 65536 / NTHREADS;
  // Register budgets per thread (setmaxnreg) of the compute warpgroups (two),
  // the dQ drain warpgroup and the producer / MMA warpgroup; multiples of 8
  // that sum, over four 128-thread warpgroups, to the launch allocation.
  static constexpr uint32_t REGS_COMPUTE = 136, REGS_DRAIN = 160, REGS_OTHER = 80;
  static_assert(2 * REGS_COMPUTE + REGS_DRAIN + REGS_OTHER == 4 * NTHREADS_REGS,
                "register budgets must sum to the launch allocation");
  // The column plan and the shared-memory plan fit the hardware.
  static_assert(TM_R0 >= TM_DV + D && TM_R1 >= TM_R0 + 128 && TM_R1 + 128 <= TMEM_COLS,
                "TMEM regions overlap or overflow");
  static_assert(!KV_TMEM || (TM_K >= TM_R1 + 128 && TM_V + D / 2 <= TMEM_COLS),
                "TMEM copies of K / V overlap or overflow");
  static_assert(SMEM_ALLOC <= 232448, "shared memory beyond the 227 KB per-block limit");
};

struct BwdItem {
  int b, hkv, j;
  int i0;      // first Q tile visited
  int ntiles;  // (query heads of the group) x (Q tiles visited)
};

__device__ __forceinline__ BwdItem bwd_decode(int item, const BwdParams& p) {
  BwdItem it;
  it.j = item % p.n_kv;
  const int bh = item / p.n_kv;
  it.b = bh / p.Hkv;
  it.hkv = bh - it.b * p.Hkv;
  // causal: the first Q tile holding a query that sees key j*128
  it.i0 = p.causal ? max(0, it.j * 128 - p.past) / 128 : 0;
  it.ntiles = (p.H / p.Hkv) * (p.n_q - it.i0);
  return it;
}

// K/V tile s of work unit u of the persistent CTAs.  Under causal masking a
// unit is the pair of K/V tiles j and n_kv-1-j of one (batch, K/V head), the
// longer first: tile j visits n_q - j Q tiles (Lq = Lk), so every pair carries
// the same work (a plain round-robin over single tiles left CTAs with fixed
// positions j and 50% more work than others).  Without masking every tile is
// the same work and a unit is one tile (finer units shorten the last round).
// Units of one head are consecutive, so the CTAs running at the same time
// share a few heads' Q / dO in L2.  Returns false for the missing second tile
// of the middle pair when n_kv is odd.
// A causal problem of only a few rounds (snake = 1) balances better with
// single tiles instead: sorted by decreasing work (tile j before j+1, all
// heads), round r of the CTAs takes the next gridDim.x of them, CTA c the c-th
// in even rounds and the (gridDim.x-1-c)-th in odd ones.  The CTAs' loops
// then run over rounds x gridDim.x units; positions past the tiles are empty.
__device__ __forceinline__ bool bwd_unit_item(int u, int s, const BwdParams& p, int& item) {
  if (p.snake) {
    const int G = static_cast<int>(gridDim.x);
    const int r = u / G, c = u - r * G;
    const int k = r * G + ((r & 1) ? G - 1 - c : c);
    if (k >= p.n_items) return false;
    const int nbh = p.n_items / p.n_kv;
    const int j = k / nbh;
    item = (k - j * nbh) * p.n_kv + j;
    return true;
  }
  if (p.ipu == 1) {
    item = u;
    return true;
  }
  const int per = (p.n_kv + 1) / 2;
  const int bh = u / per, jp = u - bh * per;
  const int j = s ? p.n_kv - 1 - jp : jp;
  if (s && j == jp) return false;
  item = bh * p.n_kv + j;
  return true;
}

// n-th (head, Q tile) pair of an item: heads of the group outer, tiles inner.
__device__ __forceinline__ void bwd_tile(const BwdItem& it, const BwdParams& p, int n, int& h,
                                         int& i) {
  const int per = p.n_q - it.i0;
  const int g = n / per;
  // The CTA of K/V tile j starts at the j-th of its Q tiles and wraps around,
  // so the CTAs working on one head at the same time read different Q / dO
  // tiles and add into different dQ accumulator tiles.
  i = it.i0 + (n - g * per + it.j) % per;
  h = it.hkv * (p.H / p.Hkv) + g;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(512, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const BwdParams p) {
  using Ly = BwdLayout<D>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr uint32_t IDESC_S = idesc_f16(BF16, 128, 128, false, false);  // S^T, dP^T
  constexpr uint32_t IDESC_KN = idesc_f16(BF16, 128, D, false, true);    // dV, dK (A in TMEM)
  constexpr uint32_t IDESC_MN = idesc_f16(BF16, 128, D, true, true);     // dQ

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  auto bar = [&](int i) -> uint32_t { return base + Ly::BAR_OFF + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + Ly::MISC_OFF);
  AbortState* ab = reinterpret_cast<AbortState*>(smem_raw + Ly::MISC_OFF + 8);
  float* stats = reinterpret_cast<float*>(smem_raw + Ly::STAT_OFF);
  unsigned int* err = device_error_word();
  const uint32_t warp = warp_id(), lane = lane_id();

  // The swizzled operand tiles need a 1024-byte aligned shared window.
  if (base & 1023u) {
    if (threadIdx.x == 0) atomicCAS(err, 0u, 499u);
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < Ly::KVS; ++s) {
      mbar_init(bar(Ly::B_KVFULL + s), 1);
      mbar_init(bar(Ly::B_KVEMPTY + s), 1);
    }
    for (int s = 0; s < Ly::STAGES; ++s) {
      mbar_init(bar(Ly::B_QFULL + s), 1);
      mbar_init(bar(Ly::B_QEMPTY + s), 1);
      mbar_init(bar(Ly::B_DOFULL + s), 1);
      mbar_init(bar(Ly::B_DOEMPTY + s), 1);
    }
    mbar_init(bar(Ly::B_SFULL), 1);
    mbar_init(bar(Ly::B_DPFULL), 1);
    for (int c = 0; c < 2; ++c) {  // one arrival per compute warp
      mbar_init(bar(Ly::B_PFULL + c), 8);
      mbar_init(bar(Ly::B_DSFULL + c), 8);
    }
    mbar_init(bar(Ly::B_DQFULL), 1);
    mbar_init(bar(Ly::B_DQEMPTY), 4);  // one arrival per drain warp
    mbar_init(bar(Ly::B_DKVFULL), 1);
    mbar_init(bar(Ly::B_DONE), 1);
    ab->flag = 0;
    fence_barrier_init();
  }
  if (warp == 12 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
  }
  if (warp == 13) {
    tmem_alloc(base + Ly::MISC_OFF, Ly::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Persistent CTAs: work units (one or two K/V tiles, bwd_unit_item)
  // blockIdx.x, blockIdx.x + gridDim.x, ...  Every
  // per-tile barrier phase runs on the CTA's tile counter g, so one item's
  // last tiles (dQ drain, dK/dV epilogue) overlap the next item's first ones;
  // K_j / V_j of the next item load once the last MMA reading the current ones
  // completes (K/V-empty barrier).
  const int G = static_cast<int>(gridDim.x);
  // Registers per thread are re-balanced between the warpgroups: the compute
  // warpgroups (warps 0-7) hold both query halves' fp32 P^T between the
  // exponent and dS phases, the drain warpgroup (warps 8-11) a whole dQ row,
  // the producer / MMA warpgroup (12-15) needs few.  The four budgets sum to
  // the launch total of 512 x 128 (Ly::REGS_*).  Each role sets its budget
  // first thing in its own branch, so the compiler allocates that branch to it.
  constexpr bool kSplitRegs = true;

  if (warp == 12) {
    if constexpr (kSplitRegs) setmaxnreg_dec<Ly::REGS_OTHER>();
    // ------------------------------------------------------------ producer (whole warp)
    bool ok = true;
    uint32_t issued[Ly::STAGES] = {0, 0}, issued_do[Ly::STAGES] = {0, 0};
    uint32_t stage = 0, phase = 0, kv_cnt = 0;
    for (int u = p.ipu * static_cast<int>(blockIdx.x); ok && u < p.ipu * p.n_units;
         u += (u % p.ipu == p.ipu - 1) ? p.ipu * (G - 1) + 1 : 1) {
    int item;
    if (!bwd_unit_item(u / p.ipu, u % p.ipu, p, item)) continue;
    const BwdItem it = bwd_decode(item, p);
    const int kvs = static_cast<int>(kv_cnt % Ly::KVS);
    const uint32_t kv_round = kv_cnt / Ly::KVS;
    if (kv_round > 0 &&
        !mbar_wait_warp(bar(Ly::B_KVEMPTY + kvs), (kv_round - 1) & 1, ab, err, 402)) {
      ok = false;
      break;
    }
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(Ly::B_KVFULL + kvs), 2 * Ly::TILE);
      for (int c = 0; c < Ly::KCH; ++c) {
        tma_load_4d(base + Ly::k_off(kvs) + c * Ly::CHUNK, &tmK, bar(Ly::B_KVFULL + kvs), c * 64, it.hkv,
                    it.j * 128, it.b);
        tma_load_4d(base + Ly::v_off(kvs) + c * Ly::CHUNK, &tmV, bar(Ly::B_KVFULL + kvs), c * 64, it.hkv,
                    it.j * 128, it.b);
      }
    }
    ++kv_cnt;
    for (int n = 0; n < it.ntiles; ++n) {
      int h, i;
      bwd_tile(it, p, n, h, i);
      // dO_i first: its slot frees after the previous occupant's last dV,
      // before Q's (its last dK).
      if (!mbar_wait_warp(bar(Ly::B_DOEMPTY + stage), phase ^ 1u, ab, err, 403)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(Ly::B_DOFULL + stage), Ly::TILE);
        for (int c = 0; c < Ly::KCH; ++c)
          tma_load_4d(base + Ly::DO_OFF + stage * Ly::TILE + c * Ly::CHUNK, &tmdO,
                      bar(Ly::B_DOFULL + stage), c * 64, h, i * 128, it.b);
      }
      ++issued_do[stage];
      if (!mbar_wait_warp(bar(Ly::B_QEMPTY + stage), phase ^ 1u, ab, err, 401)) { ok = false; break; }
      // -LSE (pre-multiplied by log2 e) and -Delta of the 128 query rows of tile i.
      float* st = stats + stage * 256;
      const size_t row0 = (static_cast<size_t>(it.b) * p.H + h) * p.Lq;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = lane + 32 * u;
        const int q = i * 128 + c;
        const bool in = q < p.Lq;
        st[c] = in ? -p.LSE[row0 + q] * 1.4426950408889634f : 0.f;
        st[128 + c] = in ? -p.Delta[row0 + q] : 0.f;
      }
      __syncwarp();  // every lane's LSE / Delta entries precede the arrival
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(Ly::B_QFULL + stage), Ly::TILE);
        for (int c = 0; c < Ly::KCH; ++c)
          tma_load_4d(base + Ly::Q_OFF + stage * Ly::TILE + c * Ly::CHUNK, &tmQ,
                      bar(Ly::B_QFULL + stage), c * 64, h, i * 128, it.b);
      }
      ++issued[stage];
      if (++stage == Ly::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    }
    if (!ok && lane == 0) {
      for (uint32_t c = kv_cnt > Ly::KVS ? kv_cnt - Ly::KVS : 0; c < kv_cnt; ++c)
        mbar_wait_drain(bar(Ly::B_KVFULL + c % Ly::KVS), (c / Ly::KVS) & 1);
      for (int s = 0; s < Ly::STAGES; ++s) {
        if (issued[s] > 0) mbar_wait_drain(bar(Ly::B_QFULL + s), (issued[s] - 1) & 1);
        if (issued_do[s] > 0) mbar_wait_drain(bar(Ly::B_DOFULL + s), (issued_do[s] - 1) & 1);
      }
    }
  } else if (warp == 13) {
    if constexpr (kSplitRegs) setmaxnreg_dec<Ly::REGS_OTHER>();
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule (warp-uniform loop state and operand
    // descriptors); one elected lane issues each MMA group and the commits.
    // Per tile g (regions: Ra = R[g % 2], Rb = the other):
    //   [S^T(g) -> Ra, issued at the end of tile g-1, or here for an item's
    //   first tile]  dP^T(g) -> Rb (after the drain holds dQ(g-1))
    //   dV_A, dV_B (as each query half's P^T lands)  dK_A (its dS^T)
    //   [once dS^T_B is in: S^T(g+1) -> Rb, whose dP^T(g) is consumed]
    //   dK_B  dQ(g) = dS K -> Ra
    // so the compute warps start on tile g+1 while dK_B(g) and dQ(g) run.
    auto commit = [&](int b) {
      if (elect_one()) tc_commit(bar(b));
      __syncwarp();
    };
    bool ok = true;
    uint32_t stage = 0, phase = 0, g = 0, kv_cnt = 0;
    // Descriptors of the first K step (K-major operands) or of the first 16
    // rows (MN-major); later steps add their byte offset >> 4.
    uint64_t kd = 0, vd = 0, kd_mn = 0;  // the current K/V slot's (set per item)
    const uint64_t dsd_mn = sdesc_sw128(base + Ly::DS_OFF, Ly::CHUNK, 1024);
    auto koff = [](int k) -> uint64_t { return ((k >> 2) * Ly::CHUNK + (k & 3) * 32u) >> 4; };
    // S^T(gg) = K_j Q^T of the Q tile in ring stage st into R[gg % 2].  The
    // region's previous contents (dP^T(gg-1), dQ(gg-2)) were consumed before.
    auto issue_s = [&](uint32_t st, uint32_t gg) {
      const uint64_t qd = sdesc_sw128(base + Ly::Q_OFF + st * Ly::TILE, 16, 1024);
      const uint32_t dst = tmem + Ly::tm_region(gg);
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          if constexpr (Ly::KV_TMEM)
            mma_ts(dst, tmem + Ly::TM_K + 8 * k, qd + koff(k), IDESC_S, k > 0 ? 1u : 0u);
          else
            mma_ss(dst, kd + koff(k), qd + koff(k), IDESC_S, k > 0 ? 1u : 0u);
        tc_commit(bar(Ly::B_SFULL));
      }
      __syncwarp();
    };
    for (int u = p.ipu * static_cast<int>(blockIdx.x); ok && u < p.ipu * p.n_units;
         u += (u % p.ipu == p.ipu - 1) ? p.ipu * (G - 1) + 1 : 1) {
    int item;
    if (!bwd_unit_item(u / p.ipu, u % p.ipu, p, item)) continue;
    const BwdItem it = bwd_decode(item, p);
    const int kvs = static_cast<int>(kv_cnt % Ly::KVS);
    if (!mbar_wait_warp(bar(Ly::B_KVFULL + kvs), (kv_cnt / Ly::KVS) & 1, ab, err, 501)) {
      ok = false;
      break;
    }
    tc_fence_after();
    kd = sdesc_sw128(base + Ly::k_off(kvs), 16, 1024);
    vd = sdesc_sw128(base + Ly::v_off(kvs), 16, 1024);
    kd_mn = sdesc_sw128(base + Ly::k_off(kvs), Ly::CHUNK, 1024);
    if constexpr (Ly::KV_TMEM) {
      // K_j, V_j into TMEM, one 16-column K step per copy (after the previous
      // item's MMAs that read these columns, which were issued before).
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          tmem_cp_128x256b(tmem + Ly::TM_K + 8 * k, kd + koff(k));
          tmem_cp_128x256b(tmem + Ly::TM_V + 8 * k, vd + koff(k));
        }
      }
      __syncwarp();
    }
    // n: tile within the item (accumulate flags); g: tile of the CTA (phases, regions)
    for (int n = 0; ok && n < it.ntiles; ++n, ++g) {
      const uint32_t ra = tmem + Ly::tm_region(g), rb = tmem + Ly::tm_region(g + 1);
      if (n == 0) {  // an item's first S^T (later ones are issued a tile ahead)
        if (!mbar_wait_warp(bar(Ly::B_QFULL + stage), phase, ab, err, 502)) { ok = false; break; }
        tc_fence_after();
        issue_s(stage, g);
      }
      const uint32_t qa = base + Ly::Q_OFF + stage * Ly::TILE;
      const uint32_t doa = base + Ly::DO_OFF + stage * Ly::TILE;
      const uint64_t qd_mn = sdesc_sw128(qa, Ly::CHUNK, 1024);
      const uint64_t dod = sdesc_sw128(doa, 16, 1024), dod_mn = sdesc_sw128(doa, Ly::CHUNK, 1024);
      // dP^T = V_j dO_i^T into Rb, once the drain holds the previous dQ tile
      // (which occupied these columns) in registers.
      if (!mbar_wait_warp(bar(Ly::B_DOFULL + stage), phase, ab, err, 512)) { ok = false; break; }
      if (g > 0 && !mbar_wait_warp(bar(Ly::B_DQEMPTY), (g - 1) & 1, ab, err, 503)) { ok = false; break; }
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          if constexpr (Ly::KV_TMEM)
            mma_ts(rb, tmem + Ly::TM_V + 8 * k, dod + koff(k), IDESC_S, k > 0 ? 1u : 0u);
          else
            mma_ss(rb, vd + koff(k), dod + koff(k), IDESC_S, k > 0 ? 1u : 0u);
        tc_commit(bar(Ly::B_DPFULL));
      }
      __syncwarp();
      // dV += P^T_c dO_c as each query half's P^T lands in TMEM (A operand from TMEM).
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (!mbar_wait_warp(bar(Ly::B_PFULL + c), g & 1, ab, err, 504 + c)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + Ly::TM_DV, ra + 64 * c + (k >> 1) * 32u + (k & 1) * 8u,
                   dod_mn + ((2048u * (4 * c + k)) >> 4), IDESC_KN,
                   (n > 0 || c > 0 || k > 0) ? 1u : 0u);
          if (c == 1) tc_commit(bar(Ly::B_DOEMPTY + stage));  // dV_B was dO_i's last reader
        }
        __syncwarp();
      }
      if (!ok) break;
      // dK += dS^T_c Q_c as each half's dS^T lands.  Once the second half is
      // in, the compute warps have consumed dP^T(g): the next tile's S^T goes
      // into Rb first, then dK_B and dQ(g) follow.
      const bool more = n + 1 < it.ntiles;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (!mbar_wait_warp(bar(Ly::B_DSFULL + c), g & 1, ab, err, 508 + c)) { ok = false; break; }
        tc_fence_after();
        if (c == 1 && more) {
          const uint32_t ns = stage + 1 == Ly::STAGES ? 0 : stage + 1;
          const uint32_t nph = stage + 1 == Ly::STAGES ? phase ^ 1u : phase;
          if (!mbar_wait_warp(bar(Ly::B_QFULL + ns), nph, ab, err, 511)) { ok = false; break; }
          tc_fence_after();
          issue_s(ns, g + 1);
        }
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + Ly::TM_DK, ra + 64 * c + (k >> 1) * 32u + 16u + (k & 1) * 8u,
                   qd_mn + ((2048u * (4 * c + k)) >> 4), IDESC_KN,
                   (n > 0 || c > 0 || k > 0) ? 1u : 0u);
        }
        __syncwarp();
      }
      if (!ok) break;
      // Q_i is no longer read (dK_B was its last reader).
      commit(Ly::B_QEMPTY + stage);
      // dQ_i = dS K_j into Ra (dS read MN-major from the dS^T tile in shared
      // memory, K_j MN-major); the P^T / dS^T there are read by the MMAs above.
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss(ra, dsd_mn + ((2048u * k) >> 4), kd_mn + ((2048u * k) >> 4), IDESC_MN,
                 k > 0 ? 1u : 0u);
        tc_commit(bar(Ly::B_DQFULL));
      }
      __syncwarp();
      if (++stage == Ly::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    // dK / dV of this item are final; K_j / V_j are no longer read.
    if (elect_one()) {
      tc_commit(bar(Ly::B_DKVFULL));
      tc_commit(bar(Ly::B_KVEMPTY + kvs));
    }
    __syncwarp();
    ++kv_cnt;
    }
    commit(Ly::B_DONE);
    mbar_wait_drain(bar(Ly::B_DONE), 0);
  } else if (warp < 8) {
    if constexpr (kSplitRegs) setmaxnreg_inc<Ly::REGS_COMPUTE>();
    // ------------------------------------------------------------ P^T / dS^T
    // All eight warps work on each query half in turn: warp w owns key rows
    // 32*(w%4).. (its TMEM lanes) and the 32-query chunk sub = w/4 of the
    // half.  Per tile: P^T of half A, then of half B (from S^T alone, which
    // lands first), then dS^T of half A and of half B (once dP^T lands); the
    // fp32 P^T of both halves stays in registers in between.
    const int sub = warp >> 2;        // 32-query chunk within a half
    const int r = threadIdx.x & 127;  // key row within the tile == TMEM lane
    const uint32_t lane_off = ((warp & 3u) * 32u) << 16;
    const float sl2 = p.sl2;
    bool ok = true;
    uint32_t stage = 0, g = 0, kv_cnt = 0;
    for (int u = p.ipu * static_cast<int>(blockIdx.x); ok && u < p.ipu * p.n_units;
         u += (u % p.ipu == p.ipu - 1) ? p.ipu * (G - 1) + 1 : 1) {
    int item;
    if (!bwd_unit_item(u / p.ipu, u % p.ipu, p, item)) continue;
    const BwdItem it = bwd_decode(item, p);
    const int kr = it.j * 128 + r;
    for (int n = 0; ok && n < it.ntiles; ++n, ++g) {
      int h, i;
      bwd_tile(it, p, n, h, i);
      // S^T(g) and then P^T / dS^T in region R[g % 2]; dP^T(g) in the other.
      const uint32_t tSr = tmem + lane_off + Ly::tm_region(g);
      const uint32_t tPr = tmem + lane_off + Ly::tm_region(g + 1);
      if (!mbar_wait_warp(bar(Ly::B_SFULL), g & 1, ab, err, 601)) { ok = false; break; }
      tc_fence_after();
      uint32_t pf[2][32];  // P^T of each half in fp32, for dS^T
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        const int cbase = 64 * hc + 32 * sub;  // first query column of this chunk
        const uint32_t tS = tSr + cbase;
        const float* st = stats + stage * 256 + cbase;
        const int q0 = i * 128 + cbase;
        // query columns [lo, hi) of this chunk are visible to key kr
        int lo = 0, hi = min(32, p.Lq - q0);
        if (kr >= p.Lk) hi = 0;
        if (p.causal) lo = max(0, kr - p.past - q0);
        const bool full = (lo == 0 && hi == 32);
        // P^T = exp2(S^T*c - LSE*log2e), from S^T alone.
        uint32_t* sv = pf[hc];
        tmem_ld32(tS, sv);
        tmem_ld_wait32(sv);
        uint32_t pk[16];
        const uint4* nl4 = reinterpret_cast<const uint4*>(st);  // -LSE*log2e
        // Off-diagonal, in-range tiles (the common case) take a copy of the
        // loop without the per-element mask.
        auto exp_loop = [&](auto masked) {
#pragma unroll
          for (int u4 = 0; u4 < 8; ++u4) {
            const uint4 l4 = nl4[u4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int cl = 4 * u4 + 2 * e;
              // (scalar FMAs: measured slightly faster here than the paired form)
              const float p0_arg = fmaf(__uint_as_float(sv[cl]), sl2, __uint_as_float(e ? l4.z : l4.x));
              const float p1_arg = fmaf(__uint_as_float(sv[cl + 1]), sl2, __uint_as_float(e ? l4.w : l4.y));
              float p0 = ex2(p0_arg), p1 = ex2(p1_arg);
              if constexpr (decltype(masked)::value) {
                p0 = (cl >= lo && cl < hi) ? p0 : 0.f;
                p1 = (cl + 1 >= lo && cl + 1 < hi) ? p1 : 0.f;
              }
              sv[cl] = __float_as_uint(p0);  // P^T in fp32 for dS^T
              sv[cl + 1] = __float_as_uint(p1);
              pk[cl >> 1] = pack2<T>(p0, p1);
            }
          }
        };
        if (full)
          exp_loop(std::false_type{});
        else
          exp_loop(std::true_type{});
        // P^T (16-bit pairs) over the first 16 of this chunk's S^T columns.
        tmem_st16(tS, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Ly::B_PFULL + hc));
      }
      if (!mbar_wait_warp(bar(Ly::B_DPFULL), g & 1, ab, err, 602)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        // dS^T = P^T o (dP^T - Delta).
        const int cbase = 64 * hc + 32 * sub;
        const uint32_t tS = tSr + cbase;
        const float* st = stats + stage * 256 + cbase;
        const uint32_t* sv = pf[hc];
        uint32_t dp[32];
        tmem_ld32(tPr + cbase, dp);
        tmem_ld_wait32(dp);
        uint32_t dk[16];
        const uint4* nd4 = reinterpret_cast<const uint4*>(st + 128);  // -Delta
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4) {
          const uint4 d4 = nd4[u4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cl = 4 * u4 + 2 * e;
            const uint64_t nd = e ? f2_pack(__uint_as_float(d4.z), __uint_as_float(d4.w))
                                  : f2_pack(__uint_as_float(d4.x), __uint_as_float(d4.y));
            float d0, d1;
            f2_unpack(fmul2(f2_pack(__uint_as_float(sv[cl]), __uint_as_float(sv[cl + 1])),
                            fadd2(f2_pack(__uint_as_float(dp[cl]), __uint_as_float(dp[cl + 1])), nd)),
                      d0, d1);
            dk[cl >> 1] = pack2<T>(d0, d1);
          }
        }
        // dS^T over the next 16 columns, and row r of the swizzled dS^T tile
        // (queries cbase .. cbase+31: four 16-byte units).
        tmem_st16(tS + 16, dk);
        uint8_t* ds_row = smem_raw + Ly::DS_OFF + hc * Ly::CHUNK + r * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int pos = (sub * 4 + v) ^ (r & 7);
          *reinterpret_cast<uint4*>(ds_row + pos * 16) =
              make_uint4(dk[4 * v], dk[4 * v + 1], dk[4 * v + 2], dk[4 * v + 3]);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Ly::B_DSFULL + hc));
      }
      if (++stage == Ly::STAGES) stage = 0;
    }
    const int hc = sub;  // epilogue role: warps 0-3 write dK, warps 4-7 write dV
    // Epilogue: warpgroup A writes dK (scaled by 1/sqrt(D)), B writes dV.
    if (!ok) break;
    if (!mbar_wait_warp(bar(Ly::B_DKVFULL), kv_cnt & 1, ab, err, 603)) { ok = false; break; }
    {
      tc_fence_after();
      void* dst_base = hc == 0 ? p.dK : p.dV;
      const float sc = hc == 0 ? p.scale : 1.f;
      const uint32_t tsrc = tmem + lane_off + (hc == 0 ? Ly::TM_DK : Ly::TM_DV);
      T* row = reinterpret_cast<T*>(dst_base) +
               ((static_cast<size_t>(it.b) * p.Lk + kr) * p.Hkv + it.hkv) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tsrc + 32 * cc, o);
        tmem_ld_wait32(o);
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack2<T>(__uint_as_float(o[2 * u]) * sc, __uint_as_float(o[2 * u + 1]) * sc);
        if (kr < p.Lk) {
          uint4* dst = reinterpret_cast<uint4*>(row + 32 * cc);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
    }
    ++kv_cnt;
    }
  } else if (warp < 12) {
    if constexpr (kSplitRegs) setmaxnreg_inc<Ly::REGS_DRAIN>();
    // ------------------------------------------------------------ dQ drain
    const int r = threadIdx.x & 127;  // query row within the Q tile == TMEM lane
    const uint32_t lane_off = ((warp & 3u) * 32u) << 16;
    bool ok = true;
    uint32_t g = 0;
    for (int u = p.ipu * static_cast<int>(blockIdx.x); ok && u < p.ipu * p.n_units;
         u += (u % p.ipu == p.ipu - 1) ? p.ipu * (G - 1) + 1 : 1) {
    int item;
    if (!bwd_unit_item(u / p.ipu, u % p.ipu, p, item)) continue;
    const BwdItem it = bwd_decode(item, p);
    for (int n = 0; n < it.ntiles; ++n, ++g) {
      int h, i;
      bwd_tile(it, p, n, h, i);
      if (!mbar_wait_warp(bar(Ly::B_DQFULL), g & 1, ab, err, 701)) { ok = false; break; }
      tc_fence_after();
      const int q = i * 128 + r;
      // accumulator layout [B, H, D/4, Lpad, 4]: a warp's 32 rows of one
      // 4-column group are 512 contiguous bytes.
      float4* acc = reinterpret_cast<float4*>(p.dq_accum) +
                    (static_cast<size_t>(it.b) * p.H + h) * (D / 4) * p.Lpad + q;
      // The whole dQ row (D fp32) in registers, then its columns go back to
      // the MMA warp before any reduction is issued.
      uint32_t gq[D];
      const uint32_t tq = tmem + lane_off + Ly::tm_region(g);  // dQ(g) lies in R[g % 2]
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tq + 32 * cc, gq + 32 * cc);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld_wait32(gq + 32 * cc);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::B_DQEMPTY));
      if (q < p.Lq) {
#pragma unroll
        for (int c4 = 0; c4 < D / 4; ++c4) {
          // Paced: issued back to back, a tile's reductions hold the SM's
          // memory-instruction path for ~1,000 cycles and slow the MMAs that
          // read shared memory meanwhile.  Measured at B8 H32 L4096 D128 fp16
          // (a tile every ~2.5 us, 2070 MHz): no pause 5.3-5.6 ms; a pause
          // after every second reduction (15 pauses) requested as 64 ns or
          // 100 ns 4.46 ms, as 128 ns 7.31 ms (the pauses then outlast the
          // tile and the drain holds up the next dP^T); 50 ns after each
          // 4.52; 200 ns after every eighth 5.60.  (__nanosleep's duration
          // is only approximately its argument.)
          if ((D == 128 || FA_BWD_PACE_D64) && FA_BWD_PACE_NS > 0 &&
              (c4 % FA_BWD_PACE_EVERY) == FA_BWD_PACE_EVERY - 1 && c4 < D / 4 - 1)
            __nanosleep(FA_BWD_PACE_NS);
          red_add_v4(reinterpret_cast<float*>(acc + static_cast<size_t>(c4) * p.Lpad),
                     __uint_as_float(gq[4 * c4]), __uint_as_float(gq[4 * c4 + 1]),
                     __uint_as_float(gq[4 * c4 + 2]), __uint_as_float(gq[4 * c4 + 3]));
        }
      }
    }
    }
  } else {
    // warps 14-15: idle, but they belong to the producer / MMA warpgroup
    if constexpr (kSplitRegs) setmaxnreg_dec<Ly::REGS_OTHER>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Ly::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- preprocess
// One CTA per (batch, 32-row chunk of the padded sequence, group of HG
// heads).  Reads the chunk's O and dO rows of its heads (32 blocks of
// HG*D contiguous elements), reduces each row in fp32, and writes Delta for
// each head as 32 contiguous floats.  When an accumulator is given it also
// zeroes that part of it.  HG is chosen by the launcher so that small
// batches still give every SM work.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
    fa_bwd_prep_kernel(const void* __restrict__ O, const void* __restrict__ dO,
                       float* __restrict__ Delta, float* __restrict__ dq_accum, int B, int L, int H,
                       int Lpad, int HG) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int TPR = D / 8;  // threads per row (16 bytes each)
  extern __shared__ float dsm[];  // [HG][32]
  const int chunks = Lpad / 32;
  const int groups = (H + HG - 1) / HG;
  const int hg = blockIdx.x % groups;
  const int bc = blockIdx.x / groups;
  const int b = bc / chunks;
  const int l0 = (bc - b * chunks) * 32;
  const int h0 = hg * HG;
  const int nh = min(HG, H - h0);                // heads of this group
  const int nrow = max(0, min(32, L - l0)) * nh;  // rows (l, h) with l < L
  const int sub = threadIdx.x % TPR;
  for (int row = threadIdx.x / TPR; row < ((nrow + (256 / TPR) - 1) / (256 / TPR)) * (256 / TPR);
       row += 256 / TPR) {
    float acc = 0.f;
    const int l = row / nh, hh = row - l * nh;
    if (row < nrow) {
      const size_t off = ((static_cast<size_t>(b) * L + l0 + l) * H + h0 + hh) * TPR + sub;
      const uint4 a = reinterpret_cast<const uint4*>(O)[off];
      const uint4 c = reinterpret_cast<const uint4*>(dO)[off];
      const T* ea = reinterpret_cast<const T*>(&a);
      const T* ec = reinterpret_cast<const T*>(&c);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(static_cast<float>(ea[e]), static_cast<float>(ec[e]), acc);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0 && row < nrow) dsm[hh * 32 + l] = acc;
  }
  __syncthreads();
  const int nl = max(0, min(32, L - l0));
  for (int idx = threadIdx.x; idx < nh * 32; idx += 256) {
    const int hh = idx / 32, l = idx - hh * 32;
    if (l < nl) Delta[(static_cast<size_t>(b) * H + h0 + hh) * L + l0 + l] = dsm[idx];
  }
  if (dq_accum) {
    // [B, H, D/4, Lpad, 4]: for each (h, column group) the chunk is 32 float4.
    float4* acc = reinterpret_cast<float4*>(dq_accum);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int idx = threadIdx.x; idx < nh * (D / 4) * 32; idx += 256) {
      const int seg = idx / 32, l = idx - seg * 32;  // seg = hh * (D/4) + c4
      const int hh = seg / (D / 4), c4 = seg - hh * (D / 4);
      acc[((static_cast<size_t>(b) * H + h0 + hh) * (D / 4) + c4) * Lpad + l0 + l] = z;
    }
  }
}

// ---------------------------------------------------------------- dQ post-process
// One CTA per (batch, head, chunk of CR rows): every thread first loads its
// share of the accumulator chunk (column groups of CR contiguous float4, read
// once, streaming), then the chunk is transposed through shared memory with
// 16-byte accesses, scaled by 1/sqrt(D) and written as BSHD rows.
constexpr int kConvRows = 64;                 // accumulator rows per CTA
constexpr int kConvThreads = 4 * kConvRows;
template <int D>
constexpr size_t conv_smem_bytes() { return static_cast<size_t>(kConvRows) * (D + 4) * sizeof(float); }

template <int D, bool BF16>
__global__ void __launch_bounds__(kConvThreads)
    fa_dq_convert_kernel(const float* __restrict__ dq_accum, void* __restrict__ dQ, int B, int L,
                         int H, int Lpad, float scale) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int CR = kConvRows, NT = kConvThreads;
  constexpr int RS = D + 4;                 // row stride in floats (16-byte aligned, skewed banks)
  constexpr int PER = (D / 4) * CR / NT;    // float4 loads per thread
  extern __shared__ __align__(16) float tile[];  // [CR][RS]
  const int chunks = Lpad / CR;
  const int bh = blockIdx.x / chunks;
  const int l0 = (blockIdx.x - bh * chunks) * CR;
  const int b = bh / H, h = bh - b * H;
  const float4* src = reinterpret_cast<const float4*>(dq_accum) + static_cast<size_t>(bh) * (D / 4) * Lpad + l0;
  float4 v[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int idx = threadIdx.x + NT * k;
    const int c4 = idx / CR, l = idx - c4 * CR;
    v[k] = __ldcs(src + static_cast<size_t>(c4) * Lpad + l);
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int idx = threadIdx.x + NT * k;
    const int c4 = idx / CR, l = idx - c4 * CR;
    *reinterpret_cast<float4*>(tile + l * RS + 4 * c4) = v[k];
  }
  __syncthreads();
  constexpr int UPR = D / 8;  // 16-byte output units per row
#pragma unroll
  for (int k = 0; k < CR * UPR / NT; ++k) {
    const int idx = threadIdx.x + NT * k;
    const int l = idx / UPR, u = idx - l * UPR;
    if (l0 + l >= L) continue;
    const float4 a = *reinterpret_cast<const float4*>(tile + l * RS + 8 * u);
    const float4 c = *reinterpret_cast<const float4*>(tile + l * RS + 8 * u + 4);
    uint4 o;
    o.x = pack2<T>(a.x * scale, a.y * scale);
    o.y = pack2<T>(a.z * scale, a.w * scale);
    o.z = pack2<T>(c.x * scale, c.y * scale);
    o.w = pack2<T>(c.z * scale, c.w * scale);
    T* row = reinterpret_cast<T*>(dQ) + ((static_cast<size_t>(b) * L + l0 + l) * H + h) * D;
    __stcs(reinterpret_cast<uint4*>(row) + u, o);
  }
}

}  // namespace fa
