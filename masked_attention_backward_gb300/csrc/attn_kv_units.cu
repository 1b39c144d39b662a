// attn_kv_units.cu -- persistent form of the key-stationary dK/dV kernel, for
// walks of a few steps (short sliding windows, block masks).
//
// The work, the TMEM layout and the per-step protocol are those of k_dkdv
// (attn_kv.cu): a unit is (b, kv head c, KV_TILE key rows), walked over
// (query head of the group, KV_SUB-row query sub-tile) steps with
//   S^T = K Q^T, dP^T = V dO^T, P^T, dS^T, dV += P^T dO, dK += dS^T Q
// and two step buffers of S^T / dP^T in TMEM.  What changes is what happens
// between units.  When a unit has only a handful of steps (a 128-key window
// gives 16, a bigbird key tile about 14), a CTA per unit spends about a third
// of its time starting, waiting for its first K / V tile and its first step,
// and storing dK / dV while nothing else runs on the SM.  Here one CTA per SM
// runs unit after unit:
//   - the producer claims the next unit from a global counter, publishes it in
//     a ring of unit slots that every other warp reads in order, brings the
//     next K / V tile into L2, and loads it as soon as the current unit's last
//     S^T / dP^T MMAs have completed; the Q / dO ring, the step buffers and
//     their barrier phases run on across units (one step counter);
//   - four epilogue warps (one per TMEM lane quarter) read a finished unit's
//     dV, then dK accumulator out of TMEM and store the rows while the other
//     warps run the next unit; the next unit's first dV (dK) MMA, which starts
//     its accumulator from zero, waits only for that read-out.
// One warp issues both accumulations (dV, then dK of each step, in the order
// the softmax warps produce their operands), so that the CTA keeps 24 warps
// and 80 registers per thread.
//
// Sources: as k_dkdv -- tilelang-ascend PR #1 "Add GQA Sink Backward BHSD",
// commit notes (five contractions + softmax + dS per step, the GQA group per
// kv head); cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook,
// optimisation 2 (key-major select table) and 3 (contiguous dK/dV write-back).
//
// Warp roles (768 threads): warp 0 loads; warp 1 issues S^T (and owns TMEM),
// warp 2 dP^T, warp 3 dV and dK; warps 4..19 are the softmax warps (warp
// (sp, g), sp = warp % 4, owns TMEM lanes 32 sp .. 32 sp + 31 and query
// columns 16 g .. 16 g + 15); warps 20..23 are the epilogue warps.
#include "kv_softmax.cuh"

namespace mab {

namespace kvu_side {

constexpr int STAGES = 4;      // Q/dO ring depth
constexpr int COL_DV = 0;
constexpr int COL_DK = 128;
constexpr int COL_BUF = 256;   // buffer b at COL_BUF + 128 b: S^T at +0, dP^T at +64
constexpr int MMA_WARPS = 3;   // warps 1..3
constexpr int SM_WARPS = 16;   // softmax warps
constexpr int SM_WARP0 = 1 + MMA_WARPS;
constexpr int EP_WARPS = 4;    // epilogue warps
constexpr int EP_WARP0 = SM_WARP0 + SM_WARPS;
constexpr int NUM_THREADS = 32 * (EP_WARP0 + EP_WARPS);
constexpr int USLOTS = 4;      // published units in flight
constexpr unsigned int EP_SLEEP_NS = 256;  // polling period of the epilogue warps' waits

struct __align__(1024) Smem {
  uint8_t K[2 * KV_TILE * 128];
  uint8_t V[2 * KV_TILE * 128];
  uint8_t Q[STAGES][2 * KV_SUB * 128];
  uint8_t dO[STAGES][2 * KV_SUB * 128];
  uint8_t ep_stage[EP_WARPS][4096];  // row staging, 4 KB per epilogue warp
  float nlse2[STAGES][KV_SUB];   // -lse log2(e) of the stage's query rows
  float delta[STAGES][KV_SUB];
  int step_r[STAGES];            // query sub-tile of the step in the stage
  int step_hh[STAGES];           // its query head within the group
  uint32_t step_vis[STAGES];     // aligned block masks: bit 4 sp + g = region (sp, g) visible
  int unit[USLOTS];              // published units (-1: none left)
  uint64_t bar_unit_full[USLOTS];
  uint64_t bar_unit_empty[USLOTS];  // every consumer warp took the unit
  uint64_t bar_kv_full;          // K, V of a unit landed (once per unit with steps)
  uint64_t bar_k_free;           // every S^T MMA of the unit complete
  uint64_t bar_v_free;           // every dP^T MMA of the unit complete
  uint64_t bar_q_full[STAGES];
  uint64_t bar_q_empty[STAGES];  // dV and dK of the step complete
  uint64_t bar_s_full[2];
  uint64_t bar_dp_full[2];
  uint64_t bar_p_full[2];        // P^T written over the buffer's S^T (every softmax warp)
  uint64_t bar_ds_full[2];       // dS^T written over the buffer's dP^T (every softmax warp)
  uint64_t bar_s_free[2];        // dV that read the buffer's P^T complete
  uint64_t bar_dp_free[2];       // dK that read the buffer's dS^T complete
  uint64_t bar_acc_full;         // every dV and dK MMA of the unit complete
  uint64_t bar_acc_empty_v;      // dV accumulator read out (every epilogue warp)
  uint64_t bar_acc_empty_k;      // dK accumulator read out (every epilogue warp)
  uint64_t bar_x_done[MMA_WARPS];  // every MMA of issuing warp 1 + i complete (exit)
  uint32_t tmem_base;
  int abort_flag;
  int is_last;                   // this CTA finished last: it sums dSink
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;
static_assert(SMEM_BYTES <= 232448, "over the 227 KB of shared memory a CTA may use");

enum { TAG_KV = 0x701, TAG_Q_EMPTY, TAG_Q_FULL, TAG_S_FREE, TAG_P_FULL, TAG_S_FULL, TAG_DP_FULL,
       TAG_DS_FULL, TAG_ACC, TAG_X_DONE, TAG_DP_FREE, TAG_UNIT_FULL, TAG_UNIT_EMPTY, TAG_KV_FREE,
       TAG_ACC_EMPTY };

// A unit: key tile t of kv head (b, c) and its walk, numbered low key tiles
// (the longest causal walks) first, as the per-tile kernel's grid.
struct KvUnit {
  int t, bc, b, c, k0, Lq, Lk, N;
  KVWalk walk;
  __device__ __forceinline__ void init(const AttnParams& p, int u) {
    const int BHkv = p.B * p.Hkv;
    t = u / BHkv;
    bc = u % BHkv;
    b = bc / p.Hkv;
    c = bc % p.Hkv;
    k0 = t * KV_TILE;
    Lq = len_q(p, b);
    Lk = len_k(p, b);
    walk.init(p, b, c, t, Lq, Lk);
    N = walk.total(p);
  }
};

// Zero P^T (or dS^T) of a softmax warp's 16 columns at TMEM address `taddr`
// (and, compensated, a zero remainder over the next 8), then waits for the
// store: the packed values of a region none of whose logits is visible.
template <bool HILO>
__device__ __forceinline__ void kv_write_zero(uint32_t taddr) {
  const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  tmem_st8(taddr, z);
  if constexpr (HILO) tmem_st8(taddr + 8, z);
  tmem_wait_st();
}

}  // namespace kvu_side

// BHSD layout only (the packed layout keeps the per-tile kernel).
// HILO: P^T and dS^T enter dV and dK as high part + remainder (compensated).
// MK: the mask kind (MK_NONE, MK_CAUSAL, MK_SLIDING or MK_BLOCK).
template <bool BF16, bool HILO, int MK>
__global__ void __launch_bounds__(kvu_side::NUM_THREADS, 1)
k_dkdv_units(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tdO,
             const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV,
             uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, const AttnParams p) {
  using namespace kvu_side;
  constexpr int NST = STAGES;
  constexpr bool BLOCK = MK == MK_BLOCK;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int U = p.nKT_k * p.B * p.Hkv;
  const bool blk_regions = BLOCK && (p.by & 31) == 0 && (p.bx & 15) == 0;
  WaitCtx wc{p.status, &s.abort_flag, p.timeout_ns};

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    for (int i = 0; i < USLOTS; ++i) {
      mbar_init(smem_u32(&s.bar_unit_full[i]), 1);
      mbar_init(smem_u32(&s.bar_unit_empty[i]), MMA_WARPS + SM_WARPS + EP_WARPS);
    }
    mbar_init(smem_u32(&s.bar_kv_full), 1);
    mbar_init(smem_u32(&s.bar_k_free), 1);
    mbar_init(smem_u32(&s.bar_v_free), 1);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.bar_q_full[i]), 1);
      mbar_init(smem_u32(&s.bar_q_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_dp_full[i]), 1);
      mbar_init(smem_u32(&s.bar_p_full[i]), SM_WARPS);
      mbar_init(smem_u32(&s.bar_ds_full[i]), SM_WARPS);
      mbar_init(smem_u32(&s.bar_s_free[i]), 1);
      mbar_init(smem_u32(&s.bar_dp_free[i]), 1);
    }
    mbar_init(smem_u32(&s.bar_acc_full), 1);
    mbar_init(smem_u32(&s.bar_acc_empty_v), EP_WARPS);
    mbar_init(smem_u32(&s.bar_acc_empty_k), EP_WARPS);
    for (int i = 0; i < MMA_WARPS; ++i) mbar_init(smem_u32(&s.bar_x_done[i]), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  // Launched behind the preprocess kernel with programmatic serialization:
  // wait for it (and, block masks, for the table kernel it waited for) before
  // any of their results is read; then let the dQ kernel behind this one be
  // scheduled (its CTAs take the SMs this grid's CTAs leave when no unit is
  // left).
  grid_dependency_wait();
  grid_launch_dependents();

  // Every warp but the producer takes each published unit in order: it waits
  // for the slot, reads it and frees it (one arrive per warp).
  auto take_unit = [&](int j, int* u, bool lazy) -> bool {
    const int slot = j % USLOTS;
    const uint32_t bar = smem_u32(&s.bar_unit_full[slot]);
    const bool ok = lazy ? mbar_wait_sleep(bar, (j / USLOTS) & 1, wc, TAG_UNIT_FULL, EP_SLEEP_NS)
                         : mbar_wait(bar, (j / USLOTS) & 1, wc, TAG_UNIT_FULL);
    if (!__all_sync(0xffffffffu, ok)) return false;
    *u = s.unit[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.bar_unit_empty[slot]));
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the walk; lane 0 claims units and issues the copies.
    // Every 32 steps the lanes look up the next 32 steps at once (query head,
    // sub-tile from the select table, aligned block masks' region word from
    // the transposed mask), so that no step waits for a chain of global
    // loads of its own.
    if (lane == 0) {
      tma_prefetch_desc(&tQ);
      tma_prefetch_desc(&tdO);
      tma_prefetch_desc(&tK);
      tma_prefetch_desc(&tV);
    }
    const uint32_t kvbar = smem_u32(&s.bar_kv_full);
    // lane 0 waits; the rest of the warp waits for its answer
    auto wait0 = [&](uint32_t bar, uint32_t parity, unsigned int tag) -> bool {
      bool r = true;
      if (lane == 0) r = mbar_wait(bar, parity, wc, tag);
      return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    bool ok = true;
    int gn = 0;               // steps issued, across units
    int up = 0;               // units with steps so far
    bool kv_pending = false;  // a K / V load was issued (the last one: phase up - 1)
    for (int j = 0; ok; ++j) {
      const int slot = j % USLOTS;
      if (j >= USLOTS &&
          !wait0(smem_u32(&s.bar_unit_empty[slot]), ((j / USLOTS) - 1) & 1, TAG_UNIT_EMPTY)) {
        ok = false;
        break;
      }
      int u = 0;
      if (lane == 0) {
        u = j == 0 ? (int)blockIdx.x : (int)(gridDim.x + atomicAdd(&p.status->next_unit_kv, 1u));
        if (u >= U) u = -1;
        s.unit[slot] = u;  // published by the arrive
        mbar_arrive(smem_u32(&s.bar_unit_full[slot]));
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u < 0) break;
      KvUnit un;
      un.init(p, u);
      // a key tile without any step only gets zeros: K and V are not loaded
      if (un.N == 0) continue;
      if (up >= 1) {
        // bring the tile into L2 while the current unit's last MMAs run, and
        // load it once they no longer read K and V
        if (lane == 0) {
          tma_prefetch_l2_3d(&tK, 0, un.k0, un.bc);
          tma_prefetch_l2_3d(&tK, 64, un.k0, un.bc);
          tma_prefetch_l2_3d(&tV, 0, un.k0, un.bc);
          tma_prefetch_l2_3d(&tV, 64, un.k0, un.bc);
        }
        if (!wait0(smem_u32(&s.bar_k_free), (up - 1) & 1, TAG_KV_FREE) ||
            !wait0(smem_u32(&s.bar_v_free), (up - 1) & 1, TAG_KV_FREE)) {
          ok = false;
          break;
        }
      }
      if (!p.test_no_loads) {
        if (lane == 0) {
          mbar_arrive_expect_tx(kvbar, 4 * KV_TILE * 128);
          tma_load_3d(smem_u32(s.K), &tK, 0, un.k0, un.bc, kvbar);
          tma_load_3d(smem_u32(s.K + KV_TILE * 128), &tK, 64, un.k0, un.bc, kvbar);
          tma_load_3d(smem_u32(s.V), &tV, 0, un.k0, un.bc, kvbar);
          tma_load_3d(smem_u32(s.V + KV_TILE * 128), &tV, 64, un.k0, un.bc, kvbar);
        }
        kv_pending = true;
      }
      ++up;
      for (int n0 = 0; ok && n0 < un.N; n0 += 32) {
        // lane l: step n0 + l (head-major over the group's query heads)
        int hh = 0, r = 0;
        uint32_t w = 0;
        if (n0 + lane < un.N) {
          int idx = n0 + lane;
          for (int c; hh < p.group - 1 && idx >= (c = un.walk.count(p, hh)); ++hh) idx -= c;
          r = un.walk.tile(p, hh, idx);
          if (blk_regions) {
            // the mask byte of each softmax warp's 32-key x 16-query region
            // (indices clamped into the mask, ranges applied after)
            const int bh = un.b * p.Hq + un.c * p.group + hh;
            const uint8_t* mt = p.maskT + (size_t)bh * p.nkb * p.nqb;
            uint32_t mv[16];
#pragma unroll
            for (int sp2 = 0; sp2 < 4; ++sp2) {
              const int kb = min((un.k0 + 32 * sp2) / p.by, p.nkb - 1);
#pragma unroll
              for (int g2 = 0; g2 < 4; ++g2) {
                const int qb = min((r * KV_SUB + 16 * g2) / p.bx, p.nqb - 1);
                mv[4 * sp2 + g2] = mt[(size_t)kb * p.nqb + qb];
              }
            }
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (mv[e] && un.k0 + 32 * (e >> 2) < p.Skv && r * KV_SUB + 16 * (e & 3) < p.Sq)
                w |= 1u << e;
          }
        }
        const int cnt = min(32, un.N - n0);
        for (int k = 0; k < cnt; ++k, ++gn) {
          const int st = gn % NST;
          const int rk = __shfl_sync(0xffffffffu, r, k);
          const int hk = __shfl_sync(0xffffffffu, hh, k);
          const uint32_t wk = __shfl_sync(0xffffffffu, w, k);
          if (gn >= NST &&
              !wait0(smem_u32(&s.bar_q_empty[st]), ((gn / NST) - 1) & 1, TAG_Q_EMPTY)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            s.step_r[st] = rk;  // published with the loads by the arrive below
            s.step_hh[st] = hk;
            s.step_vis[st] = wk;
            if (!p.test_no_loads) {
              const int bh = un.b * p.Hq + un.c * p.group + hk;
              const uint32_t fb = smem_u32(&s.bar_q_full[st]);
              mbar_arrive_expect_tx(fb, 4 * KV_SUB * 128 + 2 * KV_SUB * 4);
              tma_load_3d(smem_u32(s.Q[st]), &tQ, 0, rk * KV_SUB, bh, fb);
              tma_load_3d(smem_u32(s.Q[st] + KV_SUB * 128), &tQ, 64, rk * KV_SUB, bh, fb);
              tma_load_3d(smem_u32(s.dO[st]), &tdO, 0, rk * KV_SUB, bh, fb);
              tma_load_3d(smem_u32(s.dO[st] + KV_SUB * 128), &tdO, 64, rk * KV_SUB, bh, fb);
              const size_t srow = (size_t)bh * p.Sq_pad + (size_t)rk * KV_SUB;
              bulk_load(smem_u32(s.nlse2[st]), p.nlse2 + srow, KV_SUB * 4, fb);
              bulk_load(smem_u32(s.delta[st]), p.delta + srow, KV_SUB * 4, fb);
            }
          }
          __syncwarp();
        }
      }
    }
    if (!ok && !p.test_no_loads && lane == 0) {
      // the CTA gave up: let the copies still in flight land before it exits
      if (kv_pending) mbar_drain(kvbar, (up - 1) & 1, wc.timeout_ns);
      for (int k = gn > NST ? gn - NST : 0; k < gn; ++k)
        mbar_drain(smem_u32(&s.bar_q_full[k % NST]), (k / NST) & 1, wc.timeout_ns);
    }
  } else if (warp < SM_WARP0) {
    // ------------------------------------------------------------ MMA issuers (whole warps)
    constexpr uint32_t ID_S = idesc_f16(BF16, KV_TILE, KV_SUB, false, false);
    constexpr uint32_t ID_ACC = idesc_f16(BF16, KV_TILE, HEAD_DIM, false, true);
    bool ok = true;
    int gn = 0, up = 0;
    if (warp == 1 || warp == 2) {
      // warp 1: S^T(m) = K Q^T; warp 2: dP^T(m) = V dO^T, into buffer m & 1
      // (both operands K-major in shared memory); each waits for the
      // accumulation that read the buffer two steps ago
      const bool is_s = warp == 1;
      const uint64_t aKV = sdesc_sw128(smem_u32(is_s ? s.K : s.V), 16, 1024);
      for (int j = 0; ok; ++j) {
        int u;
        if (!take_unit(j, &u, false) || u < 0) break;
        KvUnit un;
        un.init(p, u);
        if (un.N == 0) continue;
        ok = mbar_wait_warp(smem_u32(&s.bar_kv_full), up & 1, wc, TAG_KV);
        for (int n = 0; ok && n < un.N; ++n, ++gn) {
          const int st = gn % NST, bf = gn & 1;
          ok = mbar_wait_warp(smem_u32(&s.bar_q_full[st]), (gn / NST) & 1, wc, TAG_Q_FULL);
          if (ok && gn >= 2)
            ok = mbar_wait_warp(smem_u32(is_s ? &s.bar_s_free[bf] : &s.bar_dp_free[bf]),
                                ((gn - 2) >> 1) & 1, wc, is_s ? TAG_S_FREE : TAG_DP_FREE);
          if (!ok) break;
          tc_fence_after();
          const uint64_t bB = sdesc_sw128(smem_u32(is_s ? s.Q[st] : s.dO[st]), 16, 1024);
          const uint32_t d = tbase + COL_BUF + 128 * bf + (is_s ? 0 : 64);
#pragma unroll
          for (int kk = 0; kk < HEAD_DIM / 16; ++kk)
            mma_ss_w(d, aKV + (uint64_t)(((kk >> 2) * (KV_TILE * 128) + (kk & 3) * 32) >> 4),
                     bB + (uint64_t)(((kk >> 2) * (KV_SUB * 128) + (kk & 3) * 32) >> 4), ID_S,
                     kk > 0 ? 1u : 0u);
          mma_commit_w(smem_u32(is_s ? &s.bar_s_full[bf] : &s.bar_dp_full[bf]));
        }
        if (!ok) break;
        // the unit's K (V) tile may be replaced once these MMAs completed
        mma_commit_w(smem_u32(is_s ? &s.bar_k_free : &s.bar_v_free));
        ++up;
      }
    } else {
      // warp 3: dV += P^T(n) dO, then dK += dS^T(n) Q (A = the packed values
      // in buffer n & 1, B read MN-major).  The first MMA of a unit into each
      // accumulator (which starts it from zero) waits until the epilogue warps
      // have read the previous unit's out.
      for (int j = 0; ok; ++j) {
        int u;
        if (!take_unit(j, &u, false) || u < 0) break;
        KvUnit un;
        un.init(p, u);
        if (un.N == 0) continue;
        for (int n = 0; ok && n < un.N; ++n, ++gn) {
          const int st = gn % NST, bf = gn & 1;
#pragma unroll 1
          for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK
            ok = mbar_wait_warp(smem_u32(which ? &s.bar_ds_full[bf] : &s.bar_p_full[bf]),
                                (gn >> 1) & 1, wc, which ? TAG_DS_FULL : TAG_P_FULL);
            if (ok && n == 0 && up >= 1)
              ok = mbar_wait_warp(smem_u32(which ? &s.bar_acc_empty_k : &s.bar_acc_empty_v),
                                  (up - 1) & 1, wc, TAG_ACC_EMPTY);
            if (!ok) break;
            tc_fence_after();
            const uint32_t acc = tbase + (which ? COL_DK : COL_DV);
            const uint32_t a = tbase + COL_BUF + 128 * bf + (which ? 64 : 0);
            const uint64_t bB =
                sdesc_sw128(smem_u32(which ? s.Q[st] : s.dO[st]), KV_SUB * 128, 1024);
#pragma unroll
            for (int kk = 0; kk < KV_SUB / 16; ++kk)
              mma_ts_w(acc, a + 16 * kk, bB + (uint64_t)((kk * 2048) >> 4), ID_ACC,
                       (n > 0 || kk > 0) ? 1u : 0u);
            if (HILO) {
#pragma unroll
              for (int kk = 0; kk < KV_SUB / 16; ++kk)
                mma_ts_w(acc, a + 16 * kk + 8, bB + (uint64_t)((kk * 2048) >> 4), ID_ACC, 1u);
            }
            // frees this half of the buffer
            mma_commit_w(smem_u32(which ? &s.bar_dp_free[bf] : &s.bar_s_free[bf]));
          }
          if (!ok) break;
          // S^T(n) and dP^T(n) completed before P^T(n) / dS^T(n) could be
          // written, so the commit also frees the Q / dO stage
          mma_commit_w(smem_u32(&s.bar_q_empty[st]));
        }
        if (!ok) break;
        mma_commit_w(smem_u32(&s.bar_acc_full));
        ++up;
      }
    }
    // this warp's MMAs must be complete before TMEM is freed (also when the
    // CTA gave up, hence a wait that ignores the abort flag)
    const uint32_t done = smem_u32(&s.bar_x_done[warp - 1]);
    mma_commit_w(done);
    mbar_drain_warp(done, 0, wc.timeout_ns);
  } else if (warp < EP_WARP0) {
    // ------------------------------------------------------------ softmax warps
    const int sp = warp & 3, g = (warp - SM_WARP0) >> 2;
    const int rloc = sp * 32 + lane;
    const uint32_t lane_base = tbase + ((uint32_t)(sp * 32) << 16);
    auto warp_arrive = [&](uint64_t* bar) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(bar));
    };
    bool ok = true;
    int gn = 0;
    for (int jj = 0; ok; ++jj) {
      int u;
      if (!take_unit(jj, &u, false) || u < 0) break;
      KvUnit un;
      un.init(p, u);
      if (un.N == 0) continue;
      const int j = un.k0 + rloc;
      // block masks: this lane's row of the transposed mask for the unit's
      // first query head (the step's head adds whole heads)
      const uint8_t* rowT =
          BLOCK ? p.maskT + ((size_t)(un.b * p.Hq + un.c * p.group) * p.nkb + min(j, p.Skv - 1) / p.by) *
                                p.nqb
                : nullptr;
      int flo, fhi;  // query sub-tiles that are entirely visible
      full_range_kv(p.mask_kind, p.window, un.Lq, un.Lk, un.k0, &flo, &fhi);
      for (int n = 0; n < un.N; ++n, ++gn) {
        const int st = gn % NST, bf = gn & 1;
        const uint32_t colS = COL_BUF + 128 * bf + 16 * g;
        // the stage's loads (and with them the step's coordinates and the
        // bulk-copied statistics) first: the visibility word is worked out
        // while S^T is still being computed
        if (!mbar_wait(smem_u32(&s.bar_q_full[st]), (gn / NST) & 1, wc, TAG_Q_FULL)) {
          ok = false;
          break;
        }
        const int r = s.step_r[st];
        const bool full = !BLOCK && r >= flo && r <= fhi;  // (block masks: never)
        uint32_t vis;
        if (full) {
          vis = 0xffffu;
        } else if (blk_regions) {
          vis = ((s.step_vis[st] >> (4 * sp + g)) & 1u) && j < un.Lk
                    ? bit_range(0, un.Lq - 1 - (r * KV_SUB + 16 * g))
                    : 0u;
        } else if constexpr (BLOCK) {
          {
            // key j against queries i0 .. i0 + 15 (the lane's mask row is
            // found once per unit; the query-block quotient by a reciprocal,
            // measured 10 % faster on bigbird than the division per step)
            const uint8_t* row = rowT + (size_t)s.step_hh[st] * p.nkb * p.nqb;
            const int i0 = r * KV_SUB + 16 * g;
            const int iend = min(i0 + 15, un.Lq - 1);
            uint32_t m = 0;
            if (j < un.Lk && iend >= i0) {
              for (int qb = div_by(i0, p.bx, p.inv_bx); qb * p.bx <= iend; ++qb)
                if (row[qb]) m |= bit_range(qb * p.bx - i0, (qb + 1) * p.bx - 1 - i0);
              m &= bit_range(0, iend - i0);
            }
            vis = m;
          }
        } else {
          vis = vis_key_row_closed<MK>(p, j, r * KV_SUB + 16 * g, un.Lq, un.Lk);
        }
        // no logit of the warp's region is visible: P^T and dS^T are zero
        // (written without loading S^T or dP^T, once the MMA that writes
        // those columns has completed)
        const bool none = !full && __all_sync(0xffffffffu, vis == 0u);
        float lv[16];
        load16_shared(&s.nlse2[st][16 * g], lv);
        if (!mbar_wait(smem_u32(&s.bar_s_full[bf]), (gn >> 1) & 1, wc, TAG_S_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float pv[16];
        if (none) {
          kv_write_zero<HILO>(lane_base + colS);
        } else {
          float sv[16];
          tmem_ld16(lane_base + colS, sv);
          tmem_wait_ld_regs(sv);
          kv_write_p<BF16, HILO>(lane_base + colS, sv, lv, full, vis, p.scale_log2, pv);
        }
        warp_arrive(&s.bar_p_full[bf]);

        float dl[16];
        load16_shared(&s.delta[st][16 * g], dl);
        if (!mbar_wait(smem_u32(&s.bar_dp_full[bf]), (gn >> 1) & 1, wc, TAG_DP_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (none) {
          kv_write_zero<HILO>(lane_base + colS + 64);
        } else {
          float dp[16];
          tmem_ld16(lane_base + colS + 64, dp);
          tmem_wait_ld_regs(dp);
          uint32_t pk[8];
          kv_write_ds<BF16, HILO>(lane_base + colS + 64, pv, dp, dl, pk);
        }
        warp_arrive(&s.bar_ds_full[bf]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    // Warp (EP_WARP0 + e) reads TMEM lanes 32 (warp % 4) .. + 31, 32 key rows
    // of the unit: all 128 columns of dV, then of dK, 64 at a time, each
    // stored through its own staging buffer with 128-byte coalesced rows.
    // Its waits poll with a sleep: on a long walk they last the whole unit.
    const int sp = warp & 3;
    const uint32_t lane_base = tbase + ((uint32_t)(sp * 32) << 16);
    uint8_t* stage = s.ep_stage[warp - EP_WARP0];
    bool ok = true;
    int up = 0;
    for (int j = 0;; ++j) {
      int u;
      if (!take_unit(j, &u, true) || u < 0) break;
      KvUnit un;
      un.init(p, u);
      const int r0 = un.k0 + sp * 32;
      const int nvalid = min(32, p.Skv - r0);
      const size_t elem = ((size_t)un.bc * p.Skv + r0) * HEAD_DIM;
      bool have = false;
      if (un.N > 0) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_sleep(smem_u32(&s.bar_acc_full), up & 1,
                                                               wc, TAG_ACC, EP_SLEEP_NS));
        have = ok;
        ++up;
      }
      tc_fence_after();
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK
        uint16_t* orow = (which ? dk : dv) + elem;
        if (!have) {
          // a key tile without steps, or a CTA that gave up: zeros
          warp_zero_rows(orow, HEAD_DIM, nvalid);
          continue;
        }
        const float sc = which ? p.scale : 1.f;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            float v[32];
            tmem_ld32(lane_base + (which ? COL_DK : COL_DV) + 64 * h + 32 * q, v);
            tmem_wait_ld_regs(v);
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
              pk[16 * q + cc] = pack2<BF16>(v[2 * cc] * sc, v[2 * cc + 1] * sc);
          }
          if (h == 1) {
            // the accumulator is read out: the next unit's first MMA into it may run
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
              mbar_arrive(smem_u32(which ? &s.bar_acc_empty_k : &s.bar_acc_empty_v));
          }
          warp_store_rows(stage, pk, orow + 64 * h, nvalid);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // dSink by the grid's last CTA (the partials come from the preprocess grid,
  // which every CTA waited for above)
  if (p.dsink) {
    if (threadIdx.x == 0) s.is_last = atomicAdd(&p.status->kv_done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (s.is_last)
      for (int h = warp; h < p.Hq; h += NUM_THREADS / 32) {
        const float v = dsink_of_head(p.dsink_part, p.dsink_nparts, h, lane);
        if (lane == 0) p.dsink[h] = v;
      }
  }
}

cudaError_t launch_dkdv_units(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                              const CUtensorMap& tdO, const CUtensorMap& tK,
                              const CUtensorMap& tV, void* dk, void* dv, cudaStream_t st) {
  using Kern = decltype(&k_dkdv_units<true, false, MK_NONE>);
#define MAB_KVU_ROW(BF, HL)                                                                     \
  {k_dkdv_units<BF, HL, MK_NONE>, k_dkdv_units<BF, HL, MK_CAUSAL>,                              \
   k_dkdv_units<BF, HL, MK_SLIDING>, k_dkdv_units<BF, HL, MK_BLOCK>}
  static const Kern table[2][2][4] = {{MAB_KVU_ROW(false, false), MAB_KVU_ROW(false, true)},
                                      {MAB_KVU_ROW(true, false), MAB_KVU_ROW(true, true)}};
#undef MAB_KVU_ROW
  const Kern kern = table[bf16 ? 1 : 0][p.compensated ? 1 : 0][p.mask_kind];
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kvu_side::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int units = p.nKT_k * p.B * p.Hkv;
  const int sms = p.num_sms > 0 ? p.num_sms : 1;
  // programmatic stream serialization behind the preprocess kernel: this
  // grid's launch and set-up overlap its tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units < sms ? units : sms));
  cfg.blockDim = dim3(kvu_side::NUM_THREADS);
  cfg.dynamicSmemBytes = kvu_side::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tQ, tdO, tK, tV, (uint16_t*)dk, (uint16_t*)dv, p);
}

}  // namespace mab
