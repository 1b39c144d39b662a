// attn_kv.cu -- key-stationary dK/dV kernel on tcgen05 / TMEM, fed by TMA.
//
// One CTA per (b, kv head c, KV_TILE key rows).  K and V of the tile are
// loaded once into shared memory.  The CTA walks every query head of the
// GQA group and, for each, every active query sub-tile r of KV_SUB rows
// (closed-form range for causal / sliding / none, the key-major select table
// for block masks):
//   S^T  = K Q_r^T            (A = K, B = Q_r from shared memory)
//   dP^T = V dO_r^T           (A = V, B = dO_r from shared memory)
//   P^T  = exp2(S^T * scale*log2e - lse_r log2e),  dS^T = P^T (dP^T - Delta_r)
//   dV  += P^T dO_r,  dK += dS^T Q_r          (A = P^T / dS^T from TMEM)
// The group reduction happens in the TMEM accumulators; the epilogue scales
// dK, rounds both to the input dtype and writes each row once, contiguously.
//
// Sources: tilelang-ascend PR #1 "Add GQA Sink Backward BHSD", commit notes
// (five contractions + softmax + dS per step; GQA group of query heads per
// key/value head); cannbot-knowledge PR #174, BlockSparseAttentionGrad
// runbook, optimisation 2 (key-major select table over the transposed mask),
// optimisation 3 (contiguous dK/dV write-back, no atomics) and the precision
// notes (p = exp(s - lse), ds = p (dp - delta)).
//
// Computing S^T rather than S puts key rows on the TMEM lanes, which is the
// row layout the A operand of dV += P^T dO and dK += dS^T Q needs, so P^T and
// dS^T go back into TMEM and never touch shared memory.
//
// TMEM columns (512): dV [0,128), dK [128,256) and two step buffers of 128
// columns at 256 and 384, step n using buffer n & 1: fp32 S^T in its first 64
// columns, fp32 dP^T in the next 64.  Softmax group g owns query columns
// 16 g .. 16 g + 15 of each half and writes its 16 packed P^T values over the
// first 8 of its own S^T columns (and dS^T over its dP^T columns), so the 16
// queries of MMA K-step g sit at column 16 g of the half.  S^T(n + 2) may
// overwrite a buffer once dV(n) has read the P^T in it, dP^T(n + 2) once dK(n)
// has read the dS^T: every MMA has a whole step in which to run ahead of the
// softmax warps, and the softmax warps never wait for an MMA to finish
// reading, only for their own inputs.  K stays in shared memory: S^T = K Q^T
// reads both operands from there, as dP^T = V dO^T does.
//
// Four warps issue MMAs into the one tensor pipe, each waiting only on its own
// inputs: warp 1 S^T(m), warp 2 dP^T(m), warp 3 dV(n), warp 4 dK(n).  The pipe
// accepts only a few MMAs ahead of the one executing and a barrier wait costs
// a few hundred cycles while the softmax warps keep the SM busy, so one
// issuing warp would drain the pipe at every wait.
//
// Warp roles (672 threads): warp 0 issues TMA loads, warp 1 owns TMEM; warps
// 1..4 issue MMAs (whole warps, one elected lane); warps 5..20 are the
// softmax warps: warp (sp, g) with sp = warp % 4 owns TMEM lanes
// 32 sp .. 32 sp + 31 (key rows) and query columns 16 g .. 16 g + 15.
#include <math.h>

#include "kv_softmax.cuh"

namespace mab {

namespace kv_side {

constexpr int STAGES = 4;      // Q/dO ring depth
constexpr int COL_DV = 0;
constexpr int COL_DK = 128;
constexpr int COL_BUF = 256;   // buffer b at COL_BUF + 128 b: S^T at +0, dP^T at +64
constexpr int SM_WARPS = 16;   // softmax warps
constexpr int SM_WARP0 = 5;     // first softmax warp
constexpr int NUM_THREADS = 32 * (SM_WARP0 + SM_WARPS);

struct __align__(1024) Smem {
  uint8_t K[2 * KV_TILE * 128];
  uint8_t V[2 * KV_TILE * 128];
  uint8_t Q[STAGES][2 * KV_SUB * 128];   // the first two stages stage the epilogue rows
  uint8_t dO[STAGES][2 * KV_SUB * 128];
  float nlse2[STAGES][KV_SUB];  // -lse log2(e) of the stage's query rows
  float delta[STAGES][KV_SUB];
  int step_r[STAGES];            // query sub-tile of the step in the stage
  int step_hh[STAGES];           // its query head within the group
  uint32_t step_vis[STAGES];     // aligned block masks: bit 4 sp + g = region (sp, g) visible
  uint64_t bar_kv_full;          // K, V landed
  uint64_t bar_q_full[STAGES];
  uint64_t bar_q_empty[STAGES];  // dV and dK of the step complete (one commit each)
  uint64_t bar_s_full[2];        // S^T of the buffer complete
  uint64_t bar_dp_full[2];       // dP^T of the buffer complete
  uint64_t bar_p_full[2];        // P^T written over the buffer's S^T (every softmax warp)
  uint64_t bar_ds_full[2];       // dS^T written over the buffer's dP^T (every softmax warp)
  uint64_t bar_s_free[2];        // dV that read the buffer's P^T complete
  uint64_t bar_dp_free[2];       // dK that read the buffer's dS^T complete
  uint64_t bar_x_done[2];        // every S^T (0) / dP^T (1) MMA complete
  uint64_t bar_acc_full;         // every dV and dK MMA complete (one commit each)
  uint32_t tmem_base;
  int abort_flag;
  int is_last;                   // this CTA finished last: it sums dSink
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;
static_assert(SMEM_BYTES <= 232448, "over the 227 KB of shared memory a CTA may use");
static_assert(2 * (2 * KV_SUB * 128) >= SM_WARPS * 2048, "epilogue staging fits in two Q stages");

enum { TAG_KV = 0x201, TAG_Q_EMPTY = 0x203, TAG_Q_FULL, TAG_S_FREE, TAG_P_FULL, TAG_S_FULL,
       TAG_DP_FULL, TAG_DS_FULL, TAG_ACC, TAG_X_DONE, TAG_DP_FREE };

}  // namespace kv_side

// HILO: P^T and dS^T enter dV and dK as a 16-bit high part plus a 16-bit
// remainder, the remainder packed over the second 8 of the softmax group's
// own columns.
// PACKED: the token-major layout with cumulative sequence offsets (the BHSD
// instances keep their plain row addressing).
template <bool BF16, bool HILO, bool PACKED>
__global__ void __launch_bounds__(kv_side::NUM_THREADS, 1)
k_dkdv(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tdO,
       const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV,
       uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, const AttnParams p) {
  using namespace kv_side;
  constexpr int NST = STAGES;  // Q/dO ring length
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BHkv = p.B * p.Hkv;
  const int t = (int)(blockIdx.x / BHkv);  // low key tiles (longest causal walks) first
  const int bc = (int)(blockIdx.x % BHkv);
  const int b = bc / p.Hkv, c = bc % p.Hkv;
  const int k0 = t * KV_TILE;
  const int Lq = len_q(p, b), Lk = len_k(p, b);  // valid rows and keys of the batch
  // block masks: the walk reads the select tables, which the grids before
  // this one (launched with programmatic serialization) are still writing
  if (p.mask_kind == MK_BLOCK) grid_dependency_wait();
  KVWalk walk;
  walk.init(p, b, c, t, Lq, Lk);
  const int N = walk.total(p);
  // a block mask whose blocks hold whole softmax-warp regions (32 keys x 16
  // queries): each region is visible entirely or not at all
  const bool blk_regions = p.mask_kind == MK_BLOCK && (p.by & 31) == 0 && (p.bx & 15) == 0;
  WaitCtx wc{p.status, &s.abort_flag, p.timeout_ns};

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar_kv_full), 1);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.bar_q_full[i]), 1);
      mbar_init(smem_u32(&s.bar_q_empty[i]), 2);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_dp_full[i]), 1);
      mbar_init(smem_u32(&s.bar_p_full[i]), SM_WARPS);
      mbar_init(smem_u32(&s.bar_ds_full[i]), SM_WARPS);
      mbar_init(smem_u32(&s.bar_s_free[i]), 1);
      mbar_init(smem_u32(&s.bar_dp_free[i]), 1);
      mbar_init(smem_u32(&s.bar_x_done[i]), 1);
    }
    mbar_init(smem_u32(&s.bar_acc_full), 2);
    fence_mbar_init();
    // K and V of the tile, loaded while the rest of the CTA sets up (they do
    // not depend on the kernels before this one); a key tile without any step
    // only gets zeros: K and V are not loaded (and no warp waits for them)
    if (N > 0 && !p.test_no_loads) {
      tma_prefetch_desc(&tK);
      tma_prefetch_desc(&tV);
      const uint32_t kvbar = smem_u32(&s.bar_kv_full);
      const RowAddr ka = PACKED ? row_k(p, b, c, k0) : RowAddr{k0, bc, 0, HEAD_DIM};
      mbar_arrive_expect_tx(kvbar, 4 * KV_TILE * 128);
      tma_load_3d(smem_u32(s.K), &tK, 0, ka.c1, ka.c2, kvbar);
      tma_load_3d(smem_u32(s.K + KV_TILE * 128), &tK, 64, ka.c1, ka.c2, kvbar);
      tma_load_3d(smem_u32(s.V), &tV, 0, ka.c1, ka.c2, kvbar);
      tma_load_3d(smem_u32(s.V + KV_TILE * 128), &tV, 64, ka.c1, ka.c2, kvbar);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  // Launched behind the preprocess kernel with programmatic serialization,
  // this grid may start before that one has finished: wait for it before any
  // of its results are read (block masks waited above already).  Only then let the dQ
  // kernel that follows start (it needs nothing from this grid, but reads the
  // preprocess results): it may take the SMs this grid's last CTAs leave idle.
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !p.test_no_loads) {
      tma_prefetch_desc(&tQ);
      tma_prefetch_desc(&tdO);
      const uint32_t kvbar = smem_u32(&s.bar_kv_full);
      // a short walk ends soon: bring the K / V tile of the CTA that will
      // likely take this SM next (the grid is dispatched in order, one CTA per
      // SM) into L2 now, so that its first wait is for L2 rather than HBM
      const int succ = (int)blockIdx.x + p.num_sms;
      if (N <= 64 && succ < (int)gridDim.x) {
        const int t2 = succ / BHkv, bc2 = succ % BHkv;
        const RowAddr a2 = PACKED ? row_k(p, bc2 / p.Hkv, bc2 % p.Hkv, t2 * KV_TILE)
                                  : RowAddr{t2 * KV_TILE, bc2, 0, HEAD_DIM};
        tma_prefetch_l2_3d(&tK, 0, a2.c1, a2.c2);
        tma_prefetch_l2_3d(&tK, 64, a2.c1, a2.c2);
        tma_prefetch_l2_3d(&tV, 0, a2.c1, a2.c2);
        tma_prefetch_l2_3d(&tV, 64, a2.c1, a2.c2);
      }
      KVCursor cur;
      cur.start(p, walk);
      int issued = 0;  // steps whose loads were issued
      for (int n = 0; n < N; ++n) {
        const int st = n % NST;
        int r, hh;
        kv_step(p, walk, cur, &hh, &r);
        const int bh = b * p.Hq + c * p.group + hh;
        // aligned block masks: the mask byte of each softmax warp's 32-key x
        // 16-query region, loaded before the waits below (which hide the
        // latency; indices clamped into the mask, ranges applied after)
        uint32_t mv[16];
        if (blk_regions) {
          const uint8_t* mt = p.maskT + (size_t)bh * p.nkb * p.nqb;
#pragma unroll
          for (int sp2 = 0; sp2 < 4; ++sp2) {
            const int kb = min((k0 + 32 * sp2) / p.by, p.nkb - 1);
#pragma unroll
            for (int g2 = 0; g2 < 4; ++g2) {
              const int qb = min((r * KV_SUB + 16 * g2) / p.bx, p.nqb - 1);
              mv[4 * sp2 + g2] = mt[(size_t)kb * p.nqb + qb];
            }
          }
        }
        if (n >= NST &&
            !mbar_wait(smem_u32(&s.bar_q_empty[st]), ((n / NST) - 1) & 1, wc, TAG_Q_EMPTY))
          break;
        // the step's coordinates for the softmax warps, published by the
        // arrive below together with the loads
        s.step_r[st] = r;
        s.step_hh[st] = hh;
        if (blk_regions) {
          uint32_t w = 0;
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (mv[e] && k0 + 32 * (e >> 2) < p.Skv && r * KV_SUB + 16 * (e & 3) < p.Sq)
              w |= 1u << e;
          s.step_vis[st] = w;
        }
        const uint32_t fb = smem_u32(&s.bar_q_full[st]);
        mbar_arrive_expect_tx(fb, 4 * KV_SUB * 128 + 2 * KV_SUB * 4);
        uint8_t* sq = s.Q[st];
        uint8_t* sd = s.dO[st];
        const RowAddr qa = PACKED ? row_q(p, b, c * p.group + hh, r * KV_SUB)
                                  : RowAddr{r * KV_SUB, bh, 0, HEAD_DIM};
        tma_load_3d(smem_u32(sq), &tQ, 0, qa.c1, qa.c2, fb);
        tma_load_3d(smem_u32(sq + KV_SUB * 128), &tQ, 64, qa.c1, qa.c2, fb);
        tma_load_3d(smem_u32(sd), &tdO, 0, qa.c1, qa.c2, fb);
        tma_load_3d(smem_u32(sd + KV_SUB * 128), &tdO, 64, qa.c1, qa.c2, fb);
        const size_t srow = (size_t)bh * p.Sq_pad + (size_t)r * KV_SUB;
        bulk_load(smem_u32(s.nlse2[st]), p.nlse2 + srow, KV_SUB * 4, fb);
        bulk_load(smem_u32(s.delta[st]), p.delta + srow, KV_SUB * 4, fb);
        issued = n + 1;
      }
      if (issued < N) {
        // the CTA gave up: let the copies still in flight land before it exits
        mbar_drain(kvbar, 0, wc.timeout_ns);
        for (int n = issued > NST ? issued - NST : 0; n < issued; ++n)
          mbar_drain(smem_u32(&s.bar_q_full[n % NST]), (n / NST) & 1, wc.timeout_ns);
      }
    }
  } else if (warp >= 1 && warp < SM_WARP0) {
    // ------------------------------------------------------------ MMA issuers (whole warps)
    constexpr uint32_t ID_S = idesc_f16(BF16, KV_TILE, KV_SUB, false, false);
    constexpr uint32_t ID_ACC = idesc_f16(BF16, KV_TILE, HEAD_DIM, false, true);
    if (warp == 1 || warp == 2) {
      // warp 1: S^T(m) = K Q^T; warp 2: dP^T(m) = V dO^T, into buffer m & 1
      // (A = K / V tile, B = Q / dO tile, both K-major in shared memory).
      // Each waits for the accumulation that read the buffer two steps ago.
      const bool is_s = warp == 1;
      const uint64_t aKV = sdesc_sw128(smem_u32(is_s ? s.K : s.V), 16, 1024);
      bool ok = N == 0 || mbar_wait_warp(smem_u32(&s.bar_kv_full), 0, wc, TAG_KV);
      for (int m = 0; ok && m < N; ++m) {
        const int st = m % NST, bf = m & 1;
        ok = mbar_wait_warp(smem_u32(&s.bar_q_full[st]), (m / NST) & 1, wc, TAG_Q_FULL);
        if (ok && m >= 2)
          ok = mbar_wait_warp(smem_u32(is_s ? &s.bar_s_free[bf] : &s.bar_dp_free[bf]),
                              ((m - 2) >> 1) & 1, wc, is_s ? TAG_S_FREE : TAG_DP_FREE);
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
      // this warp's MMAs must be complete before TMEM is freed (also when the
      // CTA gave up, hence a wait that ignores the abort flag)
      const uint32_t done = smem_u32(&s.bar_x_done[is_s ? 0 : 1]);
      mma_commit_w(done);
      mbar_drain_warp(done, 0, wc.timeout_ns);
    } else {
      // warp 3: dV += P^T(n) dO; warp 4: dK += dS^T(n) Q (A = the packed
      // values in buffer n & 1, B MN-major).  Each commit frees its half of
      // the buffer; both commit to q_empty and acc_full, which complete on
      // the two commits.
      const bool dkside = warp == 4;
      const uint32_t acc = tbase + (dkside ? COL_DK : COL_DV);
      bool ok = true;
      for (int n = 0; ok && n < N; ++n) {
        const int st = n % NST, bf = n & 1;
        ok = mbar_wait_warp(smem_u32(dkside ? &s.bar_ds_full[bf] : &s.bar_p_full[bf]),
                            (n >> 1) & 1, wc, dkside ? TAG_DS_FULL : TAG_P_FULL);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a = tbase + COL_BUF + 128 * bf + (dkside ? 64 : 0);
        const uint64_t bB =
            sdesc_sw128(smem_u32(dkside ? s.Q[st] : s.dO[st]), KV_SUB * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < KV_SUB / 16; ++kk)
          mma_ts_w(acc, a + 16 * kk, bB + (uint64_t)((kk * 2048) >> 4), ID_ACC,
                   (n > 0 || kk > 0) ? 1u : 0u);
        if (HILO) {
#pragma unroll
          for (int kk = 0; kk < KV_SUB / 16; ++kk)
            mma_ts_w(acc, a + 16 * kk + 8, bB + (uint64_t)((kk * 2048) >> 4), ID_ACC, 1u);
        }
        mma_commit_w(smem_u32(dkside ? &s.bar_dp_free[bf] : &s.bar_s_free[bf]));
        // S^T(n) and dP^T(n) completed before the softmax warps could write
        // P^T(n) / dS^T(n), so the two commits also free the Q / dO stage
        mma_commit_w(smem_u32(&s.bar_q_empty[st]));
      }
      // completes when every MMA of both warps has (also when the CTA gave
      // up, so that TMEM is idle before it is freed)
      mma_commit_w(smem_u32(&s.bar_acc_full));
      mbar_drain_warp(smem_u32(&s.bar_acc_full), 0, wc.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int sp = warp & 3, g = (warp - SM_WARP0) >> 2;
    const int rloc = sp * 32 + lane;
    const int j = k0 + rloc;
    const uint32_t lane_base = tbase + ((uint32_t)(sp * 32) << 16);
    bool ok = true;

    // signal one barrier from this warp once its TMEM accesses are done
    auto warp_arrive = [&](uint64_t* bar) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(bar));
    };
    int flo, fhi;  // query sub-tiles that are entirely visible
    full_range_kv(p.mask_kind, p.window, Lq, Lk, k0, &flo, &fhi);
    for (int n = 0; ok && n < N; ++n) {
      const int st = n % NST, bf = n & 1;
      const uint32_t colS = COL_BUF + 128 * bf + 16 * g;  // this warp's S^T / P^T columns
      // ---- P^T(n) = exp2(S^T(n) * scale*log2e - lse log2e)
      // s_full implies the stage's loads landed; waiting on q_full as well
      // makes the bulk-copied -lse log2e / Delta rows visible to this thread
      if (!mbar_wait(smem_u32(&s.bar_s_full[bf]), (n >> 1) & 1, wc, TAG_S_FULL) ||
          !mbar_wait(smem_u32(&s.bar_q_full[st]), (n / NST) & 1, wc, TAG_Q_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[16];
      tmem_ld16(lane_base + colS, sv);
      const int r = s.step_r[st];
      // warp-uniform: the whole 64 x 128 sub-tile is visible
      const bool full = r >= flo && r <= fhi;
      uint32_t vis;
      if (full) {
        vis = 0xffffu;
      } else if (blk_regions) {
        vis = ((s.step_vis[st] >> (4 * sp + g)) & 1u) && j < Lk
                  ? bit_range(0, Lq - 1 - (r * KV_SUB + 16 * g))
                  : 0u;
      } else {
        vis = vis_key_row(p, b * p.Hq + c * p.group + s.step_hh[st], j, r * KV_SUB + 16 * g, Lq,
                          Lk);
      }
      float lv[16];
      load16_shared(&s.nlse2[st][16 * g], lv);
      tmem_wait_ld_regs(sv);
      float pv[16];
      kv_write_p<BF16, HILO>(lane_base + colS, sv, lv, full, vis, p.scale_log2, pv);
      warp_arrive(&s.bar_p_full[bf]);

      // ---- dS^T(n) = P^T(n) (dP^T(n) - Delta)
      float dl[16];
      load16_shared(&s.delta[st][16 * g], dl);
      if (!mbar_wait(smem_u32(&s.bar_dp_full[bf]), (n >> 1) & 1, wc, TAG_DP_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float dp[16];
      tmem_ld16(lane_base + colS + 64, dp);
      tmem_wait_ld_regs(dp);
      uint32_t pk[8];
      kv_write_ds<BF16, HILO>(lane_base + colS + 64, pv, dp, dl, pk);
      warp_arrive(&s.bar_ds_full[bf]);
    }
    // ---------------------------------------------------------- epilogue
    bool have = ok && N > 0;
    if (have) have = mbar_wait(smem_u32(&s.bar_acc_full), 0, wc, TAG_ACC);
    tc_fence_after();
    // After a complete walk every MMA has completed and every stage was
    // consumed, so no stage is being read or loaded: the first two Q tiles
    // stage the output rows.  A key tile without steps loaded nothing.  A CTA
    // that gave up may still have copies in flight into the stages, so it
    // stores its zeros straight to global memory instead.
    named_bar_sync(1, 32 * SM_WARPS);
    const int r0 = k0 + sp * 32;
    const int nvalid = PACKED ? rows_to_store_k(p, b, r0) : min(32, p.Skv - r0);
    const RowAddr oa = PACKED ? row_k(p, b, c, r0)
                              : RowAddr{r0, bc, ((size_t)bc * p.Skv + r0) * HEAD_DIM, HEAD_DIM};
    uint8_t* stage = s.Q[0] + (warp - SM_WARP0) * 2048;
    const bool staged = __all_sync(0xffffffffu, have || (ok && N == 0));
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK
      uint16_t* base = which ? dk : dv;
      uint16_t* orow = base + oa.elem + 32 * g;
      if (!staged) {
        warp_zero_rows(orow, 32, nvalid, oa.stride);
        continue;
      }
      uint32_t pk[16];
      if (have) {
        const float sc = which ? p.scale : 1.f;
        float v[32];
        tmem_ld32(lane_base + (which ? COL_DK : COL_DV) + 32 * g, v);
        tmem_wait_ld_regs(v);
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) pk[cc] = pack2<BF16>(v[2 * cc] * sc, v[2 * cc + 1] * sc);
      } else {
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) pk[cc] = 0u;
      }
      warp_store_rows32(stage, pk, orow, nvalid, oa.stride);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // dSink by the grid's last CTA, off the critical path of the dQ grid that
  // runs beside this one's tail (the partials come from the preprocess grid,
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

// Whether the persistent form (attn_kv_units.cu) runs the dK/dV walk: for the
// BHSD layout when there are at least two units per SM and the walks are
// short -- block masks, or closed-form masks whose key tiles average at most
// 64 steps at the full lengths -- where a CTA per unit would spend much of
// its time starting and storing.  On long walks the per-tile grid is faster.
static bool use_units(const AttnParams& p) {
  if (p.cu_q) return false;
  if (p.kv_schedule != 0) return p.kv_schedule == 2;
  const long long units = (long long)p.nKT_k * p.B * p.Hkv;
  if (units < 2LL * (p.num_sms > 0 ? p.num_sms : 1)) return false;
  if (p.mask_kind == MK_BLOCK) return true;
  long long steps = 0;
  for (int t = 0; t < p.nKT_k; ++t) {
    int lo;
    steps += kv_tile_range_full(p.mask_kind, p.window, p.Sq, p.Skv, t, &lo);
  }
  return steps * p.group <= 64LL * p.nKT_k;
}

cudaError_t launch_dkdv(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                        const CUtensorMap& tdO, const CUtensorMap& tK, const CUtensorMap& tV,
                        void* dk, void* dv, cudaStream_t st) {
  if (use_units(p)) return launch_dkdv_units(bf16, p, tQ, tdO, tK, tV, dk, dv, st);
  using Kern = decltype(&k_dkdv<true, false, false>);
  static const Kern table[2][2][2] = {
      {{k_dkdv<false, false, false>, k_dkdv<false, false, true>},
       {k_dkdv<false, true, false>, k_dkdv<false, true, true>}},
      {{k_dkdv<true, false, false>, k_dkdv<true, false, true>},
       {k_dkdv<true, true, false>, k_dkdv<true, true, true>}}};
  const Kern kern = table[bf16 ? 1 : 0][p.compensated ? 1 : 0][p.cu_q ? 1 : 0];
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kv_side::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int nKT = (p.Skv + KV_TILE - 1) / KV_TILE;
  // programmatic stream serialization behind the preprocess kernel, so that
  // this grid's launch and (closed-form masks) set-up and K / V loads overlap
  // its tail; block-mask CTAs wait for it before they read the select tables
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nKT * p.B * p.Hkv));
  cfg.blockDim = dim3(kv_side::NUM_THREADS);
  cfg.dynamicSmemBytes = kv_side::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tQ, tdO, tK, tV, (uint16_t*)dk, (uint16_t*)dv, p);
}

}  // namespace mab
