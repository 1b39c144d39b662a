// attn_fused.cu -- single-pass backward (ATTN_FLAG_SINGLE_PASS): the
// key-stationary kernel computes dQ as well, so S and dP are computed once per
// visible tile instead of twice, and a deterministic reduction sums the dQ
// partials.
//
//   k_dkdvq        one CTA per (b, kv head, KV_TILE key rows), as k_dkdv: for
//                  every step (query head of the group, query sub-tile r of
//                  KV_SUB rows) S^T = K Q^T, dP^T = V dO^T, P^T, dS^T,
//                  dV += P^T dO, dK += dS^T Q, and in addition the step's dQ
//                  partial dQ_r^T = K^T dS^T (128 head dims x 64 queries),
//                  which the softmax warps drain into its own fp32 slot of
//                  the workspace and mark as written.
//   k_dq_reduce    per (b, q head, query sub-tile): the written partials of
//                  the sub-tile, in ascending key-tile order (a fixed order,
//                  so the result does not depend on scheduling), times the
//                  softmax scale, rounded to the input dtype.
//
// Sources: cannbot-knowledge PR #174, BlockSparseAttentionGrad change log
// (single-pass fusion of the five contractions with a dK/dV partial workspace
// and a reduce kernel), turned around here: dK/dV stay in TMEM for the whole
// GQA group (contiguous write-back, optimisation 3), and dQ is the quantity
// whose partials go through the workspace; tilelang-ascend PR #1 commit notes
// (one backward kernel: five contractions + softmax + dS per step).
//
// TMEM columns (512): dV [0,128), dK [128,256), S^T / P^T [256,320), dP^T /
// dS^T [320,384) (one step buffer: P^T and dS^T are written over the fp32
// values, each softmax warp over its own columns), dQ^T partial [384,448).
// dS^T also goes to shared memory as a 16-bit 128-key x 64-query tile, the B
// operand of dQ^T = K^T dS^T (A = the K tile read M-major).
//
// Warp roles (672 threads): warp 0 loads, warp 1 issues S^T (and owns TMEM),
// warp 2 dP^T, warp 3 dV, warp 4 dK and dQ^T; warps 5..20 are the softmax
// warps: warp (sp, g) owns TMEM lanes 32 sp .. 32 sp + 31 and query columns
// 16 g .. 16 g + 15, and drains head dims 32 sp + lane x queries
// 16 g .. 16 g + 15 of each dQ partial.
#include <math.h>

#include "kv_softmax.cuh"

namespace mab {

namespace fused_side {

constexpr int STAGES = 4;
constexpr int COL_DV = 0;
constexpr int COL_DK = 128;
constexpr int COL_S = 256;   // S^T, then P^T over it
constexpr int COL_DP = 320;  // dP^T, then dS^T over it
constexpr int COL_DQ = 384;  // dQ^T partial of the step
constexpr int SM_WARPS = 16;
constexpr int SM_WARP0 = 5;
constexpr int NUM_THREADS = 32 * (SM_WARP0 + SM_WARPS);

struct __align__(1024) Smem {
  uint8_t K[2 * KV_TILE * 128];
  uint8_t V[2 * KV_TILE * 128];
  uint8_t Q[STAGES][2 * KV_SUB * 128];  // the first two stages stage the epilogue rows
  uint8_t dO[STAGES][2 * KV_SUB * 128];
  uint8_t dS[KV_TILE * 128];             // dS^T, 128 keys x 64 queries, 128B swizzle
  float nlse2[STAGES][KV_SUB];
  float delta[STAGES][KV_SUB];
  int step_r[STAGES];
  int step_hh[STAGES];
  uint32_t step_vis[STAGES];
  long long slot_pre;            // dQ partial slots of the key tiles before this one
  int slot_lo;                   // first query sub-tile of this tile's full-length range
  uint64_t bar_kv_full;
  uint64_t bar_q_full[STAGES];
  uint64_t bar_q_empty[STAGES];  // dV and dK of the step complete
  uint64_t bar_s_full;           // S^T complete
  uint64_t bar_s_free;           // dV that read P^T complete
  uint64_t bar_dp_full;          // dP^T complete
  uint64_t bar_dp_free;          // dK that read dS^T complete
  uint64_t bar_p_full;           // P^T written (every softmax warp)
  uint64_t bar_ds_full;          // dS^T written to TMEM and shared memory (every softmax warp)
  uint64_t bar_dq_full;          // dQ^T partial complete
  uint64_t bar_dq_free;          // dQ^T partial drained (every softmax warp)
  uint64_t bar_x_done[2];
  uint64_t bar_acc_full;         // every dV, dK and dQ^T MMA complete (two commits)
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;
static_assert(SMEM_BYTES <= 232448, "over the 227 KB of shared memory a CTA may use");

enum { TAG_KV = 0x601, TAG_Q_EMPTY, TAG_Q_FULL, TAG_S_FREE, TAG_P_FULL, TAG_S_FULL, TAG_DP_FULL,
       TAG_DS_FULL, TAG_ACC, TAG_X_DONE, TAG_DP_FREE, TAG_DQ_FULL, TAG_DQ_FREE };

}  // namespace fused_side

// Workspace slot of the dQ partial of query head bh and query sub-tile r in
// a key tile whose slots start at `pre` (within the head) and whose
// full-length range starts at sub-tile `lo`; a slot is KV_SUB x HEAD_DIM
// floats, row-major.
__device__ __forceinline__ size_t dq_slot(const AttnParams& p, int bh, long long pre, int lo,
                                          int r) {
  return (size_t)((long long)bh * p.dq_steps_head + pre + (r - lo));
}

// Sum over key tiles u = i, i + n, ... below t of their full-length range
// lengths: one thread's share of the slots before key tile t.
__device__ __forceinline__ long long slots_before_share(const AttnParams& p, int t, int i, int n) {
  long long acc = 0;
  for (int u = i; u < t; u += n) {
    int lo;
    acc += kv_tile_range_full(p.mask_kind, p.window, p.Sq, p.Skv, u, &lo);
  }
  return acc;
}

template <bool BF16>
__global__ void __launch_bounds__(fused_side::NUM_THREADS, 1)
k_dkdvq(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tdO,
        const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV,
        uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, const AttnParams p) {
  using namespace fused_side;
  constexpr int NST = STAGES;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BHkv = p.B * p.Hkv;
  const int t = (int)(blockIdx.x / BHkv);
  const int bc = (int)(blockIdx.x % BHkv);
  const int b = bc / p.Hkv, c = bc % p.Hkv;
  const int k0 = t * KV_TILE;
  const int Lq = len_q(p, b), Lk = len_k(p, b);
  // block masks: the walk reads the select tables, which the grids before
  // this one (launched with programmatic serialization) are still writing
  if (p.mask_kind == MK_BLOCK) grid_dependency_wait();
  KVWalk walk;
  walk.init(p, b, c, t, Lq, Lk);
  const int N = walk.total(p);
  const bool blk_regions = p.mask_kind == MK_BLOCK && (p.by & 31) == 0 && (p.bx & 15) == 0;
  WaitCtx wc{p.status, &s.abort_flag, p.timeout_ns};

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar_kv_full), 1);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.bar_q_full[i]), 1);
      mbar_init(smem_u32(&s.bar_q_empty[i]), 2);
    }
    mbar_init(smem_u32(&s.bar_s_full), 1);
    mbar_init(smem_u32(&s.bar_s_free), 1);
    mbar_init(smem_u32(&s.bar_dp_full), 1);
    mbar_init(smem_u32(&s.bar_dp_free), 1);
    mbar_init(smem_u32(&s.bar_p_full), SM_WARPS);
    mbar_init(smem_u32(&s.bar_ds_full), SM_WARPS);
    mbar_init(smem_u32(&s.bar_dq_full), 1);
    mbar_init(smem_u32(&s.bar_dq_free), SM_WARPS);
    mbar_init(smem_u32(&s.bar_x_done[0]), 1);
    mbar_init(smem_u32(&s.bar_x_done[1]), 1);
    mbar_init(smem_u32(&s.bar_acc_full), 2);
    fence_mbar_init();
    if (N > 0 && !p.test_no_loads) {
      tma_prefetch_desc(&tK);
      tma_prefetch_desc(&tV);
      const uint32_t kvbar = smem_u32(&s.bar_kv_full);
      mbar_arrive_expect_tx(kvbar, 4 * KV_TILE * 128);
      tma_load_3d(smem_u32(s.K), &tK, 0, k0, bc, kvbar);
      tma_load_3d(smem_u32(s.K + KV_TILE * 128), &tK, 64, k0, bc, kvbar);
      tma_load_3d(smem_u32(s.V), &tV, 0, k0, bc, kvbar);
      tma_load_3d(smem_u32(s.V + KV_TILE * 128), &tV, 64, k0, bc, kvbar);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == 3) {
    // where this key tile's dQ partial slots start within a query head
    long long pre = slots_before_share(p, t, lane, 32);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
    if (lane == 0) {
      int lo;
      kv_tile_range_full(p.mask_kind, p.window, p.Sq, p.Skv, t, &lo);
      s.slot_pre = pre;
      s.slot_lo = lo;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  // Launched behind the preprocess kernel with programmatic serialization
  // (closed-form masks): wait for its results before any is read.
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !p.test_no_loads) {
      tma_prefetch_desc(&tQ);
      tma_prefetch_desc(&tdO);
      const uint32_t kvbar = smem_u32(&s.bar_kv_full);
      KVCursor cur;
      cur.start(p, walk);
      int issued = 0;
      for (int n = 0; n < N; ++n) {
        const int st = n % NST;
        int r, hh;
        kv_step(p, walk, cur, &hh, &r);
        const int bh = b * p.Hq + c * p.group + hh;
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
        tma_load_3d(smem_u32(s.Q[st]), &tQ, 0, r * KV_SUB, bh, fb);
        tma_load_3d(smem_u32(s.Q[st] + KV_SUB * 128), &tQ, 64, r * KV_SUB, bh, fb);
        tma_load_3d(smem_u32(s.dO[st]), &tdO, 0, r * KV_SUB, bh, fb);
        tma_load_3d(smem_u32(s.dO[st] + KV_SUB * 128), &tdO, 64, r * KV_SUB, bh, fb);
        const size_t srow = (size_t)bh * p.Sq_pad + (size_t)r * KV_SUB;
        bulk_load(smem_u32(s.nlse2[st]), p.nlse2 + srow, KV_SUB * 4, fb);
        bulk_load(smem_u32(s.delta[st]), p.delta + srow, KV_SUB * 4, fb);
        issued = n + 1;
      }
      if (issued < N) {
        mbar_drain(kvbar, 0, wc.timeout_ns);
        for (int n = issued > NST ? issued - NST : 0; n < issued; ++n)
          mbar_drain(smem_u32(&s.bar_q_full[n % NST]), (n / NST) & 1, wc.timeout_ns);
      }
    }
  } else if (warp >= 1 && warp < SM_WARP0) {
    // ------------------------------------------------------------ MMA issuers
    constexpr uint32_t ID_S = idesc_f16(BF16, KV_TILE, KV_SUB, false, false);
    constexpr uint32_t ID_ACC = idesc_f16(BF16, KV_TILE, HEAD_DIM, false, true);
    // dQ^T (M = 128 head dims, N = 64 queries, K = 128 keys): A = K^T and
    // B = dS^T, both read M- / N-major from shared memory
    constexpr uint32_t ID_DQ = idesc_f16(BF16, HEAD_DIM, KV_SUB, true, true);
    if (warp == 1 || warp == 2) {
      const bool is_s = warp == 1;
      const uint64_t aKV = sdesc_sw128(smem_u32(is_s ? s.K : s.V), 16, 1024);
      bool ok = N == 0 || mbar_wait_warp(smem_u32(&s.bar_kv_full), 0, wc, TAG_KV);
      for (int m = 0; ok && m < N; ++m) {
        const int st = m % NST;
        ok = mbar_wait_warp(smem_u32(&s.bar_q_full[st]), (m / NST) & 1, wc, TAG_Q_FULL);
        if (ok && m >= 1)
          ok = mbar_wait_warp(smem_u32(is_s ? &s.bar_s_free : &s.bar_dp_free), (m - 1) & 1, wc,
                              is_s ? TAG_S_FREE : TAG_DP_FREE);
        if (!ok) break;
        tc_fence_after();
        const uint64_t bB = sdesc_sw128(smem_u32(is_s ? s.Q[st] : s.dO[st]), 16, 1024);
        const uint32_t d = tbase + (is_s ? COL_S : COL_DP);
#pragma unroll
        for (int kk = 0; kk < HEAD_DIM / 16; ++kk)
          mma_ss_w(d, aKV + (uint64_t)(((kk >> 2) * (KV_TILE * 128) + (kk & 3) * 32) >> 4),
                   bB + (uint64_t)(((kk >> 2) * (KV_SUB * 128) + (kk & 3) * 32) >> 4), ID_S,
                   kk > 0 ? 1u : 0u);
        mma_commit_w(smem_u32(is_s ? &s.bar_s_full : &s.bar_dp_full));
      }
      const uint32_t done = smem_u32(&s.bar_x_done[is_s ? 0 : 1]);
      mma_commit_w(done);
      mbar_drain_warp(done, 0, wc.timeout_ns);
    } else {
      // warp 3: dV += P^T(n) dO; warp 4: dK += dS^T(n) Q, then the step's
      // dQ^T partial once the previous one has been drained
      const bool dkside = warp == 4;
      const uint32_t acc = tbase + (dkside ? COL_DK : COL_DV);
      const uint32_t a = tbase + (dkside ? COL_DP : COL_S);
      const uint64_t aKt = sdesc_sw128(smem_u32(s.K), KV_TILE * 128, 1024);
      const uint64_t bdS = sdesc_sw128(smem_u32(s.dS), KV_TILE * 128, 1024);
      bool ok = true;
      for (int n = 0; ok && n < N; ++n) {
        const int st = n % NST;
        ok = mbar_wait_warp(smem_u32(dkside ? &s.bar_ds_full : &s.bar_p_full), n & 1, wc,
                            dkside ? TAG_DS_FULL : TAG_P_FULL);
        if (!ok) break;
        tc_fence_after();
        const uint64_t bB =
            sdesc_sw128(smem_u32(dkside ? s.Q[st] : s.dO[st]), KV_SUB * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < KV_SUB / 16; ++kk)
          mma_ts_w(acc, a + 16 * kk, bB + (uint64_t)((kk * 2048) >> 4), ID_ACC,
                   (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(smem_u32(dkside ? &s.bar_dp_free : &s.bar_s_free));
        mma_commit_w(smem_u32(&s.bar_q_empty[st]));
        if (dkside) {
          // dQ^T(n) = K^T dS^T(n) into the partial's columns, once every
          // softmax warp has drained dQ^T(n - 1)
          if (n >= 1) ok = mbar_wait_warp(smem_u32(&s.bar_dq_free), (n - 1) & 1, wc, TAG_DQ_FREE);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < KV_TILE / 16; ++kk)
            mma_ss_w(tbase + COL_DQ, aKt + (uint64_t)((kk * 2048) >> 4),
                     bdS + (uint64_t)((kk * 2048) >> 4), ID_DQ, kk > 0 ? 1u : 0u);
          mma_commit_w(smem_u32(&s.bar_dq_full));
        }
      }
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
    const long long slot_pre = s.slot_pre;
    const int slot_lo = s.slot_lo;
    auto warp_arrive = [&](uint64_t* bar) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(bar));
    };
    // Drains this warp's share of the dQ^T partial of step n (query sub-tile
    // r of query head hh): head dims 32 sp + lane of queries 16 g .. 16 g + 15
    // into the step's slot (each store 32 consecutive floats of one query
    // row).  One thread marks the slot as written; the reduction reads it only
    // after this grid has completed, when every share is in memory.
    auto drain = [&](int n, int r, int hh) -> bool {
      if (!mbar_wait(smem_u32(&s.bar_dq_full), n & 1, wc, TAG_DQ_FULL)) return false;
      tc_fence_after();
      float v[16];
      tmem_ld16(lane_base + COL_DQ + 16 * g, v);
      tmem_wait_ld_regs(v);
      warp_arrive(&s.bar_dq_free);
      const size_t slot = dq_slot(p, b * p.Hq + c * p.group + hh, slot_pre, slot_lo, r);
      float* dst = p.dq_part + slot * (KV_SUB * HEAD_DIM) + (16 * g) * HEAD_DIM + rloc;
#pragma unroll
      for (int q = 0; q < 16; ++q) __stcg(dst + q * HEAD_DIM, v[q]);
      if (warp == SM_WARP0 && lane == 0) p.dq_flag[slot] = 1;
      return true;
    };
    int flo, fhi;
    full_range_kv(p.mask_kind, p.window, Lq, Lk, k0, &flo, &fhi);
    int prev_r = 0, prev_hh = 0;
    for (int n = 0; ok && n < N; ++n) {
      const int st = n % NST;
      // ---- P^T(n)
      if (!mbar_wait(smem_u32(&s.bar_s_full), n & 1, wc, TAG_S_FULL) ||
          !mbar_wait(smem_u32(&s.bar_q_full[st]), (n / NST) & 1, wc, TAG_Q_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[16];
      tmem_ld16(lane_base + COL_S + 16 * g, sv);
      const int r = s.step_r[st], hh = s.step_hh[st];
      const bool full = r >= flo && r <= fhi;
      uint32_t vis;
      if (full) {
        vis = 0xffffu;
      } else if (blk_regions) {
        vis = ((s.step_vis[st] >> (4 * sp + g)) & 1u) && j < Lk
                  ? bit_range(0, Lq - 1 - (r * KV_SUB + 16 * g))
                  : 0u;
      } else {
        vis = vis_key_row(p, b * p.Hq + c * p.group + hh, j, r * KV_SUB + 16 * g, Lq, Lk);
      }
      float lv[16];
      load16_shared(&s.nlse2[st][16 * g], lv);
      tmem_wait_ld_regs(sv);
      float pv[16];
      kv_write_p<BF16, false>(lane_base + COL_S + 16 * g, sv, lv, full, vis, p.scale_log2, pv);
      warp_arrive(&s.bar_p_full);

      // ---- the previous step's dQ partial (its completion also frees the
      // shared-memory dS^T tile for this step's)
      if (n >= 1 && !drain(n - 1, prev_r, prev_hh)) {
        ok = false;
        break;
      }

      // ---- dS^T(n) = P^T(n) (dP^T(n) - Delta), to TMEM and shared memory
      float dl[16];
      load16_shared(&s.delta[st][16 * g], dl);
      if (!mbar_wait(smem_u32(&s.bar_dp_full), n & 1, wc, TAG_DP_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float dp[16];
      tmem_ld16(lane_base + COL_DP + 16 * g, dp);
      tmem_wait_ld_regs(dp);
      uint32_t pk[8];
      kv_write_ds<BF16, false>(lane_base + COL_DP + 16 * g, pv, dp, dl, pk);
      // key row rloc, queries 16 g .. 16 g + 15: two 16-byte chunks of the
      // 128-byte row, 128B-swizzled (chunk index xor row % 8)
      uint8_t* row = s.dS + rloc * 128;
      *reinterpret_cast<uint4*>(row + (((2 * g) ^ (rloc & 7)) << 4)) =
          make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4*>(row + (((2 * g + 1) ^ (rloc & 7)) << 4)) =
          make_uint4(pk[4], pk[5], pk[6], pk[7]);
      // the dQ^T MMA reads the tile through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      warp_arrive(&s.bar_ds_full);
      prev_r = r;
      prev_hh = hh;
    }
    if (ok && N > 0) ok = drain(N - 1, prev_r, prev_hh);
    // ---------------------------------------------------------- epilogue
    bool have = ok && N > 0;
    if (have) have = mbar_wait(smem_u32(&s.bar_acc_full), 0, wc, TAG_ACC);
    tc_fence_after();
    named_bar_sync(1, 32 * SM_WARPS);
    const int r0 = k0 + sp * 32;
    const int nvalid = min(32, p.Skv - r0);
    uint8_t* stage = s.Q[0] + (warp - SM_WARP0) * 2048;
    const bool staged = __all_sync(0xffffffffu, have || (ok && N == 0));
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
      uint16_t* base = which ? dk : dv;
      uint16_t* orow = base + ((size_t)bc * p.Skv + r0) * HEAD_DIM + 32 * g;
      if (!staged) {
        warp_zero_rows(orow, 32, nvalid);
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
      warp_store_rows32(stage, pk, orow, nvalid);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// One block per (query sub-tile r, b * Hq + h): sums the written dQ partials
// of the sub-tile over key tiles in ascending order, scales, rounds and
// writes its KV_SUB rows (zeros for rows no key tile reached, and for every
// row after a device wait of the call ran out).
template <bool BF16>
__global__ void __launch_bounds__(256)
k_dq_reduce(const AttnParams p, uint16_t* __restrict__ dq) {
  __shared__ long long part[8];
  grid_dependency_wait();
  const int r = blockIdx.x, bh = blockIdx.y;
  const int nKT = (p.Skv + KV_TILE - 1) / KV_TILE;
  // key tiles that can meet this sub-tile, and the slots of the head before
  // the first of them
  int tlo = 0, thi = nKT - 1;
  if (p.mask_kind != MK_BLOCK)
    partner_range(p.mask_kind, p.window, true, r * KV_SUB, min(r * KV_SUB + KV_SUB, p.Sq), KV_TILE,
                  p.Skv, &tlo, &thi);
  long long pre = slots_before_share(p, tlo, threadIdx.x, blockDim.x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = pre;
  __syncthreads();
  pre = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) pre += part[w];
  const bool failed = p.status->code != 0;
  // thread -> (row q of the sub-tile, 32 consecutive head dims)
  const int q = threadIdx.x >> 2, d0 = (threadIdx.x & 3) * 32;
  float acc[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) acc[e] = 0.f;
  for (int t = tlo; t <= thi && !failed; ++t) {
    int lo;
    const int cnt = kv_tile_range_full(p.mask_kind, p.window, p.Sq, p.Skv, t, &lo);
    if (r >= lo && r < lo + cnt) {
      const size_t slot = dq_slot(p, bh, pre, lo, r);
      if (p.dq_flag[slot]) {
        const float4* src = reinterpret_cast<const float4*>(p.dq_part + slot * (KV_SUB * HEAD_DIM) +
                                                            q * HEAD_DIM + d0);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 v = __ldcs(src + e);
          acc[4 * e] += v.x;
          acc[4 * e + 1] += v.y;
          acc[4 * e + 2] += v.z;
          acc[4 * e + 3] += v.w;
        }
      }
    }
    pre += cnt;
  }
  const int row = r * KV_SUB + q;
  if (row >= p.Sq) return;
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) pk[e] = pack2<BF16>(acc[2 * e] * p.scale, acc[2 * e + 1] * p.scale);
  uint4* out = reinterpret_cast<uint4*>(dq + ((size_t)bh * p.Sq + row) * HEAD_DIM + d0);
#pragma unroll
  for (int e = 0; e < 4; ++e)
    out[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
}

cudaError_t launch_dkdvq(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                         const CUtensorMap& tdO, const CUtensorMap& tK, const CUtensorMap& tV,
                         void* dk, void* dv, cudaStream_t st) {
  const auto kern = bf16 ? k_dkdvq<true> : k_dkdvq<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)fused_side::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int nKT = (p.Skv + KV_TILE - 1) / KV_TILE;
  // programmatic serialization behind the preprocess kernel (block-mask CTAs
  // wait for it before they read the select tables)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nKT * p.B * p.Hkv));
  cfg.blockDim = dim3(fused_side::NUM_THREADS);
  cfg.dynamicSmemBytes = fused_side::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tQ, tdO, tK, tV, (uint16_t*)dk, (uint16_t*)dv, p);
}

cudaError_t launch_dq_reduce(bool bf16, const AttnParams& p, void* dq, cudaStream_t st) {
  const auto kern = bf16 ? k_dq_reduce<true> : k_dq_reduce<false>;
  // programmatic serialization: the blocks start as the key-stationary grid
  // drains and wait (griddepcontrol.wait) for its completion
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.nQT_k, (unsigned)(p.B * p.Hq));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, (uint16_t*)dq);
}

}  // namespace mab
