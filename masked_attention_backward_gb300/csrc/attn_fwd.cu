// attn_fwd.cu -- forward kernel producing O and LSE (the inputs of the
// backward), query-stationary on tcgen05 / TMEM, fed by TMA.
//
// Work unit: (b, query head h, Q_TILE query rows).  Q is loaded once and
// copied into TMEM, where it is the A operand of every S = Q K_t^T.  One pass
// over the active key sub-tiles t (Q_SUB rows) with an online softmax:
//   S   = Q K_t^T                                  (A = Q from TMEM, fp32 in TMEM)
//   M   = max(M, rowmax(S) * scale*log2e)          (only when it grows by more
//                                                   than 8; O and l rescaled then)
//   P   = exp2(S * scale*log2e - M),  l += rowsum(P)
//   O  += P V_t                                    (A = P packed in TMEM)
// and at the end O / l and LSE = (M + log2 l) ln 2.  The sink logit seeds M
// and adds exp2(sink log2e - M) to l: it joins the denominator only.
//
// Sources: tilelang-ascend PR #1 "Add GQA Sink Backward BHSD", Summary
// (online softmax with an attention sink and a sliding window);
// cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook, precision
// notes (a row that sees no key gets zeros).
//
// M only moves when a row's maximum exceeds it by more than 8 (log2 domain),
// so P stays below 2^8; in between P is taken against the stale M, which is
// exact up to rounding because the same M scales O and l.  A rescale
// multiplies the row's O and l by exp2(M_old - M_new) once the previous
// O += P V into that accumulator has completed; a row that has seen no key
// yet (O = 0, l = 0) just takes the new M.
//
// Two groups of softmax warps take alternate sub-tiles of a unit (group
// n % 2 takes step n), each with its own M, l and O accumulator, so a group
// has two steps' worth of tensor work to hide one step of softmax, and no
// per-step exchange between warps is needed.  At the end of the unit the two
// groups swap (M, l) per row through shared memory and each writes half of
//   O = (O_0 exp2(M_0 - M) + O_1 exp2(M_1 - M)) / l,   M = max(M_0, M_1).
//
// Persistent: one CTA per SM.  Units are numbered heaviest causal rows first;
// CTA b starts with unit b and then claims the next unit from a global
// counter when it starts loading one.  The producer publishes each claimed
// unit (or -1 when none is left) with its Q load, and loads the next unit's Q
// only once every other warp has taken the current one (unit_free), so no
// per-unit barrier can run two phases ahead of a warp that waits on it.  The
// K / V ring, the S buffers and their barrier phases continue across units
// (counted by one step counter m).  The epilogue of unit j overlaps the first
// S MMAs of unit j + 1 and meets its first O MMA at acc_empty.
//
// TMEM columns (512): O accumulators of groups 0 and 1 [0,128) and [128,256),
// Q as 16-bit pairs [256,320), three S buffers of 64 fp32 columns at
// 320 + 64 b.  The group's warp of a row quarter packs the 64 P values of its
// rows over the first 32 columns of the buffer, so the 16 keys of MMA K-step
// kk sit at buffer column 8 kk.
//
// Warp roles (352 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues S, warp 2 issues O += P V (whole warps, one elected lane); warps
// 3..10 are the softmax warps: warp (sp, grp) with sp = warp % 4 owns TMEM
// lanes 32 sp .. 32 sp + 31 (query rows), grp = (warp - 3) / 4.
#include <math.h>

#include "tiles.cuh"

namespace mab {

namespace fwd_side {

constexpr int STAGES = 5;        // K/V ring depth
constexpr int NBUF = 3;          // S / P buffers
constexpr int COL_O = 0;         // O accumulator of group g at COL_O + 128 g
constexpr int COL_QA = 256;      // Q as the A operand, 64 columns of 16-bit pairs
constexpr int COL_S = 320;       // S buffer b at COL_S + 64 b
constexpr int SM_WARP0 = 3;      // first softmax warp
constexpr int SM_WARPS = 8;      // softmax warps, two groups of four
constexpr int NUM_THREADS = 32 * (SM_WARP0 + SM_WARPS);
constexpr float RESCALE_LOG2 = 8.f;  // M moves when a row maximum exceeds it by this

struct __align__(1024) Smem {
  uint8_t Q[2 * Q_TILE * 128];  // two 64-column chunks, 128B swizzle; once copied
                                // into TMEM, the epilogue staging (4 KB per warp)
  uint8_t K[STAGES][2 * Q_SUB * 128];
  uint8_t V[STAGES][2 * Q_SUB * 128];
  float xml[2][2][Q_TILE][2];   // [unit parity][group][row]: (M, l) at the unit's end
  int step_t[STAGES];           // key sub-tile of the step in the stage
  int unit;                     // unit of the latest Q load, -1: none left
  uint64_t bar_q_full;          // Q of the unit landed in shared memory
  uint64_t bar_qa_full;         // Q copied into TMEM (all softmax warps)
  uint64_t bar_kv_full[STAGES];
  uint64_t bar_kv_empty[STAGES];
  uint64_t bar_s_full[2][2];    // [group][its step count parity]: S of the step complete
  uint64_t bar_p_full[NBUF];    // P of the buffer packed (the four warps of its group)
  uint64_t bar_p_free[NBUF];    // O += P V that read the buffer complete
  uint64_t bar_xml[4][2];       // [row quarter][unit parity]: both groups posted (M, l)
  uint64_t bar_acc_full;        // every O MMA of the unit complete
  uint64_t bar_acc_empty;       // the unit's accumulators read and stored (all softmax warps)
  uint64_t bar_unit_free;       // every other warp took the unit (and, softmax warps,
                                // stored the previous unit's epilogue)
  uint64_t bar_x_done[2];       // every MMA of the S / O warp complete
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;
static_assert(SMEM_BYTES <= 232448, "over the 227 KB of shared memory a CTA may use");

// Wait tags recorded in the status word when a wait runs out.
enum { TAG_Q = 0x101, TAG_QA, TAG_KV_EMPTY, TAG_KV_FULL, TAG_S_FULL, TAG_P_FULL, TAG_P_FREE,
       TAG_ACC, TAG_ACC_EMPTY, TAG_UNIT_FREE, TAG_XML, TAG_X_DONE };

// Position in a ring of NS slots and the parity of the slot's current use
// (kept as counters: NS need not be a power of two).
template <int NS>
struct Cyc {
  int i = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    if (++i == NS) {
      i = 0;
      ph ^= 1u;
    }
  }
};

// Coordinates of work unit u: heaviest causal query tiles first.
struct FwdUnit {
  int bh, q0, kvh, h, Lq, Lk;  // Lq, Lk: valid rows and keys of the batch
  QWalk walk;
  __device__ __forceinline__ void init(const AttnParams& p, int u) {
    const int BH = p.B * p.Hq;
    const int qt = p.nQT_q - 1 - u / BH;
    bh = u % BH;
    h = bh % p.Hq;
    const int b = bh / p.Hq;
    kvh = b * p.Hkv + h / p.group;
    q0 = qt * Q_TILE;
    Lq = len_q(p, b);
    Lk = len_k(p, b);
    walk.init(p, bh, qt, Lq, Lk);
  }
};

// What the epilogue of a finished unit needs of it.
struct FwdDone {
  int bh, q0, cnt, Lq;
};

}  // namespace fwd_side

// PACKED: the token-major layout with cumulative sequence offsets (the BHSD
// instance keeps its plain row addressing).
template <bool BF16, bool PACKED>
__global__ void __launch_bounds__(fwd_side::NUM_THREADS, 1)
k_attn_fwd(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tK,
           const __grid_constant__ CUtensorMap tV, uint16_t* __restrict__ out,
           const AttnParams p) {
  using namespace fwd_side;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int U = p.nQT_q * p.B * p.Hq;
  WaitCtx wc{p.status, &s.abort_flag, p.timeout_ns};

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar_q_full), 1);
    mbar_init(smem_u32(&s.bar_qa_full), SM_WARPS);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.bar_kv_full[i]), 1);
      mbar_init(smem_u32(&s.bar_kv_empty[i]), 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i >> 1][i & 1]), 1);
      mbar_init(smem_u32(&s.bar_xml[i][0]), 2);
      mbar_init(smem_u32(&s.bar_xml[i][1]), 2);
    }
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(smem_u32(&s.bar_p_full[i]), SM_WARPS / 2);
      mbar_init(smem_u32(&s.bar_p_free[i]), 1);
    }
    mbar_init(smem_u32(&s.bar_acc_full), 1);
    mbar_init(smem_u32(&s.bar_acc_empty), SM_WARPS);
    mbar_init(smem_u32(&s.bar_unit_free), SM_WARPS + 2);
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&s.bar_x_done[i]), 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !p.test_no_loads) {
      tma_prefetch_desc(&tQ);
      tma_prefetch_desc(&tK);
      tma_prefetch_desc(&tV);
      bool ok = true;
      int m = 0;  // step counter across units
      int q_loaded = -1;  // last unit whose Q tile was loaded
      Cyc<STAGES> rg;
      const uint32_t qbar = smem_u32(&s.bar_q_full);
      for (int j = 0; ok; ++j) {
        // the Q tile and the unit slot are free once every other warp has
        // taken the previous unit (the softmax warps: copied its Q into TMEM
        // and stored the epilogue before it, staged in the Q tile)
        if (j >= 1 && !mbar_wait(smem_u32(&s.bar_unit_free), (j - 1) & 1, wc, TAG_UNIT_FREE)) {
          ok = false;
          break;
        }
        int u = j == 0 ? (int)blockIdx.x : (int)(gridDim.x + atomicAdd(&p.status->next_unit, 1u));
        if (u >= U) u = -1;
        s.unit = u;  // published by the arrive on q_full
        if (u < 0) {
          mbar_arrive(qbar);
          break;
        }
        FwdUnit un;
        un.init(p, u);
        if (un.walk.cnt == 0) {
          // nothing to contract: the unit's rows only get O = 0, so its Q
          // tile is not loaded
          mbar_arrive(qbar);
        } else {
          const RowAddr qa =
              PACKED ? row_q(p, un.bh / p.Hq, un.h, un.q0) : RowAddr{un.q0, un.bh, 0, HEAD_DIM};
          mbar_arrive_expect_tx(qbar, 2 * Q_TILE * 128);
          tma_load_3d(smem_u32(s.Q), &tQ, 0, qa.c1, qa.c2, qbar);
          tma_load_3d(smem_u32(s.Q + Q_TILE * 128), &tQ, 64, qa.c1, qa.c2, qbar);
          q_loaded = j;
        }
        for (int n = 0; n < un.walk.cnt; ++n, ++m, rg.next()) {
          const int st = rg.i;
          if (m >= STAGES &&
              !mbar_wait(smem_u32(&s.bar_kv_empty[st]), rg.ph ^ 1u, wc, TAG_KV_EMPTY)) {
            ok = false;
            break;
          }
          const int t = un.walk.tile(n);
          s.step_t[st] = t;  // published by the arrive below together with the loads
          const uint32_t fb = smem_u32(&s.bar_kv_full[st]);
          const RowAddr ka = PACKED ? row_k(p, un.kvh / p.Hkv, un.kvh % p.Hkv, t * Q_SUB)
                                    : RowAddr{t * Q_SUB, un.kvh, 0, HEAD_DIM};
          mbar_arrive_expect_tx(fb, 4 * Q_SUB * 128);
          tma_load_3d(smem_u32(s.K[st]), &tK, 0, ka.c1, ka.c2, fb);
          tma_load_3d(smem_u32(s.K[st] + Q_SUB * 128), &tK, 64, ka.c1, ka.c2, fb);
          tma_load_3d(smem_u32(s.V[st]), &tV, 0, ka.c1, ka.c2, fb);
          tma_load_3d(smem_u32(s.V[st] + Q_SUB * 128), &tV, 64, ka.c1, ka.c2, fb);
        }
      }
      if (!ok) {
        // the CTA gave up: let the copies still in flight land before it exits
        if (q_loaded >= 0) mbar_drain(qbar, q_loaded & 1, wc.timeout_ns);
        for (int k = m > STAGES ? m - STAGES : 0; k < m; ++k)
          mbar_drain(smem_u32(&s.bar_kv_full[k % STAGES]), (k / STAGES) & 1, wc.timeout_ns);
      }
    }
  } else if (warp < SM_WARP0) {
    // ------------------------------------------------------------ MMA issuers (whole warps)
    bool ok = true;
    int m = 0;  // step counter across units
    Cyc<STAGES> rg;
    Cyc<NBUF> bc;
    if (warp == 1) {
      // S(m) = Q K^T into buffer m % NBUF (A = Q from TMEM, B = K tile, K-major)
      constexpr uint32_t ID_S = idesc_f16(BF16, Q_TILE, Q_SUB, false, false);
      int cnt0 = 0, cnt1 = 0;  // steps of each group so far
      for (int j = 0; ok; ++j) {
        if (!mbar_wait_warp(smem_u32(&s.bar_q_full), j & 1, wc, TAG_Q)) break;
        const int u = s.unit;
        if (u < 0) break;
        FwdUnit un;
        un.init(p, u);
        const int N = un.walk.cnt;
        ok = mbar_wait_warp(smem_u32(&s.bar_qa_full), j & 1, wc, TAG_QA);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_unit_free));
        for (int n = 0; ok && n < N; ++n, ++m, rg.next(), bc.next()) {
          const int st = rg.i, bf = bc.i, grp = n & 1;
          ok = mbar_wait_warp(smem_u32(&s.bar_kv_full[st]), rg.ph, wc, TAG_KV_FULL);
          // the buffer held P(m - NBUF), read by O += P V
          if (ok && m >= NBUF)
            ok = mbar_wait_warp(smem_u32(&s.bar_p_free[bf]), bc.ph ^ 1u, wc, TAG_P_FREE);
          if (!ok) break;
          tc_fence_after();
          const uint64_t bK = sdesc_sw128(smem_u32(s.K[st]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < HEAD_DIM / 16; ++kk)
            mma_ts_w(tbase + COL_S + 64 * bf, tbase + COL_QA + 8 * kk,
                     bK + (uint64_t)(((kk >> 2) * (Q_SUB * 128) + (kk & 3) * 32) >> 4), ID_S,
                     kk > 0 ? 1u : 0u);
          const int c = grp ? cnt1 : cnt0;
          mma_commit_w(smem_u32(&s.bar_s_full[grp][c & 1]));
          if (grp) ++cnt1; else ++cnt0;
        }
      }
    } else {
      // O_{n % 2} += P(m) V (A = P packed in buffer m % NBUF, B = V tile, MN-major)
      constexpr uint32_t ID_O = idesc_f16(BF16, Q_TILE, HEAD_DIM, false, true);
      for (int j = 0; ok; ++j) {
        // the unit's first accumulations overwrite the accumulators: the
        // softmax warps must have read the previous unit's
        if (j >= 1 &&
            !mbar_wait_warp(smem_u32(&s.bar_acc_empty), (j - 1) & 1, wc, TAG_ACC_EMPTY))
          break;
        if (!mbar_wait_warp(smem_u32(&s.bar_q_full), j & 1, wc, TAG_Q)) break;
        const int u = s.unit;
        if (u < 0) break;
        FwdUnit un;
        un.init(p, u);
        const int N = un.walk.cnt;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_unit_free));
        for (int n = 0; ok && n < N; ++n, ++m, rg.next(), bc.next()) {
          const int st = rg.i, bf = bc.i;
          ok = mbar_wait_warp(smem_u32(&s.bar_p_full[bf]), bc.ph, wc, TAG_P_FULL);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a = tbase + COL_S + 64 * bf;
          const uint64_t bV = sdesc_sw128(smem_u32(s.V[st]), Q_SUB * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < Q_SUB / 16; ++kk)
            mma_ts_w(tbase + COL_O + 128 * (n & 1), a + 8 * kk,
                     bV + (uint64_t)((kk * 2048) >> 4), ID_O, (n >= 2 || kk > 0) ? 1u : 0u);
          // S(m) completed before the softmax warps could signal step m, so
          // this commit also frees the K / V stage
          mma_commit_w(smem_u32(&s.bar_kv_empty[st]));
          mma_commit_w(smem_u32(&s.bar_p_free[bf]));
        }
        if (ok) mma_commit_w(smem_u32(&s.bar_acc_full));  // the unit's accumulators are complete
      }
    }
    // this warp's MMAs must be complete before TMEM is freed (also when the
    // CTA gave up, hence a wait that ignores the abort flag)
    const uint32_t done = smem_u32(&s.bar_x_done[warp - 1]);
    mma_commit_w(done);
    mbar_drain_warp(done, 0, wc.timeout_ns);
  } else {
    // ------------------------------------------------------------ softmax warps
    const int sp = warp & 3, grp = (warp - SM_WARP0) >> 2;
    const int rloc = sp * 32 + lane;
    const uint32_t lane_base = tbase + ((uint32_t)(sp * 32) << 16);
    // the epilogue stages through the Q rows this warp itself copies
    uint8_t* stage = s.Q + grp * (Q_TILE * 128) + sp * 4096;
    // Combines both groups' accumulators of unit j into the unit's O columns
    // [64 grp, 64 grp + 64) of this warp's 32 rows (zeros when the unit had
    // no step) and its LSE, then releases the accumulators and the staging
    // space.  (M, l) of the own group come in; the other group's are taken
    // from shared memory.
    auto epilogue = [&](int j, const FwdDone& un, float M, float l, float sink2, bool ok) {
      s.xml[j & 1][grp][rloc][0] = M;
      s.xml[j & 1][grp][rloc][1] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_xml[sp][j & 1]));
      const int N = un.cnt;
      bool have = ok && N > 0;
      if (have) have = mbar_wait(smem_u32(&s.bar_xml[sp][j & 1]), (j >> 1) & 1, wc, TAG_XML);
      if (have) have = mbar_wait(smem_u32(&s.bar_acc_full), j & 1, wc, TAG_ACC);
      tc_fence_after();
      float w[2] = {0.f, 0.f};  // weights of O_0 and O_1, divided by l
      float lse = INFINITY;
      if (have) {
        const float Mo = s.xml[j & 1][grp ^ 1][rloc][0], lo = s.xml[j & 1][grp ^ 1][rloc][1];
        const float Mg[2] = {grp == 0 ? M : Mo, grp == 0 ? Mo : M};
        const float lg[2] = {grp == 0 ? l : lo, grp == 0 ? lo : l};
        const float Mx = fmaxf(Mg[0], Mg[1]);
        if (Mx > -INFINITY) {
          // group 1 has steps only when the unit has two or more; a group's
          // weight is zero when its row saw nothing (l = 0)
          const float e0 = lg[0] > 0.f ? fast_exp2(Mg[0] - Mx) : 0.f;
          const float e1 = (N >= 2 && lg[1] > 0.f) ? fast_exp2(Mg[1] - Mx) : 0.f;
          float lt = lg[0] * e0 + lg[1] * e1;
          if (sink2 > -INFINITY) lt += fast_exp2(sink2 - Mx);
          if (lt > 0.f) {
            const float inv = 1.f / lt;
            w[0] = e0 * inv;
            w[1] = e1 * inv;
            lse = (Mx + log2f(lt)) * 0.6931471805599453f;
          }
        }
      } else if (ok && sink2 > -INFINITY) {
        lse = sink2 * 0.6931471805599453f;  // no key at all: only the sink
      }
      uint32_t pk[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float acc[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) acc[c] = 0.f;
        if (have) {
#pragma unroll
          for (int gg = 0; gg < 2; ++gg) {
            if (__any_sync(0xffffffffu, w[gg] != 0.f)) {
              float v[32];
              tmem_ld32(lane_base + COL_O + 128 * gg + 64 * grp + 32 * half, v);
              tmem_wait_ld_regs(v);
#pragma unroll
              for (int c = 0; c < 32; ++c) acc[c] = fmaf(v[c], w[gg], acc[c]);
            }
          }
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[16 * half + c] = pack2<BF16>(acc[2 * c], acc[2 * c + 1]);
      }
      const int r0 = un.q0 + sp * 32;
      const int bq = un.bh / p.Hq, h = un.bh % p.Hq;
      const int nvalid = PACKED ? rows_to_store_q(p, bq, r0) : min(32, p.Sq - r0);
      if (r0 + lane >= un.Lq) lse = INFINITY;  // past the batch's length: outside the problem
      if (grp == 0 && lane < nvalid) {
        // lse: [B*Hq, Sq] in the BHSD layout, [Hq, total_q] in the packed one
        const size_t li = PACKED ? (size_t)h * p.total_q + packed_off(p.cu_q, bq, p.total_q) + r0 +
                                       lane
                                 : (size_t)un.bh * p.Sq + r0 + lane;
        p.lse_out[li] = lse;
      }
      const RowAddr oa =
          PACKED ? row_q(p, bq, h, r0)
                 : RowAddr{r0, un.bh, ((size_t)un.bh * p.Sq + r0) * HEAD_DIM, HEAD_DIM};
      uint16_t* orow = out + oa.elem + 64 * grp;
      if (!__all_sync(0xffffffffu, ok && (N == 0 || have))) {
        // the CTA gave up: a copy may still be landing in the Q tile, so the
        // zeros go straight to global memory
        warp_zero_rows(orow, 64, nvalid, oa.stride);
        return;
      }
      warp_store_rows(stage, pk, orow, nvalid, oa.stride);
      // the next TMA load into the Q tile comes after this warp's generic
      // accesses to it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_acc_empty));
    };
    bool ok = true;
    int m = 0;    // step counter across units
    int cnt = 0;  // steps of this group so far
    Cyc<STAGES> rg;
    Cyc<NBUF> bc;
    FwdDone prev{0, 0, 0, 0};
    float prev_M = -INFINITY, prev_l = 0.f, prev_sink2 = -INFINITY;
    int j = 0;
    for (; ok; ++j) {
      ok = mbar_wait(smem_u32(&s.bar_q_full), j & 1, wc, TAG_Q);
      const int u = ok ? s.unit : -1;
      if (u < 0) break;
      FwdUnit un;
      un.init(p, u);
      // Q rows into TMEM as 16-bit pairs (element 2c in the low half of
      // column c): this warp copies d columns 64 grp .. 64 grp + 63 of its
      // rows.  Every S MMA of the previous unit completed before its last
      // step was signalled, so the columns are free.
      {
        const uint8_t* src = s.Q + grp * (Q_TILE * 128) + rloc * 128;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(src + ((c ^ (rloc & 7)) << 4));
          w[4 * c] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        tmem_st32(lane_base + COL_QA + 32 * grp, w);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_qa_full));
      // the previous unit's epilogue overlaps this unit's first MMAs
      if (j >= 1) epilogue(j - 1, prev, prev_M, prev_l, prev_sink2, ok);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_unit_free));

      const int i = un.q0 + rloc;
      // this group's running maximum M (log2 domain), seeded with the sink,
      // and its row sum
      const float sink2 = p.sink ? p.sink[un.h] * LOG2E : -INFINITY;
      float M = sink2, l = 0.f;
      int flo, fhi;  // key sub-tiles that are entirely visible
      full_range_q(p.mask_kind, p.window, un.Lq, un.Lk, un.q0, &flo, &fhi);
      int last_bf = 0;       // buffer of this group's previous step of the unit
      uint32_t last_ph = 0;  // and the parity of its use
      for (int n = 0; ok && n < un.walk.cnt; ++n, ++m, rg.next(), bc.next()) {
        if ((n & 1) != grp) continue;
        const int st = rg.i, bf = bc.i;
        // s_full implies the stage's loads landed; waiting on kv_full as well
        // makes the step's tile index (written by the producer) visible
        if (!mbar_wait(smem_u32(&s.bar_s_full[grp][cnt & 1]), (cnt >> 1) & 1, wc, TAG_S_FULL) ||
            !mbar_wait(smem_u32(&s.bar_kv_full[st]), rg.ph, wc, TAG_KV_FULL)) {
          ok = false;
          break;
        }
        ++cnt;
        tc_fence_after();
        const uint32_t col = COL_S + 64 * bf;
        float sv[64];
        tmem_ld32(lane_base + col, *reinterpret_cast<float(*)[32]>(&sv[0]));
        tmem_ld32(lane_base + col + 32, *reinterpret_cast<float(*)[32]>(&sv[32]));
        const int t = s.step_t[st];
        // warp-uniform: the whole 128 x 64 sub-tile is visible
        const bool full = t >= flo && t <= fhi;
        const uint32_t vis0 =
            full ? 0xffffffffu : vis_query_row(p, un.bh, i, t * Q_SUB, un.Lq, un.Lk);
        const uint32_t vis1 =
            full ? 0xffffffffu : vis_query_row(p, un.bh, i, t * Q_SUB + 32, un.Lq, un.Lk);
        tmem_wait_ld_regs(sv);
        // row maximum of the visible raw logits (the scale is positive, so
        // it is applied once afterwards); eight partial maxima and sums keep
        // the dependency chains short
        float mp[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) mp[c] = -INFINITY;
        if (!full) {
          // invisible logits drop out of the maximum
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sv[c] = ((vis0 >> c) & 1u) ? sv[c] : -INFINITY;
            sv[32 + c] = ((vis1 >> c) & 1u) ? sv[32 + c] : -INFINITY;
          }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) mp[c & 7] = fmax3f(mp[c & 7], sv[2 * c], sv[2 * c + 1]);
        const float mx = fmax3f(fmax3f(mp[0], mp[1], mp[2]), fmax3f(mp[3], mp[4], mp[5]),
                                fmaxf(mp[6], mp[7]));
        const float mx2 = mx == -INFINITY ? -INFINITY : mx * p.scale_log2;
        // move M when the row maximum exceeds it by more than 8; a row that
        // has seen nothing yet (M = -inf, so O and l are still zero) just
        // takes the new value
        float alpha = 1.f;
        if (mx2 > M + RESCALE_LOG2) {
          if (M != -INFINITY) alpha = fast_exp2(M - mx2);
          M = mx2;
          l *= alpha;
        }
        // P = exp2(S scale log2e - M): an invisible logit (-inf here) gives 0;
        // a row with nothing visible keeps M = -inf and all its logits at
        // -inf, and the finite stand-in keeps -inf - (-inf) out
        const float Ms = M == -INFINITY ? 0.f : M;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-Ms, -Ms);
        uint32_t pk[32];
        float2 lp[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) lp[c] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 x = ffma2(make_float2(sv[2 * c], sv[2 * c + 1]), sc2, nm2);
          const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          lp[c & 3] = fadd2(lp[c & 3], pp);
          pk[c] = pack2<BF16>(pp.x, pp.y);
        }
        const float2 ls = fadd2(fadd2(lp[0], lp[1]), fadd2(lp[2], lp[3]));
        l += ls.x + ls.y;
        // rescale this group's O rows whose M moved, once the group's
        // previous O += P V of the unit has completed (the unit's first
        // accumulation of the group overwrites instead)
        if (n >= 2 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!mbar_wait(smem_u32(&s.bar_p_free[last_bf]), last_ph, wc, TAG_P_FREE)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t v[32];
            tmem_ld32(lane_base + COL_O + 128 * grp + 32 * q, reinterpret_cast<float(&)[32]>(v));
            tmem_wait_ld_regs(reinterpret_cast<float(&)[32]>(v));
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
            tmem_st32(lane_base + COL_O + 128 * grp + 32 * q, v);
          }
        }
        tmem_st32(lane_base + col, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_p_full[bf]));
        last_bf = bf;
        last_ph = bc.ph;
      }
      prev = FwdDone{un.bh, un.q0, un.walk.cnt, un.Lq};
      prev_M = M;
      prev_l = l;
      prev_sink2 = sink2;
    }
    if (j >= 1) epilogue(j - 1, prev, prev_M, prev_l, prev_sink2, ok);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

cudaError_t launch_fwd(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                       const CUtensorMap& tK, const CUtensorMap& tV, void* o, cudaStream_t st) {
  const bool packed = p.cu_q != nullptr;
  auto kern = bf16 ? (packed ? k_attn_fwd<true, true> : k_attn_fwd<true, false>)
                   : (packed ? k_attn_fwd<false, true> : k_attn_fwd<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)fwd_side::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int units = p.nQT_q * p.B * p.Hq;
  dim3 grid((unsigned)(units < sms ? units : sms));
  kern<<<grid, fwd_side::NUM_THREADS, fwd_side::SMEM_BYTES, st>>>(tQ, tK, tV, (uint16_t*)o, p);
  return cudaGetLastError();
}

}  // namespace mab
