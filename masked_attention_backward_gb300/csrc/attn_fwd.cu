// attn_fwd.cu -- forward kernel producing O and LSE (the inputs of the
// backward), query-stationary on tcgen05 / TMEM, fed by TMA.
//
// One CTA per (b, query head, Q_TILE query rows); two passes over the same
// active key sub-tiles t (Q_SUB rows):
//   pass A: S = Q K_t^T, running max / sum per row in the log2 domain,
//           seeded with the sink logit (which joins only the denominator);
//   pass B: S again, P = exp2(S * scale*log2e - lse2) exactly, O += P V_t.
// No rescaling of O is ever needed because pass B knows the final LSE.
//
// Sources: tilelang-ascend PR #1 "Add GQA Sink Backward BHSD", Summary
// (online softmax with an attention sink and a sliding window);
// cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook, precision
// notes (a row that sees no key gets zeros).
//
// Warp roles (320 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs (one thread), warps 2..9 are two groups of four warps that
// each own 32 of the 64 key columns of a sub-tile for all 128 rows.
#include <math.h>

#include "tiles.cuh"

namespace mab {

namespace fwd_side {

constexpr int STAGES = 3;   // K/V ring depth
constexpr int NBUF = 3;     // S/dP buffers in TMEM
constexpr int COL_ACC = 0;  // O accumulator: 128 fp32 columns
constexpr int COL_S = 128;  // buffer b: S at COL_S + 128 b
constexpr int NUM_THREADS = 320;

struct __align__(1024) Smem {
  uint8_t Q[2 * Q_TILE * 128];          // two 64-column chunks, 128B swizzle
  uint8_t K[STAGES][2 * Q_SUB * 128];
  uint8_t V[STAGES][2 * Q_SUB * 128];
  float ml[2][Q_TILE][2];               // per-group (max, sum) per row
  uint64_t bar_q_full;
  uint64_t bar_kv_full[STAGES];
  uint64_t bar_kv_empty[STAGES];
  uint64_t bar_s_full[NBUF];
  uint64_t bar_p_full[NBUF];
  uint64_t bar_s_free[NBUF];
  uint64_t bar_acc_full;
  uint64_t bar_ml;
  uint64_t bar_drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;

// Wait tags recorded in the status word when a wait runs out.
enum { TAG_Q = 0x101, TAG_KV_EMPTY, TAG_KV_FULL, TAG_S_FREE, TAG_P_FULL, TAG_S_FULL, TAG_ACC,
       TAG_ML, TAG_DRAIN };

}  // namespace fwd_side

template <bool BF16>
__global__ void __launch_bounds__(fwd_side::NUM_THREADS, 1)
k_attn_fwd(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tK,
           const __grid_constant__ CUtensorMap tV, uint16_t* __restrict__ out,
           const AttnParams p) {
  using namespace fwd_side;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = p.B * p.Hq;
  const int qt = p.nQT_q - 1 - (int)(blockIdx.x / BH);  // longest causal rows first
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int kvh = b * p.Hkv + h / p.group;
  const int q0 = qt * Q_TILE;
  QWalk walk;
  walk.init(p, bh, qt);
  const int N = walk.cnt;
  const int NT = 2 * N;  // pass A, then pass B
  WaitCtx wc{p.status, &s.abort_flag, p.timeout_ns};

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar_q_full), 1);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.bar_kv_full[i]), 1);
      mbar_init(smem_u32(&s.bar_kv_empty[i]), 1);
    }
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_p_full[i]), 8);
      mbar_init(smem_u32(&s.bar_s_free[i]), 1);
    }
    mbar_init(smem_u32(&s.bar_acc_full), 1);
    mbar_init(smem_u32(&s.bar_ml), 256);
    mbar_init(smem_u32(&s.bar_drain), 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&tQ);
      tma_prefetch_desc(&tK);
      tma_prefetch_desc(&tV);
      const uint32_t qbar = smem_u32(&s.bar_q_full);
      mbar_arrive_expect_tx(qbar, 2 * Q_TILE * 128);
      tma_load_3d(smem_u32(s.Q), &tQ, 0, q0, bh, qbar);
      tma_load_3d(smem_u32(s.Q + Q_TILE * 128), &tQ, 64, q0, bh, qbar);
      for (int n = 0; n < NT; ++n) {
        const int st = n % STAGES;
        if (n >= STAGES &&
            !mbar_wait(smem_u32(&s.bar_kv_empty[st]), ((n / STAGES) - 1) & 1, wc, TAG_KV_EMPTY))
          break;
        const int t = walk.tile(n >= N ? n - N : n);
        const bool loadV = n >= N;  // pass A needs K only
        const uint32_t fb = smem_u32(&s.bar_kv_full[st]);
        mbar_arrive_expect_tx(fb, loadV ? 4 * Q_SUB * 128 : 2 * Q_SUB * 128);
        tma_load_3d(smem_u32(s.K[st]), &tK, 0, t * Q_SUB, kvh, fb);
        tma_load_3d(smem_u32(s.K[st] + Q_SUB * 128), &tK, 64, t * Q_SUB, kvh, fb);
        if (loadV) {
          tma_load_3d(smem_u32(s.V[st]), &tV, 0, t * Q_SUB, kvh, fb);
          tma_load_3d(smem_u32(s.V[st] + Q_SUB * 128), &tV, 64, t * Q_SUB, kvh, fb);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_f16(BF16, Q_TILE, Q_SUB, false, false);
      constexpr uint32_t ID_ACC = idesc_f16(BF16, Q_TILE, HEAD_DIM, false, true);
      const uint32_t sQ = smem_u32(s.Q);
      auto consume = [&](int m) -> bool {
        const int bf = m % NBUF, st = m % STAGES;
        if (!mbar_wait(smem_u32(&s.bar_p_full[bf]), (m / NBUF) & 1, wc, TAG_P_FULL)) return false;
        tc_fence_after();
        if (m >= N) {  // pass B: O += P V
          const uint32_t colS = tbase + COL_S + bf * 128;
          const uint32_t bop = smem_u32(s.V[st]);
#pragma unroll
          for (int kk = 0; kk < Q_SUB / 16; ++kk) {
            const uint32_t a_tmem = colS + 32 * (kk >> 1) + 8 * (kk & 1);
            mma_ts(tbase + COL_ACC, a_tmem, sdesc_sw128(bop + kk * 2048, Q_SUB * 128, 1024), ID_ACC,
                   (m > N || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(smem_u32(&s.bar_kv_empty[st]));
        mma_commit(smem_u32(&s.bar_s_free[bf]));
        return true;
      };
      bool ok = mbar_wait(smem_u32(&s.bar_q_full), 0, wc, TAG_Q);
      tc_fence_after();
      for (int n = 0; ok && n < NT; ++n) {
        const int st = n % STAGES, bf = n % NBUF;
        if (!mbar_wait(smem_u32(&s.bar_kv_full[st]), (n / STAGES) & 1, wc, TAG_KV_FULL)) {
          ok = false;
          break;
        }
        if (n >= NBUF &&
            !mbar_wait(smem_u32(&s.bar_s_free[bf]), ((n / NBUF) - 1) & 1, wc, TAG_S_FREE)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t colS = tbase + COL_S + bf * 128;
        const uint32_t sK = smem_u32(s.K[st]), sV = smem_u32(s.V[st]);
#pragma unroll
        for (int kk = 0; kk < HEAD_DIM / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * (Q_TILE * 128) + (kk & 3) * 32;
          const uint32_t bo = (kk >> 2) * (Q_SUB * 128) + (kk & 3) * 32;
          mma_ss(colS, sdesc_sw128(sQ + ao, 16, 1024), sdesc_sw128(sK + bo, 16, 1024), ID_S,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&s.bar_s_full[bf]));
        if (n >= 1 && !consume(n - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && NT >= 1) ok = consume(NT - 1);
      mma_commit(smem_u32(&s.bar_acc_full));
      mma_commit(smem_u32(&s.bar_drain));
      mbar_wait(smem_u32(&s.bar_drain), 0, wc, TAG_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int sp = warp & 3, g = (warp - 2) >> 2;
    const int rloc = sp * 32 + lane;
    const int i = q0 + rloc;
    const uint32_t lane_base = tbase + ((uint32_t)(sp * 32) << 16);
    float lse2_i = 0.f;
    bool ok = true;
    {
      // pass A: running max / sum in the log2 domain
      float m_run = -INFINITY, l_run = 0.f;
      if (g == 0 && p.sink) {
        m_run = p.sink[h] * LOG2E;
        l_run = 1.f;
      }
      for (int n = 0; n < N; ++n) {
        const int bf = n % NBUF;
        if (!mbar_wait(smem_u32(&s.bar_s_full[bf]), (n / NBUF) & 1, wc, TAG_S_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int t = walk.tile(n);
        const uint32_t vis = vis_query_row(p, bh, i, t * Q_SUB + 32 * g);
        float sv[32];
        tmem_ld32(lane_base + COL_S + bf * 128 + 32 * g, sv);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_p_full[bf]));
        float mx = m_run;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          sv[c] = ((vis >> c) & 1u) ? sv[c] * p.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sv[c]);
        }
        if (mx != -INFINITY) {
          float acc = l_run * fast_exp2(m_run - mx);
#pragma unroll
          for (int c = 0; c < 32; ++c) acc += fast_exp2(sv[c] - mx);
          l_run = acc;
          m_run = mx;
        }
      }
      // combine the two column groups of each row
      s.ml[g][rloc][0] = m_run;
      s.ml[g][rloc][1] = l_run;
      mbar_arrive(smem_u32(&s.bar_ml));
      if (!mbar_wait(smem_u32(&s.bar_ml), 0, wc, TAG_ML)) ok = false;
      {
        const float m0 = s.ml[0][rloc][0], l0 = s.ml[0][rloc][1];
        const float m1 = s.ml[1][rloc][0], l1 = s.ml[1][rloc][1];
        const float m = fmaxf(m0, m1);
        float l = 0.f;
        if (m != -INFINITY) l = l0 * fast_exp2(m0 - m) + l1 * fast_exp2(m1 - m);
        lse2_i = (l > 0.f) ? m + log2f(l) : INFINITY;
        if (g == 0 && i < p.Sq) p.lse_out[(size_t)bh * p.Sq + i] = lse2_i * 0.6931471805599453f;
      }
      // pass B: exact probabilities into TMEM for O += P V
      for (int n = N; ok && n < 2 * N; ++n) {
        const int bf = n % NBUF;
        if (!mbar_wait(smem_u32(&s.bar_s_full[bf]), (n / NBUF) & 1, wc, TAG_S_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int t = walk.tile(n - N);
        const uint32_t vis = vis_query_row(p, bh, i, t * Q_SUB + 32 * g);
        const uint32_t col = COL_S + bf * 128 + 32 * g;
        float sv[32];
        tmem_ld32(lane_base + col, sv);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float p0 = fast_exp2(fmaf(sv[2 * c], p.scale_log2, -lse2_i));
          float p1 = fast_exp2(fmaf(sv[2 * c + 1], p.scale_log2, -lse2_i));
          p0 = ((vis >> (2 * c)) & 1u) ? p0 : 0.f;
          p1 = ((vis >> (2 * c + 1)) & 1u) ? p1 : 0.f;
          pk[c] = pack2<BF16>(p0, p1);
        }
        tmem_st16(lane_base + col, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_p_full[bf]));
      }
    }
    // ---------------------------------------------------------- epilogue
    // Columns [64 g, 64 g + 64) of the accumulator, one row per lane.
    uint32_t pk[32];
    bool have = ok && N > 0;
    if (have) have = mbar_wait(smem_u32(&s.bar_acc_full), 0, wc, TAG_ACC);
    tc_fence_after();
    if (have) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[32];
        tmem_ld32(lane_base + COL_ACC + 64 * g + 32 * half, v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[16 * half + c] = pack2<BF16>(v[2 * c], v[2 * c + 1]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) pk[c] = 0u;
    }
    // the Q tile is dead once the accumulator is complete (or there was no
    // work): make sure its TMA load has landed before reusing it as staging
    if (mbar_wait(smem_u32(&s.bar_q_full), 0, wc, TAG_Q)) {
      uint8_t* stage = s.Q + (warp - 2) * 4096;
      const int r0 = q0 + sp * 32;
      uint16_t* orow = out + ((size_t)bh * p.Sq + r0) * HEAD_DIM + 64 * g;
      warp_store_rows(stage, pk, orow, min(32, p.Sq - r0));
    }
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
  auto kern = bf16 ? k_attn_fwd<true> : k_attn_fwd<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)fwd_side::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(p.nQT_q * p.B * p.Hq));
  kern<<<grid, fwd_side::NUM_THREADS, fwd_side::SMEM_BYTES, st>>>(tQ, tK, tV, (uint16_t*)o, p);
  return cudaGetLastError();
}

}  // namespace mab
