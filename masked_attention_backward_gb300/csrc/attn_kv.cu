// attn_kv.cu -- key-stationary dK/dV kernel on tcgen05 / TMEM, fed by TMA.
//
// One CTA per (b, kv head c, KV_TILE key rows).  K and V of the tile are
// loaded once; K is copied into TMEM.  The CTA walks every query head of the
// GQA group and, for each, every active query sub-tile r of KV_SUB rows
// (closed-form range for causal / sliding / none, the key-major select table
// for block masks):
//   S^T  = K Q_r^T            (A = K from TMEM)
//   dP^T = V dO_r^T           (A = V from shared memory)
//   P^T  = exp2(S^T * scale*log2e - lse2_r),  dS^T = P^T (dP^T - Delta_r)
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
// TMEM columns (512): dV [0,128), dK [128,256), K as 16-bit pairs [256,320),
// two S^T buffers [320,384) and [384,448), dP^T [448,512).  Softmax group g
// owns query columns 32 g .. 32 g + 31 of a sub-tile, i.e. 32 fp32 columns of
// an S^T buffer; it packs P^T into the first 16 of them and dS^T into the
// last 16.  dS^T therefore does not occupy the dP^T buffer, which is free
// again as soon as the softmax warps have read it.
//
// MMA order per step n: dV(n), dK(n), dP(n+1), S(n+2).  S(n+2) overwrites the
// buffer that dV(n) / dK(n) read, and its wait for them is covered by dP(n+1)
// queued behind; dP(n+1) waits only on the softmax warps having read dP(n).
// Between dP(n+1) completing and dK(n+1) being needed lie S(n+2) and dV(n+1),
// and between S(n+2) completing and dV(n+2) lie three more groups, so the
// softmax work of a step is hidden behind the tensor pipe.
//
// Warp roles (320 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues the MMAs (whole warp, one elected lane), warps 2..9 are the softmax
// warps: warp (sp, g) owns TMEM lanes 32 sp .. 32 sp + 31 (key rows).
#include <math.h>

#include "tiles.cuh"

namespace mab {

namespace kv_side {

constexpr int STAGES = 4;      // Q/dO ring depth
constexpr int COL_DV = 0;
constexpr int COL_DK = 128;
constexpr int COL_KA = 256;    // K as the A operand (64 columns of 16-bit pairs)
constexpr int COL_ST = 320;    // S^T buffer b at COL_ST + 64 b
constexpr int COL_DPT = 448;   // dP^T
constexpr int NUM_THREADS = 320;

struct __align__(1024) Smem {
  uint8_t K[2 * KV_TILE * 128];  // dead once copied into TMEM: stages the output
  uint8_t V[2 * KV_TILE * 128];
  uint8_t Q[STAGES][2 * KV_SUB * 128];
  uint8_t dO[STAGES][2 * KV_SUB * 128];
  float lse2[STAGES][KV_SUB];
  float delta[STAGES][KV_SUB];
  uint64_t bar_kv_full;          // K, V landed
  uint64_t bar_ka_full;          // K copied into TMEM (8 softmax warps)
  uint64_t bar_q_full[STAGES];
  uint64_t bar_q_empty[STAGES];
  uint64_t bar_s_full[2];        // S^T of the buffer complete
  uint64_t bar_p_full[2];        // P^T of the buffer packed (8 warps)
  uint64_t bar_st_free[2];       // dV / dK MMAs that read the buffer complete
  uint64_t bar_dp_full;          // dP^T complete
  uint64_t bar_ds_full;          // dS^T packed, dP^T read (8 warps)
  uint64_t bar_acc_full;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;

enum { TAG_KV = 0x201, TAG_KA, TAG_Q_EMPTY, TAG_Q_FULL, TAG_ST_FREE, TAG_P_FULL, TAG_S_FULL,
       TAG_DP_FULL, TAG_DS_FULL, TAG_ACC };

}  // namespace kv_side

template <bool BF16>
__global__ void __launch_bounds__(kv_side::NUM_THREADS, 1)
k_dkdv(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tdO,
       const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV,
       uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, const AttnParams p) {
  using namespace kv_side;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BHkv = p.B * p.Hkv;
  const int t = (int)(blockIdx.x / BHkv);  // low key tiles (longest causal walks) first
  const int bc = (int)(blockIdx.x % BHkv);
  const int b = bc / p.Hkv, c = bc % p.Hkv;
  const int k0 = t * KV_TILE;
  KVWalk walk;
  walk.init(p, b, c, t);
  const int N = walk.total(p);
  WaitCtx wc{p.status, &s.abort_flag, p.timeout_ns};

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar_kv_full), 1);
    mbar_init(smem_u32(&s.bar_ka_full), 8);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.bar_q_full[i]), 1);
      mbar_init(smem_u32(&s.bar_q_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_p_full[i]), 8);
      mbar_init(smem_u32(&s.bar_st_free[i]), 1);
    }
    mbar_init(smem_u32(&s.bar_dp_full), 1);
    mbar_init(smem_u32(&s.bar_ds_full), 8);
    mbar_init(smem_u32(&s.bar_acc_full), 1);
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
      tma_prefetch_desc(&tdO);
      tma_prefetch_desc(&tK);
      tma_prefetch_desc(&tV);
      const uint32_t kvbar = smem_u32(&s.bar_kv_full);
      mbar_arrive_expect_tx(kvbar, 4 * KV_TILE * 128);
      tma_load_3d(smem_u32(s.K), &tK, 0, k0, bc, kvbar);
      tma_load_3d(smem_u32(s.K + KV_TILE * 128), &tK, 64, k0, bc, kvbar);
      tma_load_3d(smem_u32(s.V), &tV, 0, k0, bc, kvbar);
      tma_load_3d(smem_u32(s.V + KV_TILE * 128), &tV, 64, k0, bc, kvbar);
      KVCursor cur;
      cur.start(p, walk);
      for (int n = 0; n < N; ++n) {
        const int st = n % STAGES;
        if (n >= STAGES &&
            !mbar_wait(smem_u32(&s.bar_q_empty[st]), ((n / STAGES) - 1) & 1, wc, TAG_Q_EMPTY))
          break;
        const int r = walk.tile(p, cur.hh, cur.idx);
        const int bh = b * p.Hq + c * p.group + cur.hh;
        cur.next(p, walk);
        const uint32_t fb = smem_u32(&s.bar_q_full[st]);
        mbar_arrive_expect_tx(fb, 4 * KV_SUB * 128 + 2 * KV_SUB * 4);
        tma_load_3d(smem_u32(s.Q[st]), &tQ, 0, r * KV_SUB, bh, fb);
        tma_load_3d(smem_u32(s.Q[st] + KV_SUB * 128), &tQ, 64, r * KV_SUB, bh, fb);
        tma_load_3d(smem_u32(s.dO[st]), &tdO, 0, r * KV_SUB, bh, fb);
        tma_load_3d(smem_u32(s.dO[st] + KV_SUB * 128), &tdO, 64, r * KV_SUB, bh, fb);
        const size_t srow = (size_t)bh * p.Sq_pad + (size_t)r * KV_SUB;
        bulk_load(smem_u32(s.lse2[st]), p.lse2 + srow, KV_SUB * 4, fb);
        bulk_load(smem_u32(s.delta[st]), p.delta + srow, KV_SUB * 4, fb);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (whole warp)
    constexpr uint32_t ID_S = idesc_f16(BF16, KV_TILE, KV_SUB, false, false);
    constexpr uint32_t ID_ACC = idesc_f16(BF16, KV_TILE, HEAD_DIM, false, true);
    // S^T(m) = K Q^T into buffer m & 1 (A = K from TMEM, B = Q tile, K-major)
    auto issue_s = [&](int m) {
      const uint32_t d = tbase + COL_ST + 64 * (m & 1);
      const uint64_t bQ = sdesc_sw128(smem_u32(s.Q[m % STAGES]), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < HEAD_DIM / 16; ++kk)
        mma_ts_w(d, tbase + COL_KA + 8 * kk,
                 bQ + (uint64_t)(((kk >> 2) * (KV_SUB * 128) + (kk & 3) * 32) >> 4), ID_S,
                 kk > 0 ? 1u : 0u);
    };
    // dP^T(m) = V dO^T (A = V tile, B = dO tile, both K-major in shared memory)
    auto issue_dp = [&](int m) {
      const uint64_t aV = sdesc_sw128(smem_u32(s.V), 16, 1024);
      const uint64_t bO = sdesc_sw128(smem_u32(s.dO[m % STAGES]), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < HEAD_DIM / 16; ++kk)
        mma_ss_w(tbase + COL_DPT,
                 aV + (uint64_t)(((kk >> 2) * (KV_TILE * 128) + (kk & 3) * 32) >> 4),
                 bO + (uint64_t)(((kk >> 2) * (KV_SUB * 128) + (kk & 3) * 32) >> 4), ID_S,
                 kk > 0 ? 1u : 0u);
    };
    // dV += P^T(m) dO, dK += dS^T(m) Q (A from buffer m & 1, B MN-major)
    auto issue_acc = [&](int m, bool dkside) {
      const uint32_t a = tbase + COL_ST + 64 * (m & 1) + (dkside ? 16 : 0);
      const uint64_t bB = sdesc_sw128(smem_u32(dkside ? s.Q[m % STAGES] : s.dO[m % STAGES]),
                                      KV_SUB * 128, 1024);
#pragma unroll
      for (int kk = 0; kk < KV_SUB / 16; ++kk)
        mma_ts_w(tbase + (dkside ? COL_DK : COL_DV), a + 32 * (kk >> 1) + 8 * (kk & 1),
                 bB + (uint64_t)((kk * 2048) >> 4), ID_ACC, (m > 0 || kk > 0) ? 1u : 0u);
    };
    bool ok = true;
    if (N > 0) {
      ok = mbar_wait_warp(smem_u32(&s.bar_kv_full), 0, wc, TAG_KV) &&
           mbar_wait_warp(smem_u32(&s.bar_ka_full), 0, wc, TAG_KA) &&
           mbar_wait_warp(smem_u32(&s.bar_q_full[0]), 0, wc, TAG_Q_FULL);
      tc_fence_after();
      if (ok) {
        issue_s(0);
        mma_commit_w(smem_u32(&s.bar_s_full[0]));
        issue_dp(0);
        mma_commit_w(smem_u32(&s.bar_dp_full));
      }
      if (ok && N > 1) {
        ok = mbar_wait_warp(smem_u32(&s.bar_q_full[1 % STAGES]), 0, wc, TAG_Q_FULL);
        tc_fence_after();
        if (ok) {
          issue_s(1);
          mma_commit_w(smem_u32(&s.bar_s_full[1]));
        }
      }
    }
    for (int n = 0; ok && n < N; ++n) {
      const int bf = n & 1;
      ok = mbar_wait_warp(smem_u32(&s.bar_p_full[bf]), (n >> 1) & 1, wc, TAG_P_FULL);
      if (!ok) break;
      tc_fence_after();
      issue_acc(n, false);  // dV += P^T dO
      ok = mbar_wait_warp(smem_u32(&s.bar_ds_full), n & 1, wc, TAG_DS_FULL);
      if (!ok) break;
      tc_fence_after();
      issue_acc(n, true);   // dK += dS^T Q
      mma_commit_w(smem_u32(&s.bar_q_empty[n % STAGES]));
      mma_commit_w(smem_u32(&s.bar_st_free[bf]));
      if (n + 1 < N) {
        // the softmax warps have read dP^T(n) (ds_full); Q/dO of step n + 1
        // were waited for before S(n + 1)
        issue_dp(n + 1);
        mma_commit_w(smem_u32(&s.bar_dp_full));
      }
      const int m = n + 2;
      if (m < N) {
        ok = mbar_wait_warp(smem_u32(&s.bar_q_full[m % STAGES]), (m / STAGES) & 1, wc,
                            TAG_Q_FULL) &&
             mbar_wait_warp(smem_u32(&s.bar_st_free[bf]), (n >> 1) & 1, wc, TAG_ST_FREE);
        if (!ok) break;
        tc_fence_after();
        issue_s(m);  // overwrites P^T(n) / dS^T(n), which dV(n) / dK(n) have read
        mma_commit_w(smem_u32(&s.bar_s_full[bf]));
      }
    }
    // completes when every MMA issued above has (also on the abort path, so
    // that TMEM is idle before it is freed)
    mma_commit_w(smem_u32(&s.bar_acc_full));
    mbar_wait_warp(smem_u32(&s.bar_acc_full), 0, wc, TAG_ACC);
  } else {
    // ------------------------------------------------------------ softmax warps
    const int sp = warp & 3, g = (warp - 2) >> 2;
    const int rloc = sp * 32 + lane;
    const int j = k0 + rloc;
    const uint32_t lane_base = tbase + ((uint32_t)(sp * 32) << 16);
    bool ok = mbar_wait(smem_u32(&s.bar_kv_full), 0, wc, TAG_KV);
    if (ok) {
      // K rows into TMEM as 16-bit pairs (element 2c in the low half of column
      // c): this warp copies d columns 64 g .. 64 g + 63 of its rows.
      const uint8_t* src = s.K + g * (KV_TILE * 128) + rloc * 128;
      uint32_t w[32];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + ((cc ^ (rloc & 7)) << 4));
        w[4 * cc] = v.x;
        w[4 * cc + 1] = v.y;
        w[4 * cc + 2] = v.z;
        w[4 * cc + 3] = v.w;
      }
      tmem_st32(lane_base + COL_KA + 32 * g, w);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.bar_ka_full));

    KVCursor cur;
    cur.start(p, walk);
    for (int n = 0; ok && n < N; ++n) {
      const int bf = n & 1, st = n % STAGES;
      const uint32_t col = COL_ST + 64 * bf + 32 * g;
      // s_full implies the stage's loads landed; waiting on q_full as well
      // makes the bulk-copied lse2 / Delta rows visible to this thread
      if (!mbar_wait(smem_u32(&s.bar_s_full[bf]), (n >> 1) & 1, wc, TAG_S_FULL) ||
          !mbar_wait(smem_u32(&s.bar_q_full[st]), (n / STAGES) & 1, wc, TAG_Q_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int r = walk.tile(p, cur.hh, cur.idx);
      const int bh = b * p.Hq + c * p.group + cur.hh;
      cur.next(p, walk);
      const uint32_t vis = vis_key_row(p, bh, j, r * KV_SUB + 32 * g);
      float pv[32];
      {
        float sv[32];
        tmem_ld32(lane_base + col, sv);
        tmem_wait_ld();
        const float4* l4 = reinterpret_cast<const float4*>(&s.lse2[st][32 * g]);
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 L = l4[q];
          const float lv[4] = {L.x, L.y, L.z, L.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int cc = 4 * q + e;
            const float pe = fast_exp2(fmaf(sv[cc], p.scale_log2, -lv[e]));
            pv[cc] = ((vis >> cc) & 1u) ? pe : 0.f;
          }
          pk[2 * q] = pack2<BF16>(pv[4 * q], pv[4 * q + 1]);
          pk[2 * q + 1] = pack2<BF16>(pv[4 * q + 2], pv[4 * q + 3]);
        }
        tmem_st16(lane_base + col, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_p_full[bf]));
      }
      if (!mbar_wait(smem_u32(&s.bar_dp_full), n & 1, wc, TAG_DP_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        float dp[32];
        tmem_ld32(lane_base + COL_DPT + 32 * g, dp);
        tmem_wait_ld();
        const float4* d4 = reinterpret_cast<const float4*>(&s.delta[st][32 * g]);
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 D = d4[q];
          pk[2 * q] = pack2<BF16>(pv[4 * q] * (dp[4 * q] - D.x), pv[4 * q + 1] * (dp[4 * q + 1] - D.y));
          pk[2 * q + 1] =
              pack2<BF16>(pv[4 * q + 2] * (dp[4 * q + 2] - D.z), pv[4 * q + 3] * (dp[4 * q + 3] - D.w));
        }
        tmem_st16(lane_base + col + 16, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_ds_full));
      }
    }
    // ---------------------------------------------------------- epilogue
    bool have = ok && N > 0;
    if (have) have = mbar_wait(smem_u32(&s.bar_acc_full), 0, wc, TAG_ACC);
    tc_fence_after();
    // K in shared memory is dead once every softmax warp has copied it
    named_bar_sync(1, 256);
    const int r0 = k0 + sp * 32;
    const int nvalid = min(32, p.Skv - r0);
    uint8_t* stage = s.K + (warp - 2) * 4096;
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK
      uint32_t pk[32];
      if (have) {
        const float sc = which ? p.scale : 1.f;
        const uint32_t colA = (which ? COL_DK : COL_DV) + 64 * g;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld32(lane_base + colA + 32 * half, v);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 16; ++cc)
            pk[16 * half + cc] = pack2<BF16>(v[2 * cc] * sc, v[2 * cc + 1] * sc);
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) pk[cc] = 0u;
      }
      uint16_t* base = which ? dk : dv;
      uint16_t* orow = base + ((size_t)bc * p.Skv + r0) * HEAD_DIM + 64 * g;
      warp_store_rows(stage, pk, orow, nvalid);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

cudaError_t launch_dkdv(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                        const CUtensorMap& tdO, const CUtensorMap& tK, const CUtensorMap& tV,
                        void* dk, void* dv, cudaStream_t st) {
  auto kern = bf16 ? k_dkdv<true> : k_dkdv<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kv_side::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int nKT = (p.Skv + KV_TILE - 1) / KV_TILE;
  dim3 grid((unsigned)(nKT * p.B * p.Hkv));
  kern<<<grid, kv_side::NUM_THREADS, kv_side::SMEM_BYTES, st>>>(tQ, tdO, tK, tV, (uint16_t*)dk,
                                                                 (uint16_t*)dv, p);
  return cudaGetLastError();
}

}  // namespace mab
