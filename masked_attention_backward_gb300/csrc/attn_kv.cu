// attn_kv.cu -- key-stationary dK/dV kernel on tcgen05 / TMEM, fed by TMA.
//
// One CTA per (b, kv head c, KV_TILE key rows).  K and V of the tile are
// loaded once.  The CTA walks every query head of the GQA group and, for each,
// every active query sub-tile r of KV_SUB rows (closed-form range for causal /
// sliding / none, the key-major select table for block masks):
//   S^T  = K Q_r^T,   dP^T = V dO_r^T                (SS MMA, fp32 in TMEM)
//   P^T  = exp2(S^T * scale*log2e - lse2_r),  dS^T = P^T (dP^T - Delta_r)
//   dV  += P^T dO_r,  dK += dS^T Q_r                 (TS MMA, P^T / dS^T from TMEM)
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
#include <math.h>

#include "tiles.cuh"

namespace mab {

namespace kv_side {

constexpr int STAGES = 3;   // Q/dO ring depth
constexpr int NBUF = 2;     // S/dP buffers in TMEM
constexpr int COL_DV = 0;
constexpr int COL_DK = 128;
constexpr int COL_S = 256;  // buffer b: S^T at COL_S + 128 b, dP^T at +64
constexpr int NUM_THREADS = 320;

struct __align__(1024) Smem {
  uint8_t K[2 * KV_TILE * 128];
  uint8_t V[2 * KV_TILE * 128];
  uint8_t Q[STAGES][2 * KV_SUB * 128];
  uint8_t dO[STAGES][2 * KV_SUB * 128];
  float lse2[STAGES][KV_SUB];
  float delta[STAGES][KV_SUB];
  uint64_t bar_kv_full;
  uint64_t bar_q_full[STAGES];
  uint64_t bar_q_empty[STAGES];
  uint64_t bar_s_full[NBUF];
  uint64_t bar_p_full[NBUF];
  uint64_t bar_s_free[NBUF];
  uint64_t bar_acc_full;
  uint64_t bar_drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;

enum { TAG_KV = 0x201, TAG_Q_EMPTY, TAG_Q_FULL, TAG_S_FREE, TAG_P_FULL, TAG_S_FULL, TAG_ACC,
       TAG_DRAIN };

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
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.bar_q_full[i]), 1);
      mbar_init(smem_u32(&s.bar_q_empty[i]), 1);
    }
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_p_full[i]), 8);
      mbar_init(smem_u32(&s.bar_s_free[i]), 1);
    }
    mbar_init(smem_u32(&s.bar_acc_full), 1);
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
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_f16(BF16, KV_TILE, KV_SUB, false, false);
      constexpr uint32_t ID_ACC = idesc_f16(BF16, KV_TILE, HEAD_DIM, false, true);
      const uint32_t sK = smem_u32(s.K), sV = smem_u32(s.V);
      auto consume = [&](int m) -> bool {
        const int bf = m % NBUF, st = m % STAGES;
        if (!mbar_wait(smem_u32(&s.bar_p_full[bf]), (m / NBUF) & 1, wc, TAG_P_FULL)) return false;
        tc_fence_after();
        const uint32_t colS = tbase + COL_S + bf * 128;
        const uint32_t sQ = smem_u32(s.Q[st]), sdO = smem_u32(s.dO[st]);
#pragma unroll
        for (int kk = 0; kk < KV_SUB / 16; ++kk) {
          const uint32_t a_off = 32 * (kk >> 1) + 8 * (kk & 1);
          mma_ts(tbase + COL_DV, colS + a_off, sdesc_sw128(sdO + kk * 2048, KV_SUB * 128, 1024),
                 ID_ACC, (m > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < KV_SUB / 16; ++kk) {
          const uint32_t a_off = 32 * (kk >> 1) + 8 * (kk & 1);
          mma_ts(tbase + COL_DK, colS + 64 + a_off, sdesc_sw128(sQ + kk * 2048, KV_SUB * 128, 1024),
                 ID_ACC, (m > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&s.bar_q_empty[st]));
        mma_commit(smem_u32(&s.bar_s_free[bf]));
        return true;
      };
      bool ok = mbar_wait(smem_u32(&s.bar_kv_full), 0, wc, TAG_KV);
      tc_fence_after();
      for (int n = 0; ok && n < N; ++n) {
        const int st = n % STAGES, bf = n % NBUF;
        if (!mbar_wait(smem_u32(&s.bar_q_full[st]), (n / STAGES) & 1, wc, TAG_Q_FULL)) {
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
        const uint32_t sQ = smem_u32(s.Q[st]), sdO = smem_u32(s.dO[st]);
#pragma unroll
        for (int kk = 0; kk < HEAD_DIM / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * (KV_TILE * 128) + (kk & 3) * 32;
          const uint32_t bo = (kk >> 2) * (KV_SUB * 128) + (kk & 3) * 32;
          mma_ss(colS, sdesc_sw128(sK + ao, 16, 1024), sdesc_sw128(sQ + bo, 16, 1024), ID_S,
                 kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < HEAD_DIM / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * (KV_TILE * 128) + (kk & 3) * 32;
          const uint32_t bo = (kk >> 2) * (KV_SUB * 128) + (kk & 3) * 32;
          mma_ss(colS + 64, sdesc_sw128(sV + ao, 16, 1024), sdesc_sw128(sdO + bo, 16, 1024), ID_S,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&s.bar_s_full[bf]));
        if (n >= 1 && !consume(n - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && N >= 1) ok = consume(N - 1);
      mma_commit(smem_u32(&s.bar_acc_full));
      mma_commit(smem_u32(&s.bar_drain));
      mbar_wait(smem_u32(&s.bar_drain), 0, wc, TAG_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int sp = warp & 3, g = (warp - 2) >> 2;
    const int rloc = sp * 32 + lane;
    const int j = k0 + rloc;
    const uint32_t lane_base = tbase + ((uint32_t)(sp * 32) << 16);
    bool ok = true;
    KVCursor cur;
    cur.start(p, walk);
    for (int n = 0; n < N; ++n) {
      const int bf = n % NBUF, st = n % STAGES;
      // s_full implies the stage's loads landed; waiting on q_full as well
      // makes the bulk-copied lse2 / Delta rows visible to this thread
      if (!mbar_wait(smem_u32(&s.bar_s_full[bf]), (n / NBUF) & 1, wc, TAG_S_FULL) ||
          !mbar_wait(smem_u32(&s.bar_q_full[st]), (n / STAGES) & 1, wc, TAG_Q_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int r = walk.tile(p, cur.hh, cur.idx);
      const int bh = b * p.Hq + c * p.group + cur.hh;
      cur.next(p, walk);
      const uint32_t vis = vis_key_row(p, bh, j, r * KV_SUB + 32 * g);
      const uint32_t col = COL_S + bf * 128 + 32 * g;
      float sv[32], dp[32];
      tmem_ld32(lane_base + col, sv);
      tmem_ld32(lane_base + col + 64, dp);
      tmem_wait_ld();
      const float4* l4 = reinterpret_cast<const float4*>(&s.lse2[st][32 * g]);
      const float4* d4 = reinterpret_cast<const float4*>(&s.delta[st][32 * g]);
      uint32_t pkP[16], pkD[16];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 L = l4[q], Dl = d4[q];
        const float lv[4] = {L.x, L.y, L.z, L.w};
        const float dv4[4] = {Dl.x, Dl.y, Dl.z, Dl.w};
        float pv[4], dsv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int cc = 4 * q + e;
          float pe = fast_exp2(fmaf(sv[cc], p.scale_log2, -lv[e]));
          pe = ((vis >> cc) & 1u) ? pe : 0.f;
          pv[e] = pe;
          dsv[e] = pe * (dp[cc] - dv4[e]);
        }
        pkP[2 * q] = pack2<BF16>(pv[0], pv[1]);
        pkP[2 * q + 1] = pack2<BF16>(pv[2], pv[3]);
        pkD[2 * q] = pack2<BF16>(dsv[0], dsv[1]);
        pkD[2 * q + 1] = pack2<BF16>(dsv[2], dsv[3]);
      }
      tmem_st16(lane_base + col, pkP);
      tmem_st16(lane_base + col + 64, pkD);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_p_full[bf]));
    }
    // ---------------------------------------------------------- epilogue
    bool have = ok && N > 0;
    if (have) have = mbar_wait(smem_u32(&s.bar_acc_full), 0, wc, TAG_ACC);
    tc_fence_after();
    const int r0 = k0 + sp * 32;
    const int nvalid = min(32, p.Skv - r0);
    uint8_t* stage = &s.Q[0][0] + (warp - 2) * 4096;  // Q stages are idle now
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
