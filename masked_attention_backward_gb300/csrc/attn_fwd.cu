// attn_fwd.cu -- forward kernel producing O and LSE (the inputs of the
// backward), query-stationary on tcgen05 / TMEM, fed by TMA.
//
// One CTA per (b, query head, Q_TILE query rows); Q is loaded once and copied
// into TMEM, where it is the A operand of every S = Q K_t^T.  Two passes over
// the same active key sub-tiles t (Q_SUB rows):
//   pass A: S, the row maximum m of the scaled logits and of the sink logit
//           (which joins only the denominator) -- no exponentials;
//   pass B: S again, P' = exp2(S * scale*log2e - m), O' += P' V_t, and the
//           row sum l of P' in fp32.
// At the end O = O' / l and LSE = (m + log2 l) ln 2, with the sink's
// exp2(sink log2e - m) added to l.  Because pass B already knows the final
// maximum, O' never needs rescaling, and each logit is exponentiated once.
//
// Sources: tilelang-ascend PR #1 "Add GQA Sink Backward BHSD", Summary
// (online softmax with an attention sink and a sliding window);
// cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook, precision
// notes (a row that sees no key gets zeros).
//
// TMEM columns (512): O accumulator [0,128), Q as 16-bit pairs [128,192), two
// fp32 S buffers [192,320), two packed P buffers [320,384).  Softmax group g
// owns key columns 16 g .. 16 g + 15 of a sub-tile, so the 16 keys of MMA
// K-step g sit at column 8 g of a P buffer.  S(n) reuses the buffer of
// S(n-2) once the softmax warps have loaded it; P(k) reuses the buffer of
// P(k-2) once O += P(k-2) V has read it.
//
// Warp roles (608 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues S, warp 2 issues O += P V (whole warps, one elected lane); warps
// 3..18 are the softmax warps: warp (sp, g) with sp = warp % 4 owns TMEM lanes
// 32 sp .. 32 sp + 31 (query rows) and key columns 16 g .. 16 g + 15.
#include <math.h>

#include "tiles.cuh"

namespace mab {

namespace fwd_side {

constexpr int STAGES = 4;     // K/V ring depth (pass A stages hold K only)
constexpr int COL_O = 0;      // O accumulator, 128 fp32 columns
constexpr int COL_QA = 128;   // Q as the A operand
constexpr int COL_S = 192;    // S buffer b at COL_S + 64 b, fp32
constexpr int COL_P = 320;    // P buffer b at COL_P + 32 b, 16-bit pairs
constexpr int SM_WARP0 = 3;   // first softmax warp
constexpr int SM_WARPS = 16;  // softmax warps
constexpr int NUM_THREADS = 32 * (SM_WARP0 + SM_WARPS);

struct __align__(1024) Smem {
  uint8_t Q[2 * Q_TILE * 128];  // two 64-column chunks, 128B swizzle; stages the output
  uint8_t K[STAGES][2 * Q_SUB * 128];
  uint8_t V[STAGES][2 * Q_SUB * 128];
  float ml[4][Q_TILE][2];       // per-group (max of S, sum of P') per row
  uint64_t bar_q_full;          // Q landed in shared memory
  uint64_t bar_qa_full;         // Q copied into TMEM (all softmax warps)
  uint64_t bar_kv_full[STAGES];
  uint64_t bar_kv_empty[STAGES];
  uint64_t bar_s_full[2];       // S of the buffer complete
  uint64_t bar_s_free[2];       // S of the buffer loaded by every softmax warp
  uint64_t bar_p_full[2];       // P of the buffer written (all softmax warps)
  uint64_t bar_p_free[2];       // O += P V that read the buffer complete
  uint64_t bar_x_done;          // every S MMA complete
  uint64_t bar_acc_full;        // every O MMA complete
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;

// Wait tags recorded in the status word when a wait runs out.
enum { TAG_Q = 0x101, TAG_QA, TAG_KV_EMPTY, TAG_KV_FULL, TAG_S_FULL, TAG_S_FREE, TAG_P_FULL,
       TAG_P_FREE, TAG_ACC, TAG_X_DONE };

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
    mbar_init(smem_u32(&s.bar_qa_full), SM_WARPS);
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&s.bar_kv_full[i]), 1);
      mbar_init(smem_u32(&s.bar_kv_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_s_free[i]), SM_WARPS);
      mbar_init(smem_u32(&s.bar_p_full[i]), SM_WARPS);
      mbar_init(smem_u32(&s.bar_p_free[i]), 1);
    }
    mbar_init(smem_u32(&s.bar_x_done), 1);
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
    // ------------------------------------------------------------ S issuer (whole warp)
    constexpr uint32_t ID_S = idesc_f16(BF16, Q_TILE, Q_SUB, false, false);
    bool ok = N == 0 || mbar_wait_warp(smem_u32(&s.bar_qa_full), 0, wc, TAG_QA);
    for (int n = 0; ok && n < NT; ++n) {
      const int bf = n & 1, st = n % STAGES;
      ok = mbar_wait_warp(smem_u32(&s.bar_kv_full[st]), (n / STAGES) & 1, wc, TAG_KV_FULL);
      // the buffer held S(n - 2): the softmax warps must have loaded it
      if (ok && n >= 2)
        ok = mbar_wait_warp(smem_u32(&s.bar_s_free[bf]), ((n - 2) >> 1) & 1, wc, TAG_S_FREE);
      if (!ok) break;
      tc_fence_after();
      const uint64_t bK = sdesc_sw128(smem_u32(s.K[st]), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < HEAD_DIM / 16; ++kk)
        mma_ts_w(tbase + COL_S + 64 * bf, tbase + COL_QA + 8 * kk,
                 bK + (uint64_t)(((kk >> 2) * (Q_SUB * 128) + (kk & 3) * 32) >> 4), ID_S,
                 kk > 0 ? 1u : 0u);
      mma_commit_w(smem_u32(&s.bar_s_full[bf]));
      // a pass-A stage holds K only, which S(n) has read once it completes
      if (n < N) mma_commit_w(smem_u32(&s.bar_kv_empty[st]));
    }
    // this warp's MMAs must be complete before TMEM is freed (abort path)
    mma_commit_w(smem_u32(&s.bar_x_done));
    mbar_wait_warp(smem_u32(&s.bar_x_done), 0, wc, TAG_X_DONE);
  } else if (warp == 2) {
    // ------------------------------------------------------------ O issuer (whole warp)
    constexpr uint32_t ID_O = idesc_f16(BF16, Q_TILE, HEAD_DIM, false, true);
    bool ok = true;
    for (int k = 0; ok && k < N; ++k) {
      const int n = N + k, bf = k & 1, st = n % STAGES;
      ok = mbar_wait_warp(smem_u32(&s.bar_kv_full[st]), (n / STAGES) & 1, wc, TAG_KV_FULL) &&
           mbar_wait_warp(smem_u32(&s.bar_p_full[bf]), (k >> 1) & 1, wc, TAG_P_FULL);
      if (!ok) break;
      tc_fence_after();
      const uint64_t bV = sdesc_sw128(smem_u32(s.V[st]), Q_SUB * 128, 1024);
#pragma unroll
      for (int kk = 0; kk < Q_SUB / 16; ++kk)
        mma_ts_w(tbase + COL_O, tbase + COL_P + 32 * bf + 8 * kk,
                 bV + (uint64_t)((kk * 2048) >> 4), ID_O, (k > 0 || kk > 0) ? 1u : 0u);
      mma_commit_w(smem_u32(&s.bar_p_free[bf]));
      // S(n) completed before the softmax warps could write P(k), so this
      // commit frees the K / V stage
      mma_commit_w(smem_u32(&s.bar_kv_empty[st]));
    }
    // completes when every MMA issued above has (also on the abort path, so
    // that TMEM is idle before it is freed)
    mma_commit_w(smem_u32(&s.bar_acc_full));
    mbar_wait_warp(smem_u32(&s.bar_acc_full), 0, wc, TAG_ACC);
  } else {
    // ------------------------------------------------------------ softmax warps
    const int sp = warp & 3, g = (warp - SM_WARP0) >> 2;
    const int rloc = sp * 32 + lane;
    const int i = q0 + rloc;
    const uint32_t lane_base = tbase + ((uint32_t)(sp * 32) << 16);
    bool ok = mbar_wait(smem_u32(&s.bar_q_full), 0, wc, TAG_Q);
    if (ok) {
      // Q rows into TMEM as 16-bit pairs (element 2c in the low half of column
      // c): this warp copies d columns 32 g .. 32 g + 31 of its rows.
      const int u0 = (g & 1) * 4;
      const uint8_t* src = s.Q + (g >> 1) * (Q_TILE * 128) + rloc * 128;
      uint32_t w[16];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + (((u0 + u) ^ (rloc & 7)) << 4));
        w[4 * u] = v.x;
        w[4 * u + 1] = v.y;
        w[4 * u + 2] = v.z;
        w[4 * u + 3] = v.w;
      }
      tmem_st16(lane_base + COL_QA + 16 * g, w);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.bar_qa_full));

    int flo, fhi;  // key sub-tiles that are entirely visible
    full_range_q(p.mask_kind, p.window, p.Sq, p.Skv, q0, &flo, &fhi);
    // Loads this warp's 16 columns of S(n) into registers and releases the
    // buffer; returns the visibility of the columns.
    auto load_s = [&](int n, float (&x)[16]) -> uint32_t {
      const int bf = n & 1;
      tmem_ld16(lane_base + COL_S + 64 * bf + 16 * g, x);
      const int t = walk.tile(n >= N ? n - N : n);
      const uint32_t vis =
          (t >= flo && t <= fhi) ? 0xffffu : vis_query_row(p, bh, i, t * Q_SUB + 16 * g);
      tmem_wait_ld_regs(x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_s_free[bf]));
      return vis;
    };

    // pass A: the maximum of this warp's visible logits of the row (raw S;
    // the scale is positive, so it is applied once afterwards)
    float mx = -INFINITY;
    for (int n = 0; ok && n < N; ++n) {
      if (!mbar_wait(smem_u32(&s.bar_s_full[n & 1]), (n >> 1) & 1, wc, TAG_S_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[16];
      const uint32_t vis = load_s(n, x);
#pragma unroll
      for (int c = 0; c < 16; ++c) mx = ((vis >> c) & 1u) ? fmaxf(mx, x[c]) : mx;
    }
    // combine the four column groups of each row, and the sink
    s.ml[g][rloc][0] = mx;
    named_bar_sync(1, 32 * SM_WARPS);
    const float sink2 = p.sink ? p.sink[h] * LOG2E : -INFINITY;
    float m2;  // row maximum in the log2 domain
    {
      float m = -INFINITY;
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) m = fmaxf(m, s.ml[gg][rloc][0]);
      m2 = fmaxf(m == -INFINITY ? -INFINITY : m * p.scale_log2, sink2);
    }
    // a row that sees nothing keeps every P' at zero through the visibility
    // mask; the finite stand-in only avoids inf - inf
    const float m2s = m2 == -INFINITY ? 0.f : m2;
    // pass B: P' into TMEM for O' += P' V, row sums in fp32
    float l_acc = 0.f;
    for (int k = 0; ok && k < N; ++k) {
      const int n = N + k, bf = k & 1;
      if (!mbar_wait(smem_u32(&s.bar_s_full[n & 1]), (n >> 1) & 1, wc, TAG_S_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[16];
      const uint32_t vis = load_s(n, x);
      uint32_t pk[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float p0 = fast_exp2(fmaf(x[2 * c], p.scale_log2, -m2s));
        float p1 = fast_exp2(fmaf(x[2 * c + 1], p.scale_log2, -m2s));
        p0 = ((vis >> (2 * c)) & 1u) ? p0 : 0.f;
        p1 = ((vis >> (2 * c + 1)) & 1u) ? p1 : 0.f;
        l_acc += p0 + p1;
        pk[c] = pack2<BF16>(p0, p1);
      }
      // O' += P'(k - 2) V must have read this P buffer
      if (k >= 2 && !mbar_wait(smem_u32(&s.bar_p_free[bf]), ((k - 2) >> 1) & 1, wc, TAG_P_FREE)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st8(lane_base + COL_P + 32 * bf + 8 * g, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_p_full[bf]));
    }
    // row sum over the four column groups, plus the sink
    s.ml[g][rloc][1] = l_acc;
    named_bar_sync(1, 32 * SM_WARPS);
    float inv_l;
    {
      float l = p.sink ? fast_exp2(sink2 - m2s) : 0.f;
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) l += s.ml[gg][rloc][1];
      const float lse2 = (l > 0.f) ? m2s + log2f(l) : INFINITY;
      if (g == 0 && i < p.Sq) p.lse_out[(size_t)bh * p.Sq + i] = lse2 * 0.6931471805599453f;
      inv_l = (l > 0.f) ? 1.f / l : 0.f;
    }
    // ---------------------------------------------------------- epilogue
    // Columns [32 g, 32 g + 32) of the accumulator, one row per lane.
    uint32_t pk[16];
    bool have = ok && N > 0;
    if (have) have = mbar_wait(smem_u32(&s.bar_acc_full), 0, wc, TAG_ACC);
    tc_fence_after();
    if (have) {
      float v[32];
      tmem_ld32(lane_base + COL_O + 32 * g, v);
      tmem_wait_ld_regs(v);
#pragma unroll
      for (int c = 0; c < 16; ++c) pk[c] = pack2<BF16>(v[2 * c] * inv_l, v[2 * c + 1] * inv_l);
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) pk[c] = 0u;
    }
    // the Q tile is dead once every softmax warp has copied it into TMEM
    // (they all passed the merge barrier after their copy): it stages the rows
    uint8_t* stage = s.Q + (warp - SM_WARP0) * 2048;
    const int r0 = q0 + sp * 32;
    uint16_t* orow = out + ((size_t)bh * p.Sq + r0) * HEAD_DIM + 32 * g;
    warp_store_rows32(stage, pk, orow, min(32, p.Sq - r0));
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
