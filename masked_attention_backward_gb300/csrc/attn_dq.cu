// attn_dq.cu -- query-stationary dQ kernel on tcgen05 / TMEM, fed by TMA.
//
// Work unit: (b, query head h, Q_TILE query rows).  Q and dO of the unit are
// loaded once and copied into TMEM, where they serve as the A operand of
// every score contraction.  For each active key sub-tile t of Q_SUB rows:
//   S  = Q K_t^T,  dP = dO V_t^T                 (A from TMEM, fp32 in TMEM)
//   P  = exp2(S * scale*log2e - lse log2e),  dS = P (dP - Delta)   (softmax warps)
//   dQ += dS K_t                                  (A = dS from TMEM)
// then dQ *= scale, rounded to the input dtype and written once.
//
// Sources: tilelang-ascend PR #1 "Add GQA Sink Backward BHSD", commit notes
// (five contractions + softmax + dS per KV step; P recomputed from LSE);
// cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook, skeleton
// "delta -> dq -> dkdv" with dq walking the query-major select table, and the
// precision notes (p = exp(s - lse), ds = p (dp - delta), fp16 / bf16
// operands into the contraction with fp32 accumulation).
//
// Why the operands sit where they do: an MMA whose A and B both come from
// shared memory at N = 64 is limited by shared-memory bandwidth (it reads
// 6 KB per 32 cycles of math), while with A in TMEM it reads only its 2 KB B
// tile and runs at the tensor pipe's rate.  Q and dO are the same for the
// whole walk of a unit, so they move to TMEM once.
//
// Persistent: one CTA per SM.  Units are numbered heaviest causal rows first;
// CTA b starts with unit b and then claims the next unnumbered unit from a
// global counter whenever it starts loading one, so the SMs finish together.
// TMEM is allocated and the barriers set up once, the next unit's Q / dO
// tiles load while the current unit runs, and the K / V ring, the S / dP
// buffers and their barrier phases simply continue across units (counted by
// one step counter m).  The producer publishes each claimed unit (or -1 when
// none is left) in shared memory with the Q / dO load, and loads the next
// unit's Q / dO only once every other warp has taken the current one
// (unit_free): so no per-unit barrier can run two phases ahead of a warp that
// waits on it, units without active tiles included.  Between units the
// epilogue of unit j and the first dQ MMA of unit j + 1 meet at acc_empty.
//
// TMEM columns (512): dQ accumulator [0,128), Q [128,192), dO [192,256)
// (16-bit pairs), and two S/dP buffers of 128 columns at 256 and 384 (S in
// the first 64, dP in the next 64).  Softmax group g owns key columns
// 32 g .. 32 g + 31 and packs its 32 dS values over the first 16 of them, so
// the 16 keys of MMA K-step kk sit at buffer column 32 (kk / 2) + 8 (kk % 2).
//
// Three warps issue MMAs into the one tensor pipe: warp 1 S(m), warp 2 dP(m),
// warp 3 the accumulation dQ(n), each waiting only on its own inputs.  The
// pipe accepts only a few MMAs ahead of the one executing and a barrier wait
// costs a few hundred cycles while the softmax warps keep the SM busy, so
// with a single issuer every wait drained the pipe.
//
// Warp roles (384 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues S, warp 2 issues dP, warp 3 issues dQ (whole warps, one elected
// lane), warps 4..11 are two groups of four softmax warps; warp (sp, g) with
// sp = warp % 4 owns TMEM lanes 32 sp .. 32 sp + 31 (query rows) and key
// columns 32 g .. 32 g + 31 of each sub-tile (eight softmax warps measured 7 %
// faster than sixteen: each step's fixed work of waits, fences and signals
// is spread over twice the elements).
#include <math.h>

#include "tiles.cuh"

namespace mab {

namespace dq_side {

constexpr int STAGES = 5;     // K/V ring depth
constexpr int COL_ACC = 0;    // dQ accumulator, 128 fp32 columns
constexpr int COL_QA = 128;   // Q as the A operand, 64 columns of 16-bit pairs
constexpr int COL_DOA = 192;  // dO as the A operand
constexpr int COL_BUF = 256;  // buffer b: S at COL_BUF + 128 b, dP at +64
constexpr int SM_WARP0 = 4;   // first softmax warp
constexpr int SM_WARPS = 8;   // softmax warps
constexpr int NUM_THREADS = 32 * (SM_WARP0 + SM_WARPS);

struct __align__(1024) Smem {
  uint8_t Q[2 * Q_TILE * 128];  // two 64-column chunks, 128B swizzle; once copied
                                // into TMEM, the epilogue staging (4 KB per warp)
  uint8_t dO[2 * Q_TILE * 128];
  uint8_t K[STAGES][2 * Q_SUB * 128];
  uint8_t V[STAGES][2 * Q_SUB * 128];
  int step_t[STAGES];           // key sub-tile of the step in the stage
  uint32_t step_vis[STAGES];    // aligned block masks: bit 2 sp + g = region (sp, g) visible
  int unit;                     // unit of the latest Q / dO load, -1: none left
  uint64_t bar_q_full;          // Q, dO of the unit landed in shared memory
  uint64_t bar_qa_full;         // Q, dO copied into TMEM (all softmax warps)
  uint64_t bar_kv_full[STAGES];
  uint64_t bar_kv_empty[STAGES];
  uint64_t bar_s_full[2];       // S and dP of the buffer complete (one commit each)
  uint64_t bar_p_full[2];       // dS of the buffer packed (all softmax warps)
  uint64_t bar_acc_free[2];     // dQ MMA that read the buffer's dS complete
  uint64_t bar_acc_full;        // every dQ MMA of the unit complete
  uint64_t bar_acc_empty;       // the unit's accumulator read and stored (all softmax warps)
  uint64_t bar_unit_free;       // every other warp took the unit (and, softmax warps,
                                // stored the previous unit's epilogue)
  uint64_t bar_x_done[3];       // every MMA of the S / dP / dQ warp complete
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;
static_assert(SMEM_BYTES <= 232448, "over the 227 KB of shared memory a CTA may use");

enum { TAG_Q = 0x301, TAG_QA, TAG_KV_EMPTY, TAG_KV_FULL, TAG_P_FULL, TAG_S_FULL, TAG_ACC_FREE,
       TAG_ACC, TAG_X_DONE, TAG_ACC_EMPTY, TAG_UNIT_FREE };

// Stage of the K/V ring and the parity of its current use (kept as counters:
// STAGES is not a power of two).
struct Ring {
  int st = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    if (++st == STAGES) {
      st = 0;
      ph ^= 1u;
    }
  }
};

// Coordinates of work unit u: heaviest causal query tiles first.
struct DqUnit {
  int bh, q0, kvh, h;
  QWalk walk;
  // VARLEN: the call gave per-batch lengths (otherwise every batch element
  // has all Sq rows and Skv keys, and none is read)
  template <bool VARLEN>
  __device__ __forceinline__ void init(const AttnParams& p, int u) {
    const int BH = p.B * p.Hq;
    const int qt = p.nQT_q - 1 - u / BH;
    bh = u % BH;
    h = bh % p.Hq;
    const int b = bh / p.Hq;
    kvh = b * p.Hkv + h / p.group;
    q0 = qt * Q_TILE;
    walk.init(p, bh, qt, VARLEN ? len_q(p, b) : p.Sq, VARLEN ? len_k(p, b) : p.Skv);
  }
};

}  // namespace dq_side

// MK: the mask kind (MK_NONE, MK_CAUSAL, MK_SLIDING or MK_BLOCK); each instance keeps
// only its own visibility code in the softmax loop (measured 1.5 to 3.5 %
// faster on the short-walk and variable-length workloads).
// HILO: dS enters the dQ contraction as a 16-bit high part (columns
// 32 g .. 32 g + 15 of group g's slice) plus a 16-bit remainder (columns
// 32 g + 16 .. 32 g + 31, whose fp32 S values are already in registers).
template <bool BF16, bool VARLEN, bool HILO, int MK>
__global__ void __launch_bounds__(dq_side::NUM_THREADS, 1)
k_dq(const __grid_constant__ CUtensorMap tQ, const __grid_constant__ CUtensorMap tdO,
     const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV,
     uint16_t* __restrict__ dq, const AttnParams p) {
  using namespace dq_side;
  constexpr bool BLOCK = MK == MK_BLOCK;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int U = p.nQT_q * p.B * p.Hq;
  // a block mask whose blocks hold whole softmax-warp regions (32 queries x
  // 32 keys): each region is visible entirely or not at all (with per-batch
  // lengths the per-element path is kept, which spares that instance's registers)
  const bool blk_regions =
      !VARLEN && BLOCK && (p.bx & 31) == 0 && (p.by & 31) == 0;
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
      mbar_init(smem_u32(&s.bar_s_full[i]), 2);
      mbar_init(smem_u32(&s.bar_p_full[i]), SM_WARPS);
      mbar_init(smem_u32(&s.bar_acc_free[i]), 1);
    }
    mbar_init(smem_u32(&s.bar_acc_full), 1);
    mbar_init(smem_u32(&s.bar_acc_empty), SM_WARPS);
    mbar_init(smem_u32(&s.bar_unit_free), SM_WARPS + 3);
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&s.bar_x_done[i]), 1);
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
    // Without per-batch lengths the whole warp runs the walk and lane 0
    // claims units and issues the copies: every 32 steps the lanes look up
    // the next 32 steps at once (key sub-tile from the select table, aligned
    // block masks' region word from the mask), so that no step waits for a
    // chain of global loads of its own (random 30 % blocks: k_dq 0.411 ->
    // 0.302 ms).  The per-batch-length instance, whose registers are at their
    // limit, keeps lane 0 walking alone (the warp-wide form measured 7 %
    // slower there).
    if constexpr (VARLEN) {
      if (lane == 0 && !p.test_no_loads) {
        tma_prefetch_desc(&tQ);
        tma_prefetch_desc(&tdO);
        tma_prefetch_desc(&tK);
        tma_prefetch_desc(&tV);
        bool ok = true;
        int m = 0;  // step counter across units
        int q_loaded = -1;  // last unit whose Q / dO tiles were loaded
        Ring rg;
        const uint32_t qbar = smem_u32(&s.bar_q_full);
        for (int j = 0; ok; ++j) {
          // the Q / dO tiles and the unit slot are free once every other warp
          // has taken the previous unit (the softmax warps: copied its Q / dO
          // into TMEM and stored the epilogue before it, staged in the Q tile)
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
          DqUnit un{};
          un.template init<VARLEN>(p, u);
          if (un.walk.cnt == 0) {
            // nothing to contract: the unit's rows only get zeros, so its
            // Q / dO tiles are not loaded
            mbar_arrive(qbar);
          } else {
            // packed layout (always with per-batch lengths): token coordinates;
            // BHSD: (row, head)
            const RowAddr qa = VARLEN ? row_q(p, un.bh / p.Hq, un.h, un.q0)
                                      : RowAddr{un.q0, un.bh, 0, HEAD_DIM};
            mbar_arrive_expect_tx(qbar, 4 * Q_TILE * 128);
            tma_load_3d(smem_u32(s.Q), &tQ, 0, qa.c1, qa.c2, qbar);
            tma_load_3d(smem_u32(s.Q + Q_TILE * 128), &tQ, 64, qa.c1, qa.c2, qbar);
            tma_load_3d(smem_u32(s.dO), &tdO, 0, qa.c1, qa.c2, qbar);
            tma_load_3d(smem_u32(s.dO + Q_TILE * 128), &tdO, 64, qa.c1, qa.c2, qbar);
            q_loaded = j;
          }
          for (int n = 0; n < un.walk.cnt; ++n, ++m, rg.next()) {
            const int st = rg.st;
            const int t = un.walk.tile(n);
            // aligned block masks: the mask byte of each softmax warp's 32-query
            // x 32-key region, loaded before the wait below (which hides the
            // latency; indices clamped into the mask, ranges applied after)
            uint32_t mv[8];
            if (blk_regions) {
              const uint8_t* mb = p.mask + (size_t)un.bh * p.nqb * p.nkb;
#pragma unroll
              for (int sp2 = 0; sp2 < 4; ++sp2) {
                const int qb = min((un.q0 + 32 * sp2) / p.bx, p.nqb - 1);
#pragma unroll
                for (int g2 = 0; g2 < 2; ++g2) {
                  const int kb = min((t * Q_SUB + 32 * g2) / p.by, p.nkb - 1);
                  mv[2 * sp2 + g2] = mb[(size_t)qb * p.nkb + kb];
                }
              }
            }
            if (m >= STAGES &&
                !mbar_wait(smem_u32(&s.bar_kv_empty[st]), rg.ph ^ 1u, wc,
                           TAG_KV_EMPTY)) {
              ok = false;
              break;
            }
            s.step_t[st] = t;  // published by the arrive below together with the loads
            if (blk_regions) {
              uint32_t w = 0;
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (mv[e] && un.q0 + 32 * (e >> 1) < p.Sq && t * Q_SUB + 32 * (e & 1) < p.Skv)
                  w |= 1u << e;
              s.step_vis[st] = w;
            }
            const uint32_t fb = smem_u32(&s.bar_kv_full[st]);
            const RowAddr ka = VARLEN ? row_k(p, un.kvh / p.Hkv, un.kvh % p.Hkv, t * Q_SUB)
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
    } else {
      if (!p.test_no_loads) {
        if (lane == 0) {
          tma_prefetch_desc(&tQ);
          tma_prefetch_desc(&tdO);
          tma_prefetch_desc(&tK);
          tma_prefetch_desc(&tV);
        }
        // lane 0 waits; the rest of the warp waits for its answer
        auto wait0 = [&](uint32_t bar, uint32_t parity, unsigned int tag) -> bool {
          bool r = true;
          if (lane == 0) r = mbar_wait(bar, parity, wc, tag);
          return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
        };
        bool ok = true;
        int m = 0;  // step counter across units
        int q_loaded = -1;  // last unit whose Q / dO tiles were loaded
        Ring rg;
        const uint32_t qbar = smem_u32(&s.bar_q_full);
        for (int j = 0; ok; ++j) {
          // the Q / dO tiles and the unit slot are free once every other warp
          // has taken the previous unit (the softmax warps: copied its Q / dO
          // into TMEM and stored the epilogue before it, staged in the Q tile)
          if (j >= 1 && !wait0(smem_u32(&s.bar_unit_free), (j - 1) & 1, TAG_UNIT_FREE)) {
            ok = false;
            break;
          }
          int u = 0;
          if (lane == 0) {
            u = j == 0 ? (int)blockIdx.x : (int)(gridDim.x + atomicAdd(&p.status->next_unit, 1u));
            if (u >= U) u = -1;
          }
          u = __shfl_sync(0xffffffffu, u, 0);
          DqUnit un{};
          if (u >= 0) un.template init<VARLEN>(p, u);
          if (lane == 0) {
            s.unit = u;  // published by the arrive on q_full
            if (u < 0 || un.walk.cnt == 0) {
              // nothing to contract: the unit's rows only
              // get zeros, so its Q / dO tiles are not loaded
              mbar_arrive(qbar);
            } else {
              // packed layout (always with per-batch lengths): token coordinates;
              // BHSD: (row, head)
              const RowAddr qa = VARLEN ? row_q(p, un.bh / p.Hq, un.h, un.q0)
                                        : RowAddr{un.q0, un.bh, 0, HEAD_DIM};
              mbar_arrive_expect_tx(qbar, 4 * Q_TILE * 128);
              tma_load_3d(smem_u32(s.Q), &tQ, 0, qa.c1, qa.c2, qbar);
              tma_load_3d(smem_u32(s.Q + Q_TILE * 128), &tQ, 64, qa.c1, qa.c2, qbar);
              tma_load_3d(smem_u32(s.dO), &tdO, 0, qa.c1, qa.c2, qbar);
              tma_load_3d(smem_u32(s.dO + Q_TILE * 128), &tdO, 64, qa.c1, qa.c2, qbar);
              q_loaded = j;
            }
          }
          if (u < 0) break;
          for (int n0 = 0; ok && n0 < un.walk.cnt; n0 += 32) {
            // lane l: step n0 + l
            int t = 0;
            uint32_t w = 0;
            if (n0 + lane < un.walk.cnt) {
              t = un.walk.tile(n0 + lane);
              if (blk_regions) {
                // the mask byte of each softmax warp's 32-query x 32-key region
                // (indices clamped into the mask, ranges applied after)
                const uint8_t* mb = p.mask + (size_t)un.bh * p.nqb * p.nkb;
                uint32_t mv[8];
#pragma unroll
                for (int sp2 = 0; sp2 < 4; ++sp2) {
                  const int qb = min((un.q0 + 32 * sp2) / p.bx, p.nqb - 1);
#pragma unroll
                  for (int g2 = 0; g2 < 2; ++g2) {
                    const int kb = min((t * Q_SUB + 32 * g2) / p.by, p.nkb - 1);
                    mv[2 * sp2 + g2] = mb[(size_t)qb * p.nkb + kb];
                  }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  if (mv[e] && un.q0 + 32 * (e >> 1) < p.Sq && t * Q_SUB + 32 * (e & 1) < p.Skv)
                    w |= 1u << e;
              }
            }
            const int cnt = min(32, un.walk.cnt - n0);
            for (int k = 0; k < cnt; ++k, ++m, rg.next()) {
              const int st = rg.st;
              const int tk = __shfl_sync(0xffffffffu, t, k);
              const uint32_t wk = __shfl_sync(0xffffffffu, w, k);
              if (m >= STAGES && !wait0(smem_u32(&s.bar_kv_empty[st]), rg.ph ^ 1u, TAG_KV_EMPTY)) {
                ok = false;
                break;
              }
              if (lane == 0) {
                s.step_t[st] = tk;  // published by the arrive below together with the loads
                s.step_vis[st] = wk;
                {
                  const uint32_t fb = smem_u32(&s.bar_kv_full[st]);
                  const RowAddr ka = VARLEN ? row_k(p, un.kvh / p.Hkv, un.kvh % p.Hkv, tk * Q_SUB)
                                            : RowAddr{tk * Q_SUB, un.kvh, 0, HEAD_DIM};
                  mbar_arrive_expect_tx(fb, 4 * Q_SUB * 128);
                  tma_load_3d(smem_u32(s.K[st]), &tK, 0, ka.c1, ka.c2, fb);
                  tma_load_3d(smem_u32(s.K[st] + Q_SUB * 128), &tK, 64, ka.c1, ka.c2, fb);
                  tma_load_3d(smem_u32(s.V[st]), &tV, 0, ka.c1, ka.c2, fb);
                  tma_load_3d(smem_u32(s.V[st] + Q_SUB * 128), &tV, 64, ka.c1, ka.c2, fb);
                }
              }
              __syncwarp();
            }
          }
        }
        if (!ok && lane == 0) {
          // the CTA gave up: let the copies still in flight land before it exits
          if (q_loaded >= 0) mbar_drain(qbar, q_loaded & 1, wc.timeout_ns);
          for (int k = m > STAGES ? m - STAGES : 0; k < m; ++k)
            mbar_drain(smem_u32(&s.bar_kv_full[k % STAGES]), (k / STAGES) & 1, wc.timeout_ns);
        }
      }
    }
  } else if (warp >= 1 && warp < SM_WARP0) {
    // ------------------------------------------------------------ MMA issuers (whole warps)
    constexpr uint32_t ID_S = idesc_f16(BF16, Q_TILE, Q_SUB, false, false);
    constexpr uint32_t ID_ACC = idesc_f16(BF16, Q_TILE, HEAD_DIM, false, true);
    bool ok = true;
    int m = 0;  // step counter across units
    Ring rg;
    if (warp == 1 || warp == 2) {
      // warp 1: S(m) = Q K^T into the S half of buffer m & 1; warp 2: dP(m) =
      // dO V^T into its dP half (A = Q / dO from TMEM, B = K / V tile, K-major)
      const bool is_s = warp == 1;
      const uint32_t a0 = tbase + (is_s ? COL_QA : COL_DOA);
      for (int j = 0; ok; ++j) {
        if (!mbar_wait_warp(smem_u32(&s.bar_q_full), j & 1, wc, TAG_Q)) break;
        const int u = s.unit;
        if (u < 0) break;
        DqUnit un{};
        un.template init<VARLEN>(p, u);
        const int N = un.walk.cnt;
        ok = mbar_wait_warp(smem_u32(&s.bar_qa_full), j & 1, wc, TAG_QA);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_unit_free));
        for (int n = 0; ok && n < N; ++n, ++m, rg.next()) {
          const int bf = m & 1, st = rg.st;
          ok = mbar_wait_warp(smem_u32(&s.bar_kv_full[st]), rg.ph, wc, TAG_KV_FULL);
          if (ok && m >= 2) {
            // S half: held dS(m - 2), read by dQ(m - 2); dP half: read by the
            // softmax warps before they signalled step m - 2
            ok = is_s ? mbar_wait_warp(smem_u32(&s.bar_acc_free[bf]), ((m - 2) >> 1) & 1, wc,
                                       TAG_ACC_FREE)
                      : mbar_wait_warp(smem_u32(&s.bar_p_full[bf]), ((m - 2) >> 1) & 1, wc,
                                       TAG_P_FULL);
          }
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tbase + COL_BUF + bf * 128 + (is_s ? 0 : 64);
          const uint64_t bB = sdesc_sw128(smem_u32(is_s ? s.K[st] : s.V[st]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < HEAD_DIM / 16; ++kk)
            mma_ts_w(d, a0 + 8 * kk,
                     bB + (uint64_t)(((kk >> 2) * (Q_SUB * 128) + (kk & 3) * 32) >> 4), ID_S,
                     kk > 0 ? 1u : 0u);
          mma_commit_w(smem_u32(&s.bar_s_full[bf]));
        }
      }
    } else {
      // dQ += dS(n) K (A = dS packed in buffer m & 1, B = K tile, MN-major)
      for (int j = 0; ok; ++j) {
        // the unit's first accumulation overwrites the accumulator: the
        // softmax warps must have read the previous unit's
        if (j >= 1 &&
            !mbar_wait_warp(smem_u32(&s.bar_acc_empty), (j - 1) & 1, wc, TAG_ACC_EMPTY))
          break;
        if (!mbar_wait_warp(smem_u32(&s.bar_q_full), j & 1, wc, TAG_Q)) break;
        const int u = s.unit;
        if (u < 0) break;
        DqUnit un{};
        un.template init<VARLEN>(p, u);
        const int N = un.walk.cnt;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_unit_free));
        for (int n = 0; ok && n < N; ++n, ++m, rg.next()) {
          const int bf = m & 1, st = rg.st;
          ok = mbar_wait_warp(smem_u32(&s.bar_p_full[bf]), (m >> 1) & 1, wc, TAG_P_FULL);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a = tbase + COL_BUF + bf * 128;
          const uint64_t bK = sdesc_sw128(smem_u32(s.K[st]), Q_SUB * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < Q_SUB / 16; ++kk)
            mma_ts_w(tbase + COL_ACC, a + 32 * (kk >> 1) + 8 * (kk & 1),
                     bK + (uint64_t)((kk * 2048) >> 4), ID_ACC, (n > 0 || kk > 0) ? 1u : 0u);
          if (HILO) {
#pragma unroll
            for (int kk = 0; kk < Q_SUB / 16; ++kk)
              mma_ts_w(tbase + COL_ACC, a + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                       bK + (uint64_t)((kk * 2048) >> 4), ID_ACC, 1u);
          }
          // S(m) and dP(m) completed before the softmax warps could signal
          // step m, so this commit also frees the K / V stage
          mma_commit_w(smem_u32(&s.bar_kv_empty[st]));
          mma_commit_w(smem_u32(&s.bar_acc_free[bf]));
        }
        if (ok) mma_commit_w(smem_u32(&s.bar_acc_full));  // the unit's accumulator is complete
      }
    }
    // this warp's MMAs must be complete before TMEM is freed (also when the
    // CTA gave up, hence a wait that ignores the abort flag)
    const uint32_t done = smem_u32(&s.bar_x_done[warp - 1]);
    mma_commit_w(done);
    mbar_drain_warp(done, 0, wc.timeout_ns);
  } else {
    // ------------------------------------------------------------ softmax warps
    const int sp = warp & 3, g = (warp - SM_WARP0) >> 2;
    const int rloc = sp * 32 + lane;
    const uint32_t lane_base = tbase + ((uint32_t)(sp * 32) << 16);
    uint8_t* stage = s.Q + (warp - SM_WARP0) * 4096;
    // Reads (or zero-fills) the accumulator of unit j, writes the unit's dQ
    // columns [64 g, 64 g + 64) of this warp's 32 rows and releases both the
    // accumulator and the staging space.
    auto epilogue = [&](int j, const DqUnit& un, bool ok) {
      uint32_t pk[32];
      const bool acc_ok = ok && mbar_wait(smem_u32(&s.bar_acc_full), j & 1, wc, TAG_ACC);
      const bool have = acc_ok && un.walk.cnt > 0;
      tc_fence_after();
      const int r0 = un.q0 + sp * 32;
      const int bq = un.bh / p.Hq;
      const RowAddr oa =
          VARLEN ? row_q(p, bq, un.h, r0)
                 : RowAddr{r0, un.bh, ((size_t)un.bh * p.Sq + r0) * HEAD_DIM, HEAD_DIM};
      const int nvalid = VARLEN ? rows_to_store_q(p, bq, r0) : min(32, p.Sq - r0);
      uint16_t* orow = dq + oa.elem + 64 * g;
      if (!__all_sync(0xffffffffu, acc_ok)) {
        // the CTA gave up: a copy may still be landing in the Q tile, so the
        // zeros go straight to global memory
        warp_zero_rows(orow, 64, nvalid, oa.stride);
        return;
      }
      if (have) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld32(lane_base + COL_ACC + 64 * g + 32 * half, v);
          tmem_wait_ld_regs(v);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[16 * half + c] = pack2<BF16>(v[2 * c] * p.scale, v[2 * c + 1] * p.scale);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = 0u;
      }
      // the accumulator is in registers: the next unit's first dQ MMA may
      // overwrite it while this warp stores the rows
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_acc_empty));
      warp_store_rows(stage, pk, orow, nvalid, oa.stride);
      // the next TMA load into the Q tile (after unit_free) comes after this
      // warp's generic accesses to it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    };
    bool ok = true;
    int m = 0;  // step counter across units
    Ring rg;
    DqUnit prev;
    int j = 0;
    for (; ok; ++j) {
      ok = mbar_wait(smem_u32(&s.bar_q_full), j & 1, wc, TAG_Q);
      const int u = ok ? s.unit : -1;
      if (u < 0) break;
      DqUnit un{};
      un.template init<VARLEN>(p, u);
      // this row's statistics, loaded now so that their latency passes while
      // the warp copies Q / dO and stores the previous unit
      const int i = un.q0 + rloc;
      const size_t srow = (size_t)un.bh * p.Sq_pad + i;
      const float nlse2_i = p.nlse2[srow];  // -lse log2(e)
      const float delta_i = p.delta[srow];
      // block masks: this row's mask row, found once per unit
      const uint8_t* rowM =
          BLOCK ? p.mask + ((size_t)un.bh * p.nqb + min(i, p.Sq - 1) / p.bx) * p.nkb : nullptr;
      // Q and dO rows of the unit into TMEM as 16-bit pairs (element 2c in
      // the low half of column c): this warp copies d columns
      // 64 g .. 64 g + 63 of its rows.  Every S / dP MMA of the previous unit
      // completed before its last step was signalled, so the columns are free.
      {
        const uint8_t* src[2] = {s.Q + g * (Q_TILE * 128) + rloc * 128,
                                 s.dO + g * (Q_TILE * 128) + rloc * 128};
        const uint32_t dst[2] = {COL_QA + 32u * g, COL_DOA + 32u * g};
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(src[which] + ((c ^ (rloc & 7)) << 4));
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
          }
          tmem_st32(lane_base + dst[which], w);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_qa_full));
      // the previous unit's epilogue overlaps this unit's first MMAs
      if (j >= 1) epilogue(j - 1, prev, ok);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.bar_unit_free));

      int flo, fhi;  // key sub-tiles that are entirely visible
      // keys past the batch's length are masked here; rows past its length
      // need no mask: their -lse log2 e is -inf, so their P and dS are 0
      const int Lk = VARLEN ? len_k(p, un.bh / p.Hq) : 0;
      full_range_q(p.mask_kind, p.window, p.Sq, VARLEN ? Lk : p.Skv, un.q0, &flo, &fhi);
      for (int n = 0; ok && n < un.walk.cnt; ++n, ++m, rg.next()) {
        const int bf = m & 1, st = rg.st;
        // s_full implies the stage's loads landed; waiting on kv_full as well
        // makes the step's tile index (written by the producer) visible
        // the step's tile index (and, block masks, the mask bytes its
        // visibility needs) are read while S and dP are still being computed
        if (!mbar_wait(smem_u32(&s.bar_kv_full[st]), rg.ph, wc, TAG_KV_FULL)) {
          ok = false;
          break;
        }
        const int t = s.step_t[st];
        // warp-uniform: the whole 128 x 64 sub-tile is visible
        const bool full = !BLOCK && t >= flo && t <= fhi;  // (block masks: never)
        uint32_t vis;
        if (full) {
          vis = 0xffffffffu;
        } else if (blk_regions) {
          vis = ((s.step_vis[st] >> (2 * sp + g)) & 1u) && i < p.Sq
                    ? bit_range(0, (VARLEN ? Lk : p.Skv) - 1 - (t * Q_SUB + 32 * g))
                    : 0u;
        } else {
          if constexpr (BLOCK) {
            // row i against keys j0 .. j0 + 31; the key-block quotient by a
            // reciprocal
            const int j0 = t * Q_SUB + 32 * g;
            const int jend = min(j0 + 31, (VARLEN ? Lk : p.Skv) - 1);
            uint32_t bits = 0;
            if (i < p.Sq && jend >= j0) {
              for (int kb = div_by(j0, p.by, p.inv_by); kb * p.by <= jend; ++kb)
                if (rowM[kb]) bits |= bit_range(kb * p.by - j0, (kb + 1) * p.by - 1 - j0);
              bits &= bit_range(0, jend - j0);
            }
            vis = bits;
          } else {
            vis = vis_query_row_closed<MK>(p, i, t * Q_SUB + 32 * g, p.Sq, VARLEN ? Lk : p.Skv);
          }
        }
        if constexpr (!VARLEN) {
          // no key of the warp's region is visible for any of its rows: dS is
          // zero, written without loading S or dP once both MMAs completed
          // (not in the per-batch-length instances, whose registers are at
          // their limit)
          if (!full && __all_sync(0xffffffffu, vis == 0u)) {
            if (!mbar_wait(smem_u32(&s.bar_s_full[bf]), (m >> 1) & 1, wc, TAG_S_FULL)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint32_t z[HILO ? 32 : 16];
#pragma unroll
            for (int c = 0; c < (HILO ? 32 : 16); ++c) z[c] = 0u;
            if constexpr (HILO)
              tmem_st32(lane_base + COL_BUF + bf * 128 + 32 * g, z);
            else
              tmem_st16(lane_base + COL_BUF + bf * 128 + 32 * g, z);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.bar_p_full[bf]));
            continue;
          }
        }
        if (!mbar_wait(smem_u32(&s.bar_s_full[bf]), (m >> 1) & 1, wc, TAG_S_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col = COL_BUF + bf * 128 + 32 * g;
        // every key of the region visible for every row: no masking
        const bool fullw = full || (!VARLEN && __all_sync(0xffffffffu, vis == 0xffffffffu));
        float sv[32], dp[32];
        tmem_ld32(lane_base + col, sv);
        tmem_ld32(lane_base + col + 64, dp);
        tmem_wait_ld_regs(sv);
#pragma unroll
        for (int c = 0; c < 32; ++c) asm volatile("" : "+f"(dp[c]));
        uint32_t pk[HILO ? 32 : 16];
        // packs dS of keys 2c, 2c + 1 (and, compensated, the remainder)
        auto put = [&](int c, float d0, float d1) {
          pk[c] = pack2<BF16>(d0, d1);
          if (HILO) {
            const float2 h = unpack2<BF16>(pk[c]);
            pk[(HILO ? 16 : 0) + c] = pack2<BF16>(d0 - h.x, d1 - h.y);
          }
        };
        if (fullw) {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float p0 = fast_exp2(fmaf(sv[2 * c], p.scale_log2, nlse2_i));
            const float p1 = fast_exp2(fmaf(sv[2 * c + 1], p.scale_log2, nlse2_i));
            put(c, p0 * (dp[2 * c] - delta_i), p1 * (dp[2 * c + 1] - delta_i));
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            float p0 = fast_exp2(fmaf(sv[2 * c], p.scale_log2, nlse2_i));
            float p1 = fast_exp2(fmaf(sv[2 * c + 1], p.scale_log2, nlse2_i));
            p0 = ((vis >> (2 * c)) & 1u) ? p0 : 0.f;
            p1 = ((vis >> (2 * c + 1)) & 1u) ? p1 : 0.f;
            put(c, p0 * (dp[2 * c] - delta_i), p1 * (dp[2 * c + 1] - delta_i));
          }
        }
        if constexpr (HILO)
          tmem_st32(lane_base + col, pk);
        else
          tmem_st16(lane_base + col, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_p_full[bf]));
      }
      prev = un;
    }
    if (j >= 1) epilogue(j - 1, prev, ok);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // launched to overlap the dK/dV grid's tail: one thread of one CTA keeps
  // this grid from completing before that one has, so whatever follows on the
  // stream sees both complete, while every other CTA frees its SM at once
  // (for kernels of other streams too)
  if (blockIdx.x == 0 && threadIdx.x == 0) grid_dependency_wait();
}

cudaError_t launch_dq(bool bf16, const AttnParams& p, const CUtensorMap& tQ, const CUtensorMap& tdO,
                      const CUtensorMap& tK, const CUtensorMap& tV, void* dq, cudaStream_t st) {
  const bool varlen = p.seqlen_q != nullptr || p.seqlen_k != nullptr || p.cu_q != nullptr;
  using Kern = decltype(&k_dq<true, false, false, MK_NONE>);
#define MAB_DQ_ROW(BF, VL, HL)                                                                  \
  {k_dq<BF, VL, HL, MK_NONE>, k_dq<BF, VL, HL, MK_CAUSAL>, k_dq<BF, VL, HL, MK_SLIDING>,       \
   k_dq<BF, VL, HL, MK_BLOCK>}
  static const Kern table[2][2][2][4] = {
      {{MAB_DQ_ROW(false, false, false), MAB_DQ_ROW(false, false, true)},
       {MAB_DQ_ROW(false, true, false), MAB_DQ_ROW(false, true, true)}},
      {{MAB_DQ_ROW(true, false, false), MAB_DQ_ROW(true, false, true)},
       {MAB_DQ_ROW(true, true, false), MAB_DQ_ROW(true, true, true)}}};
#undef MAB_DQ_ROW
  const Kern kern = table[bf16 ? 1 : 0][varlen ? 1 : 0][p.compensated ? 1 : 0][p.mask_kind];
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)dq_side::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int units = p.nQT_q * p.B * p.Hq;
  // programmatic stream serialization: the grid may start while the dK/dV
  // grid before it finishes (this one reads none of that grid's outputs)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units < sms ? units : sms));
  cfg.blockDim = dim3(dq_side::NUM_THREADS);
  cfg.dynamicSmemBytes = dq_side::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tQ, tdO, tK, tV, (uint16_t*)dq, p);
}

}  // namespace mab
