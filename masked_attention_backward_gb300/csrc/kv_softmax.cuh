// kv_softmax.cuh -- the softmax warps' arithmetic of one step of the
// key-stationary walk, shared by the dK/dV kernels (per-tile and persistent)
// and the single-pass kernel.
//
// A softmax warp owns 32 key rows (TMEM lanes) and 16 query columns of the
// step's 128-key x 64-query tile.  From its fp32 S^T values it forms
//   P^T  = exp2(S^T * scale*log2e + nlse2)   (nlse2 = -lse log2 e per query)
// and from its fp32 dP^T values
//   dS^T = P^T (dP^T - Delta),
// writing each packed to 16-bit pairs over the first 8 of its own columns
// (and, compensated, the remainder value - high part over the next 8).
// Sources: cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook,
// precision notes (p = exp(s - lse), ds = p (dp - delta)).
#pragma once
#include <math.h>

#include "tiles.cuh"

namespace mab {

// 16 consecutive floats from shared memory (16-byte aligned), as 4 vector loads.
__device__ __forceinline__ void load16_shared(const float* src, float (&v)[16]) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 x = s4[q];
    v[4 * q] = x.x;
    v[4 * q + 1] = x.y;
    v[4 * q + 2] = x.z;
    v[4 * q + 3] = x.w;
  }
}

// P^T of the warp's 16 columns from the loaded S^T values sv (invisible ones
// masked to -inf unless `full`): returns P in pv and writes it, packed, at
// TMEM address `taddr` (the warp's first S^T column), then waits for the
// store.
template <bool BF16, bool HILO>
__device__ __forceinline__ void kv_write_p(uint32_t taddr, float (&sv)[16], const float (&lv)[16],
                                           bool full, uint32_t vis, float scale_log2,
                                           float (&pv)[16]) {
  // an invisible logit becomes -inf, so its P is 0 (and so is its dS)
  if (!full) {
#pragma unroll
    for (int cc = 0; cc < 16; ++cc) sv[cc] = ((vis >> cc) & 1u) ? sv[cc] : -INFINITY;
  }
  const float2 sc2 = make_float2(scale_log2, scale_log2);
  uint32_t pk[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float2 x = ffma2(make_float2(sv[2 * q], sv[2 * q + 1]), sc2,
                           make_float2(lv[2 * q], lv[2 * q + 1]));
    pv[2 * q] = fast_exp2(x.x);
    pv[2 * q + 1] = fast_exp2(x.y);
    pk[q] = pack2<BF16>(pv[2 * q], pv[2 * q + 1]);
  }
  // over this warp's own S^T columns, which it has just loaded
  tmem_st8(taddr, pk);
  if constexpr (HILO) {
    uint32_t pl[8];  // remainders P - high part
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float2 h = unpack2<BF16>(pk[q]);
      pl[q] = pack2<BF16>(pv[2 * q] - h.x, pv[2 * q + 1] - h.y);
    }
    tmem_st8(taddr + 8, pl);
  }
  tmem_wait_st();
}

// dS^T = P^T (dP^T - Delta) of the warp's 16 columns, written packed at TMEM
// address `taddr` (the warp's first dP^T column); the packed high parts are
// also returned in pk.  Waits for the store.
template <bool BF16, bool HILO>
__device__ __forceinline__ void kv_write_ds(uint32_t taddr, const float (&pv)[16], float (&dp)[16],
                                            const float (&dl)[16], uint32_t (&pk)[8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float2 ds = fmul2(make_float2(pv[2 * q], pv[2 * q + 1]),
                            fsub2(make_float2(dp[2 * q], dp[2 * q + 1]),
                                  make_float2(dl[2 * q], dl[2 * q + 1])));
    pk[q] = pack2<BF16>(ds.x, ds.y);
    if (HILO) {
      dp[2 * q] = ds.x;
      dp[2 * q + 1] = ds.y;
    }
  }
  tmem_st8(taddr, pk);
  if constexpr (HILO) {
    uint32_t pl[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float2 h = unpack2<BF16>(pk[q]);
      pl[q] = pack2<BF16>(dp[2 * q] - h.x, dp[2 * q + 1] - h.y);
    }
    tmem_st8(taddr + 8, pl);
  }
  tmem_wait_st();
}

}  // namespace mab
