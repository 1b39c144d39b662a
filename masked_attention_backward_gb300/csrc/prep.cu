// prep.cu -- the memory-bound steps before the two contraction kernels:
//   k_preprocess      Delta = rowsum(dO * O), nlse2 = -lse * log2(e) (padded),
//                     and per-block partial sums of exp(sink - lse) * Delta;
//   k_dsink_finalize  dSink_h = -(fixed-order sum of the partials);
//   k_mask_transpose  uint8 block mask [BH,nQB,nKB] -> [BH,nKB,nQB];
//   k_build_sel       select tables: per key tile the ascending list of query
//                     sub-tiles that share an active block, and vice versa.
//
// Sources: tilelang-ascend PR #1 "Add GQA Sink Backward BHSD", commit notes of
// the 2-kernel design (Phase0 Delta = sum(O*dO); Phase5 dSink);
// cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook, optimisation 1
// (tables built on the device by an exclusive prefix count of kept entries,
// no dense token mask on the host) and optimisation 2 (transpose the uint8
// mask on the device once, then read only contiguous rows).
#include <math.h>

#include "internal.h"

namespace mab {

// One block = PREP_BLOCK_ROWS rows of one (b, h).  Each half-warp owns a row:
// 16 lanes x 16 bytes cover the 128-element row of O and of dO, so every warp
// load is a fully coalesced 512-byte request.  A thread holds 4 rows of each
// in flight; small blocks keep several per SM resident, so that one block's
// loads are in flight while another reduces and exits.
template <bool BF16>
__global__ void __launch_bounds__(256, 4)
k_preprocess(const uint4* __restrict__ O, const uint4* __restrict__ dO,
             const float* __restrict__ lse, const float* __restrict__ sink,
             float* __restrict__ nlse2, float* __restrict__ delta, float* __restrict__ part, int Hq,
             int Sq, int Sq_pad, int nparts, const int* __restrict__ seqlen_q,
             const int* __restrict__ cu_q, int total_q) {
  constexpr int ROWS_PER_WARP = PREP_BLOCK_ROWS / 8;  // 8
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const int blk = blockIdx.x, bh = blockIdx.y;
  const int h = bh % Hq, b = bh / Hq;
  const int row0 = blk * PREP_BLOCK_ROWS + warp * ROWS_PER_WARP;
  const size_t head_rows = (size_t)bh * Sq;
  // the dK/dV kernel behind this one (launched with programmatic
  // serialization) may be scheduled once every block of this grid has
  // started; it waits for this grid's completion before it reads any result
  grid_launch_dependents();
  // rows past the batch's length are outside the problem: treated like the
  // padding (Delta 0, -lse log2 e = -inf, no dSink term)
  const int Lq = cu_q ? packed_len(cu_q, b, total_q, Sq)
                      : (seqlen_q ? min(max(seqlen_q[b], 0), Sq) : Sq);
  // BHSD: row r of (b, h) is row bh * Sq + r of O and dO, lse [B*Hq, Sq];
  // packed: token cu_q[b] + r of the token-major O and dO, lse [Hq, total_q]
  const int off = cu_q ? packed_off(cu_q, b, total_q) : 0;
  auto row_elem16 = [&](int row) -> size_t {  // uint4 index of a row's first element
    return cu_q ? ((size_t)(off + row) * Hq + h) * 16 : (head_rows + row) * 16;
  };
  auto lse_index = [&](int row) -> size_t {
    return cu_q ? (size_t)h * total_q + off + row : head_rows + row;
  };

  uint4 vo[ROWS_PER_WARP / 2], vd[ROWS_PER_WARP / 2];
#pragma unroll
  for (int it = 0; it < ROWS_PER_WARP / 2; ++it) {
    int row = row0 + it * 2 + half;
    if (row < Lq) {
      size_t idx = row_elem16(row) + l16;
      vo[it] = __ldg(O + idx);
      vd[it] = __ldg(dO + idx);
    } else {
      vo[it] = make_uint4(0, 0, 0, 0);
      vd[it] = make_uint4(0, 0, 0, 0);
    }
  }
  const float sink2 = sink ? sink[h] * LOG2E : -INFINITY;
  float term_acc = 0.f;
#pragma unroll
  for (int it = 0; it < ROWS_PER_WARP / 2; ++it) {
    const uint32_t* po = reinterpret_cast<const uint32_t*>(&vo[it]);
    const uint32_t* pd = reinterpret_cast<const uint32_t*>(&vd[it]);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 a = unpack2<BF16>(po[e]), c = unpack2<BF16>(pd[e]);
      acc = fmaf(a.x, c.x, acc);
      acc = fmaf(a.y, c.y, acc);
    }
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    int row = row0 + it * 2 + half;
    if (l16 == 0) {
      size_t o = (size_t)bh * Sq_pad + row;
      if (row < Lq) {
        float l2 = lse[lse_index(row)] * LOG2E;
        delta[o] = acc;
        nlse2[o] = -l2;
        if (sink) term_acc += exp2f(sink2 - l2) * acc;
      } else {
        delta[o] = 0.f;
        nlse2[o] = -INFINITY;
      }
    }
  }
  if (sink) {
    // lanes 0 and 16 hold the per-warp sums of their rows; fixed-order reduction
    float t = term_acc + __shfl_xor_sync(0xffffffffu, term_acc, 16);
    __shared__ float wsum[8];
    if (lane == 0) wsum[warp] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
      for (int w = 0; w < 8; ++w) s += wsum[w];
      part[(size_t)h * nparts + (size_t)b * gridDim.x + blk] = s;
    }
  }
}

__global__ void k_dsink_finalize(const float* __restrict__ part, int nparts,
                                 float* __restrict__ dsink) {
  const int h = blockIdx.x, lane = threadIdx.x;
  double s = 0.0;
  for (int i = lane; i < nparts; i += 32) s += (double)part[(size_t)h * nparts + i];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) dsink[h] = (float)(-s);
}

// 32x32 byte tiles through shared memory.
__global__ void k_mask_transpose(const uint8_t* __restrict__ mask, uint8_t* __restrict__ maskT,
                                 int BH, int nqb, int nkb) {
  __shared__ uint8_t tile[32][33];
  const int kb0 = blockIdx.x * 32, qb0 = blockIdx.y * 32;
  for (int bh = blockIdx.z; bh < BH; bh += gridDim.z) {
    const uint8_t* src = mask + (size_t)bh * nqb * nkb;
    uint8_t* dst = maskT + (size_t)bh * nqb * nkb;
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
      int qb = qb0 + r, kb = kb0 + threadIdx.x;
      if (qb < nqb && kb < nkb) tile[r][threadIdx.x] = src[(size_t)qb * nkb + kb];
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
      int kb = kb0 + r, qb = qb0 + threadIdx.x;
      if (qb < nqb && kb < nkb) dst[(size_t)kb * nqb + qb] = tile[threadIdx.x][r];
    }
    __syncthreads();
  }
}

// One warp per table row.  The row's own tile covers [o0, o1) on its axis;
// candidate partner tile t covers [t*psize, min((t+1)*psize, plen)).  A pair
// is active when some mask block with a nonzero byte overlaps both ranges.
// `rows` points at the mask rows of this (b,h) laid out [own block][partner
// block] (maskT for key-major walks, the mask itself for query-major walks),
// so each probe reads a contiguous run of bytes.  Entries are written at the
// exclusive prefix count of active candidates (warp ballot + popc).
__device__ void build_row(const uint8_t* __restrict__ rows, int npb, int own_bs, int part_bs,
                          int o0, int o1, int psize, int plen, int* __restrict__ sel_row,
                          int nP, int* __restrict__ cnt) {
  const int lane = threadIdx.x & 31;
  const int ob_lo = o0 / own_bs, ob_hi = (o1 - 1) / own_bs;
  int n = 0;
  for (int base = 0; base < nP; base += 32) {
    int t = base + lane;
    bool act = false;
    if (t < nP) {
      int p0 = t * psize, p1 = min(p0 + psize, plen);
      int pb_lo = p0 / part_bs, pb_hi = (p1 - 1) / part_bs;
      for (int ob = ob_lo; ob <= ob_hi && !act; ++ob) {
        const uint8_t* r = rows + (size_t)ob * npb;
        for (int pb = pb_lo; pb <= pb_hi; ++pb)
          if (r[pb]) {
            act = true;
            break;
          }
      }
    }
    unsigned bal = __ballot_sync(0xffffffffu, act);
    if (act) sel_row[n + __popc(bal & ((1u << lane) - 1u))] = t;
    n += __popc(bal);
  }
  for (int t = n + lane; t < nP; t += 32) sel_row[t] = -1;
  if (lane == 0) *cnt = n;
}

// grid.x covers rows of both tables: first BH*nKT_k key-major rows, then
// BH*nQT_q query-major rows; 4 warps per block.
__global__ void k_build_sel(AttnParams p, int* __restrict__ sel_k, int* __restrict__ cnt_k,
                            int* __restrict__ sel_q, int* __restrict__ cnt_q) {
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int BH = p.B * p.Hq;
  const int nk_rows = BH * p.nKT_k;
  if (gw < nk_rows) {
    int bh = gw / p.nKT_k, kt = gw % p.nKT_k;
    int o0 = kt * KV_TILE, o1 = min(o0 + KV_TILE, p.Skv);
    build_row(p.maskT + (size_t)bh * p.nkb * p.nqb, p.nqb, p.by, p.bx, o0, o1, KV_SUB, p.Sq,
              sel_k + (size_t)gw * p.nQT_k, p.nQT_k, cnt_k + gw);
  } else if (gw < nk_rows + BH * p.nQT_q) {
    int r = gw - nk_rows;
    int bh = r / p.nQT_q, qt = r % p.nQT_q;
    int o0 = qt * Q_TILE, o1 = min(o0 + Q_TILE, p.Sq);
    build_row(p.mask + (size_t)bh * p.nqb * p.nkb, p.nkb, p.bx, p.by, o0, o1, Q_SUB, p.Skv,
              sel_q + (size_t)r * p.nKT_q, p.nKT_q, cnt_q + r);
  }
}

cudaError_t launch_preprocess(bool bf16, const void* O, const void* dO, const float* lse,
                              const float* sink, float* nlse2, float* delta, float* part, int B,
                              int Hq, int Sq, int Sq_pad, const int* seqlen_q, const int* cu_q,
                              int total_q, cudaStream_t st) {
  dim3 grid(Sq_pad / PREP_BLOCK_ROWS, B * Hq);
  int nparts = B * (Sq_pad / PREP_BLOCK_ROWS);
  if (bf16)
    k_preprocess<true><<<grid, 256, 0, st>>>((const uint4*)O, (const uint4*)dO, lse, sink, nlse2,
                                              delta, part, Hq, Sq, Sq_pad, nparts, seqlen_q, cu_q, total_q);
  else
    k_preprocess<false><<<grid, 256, 0, st>>>((const uint4*)O, (const uint4*)dO, lse, sink, nlse2,
                                               delta, part, Hq, Sq, Sq_pad, nparts, seqlen_q, cu_q, total_q);
  return cudaGetLastError();
}

cudaError_t launch_dsink_finalize(const float* part, int Hq, int nparts, float* dsink,
                                  cudaStream_t st) {
  k_dsink_finalize<<<Hq, 32, 0, st>>>(part, nparts, dsink);
  return cudaGetLastError();
}

cudaError_t launch_mask_transpose(const uint8_t* mask, uint8_t* maskT, int BH, int nqb, int nkb,
                                  cudaStream_t st) {
  dim3 grid((nkb + 31) / 32, (nqb + 31) / 32, BH < 65535 ? BH : 65535);
  k_mask_transpose<<<grid, dim3(32, 8), 0, st>>>(mask, maskT, BH, nqb, nkb);
  return cudaGetLastError();
}

cudaError_t launch_build_sel(const AttnParams& p, int* sel_k, int* cnt_k, int* sel_q, int* cnt_q,
                             cudaStream_t st) {
  long long rows = (long long)p.B * p.Hq * ((long long)p.nKT_k + p.nQT_q);
  int blocks = (int)((rows + 3) / 4);
  k_build_sel<<<blocks, 128, 0, st>>>(p, sel_k, cnt_k, sel_q, cnt_q);
  return cudaGetLastError();
}

}  // namespace mab
