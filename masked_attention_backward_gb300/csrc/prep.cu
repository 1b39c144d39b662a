// prep.cu -- the memory-bound steps before the two contraction kernels:
//   k_preprocess      Delta = rowsum(dO * O), nlse2 = -lse * log2(e) (padded),
//                     and per-block partial sums of exp(sink - lse) * Delta;
//   k_dsink_finalize  dSink_h = -(fixed-order sum of the partials);
//   k_mask_tables     uint8 block mask [BH,nQB,nKB] -> [BH,nKB,nQB] (transpose)
//                     and the select tables: per key tile the ascending list
//                     of query sub-tiles that share an active block, and vice
//                     versa (one launch).
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
             const int* __restrict__ cu_q, int total_q, DevStatus* __restrict__ status) {
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
  // the call's status word starts at zero: every kernel that reads or writes
  // it runs after this grid has completed (in stream order, or behind a wait
  // for this grid), and the table kernel beside it does not touch it
  if (blk == 0 && bh == 0 && threadIdx.x < sizeof(DevStatus) / sizeof(unsigned int))
    reinterpret_cast<unsigned int*>(status)[threadIdx.x] = 0u;
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
  // Behind the mask-table kernel (block masks) this grid is launched with
  // programmatic serialization and runs beside it: one thread keeps this grid
  // from completing before that one has, so the kernels waiting for this
  // grid see both complete (a no-op after an ordinary launch).
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) grid_dependency_wait();
}

__global__ void k_dsink_finalize(const float* __restrict__ part, int nparts,
                                 float* __restrict__ dsink) {
  const int h = blockIdx.x, lane = threadIdx.x;
  const float v = dsink_of_head(part, nparts, h, lane);
  if (lane == 0) dsink[h] = v;
}

// Transpose of one 32 x 32 tile of query blocks x key blocks of one (b, h)
// through shared memory (128 threads: 32 columns x 4 rows at a time).
__device__ void transpose_tile(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int nqb,
                               int nkb, int qb0, int kb0) {
  __shared__ uint8_t tile[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int r = ty; r < 32; r += 4) {
    const int qb = qb0 + r, kb = kb0 + tx;
    if (qb < nqb && kb < nkb) tile[r][tx] = src[(size_t)qb * nkb + kb];
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 4) {
    const int kb = kb0 + r, qb = qb0 + tx;
    if (qb < nqb && kb < nkb) dst[(size_t)kb * nqb + qb] = tile[tx][r];
  }
}

// One warp per table row.  The row's own tile covers [o0, o1) on its axis;
// candidate partner tile t covers [t*psize, min((t+1)*psize, plen)).  A pair
// is active when some mask block with a nonzero byte overlaps both ranges.
// The mask byte of (own block ob, partner block pb) is
// m[ob * own_stride + pb * part_stride] (the (b, h) mask read along either
// axis).  Entries are written at the exclusive prefix count of active
// candidates (warp ballot + popc).
__device__ void build_row(const uint8_t* __restrict__ m, size_t own_stride, size_t part_stride,
                          int own_bs, int part_bs, int o0, int o1, int psize, int plen,
                          int* __restrict__ sel_row, int nP, int* __restrict__ cnt) {
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
        const uint8_t* r = m + (size_t)ob * own_stride;
        for (int pb = pb_lo; pb <= pb_hi; ++pb)
          if (r[(size_t)pb * part_stride]) {
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

// Both mask steps in one launch of 128-thread blocks: the first n_tr blocks
// transpose the mask (32 x 32 tiles; the key-stationary kernels read the
// transposed rows), the rest build the select tables, one warp per row: first
// BH*nKT_k key-major rows, then BH*nQT_q query-major rows.  The tables read
// the mask itself along either axis, so neither part waits for the other.
__global__ void __launch_bounds__(128)
k_mask_tables(const AttnParams p, uint8_t* __restrict__ maskT, int n_tr, int* __restrict__ sel_k,
              int* __restrict__ cnt_k, int* __restrict__ sel_q, int* __restrict__ cnt_q) {
  // the preprocess grid behind this one reads nothing of it: let it start
  grid_launch_dependents();
  const int BH = p.B * p.Hq;
  const size_t per_head = (size_t)p.nqb * p.nkb;
  if ((int)blockIdx.x < n_tr) {
    const int tk = (p.nkb + 31) / 32, tq = (p.nqb + 31) / 32;
    const int bh = blockIdx.x / (tk * tq), rem = blockIdx.x % (tk * tq);
    transpose_tile(p.mask + bh * per_head, maskT + bh * per_head, p.nqb, p.nkb, (rem / tk) * 32,
                   (rem % tk) * 32);
    return;
  }
  const int gw = (blockIdx.x - n_tr) * 4 + (threadIdx.x >> 5);
  const int nk_rows = BH * p.nKT_k;
  if (gw < nk_rows) {
    int bh = gw / p.nKT_k, kt = gw % p.nKT_k;
    int o0 = kt * KV_TILE, o1 = min(o0 + KV_TILE, p.Skv);
    build_row(p.mask + bh * per_head, 1, p.nkb, p.by, p.bx, o0, o1, KV_SUB, p.Sq,
              sel_k + (size_t)gw * p.nQT_k, p.nQT_k, cnt_k + gw);
  } else if (gw < nk_rows + BH * p.nQT_q) {
    int r = gw - nk_rows;
    int bh = r / p.nQT_q, qt = r % p.nQT_q;
    int o0 = qt * Q_TILE, o1 = min(o0 + Q_TILE, p.Sq);
    build_row(p.mask + bh * per_head, p.nkb, 1, p.bx, p.by, o0, o1, Q_SUB, p.Skv,
              sel_q + (size_t)r * p.nKT_q, p.nKT_q, cnt_q + r);
  }
}

cudaError_t launch_preprocess(bool bf16, const void* O, const void* dO, const float* lse,
                              const float* sink, float* nlse2, float* delta, float* part, int B,
                              int Hq, int Sq, int Sq_pad, const int* seqlen_q, const int* cu_q,
                              int total_q, DevStatus* status, bool overlap_prev, cudaStream_t st) {
  const int nparts = B * (Sq_pad / PREP_BLOCK_ROWS);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Sq_pad / PREP_BLOCK_ROWS, B * Hq);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_prev ? 1 : 0;
  const uint4* o4 = (const uint4*)O;
  const uint4* d4 = (const uint4*)dO;
  return bf16 ? cudaLaunchKernelEx(&cfg, k_preprocess<true>, o4, d4, lse, sink, nlse2, delta, part,
                                   Hq, Sq, Sq_pad, nparts, seqlen_q, cu_q, total_q, status)
              : cudaLaunchKernelEx(&cfg, k_preprocess<false>, o4, d4, lse, sink, nlse2, delta,
                                   part, Hq, Sq, Sq_pad, nparts, seqlen_q, cu_q, total_q, status);
}

cudaError_t launch_dsink_finalize(const float* part, int Hq, int nparts, float* dsink,
                                  cudaStream_t st) {
  k_dsink_finalize<<<Hq, 32, 0, st>>>(part, nparts, dsink);
  return cudaGetLastError();
}

cudaError_t launch_mask_tables(const AttnParams& p, uint8_t* maskT, int* sel_k, int* cnt_k,
                               int* sel_q, int* cnt_q, cudaStream_t st) {
  const long long BH = (long long)p.B * p.Hq;
  const long long n_tr = BH * ((p.nkb + 31) / 32) * ((p.nqb + 31) / 32);
  const long long rows = BH * ((long long)p.nKT_k + p.nQT_q);
  const long long blocks = n_tr + (rows + 3) / 4;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  k_mask_tables<<<(unsigned)blocks, 128, 0, st>>>(p, maskT, (int)n_tr, sel_k, cnt_k, sel_q, cnt_q);
  return cudaGetLastError();
}

}  // namespace mab
