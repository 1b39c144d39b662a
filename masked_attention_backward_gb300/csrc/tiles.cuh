// tiles.cuh -- device helpers shared by the contraction kernels: per-thread
// visibility bitmasks for 32 consecutive partner positions, the walk over
// active partner tiles (closed form for causal / sliding / none, select tables
// for block masks), and a coalesced per-warp row store.
#pragma once
#include "internal.h"

namespace mab {

// a / b for 0 <= a < 2^24 and b >= 1, given inv_b = 1 / b rounded to float:
// the float quotient is within 2 / b of a / b (exact for b = 1, 2), so one
// correction each way gives the exact floor.
__device__ __forceinline__ int div_by(int a, int b, float inv_b) {
  int q = __float2int_rz((float)a * inv_b);
  q += (q + 1) * b <= a ? 1 : 0;
  q -= q * b > a ? 1 : 0;
  return q;
}

// Bits [lo, hi] (inclusive, clipped to [0, 31]) set.
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
  if (lo < 0) lo = 0;
  if (hi > 31) hi = 31;
  if (hi < lo) return 0u;
  uint32_t upper = (hi == 31) ? 0xffffffffu : ((1u << (hi + 1)) - 1u);
  return upper & ~((1u << lo) - 1u);
}

// Query row i against keys j0 .. j0+31 (bit c <-> key j0 + c); Lq, Lk are
// the valid rows and keys of the row's batch.
__device__ __forceinline__ uint32_t vis_query_row(const AttnParams& p, int bh, int i, int j0,
                                                  int Lq, int Lk) {
  if (i >= Lq) return 0u;
  uint32_t inrange = bit_range(0, Lk - 1 - j0);
  switch (p.mask_kind) {
    case MK_NONE:
      return inrange;
    case MK_CAUSAL:
      return inrange & bit_range(0, i - j0);
    case MK_SLIDING:
      return inrange & bit_range(i - p.window + 1 - j0, i - j0);
    default: {
      const uint8_t* row = p.mask + ((size_t)bh * p.nqb + i / p.bx) * p.nkb;
      int jend = min(j0 + 31, Lk - 1);
      if (jend < j0) return 0u;
      uint32_t m = 0;
      for (int kb = j0 / p.by; kb * p.by <= jend; ++kb)
        if (row[kb]) m |= bit_range(kb * p.by - j0, (kb + 1) * p.by - 1 - j0);
      return m & inrange;
    }
  }
}

// Key row j against queries i0 .. i0+31 (bit c <-> query i0 + c); Lq, Lk
// are the valid rows and keys of the batch.
__device__ __forceinline__ uint32_t vis_key_row(const AttnParams& p, int bh, int j, int i0,
                                                int Lq, int Lk) {
  if (j >= Lk) return 0u;
  uint32_t inrange = bit_range(0, Lq - 1 - i0);
  switch (p.mask_kind) {
    case MK_NONE:
      return inrange;
    case MK_CAUSAL:
      return inrange & bit_range(j - i0, 31);
    case MK_SLIDING:
      return inrange & bit_range(j - i0, j + p.window - 1 - i0);
    default: {
      const uint8_t* row = p.maskT + ((size_t)bh * p.nkb + j / p.by) * p.nqb;
      int iend = min(i0 + 31, Lq - 1);
      if (iend < i0) return 0u;
      uint32_t m = 0;
      for (int qb = i0 / p.bx; qb * p.bx <= iend; ++qb)
        if (row[qb]) m |= bit_range(qb * p.bx - i0, (qb + 1) * p.bx - 1 - i0);
      return m & inrange;
    }
  }
}

// The closed-form half of vis_key_row, for instances that know the mask kind
// (16 queries: the dK/dV softmax warps' share).  Keeping the other kinds'
// code out of the softmax loop measured 3 to 4 % faster on short walks in the
// persistent dK/dV kernel.
template <int MK>
__device__ __forceinline__ uint32_t vis_key_row_closed(const AttnParams& p, int j, int i0, int Lq,
                                                       int Lk) {
  if (j >= Lk) return 0u;
  const uint32_t inrange = bit_range(0, Lq - 1 - i0);
  if constexpr (MK == MK_NONE) return inrange;
  else if constexpr (MK == MK_CAUSAL) return inrange & bit_range(j - i0, 31);
  else return inrange & bit_range(j - i0, j + p.window - 1 - i0);
}
// The closed-form half of vis_query_row, for instances that know the mask
// kind (32 keys: a dQ softmax warp's share).
template <int MK>
__device__ __forceinline__ uint32_t vis_query_row_closed(const AttnParams& p, int i, int j0,
                                                         int Lq, int Lk) {
  if (i >= Lq) return 0u;
  const uint32_t inrange = bit_range(0, Lk - 1 - j0);
  if constexpr (MK == MK_NONE) return inrange;
  else if constexpr (MK == MK_CAUSAL) return inrange & bit_range(0, i - j0);
  else return inrange & bit_range(i - p.window + 1 - j0, i - j0);
}

// The sub-tiles of a walk that are entirely visible form one contiguous
// range [lo, hi] of partner tile indices under the closed-form masks (empty,
// hi < lo, for block masks, whose tiles always take the per-element path).
// Computed once per CTA, so that a step decides with two compares.
//
// Key-tile CTA [k0, k0 + KV_TILE) against query sub-tiles r of KV_SUB rows:
// every (i, j) with i in [r KV_SUB, r KV_SUB + KV_SUB), j in [k0, k0 + KV_TILE)
// must exist (i < Sq, j < Skv) and, causal / sliding, satisfy j <= i
// (r KV_SUB >= k0 + KV_TILE - 1) and, sliding, i - j < window
// (r KV_SUB + KV_SUB - 1 - k0 <= window - 1).
__host__ __device__ inline void full_range_kv(int kind, int window, int Sq, int Skv, int k0,
                                              int* lo, int* hi) {
  *lo = 0;
  *hi = Sq / KV_SUB - 1;  // r KV_SUB + KV_SUB <= Sq
  if (kind == MK_BLOCK || k0 + KV_TILE > Skv) *hi = -1;
  if (kind == MK_CAUSAL || kind == MK_SLIDING) *lo = (k0 + KV_TILE - 1 + KV_SUB - 1) / KV_SUB;
  if (kind == MK_SLIDING) {
    const int top = window + k0 - KV_SUB;  // r KV_SUB <= top
    const int h = top < 0 ? -1 : top / KV_SUB;
    if (h < *hi) *hi = h;
  }
}

// Query-tile CTA [q0, q0 + Q_TILE) against key sub-tiles t of Q_SUB rows:
// every i in [q0, q0 + Q_TILE), j in [t Q_SUB, t Q_SUB + Q_SUB) must exist
// and, causal / sliding, satisfy j <= i (t Q_SUB + Q_SUB - 1 <= q0) and,
// sliding, i - j < window (q0 + Q_TILE - 1 - t Q_SUB <= window - 1).
__host__ __device__ inline void full_range_q(int kind, int window, int Sq, int Skv, int q0,
                                             int* lo, int* hi) {
  *lo = 0;
  *hi = Skv / Q_SUB - 1;  // t Q_SUB + Q_SUB <= Skv
  if (kind == MK_BLOCK || q0 + Q_TILE > Sq) *hi = -1;
  if (kind == MK_CAUSAL || kind == MK_SLIDING) {
    const int top = q0 - (Q_SUB - 1);  // t Q_SUB <= top
    const int h = top < 0 ? -1 : top / Q_SUB;
    if (h < *hi) *hi = h;
  }
  if (kind == MK_SLIDING) {
    const int bot = q0 + Q_TILE - window;  // t Q_SUB >= bot
    const int l = bot <= 0 ? 0 : (bot + Q_SUB - 1) / Q_SUB;
    if (l > *lo) *lo = l;
  }
}

// Walk of a query-tile CTA (Q_TILE rows of head bh) over key sub-tiles of
// Q_SUB rows; Lq, Lk are the valid rows and keys of the batch (a tile that
// starts past Lq walks nothing).
struct QWalk {
  int lo, cnt;
  const int* list;  // select-table row, or nullptr for the closed form
  __device__ __forceinline__ void init(const AttnParams& p, int bh, int qt, int Lq, int Lk) {
    if (qt * Q_TILE >= Lq || Lk <= 0) {
      lo = 0;
      cnt = 0;
      list = nullptr;
    } else if (p.mask_kind == MK_BLOCK) {
      size_t row = (size_t)bh * p.nQT_q + qt;
      list = p.sel_q + row * p.nKT_q;
      cnt = p.cnt_q[row];
      lo = 0;
    } else {
      int hi;
      int q0 = qt * Q_TILE;
      partner_range(p.mask_kind, p.window, true, q0, min(q0 + Q_TILE, Lq), Q_SUB, Lk, &lo, &hi);
      cnt = hi - lo + 1;
      if (cnt < 0) cnt = 0;
      list = nullptr;
    }
  }
  __device__ __forceinline__ int tile(int n) const { return list ? list[n] : lo + n; }
};

// Walk of a key-tile CTA (KV_TILE rows of kv head (b, c)) over (query head of
// the group, query sub-tile of KV_SUB rows) pairs, head-major; Lq, Lk are the
// valid rows and keys of batch b (a tile that starts past Lk walks nothing).
struct KVWalk {
  int lo, cnt_closed;
  int b, c, t;
  bool none;
  __device__ __forceinline__ void init(const AttnParams& p, int b_, int c_, int t_, int Lq,
                                       int Lk) {
    b = b_;
    c = c_;
    t = t_;
    lo = 0;
    cnt_closed = 0;
    const int k0 = t * KV_TILE;
    none = k0 >= Lk || Lq <= 0;
    if (!none && p.mask_kind != MK_BLOCK) {
      int hi;
      partner_range(p.mask_kind, p.window, false, k0, min(k0 + KV_TILE, Lk), KV_SUB, Lq, &lo,
                    &hi);
      cnt_closed = hi - lo + 1;
      if (cnt_closed < 0) cnt_closed = 0;
    }
  }
  __device__ __forceinline__ int count(const AttnParams& p, int hh) const {
    if (none) return 0;
    if (p.mask_kind != MK_BLOCK) return cnt_closed;
    int bh = b * p.Hq + c * p.group + hh;
    return p.cnt_k[(size_t)bh * p.nKT_k + t];
  }
  __device__ __forceinline__ int tile(const AttnParams& p, int hh, int idx) const {
    if (p.mask_kind != MK_BLOCK) return lo + idx;
    int bh = b * p.Hq + c * p.group + hh;
    return p.sel_k[((size_t)bh * p.nKT_k + t) * p.nQT_k + idx];
  }
  __device__ __forceinline__ int total(const AttnParams& p) const {
    if (none) return 0;
    if (p.mask_kind != MK_BLOCK) return cnt_closed * p.group;
    int s = 0;
    for (int hh = 0; hh < p.group; ++hh) s += count(p, hh);
    return s;
  }
};

// Sequential cursor over a KVWalk: yields (hh, idx) in walk order.
struct KVCursor {
  int hh, idx, cnt;
  __device__ __forceinline__ void start(const AttnParams& p, const KVWalk& w) {
    hh = 0;
    idx = 0;
    cnt = w.count(p, 0);
    skip(p, w);
  }
  __device__ __forceinline__ void skip(const AttnParams& p, const KVWalk& w) {
    while (idx >= cnt && hh < p.group) {
      ++hh;
      idx = 0;
      cnt = hh < p.group ? w.count(p, hh) : 0;
    }
  }
  __device__ __forceinline__ void next(const AttnParams& p, const KVWalk& w) {
    ++idx;
    skip(p, w);
  }
};

// Step n of a KVWalk: query head hh of the group and query sub-tile r,
// head-major with ascending sub-tiles (the cursor advances here).  Key tiles
// t and t + 1 of a kv head, which run side by side, then read the same query
// rows two steps apart, so the second read comes from L2.
__device__ __forceinline__ void kv_step(const AttnParams& p, const KVWalk& w, KVCursor& cur,
                                        int* hh, int* r) {
  *hh = cur.hh;
  *r = w.tile(p, cur.hh, cur.idx);
  cur.next(p, w);
}

// Store 32 rows x 64 columns (16-bit elements, packed as 32 u32 per lane, one
// row per lane) through a per-warp 4 KB staging buffer so that global stores
// are 128-byte coalesced.  out_row0 points at column col0 of the warp's first
// row; rows are `stride` elements apart; rows >= nvalid are skipped.
__device__ __forceinline__ void warp_store_rows(uint8_t* stage, const uint32_t (&pk)[32],
                                                uint16_t* out_row0, int nvalid,
                                                int stride = HEAD_DIM) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    *reinterpret_cast<uint4*>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) = v;
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    int row = k * 4 + (lane >> 3), c = lane & 7;
    uint4 v = *reinterpret_cast<const uint4*>(stage + row * 128 + ((c ^ (row & 7)) << 4));
    if (row < nvalid) *reinterpret_cast<uint4*>(out_row0 + (size_t)row * stride + c * 8) = v;
  }
  __syncwarp();
}

// Store 32 rows x 32 columns (16-bit elements, packed as 16 u32 per lane, one
// row per lane) through a per-warp 2 KB staging buffer, so that each global
// store instruction writes 8 rows of 64 contiguous bytes.  out_row0 points at
// column col0 of the warp's first row; rows are `stride` elements apart; rows
// >= nvalid are skipped.
__device__ __forceinline__ void warp_store_rows32(uint8_t* stage, const uint32_t (&pk)[16],
                                                  uint16_t* out_row0, int nvalid,
                                                  int stride = HEAD_DIM) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    *reinterpret_cast<uint4*>(stage + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = v;
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int row = k * 8 + (lane >> 2), c = lane & 3;
    uint4 v = *reinterpret_cast<const uint4*>(stage + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
    if (row < nvalid) *reinterpret_cast<uint4*>(out_row0 + (size_t)row * stride + c * 8) = v;
  }
  __syncwarp();
}

// Zeros for `ncols` 16-bit columns (a multiple of 8) of 32 rows, one row per
// lane, stored straight to global memory (rows >= nvalid skipped).  Used by
// a CTA that gave up waiting, whose shared-memory staging space may still be
// the target of a copy in flight.
__device__ __forceinline__ void warp_zero_rows(uint16_t* out_row0, int ncols, int nvalid,
                                               int stride = HEAD_DIM) {
  const int lane = threadIdx.x & 31;
  if (lane >= nvalid) return;
  uint4* dst = reinterpret_cast<uint4*>(out_row0 + (size_t)lane * stride);
  for (int c = 0; c < ncols / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace mab
