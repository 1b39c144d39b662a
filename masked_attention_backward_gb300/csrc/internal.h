// internal.h -- shared definitions between the C-ABI front end (api.cu) and
// the kernel translation units.  Not part of the public interface.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace mab {

// Tile sizes.  dK/dV CTAs own KV_TILE key rows and walk query sub-tiles of
// KV_SUB rows; dQ (and forward) CTAs own Q_TILE query rows and walk key
// sub-tiles of Q_SUB rows.
constexpr int HEAD_DIM = 128;
constexpr int KV_TILE = 128;
constexpr int KV_SUB = 64;
constexpr int Q_TILE = 128;
constexpr int Q_SUB = 64;
constexpr int PREP_ROWS = 128;  // padding unit of the per-row statistics
constexpr int PREP_BLOCK_ROWS = 64;  // rows per preprocess block (divides PREP_ROWS)
constexpr float LOG2E = 1.4426950408889634f;

enum MaskKind { MK_NONE = 0, MK_CAUSAL = 1, MK_SLIDING = 2, MK_BLOCK = 3 };

// Byte offsets of the workspace regions (each 256-byte aligned).
struct WsLayout {
  size_t status;     // DevStatus
  size_t nlse2;      // float [B*Hq, Sq_pad]: -lse * log2(e), padded with -inf
  size_t delta;      // float [B*Hq, Sq_pad]: rowsum(dO * O), padded with 0
  size_t dsink_part; // float [Hq, B * n_row_blocks]
  size_t maskT;      // uint8 [B*Hq, nKB, nQB]
  size_t sel_k;      // int32 [B*Hq, nKT_k, nQT_k]  (key tiles of KV_TILE, query tiles of KV_SUB)
  size_t cnt_k;      // int32 [B*Hq, nKT_k]
  size_t sel_q;      // int32 [B*Hq, nQT_q, nKT_q]  (query tiles of Q_TILE, key tiles of Q_SUB)
  size_t cnt_q;      // int32 [B*Hq, nQT_q]
  size_t dq_flag;    // single pass: uint8 [B*Hq, steps per head], 1 = partial written
  size_t dq_part;    // single pass: float [B*Hq, steps per head, KV_SUB, HEAD_DIM]
  size_t total;
};

// Everything the attention kernels read besides the tensor maps.
struct AttnParams {
  int B, Hq, Hkv, Sq, Skv, group, Sq_pad;
  int mask_kind, window, bx, by, nqb, nkb;
  float inv_bx, inv_by;  // 1 / bx, 1 / by (block masks; quotients corrected to exact)
  const uint8_t* mask;   // [B*Hq, nqb, nkb]
  const uint8_t* maskT;  // [B*Hq, nkb, nqb]
  const int* sel_k;
  const int* cnt_k;
  int nQT_k, nKT_k;
  const int* sel_q;
  const int* cnt_q;
  int nQT_q, nKT_q;
  const float* nlse2;  // [B*Hq, Sq_pad]
  const float* delta;  // [B*Hq, Sq_pad]
  const float* sink;   // forward: [Hq] or nullptr
  float* lse_out;      // forward: [B*Hq, Sq]
  float scale;         // softmax scale
  float scale_log2;    // scale * log2(e)
  DevStatus* status;
  unsigned long long timeout_ns;
  int test_no_loads;   // test hook: the producers issue no loads (every wait runs out)
  int compensated;     // backward: P and dS enter the contractions as high part + remainder
  const int* seqlen_q; // [B] valid query rows per batch, or nullptr (= Sq)
  const int* seqlen_k; // [B] valid keys per batch, or nullptr (= Skv)
  int num_sms;         // SMs of the device (CTAs resident at once in one-CTA-per-SM grids)
  int kv_schedule;     // test hook: 0 = chosen by the walk lengths, 1 = per tile, 2 = persistent
  // Packed layout: sequence b holds tokens [cu_q[b], cu_q[b + 1]) of the
  // token-major tensors q, o, dO, dq [total_q, Hq, 128] (lse [Hq, total_q])
  // and [cu_k[b], cu_k[b + 1]) of k, v, dk, dv [total_k, Hkv, 128]; Sq and
  // Skv are then the longest lengths.  nullptr / 0 for the BHSD layout.
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;
  // dSink, summed from the preprocess kernel's partials ([Hq, nparts]) by the
  // dK/dV grid's last CTA; nullptr when that grid does not (no sink, or the
  // single-pass kernels, which leave it to k_dsink_finalize).
  float* dsink;
  const float* dsink_part;
  int dsink_nparts;
  // Single pass: the dq partial of each step of the dK/dV walk and its
  // written flag.  Slots of one query head: key tile t's steps follow those of
  // the tiles before it, query sub-tile r of the tile at (r - its range's
  // first sub-tile), over the full-length ranges (kv_tile_range_full).
  float* dq_part;
  uint8_t* dq_flag;
  long long dq_steps_head;  // slots per query head
};

#ifdef __CUDACC__
// Token offset and valid length of sequence b in a packed tensor of `total`
// tokens, the length clamped to [0, smax] and to the tensor's end.
__device__ __forceinline__ int packed_off(const int* cu, int b, int total) {
  return min(max(cu[b], 0), total);
}
__device__ __forceinline__ int packed_len(const int* cu, int b, int total, int smax) {
  const int o = packed_off(cu, b, total);
  return min(min(max(cu[b + 1], o), total) - o, smax);
}

// -(sum of head h's dSink partials), summed by one warp in a fixed order
// (lane-strided in fp64, then a butterfly): every caller gets the same bits.
__device__ __forceinline__ float dsink_of_head(const float* part, int nparts, int h, int lane) {
  double s = 0.0;
  for (int i = lane; i < nparts; i += 32) s += (double)part[(size_t)h * nparts + i];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return (float)(-s);
}

// Valid query rows / keys of batch b: the per-batch lengths clamped to
// [0, Sq] / [0, Skv], or the full lengths.
__device__ __forceinline__ int len_q(const AttnParams& p, int b) {
  if (p.cu_q) return packed_len(p.cu_q, b, p.total_q, p.Sq);
  return p.seqlen_q ? min(max(p.seqlen_q[b], 0), p.Sq) : p.Sq;
}
__device__ __forceinline__ int len_k(const AttnParams& p, int b) {
  if (p.cu_k) return packed_len(p.cu_k, b, p.total_k, p.Skv);
  return p.seqlen_k ? min(max(p.seqlen_k[b], 0), p.Skv) : p.Skv;
}

// Where row `row` of head h (of H heads) of batch b lives.  BHSD [B*H, S, 128]
// tensor maps take the coordinates (row, b*H + h); packed [T, H, 128] maps
// take (h, token).  In memory a row starts at element `elem` and consecutive
// rows of the head are `stride` elements apart.
struct RowAddr {
  int c1, c2;
  size_t elem;
  int stride;
};
__device__ __forceinline__ RowAddr row_q(const AttnParams& p, int b, int h, int row) {
  if (p.cu_q) {
    const int tok = packed_off(p.cu_q, b, p.total_q) + row;
    return {h, tok, ((size_t)tok * p.Hq + h) * 128, p.Hq * 128};
  }
  const int bh = b * p.Hq + h;
  return {row, bh, ((size_t)bh * p.Sq + row) * 128, 128};
}
__device__ __forceinline__ RowAddr row_k(const AttnParams& p, int b, int c, int row) {
  if (p.cu_k) {
    const int tok = packed_off(p.cu_k, b, p.total_k) + row;
    return {c, tok, ((size_t)tok * p.Hkv + c) * 128, p.Hkv * 128};
  }
  const int bc = b * p.Hkv + c;
  return {row, bc, ((size_t)bc * p.Skv + row) * 128, 128};
}
// Rows of head h (batch b) the epilogue writes starting at row r0, at most
// 32: up to the padded length in the BHSD layout (rows past a batch's valid
// length are zeros there), only the sequence's own rows in the packed one.
__device__ __forceinline__ int rows_to_store_q(const AttnParams& p, int b, int r0) {
  return max(0, min(32, (p.cu_q ? len_q(p, b) : p.Sq) - r0));
}
__device__ __forceinline__ int rows_to_store_k(const AttnParams& p, int b, int r0) {
  return max(0, min(32, (p.cu_k ? len_k(p, b) : p.Skv) - r0));
}
#endif

// ---- launchers (each returns the launch error, if any) ----
cudaError_t launch_preprocess(bool bf16, const void* O, const void* dO, const float* lse,
                              const float* sink, float* nlse2, float* delta, float* part, int B,
                              int Hq, int Sq, int Sq_pad, const int* seqlen_q, const int* cu_q,
                              int total_q, DevStatus* status, bool overlap_prev, cudaStream_t st);
cudaError_t launch_dsink_finalize(const float* part, int Hq, int nparts, float* dsink,
                                  cudaStream_t st);
cudaError_t launch_mask_tables(const AttnParams& p, uint8_t* maskT, int* sel_k, int* cnt_k,
                               int* sel_q, int* cnt_q, cudaStream_t st);
cudaError_t launch_dkdv(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                        const CUtensorMap& tdO, const CUtensorMap& tK, const CUtensorMap& tV,
                        void* dk, void* dv, cudaStream_t st);
cudaError_t launch_dkdv_units(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                              const CUtensorMap& tdO, const CUtensorMap& tK,
                              const CUtensorMap& tV, void* dk, void* dv, cudaStream_t st);
cudaError_t launch_dq(bool bf16, const AttnParams& p, const CUtensorMap& tQ, const CUtensorMap& tdO,
                      const CUtensorMap& tK, const CUtensorMap& tV, void* dq, cudaStream_t st);
cudaError_t launch_fwd(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                       const CUtensorMap& tK, const CUtensorMap& tV, void* o, cudaStream_t st);

// ---- tile-range helpers shared by host and device ----

// For the closed-form masks: the inclusive range [lo, hi] of partner tiles of
// `psize` rows (over a sequence of `plen`) that hold at least one visible pair
// with the own tile [o0, o1) (o1 exclusive).  own_is_query selects whether the
// own rows are queries (i) or keys (j).  Visibility: 0 <= i - j < window
// (causal: unbounded window), or everything for MK_NONE.  Returns hi < lo when
// empty.  Every tile in the range holds at least one visible pair.
__host__ __device__ inline void partner_range(int kind, int window, bool own_is_query, int o0,
                                              int o1, int psize, int plen, int* lo, int* hi) {
  int nP = (plen + psize - 1) / psize;
  if (kind == MK_NONE) {
    *lo = 0;
    *hi = nP - 1;
    return;
  }
  long long w = (kind == MK_CAUSAL) ? (long long)1 << 40 : (long long)window;
  long long a, b;  // partner token range that can be visible: [a, b]
  if (own_is_query) {
    // keys j with i - w < j <= i for some i in [o0, o1)
    a = (long long)o0 - w + 1;
    b = (long long)o1 - 1;
  } else {
    // queries i with j <= i < j + w for some j in [o0, o1)
    a = o0;
    b = (long long)o1 - 1 + w - 1;
  }
  if (a < 0) a = 0;
  if (b > plen - 1) b = plen - 1;
  if (b < a) {
    *lo = 0;
    *hi = -1;
    return;
  }
  *lo = (int)(a / psize);
  *hi = (int)(b / psize);
}

// Query sub-tiles of KV_SUB rows key tile t (KV_TILE keys) can meet at the
// full lengths: the partner range of the closed-form masks (first sub-tile in
// *lo), or all of them for block masks (*lo = 0).  Shorter per-batch lengths
// only cut a range's end, so these ranges hold every step of any walk.
__host__ __device__ inline int kv_tile_range_full(int kind, int window, int Sq, int Skv, int t,
                                                  int* lo) {
  const int nQT = (Sq + KV_SUB - 1) / KV_SUB;
  if (kind == MK_BLOCK) {
    *lo = 0;
    return nQT;
  }
  const int k0 = t * KV_TILE;
  const int k1 = k0 + KV_TILE < Skv ? k0 + KV_TILE : Skv;
  int hi;
  partner_range(kind, window, false, k0, k1, KV_SUB, Sq, lo, &hi);
  return hi >= *lo ? hi - *lo + 1 : 0;
}

cudaError_t launch_dkdvq(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                         const CUtensorMap& tdO, const CUtensorMap& tK, const CUtensorMap& tV,
                         void* dk, void* dv, cudaStream_t st);
cudaError_t launch_dq_reduce(bool bf16, const AttnParams& p, void* dq, cudaStream_t st);

}  // namespace mab
