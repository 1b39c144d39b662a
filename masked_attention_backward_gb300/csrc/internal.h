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
  size_t total;
};

// Everything the attention kernels read besides the tensor maps.
struct AttnParams {
  int B, Hq, Hkv, Sq, Skv, group, Sq_pad;
  int mask_kind, window, bx, by, nqb, nkb;
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
};

#ifdef __CUDACC__
// Valid query rows / keys of batch b: the per-batch lengths clamped to
// [0, Sq] / [0, Skv], or the full lengths.
__device__ __forceinline__ int len_q(const AttnParams& p, int b) {
  return p.seqlen_q ? min(max(p.seqlen_q[b], 0), p.Sq) : p.Sq;
}
__device__ __forceinline__ int len_k(const AttnParams& p, int b) {
  return p.seqlen_k ? min(max(p.seqlen_k[b], 0), p.Skv) : p.Skv;
}
#endif

// ---- launchers (each returns the launch error, if any) ----
cudaError_t launch_preprocess(bool bf16, const void* O, const void* dO, const float* lse,
                              const float* sink, float* nlse2, float* delta, float* part, int B,
                              int Hq, int Sq, int Sq_pad, const int* seqlen_q, cudaStream_t st);
cudaError_t launch_dsink_finalize(const float* part, int Hq, int nparts, float* dsink,
                                  cudaStream_t st);
cudaError_t launch_mask_transpose(const uint8_t* mask, uint8_t* maskT, int BH, int nqb, int nkb,
                                  cudaStream_t st);
cudaError_t launch_build_sel(const AttnParams& p, int* sel_k, int* cnt_k, int* sel_q, int* cnt_q,
                             cudaStream_t st);
cudaError_t launch_dkdv(bool bf16, const AttnParams& p, const CUtensorMap& tQ,
                        const CUtensorMap& tdO, const CUtensorMap& tK, const CUtensorMap& tV,
                        void* dk, void* dv, cudaStream_t st);
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

}  // namespace mab
