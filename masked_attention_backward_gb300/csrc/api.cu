// api.cu -- the C ABI of libmaskattn (declared in include/maskattn.h).
//
// The host side only checks arguments, carves the caller's workspace and
// enqueues kernels on the caller's stream: no dense token mask is built and
// nothing is allocated (cannbot-knowledge PR #174, BlockSparseAttentionGrad
// runbook, optimisation 1: the host does shape, alloc and view only).
//
// attn_bwd enqueues, in order:
//   k_mask_tables       block masks only: transposed mask and both select
//                         tables
//   k_preprocess        Delta, lse*log2(e) (padded), dSink partials (beside
//                         the tables)
//   k_dkdv              key-stationary dK / dV; with a sink its last CTA
//                         sums dSink = -(sum of the partials)
//   k_dq                query-stationary dQ
// and with ATTN_FLAG_SINGLE_PASS k_dkdvq (dK / dV and the dQ partials),
// k_dq_reduce and k_dsink_finalize (sink only) in place of k_dkdv and k_dq.
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "maskattn.h"
#include "internal.h"
#include "tmap.h"

using namespace mab;

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

attn_status_t check_shape_mask(const attn_shape_t* sh, const attn_mask_desc_t* mk) {
  if (!sh || !mk) return ATTN_ERR_INVALID_ARG;
  if (sh->B <= 0 || sh->Hq <= 0 || sh->Hkv <= 0 || sh->Sq <= 0 || sh->Skv <= 0 || sh->D <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (sh->Hq % sh->Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (sh->dtype != ATTN_F16 && sh->dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (sh->flags & ~(ATTN_FLAG_COMPENSATED | ATTN_FLAG_SINGLE_PASS)) return ATTN_ERR_INVALID_ARG;
  // sequence lengths up to 2^24 and B*Hq up to 65535 keep every index and
  // grid dimension in range
  if (sh->Sq > (1 << 24) || sh->Skv > (1 << 24) || (long long)sh->B * sh->Hq > 65535)
    return ATTN_ERR_INVALID_ARG;
  switch (mk->kind) {
    case ATTN_MASK_NONE:
      break;
    case ATTN_MASK_CAUSAL:
      if (sh->Sq != sh->Skv) return ATTN_ERR_INVALID_ARG;
      break;
    case ATTN_MASK_SLIDING:
      if (sh->Sq != sh->Skv || mk->window < 1) return ATTN_ERR_INVALID_ARG;
      break;
    case ATTN_MASK_BLOCK:
      if (mk->bx < 1 || mk->by < 1) return ATTN_ERR_INVALID_ARG;
      break;
    default:
      return ATTN_ERR_INVALID_ARG;
  }
  if ((mk->seqlen_q && !aligned(mk->seqlen_q, 4)) || (mk->seqlen_k && !aligned(mk->seqlen_k, 4)))
    return ATTN_ERR_INVALID_ARG;
  // packed layout: both offset arrays, no per-batch length arrays, and the
  // token totals of the tensors (which bound every access)
  if (mk->cu_seqlens_q || mk->cu_seqlens_k) {
    if (!mk->cu_seqlens_q || !mk->cu_seqlens_k || mk->seqlen_q || mk->seqlen_k ||
        !aligned(mk->cu_seqlens_q, 4) || !aligned(mk->cu_seqlens_k, 4) || mk->total_q < 1 ||
        mk->total_k < 1)
      return ATTN_ERR_INVALID_ARG;
  }
  if (sh->D != HEAD_DIM) return ATTN_ERR_UNSUPPORTED;
  // the single-pass kernels have neither the compensated nor the packed form
  if ((sh->flags & ATTN_FLAG_SINGLE_PASS) &&
      ((sh->flags & ATTN_FLAG_COMPENSATED) || mk->cu_seqlens_q))
    return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Single pass: dq partial slots per query head (kv_tile_range_full summed over
// the key tiles).
long long single_pass_steps_head(const attn_shape_t* sh, const attn_mask_desc_t* mk) {
  const int nKT = (sh->Skv + KV_TILE - 1) / KV_TILE;
  const int kind = mk->kind;
  const int window = kind == ATTN_MASK_SLIDING ? mk->window : 0;
  long long n = 0;
  for (int t = 0; t < nKT; ++t) {
    int lo;
    n += kv_tile_range_full(kind, window, sh->Sq, sh->Skv, t, &lo);
  }
  return n;
}

struct Dims {
  int Sq_pad, nqb, nkb, nQT_k, nKT_k, nQT_q, nKT_q, nparts;
};

Dims dims_of(const attn_shape_t* sh, const attn_mask_desc_t* mk) {
  Dims d;
  d.Sq_pad = (sh->Sq + PREP_ROWS - 1) / PREP_ROWS * PREP_ROWS;
  const bool blk = mk->kind == ATTN_MASK_BLOCK;
  d.nqb = blk ? (sh->Sq + mk->bx - 1) / mk->bx : 0;
  d.nkb = blk ? (sh->Skv + mk->by - 1) / mk->by : 0;
  d.nQT_k = (sh->Sq + KV_SUB - 1) / KV_SUB;
  d.nKT_k = (sh->Skv + KV_TILE - 1) / KV_TILE;
  d.nQT_q = (sh->Sq + Q_TILE - 1) / Q_TILE;
  d.nKT_q = (sh->Skv + Q_SUB - 1) / Q_SUB;
  d.nparts = sh->B * (d.Sq_pad / PREP_BLOCK_ROWS);
  return d;
}

WsLayout layout_of(const attn_shape_t* sh, const attn_mask_desc_t* mk) {
  Dims d = dims_of(sh, mk);
  const size_t BH = (size_t)sh->B * sh->Hq;
  WsLayout L;
  size_t off = 0;
  L.status = off;
  off = align256(off + sizeof(DevStatus));
  L.nlse2 = off;
  off = align256(off + BH * d.Sq_pad * sizeof(float));
  L.delta = off;
  off = align256(off + BH * d.Sq_pad * sizeof(float));
  L.dsink_part = off;
  off = align256(off + (size_t)sh->Hq * d.nparts * sizeof(float));
  L.maskT = L.sel_k = L.cnt_k = L.sel_q = L.cnt_q = off;
  if (mk->kind == ATTN_MASK_BLOCK) {
    L.maskT = off;
    off = align256(off + BH * d.nqb * d.nkb);
    L.sel_k = off;
    off = align256(off + BH * d.nKT_k * d.nQT_k * sizeof(int));
    L.cnt_k = off;
    off = align256(off + BH * d.nKT_k * sizeof(int));
    L.sel_q = off;
    off = align256(off + BH * d.nQT_q * d.nKT_q * sizeof(int));
    L.cnt_q = off;
    off = align256(off + BH * d.nQT_q * sizeof(int));
  }
  L.dq_flag = L.dq_part = off;
  if (sh->flags & ATTN_FLAG_SINGLE_PASS) {
    const size_t slots = BH * (size_t)single_pass_steps_head(sh, mk);
    L.dq_flag = off;
    off = align256(off + slots);
    L.dq_part = off;
    off = align256(off + slots * KV_SUB * HEAD_DIM * sizeof(float));
  }
  L.total = off;
  return L;
}

// Test hook (MASKATTN_TEST_NO_LOADS=1): the producer warps of the tcgen05
// kernels issue no loads and signal nothing, so the first wait of every CTA
// runs out with nothing in flight -- the way the tests reach the bounded-wait
// error path without disturbing the GPU.
int test_no_loads() {
  const char* e = getenv("MASKATTN_TEST_NO_LOADS");
  return (e && e[0] == '1') ? 1 : 0;
}

// Test hook (MASKATTN_DKDV_SCHEDULE=tile|units): forces the dK/dV kernel's
// form, so that the tests run both on any shape.
int dkdv_schedule() {
  const char* e = getenv("MASKATTN_DKDV_SCHEDULE");
  if (!e) return 0;
  if (strcmp(e, "tile") == 0) return 1;
  if (strcmp(e, "units") == 0) return 2;
  return 0;
}

unsigned long long wait_timeout_ns() {
  const char* e = getenv("MASKATTN_WAIT_TIMEOUT_NS");
  if (e && *e) {
    unsigned long long v = strtoull(e, nullptr, 10);
    if (v > 0) return v;
  }
  return kDefaultTimeoutNs;
}

AttnParams params_of(const attn_shape_t* sh, const attn_mask_desc_t* mk, const WsLayout& L,
                     uint8_t* ws, float scale) {
  Dims d = dims_of(sh, mk);
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.B = sh->B;
  p.Hq = sh->Hq;
  p.Hkv = sh->Hkv;
  p.Sq = sh->Sq;
  p.Skv = sh->Skv;
  p.group = sh->Hq / sh->Hkv;
  p.Sq_pad = d.Sq_pad;
  p.mask_kind = mk->kind;
  p.window = mk->kind == ATTN_MASK_SLIDING ? mk->window : 0;
  p.bx = mk->kind == ATTN_MASK_BLOCK ? mk->bx : 1;
  p.by = mk->kind == ATTN_MASK_BLOCK ? mk->by : 1;
  p.inv_bx = 1.0f / (float)p.bx;
  p.inv_by = 1.0f / (float)p.by;
  p.nqb = d.nqb;
  p.nkb = d.nkb;
  if (mk->kind == ATTN_MASK_BLOCK) {
    p.mask = mk->block_mask;
    p.maskT = ws + L.maskT;
    p.sel_k = reinterpret_cast<const int*>(ws + L.sel_k);
    p.cnt_k = reinterpret_cast<const int*>(ws + L.cnt_k);
    p.sel_q = reinterpret_cast<const int*>(ws + L.sel_q);
    p.cnt_q = reinterpret_cast<const int*>(ws + L.cnt_q);
  }
  p.nQT_k = d.nQT_k;
  p.nKT_k = d.nKT_k;
  p.nQT_q = d.nQT_q;
  p.nKT_q = d.nKT_q;
  p.nlse2 = reinterpret_cast<const float*>(ws + L.nlse2);
  p.delta = reinterpret_cast<const float*>(ws + L.delta);
  p.scale = scale;
  p.scale_log2 = scale * LOG2E;
  p.status = reinterpret_cast<DevStatus*>(ws + L.status);
  p.timeout_ns = wait_timeout_ns();
  p.test_no_loads = test_no_loads();
  p.kv_schedule = dkdv_schedule();
  p.compensated = (sh->flags & ATTN_FLAG_COMPENSATED) ? 1 : 0;
  if (sh->flags & ATTN_FLAG_SINGLE_PASS) {
    p.dq_part = reinterpret_cast<float*>(ws + L.dq_part);
    p.dq_flag = ws + L.dq_flag;
    p.dq_steps_head = single_pass_steps_head(sh, mk);
  }
  p.seqlen_q = mk->seqlen_q;
  p.seqlen_k = mk->seqlen_k;
  if (mk->cu_seqlens_q) {
    p.cu_q = mk->cu_seqlens_q;
    p.cu_k = mk->cu_seqlens_k;
    p.total_q = mk->total_q;
    p.total_k = mk->total_k;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
    p.num_sms = sms;
  return p;
}

attn_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Tensor map of a query-side (H = Hq, S = Sq) or key-side (H = Hkv, S = Skv)
// tensor: BHSD [B*H, S, 128], or token-major [total, H, 128] in the packed
// layout; boxes of `rows` rows of one head either way.
bool make_map(CUtensorMap* m, const void* base, bool bf16, const attn_shape_t* sh,
              const attn_mask_desc_t* mk, bool query_side, uint32_t rows) {
  const int H = query_side ? sh->Hq : sh->Hkv;
  if (mk->cu_seqlens_q)
    return make_thd_map(m, base, bf16, query_side ? mk->total_q : mk->total_k, H, rows);
  return make_bhsd_map(m, base, bf16, (int64_t)sh->B * H, query_side ? sh->Sq : sh->Skv, rows);
}

// ---- optional per-kernel events (attn_profile_enable) ----
// The mutex is taken only by calls made while profiling is on (and by the
// profiling calls themselves): with profiling off, host threads driving other
// streams or devices enqueue without waiting on one another.
struct Profiler {
  static constexpr int kMax = 16;
  std::mutex mu;
  std::atomic<bool> on{false};
  bool created = false;
  int device = -1;
  cudaEvent_t ev[kMax][2];
  const char* names[kMax];
  int n = 0;
};
Profiler g_prof;

// Brackets one launch with events when the call is profiled (the caller then
// holds the profiler's mutex).
struct ProfScope {
  cudaStream_t st;
  bool active;
  int slot;
  ProfScope(bool profiled, const char* name, cudaStream_t s) : st(s), active(false), slot(-1) {
    if (!profiled || !g_prof.created || g_prof.n >= Profiler::kMax) return;
    slot = g_prof.n++;
    g_prof.names[slot] = name;
    active = cudaEventRecord(g_prof.ev[slot][0], st) == cudaSuccess;
  }
  ~ProfScope() {
    if (active) cudaEventRecord(g_prof.ev[slot][1], st);
  }
};

// Called at the start of every profiled API call, with the mutex held.
void prof_begin() { g_prof.n = 0; }

// Takes the profiler's mutex only when profiling is on; returns whether this
// call is profiled.
bool prof_lock(std::unique_lock<std::mutex>& lock) {
  if (!g_prof.on.load(std::memory_order_acquire)) return false;
  lock.lock();
  if (!g_prof.on.load(std::memory_order_relaxed)) return false;  // switched off meanwhile
  prof_begin();
  return true;
}

// Transposed mask and both select tables (block masks only), one launch.
cudaError_t enqueue_tables(const WsLayout& L, uint8_t* ws, const AttnParams& p, cudaStream_t st) {
  return launch_mask_tables(p, ws + L.maskT, reinterpret_cast<int*>(ws + L.sel_k),
                            reinterpret_cast<int*>(ws + L.cnt_k),
                            reinterpret_cast<int*>(ws + L.sel_q),
                            reinterpret_cast<int*>(ws + L.cnt_q), st);
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

attn_status_t attn_workspace_size(const attn_shape_t* shape, const attn_mask_desc_t* mask,
                                  size_t* bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  attn_status_t r = check_shape_mask(shape, mask);
  if (r != ATTN_OK) return r;
  *bytes = layout_of(shape, mask).total;
  return ATTN_OK;
}

attn_status_t attn_fwd(const attn_shape_t* shape, const void* q, const void* k, const void* v,
                       const float* sink, const attn_mask_desc_t* mask, float scale, void* o,
                       float* lse, void* ws, size_t ws_bytes, void* stream) {
  attn_status_t r = check_shape_mask(shape, mask);
  if (r != ATTN_OK) return r;
  if (!q || !k || !v || !o || !lse || !ws) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(ws, 256) || (sink && !aligned(sink, 4)))
    return ATTN_ERR_INVALID_ARG;
  if (mask->kind == ATTN_MASK_BLOCK && !mask->block_mask) return ATTN_ERR_INVALID_ARG;
  // the forward needs none of the backward's single-pass regions
  attn_shape_t fsh = *shape;
  fsh.flags &= ~ATTN_FLAG_SINGLE_PASS;
  shape = &fsh;
  const WsLayout L = layout_of(shape, mask);
  if (ws_bytes < L.total) return ATTN_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const bool bf16 = shape->dtype == ATTN_BF16;
  AttnParams p = params_of(shape, mask, L, w, scale);
  p.sink = sink;
  p.lse_out = lse;
  CUtensorMap tQ, tK, tV;
  if (!make_map(&tQ, q, bf16, shape, mask, true, Q_TILE) ||
      !make_map(&tK, k, bf16, shape, mask, false, Q_SUB) ||
      !make_map(&tV, v, bf16, shape, mask, false, Q_SUB))
    return ATTN_ERR_CUDA;
  std::unique_lock<std::mutex> lock(g_prof.mu, std::defer_lock);
  const bool prof = prof_lock(lock);
  cudaError_t e = cudaMemsetAsync(w + L.status, 0, sizeof(DevStatus), st);
  if (e == cudaSuccess && mask->kind == ATTN_MASK_BLOCK) {
    ProfScope ps(prof, "k_mask_tables", st);
    e = enqueue_tables(L, w, p, st);
  }
  if (e == cudaSuccess) {
    ProfScope ps(prof, "k_attn_fwd", st);
    e = launch_fwd(bf16, p, tQ, tK, tV, o, st);
  }
  return cuda_status(e);
}

attn_status_t attn_bwd(const attn_shape_t* shape, const void* q, const void* k, const void* v,
                       const void* o, const void* dO, const float* lse, const float* sink,
                       const attn_mask_desc_t* mask, float scale, void* dq, void* dk, void* dv,
                       float* dsink, void* ws, size_t ws_bytes, void* stream) {
  attn_status_t r = check_shape_mask(shape, mask);
  if (r != ATTN_OK) return r;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !ws || (sink && !dsink))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dO, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(ws, 256) || (sink && (!aligned(sink, 4) || !aligned(dsink, 4))))
    return ATTN_ERR_INVALID_ARG;
  if (mask->kind == ATTN_MASK_BLOCK && !mask->block_mask) return ATTN_ERR_INVALID_ARG;
  const WsLayout L = layout_of(shape, mask);
  if (ws_bytes < L.total) return ATTN_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const bool bf16 = shape->dtype == ATTN_BF16;
  AttnParams p = params_of(shape, mask, L, w, scale);
  const Dims d = dims_of(shape, mask);

  // dK/dV walk query sub-tiles of KV_SUB rows over key tiles of KV_TILE rows;
  // dQ walks key sub-tiles of Q_SUB rows over query tiles of Q_TILE rows.
  CUtensorMap tQs, tdOs, tKt, tVt, tQt, tdOt, tKs, tVs;
  if (!make_map(&tQs, q, bf16, shape, mask, true, KV_SUB) ||
      !make_map(&tdOs, dO, bf16, shape, mask, true, KV_SUB) ||
      !make_map(&tKt, k, bf16, shape, mask, false, KV_TILE) ||
      !make_map(&tVt, v, bf16, shape, mask, false, KV_TILE) ||
      !make_map(&tQt, q, bf16, shape, mask, true, Q_TILE) ||
      !make_map(&tdOt, dO, bf16, shape, mask, true, Q_TILE) ||
      !make_map(&tKs, k, bf16, shape, mask, false, Q_SUB) ||
      !make_map(&tVs, v, bf16, shape, mask, false, Q_SUB))
    return ATTN_ERR_CUDA;

  const bool single = (shape->flags & ATTN_FLAG_SINGLE_PASS) != 0;

  std::unique_lock<std::mutex> lock(g_prof.mu, std::defer_lock);
  const bool prof = prof_lock(lock);
  // the status word is zeroed by the preprocess kernel, which every call runs
  // before any kernel that reads or writes it
  cudaError_t e = cudaSuccess;
  if (single) e = cudaMemsetAsync(w + L.dq_flag, 0, L.dq_part - L.dq_flag, st);
  // block masks: the tables first, and the preprocess grid beside them (it
  // reads nothing of theirs; its completion implies theirs)
  const bool blk = mask->kind == ATTN_MASK_BLOCK;
  if (e == cudaSuccess && blk) {
    ProfScope ps(prof, "k_mask_tables", st);
    e = enqueue_tables(L, w, p, st);
  }
  if (e == cudaSuccess) {
    ProfScope ps(prof, "k_preprocess", st);
    e = launch_preprocess(bf16, o, dO, lse, sink, reinterpret_cast<float*>(w + L.nlse2),
                          reinterpret_cast<float*>(w + L.delta),
                          reinterpret_cast<float*>(w + L.dsink_part), shape->B, shape->Hq,
                          shape->Sq, d.Sq_pad, mask->seqlen_q, mask->cu_seqlens_q,
                          mask->total_q, reinterpret_cast<DevStatus*>(w + L.status),
                          blk && !prof, st);
  }
  if (e == cudaSuccess && single) {
    {
      ProfScope ps(prof, "k_dkdvq", st);
      e = launch_dkdvq(bf16, p, tQs, tdOs, tKt, tVt, dk, dv, st);
    }
    if (e == cudaSuccess) {
      ProfScope ps(prof, "k_dq_reduce", st);
      e = launch_dq_reduce(bf16, p, dq, st);
    }
  } else if (e == cudaSuccess) {
    // the dK/dV grid's last CTA also sums dSink
    if (sink) {
      p.dsink = dsink;
      p.dsink_part = reinterpret_cast<const float*>(w + L.dsink_part);
      p.dsink_nparts = d.nparts;
    }
    {
      ProfScope ps(prof, "k_dkdv", st);
      e = launch_dkdv(bf16, p, tQs, tdOs, tKt, tVt, dk, dv, st);
    }
    if (e == cudaSuccess) {
      ProfScope ps(prof, "k_dq", st);
      e = launch_dq(bf16, p, tQt, tdOt, tKs, tVs, dq, st);
    }
  }
  if (e == cudaSuccess && sink && single) {
    ProfScope ps(prof, "k_dsink_finalize", st);
    e = launch_dsink_finalize(reinterpret_cast<const float*>(w + L.dsink_part), shape->Hq,
                              d.nparts, dsink, st);
  }
  return cuda_status(e);
}

attn_status_t attn_get_device_status(const void* ws, void* stream) {
  if (!ws) return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
  DevStatus h;
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  return h.code == 0 ? ATTN_OK : static_cast<attn_status_t>(h.code);
}

attn_status_t attn_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  if (on) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (g_prof.created && g_prof.device != dev) {
      for (int i = 0; i < Profiler::kMax; ++i) {
        cudaEventDestroy(g_prof.ev[i][0]);
        cudaEventDestroy(g_prof.ev[i][1]);
      }
      g_prof.created = false;
    }
    if (!g_prof.created) {
      for (int i = 0; i < Profiler::kMax; ++i)
        if (cudaEventCreate(&g_prof.ev[i][0]) != cudaSuccess ||
            cudaEventCreate(&g_prof.ev[i][1]) != cudaSuccess)
          return ATTN_ERR_CUDA;
      g_prof.created = true;
      g_prof.device = dev;
    }
  }
  g_prof.on.store(on != 0, std::memory_order_release);
  g_prof.n = 0;
  return ATTN_OK;
}

attn_status_t attn_profile_read(const char** names, float* ms, int capacity, int* count) {
  if (!count || (capacity > 0 && (!names || !ms))) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof.mu);
  *count = g_prof.created ? g_prof.n : 0;
  for (int i = 0; i < *count && i < capacity; ++i) {
    if (cudaEventSynchronize(g_prof.ev[i][1]) != cudaSuccess) return ATTN_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, g_prof.ev[i][0], g_prof.ev[i][1]) != cudaSuccess)
      return ATTN_ERR_CUDA;
    names[i] = g_prof.names[i];
    ms[i] = t;
  }
  return ATTN_OK;
}

}  // extern "C"
