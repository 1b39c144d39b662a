// api_noalloc.cu -- attn_bwd_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// Some callers only ever see the input and output buffers of an operation:
// operator or plugin interfaces that pass no workspace, and services that
// forbid device allocation once they are running (a cudaMalloc there can stall
// every stream on the device, or fail because a caching allocator has already
// reserved the memory).  For them this file keeps the backward's scratch
// (per-row statistics, dSink partial sums, block-mask tables and the status
// word) in one fixed, file-scope device array instead of a caller workspace.
//
// The array is NOALLOC_SCRATCH_BYTES (32 MiB) per GPU, reserved on every GPU
// that loads this library until the process exits.  Shapes whose scratch
// would exceed it are rejected with ATTN_ERR_WORKSPACE.
//
// Every call on a device shares the same array and it keeps whatever the last
// call left there.  Each call rewrites every byte it later reads (the status
// word is cleared first), so nothing carries over between calls, but calls
// whose work overlaps on the GPU (different streams, or different host
// threads without ordering) race on the array and give wrong results.
#include <mutex>

#include "maskattn.h"
#include "internal.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// Device-side scratch.  In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.  nullptr on failure.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

// True when `stream` belongs to the current device (the legacy default
// stream, NULL, always does).
bool stream_on_current_device(void* stream) {
  if (!stream) return true;
  int dev = -1, sdev = -2;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
    return false;
  return dev == sdev;
}

}  // namespace

extern "C" attn_status_t attn_bwd_noalloc(const attn_shape_t* shape, const void* q, const void* k,
                                          const void* v, const void* o, const void* dO,
                                          const float* lse, const float* sink,
                                          const attn_mask_desc_t* mask, float scale, void* dq,
                                          void* dk, void* dv, float* dsink, void* stream) {
  size_t need = 0;
  attn_status_t r = attn_workspace_size(shape, mask, &need);
  if (r != ATTN_OK) return r;
  if (need > NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  if (!stream_on_current_device(stream)) return ATTN_ERR_INVALID_ARG;
  void* ws = scratch_on_current_device();
  if (!ws) return ATTN_ERR_CUDA;
  return attn_bwd(shape, q, k, v, o, dO, lse, sink, mask, scale, dq, dk, dv, dsink, ws,
                  NOALLOC_SCRATCH_BYTES, stream);
}

// The status word of the last attn_bwd_noalloc call on the current device
// lives at the start of the library's scratch array, which callers cannot
// address; this reads it back the way attn_get_device_status reads a
// workspace's.
extern "C" attn_status_t attn_noalloc_get_device_status(void* stream) {
  if (!stream_on_current_device(stream)) return ATTN_ERR_INVALID_ARG;
  void* ws = scratch_on_current_device();
  if (!ws) return ATTN_ERR_CUDA;
  return attn_get_device_status(ws, stream);
}
