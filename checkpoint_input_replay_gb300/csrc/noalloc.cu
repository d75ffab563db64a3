// rs_decode_step_noalloc: a standard decode step for callers that cannot
// allocate device memory.
//
// The decode kernel needs one piece of scratch memory besides its inputs and
// outputs: an int32 arrival counter per sequence, through which the last CTA
// of a sequence learns that it may advance the cursor.  rs_decode_step takes
// those counters from the caller's `scratch` buffer.  Some callers cannot
// provide it: code that runs where cudaMalloc is not allowed or not wanted
// (for example inside an inference server whose memory pool is fixed before
// the model runs, or a plugin whose host owns every device allocation), or
// that only received the checkpoint, ring and cursor buffers from someone
// else.  This entry point keeps the counters in a fixed array of this library
// instead (kNoAllocMaxBatch int32 = 64 KiB, held by every GPU that loads the
// library until the process exits) and allocates nothing: no cudaMalloc, no
// cudaFree, no allocating library routine.
#include <stdlib.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr int kNoAllocMaxBatch = 16384;  // largest batch this entry point accepts
constexpr int kMaxDevices = 64;

// Arrival counters shared by every call on a device.  In host code this name
// is only a stand-in for the device array: its address on a device comes from
// cudaGetSymbolAddress below and is what the kernel receives.
static __device__ __align__(256) int g_noalloc_arrive[kNoAllocMaxBatch];

struct DeviceScratch {
  int* addr = nullptr;        // device address of g_noalloc_arrive on this device
  CUcontext ctx = nullptr;    // the context that address belongs to
  bool ready = false;
};

DeviceScratch g_devices[kMaxDevices];
std::mutex g_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent, found once through the runtime (no link to libcuda).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult qr{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  return fn;
}

// Once per device (and again if the device's context was replaced, e.g. after a
// cudaDeviceReset), with that device current: resolve the array's device address.
rs_status scratch_for_current_device(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RS_ERR_CUDA;
  CUcontext ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceScratch& s = g_devices[dev];
  const CtxGetCurrentFn get = ctx_get_current();
  if (s.ready && get && (get(&ctx) != CUDA_SUCCESS || ctx != s.ctx)) s.ready = false;
  if (!s.ready) {
    int* ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_arrive) != cudaSuccess || !ptr)
      return RS_ERR_CUDA;
    ctx = nullptr;
    if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    s.addr = ptr;
    s.ctx = ctx;
    s.ready = true;
  }
  *out = s.addr;
  return RS_OK;
}

}  // namespace

extern "C" rs_status rs_decode_step_noalloc(const rs_config* cfg, const rs_buffers* bufs, const rs_inputs* in,
                                            float* y, rs_stream stream) {
  if (!cfg || !bufs || !y) return RS_ERR_NULL;
  if (cfg->batch > kNoAllocMaxBatch) return RS_ERR_UNSUPPORTED;
  rs::LayerDev d{};
  rs_status st = rs::bind_layer(cfg, bufs, false, &d);
  if (st != RS_OK) return st;
  // the same debug ordering check as rs_create_cache (see the header)
  if (const char* e = getenv("RS_DEBUG_CTA_PERMUTE")) d.cta_mult = atoi(e) >= 2 ? atoi(e) : 0;
  rs::TokenIn tok{};
  st = rs::bind_inputs(cfg->kind, in, &tok);
  if (st != RS_OK) return st;
  if ((reinterpret_cast<uintptr_t>(y) & 15u) != 0) return RS_ERR_ALIGN;
  int* arrive = nullptr;
  st = scratch_for_current_device(&arrive);
  if (st != RS_OK) return st;
  d.arrive = arrive;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the counters must start at zero; a previous call may have stopped early
  if (cudaMemsetAsync(arrive, 0, static_cast<size_t>(cfg->batch) * sizeof(int), s) != cudaSuccess)
    return RS_ERR_CUDA;
  return rs::launch_decode(d, tok, y, s) == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}
