// fa_backward_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// fa_backward needs a caller-provided scratch workspace (the fp32 dQ
// accumulator and two per-row vectors).  Some callers cannot provide one:
// code running inside a host framework that hands it only its input and output
// buffers and owns every other byte of device memory, or a latency-critical
// loop that must not call cudaMalloc (which may synchronise the device).  This
// entry point serves them from a fixed-size scratch array that lives in this
// file as a device global, so nothing is allocated per call.
//
// Cost and limits:
//  * every GPU that loads this library holds FA_NOALLOC_SCRATCH_BYTES of
//    device memory for the array until the process exits;
//  * problems whose workspace (fa_backward_workspace_bytes) exceeds that size
//    are rejected with FA_ERR_SCRATCH_TOO_SMALL -- use fa_backward for them;
//  * all calls on a device share the one array: calls whose kernels may
//    overlap on the GPU (e.g. on two streams without ordering between them)
//    race on it and must be serialised by the caller;
//  * the array keeps whatever the previous call left in it; the backward's
//    first kernel rewrites every part of the workspace it reads (it zeroes
//    the dQ accumulator and recomputes the row vectors), so no stale value is
//    ever used.
//  * the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture on the device.
#include <mutex>

#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the current device's copy of the scratch array.  In host
// code the array's name only stands in for the symbol; the address a kernel
// can use has to be looked up, once per device, with that device current.
void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

fa_status fa_backward_noalloc(const fa_dims* dims, const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* L, void* dQ, void* dK, void* dV, void* stream) {
  const size_t need = fa_backward_workspace_min_bytes(dims);  // 0 for invalid dims: rejected below
  if (need > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_TOO_SMALL;
  void* scratch = scratch_for_current_device();
  if (!scratch) return FA_ERR_CUDA;
  return fa_backward_stages(dims, Q, K, V, O, dO, L, dQ, dK, dV, scratch, (size_t)FA_NOALLOC_SCRATCH_BYTES,
                            FA_BWD_ALL, stream);
}

}  // extern "C"
