// Forward pass that allocates nothing and needs no caller-provided workspace.
//
// Who needs this: callers that cannot call cudaMalloc (or any allocator) at the point
// where they compute the loss — for example a C plug-in inside another runtime that
// owns all device memory through its own pool and forbids further driver allocations,
// a serving process that reserves its memory once at start-up, or a latency-critical
// path where an allocation's implicit synchronisation is not acceptable.  They still
// pass their own inputs and outputs; only the forward's scratch comes from here.
//
// The scratch is one file-scope __device__ array of kStaticScratchBytes.  Every GPU
// that loads this library holds that much memory until the process exits.  In host
// code the array's name is only a host-side stand-in, so the device address is looked
// up once per device with cudaGetSymbolAddress (with that device current) and passed
// to the kernels like any workspace pointer.  Under CUDA's lazy module loading the
// lookup is also what loads the module on that device, so the first call per device
// may reserve the 16 MiB and synchronise; callers that cannot accept that make their
// first call at start-up.
#include <cuda_runtime.h>

#include <mutex>

#include "flce.h"
#include "host_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void* g_scratch[kMaxDevices] = {};  // device address per device, once looked up
std::mutex g_scratch_mu;

// Device address of the static scratch on the current device.  The device is checked
// first (an unsupported GPU gets FLCE_ERR_UNSUPPORTED, as from flce_forward); only a
// successful lookup is kept, so a failed one (say, made during a stream capture) is
// retried by the next call, and its error is what flce_last_cuda_error() reports.
flce_status static_scratch(void** out) {
  const int st = flce::check_device();
  if (st != FLCE_OK) return static_cast<flce_status>(st);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<flce_status>(flce::record_cuda_error(e));
  if (dev < 0 || dev >= kMaxDevices) return FLCE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return static_cast<flce_status>(flce::record_cuda_error(e));
    if (p == nullptr) return static_cast<flce_status>(flce::record_cuda_error(cudaErrorInvalidSymbol));
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" {

FLCE_API size_t flce_static_scratch_bytes(void) { return kStaticScratchBytes; }

FLCE_API flce_status flce_forward_noalloc(const void* H, const void* W, const int64_t* labels, int64_t N,
                                          int64_t Hd, int64_t V, int64_t ignore_index, float softcap,
                                          int reduction, float* loss, float* lse, float* target_logit,
                                          int64_t* counts, void* stream) {
  const size_t need = flce_forward_workspace_size(N, Hd, V);
  if (need > kStaticScratchBytes) return FLCE_ERR_WORKSPACE;  // sizes beyond the static scratch
  void* scratch = nullptr;
  if (need > 0) {
    const flce_status s = static_scratch(&scratch);
    if (s != FLCE_OK) return s;
  }
  // need == 0 means invalid sizes (or nothing to do); flce_forward reports which.
  return flce_forward(H, W, labels, N, Hd, V, ignore_index, softcap, reduction, loss, lse, target_logit, counts,
                      scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
