// noalloc.cu -- domino_mlp_fwd_noalloc: the MLP forward with its scratch memory taken from a
// fixed array inside the library instead of a caller-supplied workspace.
//
// Who needs this: callers that cannot allocate device memory at the point where they run the
// layer -- for example a plugin hosted by a framework that owns the whole device memory pool and
// hands out no workspace, a serving loop that forbids allocations after warm-up so its memory
// footprint stays fixed, or code that must not risk the device-wide synchronisation that
// cudaMalloc/cudaFree can cause.  They still pass X, A, B, Y (and optionally act_save); only the
// scratch (the first-linear output H of one row chunk and the fp32 shard partials) comes from
// here.
//
// The scratch array costs kStaticScratchBytes of device memory on every GPU that loads the
// library, for as long as the process lives.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/domino.h"

namespace dm {
void set_last_error(const std::string& msg);
domino_status check_handle(domino_handle H);
}

static constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB

// File-scope scratch.  Host code must not use its name as a pointer: on the host the symbol is
// only a handle, so the device address is looked up per device below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device `dev`.  Outside stream capture it is
// looked up on every call (cheap once the module is loaded), so a device reset that moved the
// array cannot leave a stale address behind; while `stream` is being captured into a graph the
// address of the last uncaptured call on this device is used, since the lookup may have to load
// the module, which capture does not allow.
cudaError_t scratch_address(int dev, cudaStream_t stream, void** out) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  if (cap != cudaStreamCaptureStatusNone) {
    if (g_scratch_ptr[dev] == nullptr) return cudaErrorStreamCaptureUnsupported;
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return e;
  g_scratch_ptr[dev] = p;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" {

domino_status domino_mlp_fwd_noalloc(domino_handle handle, const domino_cfg* cfg, const uint16_t* X,
                                     const uint16_t* A, const uint16_t* B, uint16_t* Y,
                                     uint16_t* act_save, void* stream) {
  // the cheap checks come first: nothing touches the device for a bad handle or problem
  domino_status s = dm::check_handle(handle);
  if (s != DOMINO_OK) return s;
  size_t need = 0;
  s = domino_workspace_size(cfg, DOMINO_PASS_FWD, &need);
  if (s != DOMINO_OK) return s;
  if (need > kStaticScratchBytes) {
    dm::set_last_error("domino_mlp_fwd_noalloc: this problem needs " + std::to_string(need) +
                       " bytes of scratch but the built-in scratch holds " +
                       std::to_string(kStaticScratchBytes) + " bytes; use domino_mlp_fwd with a workspace");
    return DOMINO_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
  void* scratch = nullptr;
  if (e == cudaSuccess) e = scratch_address(dev, static_cast<cudaStream_t>(stream), &scratch);
  if (e != cudaSuccess) {
    dm::set_last_error(std::string("domino_mlp_fwd_noalloc: scratch set-up failed (the first call on a device "
                                   "must come before any stream capture): ") + cudaGetErrorString(e));
    return DOMINO_ERR_CUDA;
  }
  // The forward overwrites every scratch byte it reads (H and the partials), so nothing from a
  // previous call has to be cleared.
  return domino_mlp_fwd(handle, cfg, X, A, B, Y, act_save, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
