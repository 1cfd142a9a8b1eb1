// fa_bwd_noalloc.cu -- fa_bwd_static_workspace(): the backward pass for
// callers that cannot allocate device memory.
//
// fa_bwd() needs scratch (the fp32 dQ accumulator and two per-row vectors)
// and asks the caller for it.  Some callers have no way to provide that: code
// that runs where device allocation is not permitted (for instance inside a
// host framework's execution step, where an allocation could block on the
// device or disturb a memory pool the framework manages), or code that simply
// has no allocator to call.  This entry point serves them by using a
// fixed-size scratch array that lives in the library's own device memory for
// as long as the library is loaded.  It performs no allocation of any kind.
//
// Limits and sharing:
//   * the array holds kNoAllocScratchBytes (64 MiB); problems whose
//     fa_bwd_workspace_bytes() exceeds that are refused with
//     FA_ERR_UNSUPPORTED before anything runs;
//   * the array belongs to this file's module of device code.  Under CUDA's
//     lazy module loading (the default) that module is loaded on a device,
//     and the 64 MiB committed there, by the first call on that device (the
//     address lookup below); with eager loading, when the library's code is
//     loaded onto the device.  Either way it stays until the process exits.
//     The first call may therefore allocate and synchronise inside the
//     driver: make it outside any region where that is not allowed;
//   * all calls share the one array, so calls whose work overlaps on the GPU
//     (for example on two concurrently running streams) race on it and give
//     wrong results; calls issued in order on one stream are fine.  Every
//     call re-initialises the parts that must start at zero (the prep kernel
//     zeroes the dQ accumulator and rewrites both vectors), so contents left
//     by an earlier call never leak into a later one.
//   * the array's device address is looked up (cudaGetSymbolAddress) by the
//     first call on each device, with that device current; make that first
//     call before any stream capture.
//   * arguments are checked exactly as fa_bwd checks them (same status
//     codes), before the size limit.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

// The scratch itself.  In host code this name is only a stand-in for the
// device array: its device address must be obtained with
// cudaGetSymbolAddress() on the device in question and passed to kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

struct ScratchAddr {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchAddr g_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  ScratchAddr& a = g_addr[dev];
  std::call_once(a.once, [&a]() {
    void* p = nullptr;
    a.err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    a.ptr = (a.err == cudaSuccess) ? p : nullptr;
  });
  *out = a.ptr;
  return a.err;
}

}  // namespace

extern "C" {

fa_status fa_bwd_static_workspace(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                  const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                  float scale, int window, fa_dtype dt, void* stream) {
  // fa_bwd's own argument checks first, so a bad argument gets the status
  // fa_bwd would give it whatever the problem's size; then the size limit.
  // Neither touches the device.
  const fa_status c = fa::check_bwd_args(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, window, dt);
  if (c != FA_OK) return c;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0) return FA_ERR_INVALID;
  if (need > kNoAllocScratchBytes) return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess || scratch == nullptr) return FA_ERR_CUDA;
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, window, dt, scratch, kNoAllocScratchBytes,
                stream);
}

}  // extern "C"
