// la_causal_fwd_noalloc: the causal forward with its scratch memory taken from
// a fixed array that lives in the library itself, for callers that must not
// allocate device memory.
//
// Who needs this: code that runs inside a host application which owns every
// byte of device memory (a plug-in inside an inference server or engine with
// a fixed, pre-reserved memory budget and no allocator handed to plug-ins), and
// latency-critical loops where a cudaMalloc -- which may synchronise the whole
// device and take milliseconds -- is not acceptable.  Such a caller still owns
// its inputs and outputs; only the workspace moves into the library.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/linattn.h"
#include "launch.h"

namespace {

// The scratch array.  Every GPU that loads this library holds it until the
// process exits.  All calls on a device share it.
static __device__ __align__(256) unsigned char g_la_scratch[LA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device (in host code the array's name is only a host-side stand-in, never a
// device address).  The cached address stays valid for the life of the CUDA
// context; a cudaDeviceReset after the first call invalidates it (see the
// header).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_la_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LA_OK;
}

}  // namespace

extern "C" int la_causal_fwd_noalloc(const void* q, const void* k, const void* v, void* out,
                                     float* den, int B, int H, int N, int D, int M, int dtype,
                                     void* stream) {
  // the same argument checks as la_causal_fwd, first, so that a bad call gets
  // the same error code whether or not a device is usable
  const int chk = la::causal_fwd_check(q, k, v, out, den, B, H, N, D, M, dtype);
  if (chk != LA_OK) return chk;
  const size_t need = la_workspace_bytes(LA_OP_CAUSAL_FWD, B, H, N, D, M, dtype);
  if (need > LA_NOALLOC_SCRATCH_BYTES) return LA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != LA_OK) return rc;
  // Nothing in the scratch array needs to start at zero: every entry the
  // forward reads there was written earlier in the same call.  Timeouts of
  // bounded waits are not kept here; they go to the library's status word,
  // which stays set until the caller clears it with la_device_status.
  return la_causal_fwd(q, k, v, out, den, scratch, LA_NOALLOC_SCRATCH_BYTES, B, H, N, D, M, dtype,
                       stream);
}
