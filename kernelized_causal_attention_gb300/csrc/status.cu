// The library's device status word and the calls that read and exercise it.
//
// Every wait in the tensor-core kernels (on an mbarrier, a TMA copy, an MMA
// commit) is bounded in time.  A wait that runs out stores a small nonzero
// code naming its site here (the first such code sticks), sets the CTA's
// abort flag so that every thread still reaches each barrier, drains what
// it has in flight with bounded waits, frees its tensor memory and returns.
// The context stays usable and the host learns of it through
// la_device_status.
#include <atomic>

#include "../../include/linattn.h"
#include "launch.h"
#include "tc.cuh"

namespace la {

namespace {

__device__ int g_status;

constexpr int kSelftestCode = 99;

// One thread waits on an mbarrier that nothing arrives at, with the same
// bounded wait the kernels use, and records the expiry.
__global__ void k_selftest_wait(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, limit_ns) && status != nullptr)
    atomicCAS(status, 0, kSelftestCode);
}

constexpr int kMaxDevices = 64;
std::atomic<int*> g_word[kMaxDevices];

}  // namespace

int* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* p = g_word[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_status) != cudaSuccess) return nullptr;
    p = static_cast<int*>(a);
    g_word[dev].store(p, std::memory_order_release);
  }
  return p;
}

int sm_count() {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 152;
  }
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 152;
    }
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace la

extern "C" {

int la_device_status(void* stream, int clear, int* code) {
  if (code != nullptr) *code = 0;
  int* w = la::status_word();
  if (w == nullptr) return LA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, w, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return LA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return LA_ERR_CUDA;
  if (clear && v != 0) {
    if (cudaMemsetAsync(w, 0, sizeof(int), st) != cudaSuccess) return LA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LA_ERR_CUDA;
  }
  if (code != nullptr) *code = v;
  return v != 0 ? LA_ERR_TIMEOUT : LA_OK;
}

int la_selftest_wait(void* stream, unsigned long long limit_ns) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return LA_ERR_INVALID_ARG;
  int* w = la::status_word();
  if (w == nullptr) return LA_ERR_CUDA;
  la::k_selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(w, limit_ns);
  return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // extern "C"
