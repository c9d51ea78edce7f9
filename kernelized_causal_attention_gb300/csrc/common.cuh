// Shared device helpers of the CUDA library (never used by the CPU oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace la {

// eq. 7 of "Transformers are RNNs" (part 2/3): phi(x) = elu(x) + 1, alpha = 1.
// The exponential is CUDA's own expf.
__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.f : expf(x); }
// Derivative of eq. 7: 1 for x > 0, exp(x) otherwise.
__device__ __forceinline__ float dphi(float x) { return x > 0.f ? 1.f : expf(x); }

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Unpacks one 16-byte vector of T into floats (4 fp32 or 8 bf16 values).
template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int n = 4;
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

enum TileOp { kRaw = 0, kPhi = 1, kDphi = 2 };

// Stages rows [n0, n0 + ROWS) of a row-major [*, W] global matrix into shared
// memory as fp32, applying op (raw, phi or phi').  Rows at or past n_end are
// written as zero (so a zeroed phi(K) row contributes nothing to any sum).
// TRANS = false stores s[r * ld + w]; TRANS = true stores s[w * ld + r].
// 16-byte vectorised, coalesced global reads.
template <typename T, int ROWS, int W, bool TRANS, int OP>
__device__ __forceinline__ void load_tile(float* s, int ld, const T* g, long n0, long n_end) {
  constexpr int VN = Vec16<T>::n;
  constexpr int VPR = W / VN;  // vectors per row
  for (int e = threadIdx.x; e < ROWS * VPR; e += blockDim.x) {
    const int r = e / VPR, c = (e % VPR) * VN;
    float f[VN];
    if (n0 + r < n_end) {
      const uint4 u = *reinterpret_cast<const uint4*>(g + (n0 + r) * W + c);
      Vec16<T>::unpack(u, f);
#pragma unroll
      for (int i = 0; i < VN; ++i) f[i] = OP == kPhi ? phi(f[i]) : (OP == kDphi ? dphi(f[i]) : f[i]);
    } else {
#pragma unroll
      for (int i = 0; i < VN; ++i) f[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < VN; ++i) {
      if (TRANS)
        s[(c + i) * ld + r] = f[i];
      else
        s[r * ld + c + i] = f[i];
    }
  }
}

// Register-tiled shared-memory product on a 16 x 16 thread grid (256 threads):
//   acc[r][c] += sum_k X(i, k) * Y(k, j),  i = ty + 16 r,  j = tx + 16 c,
// with X(i, k) = X[i * xi + k * xk] and Y(k, j) = Y[k * yk + j * yj].
// Rows and columns are strided by 16 so that, with odd leading dimensions,
// every shared load is either a broadcast or conflict-free.
template <int RR, int CC, int K>
__device__ __forceinline__ void smem_mm(float (&acc)[RR][CC], const float* X, int xi, int xk,
                                        const float* Y, int yk, int yj) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
  for (int k = 0; k < K; ++k) {
    float a[RR], b[CC];
#pragma unroll
    for (int r = 0; r < RR; ++r) a[r] = X[(ty + 16 * r) * xi + k * xk];
#pragma unroll
    for (int c = 0; c < CC; ++c) b[c] = Y[k * yk + (tx + 16 * c) * yj];
#pragma unroll
    for (int r = 0; r < RR; ++r)
#pragma unroll
      for (int c = 0; c < CC; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}

template <int RR, int CC>
__device__ __forceinline__ void zero_acc(float (&acc)[RR][CC]) {
#pragma unroll
  for (int r = 0; r < RR; ++r)
#pragma unroll
    for (int c = 0; c < CC; ++c) acc[r][c] = 0.f;
}

}  // namespace la
