// RNN-form decode step, "Transformers are RNNs" (part 2/3) §3.4 eq. 16-19:
//   s <- s + phi(k) v^T,  z <- z + phi(k),  y = phi(q)^T s / phi(q)^T z
// for B*H independent streams, with the fp32 state updated in place.  With the
// RetNet decay of "Linear Attention/zh" (variants and extensions) the state is
// decayed first: s <- gamma s + phi(k) v^T, z <- gamma z + phi(k).
//
// The step is bound by HBM traffic on the state (read and write D*M*4 bytes
// per stream); the kernel streams each stream's S once with 16-byte
// vectorised, coalesced loads and stores, and folds the read-out into the same
// pass (y uses the updated rows while they are still in registers).
#include "common.cuh"
#include "launch.h"

namespace la {
namespace {

constexpr int NT = 256;

template <int D, int M, typename T, bool DECAY>
__global__ void __launch_bounds__(NT) k_decode(const T* __restrict__ q, const T* __restrict__ k,
                                               const T* __restrict__ v, float* __restrict__ S,
                                               float* __restrict__ Z, T* __restrict__ y,
                                               float gamma) {
  constexpr int M4 = M / 4;                 // float4 columns of one state row
  constexpr int RG = NT / M4;               // threads sharing one column group
  constexpr int RPT = (D + RG - 1) / RG;    // state rows per thread
  __shared__ float sfk[D], sfq[D], sv[M], sden[2];
  __shared__ float4 sred[RG][M4];
  const int bh = blockIdx.x, tid = threadIdx.x;
  if (tid < D) {
    sfk[tid] = phi(to_f(k[(long)bh * D + tid]));
    sfq[tid] = phi(to_f(q[(long)bh * D + tid]));
  }
  if (tid < M) sv[tid] = to_f(v[(long)bh * M + tid]);
  __syncthreads();

  const int c4 = tid % M4, rg = tid / M4;
  float4* Sh = reinterpret_cast<float4*>(S + (long)bh * D * M);
  float4 s[RPT];
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    const int d = rg + r * RG;
    if (d < D) s[r] = Sh[d * M4 + c4];
  }
  const float v0 = sv[4 * c4], v1 = sv[4 * c4 + 1], v2 = sv[4 * c4 + 2], v3 = sv[4 * c4 + 3];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    const int d = rg + r * RG;
    if (d < D) {
      const float fk = sfk[d], fq = sfq[d];
      if (DECAY) {
        s[r].x *= gamma;
        s[r].y *= gamma;
        s[r].z *= gamma;
        s[r].w *= gamma;
      }
      s[r].x = fmaf(fk, v0, s[r].x);
      s[r].y = fmaf(fk, v1, s[r].y);
      s[r].z = fmaf(fk, v2, s[r].z);
      s[r].w = fmaf(fk, v3, s[r].w);
      Sh[d * M4 + c4] = s[r];
      acc.x = fmaf(fq, s[r].x, acc.x);
      acc.y = fmaf(fq, s[r].y, acc.y);
      acc.z = fmaf(fq, s[r].z, acc.z);
      acc.w = fmaf(fq, s[r].w, acc.w);
    }
  }
  sred[rg][c4] = acc;

  // z <- z + phi(k);  den = phi(q) . z
  float dp = 0.f;
  if (tid < D) {
    const float z = (DECAY ? gamma * Z[(long)bh * D + tid] : Z[(long)bh * D + tid]) + sfk[tid];
    Z[(long)bh * D + tid] = z;
    dp = sfq[tid] * z;
  }
  if (tid < 64) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dp += __shfl_xor_sync(0xffffffffu, dp, off);
    if ((tid & 31) == 0) sden[tid >> 5] = dp;
  }
  __syncthreads();
  if (tid < M) {
    const float den = sden[0] + (D > 32 ? sden[1] : 0.f);
    const int cc = tid / 4, lane = tid % 4;
    float num = 0.f;
    for (int g = 0; g < RG; ++g) {
      const float4 t = sred[g][cc];
      num += lane == 0 ? t.x : (lane == 1 ? t.y : (lane == 2 ? t.z : t.w));
    }
    y[(long)bh * M + tid] = from_f<T>(num / den);
  }
}

}  // namespace

cudaError_t decode_step(const void* q, const void* k, const void* v, float* S, float* Z, void* y,
                        const Shape& s, cudaStream_t st, float gamma) {
  const int BH = s.B * s.H;
  const bool dec = gamma != 1.f;
  if (s.dtype == 0) {
    using T = float;
    if (dec) {
      LA_DISPATCH_DM(s.D, s.M,
                     (k_decode<D_, M_, T, true><<<BH, NT, 0, st>>>((const T*)q, (const T*)k,
                                                                   (const T*)v, S, Z, (T*)y, gamma)));
    } else {
      LA_DISPATCH_DM(s.D, s.M,
                     (k_decode<D_, M_, T, false><<<BH, NT, 0, st>>>((const T*)q, (const T*)k,
                                                                    (const T*)v, S, Z, (T*)y, 1.f)));
    }
  } else {
    using T = __nv_bfloat16;
    if (dec) {
      LA_DISPATCH_DM(s.D, s.M,
                     (k_decode<D_, M_, T, true><<<BH, NT, 0, st>>>((const T*)q, (const T*)k,
                                                                   (const T*)v, S, Z, (T*)y, gamma)));
    } else {
      LA_DISPATCH_DM(s.D, s.M,
                     (k_decode<D_, M_, T, false><<<BH, NT, 0, st>>>((const T*)q, (const T*)k,
                                                                    (const T*)v, S, Z, (T*)y, 1.f)));
    }
  }
  return cudaGetLastError();
}

}  // namespace la
