// Non-causal linear attention with per-sequence valid lengths (CUDA cores).
//
// Method: "Linear Attention/zh", kernel reformulation: one shared
//   S = sum_{j<L} phi(K_j) V_j^T,  Z = sum_{j<L} phi(K_j)
// per (b, h), read by every query: out_i = phi(Q_i)^T S / phi(Q_i)^T Z.
// The gradients are eq. 13-15 of "Transformers are RNNs" (part 2/3) with the
// cumulative sums replaced by full sums over the valid rows, plus the
// denominator terms of the quotient rule:
//   grad_phiQ_i = S gt_i + gam_i Z,  R = sum_i phi(Q_i) gt_i^T,  r = sum_i gam_i phi(Q_i),
//   grad_phiK_j = R V_j + r,         dv_j = R^T phi(K_j).
// Rows i >= L are padding: they contribute nothing and are written as zero.
//
// Decomposition: segments of whole chunks write partial sums to the
// workspace, a reduction kernel sums them per (b, h), and a per-token kernel
// reads the shared state.
#include "common.cuh"
#include "launch.h"

namespace la {
namespace {

constexpr int C = kChunk;
constexpr int NT = 256;

__device__ __forceinline__ long valid_len(const int* lengths, int b, int N) {
  if (lengths == nullptr) return N;
  const int L = lengths[b];
  return L < 0 ? 0 : (L > N ? N : L);
}

// Partial S, Z of one segment: ws[bh][p] = [ dS (D x M) | dz (D) ].
template <int D, int M, typename T>
__global__ void __launch_bounds__(NT) k_nc_state(const T* __restrict__ k, const T* __restrict__ v,
                                                 const int* __restrict__ lengths, float* ws,
                                                 int N, int H, int nseg, int seg_len) {
  const int p = blockIdx.x, bh = blockIdx.y;
  extern __shared__ float sm[];
  float* sK = sm;
  float* sV = sK + C * (D + 1);
  const long L = valid_len(lengths, bh / H, N);
  const long nb = (long)p * seg_len, ne = min(L, nb + seg_len);
  const long hq = (long)bh * N * D, hv = (long)bh * N * M;
  float acc[D / 16][M / 16];
  zero_acc(acc);
  float zacc = 0.f;
  for (long n0 = nb; n0 < ne; n0 += C) {
    load_tile<T, C, D, false, kPhi>(sK, D + 1, k + hq, n0, ne);
    load_tile<T, C, M, false, kRaw>(sV, M + 1, v + hv, n0, ne);
    __syncthreads();
    smem_mm<D / 16, M / 16, C>(acc, sK, 1, D + 1, sV, M + 1, 1);
    if (threadIdx.x < D)
      for (int j = 0; j < C; ++j) zacc += sK[j * (D + 1) + threadIdx.x];
    __syncthreads();
  }
  float* dst = ws + ((long)bh * nseg + p) * (D * M + D);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int r = 0; r < D / 16; ++r)
#pragma unroll
    for (int c = 0; c < M / 16; ++c) dst[(ty + 16 * r) * M + tx + 16 * c] = acc[r][c];
  if (threadIdx.x < D) dst[D * M + threadIdx.x] = zacc;
}

// gt = G / den and gam = -(gt . O) for the chunk's rows (zero past ne).
template <typename T, int M>
__device__ __forceinline__ void grad_terms(float* sG, float* sO, float* sden, float* sgam,
                                           const T* gh, const T* oh, const float* denh, long n0,
                                           long ne) {
  load_tile<T, C, M, false, kRaw>(sG, M + 1, gh, n0, ne);
  load_tile<T, C, M, false, kRaw>(sO, M + 1, oh, n0, ne);
  if (threadIdx.x < C) sden[threadIdx.x] = (n0 + threadIdx.x < ne) ? denh[n0 + threadIdx.x] : 1.f;
  __syncthreads();
  for (int e = threadIdx.x; e < C * M; e += NT) {
    const int i = e / M, m = e % M;
    sG[i * (M + 1) + m] = sG[i * (M + 1) + m] / sden[i];
  }
  __syncthreads();
  if (threadIdx.x < C) {
    float s = 0.f;
    for (int m = 0; m < M; ++m) s += sG[threadIdx.x * (M + 1) + m] * sO[threadIdx.x * (M + 1) + m];
    sgam[threadIdx.x] = -s;
  }
}

// Partial R, r of one segment: ws[bh][p] = [ dR (D x M) | dr (D) ].
template <int D, int M, typename T>
__global__ void __launch_bounds__(NT) k_nc_state_bwd(const T* __restrict__ q,
                                                     const T* __restrict__ o,
                                                     const float* __restrict__ den,
                                                     const T* __restrict__ g,
                                                     const int* __restrict__ lengths, float* ws,
                                                     int N, int H, int nseg, int seg_len) {
  const int p = blockIdx.x, bh = blockIdx.y;
  extern __shared__ float sm[];
  float* sQ = sm;
  float* sG = sQ + C * (D + 1);
  float* sO = sG + C * (M + 1);
  float* sden = sO + C * (M + 1);
  float* sgam = sden + C;
  const long L = valid_len(lengths, bh / H, N);
  const long nb = (long)p * seg_len, ne = min(L, nb + seg_len);
  const long hq = (long)bh * N * D, hv = (long)bh * N * M;
  float acc[D / 16][M / 16];
  zero_acc(acc);
  float racc = 0.f;
  for (long n0 = nb; n0 < ne; n0 += C) {
    load_tile<T, C, D, false, kPhi>(sQ, D + 1, q + hq, n0, ne);
    grad_terms<T, M>(sG, sO, sden, sgam, g + hv, o + hv, den + (long)bh * N, n0, ne);
    __syncthreads();
    smem_mm<D / 16, M / 16, C>(acc, sQ, 1, D + 1, sG, M + 1, 1);
    if (threadIdx.x < D)
      for (int i = 0; i < C; ++i) racc += sgam[i] * sQ[i * (D + 1) + threadIdx.x];
    __syncthreads();
  }
  float* dst = ws + ((long)bh * nseg + p) * (D * M + D);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int r = 0; r < D / 16; ++r)
#pragma unroll
    for (int c = 0; c < M / 16; ++c) dst[(ty + 16 * r) * M + tx + 16 * c] = acc[r][c];
  if (threadIdx.x < D) dst[D * M + threadIdx.x] = racc;
}

// Sums the nseg records of each (b, h): entries [0, DM) go to dA[bh][.],
// entries [DM, DM + D) to dB[bh][.].
__global__ void k_seg_sum(const float* ws, int nseg, int DM, int D, float* dA, float* dB) {
  const int bh = blockIdx.x, stride = DM + D;
  const float* base = ws + (long)bh * nseg * stride;
  const int e = blockIdx.y * blockDim.x + threadIdx.x;
  if (e < stride) {
    float s = 0.f;
    for (int p = 0; p < nseg; ++p) s += base[(long)p * stride + e];
    if (e < DM)
      dA[(long)bh * DM + e] = s;
    else
      dB[(long)bh * D + e - DM] = s;
  }
}

// Loads S [D][M] (global, row-major) into shared memory [D][M+1] and Z [D].
template <int D, int M>
__device__ __forceinline__ void load_state(float* sS, float* sz, const float* S, const float* Z) {
  for (int e = threadIdx.x; e < D * M; e += NT) sS[(e / M) * (M + 1) + e % M] = S[e];
  if (threadIdx.x < D) sz[threadIdx.x] = Z[threadIdx.x];
}

// out_i = phi(Q_i)^T S / phi(Q_i)^T Z for i < L; zero rows (and den) after.
template <int D, int M, typename T>
__global__ void __launch_bounds__(NT) k_nc_out(const T* __restrict__ q, const float* __restrict__ S,
                                               const float* __restrict__ Z,
                                               const int* __restrict__ lengths,
                                               T* __restrict__ out, float* __restrict__ den, int N,
                                               int H, int nseg, int seg_len) {
  const int p = blockIdx.x, bh = blockIdx.y;
  extern __shared__ float sm[];
  float* sQ = sm;
  float* sS = sQ + C * (D + 1);
  float* sz = sS + D * (M + 1);
  float* sden = sz + D;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const long L = valid_len(lengths, bh / H, N);
  const long nb = (long)p * seg_len, ne = min((long)N, nb + seg_len), nv = min(ne, L);
  const long hq = (long)bh * N * D, hv = (long)bh * N * M;
  load_state<D, M>(sS, sz, S + (long)bh * D * M, Z + (long)bh * D);
  for (long n0 = nb; n0 < ne; n0 += C) {
    load_tile<T, C, D, false, kPhi>(sQ, D + 1, q + hq, n0, nv);
    __syncthreads();
    if (threadIdx.x < C) {
      const int i = threadIdx.x;
      float s = 0.f;
      for (int d = 0; d < D; ++d) s += sQ[i * (D + 1) + d] * sz[d];
      sden[i] = s;
      if (den != nullptr && n0 + i < ne) den[(long)bh * N + n0 + i] = n0 + i < nv ? s : 0.f;
    }
    __syncthreads();
    float o[C / 16][M / 16];
    zero_acc(o);
    smem_mm<C / 16, M / 16, D>(o, sQ, D + 1, 1, sS, M + 1, 1);
#pragma unroll
    for (int r = 0; r < C / 16; ++r) {
      const int i = ty + 16 * r;
      if (n0 + i < ne) {
        const bool valid = n0 + i < nv;
        const float inv = valid ? 1.f / sden[i] : 0.f;
#pragma unroll
        for (int c = 0; c < M / 16; ++c)
          out[hv + (n0 + i) * M + tx + 16 * c] = from_f<T>(valid ? o[r][c] * inv : 0.f);
      }
    }
    __syncthreads();
  }
}

// Per-token gradients from the shared S, Z and the reduced R, r.
template <int D, int M, typename T>
__global__ void __launch_bounds__(NT) k_nc_bwd(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const T* __restrict__ o, const float* __restrict__ den, const T* __restrict__ g,
    const float* __restrict__ S, const float* __restrict__ Z, const float* __restrict__ R,
    const float* __restrict__ r, const int* __restrict__ lengths, T* __restrict__ dq,
    T* __restrict__ dk, T* __restrict__ dv, int N, int H, int nseg, int seg_len) {
  const int p = blockIdx.x, bh = blockIdx.y;
  extern __shared__ float sm[];
  float* sK = sm;                  // phi(K) [C][D+1]
  float* sV = sK + C * (D + 1);    // V      [C][M+1]
  float* sG = sV + C * (M + 1);    // gt     [C][M+1]
  float* sO = sG + C * (M + 1);    // O      [C][M+1]
  float* sS = sO + C * (M + 1);    // S      [D][M+1]
  float* sR = sS + D * (M + 1);    // R      [D][M+1]
  float* sz = sR + D * (M + 1);    // Z      [D]
  float* sr = sz + D;              // r      [D]
  float* sden = sr + D;            // [C]
  float* sgam = sden + C;          // [C]
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const long L = valid_len(lengths, bh / H, N);
  const long nb = (long)p * seg_len, ne = min((long)N, nb + seg_len), nv = min(ne, L);
  const long hq = (long)bh * N * D, hv = (long)bh * N * M;
  load_state<D, M>(sS, sz, S + (long)bh * D * M, Z + (long)bh * D);
  load_state<D, M>(sR, sr, R + (long)bh * D * M, r + (long)bh * D);
  for (long n0 = nb; n0 < ne; n0 += C) {
    load_tile<T, C, D, false, kPhi>(sK, D + 1, k + hq, n0, nv);
    load_tile<T, C, M, false, kRaw>(sV, M + 1, v + hv, n0, nv);
    grad_terms<T, M>(sG, sO, sden, sgam, g + hv, o + hv, den + (long)bh * N, n0, nv);
    __syncthreads();
    {  // dq = (gt S^T + gam Z) * phi'(Q)
      float t[C / 16][D / 16];
      zero_acc(t);
      smem_mm<C / 16, D / 16, M>(t, sG, M + 1, 1, sS, 1, M + 1);
#pragma unroll
      for (int rr = 0; rr < C / 16; ++rr) {
        const int i = ty + 16 * rr;
        if (n0 + i < ne) {
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            const int d = tx + 16 * c;
            const long idx = hq + (n0 + i) * D + d;
            float val = 0.f;
            if (n0 + i < nv) val = (t[rr][c] + sgam[i] * sz[d]) * dphi(to_f(q[idx]));
            dq[idx] = from_f<T>(val);
          }
        }
      }
    }
    {  // dk = (V R^T + r) * phi'(K)
      float t[C / 16][D / 16];
      zero_acc(t);
      smem_mm<C / 16, D / 16, M>(t, sV, M + 1, 1, sR, 1, M + 1);
#pragma unroll
      for (int rr = 0; rr < C / 16; ++rr) {
        const int j = ty + 16 * rr;
        if (n0 + j < ne) {
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            const int d = tx + 16 * c;
            const long idx = hq + (n0 + j) * D + d;
            float val = 0.f;
            if (n0 + j < nv) val = (t[rr][c] + sr[d]) * dphi(to_f(k[idx]));
            dk[idx] = from_f<T>(val);
          }
        }
      }
    }
    {  // dv = phi(K) R
      float u[C / 16][M / 16];
      zero_acc(u);
      smem_mm<C / 16, M / 16, D>(u, sK, D + 1, 1, sR, M + 1, 1);
#pragma unroll
      for (int rr = 0; rr < C / 16; ++rr) {
        const int j = ty + 16 * rr;
        if (n0 + j < ne) {
#pragma unroll
          for (int c = 0; c < M / 16; ++c)
            dv[hv + (n0 + j) * M + tx + 16 * c] = from_f<T>(n0 + j < nv ? u[rr][c] : 0.f);
        }
      }
    }
    __syncthreads();
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int D, int M, typename T>
cudaError_t run_fwd(const T* q, const T* k, const T* v, const int* lengths, T* out, float* den,
                    float* S, float* Z, float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const SegPlan pl = plan_segments(BH, s.N);
  cudaError_t e;
  const size_t sm_state = sizeof(float) * (C * (D + 1) + C * (M + 1));
  const size_t sm_out = sizeof(float) * (C * (D + 1) + D * (M + 1) + D + C);
  auto ks = k_nc_state<D, M, T>;
  auto ko = k_nc_out<D, M, T>;
  if ((e = set_smem(ks, sm_state)) != cudaSuccess) return e;
  if ((e = set_smem(ko, sm_out)) != cudaSuccess) return e;
  ks<<<dim3(pl.nseg, BH), NT, sm_state, st>>>(k, v, lengths, ws, s.N, s.H, pl.nseg, pl.seg_len);
  k_seg_sum<<<dim3(BH, (D * M + D + 255) / 256), 256, 0, st>>>(ws, pl.nseg, D * M, D, S, Z);
  ko<<<dim3(pl.nseg, BH), NT, sm_out, st>>>(q, S, Z, lengths, out, den, s.N, s.H, pl.nseg,
                                            pl.seg_len);
  return cudaGetLastError();
}

template <int D, int M, typename T>
cudaError_t run_bwd(const T* q, const T* k, const T* v, const int* lengths, const T* o,
                    const float* den, const float* S, const float* Z, const T* g, T* dq, T* dk,
                    T* dv, float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const SegPlan pl = plan_segments(BH, s.N);
  cudaError_t e;
  float* R = ws + (size_t)BH * pl.nseg * (D * M + D);
  float* r = R + (size_t)BH * D * M;
  const size_t sm_state = sizeof(float) * (C * (D + 1) + 2 * C * (M + 1) + 2 * C);
  const size_t sm_main =
      sizeof(float) * (C * (D + 1) + 3 * C * (M + 1) + 2 * D * (M + 1) + 2 * D + 2 * C);
  auto ks = k_nc_state_bwd<D, M, T>;
  auto kb = k_nc_bwd<D, M, T>;
  if ((e = set_smem(ks, sm_state)) != cudaSuccess) return e;
  if ((e = set_smem(kb, sm_main)) != cudaSuccess) return e;
  ks<<<dim3(pl.nseg, BH), NT, sm_state, st>>>(q, o, den, g, lengths, ws, s.N, s.H, pl.nseg,
                                              pl.seg_len);
  k_seg_sum<<<dim3(BH, (D * M + D + 255) / 256), 256, 0, st>>>(ws, pl.nseg, D * M, D, R, r);
  kb<<<dim3(pl.nseg, BH), NT, sm_main, st>>>(q, k, v, o, den, g, S, Z, R, r, lengths, dq, dk, dv,
                                             s.N, s.H, pl.nseg, pl.seg_len);
  return cudaGetLastError();
}

bool use_tc(const Shape& s) { return s.D == 64 && s.M == 64; }

}  // namespace

size_t noncausal_fwd_ws_floats(const Shape& s) {
  if (use_tc(s)) return 0;
  const SegPlan pl = plan_segments(s.B * s.H, s.N);
  return (size_t)s.B * s.H * pl.nseg * (s.D * s.M + s.D);
}

size_t noncausal_bwd_ws_floats(const Shape& s) {
  if (use_tc(s)) return 0;
  const SegPlan pl = plan_segments(s.B * s.H, s.N);
  return (size_t)s.B * s.H * (pl.nseg + 1) * (s.D * s.M + s.D);
}

int noncausal_fwd_launches(const Shape& s) { return use_tc(s) ? 1 : 3; }

int noncausal_bwd_launches(const Shape& s) { return use_tc(s) ? 1 : 3; }

cudaError_t noncausal_fwd_cc(const void* q, const void* k, const void* v, const int* lengths,
                             void* out, float* den, float* S, float* Z, float* ws, const Shape& s,
                             cudaStream_t st) {
  if (use_tc(s)) return noncausal_tc_fwd(q, k, v, lengths, out, den, S, Z, s, st);
  if (s.dtype == 0) {
    using T = float;
    LA_DISPATCH_DM(s.D, s.M,
                   return (run_fwd<D_, M_, T>((const T*)q, (const T*)k, (const T*)v, lengths,
                                              (T*)out, den, S, Z, ws, s, st)));
  } else {
    using T = __nv_bfloat16;
    LA_DISPATCH_DM(s.D, s.M,
                   return (run_fwd<D_, M_, T>((const T*)q, (const T*)k, (const T*)v, lengths,
                                              (T*)out, den, S, Z, ws, s, st)));
  }
  return cudaErrorInvalidValue;
}

cudaError_t noncausal_bwd_cc(const void* q, const void* k, const void* v, const int* lengths,
                             const void* out, const float* den, const float* S, const float* Z,
                             const void* dout, void* dq, void* dk, void* dv, float* ws,
                             const Shape& s, cudaStream_t st) {
  if (use_tc(s))  // out is not read: gam comes from the dq accumulator
    return noncausal_tc_bwd(q, k, v, lengths, den, S, Z, dout, dq, dk, dv, s, st);
  if (s.dtype == 0) {
    using T = float;
    LA_DISPATCH_DM(s.D, s.M,
                   return (run_bwd<D_, M_, T>((const T*)q, (const T*)k, (const T*)v, lengths,
                                              (const T*)out, den, S, Z, (const T*)dout, (T*)dq,
                                              (T*)dk, (T*)dv, ws, s, st)));
  } else {
    using T = __nv_bfloat16;
    LA_DISPATCH_DM(s.D, s.M,
                   return (run_bwd<D_, M_, T>((const T*)q, (const T*)k, (const T*)v, lengths,
                                              (const T*)out, den, S, Z, (const T*)dout, (T*)dq,
                                              (T*)dk, (T*)dv, ws, s, st)));
  }
  return cudaErrorInvalidValue;
}

}  // namespace la
