// Causal linear attention on CUDA cores (fp32 FFMA), any supported dtype.
//
// Method: "Transformers are RNNs" (part 2/3), §3.3 eq. 9-12 (forward) and
// §3.3.1 eq. 13-15 (cumulative-sum backward, completed here with the
// denominator terms by the quotient rule).
//
// Work decomposition (the GB300 design, not the pages'): every (b, h)
// sequence is cut into segments of whole 64-token chunks so that the grid
// fills the SMs.  A first kernel writes each segment's partial sums
// (dS = sum phi(K) V^T, dz = sum phi(K); for the backward also
// dR = sum phi(Q) gt^T, dr = sum gam phi(Q)) to the workspace, a scan kernel
// turns them into exclusive prefix (S, z) and suffix (R, r) sums, and the
// main kernel walks its segment chunk by chunk, carrying S/z forward (or R/r
// backward) in fp32.  Inside a chunk the masked chunk-local terms are explicit
// 64 x 64 products, exactly the quadratic form of eq. 8 restricted to the
// chunk, and the earlier chunks enter through the carried state.
//
// The RetNet decay of "Linear Attention/zh" (variants and extensions),
// S_t = gamma S_{t-1} + phi(k_t) v_t^T with z decaying alongside S, weighs the
// pair (i, j) by gamma^(i-j).  With DECAY: the masks multiply each pair by
// gamma^(i-j) (a table of gamma^0 .. gamma^C); a query row i of a chunk reads
// the carried state with gamma^(i+1) and a key row j with gamma^(L-j) (L the
// chunk's valid length); the carried state decays by gamma^L per chunk, and a
// segment's record is taken relative to its last row (forward sums) or its
// first row (reverse sums), the scan decaying it by gamma^(segment length).
#include "common.cuh"
#include "launch.h"

namespace la {
namespace {

constexpr int C = kChunk;
constexpr int NT = 256;

// gamma^e from lg = log2(gamma) (lg = -inf for gamma = 0); gamma^0 = 1.
__device__ __forceinline__ float decay_pow(float lg, int e) {
  return e == 0 ? 1.f : exp2f(lg * static_cast<float>(e));
}

// Multiplies rows [0, C) of the [C][W+1] tile by gamma^(e0 + dir * row) for
// rows below `valid` (rows past it are zero anyway).
template <int W>
__device__ __forceinline__ void scale_rows(float* tile, float lg, int e0, int dir, int valid) {
  for (int e = threadIdx.x; e < C * W; e += NT) {
    const int j = e / W, w = e % W;
    if (j < valid) tile[j * (W + 1) + w] *= decay_pow(lg, e0 + dir * j);
  }
}

// ---------------------------------------------------------------- partial sums

// Per-segment sums of the forward state, eq. 10-11 restricted to the segment:
//   ws[bh][p] = [ dS (D x M) | dz (D) ]  (nrec records per (b, h)).
// The last segment's sums are only needed for the state after the sequence
// (all != 0); the forward itself reads exclusive prefixes only.
template <int D, int M, typename T, bool DECAY>
__global__ void __launch_bounds__(NT) k_seg_state_fwd(const T* __restrict__ k,
                                                      const T* __restrict__ v, float* ws, int N,
                                                      int nseg, int seg_len, int nrec, int all,
                                                      float lg) {
  const int p = blockIdx.x, bh = blockIdx.y;
  if (p == nseg - 1 && !all) return;
  extern __shared__ float sm[];
  float* sK = sm;                  // phi(K) [C][D+1]
  float* sV = sK + C * (D + 1);    // V      [C][M+1]
  const long nb = (long)p * seg_len, ne = min((long)N, nb + seg_len);
  const T* kh = k + (long)bh * N * D;
  const T* vh = v + (long)bh * N * M;
  float acc[D / 16][M / 16];
  zero_acc(acc);
  float zacc = 0.f;
  for (long n0 = nb; n0 < ne; n0 += C) {
    load_tile<T, C, D, false, kPhi>(sK, D + 1, kh, n0, ne);
    load_tile<T, C, M, false, kRaw>(sV, M + 1, vh, n0, ne);
    __syncthreads();
    if (DECAY) {  // relative to the segment's last row: gamma^(ne - 1 - row)
      scale_rows<D>(sK, lg, (int)(ne - 1 - n0), -1, (int)(ne - n0));
      __syncthreads();
    }
    smem_mm<D / 16, M / 16, C>(acc, sK, 1, D + 1, sV, M + 1, 1);
    if (threadIdx.x < D)
      for (int j = 0; j < C; ++j) zacc += sK[j * (D + 1) + threadIdx.x];
    __syncthreads();
  }
  float* dst = ws + ((long)bh * nrec + p) * (D * M + D);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int r = 0; r < D / 16; ++r)
#pragma unroll
    for (int c = 0; c < M / 16; ++c) dst[(ty + 16 * r) * M + tx + 16 * c] = acc[r][c];
  if (threadIdx.x < D) dst[D * M + threadIdx.x] = zacc;
}

// Loads the chunk's G and O, forms gt = G / den in place and
// gam = -(gt . O) per row (the quotient-rule terms of the backward pass).
// Rows past ne have G = 0, so gt = 0 and gam = 0 there.
template <typename T, int M>
__device__ __forceinline__ void load_grad_terms(float* sG, float* sO, float* sden, float* sgam,
                                                const T* gh, const T* oh, const float* denh,
                                                long n0, long ne) {
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

// Per-segment sums for the backward pass:
//   ws[bh][p] = [ dS (D x M) | dz (D) | dR (D x M) | dr (D) ]
// with dR = sum_i phi(Q_i) gt_i^T and dr = sum_i gam_i phi(Q_i) (the terms of
// the reverse cumulative sums of eq. 14-15).  dS/dz are skipped for the last
// segment and dR/dr for the first (never read).
template <int D, int M, typename T, bool DECAY>
__global__ void __launch_bounds__(NT) k_seg_state_bwd(const T* __restrict__ q,
                                                      const T* __restrict__ k,
                                                      const T* __restrict__ v,
                                                      const T* __restrict__ o,
                                                      const float* __restrict__ den,
                                                      const T* __restrict__ g, float* ws, int N,
                                                      int nseg, int seg_len, float lg) {
  const int p = blockIdx.x, bh = blockIdx.y;
  const bool want_s = p < nseg - 1, want_r = p > 0;
  extern __shared__ float sm[];
  float* sK = sm;                  // phi(K) [C][D+1]
  float* sQ = sK + C * (D + 1);    // phi(Q) [C][D+1]
  float* sV = sQ + C * (D + 1);    // V      [C][M+1]
  float* sG = sV + C * (M + 1);    // gt     [C][M+1]
  float* sO = sG + C * (M + 1);    // O      [C][M+1]
  float* sden = sO + C * (M + 1);  // [C]
  float* sgam = sden + C;          // [C]
  const long nb = (long)p * seg_len, ne = min((long)N, nb + seg_len);
  const long hq = (long)bh * N * D, hv = (long)bh * N * M;
  float accS[D / 16][M / 16], accR[D / 16][M / 16];
  zero_acc(accS);
  zero_acc(accR);
  float zacc = 0.f, racc = 0.f;
  for (long n0 = nb; n0 < ne; n0 += C) {
    if (want_s) {
      load_tile<T, C, D, false, kPhi>(sK, D + 1, k + hq, n0, ne);
      load_tile<T, C, M, false, kRaw>(sV, M + 1, v + hv, n0, ne);
    }
    if (want_r) {
      load_tile<T, C, D, false, kPhi>(sQ, D + 1, q + hq, n0, ne);
      load_grad_terms<T, M>(sG, sO, sden, sgam, g + hv, o + hv, den + (long)bh * N, n0, ne);
    }
    __syncthreads();
    if (DECAY) {  // forward sums relative to the segment's last row, reverse sums to its first
      if (want_s) scale_rows<D>(sK, lg, (int)(ne - 1 - n0), -1, (int)(ne - n0));
      if (want_r) scale_rows<D>(sQ, lg, (int)(n0 - nb), 1, (int)(ne - n0));
      __syncthreads();
    }
    if (want_s) {
      smem_mm<D / 16, M / 16, C>(accS, sK, 1, D + 1, sV, M + 1, 1);
      if (threadIdx.x < D)
        for (int j = 0; j < C; ++j) zacc += sK[j * (D + 1) + threadIdx.x];
    }
    if (want_r) {
      smem_mm<D / 16, M / 16, C>(accR, sQ, 1, D + 1, sG, M + 1, 1);
      if (threadIdx.x < D)
        for (int i = 0; i < C; ++i) racc += sgam[i] * sQ[i * (D + 1) + threadIdx.x];
    }
    __syncthreads();
  }
  float* dst = ws + ((long)bh * nseg + p) * 2 * (D * M + D);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int r = 0; r < D / 16; ++r)
#pragma unroll
    for (int c = 0; c < M / 16; ++c) {
      dst[(ty + 16 * r) * M + tx + 16 * c] = accS[r][c];
      dst[D * M + D + (ty + 16 * r) * M + tx + 16 * c] = accR[r][c];
    }
  if (threadIdx.x < D) {
    dst[D * M + threadIdx.x] = zacc;
    dst[2 * D * M + D + threadIdx.x] = racc;
  }
}

// In-place exclusive scans over the segments of each (b, h): entries
// [0, wf) of every record become prefix sums over earlier segments, entries
// [ro, ro + wr) suffix sums over later segments.  One thread per entry.
// With nrec > nseg, record nseg receives the forward totals.
// With the decay (lg = log2 gamma != 0) a record is relative to its segment's
// last row (forward) or first row (reverse), and the running sum decays by
// gamma^(segment length) when it passes a segment; lg = 0 multiplies by one.
__global__ void k_seg_scan(float* ws, int nseg, int stride, int wf, int ro, int wr, int nrec,
                           float lg, int seg_len, int N) {
  float* base = ws + (long)blockIdx.x * nrec * stride;
  const int e = blockIdx.y * blockDim.x + threadIdx.x;
  auto len = [&](int p) { return min(N - p * seg_len, seg_len); };
  if (e < wf) {
    float run = 0.f;
    for (int p = 0; p < nseg; ++p) {
      const float x = base[(long)p * stride + e];
      base[(long)p * stride + e] = run;
      run = lg != 0.f ? decay_pow(lg, len(p)) * run + x : run + x;
    }
    if (nrec > nseg) base[(long)nseg * stride + e] = run;
  }
  if (e < wr) {
    float run = 0.f;
    for (int p = nseg - 1; p >= 0; --p) {
      const float x = base[(long)p * stride + ro + e];
      base[(long)p * stride + ro + e] = run;
      run = lg != 0.f ? x + decay_pow(lg, len(p)) * run : run + x;
    }
  }
}

// ---------------------------------------------------------------- forward

// Causal forward, one CTA per (segment, b*h).  Per chunk:
//   A   = mask(phi(Q) phi(K)^T)                  (eq. 8 inside the chunk)
//   den = rowsum(A) + phi(Q) z                   (eq. 12 denominator)
//   out = (A V + phi(Q) S) / den                 (eq. 12 numerator)
//   S  += phi(K)^T V,  z += sum phi(K)           (eq. 10-11)
// S0, Z0 (may be null): a state the sums start from (eq. 16-19 over a prompt).
template <int D, int M, typename T, bool DECAY>
__global__ void __launch_bounds__(NT) k_causal_fwd(const T* __restrict__ q,
                                                   const T* __restrict__ k,
                                                   const T* __restrict__ v, T* __restrict__ out,
                                                   float* __restrict__ den,
                                                   const float* __restrict__ ws, int N, int nseg,
                                                   int seg_len, int nrec,
                                                   const float* __restrict__ S0,
                                                   const float* __restrict__ Z0, float lg) {
  const int p = blockIdx.x, bh = blockIdx.y;
  extern __shared__ float sm[];
  float* sQ = sm;                  // phi(Q) [C][D+1]
  float* sK = sQ + C * (D + 1);    // phi(K) [C][D+1]
  float* sV = sK + C * (D + 1);    // V      [C][M+1]
  float* sA = sV + C * (M + 1);    // A      [C][C+1]
  float* sS = sA + C * (C + 1);    // S      [D][M+1]
  float* sz = sS + D * (M + 1);    // z      [D]
  float* sden = sz + D;            // [C]
  float* spw = sden + C;           // gamma^0 .. gamma^C (with DECAY)
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const long nb = (long)p * seg_len, ne = min((long)N, nb + seg_len);
  const long hq = (long)bh * N * D, hv = (long)bh * N * M;
  if (DECAY && threadIdx.x <= C) spw[threadIdx.x] = decay_pow(lg, threadIdx.x);

  // exclusive prefix state of this segment (plus the initial state)
  const float* pre = ws + ((long)bh * nrec + p) * (D * M + D);
  float accS[D / 16][M / 16];
#pragma unroll
  for (int r = 0; r < D / 16; ++r)
#pragma unroll
    for (int c = 0; c < M / 16; ++c) {
      const int d = ty + 16 * r, m = tx + 16 * c;
      accS[r][c] = (p > 0 ? pre[d * M + m] : 0.f) + (S0 != nullptr ? S0[(long)bh * D * M + d * M + m] : 0.f);
      sS[d * (M + 1) + m] = accS[r][c];
    }
  if (threadIdx.x < D)
    sz[threadIdx.x] = (p > 0 ? pre[D * M + threadIdx.x] : 0.f) +
                      (Z0 != nullptr ? Z0[(long)bh * D + threadIdx.x] : 0.f);

  for (long n0 = nb; n0 < ne; n0 += C) {
    load_tile<T, C, D, false, kPhi>(sQ, D + 1, q + hq, n0, ne);
    load_tile<T, C, D, false, kPhi>(sK, D + 1, k + hq, n0, ne);
    load_tile<T, C, M, false, kRaw>(sV, M + 1, v + hv, n0, ne);
    __syncthreads();
    {  // A = mask(phi(Q) phi(K)^T)
      float a[C / 16][C / 16];
      zero_acc(a);
      smem_mm<C / 16, C / 16, D>(a, sQ, D + 1, 1, sK, 1, D + 1);
#pragma unroll
      for (int r = 0; r < C / 16; ++r)
#pragma unroll
        for (int c = 0; c < C / 16; ++c) {
          const int i = ty + 16 * r, j = tx + 16 * c;
          sA[i * (C + 1) + j] = j <= i ? (DECAY ? a[r][c] * spw[i - j] : a[r][c]) : 0.f;
        }
    }
    __syncthreads();
    if (threadIdx.x < C) {
      const int i = threadIdx.x;
      float s = 0.f;
      for (int j = 0; j <= i; ++j) s += sA[i * (C + 1) + j];
      if (DECAY) {  // the carried state reaches row i with gamma^(i+1)
        float t = 0.f;
        for (int d = 0; d < D; ++d) t += sQ[i * (D + 1) + d] * sz[d];
        s += spw[i + 1] * t;
      } else {
        for (int d = 0; d < D; ++d) s += sQ[i * (D + 1) + d] * sz[d];
      }
      sden[i] = s;
      if (den != nullptr && n0 + i < ne) den[(long)bh * N + n0 + i] = s;
    }
    __syncthreads();
    {  // out = (A V + phi(Q) S) / den
      float o[C / 16][M / 16];
      zero_acc(o);
      smem_mm<C / 16, M / 16, C>(o, sA, C + 1, 1, sV, M + 1, 1);
      if (DECAY) {
        float o2[C / 16][M / 16];
        zero_acc(o2);
        smem_mm<C / 16, M / 16, D>(o2, sQ, D + 1, 1, sS, M + 1, 1);
#pragma unroll
        for (int r = 0; r < C / 16; ++r)
#pragma unroll
          for (int c = 0; c < M / 16; ++c) o[r][c] += spw[ty + 16 * r + 1] * o2[r][c];
      } else {
        smem_mm<C / 16, M / 16, D>(o, sQ, D + 1, 1, sS, M + 1, 1);
      }
#pragma unroll
      for (int r = 0; r < C / 16; ++r) {
        const int i = ty + 16 * r;
        if (n0 + i < ne) {
          const float inv = 1.f / sden[i];
#pragma unroll
          for (int c = 0; c < M / 16; ++c)
            out[hv + (n0 + i) * M + tx + 16 * c] = from_f<T>(o[r][c] * inv);
        }
      }
    }
    __syncthreads();
    // S += phi(K)^T V, z += sum phi(K); with DECAY S <- gamma^L S + sum_j
    // gamma^(L-1-j) phi(K_j) V_j^T (L = the chunk's valid rows)
    const int L = (int)min((long)C, ne - n0);
    (void)L;
    if (DECAY) {
      scale_rows<D>(sK, lg, L - 1, -1, L);
      const float dl = spw[L];
#pragma unroll
      for (int r = 0; r < D / 16; ++r)
#pragma unroll
        for (int c = 0; c < M / 16; ++c) accS[r][c] *= dl;
      if (threadIdx.x < D) sz[threadIdx.x] *= dl;
      __syncthreads();
    }
    smem_mm<D / 16, M / 16, C>(accS, sK, 1, D + 1, sV, M + 1, 1);
#pragma unroll
    for (int r = 0; r < D / 16; ++r)
#pragma unroll
      for (int c = 0; c < M / 16; ++c) sS[(ty + 16 * r) * (M + 1) + tx + 16 * c] = accS[r][c];
    if (threadIdx.x < D) {
      float s = sz[threadIdx.x];
      for (int j = 0; j < C; ++j) s += sK[j * (D + 1) + threadIdx.x];
      sz[threadIdx.x] = s;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- backward

// Causal backward, grid (segment, b*h, role).
// role 0 walks the segment forward carrying S, z (eq. 13 plus the
// denominator term):
//   dA       = mask(gt V^T + gam 1^T)
//   grad_phiQ = dA phi(K) + gt S^T + gam z^T,  dq = grad_phiQ * phi'(Q)
// role 1 walks it backward carrying R, r (eq. 14-15 plus the denominator):
//   A = mask(phi(Q) phi(K)^T),  dA as above
//   grad_phiK = dA^T phi(Q) + V R^T + r,        dk = grad_phiK * phi'(K)
//   dv        = A^T gt + phi(K) R
//   R += phi(Q)^T gt,  r += phi(Q)^T gam
template <int D, int M, typename T, bool DECAY>
__global__ void __launch_bounds__(NT) k_causal_bwd(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const T* __restrict__ o, const float* __restrict__ den, const T* __restrict__ g,
    T* __restrict__ dq, T* __restrict__ dk, T* __restrict__ dv, const float* __restrict__ ws,
    int N, int nseg, int seg_len, float lg) {
  const int p = blockIdx.x, bh = blockIdx.y, role = blockIdx.z;
  extern __shared__ float sm[];
  float* sQ = sm;                  // phi(Q) [C][D+1]
  float* sK = sQ + C * (D + 1);    // phi(K) [C][D+1]
  float* sV = sK + C * (D + 1);    // V      [C][M+1]
  float* sG = sV + C * (M + 1);    // gt     [C][M+1]
  float* sO = sG + C * (M + 1);    // O      [C][M+1]
  float* sA = sO + C * (M + 1);    // A      [C][C+1]
  float* sdA = sA + C * (C + 1);   // dA     [C][C+1]
  float* sS = sdA + C * (C + 1);   // S or R [D][M+1]
  float* sz = sS + D * (M + 1);    // z or r [D]
  float* sden = sz + D;            // [C]
  float* sgam = sden + C;          // [C]
  float* spw = sgam + C;           // gamma^0 .. gamma^C (with DECAY)
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const long nb = (long)p * seg_len, ne = min((long)N, nb + seg_len);
  const long hq = (long)bh * N * D, hv = (long)bh * N * M;
  if (DECAY && threadIdx.x <= C) spw[threadIdx.x] = decay_pow(lg, threadIdx.x);
  const float* rec = ws + ((long)bh * nseg + p) * 2 * (D * M + D);
  // role 0: exclusive prefix (S, z) of the segment; role 1: exclusive suffix (R, r)
  const float* st = rec + (role == 0 ? 0 : D * M + D);
  const bool has = role == 0 ? p > 0 : p < nseg - 1;
  float acc[D / 16][M / 16];
#pragma unroll
  for (int r = 0; r < D / 16; ++r)
#pragma unroll
    for (int c = 0; c < M / 16; ++c) {
      const int d = ty + 16 * r, m = tx + 16 * c;
      acc[r][c] = has ? st[d * M + m] : 0.f;
      sS[d * (M + 1) + m] = acc[r][c];
    }
  if (threadIdx.x < D) sz[threadIdx.x] = has ? st[D * M + threadIdx.x] : 0.f;

  const int nchunks = (int)((ne - nb + C - 1) / C);
  for (int ci = 0; ci < nchunks; ++ci) {
    const long n0 = role == 0 ? nb + (long)ci * C : nb + (long)(nchunks - 1 - ci) * C;
    const int L = (int)min((long)C, ne - n0);  // valid rows of the chunk
    if (role == 1) load_tile<T, C, D, false, kPhi>(sQ, D + 1, q + hq, n0, ne);
    load_tile<T, C, D, false, kPhi>(sK, D + 1, k + hq, n0, ne);
    load_tile<T, C, M, false, kRaw>(sV, M + 1, v + hv, n0, ne);
    load_grad_terms<T, M>(sG, sO, sden, sgam, g + hv, o + hv, den + (long)bh * N, n0, ne);
    __syncthreads();
    {  // dA = mask(gt V^T + gam); role 1 also A = mask(phi(Q) phi(K)^T)
      float a[C / 16][C / 16];
      zero_acc(a);
      smem_mm<C / 16, C / 16, M>(a, sG, M + 1, 1, sV, 1, M + 1);
#pragma unroll
      for (int r = 0; r < C / 16; ++r)
#pragma unroll
        for (int c = 0; c < C / 16; ++c) {
          const int i = ty + 16 * r, j = tx + 16 * c;
          sdA[i * (C + 1) + j] = j <= i ? (DECAY ? (a[r][c] + sgam[i]) * spw[i - j] : a[r][c] + sgam[i]) : 0.f;
        }
      if (role == 1) {
        zero_acc(a);
        smem_mm<C / 16, C / 16, D>(a, sQ, D + 1, 1, sK, 1, D + 1);
#pragma unroll
        for (int r = 0; r < C / 16; ++r)
#pragma unroll
          for (int c = 0; c < C / 16; ++c) {
            const int i = ty + 16 * r, j = tx + 16 * c;
            sA[i * (C + 1) + j] = j <= i ? (DECAY ? a[r][c] * spw[i - j] : a[r][c]) : 0.f;
          }
      }
    }
    __syncthreads();
    if (role == 0) {
      float t[C / 16][D / 16], t2[C / 16][D / 16];
      zero_acc(t);
      smem_mm<C / 16, D / 16, C>(t, sdA, C + 1, 1, sK, D + 1, 1);   // dA phi(K)
      if (DECAY) {  // the carried state reaches query row i with gamma^(i+1)
        zero_acc(t2);
        smem_mm<C / 16, D / 16, M>(t2, sG, M + 1, 1, sS, 1, M + 1);  // gt S^T
      } else {
        smem_mm<C / 16, D / 16, M>(t, sG, M + 1, 1, sS, 1, M + 1);   // gt S^T
      }
#pragma unroll
      for (int r = 0; r < C / 16; ++r) {
        const int i = ty + 16 * r;
        if (n0 + i < ne) {
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            const int d = tx + 16 * c;
            const long idx = hq + (n0 + i) * D + d;
            const float gq = DECAY ? t[r][c] + spw[i + 1] * (t2[r][c] + sgam[i] * sz[d])
                                   : t[r][c] + sgam[i] * sz[d];
            dq[idx] = from_f<T>(gq * dphi(to_f(q[idx])));
          }
        }
      }
    } else {
      float t[C / 16][D / 16], t2[C / 16][D / 16];
      zero_acc(t);
      smem_mm<C / 16, D / 16, C>(t, sdA, 1, C + 1, sQ, D + 1, 1);   // dA^T phi(Q)
      if (DECAY) {  // the carried state (the sums after the chunk) reaches key row j with gamma^(L-j)
        zero_acc(t2);
        smem_mm<C / 16, D / 16, M>(t2, sV, M + 1, 1, sS, 1, M + 1);  // V R^T
      } else {
        smem_mm<C / 16, D / 16, M>(t, sV, M + 1, 1, sS, 1, M + 1);   // V R^T
      }
#pragma unroll
      for (int r = 0; r < C / 16; ++r) {
        const int j = ty + 16 * r;
        if (n0 + j < ne) {
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            const int d = tx + 16 * c;
            const long idx = hq + (n0 + j) * D + d;
            const float gk = DECAY ? t[r][c] + spw[L - j] * (t2[r][c] + sz[d]) : t[r][c] + sz[d];
            dk[idx] = from_f<T>(gk * dphi(to_f(k[idx])));
          }
        }
      }
      float u[C / 16][M / 16], u2[C / 16][M / 16];
      zero_acc(u);
      smem_mm<C / 16, M / 16, C>(u, sA, 1, C + 1, sG, M + 1, 1);    // A^T gt
      if (DECAY) {
        zero_acc(u2);
        smem_mm<C / 16, M / 16, D>(u2, sK, D + 1, 1, sS, M + 1, 1);  // phi(K) R
      } else {
        smem_mm<C / 16, M / 16, D>(u, sK, D + 1, 1, sS, M + 1, 1);   // phi(K) R
      }
#pragma unroll
      for (int r = 0; r < C / 16; ++r) {
        const int j = ty + 16 * r;
        if (n0 + j < ne) {
#pragma unroll
          for (int c = 0; c < M / 16; ++c)
            dv[hv + (n0 + j) * M + tx + 16 * c] =
                from_f<T>(DECAY ? u[r][c] + spw[L - j] * u2[r][c] : u[r][c]);
        }
      }
    }
    __syncthreads();
    if (DECAY) {  // the chunk's rows relative to where the carried state continues, and its decay
      if (role == 0)
        scale_rows<D>(sK, lg, L - 1, -1, L);  // gamma^(L-1-j)
      else
        scale_rows<D>(sQ, lg, 0, 1, L);       // gamma^i
      const float dl = spw[L];
#pragma unroll
      for (int r = 0; r < D / 16; ++r)
#pragma unroll
        for (int c = 0; c < M / 16; ++c) acc[r][c] *= dl;
      if (threadIdx.x < D) sz[threadIdx.x] *= dl;
      __syncthreads();
    }
    if (role == 0) {  // S += phi(K)^T V, z += sum phi(K)
      smem_mm<D / 16, M / 16, C>(acc, sK, 1, D + 1, sV, M + 1, 1);
      if (threadIdx.x < D) {
        float s = sz[threadIdx.x];
        for (int j = 0; j < C; ++j) s += sK[j * (D + 1) + threadIdx.x];
        sz[threadIdx.x] = s;
      }
    } else {          // R += phi(Q)^T gt, r += phi(Q)^T gam
      smem_mm<D / 16, M / 16, C>(acc, sQ, 1, D + 1, sG, M + 1, 1);
      if (threadIdx.x < D) {
        float s = sz[threadIdx.x];
        for (int i = 0; i < C; ++i) s += sgam[i] * sQ[i * (D + 1) + threadIdx.x];
        sz[threadIdx.x] = s;
      }
    }
#pragma unroll
    for (int r = 0; r < D / 16; ++r)
#pragma unroll
      for (int c = 0; c < M / 16; ++c) sS[(ty + 16 * r) * (M + 1) + tx + 16 * c] = acc[r][c];
    __syncthreads();
  }
}

template <int D, int M>
constexpr size_t fwd_smem() {
  return sizeof(float) * (2 * C * (D + 1) + C * (M + 1) + C * (C + 1) + D * (M + 1) + D + C + C + 1);
}
template <int D, int M>
constexpr size_t bwd_smem() {
  return sizeof(float) *
         (2 * C * (D + 1) + 3 * C * (M + 1) + 2 * C * (C + 1) + D * (M + 1) + D + 2 * C + C + 1);
}
template <int D, int M>
constexpr size_t state_fwd_smem() {
  return sizeof(float) * (C * (D + 1) + C * (M + 1));
}
template <int D, int M>
constexpr size_t state_bwd_smem() {
  return sizeof(float) * (2 * C * (D + 1) + 3 * C * (M + 1) + 2 * C);
}

// Segments of the main kernels, planned in whole waves: CTAs of the given
// dynamic shared memory fit two to an SM below half of it (else one; the
// registers of 256 threads allow no more), `roles` CTAs run per segment, and
// the plan minimises waves x (chunks per segment + 1) -- the longest chain of
// CTAs an SM runs, each CTA's fixed cost (its prefix state, the first loads)
// taken as about one chunk -- preferring fewer segments on a tie.  (Rounding
// the segment count up to fill one wave can leave a few CTAs for a second
// wave, which costs a whole segment's time.)
SegPlan cc_plan(int BH, int N, int roles, size_t smem) {
  const long occ = smem + 1024 <= 232448 / 2 ? 2 : 1;
  const long slots = occ * (sm_count() < 1 ? 1 : sm_count());
  const int nch = (N + C - 1) / C;
  SegPlan best{1, nch * C};
  long best_cost = -1;
  for (int want = 1; want <= nch; ++want) {
    const int per = (nch + want - 1) / want;  // chunks per segment
    const int nseg = (nch + per - 1) / per;
    if (nseg != want) continue;  // the shortest segments for this count only
    const long waves = (static_cast<long>(nseg) * BH * roles + slots - 1) / slots;
    const long cost = waves * (per + 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = SegPlan{nseg, per * C};
    }
  }
  return best;
}

// The dynamic shared memory of the main kernels, as the launches give it.
size_t fwd_smem_rt(int D, int M) {
  return sizeof(float) * (2 * C * (D + 1) + C * (M + 1) + C * (C + 1) + D * (M + 1) + D + C + C + 1);
}
size_t bwd_smem_rt(int D, int M) {
  return sizeof(float) *
         (2 * C * (D + 1) + 3 * C * (M + 1) + 2 * C * (C + 1) + D * (M + 1) + D + 2 * C + C + 1);
}
static_assert(fwd_smem<64, 64>() == sizeof(float) * 20993 && bwd_smem<64, 64>() == sizeof(float) * 33537,
              "the run-time sizes follow the templates");
SegPlan fwd_plan(int BH, int N, int D, int M) { return cc_plan(BH, N, 1, fwd_smem_rt(D, M)); }
SegPlan bwd_plan_cc(int BH, int N, int D, int M) { return cc_plan(BH, N, 2, bwd_smem_rt(D, M)); }

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// lg = log2(gamma) of the RetNet decay (0: undecayed).
template <int D, int M, typename T, bool DECAY>
cudaError_t run_fwd(const T* q, const T* k, const T* v, T* out, float* den, float* ws,
                    const Shape& s, cudaStream_t st, float lg) {
  const int BH = s.B * s.H;
  const SegPlan pl = fwd_plan(BH, s.N, D, M);
  cudaError_t e;
  if (pl.nseg > 1) {
    auto ks = k_seg_state_fwd<D, M, T, DECAY>;
    if ((e = set_smem(ks, state_fwd_smem<D, M>())) != cudaSuccess) return e;
    ks<<<dim3(pl.nseg, BH), NT, state_fwd_smem<D, M>(), st>>>(k, v, ws, s.N, pl.nseg, pl.seg_len,
                                                              pl.nseg, 0, lg);
    k_seg_scan<<<dim3(BH, (D * M + D + 255) / 256), 256, 0, st>>>(
        ws, pl.nseg, D * M + D, D * M + D, 0, 0, pl.nseg, DECAY ? lg : 0.f, pl.seg_len, s.N);
  }
  auto kf = k_causal_fwd<D, M, T, DECAY>;
  if ((e = set_smem(kf, fwd_smem<D, M>())) != cudaSuccess) return e;
  kf<<<dim3(pl.nseg, BH), NT, fwd_smem<D, M>(), st>>>(q, k, v, out, den, ws, s.N, pl.nseg,
                                                      pl.seg_len, pl.nseg, nullptr, nullptr, lg);
  return cudaGetLastError();
}

// The forward from the state (S, Z), which then receives the state after the
// sequence: every segment's sums (nseg + 1 records per (b, h), the last one
// the totals), the forward with S, Z added to each prefix, then S, Z += the
// totals (after the forward has read them).
template <int D, int M, typename T>
cudaError_t run_prefill(const T* q, const T* k, const T* v, T* out, float* den, float* S, float* Z,
                        float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const SegPlan pl = fwd_plan(BH, s.N, D, M);
  const int nrec = pl.nseg + 1;
  cudaError_t e;
  auto ks = k_seg_state_fwd<D, M, T, false>;
  if ((e = set_smem(ks, state_fwd_smem<D, M>())) != cudaSuccess) return e;
  ks<<<dim3(pl.nseg, BH), NT, state_fwd_smem<D, M>(), st>>>(k, v, ws, s.N, pl.nseg, pl.seg_len,
                                                            nrec, 1, 0.f);
  k_seg_scan<<<dim3(BH, (D * M + D + 255) / 256), 256, 0, st>>>(ws, pl.nseg, D * M + D, D * M + D,
                                                                0, 0, nrec, 0.f, pl.seg_len, s.N);
  auto kf = k_causal_fwd<D, M, T, false>;
  if ((e = set_smem(kf, fwd_smem<D, M>())) != cudaSuccess) return e;
  kf<<<dim3(pl.nseg, BH), NT, fwd_smem<D, M>(), st>>>(q, k, v, out, den, ws, s.N, pl.nseg,
                                                      pl.seg_len, nrec, S, Z, 0.f);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return state_add_records(ws, BH, nrec, D * M + D, pl.nseg, nrec, D, M, M, D * M, 1, S, Z, st);
}

template <int D, int M, typename T, bool DECAY>
cudaError_t run_bwd(const T* q, const T* k, const T* v, const T* o, const float* den, const T* g,
                    T* dq, T* dk, T* dv, float* ws, const Shape& s, cudaStream_t st, float lg) {
  const int BH = s.B * s.H;
  const SegPlan pl = bwd_plan_cc(BH, s.N, D, M);
  cudaError_t e;
  if (pl.nseg > 1) {
    auto ks = k_seg_state_bwd<D, M, T, DECAY>;
    if ((e = set_smem(ks, state_bwd_smem<D, M>())) != cudaSuccess) return e;
    ks<<<dim3(pl.nseg, BH), NT, state_bwd_smem<D, M>(), st>>>(q, k, v, o, den, g, ws, s.N,
                                                              pl.nseg, pl.seg_len, lg);
    k_seg_scan<<<dim3(BH, (D * M + D + 255) / 256), 256, 0, st>>>(
        ws, pl.nseg, 2 * (D * M + D), D * M + D, D * M + D, D * M + D, pl.nseg, DECAY ? lg : 0.f,
        pl.seg_len, s.N);
  }
  auto kb = k_causal_bwd<D, M, T, DECAY>;
  if ((e = set_smem(kb, bwd_smem<D, M>())) != cudaSuccess) return e;
  kb<<<dim3(pl.nseg, BH, 2), NT, bwd_smem<D, M>(), st>>>(q, k, v, o, den, g, dq, dk, dv, ws,
                                                         s.N, pl.nseg, pl.seg_len, lg);
  return cudaGetLastError();
}

}  // namespace

void k_seg_scan_ext(float* ws, int BH, int nseg, int stride, int wf, int ro, int wr,
                    cudaStream_t st) {
  const int w = wf > wr ? wf : wr;
  k_seg_scan<<<dim3(BH, (w + 255) / 256), 256, 0, st>>>(ws, nseg, stride, wf, ro, wr, nseg, 0.f, 1, 1);
}

namespace {

// (S, Z)[bh] += the sum of records r0 .. r1 - 1 of ws[bh] (nrec records of
// rstride floats per (b, h)); a record holds S[d][m] at d * srow + m and
// z[d] at zoff + d * zstride.
__global__ void k_state_add(const float* __restrict__ ws, int nrec, int rstride, int r0, int r1,
                            int D, int M, int srow, int zoff, int zstride, float* __restrict__ S,
                            float* __restrict__ Z) {
  const long bh = blockIdx.x;
  const float* base = ws + bh * nrec * static_cast<long>(rstride);
  const int e = blockIdx.y * blockDim.x + threadIdx.x;
  if (e >= D * M + D) return;
  const bool isz = e >= D * M;
  const int off = isz ? zoff + (e - D * M) * zstride : (e / M) * srow + e % M;
  float acc = 0.f;
  for (int r = r0; r < r1; ++r) acc += base[static_cast<long>(r) * rstride + off];
  if (isz)
    Z[bh * D + (e - D * M)] += acc;
  else
    S[bh * D * M + e] += acc;
}

}  // namespace

cudaError_t state_add_records(const float* ws, int BH, int nrec, int rstride, int r0, int r1, int D,
                              int M, int srow, int zoff, int zstride, float* S, float* Z,
                              cudaStream_t st) {
  k_state_add<<<dim3(BH, (D * M + D + 255) / 256), 256, 0, st>>>(ws, nrec, rstride, r0, r1, D, M,
                                                                 srow, zoff, zstride, S, Z);
  return cudaGetLastError();
}

size_t causal_prefill_ws_floats(const Shape& s) {
  const SegPlan pl = fwd_plan(s.B * s.H, s.N, s.D, s.M);
  return (size_t)s.B * s.H * (pl.nseg + 1) * (s.D * s.M + s.D);
}

cudaError_t causal_prefill_cc(const void* q, const void* k, const void* v, void* out, float* den,
                              float* S, float* Z, float* ws, const Shape& s, cudaStream_t st) {
  if (s.dtype == 0) {
    using T = float;
    LA_DISPATCH_DM(s.D, s.M, return (run_prefill<D_, M_, T>((const T*)q, (const T*)k, (const T*)v,
                                                             (T*)out, den, S, Z, ws, s, st)));
  } else {
    using T = __nv_bfloat16;
    LA_DISPATCH_DM(s.D, s.M, return (run_prefill<D_, M_, T>((const T*)q, (const T*)k, (const T*)v,
                                                             (T*)out, den, S, Z, ws, s, st)));
  }
  return cudaErrorInvalidValue;
}

size_t causal_fwd_ws_floats(const Shape& s) {
  const SegPlan pl = fwd_plan(s.B * s.H, s.N, s.D, s.M);
  return pl.nseg > 1 ? (size_t)s.B * s.H * pl.nseg * (s.D * s.M + s.D) : 0;
}

size_t causal_bwd_ws_floats(const Shape& s) {
  const SegPlan pl = bwd_plan_cc(s.B * s.H, s.N, s.D, s.M);
  return pl.nseg > 1 ? (size_t)s.B * s.H * pl.nseg * 2 * (s.D * s.M + s.D) : 0;
}

int causal_fwd_launches(const Shape& s) {
  return fwd_plan(s.B * s.H, s.N, s.D, s.M).nseg > 1 ? 3 : 1;
}

int causal_bwd_launches(const Shape& s) {
  return bwd_plan_cc(s.B * s.H, s.N, s.D, s.M).nseg > 1 ? 3 : 1;
}

cudaError_t causal_fwd_cc(const void* q, const void* k, const void* v, void* out, float* den,
                          float* ws, const Shape& s, cudaStream_t st, float gamma) {
  const bool dec = gamma != 1.f;
  const float lg = dec ? log2f(gamma) : 0.f;  // -inf for gamma = 0
  if (s.dtype == 0) {
    using T = float;
    if (dec) {
      LA_DISPATCH_DM(s.D, s.M, return (run_fwd<D_, M_, T, true>((const T*)q, (const T*)k, (const T*)v,
                                                                (T*)out, den, ws, s, st, lg)));
    } else {
      LA_DISPATCH_DM(s.D, s.M, return (run_fwd<D_, M_, T, false>((const T*)q, (const T*)k, (const T*)v,
                                                                 (T*)out, den, ws, s, st, 0.f)));
    }
  } else {
    using T = __nv_bfloat16;
    if (dec) {
      LA_DISPATCH_DM(s.D, s.M, return (run_fwd<D_, M_, T, true>((const T*)q, (const T*)k, (const T*)v,
                                                                (T*)out, den, ws, s, st, lg)));
    } else {
      LA_DISPATCH_DM(s.D, s.M, return (run_fwd<D_, M_, T, false>((const T*)q, (const T*)k, (const T*)v,
                                                                 (T*)out, den, ws, s, st, 0.f)));
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t causal_bwd_cc(const void* q, const void* k, const void* v, const void* out,
                          const float* den, const void* dout, void* dq, void* dk, void* dv,
                          float* ws, const Shape& s, cudaStream_t st, float gamma) {
  const bool dec = gamma != 1.f;
  const float lg = dec ? log2f(gamma) : 0.f;
#define LA_BWD_CALL(T, DEC, LG)                                                                    \
  LA_DISPATCH_DM(s.D, s.M,                                                                         \
                 return (run_bwd<D_, M_, T, DEC>((const T*)q, (const T*)k, (const T*)v,            \
                                                 (const T*)out, den, (const T*)dout, (T*)dq,       \
                                                 (T*)dk, (T*)dv, ws, s, st, LG)))
  if (s.dtype == 0) {
    if (dec) {
      LA_BWD_CALL(float, true, lg);
    } else {
      LA_BWD_CALL(float, false, 0.f);
    }
  } else {
    if (dec) {
      LA_BWD_CALL(__nv_bfloat16, true, lg);
    } else {
      LA_BWD_CALL(__nv_bfloat16, false, 0.f);
    }
  }
#undef LA_BWD_CALL
  return cudaErrorInvalidValue;
}

}  // namespace la
