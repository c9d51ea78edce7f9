// Non-causal path for D = M = 64 (fp32 or bf16 inputs, fp32 arithmetic on
// the CUDA cores).
//
// Method: "Linear Attention/zh", kernel reformulation (one shared S, Z per
// (b, h)) and eq. 13-15 of "Transformers are RNNs" (part 2/3) with full sums
// over the valid rows i < L:
//   S = sum_j phi(K_j) V_j^T,  Z = sum_j phi(K_j),
//   out_i = phi(Q_i)^T S / phi(Q_i)^T Z,
//   gt_i = dout_i / den_i,  gam_i = -(gt_i . out_i),
//   R = sum_i phi(Q_i) gt_i^T,  r = sum_i gam_i phi(Q_i),
//   dq_i = (S gt_i + gam_i Z) * phi'(Q_i),
//   dk_j = (R V_j + r) * phi'(K_j),  dv_j = R^T phi(K_j).
// Rows i >= L are padding: they enter no sum and are written as zero.
//
// Two launches per direction.  A state kernel gives every segment of whole
// 128-token chunks two partial records ([64 x 64 | 64], one per half of the
// CTA's tokens); the per-token kernel of the same (b, h) sums the records
// while staging them (no reduction launch) and runs the per-token products.
// The backward state kernel also stores gam, so the per-token backward never
// reads out.
//
// Every product is a 64-deep contraction out of shared memory in which each
// thread accumulates an 8 x 4 block (32 FMAs per three 16-byte shared loads):
//  - state sums: [64 x 64] += A^T B over a half-chunk of 64 tokens, A and B
//    staged row-major ([token][64 + 4]);
//  - per-token products: [128 tokens x 64] = A B with the token operand
//    stored transposed ([64][128 + 4], written with conflict-free stores) and
//    the 64 x 64 operand row-major ([64][64 + 4]).
// Chunks past the valid length are written as zeros without arithmetic.
#include "common.cuh"
#include "launch.h"

namespace la {
namespace {

constexpr int C64 = 128;          // tokens per chunk
constexpr int LDT = C64 + 4;      // leading dimension of a transposed token tile
constexpr int LDB = 64 + 4;       // leading dimension of a row-major 64-wide tile
constexpr int RS = 64 * 64 + 64;  // floats per partial record [64 x 64 | 64]
constexpr int NT64 = 256;

__device__ __forceinline__ long vlen(const int* lengths, int b, int N) {
  if (lengths == nullptr) return N;
  const int L = lengths[b];
  return L < 0 ? 0 : (L > N ? N : L);
}

enum LoadOp { kLoadRaw = 0, kLoadPhi = 1, kLoadScale = 2 };

template <int OP>
__device__ __forceinline__ float load_op(float x, float s) {
  return OP == kLoadPhi ? phi(x) : (OP == kLoadScale ? x * s : x);
}

// Token rows n0 .. n0+127 of a [*][64] tensor, transposed into At[64][LDT]:
// At[c][i] = op(x[n0 + i][c]); rows at or past nv are zero.  A warp step
// takes RB rows x VB 16-byte vectors, chosen so that the transposing stores
// of one warp hit 32 different banks (LDT = 4 mod 32): 16 rows x 2 vectors
// for fp32, 32 rows x 1 vector for bf16.
template <typename T, int OP>
__device__ __forceinline__ void load_t(float* At, const T* x, long n0, long nv, const float* rs) {
  constexpr int VN = Vec16<T>::n;      // elements per 16-byte vector
  constexpr int VB = VN == 4 ? 2 : 1;  // vectors per warp step
  constexpr int RB = 32 / VB;          // rows per warp step
  constexpr int NBR = C64 / RB, NB = NBR * (64 / VN / VB);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int b = w; b < NB; b += NT64 / 32) {
    const int row = RB * (b % NBR) + l % RB, cv = VB * (b / NBR) + l / RB;
    float f[VN];
    if (n0 + row < nv) {
      const uint4 u = *reinterpret_cast<const uint4*>(x + (n0 + row) * 64 + cv * VN);
      Vec16<T>::unpack(u, f);
      const float s = OP == kLoadScale ? rs[row] : 1.f;
#pragma unroll
      for (int i = 0; i < VN; ++i) f[i] = load_op<OP>(f[i], s);
    } else {
#pragma unroll
      for (int i = 0; i < VN; ++i) f[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < VN; ++i) At[(cv * VN + i) * LDT + row] = f[i];
  }
}

// Token rows n0 .. n0+127 of a [*][64] tensor, row-major into A[128][LDB]
// with op applied; rows at or past ne are zero.
template <typename T, int OP>
__device__ __forceinline__ void load_r(float* A, const T* x, long n0, long ne) {
  constexpr int VN = Vec16<T>::n, VPR = 64 / VN;
#pragma unroll
  for (int e = threadIdx.x; e < C64 * VPR; e += NT64) {
    const int row = e / VPR, cv = e % VPR;
    float f[VN];
    if (n0 + row < ne) {
      const uint4 u = *reinterpret_cast<const uint4*>(x + (n0 + row) * 64 + cv * VN);
      Vec16<T>::unpack(u, f);
#pragma unroll
      for (int i = 0; i < VN; ++i) f[i] = load_op<OP>(f[i], 1.f);
    } else {
#pragma unroll
      for (int i = 0; i < VN; ++i) f[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < VN; i += 4)
      *reinterpret_cast<float4*>(A + row * LDB + cv * VN + i) =
          make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
  }
}

// acc[r][c] += sum_{k<64} A[k * lda + r] * B[k * ldb + c]  (r < 8, c < 4);
// A and B already offset to the thread's block.
__device__ __forceinline__ void gemm_8x4(float (&acc)[8][4], const float* A, int lda,
                                         const float* B, int ldb) {
#pragma unroll 4
  for (int k = 0; k < 64; ++k) {
    const float4 a0 = *reinterpret_cast<const float4*>(A + k * lda);
    const float4 a1 = *reinterpret_cast<const float4*>(A + k * lda + 4);
    const float4 bb = *reinterpret_cast<const float4*>(B + k * ldb);
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float b[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// Four values to global memory (16 bytes of fp32 or 8 of bf16).
template <typename T>
__device__ __forceinline__ void store4(T* dst, const float* v);
template <>
__device__ __forceinline__ void store4<float>(float* dst, const float* v) {
  *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<const uint32_t*>(&a),
                                              *reinterpret_cast<const uint32_t*>(&b));
}

// Four consecutive elements of row-major global data as floats.
template <typename T>
__device__ __forceinline__ void load4(const T* src, float* v);
template <>
__device__ __forceinline__ void load4<float>(const float* src, float* v) {
  const float4 x = *reinterpret_cast<const float4*>(src);
  v[0] = x.x;
  v[1] = x.y;
  v[2] = x.z;
  v[3] = x.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* src, float* v) {
  const uint2 x = *reinterpret_cast<const uint2*>(src);
  v[0] = __uint_as_float(x.x << 16);
  v[1] = __uint_as_float(x.x & 0xffff0000u);
  v[2] = __uint_as_float(x.y << 16);
  v[3] = __uint_as_float(x.y & 0xffff0000u);
}

// Rows [r0, r1) of a [*][64] tensor set to zero by the CTA.
template <typename T>
__device__ __forceinline__ void zero_rows(T* x, long r0, long r1) {
  const float z[4] = {0.f, 0.f, 0.f, 0.f};
  for (long e = r0 * 16 + threadIdx.x; e < r1 * 16; e += NT64) store4<T>(x + e * 4, z);
}

// The CTA's partial sums to its two records: acc of half h (threads
// 128h .. 128h+127) to record h, and the column sum whose four quarters
// (threads 64q .. 64q+63 over rows 32q .. 32q+31) are in colsum; quarters
// 2h and 2h+1 go to record h.  sx: 128 floats of scratch.
__device__ __forceinline__ void put_records(float* rec2, const float (&acc)[8][4], float colsum,
                                            float* sx) {
  const int t = threadIdx.x, h = t >> 7, u = t & 127, tx = u & 15, ty = u >> 4;
  float* rec = rec2 + h * RS;
#pragma unroll
  for (int r = 0; r < 8; ++r)
    *reinterpret_cast<float4*>(rec + (8 * ty + r) * 64 + 4 * tx) =
        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  const int d = t & 63, q = t >> 6;
  if (q & 1) sx[(q >> 1) * 64 + d] = colsum;
  __syncthreads();
  if (!(q & 1)) rec2[(q >> 1) * RS + 64 * 64 + d] = colsum + sx[(q >> 1) * 64 + d];
}

// ------------------------------------------------------------ state sums
// Partial S, Z of one segment: rec[bh][2p + h] holds the sums over the
// half-chunks h of phi(K_j) V_j^T and phi(K_j).
template <typename T>
__global__ void __launch_bounds__(NT64, 2)
    k64_state(const T* __restrict__ k, const T* __restrict__ v, const int* __restrict__ lengths,
              float* __restrict__ rec, int N, int H, int seg_len, int nrec) {
  extern __shared__ __align__(16) float sm64[];
  float* sK = sm64;            // phi(K) [128][LDB]
  float* sV = sK + C64 * LDB;  // V      [128][LDB]
  float* sx = sV + C64 * LDB;  // [128]
  const int p = blockIdx.x, bh = blockIdx.y, t = threadIdx.x;
  const int h = t >> 7, u = t & 127, tx = u & 15, ty = u >> 4, zd = t & 63, zq = t >> 6;
  const long L = vlen(lengths, bh / H, N);
  const long nb = static_cast<long>(p) * seg_len, ne = min(L, nb + seg_len);
  const long hq = static_cast<long>(bh) * N * 64;
  float acc[8][4] = {};
  float zacc = 0.f;
  for (long n0 = nb; n0 < ne; n0 += C64) {
    load_r<T, kLoadPhi>(sK, k + hq, n0, ne);
    load_r<T, kLoadRaw>(sV, v + hq, n0, ne);
    __syncthreads();
    gemm_8x4(acc, sK + 64 * h * LDB + 8 * ty, LDB, sV + 64 * h * LDB + 4 * tx, LDB);
#pragma unroll 8
    for (int j = 32 * zq; j < 32 * zq + 32; ++j) zacc += sK[j * LDB + zd];
    __syncthreads();
  }
  put_records(rec + (static_cast<long>(bh) * nrec + 2 * p) * RS, acc, zacc, sx);
}

// Partial R, r of one segment, plus gam_i for its valid rows:
// rec[bh][2p + h] holds the sums over the half-chunks h of phi(Q_i) gt_i^T
// and gam_i phi(Q_i).
template <typename T>
__global__ void __launch_bounds__(NT64, 2)
    k64_state_bwd(const T* __restrict__ q, const T* __restrict__ o, const float* __restrict__ den,
                  const T* __restrict__ g, const int* __restrict__ lengths,
                  float* __restrict__ rec, float* __restrict__ gam, int N, int H, int seg_len,
                  int nrec) {
  extern __shared__ __align__(16) float sm64[];
  float* sQ = sm64;            // phi(Q) [128][LDB]
  float* sG = sQ + C64 * LDB;  // gt     [128][LDB]
  float* sx = sG + C64 * LDB;  // [128]
  float* sinv = sx + C64;      // 1 / den [128]
  float* sgam = sinv + C64;    // gam [128]
  constexpr int VN = Vec16<T>::n, VPR = 64 / VN;
  const int p = blockIdx.x, bh = blockIdx.y, t = threadIdx.x;
  const int h = t >> 7, u = t & 127, tx = u & 15, ty = u >> 4, zd = t & 63, zq = t >> 6;
  const long L = vlen(lengths, bh / H, N);
  const long nb = static_cast<long>(p) * seg_len, ne = min(L, nb + seg_len);
  const long hq = static_cast<long>(bh) * N * 64, hn = static_cast<long>(bh) * N;
  float acc[8][4] = {};
  float racc = 0.f;
  for (long n0 = nb; n0 < ne; n0 += C64) {
    if (t < C64) sinv[t] = n0 + t < ne ? 1.f / den[hn + n0 + t] : 0.f;
    load_r<T, kLoadPhi>(sQ, q + hq, n0, ne);
    __syncthreads();
    // gt = dout / den into sG; gam = -(gt . out), reduced over the VPR
    // consecutive lanes of one warp that hold a row.
#pragma unroll
    for (int e = t; e < C64 * VPR; e += NT64) {
      const int row = e / VPR, cv = e % VPR;
      float f[VN], y[VN];
      float part = 0.f;
      if (n0 + row < ne) {
        const long off = hq + (n0 + row) * 64 + cv * VN;
        Vec16<T>::unpack(*reinterpret_cast<const uint4*>(g + off), f);
        Vec16<T>::unpack(*reinterpret_cast<const uint4*>(o + off), y);
        const float s = sinv[row];
#pragma unroll
        for (int i = 0; i < VN; ++i) {
          f[i] *= s;
          part = fmaf(f[i], y[i], part);
        }
      } else {
#pragma unroll
        for (int i = 0; i < VN; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < VN; i += 4)
        *reinterpret_cast<float4*>(sG + row * LDB + cv * VN + i) =
            make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
#pragma unroll
      for (int off = VPR / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      if (cv == 0) {
        sgam[row] = -part;
        if (n0 + row < ne) gam[hn + n0 + row] = -part;
      }
    }
    __syncthreads();
    gemm_8x4(acc, sQ + 64 * h * LDB + 8 * ty, LDB, sG + 64 * h * LDB + 4 * tx, LDB);
#pragma unroll 8
    for (int j = 32 * zq; j < 32 * zq + 32; ++j) racc = fmaf(sgam[j], sQ[j * LDB + zd], racc);
    __syncthreads();
  }
  put_records(rec + (static_cast<long>(bh) * nrec + 2 * p) * RS, acc, racc, sx);
}

// Sum of the nrec records of one (b, h): the 64 x 64 part into X (row-major
// [64][LDB]) and, when Xt is given, transposed into Xt; the vector part into
// x.  When Xg is given the sums are also stored to Xg [64 * 64] and xg [64].
__device__ __forceinline__ void sum_records(const float* rec, int nrec, float* X, float* Xt,
                                            float* x, float* Xg, float* xg) {
  for (int e = threadIdx.x; e < RS / 4; e += NT64) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < nrec; ++i)
      s = add4(s, *reinterpret_cast<const float4*>(rec + static_cast<long>(i) * RS + 4 * e));
    if (e < 1024) {
      const int r = e >> 4, c = 4 * (e & 15);
      *reinterpret_cast<float4*>(X + r * LDB + c) = s;
      if (Xt != nullptr) {
        Xt[c * LDB + r] = s.x;
        Xt[(c + 1) * LDB + r] = s.y;
        Xt[(c + 2) * LDB + r] = s.z;
        Xt[(c + 3) * LDB + r] = s.w;
      }
      if (Xg != nullptr) *reinterpret_cast<float4*>(Xg + 4 * e) = s;
    } else {
      *reinterpret_cast<float4*>(x + 4 * (e - 1024)) = s;
      if (xg != nullptr) *reinterpret_cast<float4*>(xg + 4 * (e - 1024)) = s;
    }
  }
}

// ---------------------------------------------------------------- forward
// out and den of one segment; the first segment of each (b, h) also stores
// the summed S and Z.
template <typename T>
__global__ void __launch_bounds__(NT64, 2)
    k64_out(const T* __restrict__ q, const float* __restrict__ rec, const int* __restrict__ lengths,
            T* __restrict__ out, float* __restrict__ den, float* __restrict__ S,
            float* __restrict__ Z, int N, int H, int seg_len, int nrec) {
  extern __shared__ __align__(16) float sm64[];
  float* sS = sm64;            // [64][LDB]
  float* sQt = sS + 64 * LDB;  // phi(Q)^T [64][LDT]
  float* sz = sQt + 64 * LDT;  // [64]
  float* sden = sz + 64;       // [128]
  const int p = blockIdx.x, bh = blockIdx.y;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const long L = vlen(lengths, bh / H, N);
  const long nb = static_cast<long>(p) * seg_len, ne = min(static_cast<long>(N), nb + seg_len);
  const long nv = min(ne, L);
  const long hq = static_cast<long>(bh) * N * 64;
  T* outh = out + hq;
  float* denh = den == nullptr ? nullptr : den + static_cast<long>(bh) * N;
  if (nv < ne) {  // padding: zero rows (and den) without arithmetic
    zero_rows<T>(outh, max(nb, nv), ne);
    if (denh != nullptr)
      for (long i = max(nb, nv) + threadIdx.x; i < ne; i += NT64) denh[i] = 0.f;
  }
  const bool first = p == 0;
  if (nb >= nv && !first) return;
  sum_records(rec + static_cast<long>(bh) * nrec * RS, nrec, sS, nullptr, sz,
              first ? S + static_cast<long>(bh) * 4096 : nullptr,
              first ? Z + static_cast<long>(bh) * 64 : nullptr);
  for (long n0 = nb; n0 < nv; n0 += C64) {
    __syncthreads();  // the state sums, or the previous chunk's readers
    load_t<T, kLoadPhi>(sQt, q + hq, n0, nv, nullptr);
    __syncthreads();
    if (threadIdx.x < C64) {  // den_i = phi(Q_i) . Z
      const int i = threadIdx.x;
      float s = 0.f;
#pragma unroll 8
      for (int d = 0; d < 64; ++d) s = fmaf(sQt[d * LDT + i], sz[d], s);
      sden[i] = s;
      if (denh != nullptr && n0 + i < nv) denh[n0 + i] = s;
    }
    float acc[8][4] = {};
    gemm_8x4(acc, sQt + 8 * ty, LDT, sS + 4 * tx, LDB);
    __syncthreads();  // sden
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = 8 * ty + r;
      if (n0 + i < nv) {
        const float inv = 1.f / sden[i];
        float y[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) y[c] = acc[r][c] * inv;
        store4<T>(outh + (n0 + i) * 64 + 4 * tx, y);
      }
    }
  }
}

// --------------------------------------------------------------- backward
// dq, dk, dv of one segment from S, Z, the summed R, r records and gam.
template <typename T>
__global__ void __launch_bounds__(NT64, 2)
    k64_bwd(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
            const float* __restrict__ den, const float* __restrict__ gam, const T* __restrict__ g,
            const float* __restrict__ S, const float* __restrict__ Z,
            const float* __restrict__ rec, const int* __restrict__ lengths, T* __restrict__ dq,
            T* __restrict__ dk, T* __restrict__ dv, int N, int H, int seg_len, int nrec) {
  extern __shared__ __align__(16) float sm64[];
  float* sSt = sm64;            // S^T [64 m][LDB]
  float* sRt = sSt + 64 * LDB;  // R^T [64 m][LDB]
  float* sR = sRt + 64 * LDB;   // R   [64 d][LDB]
  float* sAt = sR + 64 * LDB;   // token operand, transposed [64][LDT]
  float* sz = sAt + 64 * LDT;   // Z [64]
  float* sr = sz + 64;          // r [64]
  float* sinv = sr + 64;        // 1 / den [128]
  float* sgam = sinv + C64;     // gam [128]
  const int p = blockIdx.x, bh = blockIdx.y, t = threadIdx.x;
  const int tx = t & 15, ty = t >> 4;
  const long L = vlen(lengths, bh / H, N);
  const long nb = static_cast<long>(p) * seg_len, ne = min(static_cast<long>(N), nb + seg_len);
  const long nv = min(ne, L);
  const long hq = static_cast<long>(bh) * N * 64, hn = static_cast<long>(bh) * N;
  if (nv < ne) {
    zero_rows<T>(dq + hq, max(nb, nv), ne);
    zero_rows<T>(dk + hq, max(nb, nv), ne);
    zero_rows<T>(dv + hq, max(nb, nv), ne);
  }
  if (nb >= nv) return;
  sum_records(rec + static_cast<long>(bh) * nrec * RS, nrec, sR, sRt, sr, nullptr, nullptr);
  for (int e = t; e < 4096; e += NT64)
    sSt[(e & 63) * LDB + (e >> 6)] = S[static_cast<long>(bh) * 4096 + e];
  if (t < 64) sz[t] = Z[static_cast<long>(bh) * 64 + t];
  for (long n0 = nb; n0 < nv; n0 += C64) {
    __syncthreads();  // the state, or the previous chunk's readers
    if (t < C64) {
      const long i = n0 + t;
      sinv[t] = i < nv ? 1.f / den[hn + i] : 0.f;
      sgam[t] = i < nv ? gam[hn + i] : 0.f;
    }
    __syncthreads();
    // dq = (gt S^T + gam Z) * phi'(Q), gt = dout / den
    load_t<T, kLoadScale>(sAt, g + hq, n0, nv, sinv);
    __syncthreads();
    {
      float acc[8][4] = {};
      gemm_8x4(acc, sAt + 8 * ty, LDT, sSt + 4 * tx, LDB);
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int i = 8 * ty + rr;
        if (n0 + i < nv) {
          float x[4], y[4];
          load4<T>(q + hq + (n0 + i) * 64 + 4 * tx, x);
#pragma unroll
          for (int c = 0; c < 4; ++c) y[c] = (acc[rr][c] + sgam[i] * sz[4 * tx + c]) * dphi(x[c]);
          store4<T>(dq + hq + (n0 + i) * 64 + 4 * tx, y);
        }
      }
    }
    __syncthreads();
    // dk = (V R^T + r) * phi'(K)
    load_t<T, kLoadRaw>(sAt, v + hq, n0, nv, nullptr);
    __syncthreads();
    {
      float acc[8][4] = {};
      gemm_8x4(acc, sAt + 8 * ty, LDT, sRt + 4 * tx, LDB);
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int j = 8 * ty + rr;
        if (n0 + j < nv) {
          float x[4], y[4];
          load4<T>(k + hq + (n0 + j) * 64 + 4 * tx, x);
#pragma unroll
          for (int c = 0; c < 4; ++c) y[c] = (acc[rr][c] + sr[4 * tx + c]) * dphi(x[c]);
          store4<T>(dk + hq + (n0 + j) * 64 + 4 * tx, y);
        }
      }
    }
    __syncthreads();
    // dv = phi(K) R
    load_t<T, kLoadPhi>(sAt, k + hq, n0, nv, nullptr);
    __syncthreads();
    {
      float acc[8][4] = {};
      gemm_8x4(acc, sAt + 8 * ty, LDT, sR + 4 * tx, LDB);
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int j = 8 * ty + rr;
        if (n0 + j < nv) store4<T>(dv + hq + (n0 + j) * 64 + 4 * tx, acc[rr]);
      }
    }
  }
}

constexpr size_t kStateSmem = sizeof(float) * (2 * C64 * LDB + 3 * C64);
constexpr size_t kOutSmem = sizeof(float) * (64 * LDB + 64 * LDT + 64 + C64);
constexpr size_t kBwdSmem = sizeof(float) * (3 * 64 * LDB + 64 * LDT + 2 * 64 + 2 * C64);

template <typename K>
cudaError_t smem_attr(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

template <typename T>
cudaError_t run_fwd64(const T* q, const T* k, const T* v, const int* lengths, T* out, float* den,
                      float* S, float* Z, float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const SegPlan pl = noncausal64_plan(BH, s.N);
  const int nrec = 2 * pl.nseg;
  cudaError_t e;
  if ((e = smem_attr(k64_state<T>, kStateSmem)) != cudaSuccess) return e;
  if ((e = smem_attr(k64_out<T>, kOutSmem)) != cudaSuccess) return e;
  k64_state<T><<<dim3(pl.nseg, BH), NT64, kStateSmem, st>>>(k, v, lengths, ws, s.N, s.H,
                                                             pl.seg_len, nrec);
  k64_out<T><<<dim3(pl.nseg, BH), NT64, kOutSmem, st>>>(q, ws, lengths, out, den, S, Z, s.N, s.H,
                                                         pl.seg_len, nrec);
  return cudaGetLastError();
}

template <typename T>
cudaError_t run_bwd64(const T* q, const T* k, const T* v, const int* lengths, const T* o,
                      const float* den, const float* S, const float* Z, const T* g, T* dq, T* dk,
                      T* dv, float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const SegPlan pl = noncausal64_plan(BH, s.N);
  const int nrec = 2 * pl.nseg;
  float* gam = ws + static_cast<size_t>(BH) * nrec * RS;
  cudaError_t e;
  if ((e = smem_attr(k64_state_bwd<T>, kStateSmem)) != cudaSuccess) return e;
  if ((e = smem_attr(k64_bwd<T>, kBwdSmem)) != cudaSuccess) return e;
  k64_state_bwd<T><<<dim3(pl.nseg, BH), NT64, kStateSmem, st>>>(q, o, den, g, lengths, ws, gam,
                                                                 s.N, s.H, pl.seg_len, nrec);
  k64_bwd<T><<<dim3(pl.nseg, BH), NT64, kBwdSmem, st>>>(q, k, v, den, gam, g, S, Z, ws, lengths,
                                                         dq, dk, dv, s.N, s.H, pl.seg_len, nrec);
  return cudaGetLastError();
}

}  // namespace

SegPlan noncausal64_plan(int BH, int N) { return plan_segments(BH, N, C64, kTargetCtas); }

size_t noncausal64_fwd_ws_floats(const Shape& s) {
  const SegPlan pl = noncausal64_plan(s.B * s.H, s.N);
  return static_cast<size_t>(s.B) * s.H * 2 * pl.nseg * RS;
}

size_t noncausal64_bwd_ws_floats(const Shape& s) {
  return noncausal64_fwd_ws_floats(s) + static_cast<size_t>(s.B) * s.H * s.N;
}

cudaError_t noncausal64_fwd(const void* q, const void* k, const void* v, const int* lengths,
                            void* out, float* den, float* S, float* Z, float* ws, const Shape& s,
                            cudaStream_t st) {
  if (s.dtype == 0)
    return run_fwd64<float>(static_cast<const float*>(q), static_cast<const float*>(k),
                            static_cast<const float*>(v), lengths, static_cast<float*>(out), den,
                            S, Z, ws, s, st);
  using B16 = __nv_bfloat16;
  return run_fwd64<B16>(static_cast<const B16*>(q), static_cast<const B16*>(k),
                        static_cast<const B16*>(v), lengths, static_cast<B16*>(out), den, S, Z,
                        ws, s, st);
}

cudaError_t noncausal64_bwd(const void* q, const void* k, const void* v, const int* lengths,
                            const void* out, const float* den, const float* S, const float* Z,
                            const void* dout, void* dq, void* dk, void* dv, float* ws,
                            const Shape& s, cudaStream_t st) {
  if (s.dtype == 0)
    return run_bwd64<float>(static_cast<const float*>(q), static_cast<const float*>(k),
                            static_cast<const float*>(v), lengths, static_cast<const float*>(out),
                            den, S, Z, static_cast<const float*>(dout), static_cast<float*>(dq),
                            static_cast<float*>(dk), static_cast<float*>(dv), ws, s, st);
  using B16 = __nv_bfloat16;
  return run_bwd64<B16>(static_cast<const B16*>(q), static_cast<const B16*>(k),
                        static_cast<const B16*>(v), lengths, static_cast<const B16*>(out), den, S,
                        Z, static_cast<const B16*>(dout), static_cast<B16*>(dq),
                        static_cast<B16*>(dk), static_cast<B16*>(dv), ws, s, st);
}

}  // namespace la
