// Causal linear attention with the degree-2 polynomial kernel, "Transformers
// are RNNs" (part 2/3), the feature-map discussion before eq. 7 (§3.2.1): the
// polynomial kernel has an exact finite feature map, and at degree 2 the
// method costs O(N D^2 M).  Read as sim(q, k) = (q . k)^2 in eq. 8-12, whose
// exact feature map is, for a <= b,
//   f(x)_(a,a) = x_a^2,   f(x)_(a,b) = sqrt(2) x_a x_b   (a < b),
// D (D + 1) / 2 features (55 at D = 10), so f(q) . f(k) = (q . k)^2.
//
// GB300 design: the features are formed once into 64-wide bf16 rows (zero
// past the last pair), and the causal tensor-core kernels run on them with no
// feature map of their own (feat = true), the same skeleton as elu(x) + 1.
// The backward's feature gradients come back through the chain rule:
//   dx_a = 2 x_a df_(a,a) + sqrt(2) sum_{b != a} x_b df_(min(a,b), max(a,b)).
// Both extra kernels stream rows once, 32 rows a block staged in shared
// memory; the features are an intermediate in the caller's workspace.
#include "common.cuh"
#include "launch.h"

namespace la {
namespace {

using bf16 = __nv_bfloat16;
constexpr int FW = 64;  // feature row width
constexpr float SQRT2 = 1.41421356237309505f;  // sqrt(2)

// Feature c of a row of width D: the pair (a, b), a <= b, in the order
// (0,0), (0,1), ..., (0,D-1), (1,1), ...; returns false past the last pair.
__device__ __forceinline__ bool pair_of(int c, int D, int& a, int& b) {
  int base = 0;
  for (a = 0; a < D; ++a) {
    if (c < base + (D - a)) {
      b = a + (c - base);
      return true;
    }
    base += D - a;
  }
  return false;
}

constexpr int RPB = 32;          // rows per block
constexpr int NTB = RPB * FW / 8;  // 256 threads: one 16-byte chunk of 8 features each

// The pair table of width D in shared memory: feature c <-> (a, b) and its
// coefficient (1 for a = b, sqrt 2 otherwise; 0 past the last pair).
struct PairTab {
  unsigned char a[FW], b[FW];
  float coef[FW];
};

__device__ __forceinline__ void build_pairs(PairTab& t, int D) {
  for (int c = threadIdx.x; c < FW; c += blockDim.x) {
    int a = 0, b = 0;
    const bool live = pair_of(c, D, a, b);
    t.a[c] = static_cast<unsigned char>(live ? a : 0);
    t.b[c] = static_cast<unsigned char>(live ? b : 0);
    t.coef[c] = live ? (a == b ? 1.f : SQRT2) : 0.f;
  }
}

// A block of 32 rows: their inputs staged in shared memory (coalesced), then
// thread t forms features 8 (t mod 8) .. +7 of row t / 8 and stores them as
// one 16-byte chunk (the rows' 128-byte feature rows by consecutive threads).
// q and k in one launch: blockIdx.y picks the tensor.
template <typename T>
__global__ void __launch_bounds__(NTB) k_poly_features(const T* __restrict__ x0, bf16* __restrict__ f0,
                                                       const T* __restrict__ x1, bf16* __restrict__ f1,
                                                       long rows, int D) {
  const T* __restrict__ x = blockIdx.y == 0 ? x0 : x1;
  bf16* __restrict__ f = blockIdx.y == 0 ? f0 : f1;
  __shared__ PairTab tab;
  __shared__ float xs[RPB][POLY_MAX_D];
  const long r0 = static_cast<long>(blockIdx.x) * RPB;
  const int nr = static_cast<int>(min(static_cast<long>(RPB), rows - r0));
  build_pairs(tab, D);
  for (int e = threadIdx.x; e < nr * D; e += NTB) xs[e / D][e % D] = to_f(x[r0 * D + e]);
  __syncthreads();
  const int rr = threadIdx.x / 8, j = threadIdx.x % 8;
  if (rr >= nr) return;
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const int c0 = 8 * j + e, c1 = c0 + 1;
    const float f0 = tab.coef[c0] * xs[rr][tab.a[c0]] * xs[rr][tab.b[c0]];
    const float f1 = tab.coef[c1] * xs[rr][tab.a[c1]] * xs[rr][tab.b[c1]];
    const __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
    w[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(f + (r0 + rr) * FW + 8 * j) = make_uint4(w[0], w[1], w[2], w[3]);
}

// A block of 32 rows: their feature gradients (one 16-byte chunk a thread)
// and inputs staged in shared memory, then output t < 32 D (threads striding)
// is dx_a of row t / D, a = t mod D, over the D features that involve a:
//   dx_a = 2 x_a df_(a,a) + sqrt(2) sum_{b != a} x_b df_(min(a,b), max(a,b)).
// q and k in one launch: blockIdx.y picks the tensor.
template <typename T>
__global__ void __launch_bounds__(NTB) k_poly_grad(const T* __restrict__ x0, const bf16* __restrict__ df0,
                                                   T* __restrict__ dx0, const T* __restrict__ x1,
                                                   const bf16* __restrict__ df1, T* __restrict__ dx1,
                                                   long rows, int D) {
  const T* __restrict__ x = blockIdx.y == 0 ? x0 : x1;
  const bf16* __restrict__ df = blockIdx.y == 0 ? df0 : df1;
  T* __restrict__ dx = blockIdx.y == 0 ? dx0 : dx1;
  __shared__ float xs[RPB][POLY_MAX_D];
  __shared__ __align__(16) bf16 gs[RPB][FW];
  __shared__ unsigned char first[POLY_MAX_D];  // the index of feature (a, a)
  const long r0 = static_cast<long>(blockIdx.x) * RPB;
  const int nr = static_cast<int>(min(static_cast<long>(RPB), rows - r0));
  if (threadIdx.x < D) {
    const int a = threadIdx.x;
    first[a] = static_cast<unsigned char>(a * D - a * (a - 1) / 2);
  }
  for (int e = threadIdx.x; e < nr * D; e += NTB) xs[e / D][e % D] = to_f(x[r0 * D + e]);
  {
    const int rr = threadIdx.x / 8, j = threadIdx.x % 8;
    if (rr < nr)
      *reinterpret_cast<uint4*>(&gs[rr][8 * j]) =
          *reinterpret_cast<const uint4*>(df + (r0 + rr) * FW + 8 * j);
  }
  __syncthreads();
  for (int t = threadIdx.x; t < nr * D; t += NTB) {  // 32 D outputs: more than the threads for D > 8
    const int rr = t / D, a = t % D;
    float acc = 2.f * xs[rr][a] * __bfloat162float(gs[rr][first[a]]);
    for (int b = 0; b < D; ++b) {
      if (b == a) continue;
      const int lo = min(a, b), hi = max(a, b);
      acc += SQRT2 * xs[rr][b] * __bfloat162float(gs[rr][first[lo] + (hi - lo)]);
    }
    dx[(r0 + rr) * D + a] = from_f<T>(acc);
  }
}

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

Shape feature_shape(const Shape& s) { return Shape{s.B, s.H, s.N, FW, s.M, s.dtype}; }

size_t feat_bytes(const Shape& s) {
  return align256(static_cast<size_t>(s.B) * s.H * s.N * FW * sizeof(bf16));
}

cudaError_t features(const void* q, bf16* fq, const void* k, bf16* fk, const Shape& s, cudaStream_t st) {
  const long rows = static_cast<long>(s.B) * s.H * s.N;
  k_poly_features<bf16><<<dim3(static_cast<unsigned>((rows + RPB - 1) / RPB), 2), NTB, 0, st>>>(
      static_cast<const bf16*>(q), fq, static_cast<const bf16*>(k), fk, rows, s.D);
  return cudaGetLastError();
}

cudaError_t grad(const void* q, const bf16* dfq, void* dq, const void* k, const bf16* dfk, void* dk,
                 const Shape& s, cudaStream_t st) {
  const long rows = static_cast<long>(s.B) * s.H * s.N;
  k_poly_grad<bf16><<<dim3(static_cast<unsigned>((rows + RPB - 1) / RPB), 2), NTB, 0, st>>>(
      static_cast<const bf16*>(q), dfq, static_cast<bf16*>(dq), static_cast<const bf16*>(k), dfk,
      static_cast<bf16*>(dk), rows, s.D);
  return cudaGetLastError();
}

}  // namespace

size_t causal_poly_ws_bytes(const Shape& s, bool bwd) {
  const Shape f = feature_shape(s);
  const size_t tc = bwd ? causal_bwd_tc_ws_floats(f) : causal_fwd_tc_ws_floats(f);
  return (bwd ? 4 : 2) * feat_bytes(s) + align256(tc * 4);
}

int causal_poly_launches(const Shape& s, bool bwd) {
  const Shape f = feature_shape(s);
  return bwd ? 1 + causal_bwd_tc_launches(f) + 1 : 1 + causal_fwd_tc_launches(f);
}

cudaError_t causal_fwd_poly(const void* q, const void* k, const void* v, void* out, float* den,
                            void* ws, const Shape& s, cudaStream_t st) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  bf16* fq = reinterpret_cast<bf16*>(w);
  bf16* fk = reinterpret_cast<bf16*>(w + feat_bytes(s));
  float* tcws = reinterpret_cast<float*>(w + 2 * feat_bytes(s));
  cudaError_t e;
  if ((e = features(q, fq, k, fk, s, st)) != cudaSuccess) return e;
  return causal_fwd_tc(fq, fk, v, out, den, tcws, feature_shape(s), st, true);
}

cudaError_t causal_bwd_poly(const void* q, const void* k, const void* v, const void* out,
                            const float* den, const void* dout, void* dq, void* dk, void* dv,
                            void* ws, const Shape& s, cudaStream_t st) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t fb = feat_bytes(s);
  bf16* fq = reinterpret_cast<bf16*>(w);
  bf16* fk = reinterpret_cast<bf16*>(w + fb);
  bf16* dfq = reinterpret_cast<bf16*>(w + 2 * fb);
  bf16* dfk = reinterpret_cast<bf16*>(w + 3 * fb);
  float* tcws = reinterpret_cast<float*>(w + 4 * fb);
  cudaError_t e;
  if ((e = features(q, fq, k, fk, s, st)) != cudaSuccess) return e;
  if ((e = causal_bwd_tc(fq, fk, v, out, den, dout, dfq, dfk, dv, tcws, feature_shape(s), st, true)) !=
      cudaSuccess)
    return e;
  return grad(q, dfq, dq, k, dfk, dk, s, st);
}

}  // namespace la
