// Non-causal path for fp32 inputs with D = M = 64: one kernel per direction,
// one thread-block cluster per (b, h).
//
// Method: "Linear Attention/zh", kernel reformulation (one shared S, Z per
// (b, h)) and eq. 13-15 of "Transformers are RNNs" (part 2/3) with full sums
// over the valid rows i < L:
//   S = sum_j phi(K_j) V_j^T,  Z = sum_j phi(K_j),
//   out_i = phi(Q_i)^T S / den_i,  den_i = phi(Q_i)^T Z,
//   gt_i = dout_i / den_i,  gam_i = -(gt_i . out_i),
//   R = sum_i phi(Q_i) gt_i^T,  r = sum_i gam_i phi(Q_i),
//   dq_i = (S gt_i + gam_i Z) * phi'(Q_i),
//   dk_j = (R V_j + r) * phi'(K_j),  dv_j = R^T phi(K_j).
// Rows i >= L are padding: they enter no sum and are written as zero.
//
// Layout of the work.  The nseg CTAs of a cluster share one (b, h); the
// valid rows are cut into 64-token chunks and every CTA takes an equal run
// of them.  Each kernel has two phases:
//  forward   1: partial S, Z over the CTA's rows;  cluster-wide sum through
//               distributed shared memory;  2: out, den of the CTA's rows
//               (the first CTA also stores S, Z);
//  backward  1: gt, gam, dq (S and Z are inputs) and partial R, r;  cluster
//               sum;  2: dk, dv.
// So the inputs are read once per phase that needs them, nothing goes
// through a workspace, and there is one launch per direction.
//
// Staging.  Chunks of q, k, v, dout are copied with cp.async (16 bytes per
// thread, rows past the end zero-filled) into padded tiles [64][68] in a
// two- or three-stage ring, so the copy of chunk c+1 runs under the
// arithmetic of chunk c.  phi, 1 / den and the zeroing of invalid rows are
// applied in place once a chunk has landed.
//
// Arithmetic.  fp32 FMAs; each of the 128 threads keeps an 8 x 4 block of
// the output in registers (32 FMAs per three 16-byte shared loads):
//  - state form  [64 d x 64 m] += A^T B over the chunk's tokens: thread
//    (tx, ty) owns d = 8 ty .. 8 ty + 7, m = 4 tx .. 4 tx + 3;
//  - token form  [64 tokens x 64] = A B: thread (tx, ty) owns tokens
//    ty + 8 r (r < 8) and columns 4 tx .. 4 tx + 3, so the two token rows a
//    warp reads at a time sit 68 floats apart (different banks).
#include "common.cuh"
#include "launch.h"

namespace la {
namespace {

constexpr int CC = 64;               // tokens per chunk
constexpr int LDA = 68;              // padded row of a staged tile (floats)
constexpr int TILE = CC * LDA;       // floats per tile
constexpr int NTC = 128;             // threads per CTA
constexpr int PREC = 64 * 64 + 64;   // floats of a partial-state record
constexpr int kMaxSeg = 8;           // CTAs per cluster (portable limit)

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared; zero-fills when !valid.
__device__ __forceinline__ void cp16(float* dst, const float* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Cluster-wide barrier: every thread's earlier shared-memory writes are
// visible to every thread of the cluster after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float4 phi4(float4 x) {
  return make_float4(phi(x.x), phi(x.y), phi(x.z), phi(x.w));
}
__device__ __forceinline__ float get(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// The CTA's rows of one (b, h): valid rows [r0, r1) in chunks of CC, and
// padded rows [z0, z1) to be zeroed.
struct Rows {
  long r0, r1, z0, z1;
  int nch;
};

__device__ __forceinline__ Rows my_rows(const int* lengths, int b, int N, int p, int nseg) {
  long L = N;
  if (lengths != nullptr) {
    const int l = lengths[b];
    L = l < 0 ? 0 : (l > N ? N : l);
  }
  const long nchv = (L + CC - 1) / CC;
  const long per = (nchv + nseg - 1) / nseg;
  const long c0 = min(nchv, p * per), c1 = min(nchv, c0 + per);
  Rows w;
  w.r0 = c0 * CC;
  w.r1 = min(c1 * CC, L);
  w.nch = static_cast<int>(c1 - c0);
  const long zs = (N - L + nseg - 1) / nseg;
  w.z0 = min(static_cast<long>(N), L + p * zs);
  w.z1 = min(static_cast<long>(N), w.z0 + zs);
  return w;
}

// Rows [n0, n0 + CC) of x ([*][64], fp32) into tile [CC][LDA]; rows at or
// past ne are zero-filled.  Warp-contiguous 16-byte pieces (two rows per
// warp instruction).
__device__ __forceinline__ void issue_tile(float* tile, const float* x, long n0, long ne) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = threadIdx.x + NTC * i, row = e >> 4, cv = e & 15;
    const bool ok = n0 + row < ne;
    cp16(tile + row * LDA + 4 * cv, x + (ok ? n0 + row : n0) * 64 + 4 * cv, ok);
  }
}

// Element i of a thread's share of a tile (i < 8): row (t >> 4) + 8 i,
// columns 4 (t & 15) .. +3; the 16 lanes holding a row are consecutive.
__device__ __forceinline__ int part_row(int i) { return (threadIdx.x >> 4) + 8 * i; }
__device__ __forceinline__ int part_col() { return 4 * (threadIdx.x & 15); }

// phi in place on the valid rows of a tile; rows at or past nv become 0.
__device__ __forceinline__ void phi_tile(float* tile, int nv) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = part_row(i);
    float* p = tile + row * LDA + part_col();
    st4(p, row < nv ? phi4(ld4(p)) : make_float4(0.f, 0.f, 0.f, 0.f));
  }
}

__device__ __forceinline__ float sum16(float x) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// State form: acc[r][c] += sum_{j<CC} A[j * LDA + r] * B[j * LDA + c], with
// A, B already offset to the thread's d and m.
__device__ __forceinline__ void gemm_state(float (&acc)[8][4], const float* A, const float* B) {
#pragma unroll 4
  for (int j = 0; j < CC; ++j) {
    const float4 a0 = ld4(A + j * LDA), a1 = ld4(A + j * LDA + 4), b = ld4(B + j * LDA);
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      acc[r][0] = fmaf(a[r], b.x, acc[r][0]);
      acc[r][1] = fmaf(a[r], b.y, acc[r][1]);
      acc[r][2] = fmaf(a[r], b.z, acc[r][2]);
      acc[r][3] = fmaf(a[r], b.w, acc[r][3]);
    }
  }
}

// Token form: acc[r][c] += sum_{k<64} A[8 r * LDA + k] * B[k * LDA + c],
// with A offset to the thread's first token row and B to its columns.
__device__ __forceinline__ void gemm_tok(float (&acc)[8][4], const float* A, const float* B) {
#pragma unroll 2
  for (int k = 0; k < 64; k += 4) {
    float4 a[8], b[4];
#pragma unroll
    for (int r = 0; r < 8; ++r) a[r] = ld4(A + 8 * r * LDA + k);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) b[kk] = ld4(B + (k + kk) * LDA);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float x = get(a[r], kk);
        acc[r][0] = fmaf(x, b[kk].x, acc[r][0]);
        acc[r][1] = fmaf(x, b[kk].y, acc[r][1]);
        acc[r][2] = fmaf(x, b[kk].z, acc[r][2]);
        acc[r][3] = fmaf(x, b[kk].w, acc[r][3]);
      }
  }
}

template <int R, int C>
__device__ __forceinline__ void zero(float (&a)[R][C]) {
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int c = 0; c < C; ++c) a[r][c] = 0.f;
}

// The CTA's partial state to its record P ([64 x 64] row-major | [64]):
// acc from the state form, colsum[t] the sum over rows 32 (t >> 6) .. + 31
// of column t & 63 (the two halves meet in sx).
__device__ __forceinline__ void put_partial(float* P, const float (&acc)[8][4], float colsum,
                                            float* sx) {
  const int t = threadIdx.x, tx = t & 15, ty = t >> 4;
#pragma unroll
  for (int r = 0; r < 8; ++r)
    st4(P + (8 * ty + r) * 64 + 4 * tx, make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]));
  if (t >= 64) sx[t - 64] = colsum;
  __syncthreads();
  if (t < 64) P[64 * 64 + t] = colsum + sx[t];
}

// Sum of the records P of all nseg CTAs of the cluster: thread t gets the
// float4 pieces t + 128 i (i < 8) of the matrix part in m[i] and, for
// t < 16, piece t of the vector part in vec.
__device__ __forceinline__ void cluster_sum(const float* P, int nseg, float4 (&m)[8], float4& vec) {
  const uint32_t base = saddr(P);
  const int t = threadIdx.x;
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  vec = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q = 0; q < nseg; ++q) {
    const uint32_t a = map_rank(base, static_cast<uint32_t>(q));
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = add4(m[i], ld_cluster4(a + 16u * (t + NTC * i)));
    if (t < 16) vec = add4(vec, ld_cluster4(a + 16u * (1024 + t)));
  }
}

// The thread's share of out (8 float4) and den (8 floats) for the chunk at
// n0 (rows at or past ne read as 0 and 1).
__device__ __forceinline__ void fetch_od(float4 (&on)[8], float (&dn)[8], const float* oh,
                                         const float* dh, long n0, long ne) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const long row = n0 + part_row(i);
    const bool ok = row < ne;
    on[i] = ok ? ld4(oh + row * 64 + part_col()) : make_float4(0.f, 0.f, 0.f, 0.f);
    dn[i] = ok ? dh[row] : 1.f;
  }
}

// Piece e (< 1024) of a [64 x 64] row-major matrix: row e >> 4, columns
// 4 (e & 15) .. +3.
__device__ __forceinline__ int piece_row(int e) { return e >> 4; }
__device__ __forceinline__ int piece_col(int e) { return 4 * (e & 15); }

// ---------------------------------------------------------------- forward
constexpr int kFwdFloats = 4 * TILE + PREC + 3 * 64;

__global__ void __launch_bounds__(NTC, 2)
    k_nc_fwd_cluster(const float* __restrict__ q, const float* __restrict__ k,
                     const float* __restrict__ v, const int* __restrict__ lengths,
                     float* __restrict__ out, float* __restrict__ den, float* __restrict__ S,
                     float* __restrict__ Z, int N, int H, int nseg) {
  extern __shared__ __align__(16) float smc[];
  float* U = smc;                  // phase 1: (K, V) x 2 stages; phase 2: Q x 3 stages, S
  float* P = U + 4 * TILE;         // this CTA's partial S | Z
  float* sz = P + PREC;            // Z [64]
  float* sden = sz + 64;           // den of the chunk's rows [64]
  float* sx = sden + 64;           // [64]
  const int t = threadIdx.x, tx = t & 15, ty = t >> 4;
  const int p = static_cast<int>(cluster_rank());
  const int bh = blockIdx.x / nseg;
  const Rows w = my_rows(lengths, bh / H, N, p, nseg);
  const long hq = static_cast<long>(bh) * N * 64, hn = static_cast<long>(bh) * N;

  // padded rows
  for (long e = w.z0 * 16 + t; e < w.z1 * 16; e += NTC) st4(out + hq + 4 * e, make_float4(0.f, 0.f, 0.f, 0.f));
  if (den != nullptr)
    for (long i = w.z0 + t; i < w.z1; i += NTC) den[hn + i] = 0.f;

  // phase 1: partial S, Z
  float acc[8][4];
  zero(acc);
  float zc = 0.f;
  if (w.nch > 0) {
    issue_tile(U, k + hq, w.r0, w.r1);
    issue_tile(U + TILE, v + hq, w.r0, w.r1);
  }
  cp_commit();
  for (int c = 0; c < w.nch; ++c) {
    float* sK = U + 2 * (c & 1) * TILE;
    float* sV = sK + TILE;
    cp_wait<0>();
    __syncthreads();  // chunk c landed; chunk c - 1 fully consumed
    if (c + 1 < w.nch) {
      const long n1 = w.r0 + (c + 1) * CC;
      float* nK = U + 2 * ((c + 1) & 1) * TILE;
      issue_tile(nK, k + hq, n1, w.r1);
      issue_tile(nK + TILE, v + hq, n1, w.r1);
    }
    cp_commit();
    phi_tile(sK, static_cast<int>(min(static_cast<long>(CC), w.r1 - w.r0 - c * CC)));
    __syncthreads();
    gemm_state(acc, sK + 8 * ty, sV + 4 * tx);
    const int d = t & 63, h = t >> 6;
#pragma unroll 8
    for (int j = 32 * h; j < 32 * h + 32; ++j) zc += sK[j * LDA + d];
  }
  put_partial(P, acc, zc, sx);

  cluster_sync_all();  // every partial is complete; phase 1 tiles are free

  // phase 2 prologue: the first two Q chunks, under the cluster sum
  float* sS = U + 3 * TILE;
  for (int s = 0; s < 2; ++s) {
    if (s < w.nch) issue_tile(U + s * TILE, q + hq, w.r0 + s * CC, w.r1);
    cp_commit();
  }
  {
    float4 m[8], zv;
    cluster_sum(P, nseg, m, zv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = t + NTC * i;
      st4(sS + piece_row(e) * LDA + piece_col(e), m[i]);
      if (p == 0) st4(S + static_cast<long>(bh) * 4096 + 4 * e, m[i]);
    }
    if (t < 16) {
      st4(sz + 4 * t, zv);
      if (p == 0) st4(Z + static_cast<long>(bh) * 64 + 4 * t, zv);
    }
  }
  cluster_sync_all();  // no CTA reads another's P after this; S, Z visible in the CTA

  // phase 2: out = phi(Q) S / den
  for (int c = 0; c < w.nch; ++c) {
    float* sQ = U + (c % 3) * TILE;
    cp_wait<1>();
    __syncthreads();  // chunk c landed; chunk c - 1 fully consumed
    if (c + 2 < w.nch) issue_tile(U + ((c + 2) % 3) * TILE, q + hq, w.r0 + (c + 2) * CC, w.r1);
    cp_commit();
    const long n0 = w.r0 + c * CC;
    const int nv = static_cast<int>(min(static_cast<long>(CC), w.r1 - n0));
    {  // phi(Q) in place and den = phi(Q) . Z
      const float4 zq = ld4(sz + part_col());
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = part_row(i);
        float* ptr = sQ + row * LDA + part_col();
        const float4 f = row < nv ? phi4(ld4(ptr)) : make_float4(0.f, 0.f, 0.f, 0.f);
        st4(ptr, f);
        const float dn = sum16(f.x * zq.x + f.y * zq.y + f.z * zq.z + f.w * zq.w);
        if ((t & 15) == 0) {
          sden[row] = dn;
          if (den != nullptr && row < nv) den[hn + n0 + row] = dn;
        }
      }
    }
    __syncthreads();
    float o[8][4];
    zero(o);
    gemm_tok(o, sQ + ty * LDA, sS + 4 * tx);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int row = ty + 8 * r;
      if (row < nv) {
        const float inv = 1.f / sden[row];
        st4(out + hq + (n0 + row) * 64 + 4 * tx,
            make_float4(o[r][0] * inv, o[r][1] * inv, o[r][2] * inv, o[r][3] * inv));
      }
    }
  }
  cp_wait<0>();
}

// --------------------------------------------------------------- backward
constexpr int kBwdFloats = 6 * TILE + 4 * 64;

__global__ void __launch_bounds__(NTC, 2)
    k_nc_bwd_cluster(const float* __restrict__ q, const float* __restrict__ k,
                     const float* __restrict__ v, const int* __restrict__ lengths,
                     const float* __restrict__ o, const float* __restrict__ den,
                     const float* __restrict__ S, const float* __restrict__ Z,
                     const float* __restrict__ g, float* __restrict__ dq, float* __restrict__ dk,
                     float* __restrict__ dv, int N, int H, int nseg) {
  extern __shared__ __align__(16) float smc[];
  float* U = smc;                  // phase 1: (Q, G) x 2 stages; phase 2: (V, K) x 2 stages
  float* W = U + 4 * TILE;         // phase 1: S^T, P;  phase 2: R^T, R
  float* sz = W + 2 * TILE;        // phase 1: Z;  phase 2: r
  float* sgam = sz + 64;           // gam of the chunk's rows
  float* sx = sgam + 64;
  const int t = threadIdx.x, tx = t & 15, ty = t >> 4;
  const int p = static_cast<int>(cluster_rank());
  const int bh = blockIdx.x / nseg;
  const Rows w = my_rows(lengths, bh / H, N, p, nseg);
  const long hq = static_cast<long>(bh) * N * 64, hn = static_cast<long>(bh) * N;

  for (long e = w.z0 * 16 + t; e < w.z1 * 16; e += NTC) {
    st4(dq + hq + 4 * e, make_float4(0.f, 0.f, 0.f, 0.f));
    st4(dk + hq + 4 * e, make_float4(0.f, 0.f, 0.f, 0.f));
    st4(dv + hq + 4 * e, make_float4(0.f, 0.f, 0.f, 0.f));
  }

  // phase 1: gt, gam, dq and partial R, r
  float* sSt = W;
  float* P = W + TILE;
  if (w.nch > 0) {
    issue_tile(U, q + hq, w.r0, w.r1);
    issue_tile(U + TILE, g + hq, w.r0, w.r1);
  }
  cp_commit();
  for (int e = t; e < 4096; e += NTC)  // S^T: sSt[m][d] = S[d][m]
    sSt[(e & 63) * LDA + (e >> 6)] = S[static_cast<long>(bh) * 4096 + e];
  if (t < 64) sz[t] = Z[static_cast<long>(bh) * 64 + t];
  // out and den of the next chunk, prefetched into registers
  float4 onx[8];
  float dnx[8];
  if (w.nch > 0) fetch_od(onx, dnx, o + hq, den + hn, w.r0, w.r1);
  float accR[8][4];
  zero(accR);
  float rc = 0.f;
  for (int c = 0; c < w.nch; ++c) {
    float* sQ = U + 2 * (c & 1) * TILE;
    float* sG = sQ + TILE;
    cp_wait<0>();
    __syncthreads();  // chunk c landed; chunk c - 1 fully consumed
    if (c + 1 < w.nch) {
      const long n1 = w.r0 + (c + 1) * CC;
      float* nQ = U + 2 * ((c + 1) & 1) * TILE;
      issue_tile(nQ, q + hq, n1, w.r1);
      issue_tile(nQ + TILE, g + hq, n1, w.r1);
    }
    cp_commit();
    const long n0 = w.r0 + c * CC;
    const int nv = static_cast<int>(min(static_cast<long>(CC), w.r1 - n0));
    phi_tile(sQ, nv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // gt = dout / den; gam = -(gt . out)
      const int row = part_row(i);
      float* ptr = sG + row * LDA + part_col();
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row < nv) {
        const float inv = 1.f / dnx[i];
        const float4 x = ld4(ptr);
        f = make_float4(x.x * inv, x.y * inv, x.z * inv, x.w * inv);
      }
      st4(ptr, f);
      const float gm = -sum16(f.x * onx[i].x + f.y * onx[i].y + f.z * onx[i].z + f.w * onx[i].w);
      if ((t & 15) == 0) sgam[row] = gm;
    }
    if (c + 1 < w.nch) fetch_od(onx, dnx, o + hq, den + hn, n0 + CC, w.r1);
    __syncthreads();
    gemm_state(accR, sQ + 8 * ty, sG + 4 * tx);
    {
      const int d = t & 63, h = t >> 6;
#pragma unroll 8
      for (int j = 32 * h; j < 32 * h + 32; ++j) rc = fmaf(sgam[j], sQ[j * LDA + d], rc);
    }
    float a[8][4];
    zero(a);
    gemm_tok(a, sG + ty * LDA, sSt + 4 * tx);
    const float4 zz = ld4(sz + 4 * tx);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int row = ty + 8 * r;
      if (row < nv) {
        const float gm = sgam[row];
        const float4 f = ld4(sQ + row * LDA + 4 * tx);  // phi(Q); phi' = min(phi, 1)
        st4(dq + hq + (n0 + row) * 64 + 4 * tx,
            make_float4((a[r][0] + gm * zz.x) * fminf(f.x, 1.f), (a[r][1] + gm * zz.y) * fminf(f.y, 1.f),
                        (a[r][2] + gm * zz.z) * fminf(f.z, 1.f), (a[r][3] + gm * zz.w) * fminf(f.w, 1.f)));
      }
    }
  }
  put_partial(P, accR, rc, sx);

  cluster_sync_all();  // every partial is complete; phase 1 tiles are free

  if (w.nch > 0) {
    issue_tile(U, v + hq, w.r0, w.r1);
    issue_tile(U + TILE, k + hq, w.r0, w.r1);
  }
  cp_commit();
  float4 m[8], rv;
  cluster_sum(P, nseg, m, rv);
  cluster_sync_all();  // every CTA is done reading P, which R overwrites
  float* sRt = W;
  float* sR = W + TILE;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = t + NTC * i, row = piece_row(e), col = piece_col(e);
    st4(sR + row * LDA + col, m[i]);
    sRt[col * LDA + row] = m[i].x;
    sRt[(col + 1) * LDA + row] = m[i].y;
    sRt[(col + 2) * LDA + row] = m[i].z;
    sRt[(col + 3) * LDA + row] = m[i].w;
  }
  if (t < 16) st4(sz + 4 * t, rv);

  // phase 2: dk = (V R^T + r) * phi'(K), dv = phi(K) R
  for (int c = 0; c < w.nch; ++c) {
    float* sV = U + 2 * (c & 1) * TILE;
    float* sK = sV + TILE;
    cp_wait<0>();
    __syncthreads();  // chunk c landed; chunk c - 1 (and R, r) fully written
    if (c + 1 < w.nch) {
      const long n1 = w.r0 + (c + 1) * CC;
      float* nV = U + 2 * ((c + 1) & 1) * TILE;
      issue_tile(nV, v + hq, n1, w.r1);
      issue_tile(nV + TILE, k + hq, n1, w.r1);
    }
    cp_commit();
    const long n0 = w.r0 + c * CC;
    const int nv = static_cast<int>(min(static_cast<long>(CC), w.r1 - n0));
    phi_tile(sK, nv);
    __syncthreads();
    {
      float a[8][4];
      zero(a);
      gemm_tok(a, sV + ty * LDA, sRt + 4 * tx);
      const float4 rr = ld4(sz + 4 * tx);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int row = ty + 8 * r;
        if (row < nv) {
          const float4 f = ld4(sK + row * LDA + 4 * tx);
          st4(dk + hq + (n0 + row) * 64 + 4 * tx,
              make_float4((a[r][0] + rr.x) * fminf(f.x, 1.f), (a[r][1] + rr.y) * fminf(f.y, 1.f),
                          (a[r][2] + rr.z) * fminf(f.z, 1.f), (a[r][3] + rr.w) * fminf(f.w, 1.f)));
        }
      }
    }
    {
      float a[8][4];
      zero(a);
      gemm_tok(a, sK + ty * LDA, sR + 4 * tx);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int row = ty + 8 * r;
        if (row < nv) st4(dv + hq + (n0 + row) * 64 + 4 * tx, make_float4(a[r][0], a[r][1], a[r][2], a[r][3]));
      }
    }
  }
  cp_wait<0>();
}

template <typename K, typename... Args>
cudaError_t launch_cluster(K kernel, int nseg, int BH, size_t smem, cudaStream_t st, Args... args) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nseg) * static_cast<unsigned>(BH));
  cfg.blockDim = dim3(NTC);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(nseg);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// CTAs per (b, h): up to the portable cluster size, one per 64-token chunk
// at most, and fewer when B * H alone fills the GPU several times over.
int noncausal_cluster_nseg(int BH, int N) {
  const int nch = (N + CC - 1) / CC;
  const int fill = (6 * 152 + BH - 1) / BH;
  int n = kMaxSeg;
  if (n > nch) n = nch;
  if (n > fill) n = fill;
  return n < 1 ? 1 : n;
}

cudaError_t noncausal_cluster_fwd(const float* q, const float* k, const float* v,
                                  const int* lengths, float* out, float* den, float* S, float* Z,
                                  const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H, nseg = noncausal_cluster_nseg(BH, s.N);
  return launch_cluster(k_nc_fwd_cluster, nseg, BH, sizeof(float) * kFwdFloats, st, q, k, v,
                        lengths, out, den, S, Z, s.N, s.H, nseg);
}

cudaError_t noncausal_cluster_bwd(const float* q, const float* k, const float* v,
                                  const int* lengths, const float* out, const float* den,
                                  const float* S, const float* Z, const float* dout, float* dq,
                                  float* dk, float* dv, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H, nseg = noncausal_cluster_nseg(BH, s.N);
  return launch_cluster(k_nc_bwd_cluster, nseg, BH, sizeof(float) * kBwdFloats, st, q, k, v,
                        lengths, out, den, S, Z, dout, dq, dk, dv, s.N, s.H, nseg);
}

}  // namespace la
