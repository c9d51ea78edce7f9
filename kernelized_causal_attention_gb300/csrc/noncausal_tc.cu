// Non-causal path with D = M = 64 on the tensor cores, for fp32 and bf16
// inputs (outputs in the input type; den, S, Z fp32).
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
// fp32 accuracy from bf16 products.  An operand x is split into bf16 terms
// x_0 = bf16(x), x_i = bf16(x - x_0 - ... - x_{i-1}); every term takes 9
// more bits, so n terms leave a remainder below 2^-9n |x|.  With two terms
// a product is a_0 b_0 + a_0 b_1 + a_1 b_0 (error below 2^-16 |a| |b|); with
// three, a_0 b_0 + a_0 b_1 + a_1 b_0 + a_0 b_2 + a_1 b_1 + a_2 b_0 (below
// 2^-25 |a| |b|).  Token-form products accumulate in fp32 in two 64-column
// halves of a tensor-memory accumulator that the epilogue adds (the state
// form takes its products as quadrants instead, see mma_state):
//   two terms:   A_0 [B_0 | B_1] (N = 128), A_1 B_0 -> first half
//   three terms: A_0 [B_0 | B_1], A_1 [B_0 | B_1], A_0 B_2 -> first half,
//                A_2 B_0 -> second half
// Three terms go where the result is a small difference of large sums: dq
// = S gt + gam Z and dk = R V + r cancel, exactly so for a sequence of one
// token, so S, R, S gt and R V carry them for fp32 inputs.  out and dv
// cancel nothing and take two terms, as does everything for bf16 inputs.
//
// Layout of the work.  One thread-block cluster of nseg CTAs per (b, h); the
// valid rows are cut into 128-token chunks and every CTA takes an equal run.
//  forward   phase 1: S~ += phi(K)^T V                  (state form, two A terms stacked to M = 128)
//            cluster sum of the partial S, Z through distributed shared memory
//            phase 2: O~ = phi(Q) S                     (M = 128, token form)
//  backward  phase 1: R~ += phi(Q)^T gt, dQ~ = gt S^T
//            cluster sum of the partial R, r
//            phase 2: dK~ = V R^T, dV~ = phi(K) R
// The CUDA cores load each chunk (prefetched into registers one chunk
// ahead), apply phi, 1 / den, gam and the zeroing of invalid rows, split and
// write the swizzled operand tiles (two buffers), and run the epilogue of
// chunk c - 1 while the tensor cores work on chunk c.  den, gam, Z and r are
// plain fp32 dot products on the CUDA cores.  A CTA's partial record for the
// cluster sum lives where the state operand tiles go next; a full cluster
// barrier separates the last remote read of it from the first tile write.
//
// gam without out.  out_i = S^T phi(Q_i) / den_i, so
//   gt_i . out_i = phi(Q_i) . (S gt_i) / den_i,
// and S gt_i is the accumulator dQ~ already holds for row i: the backward
// takes gam from it in the dq epilogue and never reads out.
#include "common.cuh"
#include "launch.h"
#include "tc_chunk.cuh"

namespace la {
namespace {

using namespace tcc;

constexpr int CH = 128;              // tokens per chunk
constexpr int NTX = 512;             // threads per CTA
constexpr int NU = CH * 8 / NTX;     // 8-column units of a chunk per thread
constexpr int NCG = NTX / 128;       // column groups of a 128-lane accumulator readout
constexpr int CW = 64 / NCG;         // columns per group
constexpr int BT = CH * 128;         // bytes of a [128][64] bf16 tile
constexpr int ST = 64 * 128;         // bytes of a [64][64] bf16 tile
constexpr int PREC = 64 * 64 + 64;   // floats of a partial-state record
constexpr int N_MISC = 4 * CH + 64 + (NTX / 32) * 64 + NCG * CH;
constexpr int kMaxSeg = 8;           // CTAs per cluster (portable limit)

// Terms per operand in the cancelling products (fp32 inputs: 3, bf16: 2).
template <typename T>
struct Terms {
  static constexpr int n = 2;
};
template <>
struct Terms<float> {
  static constexpr int n = 3;
};

// Shared memory for NT-term operands, bytes from a 1024-aligned base.  A
// chunk's two operands X and Y take four tiles of the chunk's buffer: X's
// terms (the operand an epilogue reads back, if any) and Y's first term, or
// both terms of each for NT = 2.  For NT = 3, Y's terms 1 and 2 go to one
// pair of tiles that both buffers share: a chunk writes them once the MMAs
// of the chunk before have finished.  Ten tiles instead of twelve keep the
// CTA under 196 KB, which leaves L1 about 60 KB (at 228 KB of shared memory
// it keeps 28 KB and throttles the register prefetch of the next chunk).
template <int NT>
struct Lay {
  static constexpr int BUF = 4 * BT;       // one operand buffer: four term tiles
  static constexpr int O_BUF = 0;          // two operand buffers
  static constexpr int O_SHY = 2 * BUF;    // NT = 3: Y's terms 1, 2 (one pair for both buffers)
  static constexpr int O_ST = O_SHY + (NT == 3 ? 2 * BT : 0);  // state tiles, NT x [64][64]; or the partial record (fp32)
  static constexpr int N_ST = NT * ST > 4 * PREC ? NT * ST : (4 * PREC + 1023) / 1024 * 1024;
  static constexpr int O_MISC = O_ST + N_ST;  // fp32: per-row [2][128] x 2, vector [64], sums [warps][64], [4][128]
  static constexpr int O_BAR = O_MISC + 4 * N_MISC;  // mbarriers: MMA done per buffer, final drain; TMEM address
  static constexpr int SMEM = O_BAR + 64 + 1024;     // + alignment slack
  // The state form reaches a term pair's second tile through the descriptor's
  // leading offset t[1] - t[0], taken unsigned: every second tile must lie
  // above its first (X: consecutive tiles; Y: in-buffer for two terms, the
  // shared pair above both buffers' Y_0 for three), so that no MMA reads a
  // tile this launch has not written.
  static_assert(NT == 2 || O_SHY > 1 * BUF + 3 * BT, "Y's shared terms must lie above every Y_0");
};
static_assert(Lay<3>::SMEM + 16 + 1024 <= 196 * 1024, "the three-term layout fits the 196 KB carveout");
static_assert(Lay<2>::SMEM + 16 + 1024 <= 164 * 1024, "the two-term layout fits the 164 KB carveout");

// The term tiles of one operand of one chunk.
template <int NT>
struct Terms8 {
  uint8_t* t[NT];
};
// X: NT consecutive tiles from b; Y: see Lay.
template <int NT>
__device__ __forceinline__ Terms8<NT> x_tiles(uint8_t* b) {
  Terms8<NT> r;
#pragma unroll
  for (int i = 0; i < NT; ++i) r.t[i] = b + i * BT;
  return r;
}
template <int NT>
__device__ __forceinline__ Terms8<NT> y_tiles(uint8_t* b, uint8_t* shy) {
  Terms8<NT> r;
  if constexpr (NT == 3) {
    r.t[0] = b + 3 * BT;
    r.t[1] = shy;
    r.t[2] = shy + BT;
  } else {
    r.t[0] = b + 2 * BT;
    r.t[1] = b + 3 * BT;
  }
  return r;
}

// TMEM columns
constexpr uint32_t T_STATE = 0;      // the state accumulators (M = 128, 2 x 128 columns)
constexpr uint32_t T_TOK = 256;      // token-form accumulators of phase 1, 128 per buffer

// ------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
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

// -------------------------------------------------------------- helpers
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ uint32_t bits(__nv_bfloat162 h) {
  return *reinterpret_cast<uint32_t*>(&h);
}

// (x0, x1) -> NT bf16 pairs w[0], w[1], ...: each term is the bf16 rounding
// of what the earlier ones leave (the subtraction is exact in fp32), so the
// terms sum to x within 2^-9NT |x|.
template <int NT>
__device__ __forceinline__ void split(float x0, float x1, uint32_t (&w)[NT]) {
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    w[i] = bits(h);
    if (i + 1 < NT) {
      const float2 f = __bfloat1622float2(h);
      x0 -= f.x;
      x1 -= f.y;
    }
  }
}

// Columns 8 c8 .. 8 c8 + 7 of row `row` into the swizzled term tiles.
template <int NT>
__device__ __forceinline__ void put_split8(const Terms8<NT>& tl, int row, int c8, const float* x) {
  uint32_t w[4][NT];
#pragma unroll
  for (int j = 0; j < 4; ++j) split<NT>(x[2 * j], x[2 * j + 1], w[j]);
  const uint32_t off = static_cast<uint32_t>(row) * 128u + ((static_cast<uint32_t>(c8) ^ (row & 7u)) << 4);
#pragma unroll
  for (int i = 0; i < NT; ++i)
    *reinterpret_cast<uint4*>(tl.t[i] + off) = make_uint4(w[0][i], w[1][i], w[2][i], w[3][i]);
}

// Four values (columns col .. col + 3, col a multiple of 4) of row `row`.
template <int NT>
__device__ __forceinline__ void put_split4(uint8_t* t, int stride, int row, int col, float4 x) {
  uint32_t a[NT], b[NT];
  split<NT>(x.x, x.y, a);
  split<NT>(x.z, x.w, b);
  const uint32_t off = sw128_offset(row, col);
#pragma unroll
  for (int i = 0; i < NT; ++i) *reinterpret_cast<uint2*>(t + i * stride + off) = make_uint2(a[i], b[i]);
}

// Columns col0 .. col0 + NC - 1 (NC a multiple of 8) of row `row` as the sum
// of the NT term tiles at t, t + stride, ... (smallest term first).
template <int NC, int NT>
__device__ __forceinline__ void get_row(const uint8_t* t, int stride, int row, int col0, float* x) {
#pragma unroll
  for (int m = 0; m < NC / 8; ++m) {
    const uint32_t off = sw128_offset(row, col0 + 8 * m);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[8 * m + j] = 0.f;
#pragma unroll
    for (int i = NT - 1; i >= 0; --i) {
      const uint4 a = *reinterpret_cast<const uint4*>(t + i * stride + off);
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[8 * m + 2 * j] += __uint_as_float(wa[j] << 16);
        x[8 * m + 2 * j + 1] += __uint_as_float(wa[j] & 0xffff0000u);
      }
    }
  }
}

// The CTA's valid rows [r0, r1) in nch chunks, and padded rows [z0, z1).
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
  const long nchv = (L + CH - 1) / CH, per = (nchv + nseg - 1) / nseg;
  const long c0 = min(nchv, p * per), c1 = min(nchv, c0 + per);
  Rows w;
  w.r0 = c0 * CH;
  w.r1 = min(c1 * CH, L);
  w.nch = static_cast<int>(c1 - c0);
  const long zs = (N - L + nseg - 1) / nseg;
  w.z0 = min(static_cast<long>(N), L + p * zs);
  w.z1 = min(static_cast<long>(N), w.z0 + zs);
  return w;
}

// A thread's share of a chunk: units i < NU, row (t >> 3) + (NTX / 8) i,
// columns 8 (t & 7) .. + 7 (the 8 lanes of a row are consecutive).
__device__ __forceinline__ int unit_row(int i) { return (threadIdx.x >> 3) + (NTX / 8) * i; }
__device__ __forceinline__ int unit_c8() { return threadIdx.x & 7; }

// The thread's share of a chunk as loaded (converted to fp32 only when
// used, so that the loads of the next chunk stay in flight meanwhile).
template <typename T>
struct Raw;
template <>
struct Raw<float> {
  float4 v[2 * NU];
};
template <>
struct Raw<__nv_bfloat16> {
  uint4 v[NU];
};

// The thread's share of rows n0 .. n0 + 127 of x ([*][64]); rows at or past
// ne read as 0.
__device__ __forceinline__ void fetch(Raw<float>& r, const float* x, long n0, long ne) {
#pragma unroll
  for (int i = 0; i < NU; ++i) {
    const long row = n0 + unit_row(i);
    if (row < ne) {
      const float* p = x + row * 64 + 8 * unit_c8();
      r.v[2 * i] = ld4(p);
      r.v[2 * i + 1] = ld4(p + 4);
    } else {
      r.v[2 * i] = r.v[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}
__device__ __forceinline__ void fetch(Raw<__nv_bfloat16>& r, const __nv_bfloat16* x, long n0,
                                      long ne) {
#pragma unroll
  for (int i = 0; i < NU; ++i) {
    const long row = n0 + unit_row(i);
    r.v[i] = row < ne ? *reinterpret_cast<const uint4*>(x + row * 64 + 8 * unit_c8())
                      : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Unit i of a fetched share as 8 floats.
__device__ __forceinline__ void unpack(const Raw<float>& r, int i, float* x) {
  const float4 a = r.v[2 * i], b = r.v[2 * i + 1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void unpack(const Raw<__nv_bfloat16>& r, int i, float* x) {
  const uint32_t w[4] = {r.v[i].x, r.v[i].y, r.v[i].z, r.v[i].w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = __uint_as_float(w[j] << 16);
    x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}

// Four output values to global memory in the output type.
__device__ __forceinline__ void st_out(float* dst, float4 v) { st4(dst, v); }
__device__ __forceinline__ void st_out(__nv_bfloat16* dst, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  *reinterpret_cast<uint2*>(dst) = make_uint2(bits(a), bits(b));
}

// The thread's den values of rows n0 .. n0 + 127 (1 at or past ne).
__device__ __forceinline__ void fetch_den(float (&rd)[NU], const float* dh, long n0, long ne) {
#pragma unroll
  for (int i = 0; i < NU; ++i) {
    const long row = n0 + unit_row(i);
    rd[i] = row < ne ? dh[row] : 1.f;
  }
}


__device__ __forceinline__ float sum8(float x) {  // over the 8 lanes of a row
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x;
}

// ------------------------------------------------------------------ MMAs
// One 16-deep step of an NT-term product into the accumulator halves d and
// d + 64: a0..a2 the A term descriptors, b01 the N = 128 pair [B_0 | B_1],
// b0 and b2 single N = 64 terms.  acc = 0 overwrites on the first
// instruction.
template <int NT>
__device__ __forceinline__ void mma_step(uint32_t d, uint64_t a0, uint64_t a1, uint64_t a2,
                                         uint64_t b01, uint64_t b0, uint64_t b2, uint32_t i128,
                                         uint32_t i64, uint32_t acc) {
  mma_bf16(d, a0, b01, i128, acc);
  if (NT == 2) {
    mma_bf16(d, a1, b0, i64, 1);
  } else {
    mma_bf16(d, a1, b01, i128, 1);
    mma_bf16(d, a0, b2, i64, 1);
    mma_bf16(d + 64, a2, b0, i64, 1);
  }
}

// Shared-memory addresses of an operand's term tiles.
struct TermAddr {
  uint32_t t[3];  // unused terms repeat the last one
};
template <int NT>
__device__ __forceinline__ TermAddr taddr(const Terms8<NT>& tl) {
  TermAddr r;
#pragma unroll
  for (int i = 0; i < 3; ++i) r.t[i] = static_cast<uint32_t>(__cvta_generic_to_shared(tl.t[i < NT ? i : NT - 1]));
  return r;
}

// State form over one chunk, A^T B with A and B each NT term tiles
// ([128 tokens][64]) read MN-major (16 tokens = 2048 bytes per step).  Two
// terms stacked along M against two along N (the second tile of a pair is
// reached by the descriptor's leading offset, so it only has to lie above
// the first) make one M = N = 128 instruction whose quadrants are the four
// products a_i b_j, i, j < 2:
//   D   (+)= [A_0; A_1]^T [B_0 | B_1]
// and with three terms a second accumulator 128 columns on holds
//   D'  (+)= [A_0; A_2]^T [B_0 | B_2],
// whose off-diagonal quadrants are a_0 b_2 and a_2 b_0 (the diagonal ones
// are not used).
template <int NT>
__device__ __forceinline__ void mma_state(uint32_t d, const TermAddr& a, const TermAddr& b,
                                          bool first) {
  constexpr uint32_t I = idesc_bf16(128, 128, true, true);
  const uint64_t da01 = sdesc(a.t[0], a.t[1] - a.t[0], 1024), db01 = sdesc(b.t[0], b.t[1] - b.t[0], 1024);
  const uint64_t da02 = sdesc(a.t[0], a.t[2] - a.t[0], 1024), db02 = sdesc(b.t[0], b.t[2] - b.t[0], 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t o = 2048 * kk, acc = !first || kk > 0;
    mma_bf16(d, dadd(da01, o), dadd(db01, o), I, acc);
    if (NT == 3) mma_bf16(d + 128, dadd(da02, o), dadd(db02, o), I, acc);
  }
}

// Token form over one chunk: D (M = 128 tokens, N = 128 as two halves) = A B,
// A NT K-major [128][64] term tiles, B NT state term tiles at b (ST apart):
// MN-major ([K = 64 rows][N]) when b_mn, else K-major ([N rows][K]; the
// first two terms' rows are contiguous, which makes the N = 128 pair).
template <int NT>
__device__ __forceinline__ void mma_tok(uint32_t d, const TermAddr& a, uint32_t b, bool b_mn) {
  const uint64_t da0 = sdesc(a.t[0], 16, 1024), da1 = sdesc(a.t[1], 16, 1024),
                 da2 = sdesc(a.t[2], 16, 1024);
  const uint64_t db0 = sdesc(b, 16, 1024), db2 = sdesc(b + 2 * ST, 16, 1024);
  if (b_mn) {
    constexpr uint32_t I128 = idesc_bf16(128, 128, false, true);
    constexpr uint32_t I64 = idesc_bf16(128, 64, false, true);
    const uint64_t db01 = sdesc(b, ST, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_step<NT>(d, dadd(da0, 32 * kk), dadd(da1, 32 * kk), dadd(da2, 32 * kk),
                   dadd(db01, 2048 * kk), dadd(db0, 2048 * kk), dadd(db2, 2048 * kk), I128, I64,
                   kk > 0);
  } else {
    constexpr uint32_t I128 = idesc_bf16(128, 128, false, false);
    constexpr uint32_t I64 = idesc_bf16(128, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_step<NT>(d, dadd(da0, 32 * kk), dadd(da1, 32 * kk), dadd(da2, 32 * kk),
                   dadd(db0, 32 * kk), dadd(db0, 32 * kk), dadd(db2, 32 * kk), I128, I64, kk > 0);
  }
}

// ------------------------------------------------------ shared pieces
struct Ctx {
  uint8_t* sm;
  uint64_t* bar;  // [0], [1]: MMA of buffer 0 / 1 done; [2]: final drain
  int* abort;
  int* err;       // the library's status word
  int site;       // this kernel's code in it
  uint32_t tm;
};

// Waits for the MMAs of global chunk g; agreed by the whole warp (the TMEM
// loads that follow are warp-collective).  Gives up after WAIT_NS, records
// the kernel's code in the status word and sets the CTA's abort flag, after
// which every wait fails at once and no further MMA is issued.
__device__ __forceinline__ bool wait_chunk(const Ctx& x, uint32_t g) {
  bool ok = false;
  if (!*reinterpret_cast<volatile int*>(x.abort)) {
    ok = mbar_wait(&x.bar[g & 1], (g >> 1) & 1, WAIT_NS);
    if (!ok) {
      *reinterpret_cast<volatile int*>(x.abort) = 1;
      fail(x.err, x.site);
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// CW columns (col .. col + CW - 1) of the thread's TMEM lane from the two
// halves of a 128-column accumulator (col and col + 64); one wait.
__device__ __forceinline__ void ld_halves(uint32_t taddr, float* a, float* b) {
#pragma unroll
  for (int j = 0; j < CW; j += 16) {
    tmem_ld16(taddr + j, a + j);
    tmem_ld16(taddr + 64 + j, b + j);
  }
  tmem_ld_wait();
}

// Readout of the state accumulators into P ([64][64] fp32): the thread
// holds accumulator row 32 (warp & 3) + lane, columns CW (warp >> 2) .. and
// the same + 64, i.e. state row (that row mod 64).  Rows < 64 are the A_0
// quadrants (plus a_0 b_2 from the second accumulator's right half), rows
// >= 64 the A_1 ones (plus a_2 b_0 from its left half); the upper rows are
// written first and the lower ones added.
template <int NT>
__device__ __forceinline__ void state_readout(const Ctx& x, bool ok, float* P) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, qd = warp & 3, cg = warp >> 2;
  const uint32_t ta = x.tm + T_STATE + ((32u * qd) << 16) + CW * cg;
  float a[CW], b[CW], c[CW];
  if (ok) {
#pragma unroll
    for (int j = 0; j < CW; j += 16) {
      tmem_ld16(ta + j, a + j);
      tmem_ld16(ta + 64 + j, b + j);
      if (NT == 3) tmem_ld16(ta + 128 + (qd < 2 ? 64 : 0) + j, c + j);
    }
    tmem_ld_wait();
  } else {
#pragma unroll
    for (int j = 0; j < CW; ++j) a[j] = b[j] = c[j] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < CW; ++j) a[j] += NT == 3 ? b[j] + c[j] : b[j];
  float* dst = P + ((32 * qd + lane) & 63) * 64 + CW * cg;
  if (qd < 2)
#pragma unroll
    for (int j = 0; j < CW; j += 4) st4(dst + j, make_float4(a[j], a[j + 1], a[j + 2], a[j + 3]));
  __syncthreads();
  if (qd >= 2)
#pragma unroll
    for (int j = 0; j < CW; j += 4) st4(dst + j, add4(ld4(dst + j), make_float4(a[j], a[j + 1], a[j + 2], a[j + 3])));
}

// Column sums of the thread's 8 columns over all threads -> P[4096 + d].
__device__ __forceinline__ void colsum_to_record(float (&cs)[8], float* scol, float* P) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    cs[j] += __shfl_xor_sync(0xffffffffu, cs[j], 8);
    cs[j] += __shfl_xor_sync(0xffffffffu, cs[j], 16);
  }
  if (lane < 8)
#pragma unroll
    for (int j = 0; j < 8; ++j) scol[warp * 64 + 8 * lane + j] = cs[j];
  __syncthreads();
  if (threadIdx.x < 64) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NTX / 32; ++w) s += scol[w * 64 + threadIdx.x];
    P[64 * 64 + threadIdx.x] = s;
  }
}

constexpr int NPC = 1024 / NTX;  // matrix pieces per thread in the cluster sum

// Sum over the cluster of the records P: thread t gets matrix pieces
// t + NTX i (i < NPC; piece e = row e >> 4, columns 4 (e & 15) ..) and, for
// t < 16, vector piece t.  Four peers' loads are in flight at a time.
__device__ __forceinline__ void cluster_sum(const float* P, int nseg, float4 (&m)[NPC], float4& vec) {
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(P));
  const int t = threadIdx.x;
#pragma unroll
  for (int i = 0; i < NPC; ++i) m[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  vec = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = 0; q0 < nseg; q0 += 4) {
    float4 part[4][NPC + 1];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (q0 + u < nseg) {
        const uint32_t a = map_rank(base, static_cast<uint32_t>(q0 + u));
#pragma unroll
        for (int i = 0; i < NPC; ++i) part[u][i] = ld_cluster4(a + 16u * (t + NTX * i));
        part[u][NPC] = t < 16 ? ld_cluster4(a + 16u * (1024 + t)) : make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
#pragma unroll
        for (int i = 0; i <= NPC; ++i) part[u][i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int i = 0; i < NPC; ++i) m[i] = add4(m[i], part[u][i]);
      vec = add4(vec, part[u][NPC]);
    }
  }
}

// Setup shared by both kernels: barriers (at byte o_bar), abort flag, TMEM.
__device__ __forceinline__ Ctx setup(uint8_t* smraw, int* s_abort, int o_bar, int* err, int site) {
  Ctx x;
  x.sm = align1024(smraw);
  x.bar = reinterpret_cast<uint64_t*>(x.sm + o_bar);
  x.abort = s_abort;
  x.err = err;
  x.site = site;
  uint32_t* slot = reinterpret_cast<uint32_t*>(x.sm + o_bar + 32);
  if (threadIdx.x == 0) {
    mbar_init(&x.bar[0], 1);
    mbar_init(&x.bar[1], 1);
    mbar_init(&x.bar[2], 1);
    fence_barrier_init();
    *s_abort = 0;
  }
  if ((threadIdx.x >> 5) == 0) tmem_alloc(slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  x.tm = *slot;
  return x;
}

// Teardown: no MMA in flight (a bounded drain), TMEM freed.  (No peer
// reads this CTA's shared memory any more: the cluster barrier after the
// sum saw to that.)
__device__ __forceinline__ void teardown(const Ctx& x) {
  if (threadIdx.x == 0) {
    mma_commit(&x.bar[2]);
    if (!mbar_wait(&x.bar[2], 0, WAIT_NS)) fail(x.err, x.site + 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(x.tm, 512);
}

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- forward
template <typename T>
__global__ void __launch_bounds__(NTX, 1)
    k_nc_fwd_tc(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                const int* __restrict__ lengths, T* __restrict__ out, float* __restrict__ den,
                float* __restrict__ S,
                float* __restrict__ Z, int N, int H, int nseg, int* err) {
  constexpr int NT = Terms<T>::n;
  using L = Lay<NT>;
  extern __shared__ uint8_t smraw[];
  __shared__ int s_abort;
  const Ctx x = setup(smraw, &s_abort, L::O_BAR, err, 31);
  uint8_t* sm = x.sm;
  float* P = reinterpret_cast<float*>(sm + L::O_ST);     // partial record, then
  uint8_t* SH = sm + L::O_ST;                            // the S terms 0, 1
  float* sden = reinterpret_cast<float*>(sm + L::O_MISC);  // [2][128]
  float* sz = sden + 2 * CH;                             // Z [64]
  float* scol = sz + 64;                                 // [warps][64]
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, qd = warp & 3, cg = warp >> 2;
  const int p = static_cast<int>(cluster_rank()), bh = blockIdx.x / nseg;
  const Rows w = my_rows(lengths, bh / H, N, p, nseg);
  const long hq = static_cast<long>(bh) * N * 64, hn = static_cast<long>(bh) * N;
  const int c8 = unit_c8();

  uint32_t g = 0;  // chunks issued so far: buffer g & 1, barrier parity (g >> 1) & 1
  Raw<T> ra, rb;
  if (w.nch > 0) {
    fetch(ra, k + hq, w.r0, w.r1);
    fetch(rb, v + hq, w.r0, w.r1);
  }

  // ---- phase 1: partial S~ and Z
  float cs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int c = 0; c < w.nch; ++c, ++g) {
    uint8_t* B0 = sm + L::O_BUF + (g & 1) * L::BUF;
    const Terms8<NT> tx = x_tiles<NT>(B0), ty = y_tiles<NT>(B0, sm + L::O_SHY);  // phi(K), V
    const long n0 = w.r0 + static_cast<long>(c) * CH;
    const int nv = static_cast<int>(min(static_cast<long>(CH), w.r1 - n0));
#pragma unroll
    for (int i = 0; i < NU; ++i) {
      const int row = unit_row(i);
      float a[8];
      unpack(ra, i, a);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        a[j] = row < nv ? phi(a[j]) : 0.f;
        cs[j] += a[j];
      }
      put_split8<NT>(tx, row, c8, a);
    }
    if (c + 1 < w.nch) fetch(ra, k + hq, n0 + CH, w.r1);
    if (c > 0) wait_chunk(x, g - 1);  // the MMAs of the chunk before: frees the shared tiles
#pragma unroll
    for (int i = 0; i < NU; ++i) {
      float b[8];
      unpack(rb, i, b);
      put_split8<NT>(ty, unit_row(i), c8, b);
    }
    if (c + 1 < w.nch) fetch(rb, v + hq, n0 + CH, w.r1);
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (t == 0 && !s_abort) {
      tc_fence_after();
      mma_state<NT>(x.tm + T_STATE, taddr(tx), taddr(ty), c == 0);
      mma_commit(&x.bar[g & 1]);
    }
  }
  {
    const bool ok = w.nch > 0 && wait_chunk(x, g - 1);
    tc_fence_after();
    state_readout<NT>(x, ok, P);
  }
  colsum_to_record(cs, scol, P);
  tc_fence_before();
  cluster_arrive();
  // padded rows, while the slower CTAs of the cluster finish phase 1
  for (long e = w.z0 * 16 + t; e < w.z1 * 16; e += NTX) st_out(out + hq + 4 * e, make_float4(0.f, 0.f, 0.f, 0.f));
  if (den != nullptr)
    for (long i = w.z0 + t; i < w.z1; i += NTX) den[hn + i] = 0.f;
  cluster_wait();  // every record complete

  // ---- phase 2: out = phi(Q) S / den
  if (w.nch > 0) fetch(ra, q + hq, w.r0, w.r1);
  {
    float4 m[NPC], zv;
    cluster_sum(P, nseg, m, zv);
    cluster_arrive();  // this CTA no longer reads the others' records
    if (p == 0) {
#pragma unroll
      for (int i = 0; i < NPC; ++i) st4(S + static_cast<long>(bh) * 4096 + 4 * (t + NTX * i), m[i]);
      if (t < 16) st4(Z + static_cast<long>(bh) * 64 + 4 * t, zv);
    }
    if (t < 16) st4(sz + 4 * t, zv);
    cluster_wait();  // nor does any other CTA read this one's: the S tiles replace it
#pragma unroll
    for (int i = 0; i < NPC; ++i) {
      const int e = t + NTX * i;
      put_split4<2>(SH, ST, e >> 4, 4 * (e & 15), m[i]);
    }
  }
  fence_proxy_async();
  __syncthreads();
  float zc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) zc[j] = sz[8 * c8 + j];
  const uint32_t tok0 = x.tm + T_TOK;
  for (int c = 0; c <= w.nch; ++c) {
    if (c < w.nch) {
      uint8_t* B0 = sm + L::O_BUF + (g & 1) * L::BUF;
      const Terms8<2> tx = x_tiles<2>(B0);  // phi(Q), two terms
      const long n0 = w.r0 + static_cast<long>(c) * CH;
      const int nv = static_cast<int>(min(static_cast<long>(CH), w.r1 - n0));
#pragma unroll
      for (int i = 0; i < NU; ++i) {
        const int row = unit_row(i);
        float a[8];
        unpack(ra, i, a);
        float dp = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          a[j] = row < nv ? phi(a[j]) : 0.f;
          dp = fmaf(a[j], zc[j], dp);
        }
        dp = sum8(dp);
        if (c8 == 0) {
          sden[(g & 1) * CH + row] = dp;
          if (den != nullptr && row < nv) den[hn + n0 + row] = dp;
        }
        put_split8<2>(tx, row, c8, a);
      }
      if (c + 1 < w.nch) fetch(ra, q + hq, n0 + CH, w.r1);
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (t == 0 && !s_abort) {
        tc_fence_after();
        mma_tok<2>(tok0 + 128 * (g & 1), taddr(tx), saddr(SH), true);
        mma_commit(&x.bar[g & 1]);
      }
      ++g;
    }
    if (c > 0) {  // epilogue of chunk c - 1 (global chunk g - 1 or g - 2)
      const uint32_t ge = c < w.nch ? g - 2 : g - 1;
      const bool ok = wait_chunk(x, ge);
      tc_fence_after();
      if (ok) {
        const long n0 = w.r0 + static_cast<long>(c - 1) * CH;
        const int nv = static_cast<int>(min(static_cast<long>(CH), w.r1 - n0));
        const int row = 32 * qd + lane;
        float a[CW], b[CW];
        ld_halves(tok0 + 128 * (ge & 1) + ((32u * qd) << 16) + CW * cg, a, b);
        if (row < nv) {
          const float inv = 1.f / sden[(ge & 1) * CH + row];
          T* dst = out + hq + (n0 + row) * 64 + CW * cg;
#pragma unroll
          for (int j = 0; j < CW; j += 4)
            st_out(dst + j, make_float4((a[j] + b[j]) * inv, (a[j + 1] + b[j + 1]) * inv,
                                     (a[j + 2] + b[j + 2]) * inv, (a[j + 3] + b[j + 3]) * inv));
        }
      }
      tc_fence_before();
      __syncthreads();  // the next transform rewrites what this epilogue read
    }
  }
  teardown(x);
}

// --------------------------------------------------------------- backward
template <typename T>
__global__ void __launch_bounds__(NTX, 1)
    k_nc_bwd_tc(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                const int* __restrict__ lengths, const float* __restrict__ den,
                const float* __restrict__ S, const float* __restrict__ Z,
                const T* __restrict__ gr, T* __restrict__ dq, T* __restrict__ dk,
                T* __restrict__ dv, int N, int H, int nseg, int* err) {
  constexpr int NT = Terms<T>::n;
  using L = Lay<NT>;
  extern __shared__ uint8_t smraw[];
  __shared__ int s_abort;
  const Ctx x = setup(smraw, &s_abort, L::O_BAR, err, 33);
  uint8_t* sm = x.sm;
  uint8_t* SH = sm + L::O_ST;  // phase 1: the S terms; then the partial record; phase 2: the R terms
  float* P = reinterpret_cast<float*>(SH);
  float* sinv = reinterpret_cast<float*>(sm + L::O_MISC);  // 1 / den [2][128]
  float* sz = sinv + 4 * CH;                             // phase 1: Z; phase 2: r
  float* scol = sz + 64;                                 // [warps][64]
  float* spart = scol + (NTX / 32) * 64;                 // [NCG][128]
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, qd = warp & 3, cg = warp >> 2;
  const int p = static_cast<int>(cluster_rank()), bh = blockIdx.x / nseg;
  const Rows w = my_rows(lengths, bh / H, N, p, nseg);
  const long hq = static_cast<long>(bh) * N * 64, hn = static_cast<long>(bh) * N;
  const int c8 = unit_c8();

  uint32_t g = 0;
  Raw<T> ra, rb;
  float rd[NU];
  if (w.nch > 0) {
    fetch(ra, q + hq, w.r0, w.r1);
    fetch(rb, gr + hq, w.r0, w.r1);
    fetch_den(rd, den + hn, w.r0, w.r1);
  }
  // S (the forward's state) as NT operand term tiles; Z
#pragma unroll
  for (int i = 0; i < NPC; ++i) {
    const int e = t + NTX * i;
    put_split4<NT>(SH, ST, e >> 4, 4 * (e & 15), ld4(S + static_cast<long>(bh) * 4096 + 4 * e));
  }
  if (t < 64) sz[t] = Z[static_cast<long>(bh) * 64 + t];
  fence_proxy_async();
  __syncthreads();  // S tiles and Z in place

  // ---- phase 1: gt, dq, gam and partial R~, r
  float rp[CW];  // r over the thread's epilogue rows, columns CW cg ..
#pragma unroll
  for (int j = 0; j < CW; ++j) rp[j] = 0.f;
  const uint32_t tok0 = x.tm + T_TOK;
  for (int c = 0; c <= w.nch; ++c) {
    if (c < w.nch) {
      uint8_t* B0 = sm + L::O_BUF + (g & 1) * L::BUF;
      const Terms8<NT> tx = x_tiles<NT>(B0), ty = y_tiles<NT>(B0, sm + L::O_SHY);  // phi(Q), gt
      const long n0 = w.r0 + static_cast<long>(c) * CH;
      const int nv = static_cast<int>(min(static_cast<long>(CH), w.r1 - n0));
#pragma unroll
      for (int i = 0; i < NU; ++i) {
        const int row = unit_row(i);
        float a[8];
        unpack(ra, i, a);
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = row < nv ? phi(a[j]) : 0.f;
        put_split8<NT>(tx, row, c8, a);
      }
      if (c + 1 < w.nch) fetch(ra, q + hq, n0 + CH, w.r1);
      if (c > 0) wait_chunk(x, g - 1);  // the MMAs of the chunk before: frees the shared tiles
#pragma unroll
      for (int i = 0; i < NU; ++i) {
        const int row = unit_row(i);
        const float inv = row < nv ? 1.f / rd[i] : 0.f;
        float b[8];
        unpack(rb, i, b);
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] *= inv;
        if (c8 == 0) sinv[(g & 1) * CH + row] = inv;
        put_split8<NT>(ty, row, c8, b);
      }
      if (c + 1 < w.nch) {
        fetch(rb, gr + hq, n0 + CH, w.r1);
        fetch_den(rd, den + hn, n0 + CH, w.r1);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (t == 0 && !s_abort) {
        tc_fence_after();
        const TermAddr ay = taddr(ty);
        mma_state<NT>(x.tm + T_STATE, taddr(tx), ay, c == 0);
        mma_tok<NT>(tok0 + 128 * (g & 1), ay, saddr(SH), false);
        mma_commit(&x.bar[g & 1]);
      }
      ++g;
    }
    if (c > 0) {  // gam, dq and r of chunk c - 1
      const uint32_t ge = c < w.nch ? g - 2 : g - 1;
      const bool ok = wait_chunk(x, ge);
      tc_fence_after();
      const long n0 = w.r0 + static_cast<long>(c - 1) * CH;
      const int nv = static_cast<int>(min(static_cast<long>(CH), w.r1 - n0));
      const int row = 32 * qd + lane;
      const uint8_t* B0 = sm + L::O_BUF + (ge & 1) * L::BUF;
      float a[CW], b[CW], f[CW];
      if (ok) {
        ld_halves(tok0 + 128 * (ge & 1) + ((32u * qd) << 16) + CW * cg, a, b);
      } else {
#pragma unroll
        for (int j = 0; j < CW; ++j) a[j] = b[j] = 0.f;
      }
      get_row<CW, NT>(B0, BT, row, CW * cg, f);  // phi(Q) (0 on invalid rows); phi' = min(phi, 1)
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < CW; ++j) {
        a[j] += b[j];  // S gt
        part = fmaf(f[j], a[j], part);
      }
      spart[cg * CH + row] = part;
      __syncthreads();
      float dsum = 0.f;
#pragma unroll
      for (int u = 0; u < NCG; ++u) dsum += spart[u * CH + row];
      const float gm = -dsum * sinv[(ge & 1) * CH + row];
      if (row < nv) {
        T* dst = dq + hq + (n0 + row) * 64 + CW * cg;
#pragma unroll
        for (int j = 0; j < CW; j += 4) {
          float r4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) r4[u] = (a[j + u] + gm * sz[CW * cg + j + u]) * fminf(f[j + u], 1.f);
          st_out(dst + j, make_float4(r4[0], r4[1], r4[2], r4[3]));
        }
      }
#pragma unroll
      for (int j = 0; j < CW; ++j) rp[j] = fmaf(gm, f[j], rp[j]);
      tc_fence_before();
      __syncthreads();  // the next transform rewrites what this epilogue read
    }
  }
  {
    const bool ok = w.nch > 0 && !*reinterpret_cast<volatile int*>(x.abort);
    tc_fence_after();
    state_readout<NT>(x, __all_sync(0xffffffffu, ok), P);
  }
  // r: the thread's CW columns summed over its warp's lanes, then over the
  // four lane quarters of its column group
#pragma unroll
  for (int j = 0; j < CW; ++j)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rp[j] += __shfl_xor_sync(0xffffffffu, rp[j], o);
  if (lane == 0)
#pragma unroll
    for (int j = 0; j < CW; ++j) scol[warp * 64 + j] = rp[j];
  __syncthreads();
  if (t < 64) {
    const int gc = t / CW, j = t % CW;
    float sr = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) sr += scol[(4 * gc + u) * 64 + j];
    P[64 * 64 + t] = sr;
  }
  tc_fence_before();
  cluster_arrive();
  // padded rows, while the slower CTAs of the cluster finish phase 1
  for (long e = w.z0 * 16 + t; e < w.z1 * 16; e += NTX) {
    st_out(dq + hq + 4 * e, make_float4(0.f, 0.f, 0.f, 0.f));
    st_out(dk + hq + 4 * e, make_float4(0.f, 0.f, 0.f, 0.f));
    st_out(dv + hq + 4 * e, make_float4(0.f, 0.f, 0.f, 0.f));
  }
  cluster_wait();  // every record complete

  // ---- phase 2: dk = (V R^T + r) * phi'(K), dv = phi(K) R
  if (w.nch > 0) {
    fetch(ra, v + hq, w.r0, w.r1);
    fetch(rb, k + hq, w.r0, w.r1);
  }
  {
    float4 m[NPC], rv;
    cluster_sum(P, nseg, m, rv);
    cluster_arrive();  // this CTA no longer reads the others' records
    if (t < 16) st4(sz + 4 * t, rv);
    cluster_wait();  // nor does any other CTA read this one's: the R tiles replace it
#pragma unroll
    for (int i = 0; i < NPC; ++i) {
      const int e = t + NTX * i;
      put_split4<NT>(SH, ST, e >> 4, 4 * (e & 15), m[i]);
    }
  }
  fence_proxy_async();
  __syncthreads();
  const uint32_t t2 = x.tm;  // phase 2: buffer b uses columns 256 b .. 256 b + 255
  for (int c = 0; c <= w.nch; ++c) {
    if (c < w.nch) {
      uint8_t* B0 = sm + L::O_BUF + (g & 1) * L::BUF;
      // phi(K): two terms in tiles 2, 3 (the epilogue reads them back);
      // V: tiles 0, 1 and, for three terms, the first shared tile
      const Terms8<2> tk = x_tiles<2>(B0 + 2 * BT);
      Terms8<NT> tv;
      tv.t[0] = B0;
      tv.t[1] = B0 + BT;
      if constexpr (NT == 3) tv.t[2] = sm + L::O_SHY;
      const long n0 = w.r0 + static_cast<long>(c) * CH;
      const int nv = static_cast<int>(min(static_cast<long>(CH), w.r1 - n0));
#pragma unroll
      for (int i = 0; i < NU; ++i) {
        const int row = unit_row(i);
        float b[8];
        unpack(rb, i, b);
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] = row < nv ? phi(b[j]) : 0.f;
        put_split8<2>(tk, row, c8, b);
      }
      if (c + 1 < w.nch) fetch(rb, k + hq, n0 + CH, w.r1);
      if (NT == 3 && c > 0) wait_chunk(x, g - 1);  // the MMAs of the chunk before: frees the shared tile
#pragma unroll
      for (int i = 0; i < NU; ++i) {
        float a[8];
        unpack(ra, i, a);
        put_split8<NT>(tv, unit_row(i), c8, a);
      }
      if (c + 1 < w.nch) fetch(ra, v + hq, n0 + CH, w.r1);
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (t == 0 && !s_abort) {
        tc_fence_after();
        const uint32_t d0 = t2 + 256 * (g & 1);
        mma_tok<NT>(d0, taddr(tv), saddr(SH), false);       // V R^T
        mma_tok<2>(d0 + 128, taddr(tk), saddr(SH), true);  // phi(K) R
        mma_commit(&x.bar[g & 1]);
      }
      ++g;
    }
    if (c > 0) {  // dk, dv of chunk c - 1
      const uint32_t ge = c < w.nch ? g - 2 : g - 1;
      const bool ok = wait_chunk(x, ge);
      tc_fence_after();
      if (ok) {
        const long n0 = w.r0 + static_cast<long>(c - 1) * CH;
        const int nv = static_cast<int>(min(static_cast<long>(CH), w.r1 - n0));
        const int row = 32 * qd + lane;
        const uint32_t acc = t2 + 256 * (ge & 1) + ((32u * qd) << 16) + CW * cg;
        const uint8_t* B0 = sm + L::O_BUF + (ge & 1) * L::BUF;
        float a[CW], b[CW];
        ld_halves(acc, a, b);
        if (row < nv) {
          float f[CW];
          get_row<CW, 2>(B0 + 2 * BT, BT, row, CW * cg, f);  // phi(K) to 2^-18, for phi'
          T* dst = dk + hq + (n0 + row) * 64 + CW * cg;
#pragma unroll
          for (int j = 0; j < CW; j += 4) {
            float r4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              r4[u] = (a[j + u] + b[j + u] + sz[CW * cg + j + u]) * fminf(f[j + u], 1.f);
            st_out(dst + j, make_float4(r4[0], r4[1], r4[2], r4[3]));
          }
        }
        ld_halves(acc + 128, a, b);
        if (row < nv) {
          T* dst = dv + hq + (n0 + row) * 64 + CW * cg;
#pragma unroll
          for (int j = 0; j < CW; j += 4)
            st_out(dst + j, make_float4(a[j] + b[j], a[j + 1] + b[j + 1], a[j + 2] + b[j + 2], a[j + 3] + b[j + 3]));
        }
      }
      tc_fence_before();
      __syncthreads();  // the next transform rewrites what this epilogue read
    }
  }
  teardown(x);
}

template <typename K, typename... Args>
cudaError_t launch_cluster(K kernel, int smem, int nseg, int BH, cudaStream_t st, Args... args) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nseg) * static_cast<unsigned>(BH));
  cfg.blockDim = dim3(NTX);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
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

template <typename T>
cudaError_t run_fwd(const T* q, const T* k, const T* v, const int* lengths, T* out, float* den,
                    float* S, float* Z, const Shape& s, int nseg, cudaStream_t st) {
  return launch_cluster(k_nc_fwd_tc<T>, Lay<Terms<T>::n>::SMEM, nseg, s.B * s.H, st, q, k, v, lengths, out, den, S, Z,
                        s.N, s.H, nseg, status_word());
}

template <typename T>
cudaError_t run_bwd(const T* q, const T* k, const T* v, const int* lengths, const float* den,
                    const float* S, const float* Z, const T* dout, T* dq, T* dk, T* dv,
                    const Shape& s, int nseg, cudaStream_t st) {
  return launch_cluster(k_nc_bwd_tc<T>, Lay<Terms<T>::n>::SMEM, nseg, s.B * s.H, st, q, k, v, lengths, den, S, Z, dout, dq,
                        dk, dv, s.N, s.H, nseg, status_word());
}

}  // namespace

// CTAs per (b, h): a power of two (clusters of 1, 2, 4 or 8 CTAs pack the
// GPCs without holes), at most one per 128-token chunk, and about one and a
// half waves of one CTA per SM over all (b, h): every CTA pays fixed costs
// (first loads, the cluster barrier and sum, the last epilogue), so fewer,
// longer CTAs win once the SMs are full (96 heads of 800-2048 tokens: 2 per
// head beat 4 by 4-12 us per call, 1 per head leaves SMs idle).
int noncausal_tc_nseg(int BH, int N) {
  const int nch = (N + CH - 1) / CH;
  const int fill = (3 * sm_count() / 2 + BH - 1) / BH;
  int n = kMaxSeg;
  while (n > 1 && (n > nch || n > fill)) n >>= 1;
  return n;
}

cudaError_t noncausal_tc_fwd(const void* q, const void* k, const void* v, const int* lengths,
                             void* out, float* den, float* S, float* Z, const Shape& s,
                             cudaStream_t st) {
  const int BH = s.B * s.H, nseg = noncausal_tc_nseg(BH, s.N);
  if (s.dtype == 0)
    return run_fwd<float>(static_cast<const float*>(q), static_cast<const float*>(k),
                          static_cast<const float*>(v), lengths, static_cast<float*>(out), den, S,
                          Z, s, nseg, st);
  using B16 = __nv_bfloat16;
  return run_fwd<B16>(static_cast<const B16*>(q), static_cast<const B16*>(k),
                      static_cast<const B16*>(v), lengths, static_cast<B16*>(out), den, S, Z, s,
                      nseg, st);
}

cudaError_t noncausal_tc_bwd(const void* q, const void* k, const void* v, const int* lengths,
                             const float* den, const float* S, const float* Z, const void* dout,
                             void* dq, void* dk, void* dv, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H, nseg = noncausal_tc_nseg(BH, s.N);
  if (s.dtype == 0)
    return run_bwd<float>(static_cast<const float*>(q), static_cast<const float*>(k),
                          static_cast<const float*>(v), lengths, den, S, Z,
                          static_cast<const float*>(dout), static_cast<float*>(dq),
                          static_cast<float*>(dk), static_cast<float*>(dv), s, nseg, st);
  using B16 = __nv_bfloat16;
  return run_bwd<B16>(static_cast<const B16*>(q), static_cast<const B16*>(k),
                      static_cast<const B16*>(v), lengths, den, S, Z,
                      static_cast<const B16*>(dout), static_cast<B16*>(dq), static_cast<B16*>(dk),
                      static_cast<B16*>(dv), s, nseg, st);
}

}  // namespace la
