// Causal linear attention on the 5th-generation tensor cores (tcgen05), for
// bf16 inputs with D = M = 64 and fp32 accumulation in tensor memory.
//
// Method: "Transformers are RNNs" (part 2/3), §3.3 eq. 9-12 (forward) and
// §3.3.1 eq. 13-15 (cumulative-sum backward with the denominator terms).
//
// GB300 design (not the pages'): each (b, h) sequence is cut into segments of
// whole 128-token chunks, one CTA per segment (one CTA per SM).  Inside a CTA
// one warp streams raw Q/K/V chunks with TMA into a two-stage shared-memory
// ring (128-byte swizzle), four compute warps apply phi in place, and one
// thread issues the tcgen05 MMAs whose fp32 accumulators live in tensor
// memory.  The value matrix is augmented with a column of ones, V~ = [V | 1],
// so one accumulator carries both the state and the normaliser,
// S~ = [S | z] = sum phi(K_j) V~_j^T, and every product that yields a
// numerator yields its denominator in column 64:
//   A    = phi(Q) phi(K)^T                        (128 x 128, K = 64)
//   P    = bf16(mask(A))                           (compute warps, TMEM -> smem)
//   O~   = P V~ + phi(Q) bf16(S~_prev)            (128 x 80)  -> out = O~[:, :64] / O~[:, 64]
//   S~  += phi(K)^T V~                             (64 x 80, carried across chunks)
// Segment prefixes come from a state pass (same kernel, MODE 0) and a scan.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace la {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int TC_C = 128;                  // tokens per chunk (MMA M)
constexpr int TC_MA = 80;                  // augmented value width [V | 1 | 0 ...]
constexpr int NST = 2;                     // TMA ring stages
constexpr int TILE = TC_C * 64 * 2;        // one [128][64] bf16 tile
constexpr int NTHR = 192;                  // warp 0 TMA, warp 1 MMA, warps 2-5 compute
constexpr uint64_t WAIT_NS = 2000000000ull;  // bound on every wait

// shared-memory map of the forward kernel (offsets from a 1024-aligned base)
constexpr int F_STAGE = 3 * TILE;          // Q, K, V
constexpr int F_ONES = NST * F_STAGE;      // [128][64], column 0 = 1
constexpr int F_P = F_ONES + TILE;         // P, keys 0-63 then 64-127
constexpr int F_SP = F_P + 2 * TILE;       // bf16 S~_prev: [64 d][64] then [64 d][z, 0...]
constexpr int F_BYTES = F_SP + 2 * 8192;
constexpr int F_SMEM = F_BYTES + 1024;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void fail(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// phi applied in place to a swizzled [128][64] bf16 tile by the 128 compute
// threads (elementwise, so the swizzle does not matter).  Rows at or past
// `valid` are zeroed: a zero phi(K) row adds nothing to any sum.
__device__ __forceinline__ void phi_tile(uint8_t* tile, int valid, int t) {
  for (int v = t; v < TILE / 16; v += 128) {
    uint4* ptr = reinterpret_cast<uint4*>(tile + v * 16);
    uint4 u = *ptr;
    if ((v >> 3) >= valid) {
      u = make_uint4(0u, 0u, 0u, 0u);
    } else {
      uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
        const float plo = lo > 0.f ? lo + 1.f : __expf(lo);
        const float phi_ = hi > 0.f ? hi + 1.f : __expf(hi);
        __nv_bfloat162 b = __floats2bfloat162_rn(plo, phi_);
        w[i] = *reinterpret_cast<uint32_t*>(&b);
      }
      u = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *ptr = u;
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Writes 8 consecutive values (columns 8c .. 8c+7) of row r of a swizzled
// [rows][64] bf16 tile.
__device__ __forceinline__ void st_row_chunk(uint8_t* tile, int r, int c, const float* x) {
  const uint32_t off = static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(c) ^ (r & 7u)) << 4);
  *reinterpret_cast<uint4*>(tile + off) =
      make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                 pack_bf16(x[6], x[7]));
}

// Loads the 80 fp32 columns of this thread's TMEM lane starting at `taddr`.
__device__ __forceinline__ void tmem_ld80(uint32_t taddr, float* v) {
  tmem_ld16(taddr + 0, v + 0);
  tmem_ld16(taddr + 16, v + 16);
  tmem_ld16(taddr + 32, v + 32);
  tmem_ld16(taddr + 48, v + 48);
  tmem_ld16(taddr + 64, v + 64);
  tmem_ld_wait();
}

// Forward kernel.  MODE 0: per-segment partial state dS~ = sum phi(K) V~^T
// written to ws[bh][p] ([64][80] fp32; the last segment is skipped).
// MODE 1: the causal forward, starting from the exclusive prefix in ws[bh][p].
template <int MODE>
__global__ void __launch_bounds__(NTHR, 1)
    k_tc_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, bf16* __restrict__ out,
             float* __restrict__ den, float* __restrict__ ws, int N, int nseg, int seg_len,
             int* err) {
  const int p = blockIdx.x, bh = blockIdx.y;
  if (MODE == 0 && p == nseg - 1) return;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  __shared__ uint64_t bar_full[NST], bar_empty[NST], bar_phi[NST];
  __shared__ uint64_t bar_a, bar_p, bar_sp, bar_o, bar_s;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p * seg_len;
  const int ne = min(N, nb + seg_len);
  const int nch = (ne - nb + TC_C - 1) / TC_C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
      mbar_init(&bar_phi[s], 128);
    }
    mbar_init(&bar_a, 1);
    mbar_init(&bar_p, 128);
    mbar_init(&bar_sp, 128);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_s, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    if (MODE == 1) prefetch_tensormap(&tmQ);
  }
  if (warp == 1) tmem_alloc(&tmem_base, 512);
  if (warp >= 2) {  // the constant ones tile: column 0 = 1, the rest 0
    const int t = threadIdx.x - 64;
    for (int v = t; v < TILE / 16; v += 128) {
      const int r = v >> 3, c = (v & 7) ^ (r & 7);  // logical 16-byte chunk of this vector
      *reinterpret_cast<uint4*>(sm + F_ONES + v * 16) =
          c == 0 ? make_uint4(0x3f80u, 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (MODE == 1)
      for (int v = t; v < 8192 / 16; v += 128)
        *reinterpret_cast<uint4*>(sm + F_SP + 8192 + v * 16) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_base;
  const uint32_t TA = tm, TO = tm + 128, TS = tm + 256;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int s = c % NST;
        if (c >= NST && !mbar_wait(&bar_empty[s], ((c / NST) - 1) & 1, WAIT_NS)) {
          fail(err, 11);
          break;
        }
        uint8_t* st = sm + s * F_STAGE;
        mbar_arrive_expect_tx(&bar_full[s], (MODE == 1 ? 3 : 2) * TILE);
        const int n0 = nb + c * TC_C;
        if (MODE == 1) tma_load_3d(st, &tmQ, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + TILE, &tmK, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + 2 * TILE, &tmV, &bar_full[s], 0, n0, bh);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_A = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_O = idesc_bf16(128, TC_MA, false, true);
      constexpr uint32_t ID_S = idesc_bf16(64, TC_MA, true, true);
      const uint32_t ones = smem_u32(sm + F_ONES);
      const uint32_t pb = smem_u32(sm + F_P), spb = smem_u32(sm + F_SP);
      for (int c = 0; c < nch; ++c) {
        const int s = c % NST;
        const uint32_t q = smem_u32(sm + s * F_STAGE), k = q + TILE, v = q + 2 * TILE;
        if (!mbar_wait(&bar_phi[s], (c / NST) & 1, WAIT_NS)) {
          fail(err, 12);
          break;
        }
        tc_fence_after();
        if (MODE == 1) {
          for (int kk = 0; kk < 4; ++kk)  // A = phi(Q) phi(K)^T
            mma_bf16(TA, sdesc(q + 32 * kk, 16, 1024), sdesc(k + 32 * kk, 16, 1024), ID_A, kk > 0);
          mma_commit(&bar_a);
          if (!mbar_wait(&bar_p, c & 1, WAIT_NS) || !mbar_wait(&bar_sp, c & 1, WAIT_NS)) {
            fail(err, 13);
            break;
          }
          tc_fence_after();
          for (int kk = 0; kk < 8; ++kk)  // O~ = P V~
            mma_bf16(TO, sdesc(pb + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024),
                     sdesc(v + kk * 2048, ones - v, 1024), ID_O, kk > 0);
          for (int kk = 0; kk < 4; ++kk)  // O~ += phi(Q) S~_prev
            mma_bf16(TO, sdesc(q + 32 * kk, 16, 1024), sdesc(spb + kk * 2048, 8192, 1024), ID_O, 1);
          mma_commit(&bar_o);
        }
        for (int kk = 0; kk < 8; ++kk)  // S~ += phi(K)^T V~
          mma_bf16(TS, sdesc(k + kk * 2048, 16, 1024), sdesc(v + kk * 2048, ones - v, 1024), ID_S, 1);
        if (MODE == 1 || c == nch - 1) mma_commit(&bar_s);  // MODE 0: only the final state
        mma_commit(&bar_empty[s]);
      }
    }
  } else {
    // -------------------------------------------------------- compute warps
    const int t = threadIdx.x - 64;        // 0..127
    const int qd = warp & 3;               // TMEM lane quarter of this warp
    const int row = 32 * qd + lane;        // chunk row == TMEM lane
    const uint32_t lq = static_cast<uint32_t>(32 * qd) << 16;
    const bool has_s = lane < 16;          // M=64 accumulators: row 16*qd + lane in lane 32*qd + lane
    const int srow = 16 * qd + lane;
    float sv[TC_MA];
    {  // initial state: the exclusive prefix (MODE 1, p > 0) or zero
      const float* pre = ws + ((static_cast<long>(bh) * nseg + p) * 64 + (has_s ? srow : 0)) * TC_MA;
      for (int j = 0; j < TC_MA; ++j) sv[j] = (MODE == 1 && p > 0 && has_s) ? pre[j] : 0.f;
      for (int j = 0; j < TC_MA; j += 16) tmem_st16(TS + lq + j, sv + j);
      tmem_st_wait();
      if (MODE == 1 && has_s) {
        for (int c8 = 0; c8 < 8; ++c8) st_row_chunk(sm + F_SP, srow, c8, sv + 8 * c8);
        float z8[8] = {sv[64], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        st_row_chunk(sm + F_SP + 8192, srow, 0, z8);
      }
      fence_proxy_async();
      tc_fence_before();
    }
    bool ok = true;
    // phi on chunk 0
    if (!mbar_wait(&bar_full[0], 0, WAIT_NS)) {
      fail(err, 14);
      ok = false;
    }
    if (ok) {
      const int valid = min(TC_C, ne - nb);
      if (MODE == 1) phi_tile(sm + 0, valid, t);
      phi_tile(sm + TILE, valid, t);
      fence_proxy_async();
      mbar_arrive(&bar_phi[0]);
      if (MODE == 1) mbar_arrive(&bar_sp);
    }
    for (int c = 0; ok && c < nch; ++c) {
      const int n0 = nb + c * TC_C;
      if (MODE == 1) {
        // P = bf16(mask(A)): row `row` keeps keys j <= row
        if (!mbar_wait(&bar_a, c & 1, WAIT_NS)) {
          fail(err, 15);
          break;
        }
        tc_fence_after();
        for (int g = 0; g < 4; ++g) {  // 32 keys per group
          float a[32];
          tmem_ld16(TA + lq + 32 * g, a);
          tmem_ld16(TA + lq + 32 * g + 16, a + 16);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * g + i > row) a[i] = 0.f;
          uint8_t* half = sm + F_P + (g >> 1) * TILE;
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) st_row_chunk(half, row, (g & 1) * 4 + c8, a + 8 * c8);
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_p);
      }
      // phi on the next chunk while the tensor cores work on this one
      if (c + 1 < nch) {
        const int s1 = (c + 1) % NST;
        if (!mbar_wait(&bar_full[s1], ((c + 1) / NST) & 1, WAIT_NS)) {
          fail(err, 16);
          break;
        }
        const int valid = min(TC_C, ne - (n0 + TC_C));
        if (MODE == 1) phi_tile(sm + s1 * F_STAGE, valid, t);
        phi_tile(sm + s1 * F_STAGE + TILE, valid, t);
        fence_proxy_async();
        mbar_arrive(&bar_phi[s1]);
      }
      if (MODE == 1) {
        // out = O~[:, :64] / O~[:, 64]
        if (!mbar_wait(&bar_o, c & 1, WAIT_NS)) {
          fail(err, 17);
          break;
        }
        tc_fence_after();
        float o[TC_MA];
        tmem_ld80(TO + lq, o);
        const int n = n0 + row;
        if (n < ne) {
          const float d = o[64];
          const float inv = 1.f / d;
          uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<long>(bh) * N + n) * 64);
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8)
            dst[c8] = make_uint4(pack_bf16(o[8 * c8] * inv, o[8 * c8 + 1] * inv),
                                 pack_bf16(o[8 * c8 + 2] * inv, o[8 * c8 + 3] * inv),
                                 pack_bf16(o[8 * c8 + 4] * inv, o[8 * c8 + 5] * inv),
                                 pack_bf16(o[8 * c8 + 6] * inv, o[8 * c8 + 7] * inv));
          if (den != nullptr) den[static_cast<long>(bh) * N + n] = d;
        }
        // next chunk's S~_prev in bf16
        if (c + 1 < nch) {
          if (!mbar_wait(&bar_s, c & 1, WAIT_NS)) {
            fail(err, 18);
            break;
          }
          tc_fence_after();
          tmem_ld80(TS + lq, sv);
          if (has_s) {
            for (int c8 = 0; c8 < 8; ++c8) st_row_chunk(sm + F_SP, srow, c8, sv + 8 * c8);
            float z8[8] = {sv[64], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            st_row_chunk(sm + F_SP + 8192, srow, 0, z8);
          }
          fence_proxy_async();
          tc_fence_before();
          mbar_arrive(&bar_sp);
        }
      }
    }
    if (MODE == 0 && ok) {
      // the segment's partial state: wait for the last S~ update
      const bool done = mbar_wait(&bar_s, 0, WAIT_NS);
      if (!done) fail(err, 19);
      if (done) {
        tc_fence_after();
        tmem_ld80(TS + lq, sv);
        if (has_s) {
          float* dst = ws + ((static_cast<long>(bh) * nseg + p) * 64 + srow) * TC_MA;
          for (int j = 0; j < TC_MA; ++j) dst[j] = sv[j];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------------ backward
//
// Quotient-rule terms per row i: gt_i = dout_i / den_i and
// gam_i = -(gt_i . out_i); augmented gt~_i = [gt_i | gam_i | 0 ...] (80 wide).
// With V~ = [V | 1]:
//   dA = mask(gt~ V~^T)                                       (dA_ij = gt_i . V_j + gam_i)
//   grad_phiQ = dP phi(K) + gt~ S~_prev^T                     (eq. 13 + denominator)
//   grad_phiK = dP^T phi(Q) + V~ R~_next^T                    (eq. 14 + denominator)
//   dv        = P^T gt + phi(K) R_next                        (eq. 15)
//   S~ += phi(K)^T V~ (forward),  R~ += phi(Q)^T gt~ (reverse) with R~ = [R | r]
// P = bf16(mask(A)), dP = bf16(mask(dA)).  MODE 0 writes each segment's
// partial S~ and R~; MODE 1 runs role 0 (dq, forward walk) or role 1 (dk and dv,
// reverse walk) by blockIdx.z.

constexpr int B_STAGE = 3 * TILE;          // Q, K, V
constexpr int B_ONES = NST * B_STAGE;
constexpr int B_GA = B_ONES + TILE;        // gt (64 cols) then [gam, 0, ...]
constexpr int B_P = B_GA + 2 * TILE;       // P  [i][j]: j 0-63 then 64-127
constexpr int B_DP = B_P + 2 * TILE;       // dP [i][j]
constexpr int B_RP = B_DP + 2 * TILE;      // bf16 carried state [64 d][64] then [64 d][col 64, 0...]
constexpr int B_BYTES = B_RP + 2 * 8192;
constexpr int B_SMEM = B_BYTES + 1024;
static_assert(B_SMEM + 256 <= 232448, "backward shared memory over the per-CTA limit");

// Builds this thread's row of gt~ (bf16, swizzled) from global dout, out, den.
__device__ __forceinline__ void build_gt_row(uint8_t* ga, const bf16* g, const bf16* o,
                                             const float* den, long rowbase, int row, bool valid) {
  float gt[64];
  float gam = 0.f;
  if (valid) {
    const float inv = 1.f / den[rowbase];
    const uint4* gp = reinterpret_cast<const uint4*>(g + rowbase * 64);
    const uint4* op = reinterpret_cast<const uint4*>(o + rowbase * 64);
    float acc = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint4 gu = gp[c8], ou = op[c8];
      float gf[8], of[8];
      Vec16<bf16>::unpack(gu, gf);
      Vec16<bf16>::unpack(ou, of);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        gt[8 * c8 + i] = gf[i] * inv;
        acc = fmaf(gt[8 * c8 + i], of[i], acc);
      }
    }
    gam = -acc;
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) gt[i] = 0.f;
  }
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) st_row_chunk(ga, row, c8, gt + 8 * c8);
  float g8[8] = {gam, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  st_row_chunk(ga + TILE, row, 0, g8);
}

// Reads 128 masked columns (j <= row) of an accumulator and stores them as
// bf16 row `row` of a [128][128] K-major operand (two 64-column tiles).
__device__ __forceinline__ void mask_to_smem(uint32_t taddr, uint8_t* dst, int row) {
  for (int g = 0; g < 4; ++g) {
    float a[32];
    tmem_ld16(taddr + 32 * g, a);
    tmem_ld16(taddr + 32 * g + 16, a + 16);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (32 * g + i > row) a[i] = 0.f;
    uint8_t* half = dst + (g >> 1) * TILE;
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) st_row_chunk(half, row, (g & 1) * 4 + c8, a + 8 * c8);
  }
}

// Stores an fp32 [64 d][80] state held in TMEM rows (M=64 layout) as the bf16
// operand tiles at `rp` (columns 0-63, then column 64 in the second tile).
__device__ __forceinline__ void state_to_smem(uint8_t* rp, const float* sv, int srow, bool has) {
  if (has) {
    for (int c8 = 0; c8 < 8; ++c8) st_row_chunk(rp, srow, c8, sv + 8 * c8);
    float z8[8] = {sv[64], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    st_row_chunk(rp + 8192, srow, 0, z8);
  }
}

// Writes one 64-wide bf16 output row: val[c] * (scale ? phi'(x[c]) : 1).
__device__ __forceinline__ void store_row(bf16* dst, const float* val, const bf16* raw) {
  uint4* d = reinterpret_cast<uint4*>(dst);
  const uint4* r = reinterpret_cast<const uint4*>(raw);
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    float f[8];
    if (raw != nullptr) {
      float x[8];
      Vec16<bf16>::unpack(r[c8], x);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = val[8 * c8 + i] * (x[i] > 0.f ? 1.f : __expf(x[i]));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = val[8 * c8 + i];
    }
    d[c8] = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                       pack_bf16(f[6], f[7]));
  }
}

template <int MODE>
__global__ void __launch_bounds__(NTHR, 1)
    k_tc_bwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const bf16* __restrict__ q,
             const bf16* __restrict__ k, const bf16* __restrict__ o,
             const float* __restrict__ den, const bf16* __restrict__ g, bf16* __restrict__ dq,
             bf16* __restrict__ dk, bf16* __restrict__ dv, float* __restrict__ ws, int N,
             int nseg, int seg_len, int* err) {
  const int p = blockIdx.x, bh = blockIdx.y;
  const int role = MODE == 0 ? 2 : blockIdx.z;  // 0: dq, 1: dk/dv, 2: partial states
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  __shared__ uint64_t bar_full[NST], bar_empty[NST];
  __shared__ uint64_t bar_in, bar_a, bar_p, bar_rp, bar_o, bar_s;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p * seg_len;
  const int ne = min(N, nb + seg_len);
  const int nch = (ne - nb + TC_C - 1) / TC_C;
  const bool need_q = role != 0;  // phi(Q) tiles: roles 1 and 2

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_in, 128);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_p, 128);
    mbar_init(&bar_rp, 128);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_s, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    if (need_q) prefetch_tensormap(&tmQ);
  }
  if (warp == 1) tmem_alloc(&tmem_base, 512);
  if (warp >= 2) {
    const int t = threadIdx.x - 64;
    for (int v = t; v < TILE / 16; v += 128) {
      const int r = v >> 3, c = (v & 7) ^ (r & 7);
      *reinterpret_cast<uint4*>(sm + B_ONES + v * 16) =
          c == 0 ? make_uint4(0x3f80u, 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(sm + B_GA + TILE + v * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int v = t; v < 8192 / 16; v += 128)
      *reinterpret_cast<uint4*>(sm + B_RP + 8192 + v * 16) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_base;
  const uint32_t TA = tm, TDA = tm + 128, TG1 = tm + 256, TG2 = tm + 320, TST = tm + 384;
  // MODE 0 keeps S~ in TG1..(80 cols at 256) and R~ in TST (384)

  // chunk order: role 1 walks its segment backwards
  auto chunk_at = [&](int c) { return role == 1 ? nch - 1 - c : c; };

  if (warp == 0) {
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int s = c % NST;
        if (c >= NST && !mbar_wait(&bar_empty[s], ((c / NST) - 1) & 1, WAIT_NS)) {
          fail(err, 21);
          break;
        }
        uint8_t* st = sm + s * B_STAGE;
        mbar_arrive_expect_tx(&bar_full[s], (need_q ? 3 : 2) * TILE);
        const int n0 = nb + chunk_at(c) * TC_C;
        if (need_q) tma_load_3d(st, &tmQ, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + TILE, &tmK, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + 2 * TILE, &tmV, &bar_full[s], 0, n0, bh);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_A = idesc_bf16(128, 128, false, false);   // A, dA
      constexpr uint32_t ID_G = idesc_bf16(128, 64, false, false);    // K-major A and B
      constexpr uint32_t ID_GMN = idesc_bf16(128, 64, false, true);   // K-major A, MN-major B
      constexpr uint32_t ID_GTT = idesc_bf16(128, 64, true, true);    // MN-major A and B
      constexpr uint32_t ID_ST = idesc_bf16(64, TC_MA, true, true);   // state updates
      const uint32_t ones = smem_u32(sm + B_ONES), ga = smem_u32(sm + B_GA);
      const uint32_t pp = smem_u32(sm + B_P), dp = smem_u32(sm + B_DP), rp = smem_u32(sm + B_RP);
      for (int c = 0; c < nch; ++c) {
        const int s = c % NST;
        const uint32_t qs = smem_u32(sm + s * B_STAGE), ks = qs + TILE, vs = qs + 2 * TILE;
        if (!mbar_wait(&bar_in, c & 1, WAIT_NS)) {
          fail(err, 22);
          break;
        }
        tc_fence_after();
        if (role == 2) {
          for (int kk = 0; kk < 8; ++kk)  // S~ += phi(K)^T V~
            mma_bf16(TG1, sdesc(ks + kk * 2048, 16, 1024), sdesc(vs + kk * 2048, ones - vs, 1024),
                     ID_ST, 1);
          for (int kk = 0; kk < 8; ++kk)  // R~ += phi(Q)^T gt~
            mma_bf16(TST, sdesc(qs + kk * 2048, 16, 1024), sdesc(ga + kk * 2048, TILE, 1024),
                     ID_ST, 1);
          mma_commit(&bar_s);
          mma_commit(&bar_empty[s]);
          continue;
        }
        // dA = gt~ V~^T: K = 80 (4 steps in gt / V, one in [gam] / ones)
        for (int kk = 0; kk < 5; ++kk) {
          const uint32_t a = kk < 4 ? ga + 32 * kk : ga + TILE;
          const uint32_t b = kk < 4 ? vs + 32 * kk : ones;
          mma_bf16(TDA, sdesc(a, 16, 1024), sdesc(b, 16, 1024), ID_A, kk > 0);
        }
        if (role == 1)  // A = phi(Q) phi(K)^T
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(TA, sdesc(qs + 32 * kk, 16, 1024), sdesc(ks + 32 * kk, 16, 1024), ID_A, kk > 0);
        mma_commit(&bar_a);
        if (!mbar_wait(&bar_p, c & 1, WAIT_NS) || !mbar_wait(&bar_rp, c & 1, WAIT_NS)) {
          fail(err, 23);
          break;
        }
        tc_fence_after();
        if (role == 0) {
          // grad_phiQ = dP phi(K) + gt~ S~_prev^T
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(TG1, sdesc(dp + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024),
                     sdesc(ks + kk * 2048, 16, 1024), ID_GMN, kk > 0);
          for (int kk = 0; kk < 5; ++kk) {
            const uint32_t a = kk < 4 ? ga + 32 * kk : ga + TILE;
            const uint32_t b = kk < 4 ? rp + 32 * kk : rp + 8192;
            mma_bf16(TG1, sdesc(a, 16, 1024), sdesc(b, 16, 1024), ID_G, 1);
          }
          mma_commit(&bar_o);
          for (int kk = 0; kk < 8; ++kk)  // S~ += phi(K)^T V~
            mma_bf16(TST, sdesc(ks + kk * 2048, 16, 1024), sdesc(vs + kk * 2048, ones - vs, 1024),
                     ID_ST, 1);
        } else {
          // grad_phiK = dP^T phi(Q) + V~ R~^T
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(TG1, sdesc(dp + kk * 2048, TILE, 1024), sdesc(qs + kk * 2048, 16, 1024),
                     ID_GTT, kk > 0);
          for (int kk = 0; kk < 5; ++kk) {
            const uint32_t a = kk < 4 ? vs + 32 * kk : ones;
            const uint32_t b = kk < 4 ? rp + 32 * kk : rp + 8192;
            mma_bf16(TG1, sdesc(a, 16, 1024), sdesc(b, 16, 1024), ID_G, 1);
          }
          // dv = P^T gt + phi(K) R
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(TG2, sdesc(pp + kk * 2048, TILE, 1024), sdesc(ga + kk * 2048, 16, 1024),
                     ID_GTT, kk > 0);
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(TG2, sdesc(ks + 32 * kk, 16, 1024), sdesc(rp + kk * 2048, 16, 1024), ID_GMN, 1);
          mma_commit(&bar_o);
          for (int kk = 0; kk < 8; ++kk)  // R~ += phi(Q)^T gt~
            mma_bf16(TST, sdesc(qs + kk * 2048, 16, 1024), sdesc(ga + kk * 2048, TILE, 1024),
                     ID_ST, 1);
        }
        mma_commit(&bar_s);
        mma_commit(&bar_empty[s]);
      }
    }
  } else {
    const int t = threadIdx.x - 64;
    const int qd = warp & 3;
    const int row = 32 * qd + lane;
    const uint32_t lq = static_cast<uint32_t>(32 * qd) << 16;
    const bool has_s = lane < 16;
    const int srow = 16 * qd + lane;
    float sv[TC_MA];
    {  // initial carried state: role 0 the exclusive prefix S~, role 1 the exclusive suffix R~
      const bool has_pre = (role == 0 && p > 0) || (role == 1 && p < nseg - 1);
      const float* pre = ws + (static_cast<long>(bh) * nseg + p) * 2 * 64 * TC_MA +
                         (role == 1 ? 64 * TC_MA : 0) + (has_s ? srow : 0) * TC_MA;
      for (int j = 0; j < TC_MA; ++j) sv[j] = (has_pre && has_s) ? pre[j] : 0.f;
      if (role == 2) {
        for (int j = 0; j < TC_MA; j += 16) tmem_st16(TG1 + lq + j, sv + j);
      }
      for (int j = 0; j < TC_MA; j += 16) tmem_st16(TST + lq + j, sv + j);
      tmem_st_wait();
      if (role != 2) state_to_smem(sm + B_RP, sv, srow, has_s);
      fence_proxy_async();
      tc_fence_before();
      if (role != 2) mbar_arrive(&bar_rp);
    }
    for (int c = 0; c < nch; ++c) {
      const int s = c % NST;
      const int n0 = nb + chunk_at(c) * TC_C;
      const int valid = min(TC_C, ne - n0);
      uint8_t* st = sm + s * B_STAGE;
      if (c > 0 && role == 2) {  // gt~ buffer is free once the previous R~ update finished
        if (!mbar_wait(&bar_s, (c - 1) & 1, WAIT_NS)) {
          fail(err, 24);
          break;
        }
        tc_fence_after();
      }
      build_gt_row(sm + B_GA, g, o, den, static_cast<long>(bh) * N + n0 + row, row, row < valid);
      if (!mbar_wait(&bar_full[s], (c / NST) & 1, WAIT_NS)) {
        fail(err, 25);
        break;
      }
      if (need_q) phi_tile(st, valid, t);
      phi_tile(st + TILE, valid, t);
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_in);
      if (role == 2) continue;

      if (!mbar_wait(&bar_a, c & 1, WAIT_NS)) {
        fail(err, 26);
        break;
      }
      tc_fence_after();
      mask_to_smem(TDA + lq, sm + B_DP, row);
      if (role == 1) mask_to_smem(TA + lq, sm + B_P, row);
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_p);

      if (!mbar_wait(&bar_o, c & 1, WAIT_NS)) {
        fail(err, 27);
        break;
      }
      tc_fence_after();
      {
        float gv[64];
        tmem_ld16(TG1 + lq, gv);
        tmem_ld16(TG1 + lq + 16, gv + 16);
        tmem_ld16(TG1 + lq + 32, gv + 32);
        tmem_ld16(TG1 + lq + 48, gv + 48);
        tmem_ld_wait();
        const long rb = (static_cast<long>(bh) * N + n0 + row) * 64;
        if (row < valid) store_row((role == 0 ? dq : dk) + rb, gv, (role == 0 ? q : k) + rb);
        if (role == 1) {
          tmem_ld16(TG2 + lq, gv);
          tmem_ld16(TG2 + lq + 16, gv + 16);
          tmem_ld16(TG2 + lq + 32, gv + 32);
          tmem_ld16(TG2 + lq + 48, gv + 48);
          tmem_ld_wait();
          if (row < valid) store_row(dv + rb, gv, nullptr);
        }
      }
      if (!mbar_wait(&bar_s, c & 1, WAIT_NS)) {
        fail(err, 28);
        break;
      }
      tc_fence_after();
      if (c + 1 < nch) {
        tmem_ld80(TST + lq, sv);
        state_to_smem(sm + B_RP, sv, srow, has_s);
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_rp);
      }
    }
    if (role == 2) {
      if (mbar_wait(&bar_s, (nch - 1) & 1, WAIT_NS)) {
        tc_fence_after();
        float* rec = ws + (static_cast<long>(bh) * nseg + p) * 2 * 64 * TC_MA;
        tmem_ld80(TG1 + lq, sv);
        if (has_s)
          for (int j = 0; j < TC_MA; ++j) rec[srow * TC_MA + j] = sv[j];
        tmem_ld80(TST + lq, sv);
        if (has_s)
          for (int j = 0; j < TC_MA; ++j) rec[64 * TC_MA + srow * TC_MA + j] = sv[j];
      } else {
        fail(err, 29);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// [BH][N][64] bf16 viewed as a 3-D tensor, 64 x 128 x 1 boxes, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int BH, int N) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {64 * 2, static_cast<cuuint64_t>(N) * 64 * 2};
  cuuint32_t box[3] = {64, TC_C, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

SegPlan tc_plan(int BH, int N) {
  const int nch = (N + TC_C - 1) / TC_C;
  int want = 152 / BH;  // whole segments per head so that all CTAs fit one wave
  if (want < 1) want = 1;
  if (want > nch) want = nch;
  const int per = (nch + want - 1) / want;
  SegPlan pl;
  pl.seg_len = per * TC_C;
  pl.nseg = (N + pl.seg_len - 1) / pl.seg_len;
  return pl;
}

bool tc_eligible(const Shape& s) { return s.dtype == 1 && s.D == 64 && s.M == 64; }

size_t causal_fwd_tc_ws_floats(const Shape& s) {
  const SegPlan pl = tc_plan(s.B * s.H, s.N);
  return static_cast<size_t>(s.B) * s.H * pl.nseg * 64 * TC_MA + 4;
}

int causal_fwd_tc_launches(const Shape& s) { return tc_plan(s.B * s.H, s.N).nseg > 1 ? 3 : 1; }

cudaError_t causal_fwd_tc(const void* q, const void* k, const void* v, void* out, float* den,
                          float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const SegPlan pl = tc_plan(BH, s.N);
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, BH, s.N) || !make_map(&mk, k, BH, s.N) || !make_map(&mv, v, BH, s.N))
    return cudaErrorInvalidValue;
  int* err = reinterpret_cast<int*>(ws + static_cast<size_t>(BH) * pl.nseg * 64 * TC_MA);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_tc_fwd<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                F_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_tc_fwd<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                F_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaMemsetAsync(err, 0, sizeof(int), st)) != cudaSuccess) return e;
  if (pl.nseg > 1) {
    k_tc_fwd<0><<<dim3(pl.nseg, BH), NTHR, F_SMEM, st>>>(mq, mk, mv, nullptr, nullptr, ws, s.N,
                                                         pl.nseg, pl.seg_len, err);
    k_seg_scan_ext(ws, BH, pl.nseg, 64 * TC_MA, 64 * TC_MA, 0, 0, st);
  }
  k_tc_fwd<1><<<dim3(pl.nseg, BH), NTHR, F_SMEM, st>>>(mq, mk, mv, static_cast<bf16*>(out), den,
                                                       ws, s.N, pl.nseg, pl.seg_len, err);
  return cudaGetLastError();
}

SegPlan tc_plan_bwd(int BH, int N) { return tc_plan(2 * BH, N); }

size_t causal_bwd_tc_ws_floats(const Shape& s) {
  const SegPlan pl = tc_plan_bwd(s.B * s.H, s.N);
  return static_cast<size_t>(s.B) * s.H * pl.nseg * 2 * 64 * TC_MA + 4;
}

int causal_bwd_tc_launches(const Shape& s) { return tc_plan_bwd(s.B * s.H, s.N).nseg > 1 ? 3 : 1; }

cudaError_t causal_bwd_tc(const void* q, const void* k, const void* v, const void* out,
                          const float* den, const void* dout, void* dq, void* dk, void* dv,
                          float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const SegPlan pl = tc_plan_bwd(BH, s.N);
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, BH, s.N) || !make_map(&mk, k, BH, s.N) || !make_map(&mv, v, BH, s.N))
    return cudaErrorInvalidValue;
  const int rec = 2 * 64 * TC_MA;
  int* err = reinterpret_cast<int*>(ws + static_cast<size_t>(BH) * pl.nseg * rec);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_tc_bwd<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                B_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_tc_bwd<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                B_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaMemsetAsync(err, 0, sizeof(int), st)) != cudaSuccess) return e;
  const bf16 *qb = static_cast<const bf16*>(q), *kb = static_cast<const bf16*>(k);
  const bf16 *ob = static_cast<const bf16*>(out), *gb = static_cast<const bf16*>(dout);
  if (pl.nseg > 1) {
    k_tc_bwd<0><<<dim3(pl.nseg, BH, 1), NTHR, B_SMEM, st>>>(mq, mk, mv, qb, kb, ob, den, gb,
                                                           nullptr, nullptr, nullptr, ws, s.N,
                                                           pl.nseg, pl.seg_len, err);
    k_seg_scan_ext(ws, BH, pl.nseg, rec, 64 * TC_MA, 64 * TC_MA, 64 * TC_MA, st);
  }
  k_tc_bwd<1><<<dim3(pl.nseg, BH, 2), NTHR, B_SMEM, st>>>(
      mq, mk, mv, qb, kb, ob, den, gb, static_cast<bf16*>(dq), static_cast<bf16*>(dk),
      static_cast<bf16*>(dv), ws, s.N, pl.nseg, pl.seg_len, err);
  return cudaGetLastError();
}

}  // namespace la
