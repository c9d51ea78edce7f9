// Causal linear attention on the 5th-generation tensor cores (tcgen05), for
// bf16 inputs with D = M = 64 and fp32 accumulation in tensor memory.
//
// Method: "Transformers are RNNs" (part 2/3), §3.3 eq. 9-12 (forward) and
// §3.3.1 eq. 13-15 (cumulative-sum backward with the denominator terms).
//
// GB300 design (not the pages'): each (b, h) sequence is cut into segments of
// whole 128-token chunks, one CTA per segment (one CTA per SM).  Inside a CTA
// one warp streams raw Q/K/V chunks with TMA into a three-stage shared-memory
// ring (128-byte swizzle), the compute warps apply phi in place, and one
// thread issues the tcgen05 MMAs whose fp32 accumulators live in tensor
// memory.  The value matrix is augmented with a column of ones, V~ = [V | 1],
// so one accumulator carries both the state and the normaliser,
// S~ = [S | z] = sum phi(K_j) V~_j^T, and every product that yields a
// numerator yields its denominator in column 64:
//   A    = phi(Q) phi(K)^T                        (128 x 128, K = 64)
//   P    = bf16(mask(A))                           (compute warps, kept in TMEM)
//   O~   = P V~ + phi(Q) bf16(S~_prev)            (128 x 80)  -> out = O~[:, :64] / O~[:, 64]
//   S~  += phi(K)^T V~                             (64 x 80, carried across chunks)
// Segment prefixes are sums of the partial states of a first pass (same
// kernel, MODE 0), added up by each CTA of the second pass.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tc_chunk.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcc;

constexpr int TC_MA = 80;                  // augmented value width [V | 1 | 0 ...]

// shared-memory map of the forward kernel (offsets from a 1024-aligned base)
constexpr int FNST = 3;                    // TMA ring stages of the forward
constexpr int F_STAGE = 3 * TILE;          // Q, K, V
constexpr int F_ONES = FNST * F_STAGE;     // [128][64], column 0 = 1
constexpr int F_SP = F_ONES + TILE;        // bf16 S~_prev: [64 d][64] then [64 d][z, 0...]
constexpr int F_OUT = F_SP + 2 * 8192;     // two output staging tiles (by chunk parity)
constexpr int F_BYTES = F_OUT + 2 * TILE;
constexpr int F_SMEM = F_BYTES + 1024;

// Forward kernel.  MODE 0: per-segment partial state dS~ = sum phi(K) V~^T
// written to ws[bh][p] ([64][80] fp32; the last segment is skipped).
// MODE 1: the causal forward, starting from the sum of ws[bh][0 .. p-1].
template <int MODE>
__global__ void __launch_bounds__(NTHR, 1)
    k_tc_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmOut,
             float* __restrict__ den, float* __restrict__ ws, int N, int nseg, int seg_len,
             int* err) {
  const int p = blockIdx.x, bh = blockIdx.y;
  if (MODE == 0 && p == nseg - 1) return;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  __shared__ uint64_t bar_full[FNST], bar_empty[FNST], bar_phi[FNST];
  __shared__ uint64_t bar_a, bar_p, bar_sp, bar_o, bar_s;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p * seg_len;
  const int ne = min(N, nb + seg_len);
  const int nch = (ne - nb + TC_C - 1) / TC_C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < FNST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
      mbar_init(&bar_phi[s], MODE == 1 ? NCOMP / 2 : NCOMP);
    }
    mbar_init(&bar_a, 1);
    mbar_init(&bar_p, NCOMP / 2);
    mbar_init(&bar_sp, NCOMP / 2);
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
    for (int v = t; v < TILE / 16; v += NCOMP) {
      const int r = v >> 3, c = (v & 7) ^ (r & 7);  // logical 16-byte chunk of this vector
      *reinterpret_cast<uint4*>(sm + F_ONES + v * 16) =
          c == 0 ? make_uint4(0x3f80u, 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (MODE == 1)
      for (int v = t; v < 8192 / 16; v += NCOMP)
        *reinterpret_cast<uint4*>(sm + F_SP + 8192 + v * 16) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();  // the previous kernel's outputs are visible from here on
  const uint32_t tm = tmem_base;
  const uint32_t TA = tm, TO = tm + 128, TS = tm + 256, TP = tm + 384;  // TP: bf16 P (A operand)

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int s = c % FNST;
        if (c >= FNST && !mbar_wait(&bar_empty[s], ((c / FNST) - 1) & 1, WAIT_NS)) {
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
      const uint64_t dSP = sdesc(smem_u32(sm + F_SP), 8192, 1024);
      for (int c = 0; c < nch; ++c) {
        const int s = c % FNST;
        const uint32_t q = smem_u32(sm + s * F_STAGE), k = q + TILE, v = q + 2 * TILE;
        const uint64_t dQ = sdesc(q, 16, 1024), dK = sdesc(k, 16, 1024);
        const uint64_t dVt = sdesc(v, ones - v, 1024);  // [V | ones] as an MN-major operand
        if (!mbar_wait(&bar_phi[s], (c / FNST) & 1, WAIT_NS)) {
          fail(err, 12);
          break;
        }
        tc_fence_after();
        if (MODE == 1) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // A = phi(Q) phi(K)^T
            mma_bf16(TA, dadd(dQ, 32 * kk), dadd(dK, 32 * kk), ID_A, kk > 0);
          mma_commit(&bar_a);
          if (!mbar_wait(&bar_p, c & 1, WAIT_NS) || !mbar_wait(&bar_sp, c & 1, WAIT_NS)) {
            fail(err, 13);
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // O~ = P V~, P read from tensor memory
            mma_bf16_ts(TO, TP + 8 * kk, dadd(dVt, kk * 2048), ID_O, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // O~ += phi(Q) S~_prev
            mma_bf16(TO, dadd(dQ, 32 * kk), dadd(dSP, kk * 2048), ID_O, 1);
          mma_commit(&bar_o);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // S~ += phi(K)^T V~
          mma_bf16(TS, dadd(dK, kk * 2048), dadd(dVt, kk * 2048), ID_S, 1);
        if (MODE == 1 || c == nch - 1) mma_commit(&bar_s);  // MODE 0: only the final state
        mma_commit(&bar_empty[s]);
      }
    }
  } else {
    // -------------------------------------------------------- compute warps
    // MODE 1: warpgroups 0-1 are consumers (P, read-out, carried state; each
    // covers all 128 rows and half of the columns), warpgroups 2-3 apply phi
    // to the chunks ahead on the TMA ring.  MODE 0: every warpgroup applies phi.
    const int t = threadIdx.x - 64;        // 0 .. NCOMP-1
    const int wg = t >> 7;
    const int qd = warp & 3;               // TMEM lane quarter of this warp
    const int row = 32 * qd + lane;        // chunk row == TMEM lane
    const uint32_t lq = static_cast<uint32_t>(32 * qd) << 16;
    const bool has_s = lane < 16;          // M=64 accumulators: row 16*qd + lane in lane 32*qd + lane
    const int srow = 16 * qd + lane;
    const bool transform = MODE == 0 || wg >= 2;
    if (wg == 0) {  // initial state: the sum of the earlier segments' partial
                    // states written by MODE 0 (MODE 1), zero otherwise
      float sv[TC_MA];
      for (int j = 0; j < TC_MA; ++j) sv[j] = 0.f;
      if (MODE == 1 && has_s)
        for (int pp = 0; pp < p; ++pp) {
          const float4* rec = reinterpret_cast<const float4*>(
              ws + ((static_cast<long>(bh) * nseg + pp) * 64 + srow) * TC_MA);
#pragma unroll
          for (int j = 0; j < TC_MA / 4; ++j) {
            const float4 x = rec[j];
            sv[4 * j] += x.x;
            sv[4 * j + 1] += x.y;
            sv[4 * j + 2] += x.z;
            sv[4 * j + 3] += x.w;
          }
        }
      for (int j = 0; j < TC_MA; j += 16) tmem_st16(TS + lq + j, sv + j);
      tmem_st_wait();
      if (MODE == 1 && has_s) {
        tile_put_cols<64>(sm + F_SP, srow, 0, sv);
        float z8[8] = {sv[64], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        st_row_chunk(sm + F_SP + 8192, srow, 0, z8);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    if (transform) {
      // ------------------------------------------------ phi on every chunk
      const int tt = MODE == 1 ? t - NCOMP / 2 : t;
      const int nt = MODE == 1 ? NCOMP / 2 : NCOMP;
      for (int c = 0; c < nch; ++c) {
        const int s = c % FNST;
        if (!mbar_wait(&bar_full[s], (c / FNST) & 1, WAIT_NS)) {
          fail(err, 14);
          break;
        }
        const int valid = min(TC_C, ne - (nb + c * TC_C));
        if (MODE == 1) phi_tile(sm + s * F_STAGE, valid, tt, nt);
        phi_tile(sm + s * F_STAGE + TILE, valid, tt, nt);
        fence_proxy_async();
        mbar_arrive(&bar_phi[s]);
      }
    } else {
      // ------------------------------------------- consumers (MODE 1 only)
      const int c0 = 32 * wg, k0 = 64 * wg;  // output columns / keys of this warpgroup
      mbar_arrive(&bar_sp);
      for (int c = 0; c < nch; ++c) {
        const int n0 = nb + c * TC_C;
        // P = bf16(mask(A)) for keys k0 .. k0+63, kept in TMEM
        if (!mbar_wait(&bar_a, c & 1, WAIT_NS)) {
          fail(err, 15);
          break;
        }
        tc_fence_after();
        {
          float a[64];
          uint32_t pk[32];
          tmem_ldn<4>(TA + lq + k0, a);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            pk[i] = pack_bf16(k0 + 2 * i <= row ? a[2 * i] : 0.f, k0 + 2 * i + 1 <= row ? a[2 * i + 1] : 0.f);
          tmem_st16u(TP + lq + k0 / 2, pk);
          tmem_st16u(TP + lq + k0 / 2 + 16, pk + 16);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bar_p);
        // out = O~[:, :64] / O~[:, 64], columns c0 .. c0+31
        if (!mbar_wait(&bar_o, c & 1, WAIT_NS)) {
          fail(err, 17);
          break;
        }
        tc_fence_after();
        float o[32], dd[16];
        tmem_ld16(TO + lq + c0, o);
        tmem_ld16(TO + lq + c0 + 16, o + 16);
        tmem_ld16(TO + lq + 64, dd);
        tmem_ld_wait();
        const float d = dd[0];
        const float inv = 1.f / d;
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= inv;
        tile_put_cols<32>(sm + F_OUT + (c & 1) * TILE, row, c0, o);
        if (den != nullptr && wg == 0 && n0 + row < ne) den[static_cast<long>(bh) * N + n0 + row] = d;
        // next chunk's S~_prev in bf16: warpgroup 0 columns 0-47, 1 columns 48-79
        if (c + 1 < nch) {
          if (!mbar_wait(&bar_s, c & 1, WAIT_NS)) {
            fail(err, 18);
            break;
          }
          tc_fence_after();
          float sv[48];
          if (wg == 0) {
            tmem_ldn<3>(TS + lq, sv);
            if (has_s) tile_put_cols<48>(sm + F_SP, srow, 0, sv);
          } else {
            tmem_ldn<2>(TS + lq + 48, sv);
            if (has_s) {
              tile_put_cols<16>(sm + F_SP, srow, 48, sv);
              float z8[8] = {sv[16], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
              st_row_chunk(sm + F_SP + 8192, srow, 0, z8);
            }
          }
          fence_proxy_async();
          tc_fence_before();
          mbar_arrive(&bar_sp);
        }
        fence_proxy_async();
        if (t == 0) bulk_wait_read();  // chunk c-1's store has left the other staging tile
        half_sync();                   // this chunk's output tile is complete
        if (t == 0) {
          tma_store_3d(&tmOut, sm + F_OUT + (c & 1) * TILE, 0, n0, bh);
          bulk_commit();
        }
      }
      if (t == 0) bulk_wait_all();
    }
    if (MODE == 0) {
      // the segment's partial state: wait for the last S~ update
      const bool done = mbar_wait(&bar_s, 0, WAIT_NS);
      if (!done) fail(err, 19);
      if (done) {
        tc_fence_after();
        float sv[16], zz[16];
        float* dst = ws + ((static_cast<long>(bh) * nseg + p) * 64 + srow) * TC_MA;
        tmem_ld16(TS + lq + 16 * wg, sv);
        if (wg == 0) tmem_ld16(TS + lq + 64, zz);
        tmem_ld_wait();
        if (has_s) {
          for (int j = 0; j < 16; ++j) dst[16 * wg + j] = sv[j];
          if (wg == 0)
            for (int j = 0; j < 16; ++j) dst[64 + j] = zz[j];
        }
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

}  // namespace

// [BH][N][64] bf16 viewed as a 3-D tensor, 64 x 128 x 1 boxes, 128-byte swizzle.
bool make_bf16_map(CUtensorMap* m, const void* base, int BH, int N) {
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

int causal_fwd_tc_launches(const Shape& s) { return tc_plan(s.B * s.H, s.N).nseg > 1 ? 2 : 1; }

cudaError_t causal_fwd_tc(const void* q, const void* k, const void* v, void* out, float* den,
                          float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const SegPlan pl = tc_plan(BH, s.N);
  CUtensorMap mq, mk, mv, mo;
  if (!make_bf16_map(&mq, q, BH, s.N) || !make_bf16_map(&mk, k, BH, s.N) ||
      !make_bf16_map(&mv, v, BH, s.N) || !make_bf16_map(&mo, out, BH, s.N))
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
    if ((e = launch_pdl(k_tc_fwd<0>, dim3(pl.nseg, BH), dim3(NTHR), F_SMEM, st, mq, mk, mv, mo,
                        static_cast<float*>(nullptr), ws, s.N, pl.nseg, pl.seg_len, err)) !=
        cudaSuccess)
      return e;
  }
  if ((e = launch_pdl(k_tc_fwd<1>, dim3(pl.nseg, BH), dim3(NTHR), F_SMEM, st, mq, mk, mv, mo, den,
                      ws, s.N, pl.nseg, pl.seg_len, err)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace la
