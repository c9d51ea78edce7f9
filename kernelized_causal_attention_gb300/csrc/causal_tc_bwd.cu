// Backward of causal linear attention on the tcgen05 tensor cores, bf16 with
// D = M = 64 and fp32 accumulation in tensor memory.
//
// Method: "Transformers are RNNs" (part 2/3) §3.3.1 eq. 13-15, the gradients
// of the numerator as cumulative sums, completed with the denominator by the
// quotient rule.  With gt_i = dout_i / den_i and gam_i = -(gt_i . out_i):
//   dA_ij      = gt_i . V_j + gam_i            (j <= i)
//   grad_phiQ  = dP phi(K) + gt S_prev^T + gam z_prev^T          (forward sums)
//   grad_phiK  = dP^T phi(Q) + V R_next^T + r_next                (reverse sums)
//   dv         = P^T gt + phi(K) R_next
//   S += phi(K)^T V, z += sum phi(K);  R += phi(Q)^T gt, r += sum gam phi(Q)
// with P = bf16(mask(phi(Q) phi(K)^T)) and dP = bf16(mask(dA)); then
// dq = grad_phiQ * phi'(Q), dk = grad_phiK * phi'(K).
//
// Two passes over segments of whole 128-token chunks.  MODE 0 (one CTA per
// segment) reads dout, out and den once, writes gt (bf16) and gam to the
// workspace, and the segment's partial S, z, R, r.  MODE 1 runs two roles per
// segment (grid z): role 0 walks forward carrying S, z and writes dq; role 1
// walks backward carrying R, r and writes dk and dv.  Each CTA adds up the
// partial states of the segments before (role 0) or after (role 1) it.  The
// matrix terms run on tcgen05 (operands TMA-fed, 128-byte swizzle); the
// vector terms z, r and the gam corrections run on CUDA cores in fp32.
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tc_chunk.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcc;

constexpr int DM = 64 * 64;
constexpr int REC = 2 * (DM + 64);  // per-segment record [S | z | R | r]

// MODE 0 shared memory: stages of Q, K, V, dout, out; the bf16 gt tile
constexpr int S_STAGE = 5 * TILE;
constexpr int S_GT = NST * S_STAGE;
constexpr int S_SMEM = S_GT + TILE + 1024;
// MODE 1 shared memory: stages of Q, K, V, gt; P; dP; bf16 carried state
constexpr int M_STAGE = 4 * TILE;
constexpr int M_P = NST * M_STAGE;
constexpr int M_DP = M_P + 2 * TILE;
constexpr int M_RP = M_DP + 2 * TILE;
constexpr int M_SMEM = M_RP + 8192 + 1024;
static_assert(S_SMEM + 2048 <= 232448 && M_SMEM + 2048 <= 232448, "shared memory");

__device__ __forceinline__ void compute_sync() {  // the four compute warps only
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Element (r, d) of a swizzled [128][64] bf16 tile, as float.
__device__ __forceinline__ float tile_at(const uint8_t* tile, int r, int d) {
  const uint32_t off = static_cast<uint32_t>(r) * 128u +
                       ((static_cast<uint32_t>(d >> 3) ^ (r & 7u)) << 4) + (d & 7) * 2;
  return __bfloat162float(*reinterpret_cast<const bf16*>(tile + off));
}

// Row r of a swizzled [128][64] bf16 tile as 64 floats.
__device__ __forceinline__ void tile_row(const uint8_t* tile, int r, float* x) {
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + r * 128 + ((c8 ^ (r & 7)) << 4));
    Vec16<bf16>::unpack(u, x + 8 * c8);
  }
}

// Column sums over half of a chunk: thread t sums column (t & 63) over rows
// 64 (t >> 6) .. + 63, weighted by w[row] when w is given.
__device__ __forceinline__ float half_colsum(const uint8_t* tile, const float* w, int t) {
  const int d = t & 63, r0 = (t >> 6) * 64;
  float acc = 0.f;
  for (int r = r0; r < r0 + 64; ++r) {
    const float x = tile_at(tile, r, d);
    acc = w != nullptr ? fmaf(w[r], x, acc) : acc + x;
  }
  return acc;
}

// 64 fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  tmem_ld16(taddr, v);
  tmem_ld16(taddr + 16, v + 16);
  tmem_ld16(taddr + 32, v + 32);
  tmem_ld16(taddr + 48, v + 48);
  tmem_ld_wait();
}

// Reads the 128 fp32 columns of row `row` of an accumulator, adds `add`,
// keeps keys j <= row and stores bf16 row `row` of a [128][128] operand held
// as two swizzled [128][64] tiles.
__device__ __forceinline__ void mask_row_to_smem(uint32_t taddr, float add, uint8_t* dst, int row) {
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    float a[64];
    tmem_ld64(taddr + 64 * h, a);
#pragma unroll
    for (int i = 0; i < 64; ++i) a[i] = (64 * h + i <= row) ? a[i] + add : 0.f;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) st_row_chunk(dst + h * TILE, row, c8, a + 8 * c8);
  }
}

__device__ __forceinline__ void store_row_bf16(bf16* dst, const float* f) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8)
    d[c8] = make_uint4(pack_bf16(f[8 * c8], f[8 * c8 + 1]), pack_bf16(f[8 * c8 + 2], f[8 * c8 + 3]),
                       pack_bf16(f[8 * c8 + 4], f[8 * c8 + 5]),
                       pack_bf16(f[8 * c8 + 6], f[8 * c8 + 7]));
}

template <int MODE>
__global__ void __launch_bounds__(NTHR, 1)
    k_tc_bwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
             const __grid_constant__ CUtensorMap tmO, const float* __restrict__ den,
             float* __restrict__ rec, bf16* __restrict__ gt_out, float* __restrict__ gam,
             bf16* __restrict__ dq, bf16* __restrict__ dk, bf16* __restrict__ dv, int N, int nseg,
             int seg_len, int* err) {
  const int p = blockIdx.x, bh = blockIdx.y;
  const int role = MODE == 0 ? 2 : static_cast<int>(blockIdx.z);  // 0 dq, 1 dk/dv, 2 partials
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  __shared__ uint64_t bar_full[NST], bar_empty[NST];
  __shared__ uint64_t bar_in, bar_a, bar_p, bar_rp, bar_o, bar_s;
  __shared__ uint32_t tmem_base;
  __shared__ float s_vec[64];        // carried z (role 0) or r (role 1)
  __shared__ float s_part[2][64];    // per-half column sums of the current chunk
  __shared__ float s_part2[2][64];   // MODE 0: second set (r)
  __shared__ float s_gam[TC_C];
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p * seg_len;
  const int ne = min(N, nb + seg_len);
  const int nch = (ne - nb + TC_C - 1) / TC_C;
  const int stage_bytes = MODE == 0 ? S_STAGE : M_STAGE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], MODE == 0 ? 1 : 1 + 128);
    }
    mbar_init(&bar_in, 128);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_p, 128);
    mbar_init(&bar_rp, 128);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_s, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmG);
    if (MODE == 0) prefetch_tensormap(&tmO);
  }
  if (threadIdx.x == 0) s_abort = 0;
  if (warp == 1) tmem_alloc(&tmem_base, 512);
  // Bounded wait shared by all roles: after the first failure every later
  // wait gives up at once, so all threads still reach the block-wide barriers.
  auto wt = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
    if (*reinterpret_cast<volatile int*>(&s_abort)) return false;
    if (mbar_wait(bar, parity, WAIT_NS)) return true;
    *reinterpret_cast<volatile int*>(&s_abort) = 1;
    fail(err, code);
    return false;
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_base;
  const uint32_t TA = tm, TDA = tm + 128, TG1 = tm + 256, TG2 = tm + 320, TST = tm + 384;
  auto chunk_at = [&](int c) { return role == 1 ? nch - 1 - c : c; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int ntile = MODE == 0 ? 5 : 4;
      for (int c = 0; c < nch; ++c) {
        const int s = c % NST;
        if (c >= NST && !wt(&bar_empty[s], ((c / NST) - 1) & 1, 21)) break;
        uint8_t* st = sm + s * stage_bytes;
        mbar_arrive_expect_tx(&bar_full[s], ntile * TILE);
        const int n0 = nb + chunk_at(c) * TC_C;
        tma_load_3d(st, &tmQ, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + TILE, &tmK, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + 2 * TILE, &tmV, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + 3 * TILE, &tmG, &bar_full[s], 0, n0, bh);
        if (MODE == 0) tma_load_3d(st + 4 * TILE, &tmO, &bar_full[s], 0, n0, bh);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_AA = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_G = idesc_bf16(128, 64, false, false);
      constexpr uint32_t ID_GMN = idesc_bf16(128, 64, false, true);
      constexpr uint32_t ID_GTT = idesc_bf16(128, 64, true, true);
      constexpr uint32_t ID_ST = idesc_bf16(64, 64, true, true);
      const uint32_t pp = smem_u32(sm + M_P), dp = smem_u32(sm + M_DP), rp = smem_u32(sm + M_RP);
      for (int c = 0; c < nch; ++c) {
        const int s = c % NST;
        const uint32_t qs = smem_u32(sm + s * stage_bytes), ks = qs + TILE, vs = qs + 2 * TILE;
        const uint32_t gs = MODE == 0 ? smem_u32(sm + S_GT) : qs + 3 * TILE;  // gt operand
        if (!wt(&bar_in, c & 1, 22)) break;
        tc_fence_after();
        if (MODE == 0) {
          for (int kk = 0; kk < 8; ++kk)  // S += phi(K)^T V
            mma_bf16(TG1, sdesc(ks + kk * 2048, 16, 1024), sdesc(vs + kk * 2048, 16, 1024), ID_ST, 1);
          for (int kk = 0; kk < 8; ++kk)  // R += phi(Q)^T gt
            mma_bf16(TST, sdesc(qs + kk * 2048, 16, 1024), sdesc(gs + kk * 2048, 16, 1024), ID_ST, 1);
          mma_commit(&bar_s);
          mma_commit(&bar_empty[s]);
          continue;
        }
        for (int kk = 0; kk < 4; ++kk)  // dA (without gam) = gt V^T
          mma_bf16(TDA, sdesc(gs + 32 * kk, 16, 1024), sdesc(vs + 32 * kk, 16, 1024), ID_AA, kk > 0);
        if (role == 1)
          for (int kk = 0; kk < 4; ++kk)  // A = phi(Q) phi(K)^T
            mma_bf16(TA, sdesc(qs + 32 * kk, 16, 1024), sdesc(ks + 32 * kk, 16, 1024), ID_AA, kk > 0);
        mma_commit(&bar_a);
        if (!wt(&bar_p, c & 1, 23) || !wt(&bar_rp, c & 1, 23)) break;
        tc_fence_after();
        if (role == 0) {
          for (int kk = 0; kk < 8; ++kk)  // dP phi(K)
            mma_bf16(TG1, sdesc(dp + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024),
                     sdesc(ks + kk * 2048, 16, 1024), ID_GMN, kk > 0);
          for (int kk = 0; kk < 4; ++kk)  // + gt S_prev^T
            mma_bf16(TG1, sdesc(gs + 32 * kk, 16, 1024), sdesc(rp + 32 * kk, 16, 1024), ID_G, 1);
          mma_commit(&bar_o);
          for (int kk = 0; kk < 8; ++kk)  // S += phi(K)^T V
            mma_bf16(TST, sdesc(ks + kk * 2048, 16, 1024), sdesc(vs + kk * 2048, 16, 1024), ID_ST, 1);
        } else {
          for (int kk = 0; kk < 8; ++kk)  // dP^T phi(Q)
            mma_bf16(TG1, sdesc(dp + kk * 2048, TILE, 1024), sdesc(qs + kk * 2048, 16, 1024), ID_GTT,
                     kk > 0);
          for (int kk = 0; kk < 4; ++kk)  // + V R^T
            mma_bf16(TG1, sdesc(vs + 32 * kk, 16, 1024), sdesc(rp + 32 * kk, 16, 1024), ID_G, 1);
          for (int kk = 0; kk < 8; ++kk)  // P^T gt
            mma_bf16(TG2, sdesc(pp + kk * 2048, TILE, 1024), sdesc(gs + kk * 2048, 16, 1024), ID_GTT,
                     kk > 0);
          for (int kk = 0; kk < 4; ++kk)  // + phi(K) R
            mma_bf16(TG2, sdesc(ks + 32 * kk, 16, 1024), sdesc(rp + kk * 2048, 16, 1024), ID_GMN, 1);
          mma_commit(&bar_o);
          for (int kk = 0; kk < 8; ++kk)  // R += phi(Q)^T gt
            mma_bf16(TST, sdesc(qs + kk * 2048, 16, 1024), sdesc(gs + kk * 2048, 16, 1024), ID_ST, 1);
        }
        mma_commit(&bar_s);
        mma_commit(&bar_empty[s]);
      }
    }
  } else {
    // ---------------------------------------------------------- compute warps
    const int t = threadIdx.x - 64;
    const int qd = warp & 3;
    const int row = 32 * qd + lane;
    const uint32_t lq = static_cast<uint32_t>(32 * qd) << 16;
    const bool has_s = lane < 16;  // M=64 accumulators: row 16*qd + lane in lane 32*qd + lane
    const int srow = 16 * qd + lane;
    const long hb = static_cast<long>(bh) * N;
    float sv[64];
    if (MODE == 1) {
      // carried state: role 0 sums the records of earlier segments (S, z),
      // role 1 those of later segments (R, r)
      const int lo = role == 0 ? 0 : p + 1, hi = role == 0 ? p : nseg;
      const int off = role == 0 ? 0 : DM + 64;
      for (int j = 0; j < 64; ++j) sv[j] = 0.f;
      float vec = 0.f;
      for (int pp = lo; pp < hi; ++pp) {
        const float* r0 = rec + (static_cast<long>(bh) * nseg + pp) * REC + off;
        if (has_s) {
          const float4* rr = reinterpret_cast<const float4*>(r0 + srow * 64);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float4 x = rr[j];
            sv[4 * j] += x.x;
            sv[4 * j + 1] += x.y;
            sv[4 * j + 2] += x.z;
            sv[4 * j + 3] += x.w;
          }
        }
        if (t < 64) vec += r0[DM + t];
      }
      if (t < 64) s_vec[t] = vec;
      for (int j = 0; j < 64; j += 16) tmem_st16(TST + lq + j, sv + j);
      tmem_st_wait();
      if (has_s)
        for (int c8 = 0; c8 < 8; ++c8) st_row_chunk(sm + M_RP, srow, c8, sv + 8 * c8);
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_rp);
    } else {
      for (int j = 0; j < 64; ++j) sv[j] = 0.f;
      for (int j = 0; j < 64; j += 16) {
        tmem_st16(TG1 + lq + j, sv + j);
        tmem_st16(TST + lq + j, sv + j);
      }
      tmem_st_wait();
      tc_fence_before();
    }
    float zacc = 0.f, racc = 0.f;  // MODE 0 column-sum accumulators
    for (int c = 0; c < nch; ++c) {
      const int s = c % NST;
      const int n0 = nb + chunk_at(c) * TC_C;
      const int valid = min(TC_C, ne - n0);
      const bool rv = row < valid;
      uint8_t* st = sm + s * stage_bytes;
      if (MODE == 0) {
        const float dn = rv ? den[hb + n0 + row] : 1.f;
        if (c > 0) {  // the gt tile is free once the previous chunk's MMAs finished
          wt(&bar_s, (c - 1) & 1, 24);
          tc_fence_after();
        }
        wt(&bar_full[s], (c / NST) & 1, 25);
        // gt = dout / den, gam = -(gt . out) for this row
        float g[64], o[64];
        tile_row(st + 3 * TILE, row, g);
        tile_row(st + 4 * TILE, row, o);
        const float inv = 1.f / dn;
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          g[i] = rv ? g[i] * inv : 0.f;
          acc = fmaf(g[i], o[i], acc);
        }
        const float gm = rv ? -acc : 0.f;
        s_gam[row] = gm;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) st_row_chunk(sm + S_GT, row, c8, g + 8 * c8);
        if (rv) {
          store_row_bf16(gt_out + (hb + n0 + row) * 64, g);
          gam[hb + n0 + row] = gm;
        }
        phi_tile(st, valid, t);
        phi_tile(st + TILE, valid, t);
        compute_sync();
        zacc += half_colsum(st + TILE, nullptr, t);
        racc += half_colsum(st, s_gam, t);
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_in);
        continue;
      }
      // ------------------------------------------------------------- MODE 1
      const float gm = rv ? gam[hb + n0 + row] : 0.f;
      wt(&bar_full[s], (c / NST) & 1, 25);
      if (role == 1) phi_tile(st, valid, t);
      phi_tile(st + TILE, valid, t);
      if (role == 1) s_gam[row] = gm;
      compute_sync();
      const float part = role == 0 ? half_colsum(st + TILE, nullptr, t) : half_colsum(st, s_gam, t);
      s_part[t >> 6][t & 63] = part;
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_in);

      wt(&bar_a, c & 1, 26);
      tc_fence_after();
      mask_row_to_smem(TDA + lq, gm, sm + M_DP, row);
      if (role == 1) mask_row_to_smem(TA + lq, 0.f, sm + M_P, row);
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_p);

      wt(&bar_o, c & 1, 27);
      tc_fence_after();
      {
        float gv[64], x[64];
        tmem_ld64(TG1 + lq, gv);
        if (role == 0) {  // dq = (grad_phiQ + gam z_prev) * phi'(Q), raw Q in the stage
          tile_row(st, row, x);
#pragma unroll
          for (int i = 0; i < 64; ++i) gv[i] = (gv[i] + gm * s_vec[i]) * (x[i] > 0.f ? 1.f : __expf(x[i]));
          if (rv) store_row_bf16(dq + (hb + n0 + row) * 64, gv);
        } else {          // dk = (grad_phiK + r_next) * phi'(K), phi'(K) = min(phi(K), 1)
          tile_row(st + TILE, row, x);
#pragma unroll
          for (int i = 0; i < 64; ++i) gv[i] = (gv[i] + s_vec[i]) * fminf(x[i], 1.f);
          if (rv) store_row_bf16(dk + (hb + n0 + row) * 64, gv);
          tmem_ld64(TG2 + lq, gv);
          if (rv) store_row_bf16(dv + (hb + n0 + row) * 64, gv);
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_empty[s]);  // this thread is done with the stage
      compute_sync();
      if (t < 64) s_vec[t] += s_part[0][t] + s_part[1][t];  // z or r now includes this chunk
      wt(&bar_s, c & 1, 28);
      tc_fence_after();
      if (c + 1 < nch) {
        tmem_ld64(TST + lq, sv);
        if (has_s)
          for (int c8 = 0; c8 < 8; ++c8) st_row_chunk(sm + M_RP, srow, c8, sv + 8 * c8);
        fence_proxy_async();
        compute_sync();  // s_vec updated before the next chunk's epilogue reads it
        tc_fence_before();
        mbar_arrive(&bar_rp);
      }
    }
    if (MODE == 0) {
      s_part[t >> 6][t & 63] = zacc;
      s_part2[t >> 6][t & 63] = racc;
      if (wt(&bar_s, (nch - 1) & 1, 29)) {
        tc_fence_after();
        float* r0 = rec + (static_cast<long>(bh) * nseg + p) * REC;
        tmem_ld64(TG1 + lq, sv);
        if (has_s)
          for (int j = 0; j < 64; ++j) r0[srow * 64 + j] = sv[j];
        tmem_ld64(TST + lq, sv);
        if (has_s)
          for (int j = 0; j < 64; ++j) r0[DM + 64 + srow * 64 + j] = sv[j];
        compute_sync();
        if (t < 64) {
          r0[DM + t] = s_part[0][t] + s_part[1][t];
          r0[2 * DM + 64 + t] = s_part2[0][t] + s_part2[1][t];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tm, 512);
}

}  // namespace

SegPlan tc_plan_bwd(int BH, int N) { return tc_plan(2 * BH, N); }

// workspace: records [BH][nseg][REC] fp32 | gt bf16 [BH][N][64] | gam fp32 [BH][N] | status
size_t causal_bwd_tc_ws_floats(const Shape& s) {
  const size_t BH = static_cast<size_t>(s.B) * s.H;
  const SegPlan pl = tc_plan_bwd(s.B * s.H, s.N);
  return BH * pl.nseg * REC + BH * s.N * 32 + BH * s.N + 4;
}

int causal_bwd_tc_launches(const Shape&) { return 2; }

cudaError_t causal_bwd_tc(const void* q, const void* k, const void* v, const void* out,
                          const float* den, const void* dout, void* dq, void* dk, void* dv,
                          float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const SegPlan pl = tc_plan_bwd(BH, s.N);
  float* rec = ws;
  bf16* gt = reinterpret_cast<bf16*>(ws + static_cast<size_t>(BH) * pl.nseg * REC);
  float* gam = ws + static_cast<size_t>(BH) * pl.nseg * REC + static_cast<size_t>(BH) * s.N * 32;
  int* err = reinterpret_cast<int*>(gam + static_cast<size_t>(BH) * s.N);
  CUtensorMap mq, mk, mv, mg, mo, mgt;
  if (!make_bf16_map(&mq, q, BH, s.N) || !make_bf16_map(&mk, k, BH, s.N) ||
      !make_bf16_map(&mv, v, BH, s.N) || !make_bf16_map(&mg, dout, BH, s.N) ||
      !make_bf16_map(&mo, out, BH, s.N) || !make_bf16_map(&mgt, gt, BH, s.N))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_tc_bwd<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                S_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_tc_bwd<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                M_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaMemsetAsync(err, 0, sizeof(int), st)) != cudaSuccess) return e;
  k_tc_bwd<0><<<dim3(pl.nseg, BH, 1), NTHR, S_SMEM, st>>>(mq, mk, mv, mg, mo, den, rec, gt, gam,
                                                          nullptr, nullptr, nullptr, s.N, pl.nseg,
                                                          pl.seg_len, err);
  k_tc_bwd<1><<<dim3(pl.nseg, BH, 2), NTHR, M_SMEM, st>>>(
      mq, mk, mv, mgt, mgt, den, rec, gt, gam, static_cast<bf16*>(dq), static_cast<bf16*>(dk),
      static_cast<bf16*>(dv), s.N, pl.nseg, pl.seg_len, err);
  return cudaGetLastError();
}

}  // namespace la
