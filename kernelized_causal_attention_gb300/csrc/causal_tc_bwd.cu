// Backward of causal linear attention on the tcgen05 tensor cores, bf16 with
// D, M in {16, 32, 64} (narrower heads zero-filled to the 64-wide tiles, phi
// zeroed on the padded features) and fp32 accumulation in tensor memory.
//
// Method: "Transformers are RNNs" (part 2/3) §3.3.1 eq. 13-15, the gradients
// of the numerator as cumulative sums, completed with the denominator by the
// quotient rule.  With gt_i = dout_i / den_i and gam_i = -(gt_i . out_i):
//   dA_ij      = gt_i . V_j + gam_i            (j <= i)
//   grad_phiQ  = dP phi(K) + gt S_prev^T + gam z_prev^T          (forward sums)
//   grad_phiK  = dP^T phi(Q) + V R_next^T + r_next                (reverse sums)
//   dv         = P^T gt + phi(K) R_next
//   S += phi(K)^T V, z += phi(K)^T 1;  R += phi(Q)^T gt, r += phi(Q)^T gam
// with P = bf16(mask(phi(Q) phi(K)^T)) and dP = bf16(mask(dA)); then
// dq = grad_phiQ * phi'(Q), dk = grad_phiK * phi'(K), and phi'(x) = min(phi(x), 1).
//
// Two kernels.  The state pass k_tc_bwd_state (one CTA per one or two
// sub-segments of whole 128-token chunks) reads q, k, v, dout, out and den
// once; it stores phi(Q), phi(K) and gt = dout / den (bf16) and gam (fp32) in
// the workspace, and each sub-segment's partial S, z, R, r.  The main pass
// k_tc_bwd_main fills one wave of CTAs with runs of whole sub-segments: role 0
// walks its run forward carrying S, z and writes dq; role 1 walks backward
// carrying R, r and writes dk and dv.  A run may cross from one (b, h) into
// the next (the state restarts from zero there), so the roles can be given
// different run lengths: a dk / dv chunk costs about 1.4 times a dq chunk,
// and the 3072-token workload runs 64 dq runs of 12 chunks beside 86 dk / dv
// runs of 9.  Each CTA first adds up the partial states of the sub-segments
// before (role 0) or after (role 1) its run.
// Every product, including the vector sums z and r (against a ones column
// or the gam column), runs on tcgen05 with TMA-fed operands; dq, dk and dv
// are staged in shared memory and written with TMA stores.
//
// Variants on the same kernels.  feat: phi(Q), phi(K) are the given rows (the
// degree-2 polynomial map) and phi' = 1.  DECAY (a template flag): the state
// pass writes phi(Q) rows scaled by gamma^i' and phi(K) rows by gamma^(127-j')
// (within the chunk) to the workspace and scales its own copies by the
// distance to its sub-segment's start (phi(Q), reverse records) or end
// (phi(K), forward records); the main pass then masks with the constant
// gamma^-128, carries S~ and R~ with a gamma^128 write-back after each
// read-out, and its epilogues restore the row frames (dq by gamma^(i'+1), dk
// by gamma^(128-j'), dv by gamma).
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tc_chunk.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcc;

constexpr int DM = 64 * 64;
constexpr int REC = 2 * (DM + 64);  // per-sub-segment record [S | z | R | r]

// Main-pass shared memory: two stages of phi(Q), phi(K), V, gt; P; dP (both
// also the output staging); two bf16 state tiles; the vector atom (role 0:
// ones, the N atom of [V | 1]; role 1: gam in column 0, the N atom of [gt | gam]).
constexpr int M_STAGE = 4 * TILE;
constexpr int M_P = NST * M_STAGE;
constexpr int M_DP = M_P + 2 * TILE;
constexpr int M_RP = M_DP + 2 * TILE;
constexpr int M_VEC = M_RP + 2 * 8192;
constexpr int M_SMEM = M_VEC + TILE + 1024;
static_assert(M_SMEM + 2048 <= 232448, "shared memory");

// Role 1: the masked bf16 rows of dA (+ gam) and of A for this warpgroup's
// KW keys from key0, loaded together so that one wait covers both.
__device__ __forceinline__ void mask2_cols(uint32_t tda, uint32_t ta, float add, uint8_t* ddst,
                                           uint8_t* adst, int row, int key0, float dscale = 1.f,
                                           float ascale = 1.f) {
  float d[KW], a[KW];
#pragma unroll
  for (int i = 0; i < KW / 16; ++i) {
    tmem_ld16(tda + 16 * i, d + 16 * i);
    tmem_ld16(ta + 16 * i, a + 16 * i);
  }
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < KW; ++i) {
    const bool keep = key0 + i <= row;
    d[i] = keep ? (d[i] + add) * dscale : 0.f;
    a[i] = keep ? a[i] * ascale : 0.f;
  }
  tile_put_cols<KW>(ddst, row, key0 & 63, d);
  tile_put_cols<KW>(adst, row, key0 & 63, a);
}

struct BwdMaps {
  CUtensorMap q, k, v, g, o;  // state-pass inputs
  CUtensorMap fq, fk, gt;     // state-pass outputs, main-pass inputs
  CUtensorMap dq, dk, dv;     // main-pass outputs (TMA stores)
};

// Main pass: each CTA takes one role over a run of whole sub-segments, a
// contiguous range [F0, F1) of flat chunk indices bh * nchh + chunk that may
// cross from one (b, h) into the next.  Role 0 (the first n0cta CTAs, upc0
// sub-segments each) walks its run forward carrying S~ = [S | z] and writes
// dq; role 1 (upc1 sub-segments each) walks it backward carrying R~ = [R | r]
// and writes dk and dv.  The run starts from the records of the sub-segments
// before it (role 0) or after it (role 1) in its first (b, h); where it enters
// the next (b, h) the carried state restarts from zero.  Per chunk: A and dA,
// then the carried-state update (it only needs the stage, so the compute warps
// read the next state out while the gradient products run), then the gradient
// products.  The vector terms gam z_prev (dq) and r_next (dk) are added in the
// epilogues.
template <bool DECAY>
__global__ void __launch_bounds__(NTHR, 1)
    k_tc_bwd_main(const __grid_constant__ BwdMaps maps, const float* __restrict__ rec,
                  const float* __restrict__ gam, int N, int nchh, int cps, int nsub, int BH,
                  int n0cta, int upc0, int upc1, int feat, float lg, int* err) {
  const int role = static_cast<int>(blockIdx.x) < n0cta ? 0 : 1;  // 0 dq, 1 dk / dv
  const int idx = static_cast<int>(blockIdx.x) - (role == 0 ? 0 : n0cta);
  const int upc = role == 0 ? upc0 : upc1;
  const int u0 = idx * upc, u1 = min(BH * nsub, u0 + upc);  // sub-segments [u0, u1) of BH * nsub
  const int F0 = (u0 / nsub) * nchh + (u0 % nsub) * cps;
  const int F1 = ((u1 - 1) / nsub) * nchh + min(nchh, ((u1 - 1) % nsub + 1) * cps);
  const int nch = F1 - F0;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  __shared__ uint64_t bar_full[NST], bar_empty[NST];
  __shared__ uint64_t bar_in, bar_a, bar_p, bar_rp, bar_o, bar_o2, bar_s;
  __shared__ uint32_t tmem_base;
  __shared__ float s_vec[2][64];  // carried z (role 0) or r (role 1) before chunk c, by c & 1
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* vec = sm + M_VEC;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1 + NCOMP);  // the MMAs and every compute thread (epilogues read phi)
    }
    mbar_init(&bar_in, NCOMP);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_p, NCOMP);
    mbar_init(&bar_rp, NCOMP);
    mbar_init(&bar_o, 1);   // dq (role 0) or dk (role 1) products done
    mbar_init(&bar_o2, 1);  // role 1: the dv products done
    mbar_init(&bar_s, 1);
    fence_barrier_init();
    s_abort = 0;
  }
  if (warp == 1) tmem_alloc(&tmem_base, 512);
  if (warp >= 2) {  // the vector atom: ones (role 0) or zeros (role 1; gam is written per chunk)
    const int t = threadIdx.x - 64;
    for (int v = t; v < TILE / 16; v += NCOMP) {
      const int r = v >> 3, c = (v & 7) ^ (r & 7);
      *reinterpret_cast<uint4*>(vec + v * 16) =
          (role == 0 && c == 0) ? make_uint4(0x3f80u, 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();
  }
  // Bounded wait: after the first failure every later wait gives up at once,
  // so all threads still reach the block-wide barriers.
  auto wt = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
    if (*reinterpret_cast<volatile int*>(&s_abort)) return false;
    if (mbar_wait(bar, parity, WAIT_NS)) return true;
    *reinterpret_cast<volatile int*>(&s_abort) = 1;
    fail(err, code);
    return false;
  };
  // the same, agreed by the whole warp (tcgen05 loads and stores that follow
  // are warp-collective)
  auto wtu = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
    return __all_sync(0xffffffffu, wt(bar, parity, code));
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();  // the state pass's outputs are visible from here on
  const uint32_t tm = tmem_base;
  const uint32_t TA = tm, TDA = tm + 128, TG1 = tm + 256, TG2 = tm + 320, TST = tm + 384;
  // the c-th chunk in walking order: its flat index, (b, h) and first token
  auto flat_at = [&](int c) { return role == 1 ? F1 - 1 - c : F0 + c; };
  auto bh_at = [&](int c) { return flat_at(c) / nchh; };
  auto n0_at = [&](int c) { return (flat_at(c) % nchh) * TC_C; };
  // chunk c opens a new (b, h) within the run: the carried state restarts at zero
  auto head_first = [&](int c) {
    return c > 0 && flat_at(c) % nchh == (role == 0 ? 0 : nchh - 1);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nch; ++c) {
        const int s = c % NST;
        if (c >= NST && !wt(&bar_empty[s], ((c / NST) - 1) & 1, 21)) break;
        // every CTA starts at once: chunk 0's tiles come in alone (they gate
        // the first products), chunk 1's follow while chunk 0 is worked on
        if (c == 1 && !wt(&bar_full[0], 0, 21)) break;
        uint8_t* st = sm + s * M_STAGE;
        mbar_arrive_expect_tx(&bar_full[s], 4 * TILE);
        const int n0 = n0_at(c), bh = bh_at(c);
        tma_load_3d(st, &maps.fq, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + TILE, &maps.fk, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + 2 * TILE, &maps.v, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + 3 * TILE, &maps.gt, &bar_full[s], 0, n0, bh);
        ++issued;
      }
      for (int i = issued > NST ? issued - NST : 0; i < issued; ++i)  // no load in flight at exit
        mbar_wait(&bar_full[i % NST], (i / NST) & 1, WAIT_NS);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_AA = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_G = idesc_bf16(128, 64, false, false);
      constexpr uint32_t ID_GMN = idesc_bf16(128, 64, false, true);
      constexpr uint32_t ID_GTT = idesc_bf16(128, 64, true, true);
      constexpr uint32_t ID_ST = idesc_bf16(64, 80, true, true);  // 64 x 80 state update
      const uint64_t dP0 = sdesc(smem_u32(sm + M_P), TILE, 1024);
      const uint64_t dDP = sdesc(smem_u32(sm + M_DP), 16, 1024);
      const uint64_t dDPT = sdesc(smem_u32(sm + M_DP), TILE, 1024);
      const uint32_t vaddr = smem_u32(vec);
      for (int c = 0; c < nch; ++c) {
        const int s = c % NST;
        const uint32_t qs = smem_u32(sm + s * M_STAGE), ks = qs + TILE, vs = qs + 2 * TILE, gs = qs + 3 * TILE;
        const uint64_t dQ = sdesc(qs, 16, 1024), dK = sdesc(ks, 16, 1024);
        const uint64_t dV = sdesc(vs, 16, 1024), dG = sdesc(gs, 16, 1024);
        const uint64_t dRP = sdesc(smem_u32(sm + M_RP + (c & 1) * 8192), 16, 1024);
        if (!wt(&bar_in, c & 1, 22)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dA (without gam) = gt V^T
          mma_bf16(TDA, dadd(dG, 32 * kk), dadd(dV, 32 * kk), ID_AA, kk > 0);
        if (role == 1)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // A = phi(Q) phi(K)^T
            mma_bf16(TA, dadd(dQ, 32 * kk), dadd(dK, 32 * kk), ID_AA, kk > 0);
        mma_commit(&bar_a);
        if (!wt(&bar_rp, c & 1, 23)) break;  // the carried state has been read out
        tc_fence_after();
        const bool fresh = head_first(c);  // a new (b, h): the state restarts from zero
        if (role == 0) {
          const uint64_t dVt = sdesc(vs, vaddr - vs, 1024);  // [V | 1]
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // S~ += phi(K)^T [V | 1]
            mma_bf16(TST, dadd(dK, kk * 2048), dadd(dVt, kk * 2048), ID_ST, kk > 0 || !fresh);
        } else {
          const uint64_t dGt = sdesc(gs, vaddr - gs, 1024);  // [gt | gam]
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // R~ += phi(Q)^T [gt | gam]
            mma_bf16(TST, dadd(dQ, kk * 2048), dadd(dGt, kk * 2048), ID_ST, kk > 0 || !fresh);
        }
        mma_commit(&bar_s);
        if (!wt(&bar_p, c & 1, 23)) break;
        tc_fence_after();
        if (role == 0) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dP phi(K)
            mma_bf16(TG1, dadd(dDP, (kk >> 2) * TILE + (kk & 3) * 32), dadd(dK, kk * 2048), ID_GMN,
                     kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // + gt S_prev^T
            mma_bf16(TG1, dadd(dG, 32 * kk), dadd(dRP, 32 * kk), ID_G, 1);
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dP^T phi(Q)
            mma_bf16(TG1, dadd(dDPT, kk * 2048), dadd(dQ, kk * 2048), ID_GTT, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // + V R^T
            mma_bf16(TG1, dadd(dV, 32 * kk), dadd(dRP, 32 * kk), ID_G, 1);
          mma_commit(&bar_o);  // the dk epilogue may start while the dv products run
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // P^T gt
            mma_bf16(TG2, dadd(dP0, kk * 2048), dadd(dG, kk * 2048), ID_GTT, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // + phi(K) R
            mma_bf16(TG2, dadd(dK, 32 * kk), dadd(dRP, kk * 2048), ID_GMN, 1);
        }
        mma_commit(role == 0 ? &bar_o : &bar_o2);
        mma_commit(&bar_empty[s]);
      }
      // every issued MMA has finished before the exit (also after an early break)
      mma_commit(&bar_s);
      mbar_wait(&bar_s, nch & 1, WAIT_NS);
    }
  } else {
    // ---------------------------------------------------------- compute warps
    // NWG warpgroups; each covers all 128 rows (TMEM lanes) and takes a slice
    // of the columns: KW keys of A / dA from k0, OW output columns from c0.
    const int t = threadIdx.x - 64;  // 0 .. NCOMP-1
    const int wg = t >> 7;
    const int qd = warp & 3;
    const int row = 32 * qd + lane;
    const uint32_t lq = static_cast<uint32_t>(32 * qd) << 16;
    const bool has_s = lane < 16;  // M=64 accumulators: row 16*qd + lane in lane 32*qd + lane
    const int srow = 16 * qd + lane;
    const int c0 = OW * wg, k0 = KW * wg;
    auto gam_at = [&](int c) {  // gam of this thread's row in chunk c
      const int n0 = n0_at(c);
      return row < min(TC_C, N - n0) ? gam[static_cast<long>(bh_at(c)) * N + n0 + row] : 0.f;
    };
    // gam_i into row i, column 0 of the vector atom (128-byte swizzle)
    auto put_gam = [&](float g) {
      *reinterpret_cast<bf16*>(vec + row * 128 + ((row & 7) << 4)) = __float2bfloat16_rn(g);
    };
    {
      // carried state: role 0 sums the records of the sub-segments before its
      // run ([S | z]), role 1 those after it ([R | r]), in the (b, h) where the
      // walk starts; every compute thread adds up a slice, into the P tile
      // (free until the first mask)
      const int ui = role == 0 ? u0 : u1 - 1;  // the first sub-segment walked
      const int bhi = ui / nsub;
      const int lo = role == 0 ? 0 : ui % nsub + 1;
      const int hi = role == 0 ? ui % nsub : nsub;
      const int off = role == 0 ? 0 : DM + 64;
      float* scr = reinterpret_cast<float*>(sm + M_P);
      // decay: a forward record (summed to its sub-segment's end) reaches the
      // run's start (sub-segment hi) through gamma^((hi - 1 - pp) sub_len); a
      // reverse record (summed from its start) reaches the run's end (the start
      // of sub-segment lo) through gamma^((pp - lo) sub_len)
      const int sub_len = cps * TC_C;
      auto wrec = [&](int pp) {
        if (!DECAY) return 1.f;
        const int e = role == 0 ? (hi - 1 - pp) : (pp - lo);
        return exp2f(lg * static_cast<float>(e) * static_cast<float>(sub_len));
      };
      const float4* rb = reinterpret_cast<const float4*>(rec + static_cast<long>(bhi) * nsub * REC + off);
      constexpr int RV = REC / 4;       // float4 per record
      constexpr int SV = (DM + 64) / 4; // float4 per state: 1040, columns t, t + 512, t + 1024
      float4 acc[3];
#pragma unroll
      for (int jj = 0; jj < 3; ++jj) acc[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int pp = lo; pp < hi; pp += 4) {  // four records of all three columns per round trip
        float4 x[4][3];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int jj = 0; jj < 3; ++jj) {
            const int j = t + jj * NCOMP;
            x[i][jj] = pp + i < hi && j < SV ? rb[static_cast<long>(pp + i) * RV + j]
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float f = DECAY && pp + i < hi ? wrec(pp + i) : 1.f;
#pragma unroll
          for (int jj = 0; jj < 3; ++jj) {
            acc[jj].x += f * x[i][jj].x;
            acc[jj].y += f * x[i][jj].y;
            acc[jj].z += f * x[i][jj].z;
            acc[jj].w += f * x[i][jj].w;
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < 3; ++jj)
        if (t + jj * NCOMP < SV) reinterpret_cast<float4*>(scr)[t + jj * NCOMP] = acc[jj];
      compute_sync();
      if (wg == 0) {  // into TMEM (the MMA's accumulator) and the bf16 state tile
        float sv[16];
#pragma unroll
        for (int j = 0; j < 5; ++j) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = 16 * j + i;
            sv[i] = !has_s ? 0.f : col < 64 ? scr[srow * 64 + col] : col == 64 ? scr[DM + srow] : 0.f;
          }
          if (has_s && j < 4) tile_put_cols<16>(sm + M_RP, srow, 16 * j, sv);
          if (has_s && j == 4) s_vec[0][srow] = sv[0];
          if (DECAY) {  // the state the first chunk adds to: gamma^128 times the carried one
            const float g128 = exp2f(128.f * lg);
#pragma unroll
            for (int i = 0; i < 16; ++i) sv[i] *= g128;
          }
          tmem_st16(TST + lq + 16 * j, sv);
        }
        tmem_st_wait();
      }
      fence_proxy_async();
      compute_sync();  // the P tile is free again
      tc_fence_before();
      mbar_arrive(&bar_rp);
      // chunk 0 inputs
      const float g0 = gam_at(0);
      wt(&bar_full[0], 0, 25);
      if (role == 1 && wg == 0) {
        put_gam(g0);
        fence_proxy_async();
      }
      mbar_arrive(&bar_in);
    }
    float gm = gam_at(0);
    for (int c = 0; c < nch; ++c) {
      const int s = c % NST;
      const int n0 = n0_at(c), bh = bh_at(c);
      uint8_t* st = sm + s * M_STAGE;
      // P, dP of chunk c
      const bool ok_a = wtu(&bar_a, c & 1, 26);
      tc_fence_after();
      if (t == 0) bulk_wait_read();  // the previous chunk's output tiles have left P / dP
      compute_sync();
      if (ok_a) {
        // decay: with the workspace's phi(Q) rows scaled by gamma^i' and phi(K) rows by
        // gamma^(127-j'), every weight gamma^(i'-j') becomes the constant gamma^-128 in a
        // row frame that the epilogues take back
        const float cm = DECAY ? exp2f(-128.f * lg) : 1.f;
        if (role == 1)
          mask2_cols(TDA + lq + k0, TA + lq + k0, gm, sm + M_DP + (k0 >> 6) * TILE,
                     sm + M_P + (k0 >> 6) * TILE, row, k0, cm, cm);
        else
          mask_cols<KW>(TDA + lq + k0, gm, sm + M_DP + (k0 >> 6) * TILE, row, k0, cm);
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_p);
      // carried state for chunk c+1 (after this chunk's update); it must be
      // read before the next chunk's gam replaces this chunk's in the vector atom
      if (c + 1 < nch) {
        const bool fresh = head_first(c + 1);  // a new (b, h): it starts from a zero state
        if (wtu(&bar_s, c & 1, 28)) {
          tc_fence_after();
          float sv[OW], vv[16];
          if (fresh) {
#pragma unroll
            for (int i = 0; i < OW; ++i) sv[i] = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) vv[i] = 0.f;
          } else {
            tmem_ldn<OW / 16>(TST + lq + c0, sv);
            tmem_ldn<1>(TST + lq + 64, vv);
          }
          if (has_s) {
            tile_put_cols<OW>(sm + M_RP + ((c + 1) & 1) * 8192, srow, c0, sv);
            if (wg == 0) s_vec[(c + 1) & 1][srow] = vv[0];
          }
          if (DECAY && !fresh) {  // the next chunk adds to gamma^128 times this state
            const float g128 = exp2f(128.f * lg);
#pragma unroll
            for (int i = 0; i < OW; ++i) sv[i] *= g128;
#pragma unroll
            for (int i = 0; i < OW / 16; ++i) tmem_st16(TST + lq + c0 + 16 * i, sv + 16 * i);
            if (wg == 0) {
#pragma unroll
              for (int i = 0; i < 16; ++i) vv[i] *= g128;
              tmem_st16(TST + lq + 64, vv);
            }
            tmem_st_wait();
          }
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_rp);
      }
      // inputs of chunk c+1 (the tensor cores may start on it)
      float gm_next = 0.f;
      if (c + 1 < nch) {
        gm_next = gam_at(c + 1);
        wt(&bar_full[(c + 1) % NST], ((c + 1) / NST) & 1, 25);
        if (role == 1 && wg == 0) {
          put_gam(gm_next);
          fence_proxy_async();
        }
        mbar_arrive(&bar_in);
      }
      // gradients of chunk c, staged in the free P / dP tiles and TMA-stored:
      // dq and dk over dP (read only by their own products), dv over P's
      // second half once the dv products are done
      if (wtu(&bar_o, c & 1, 27)) {
        tc_fence_after();
        const float* vcur = s_vec[c & 1];
        float gv[OW], x[OW];
        tmem_ldn<OW / 16>(TG1 + lq + c0, gv);
        if (role == 0) {  // dq = (grad_phiQ + gam z_prev) * phi'(Q)
          tile_row_cols<OW>(st, row, c0, x);
          // decay: the row frame gamma^-(i'+1) back; the tile holds gamma^i' phi(Q)
          const float fo = DECAY ? exp2f(lg * static_cast<float>(row + 1)) : 1.f;
          const float fx = DECAY ? exp2f(-lg * static_cast<float>(row)) : 1.f;
#pragma unroll
          for (int i = 0; i < OW; ++i)
            gv[i] = (gv[i] + gm * vcur[c0 + i]) * fo * (feat ? 1.f : fminf(x[i] * fx, 1.f));
          tile_put_cols<OW>(sm + M_DP, row, c0, gv);
        } else {          // dk = (grad_phiK + r_next) * phi'(K), dv
          tile_row_cols<OW>(st + TILE, row, c0, x);
          // decay: dk's row frame gamma^-(128-j') back, the tile holds gamma^(127-j')
          // phi(K), and dv comes out gamma^-1 times the true one
          const float fo = DECAY ? exp2f(lg * static_cast<float>(128 - row)) : 1.f;
          const float fx = DECAY ? exp2f(-lg * static_cast<float>(127 - row)) : 1.f;
#pragma unroll
          for (int i = 0; i < OW; ++i)
            gv[i] = (gv[i] + vcur[c0 + i]) * fo * (feat ? 1.f : fminf(x[i] * fx, 1.f));
          tile_put_cols<OW>(sm + M_DP, row, c0, gv);
          if (wtu(&bar_o2, c & 1, 29)) {
            tc_fence_after();
            tmem_ldn<OW / 16>(TG2 + lq + c0, gv);
            if (DECAY) {
              const float g1 = exp2f(lg);
#pragma unroll
              for (int i = 0; i < OW; ++i) gv[i] *= g1;
            }
            tile_put_cols<OW>(sm + M_P + TILE, row, c0, gv);
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_empty[s]);  // this thread is done with the stage
      compute_sync();              // s_vec[c & 1] is free again; the output tiles are complete
      if (t == 0 && !*reinterpret_cast<volatile int*>(&s_abort)) {
        if (role == 0) {
          tma_store_3d(&maps.dq, sm + M_DP, 0, n0, bh);
        } else {
          tma_store_3d(&maps.dk, sm + M_DP, 0, n0, bh);
          tma_store_3d(&maps.dv, sm + M_P + TILE, 0, n0, bh);
        }
        bulk_commit();
      }
      gm = gm_next;
    }
    if (t == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------- state pass
// One CTA per spc consecutive sub-segments (one or two).  Per chunk: phi(Q),
// phi(K) in place (and to the workspace), gt = dout / den in place over dout
// (and to the workspace), gam = -(gt . out) (to the workspace and as column 0
// of the gam tile), then
//   S~ += phi(K)^T [V | 1]   and   R~ += phi(Q)^T [gt | gam]
// as two 64 x 80 products whose last atoms are the ones tile and the gam
// tile, into the accumulator pair of the chunk's sub-segment.  Each
// sub-segment's partial [S | z | R | r] leaves by one bulk copy.
// smem: two stages of [Q | K | V | dout -> gt | out], the ones tile, two gam
// tiles (one per stage).
constexpr int SS_STAGE = 5 * TILE;
constexpr int SS_ONES = 2 * SS_STAGE;
constexpr int SS_GAMT = SS_ONES + TILE;
constexpr int SS_SMEM = SS_GAMT + 2 * TILE + 1024;
constexpr uint32_t ID_ST80 = idesc_bf16(64, 80, true, true);

struct StateMaps {
  CUtensorMap q, k, v, g, o;  // inputs
  CUtensorMap fq, fk, gt;     // the workspace rows the main pass reads (TMA stores)
};

// The constant ones tile ([128][64] bf16, column 0 = 1): the second N atom of
// the MN-major operand [V | 1].
__device__ __forceinline__ void ones_tile(uint8_t* tile, int t, int nthr) {
  for (int v = t; v < TILE / 16; v += nthr) {
    const int r = v >> 3, c = (v & 7) ^ (r & 7);
    *reinterpret_cast<uint4*>(tile + v * 16) =
        c == 0 ? make_uint4(0x3f80u, 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <bool DECAY>
__global__ void __launch_bounds__(NTHR, 1)
    k_tc_bwd_state(const __grid_constant__ StateMaps maps, const float* __restrict__ den,
                   float* __restrict__ gam, bf16* __restrict__ gt_out, bf16* __restrict__ fq_out,
                   bf16* __restrict__ fk_out, float* __restrict__ rec, int N, int sub_len, int nsub,
                   int spc, int dch, int feat, float lg, int* err) {
  const int p = blockIdx.x, bh = blockIdx.y;  // the call's first kernel
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  __shared__ uint64_t bar_full[2], bar_empty[2], bar_phi[2], bar_done, bar_st;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub0 = p * spc;                 // this CTA's first sub-segment
  const int nsb = min(spc, nsub - sub0);    // and how many
  const int cps = sub_len / TC_C;           // chunks per sub-segment
  const int nb = sub0 * sub_len;
  const int ne = min(N, nb + nsb * sub_len);
  const int nch = (ne - nb + TC_C - 1) / TC_C;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
      mbar_init(&bar_phi[s], NCOMP);
    }
    mbar_init(&bar_done, 1);
    mbar_init(&bar_st, 1);
    fence_barrier_init();
    prefetch_tensormap(&maps.q);
    prefetch_tensormap(&maps.k);
    prefetch_tensormap(&maps.v);
    prefetch_tensormap(&maps.g);
    prefetch_tensormap(&maps.o);
    s_abort = 0;
  }
  if (warp == 1) tmem_alloc(&tmem_base, 512);
  if (warp >= 2) {
    const int t = threadIdx.x - 64;
    ones_tile(sm + SS_ONES, t, NCOMP);
    for (int v = t; v < 2 * TILE / 16; v += NCOMP)
      *reinterpret_cast<uint4*>(sm + SS_GAMT + v * 16) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
  }
  auto wt = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
    if (*reinterpret_cast<volatile int*>(&s_abort)) return false;
    if (mbar_wait(bar, parity, WAIT_NS)) return true;
    *reinterpret_cast<volatile int*>(&s_abort) = 1;
    fail(err, code);
    return false;
  };
  // the same, agreed by the whole warp (shuffles and TMEM loads follow)
  auto wtu = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
    return __all_sync(0xffffffffu, wt(bar, parity, code));
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();
  const uint32_t tm = tmem_base;  // sub-segment j: S~ at column 256 j, R~ at 256 j + 128

  if (warp == 0) {
    if (lane == 0) {
      // Without decay the stage's phi(Q), phi(K) and gt tiles are the
      // workspace rows: TMA stores write them once the compute warps are done
      // with the chunk (rows past N are clipped), and a stage is reloaded only
      // after its stores have read it.
      auto store_ws = [&](int c) {
        const int s = c & 1;
        if (!wt(&bar_phi[s], (c >> 1) & 1, 45)) return false;
        const uint8_t* st = sm + s * SS_STAGE;
        const int n0 = nb + c * TC_C;
        tma_store_3d(&maps.fq, st, 0, n0, bh);
        tma_store_3d(&maps.fk, st + TILE, 0, n0, bh);
        tma_store_3d(&maps.gt, st + 3 * TILE, 0, n0, bh);
        bulk_commit();
        return true;
      };
      int issued = 0;
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        const int s = c & 1;
        if (c >= 2) {
          if (!(ok = wt(&bar_empty[s], ((c >> 1) - 1) & 1, 41))) break;
          if (!DECAY) bulk_wait_read();  // chunk c-2's stores (the only ones in flight) have read the stage
        }
        if (c == 1 && !(ok = wt(&bar_full[0], 0, 41))) break;  // chunk 0's tiles first, alone
        uint8_t* st = sm + s * SS_STAGE;
        const int n0 = nb + c * TC_C;
        mbar_arrive_expect_tx(&bar_full[s], 5 * TILE);
        tma_load_3d(st, &maps.q, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + TILE, &maps.k, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + 2 * TILE, &maps.v, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + 3 * TILE, &maps.g, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + 4 * TILE, &maps.o, &bar_full[s], 0, n0, bh);
        ++issued;
        if (!DECAY && c >= 1) ok = store_ws(c - 1);
      }
      if (!DECAY && ok && nch > 0) store_ws(nch - 1);
      for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)  // no load in flight at exit
        mbar_wait(&bar_full[i & 1], (i >> 1) & 1, WAIT_NS);
      bulk_wait_read();
      mbar_arrive(&bar_st);  // stage 0 may take the records
      bulk_wait_all();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t ones = smem_u32(sm + SS_ONES);
      for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
        const uint32_t q = smem_u32(sm + s * SS_STAGE), k = q + TILE, v = q + 2 * TILE, g = q + 3 * TILE;
        const uint32_t gt = smem_u32(sm + SS_GAMT + s * TILE);
        const uint64_t dQ = sdesc(q, 16, 1024), dK = sdesc(k, 16, 1024);
        const uint64_t dVt = sdesc(v, ones - v, 1024), dGt = sdesc(g, gt - g, 1024);
        if (!wt(&bar_phi[s], (c >> 1) & 1, 42)) break;
        tc_fence_after();
        const uint32_t tj = tm + 256 * static_cast<uint32_t>(c / cps);  // the chunk's sub-segment
        const bool first = c % cps == 0;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // S~ += phi(K)^T [V | 1]
          mma_bf16(tj, dadd(dK, kk * 2048), dadd(dVt, kk * 2048), ID_ST80, !first || kk > 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // R~ += phi(Q)^T [gt | gam]
          mma_bf16(tj + 128, dadd(dQ, kk * 2048), dadd(dGt, kk * 2048), ID_ST80, !first || kk > 0);
        mma_commit(&bar_empty[s]);
      }
      mma_commit(&bar_done);  // also after an early exit: every issued MMA has finished
    }
  } else {
    const int t = threadIdx.x - 64;  // 0 .. 511: vectors t and t + 512 of each tile
    const long hb = static_cast<long>(bh) * N;
    auto load_inv = [&](int c, float* inv) {  // 1 / den of the two rows, one chunk ahead
      const int n0 = nb + c * TC_C;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = (t >> 3) + 64 * i;
        inv[i] = (c < nch && n0 + r < ne) ? den[hb + n0 + r] : 1.f;
      }
    };
    float dn_next[2];
    load_inv(0, dn_next);
    for (int c = 0; c < nch; ++c) {
      const int s = c & 1;
      const int n0 = nb + c * TC_C;
      const int valid = min(TC_C, ne - n0);
      const int nbj = nb + (c / cps) * sub_len, nej = min(N, nbj + sub_len);  // the chunk's sub-segment
      uint8_t* st = sm + s * SS_STAGE;
      const float inv[2] = {1.f / dn_next[0], 1.f / dn_next[1]};
      load_inv(c + 1, dn_next);
      if (wtu(&bar_full[s], (c >> 1) & 1, 43)) {
        uint4 x[3][2], o[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int v = t + i * NCOMP;
          x[0][i] = *reinterpret_cast<const uint4*>(st + v * 16);             // Q
          x[1][i] = *reinterpret_cast<const uint4*>(st + TILE + v * 16);      // K
          x[2][i] = *reinterpret_cast<const uint4*>(st + 3 * TILE + v * 16);  // dout
          o[i] = *reinterpret_cast<const uint4*>(st + 4 * TILE + v * 16);     // out
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int v = t + i * NCOMP, r = v >> 3, lc = (v & 7) ^ (r & 7);
          const bool rv = r < valid;
          const long gofs = (hb + n0 + r) * 64 + lc * 8;
          // phi(Q), phi(K): in place (zero on padded features of a head
          // narrower than 64: phi(0) = 1 would add them); with decay also to
          // the workspace, scaled by chunk (the TMA stores copy the tiles else)
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint4 f = rv && lc < dch ? (feat ? x[k][i] : phi_vec(x[k][i])) : make_uint4(0u, 0u, 0u, 0u);
            if (DECAY) {
              // the workspace takes chunk-scaled rows for the main pass (phi(Q) gamma^r,
              // phi(K) gamma^(127-r)); the records take sub-segment-scaled ones (the
              // reverse sums from the sub-segment's start, the forward sums to its end)
              const float fw = exp2f(lg * static_cast<float>(k == 0 ? r : 127 - r));
              const float fs = exp2f(lg * static_cast<float>(k == 0 ? n0 + r - nbj : nej - 1 - n0 - r));
              *reinterpret_cast<uint4*>(st + k * TILE + v * 16) = scale_vec(f, fs);
              if (rv) *reinterpret_cast<uint4*>((k == 0 ? fq_out : fk_out) + gofs) = scale_vec(f, fw);
            } else {
              *reinterpret_cast<uint4*>(st + k * TILE + v * 16) = f;
            }
          }
          // gt = dout / den in place and to the workspace; gam = -(gt . out)
          float dot = 0.f;
          uint4 gv = make_uint4(0u, 0u, 0u, 0u);
          if (rv) {
            const uint32_t gw[4] = {x[2][i].x, x[2][i].y, x[2][i].z, x[2][i].w};
            const uint32_t ow[4] = {o[i].x, o[i].y, o[i].z, o[i].w};
            uint32_t rw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float g0 = __uint_as_float(gw[j] << 16) * inv[i];
              const float g1 = __uint_as_float(gw[j] & 0xffff0000u) * inv[i];
              dot = fmaf(g0, __uint_as_float(ow[j] << 16), dot);
              dot = fmaf(g1, __uint_as_float(ow[j] & 0xffff0000u), dot);
              rw[j] = pack_bf16(g0, g1);
            }
            gv = make_uint4(rw[0], rw[1], rw[2], rw[3]);
            if (DECAY) *reinterpret_cast<uint4*>(gt_out + gofs) = gv;
          }
          *reinterpret_cast<uint4*>(st + 3 * TILE + v * 16) = gv;
          dot += __shfl_xor_sync(0xffffffffu, dot, 1);  // the 8 vectors of row r
          dot += __shfl_xor_sync(0xffffffffu, dot, 2);  // sit in 8 consecutive lanes
          dot += __shfl_xor_sync(0xffffffffu, dot, 4);
          if ((t & 7) == 0) {
            const float gm = rv ? -dot : 0.f;
            *reinterpret_cast<bf16*>(sm + SS_GAMT + s * TILE + r * 128 + ((r & 7) << 4)) =
                __float2bfloat16_rn(gm);
            if (rv) gam[hb + n0 + r] = gm;
          }
        }
      }
      fence_proxy_async();
      mbar_arrive(&bar_phi[s]);
    }
    // the partial states [S | z | R | r] of each sub-segment: TMEM -> shared
    // memory (stage 0, one record after the other) -> one bulk copy each
    const int qd = warp & 3, wq = (warp - 2) >> 2;  // lane quarter, warp within it
    const uint32_t lq = static_cast<uint32_t>(32 * qd) << 16;
    const int srow = 16 * qd + lane;
    float* stg = reinterpret_cast<float*>(sm);
    static_assert(2 * REC * 4 <= SS_STAGE, "two records fit stage 0");
    if (wtu(&bar_done, 0, 44) && wtu(&bar_st, 0, 46)) {
      tc_fence_after();
      for (int blk = wq; blk < 10 * nsb; blk += 4) {  // 16-column blocks: S~ 0-4, R~ 5-9 per record
        const int j = blk / 10, which = (blk % 10) / 5, col = (blk % 5) * 16;
        float sv[16];
        tmem_ldn<1>(tm + 256 * j + which * 128 + lq + col, sv);
        float* base = stg + j * REC + which * (DM + 64);
        if (lane < 16) {
          if (col < 64) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<float4*>(base + srow * 64 + col + j) =
                  make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
          } else {
            base[DM + srow] = sv[0];  // the vector column
          }
        }
      }
    }
    fence_proxy_async();
    compute_sync();
    if (t == 0 && !*reinterpret_cast<volatile int*>(&s_abort)) {
      for (int j = 0; j < nsb; ++j)
        bulk_store(rec + (static_cast<long>(bh) * nsub + sub0 + j) * REC, stg + j * REC, REC * 4);
      bulk_commit();
      bulk_wait_all();
    }
  }
  if (warp == 1 && lane == 0) mbar_wait(&bar_done, 0, WAIT_NS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tm, 512);
}

struct BwdPlan {
  int g;           // chunks per sub-segment
  int sub_len;     // tokens per sub-segment
  int nsub;        // sub-segments per (b, h)
  int spc;         // sub-segments per state-pass CTA (1 or 2)
  int nchh;        // chunks per (b, h)
  int n0, upc0;    // main pass, role 0 (dq): CTAs and sub-segments per CTA
  int n1, upc1;    // role 1 (dk, dv)
};

// The runs of the main pass: one wave of CTAs, the dq role on n0 of them and
// the dk / dv role on the rest, each run upc whole sub-segments of the flat
// (b, h, sub-segment) order.  The sub-segment length g and the split are
// chosen to minimise the state pass's time plus the longest run, in units of
// a dq chunk (about 2.4 us on the 3072-token, 64-wide workload): a dk / dv
// chunk weighs 1.4 (3.4 us), each record a run adds up at its start 0.1, a
// state-pass chunk 1.3 and a state-pass CTA's fixed cost 1.
BwdPlan bwd_plan(int BH, int N) {
  constexpr double W1 = 1.4, WREC = 0.1, WS = 1.3, FS = 1.0;
  const int slots = sm_count() < 2 ? 2 : sm_count();
  // the last plan of this thread (every backward call and workspace query asks)
  thread_local int c_bh = -1, c_n = -1, c_slots = -1;
  thread_local BwdPlan c_plan{};
  if (BH == c_bh && N == c_n && slots == c_slots) return c_plan;
  const int nchh = (N + TC_C - 1) / TC_C;
  auto cdiv = [](long a, long b) { return (a + b - 1) / b; };
  BwdPlan best{};
  double best_cost = 1e300;
  // For a given number of sub-segments the shortest length that gives it is
  // the best one (the costs grow with g), so only those lengths are tried
  // (about 2 sqrt(nchh) of them), longest first: fewer records on a tie.
  for (int k = 1; k <= nchh; ++k) {
    const int g = static_cast<int>(cdiv(nchh, k));
    const int nsub = static_cast<int>(cdiv(nchh, g));
    if (nsub != k) continue;  // no sub-segment length gives k of them
    const long U = static_cast<long>(BH) * nsub;
    const int spc = U <= slots ? 1 : 2;
    const double state = static_cast<double>(cdiv(BH * cdiv(nsub, spc), slots)) * (FS + WS * spc * g);
    const long lo0 = cdiv(U, slots - 1);  // leave at least one CTA to role 1
    for (long upc0 = lo0; upc0 <= U && upc0 <= lo0 + 64; ++upc0) {
      const long n0 = cdiv(U, upc0);
      const long upc1 = cdiv(U, slots - n0);
      const long n1 = cdiv(U, upc1);
      const double cost = state + WREC * nsub +
                          std::max(static_cast<double>(upc0 * g), W1 * static_cast<double>(upc1 * g));
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best.g = g;
        best.nsub = nsub;
        best.n0 = static_cast<int>(n0);
        best.upc0 = static_cast<int>(upc0);
        best.n1 = static_cast<int>(n1);
        best.upc1 = static_cast<int>(upc1);
      }
    }
  }
  best.nchh = nchh;
  best.sub_len = best.g * TC_C;
  // state pass: one sub-segment per CTA while that fits one wave, else two
  // (two accumulator pairs fill the 512 tensor-memory columns)
  best.spc = static_cast<long>(BH) * best.nsub <= slots ? 1 : 2;
  c_bh = BH;
  c_n = N;
  c_slots = slots;
  c_plan = best;
  return best;
}

struct BwdWs {
  float* rec;
  bf16 *gt, *fq, *fk;
  float* gam;
  size_t floats;
};

BwdWs bwd_ws(float* ws, int BH, int N, const BwdPlan& pl) {
  BwdWs w;
  const size_t tok = static_cast<size_t>(BH) * N;
  w.rec = ws;
  size_t off = static_cast<size_t>(BH) * pl.nsub * REC;
  w.gt = reinterpret_cast<bf16*>(ws + off);
  off += tok * 32;
  w.fq = reinterpret_cast<bf16*>(ws + off);
  off += tok * 32;
  w.fk = reinterpret_cast<bf16*>(ws + off);
  off += tok * 32;
  w.gam = ws + off;
  w.floats = off + tok;
  return w;
}

}  // namespace

// workspace: records [BH][nsub][REC] | gt, phi(Q), phi(K) bf16 [BH][N][64] |
// gam fp32 [BH][N]
size_t causal_bwd_tc_ws_floats(const Shape& s) {
  const int BH = s.B * s.H;
  return bwd_ws(nullptr, BH, s.N, bwd_plan(BH, s.N)).floats;
}

int causal_bwd_tc_launches(const Shape&) { return 2; }

cudaError_t causal_bwd_tc(const void* q, const void* k, const void* v, const void* out,
                          const float* den, const void* dout, void* dq, void* dk, void* dv,
                          float* ws, const Shape& s, cudaStream_t st, bool feat, float gamma) {
  const int BH = s.B * s.H;
  const BwdPlan pl = bwd_plan(BH, s.N);
  const BwdWs w = bwd_ws(ws, BH, s.N, pl);
  BwdMaps m;
  // the caller's tensors at their own widths (loads zero-fill to 64, stores
  // write only D or M columns); the workspace's phi(Q), phi(K), gt stay 64 wide
  if (!make_bf16_map(&m.q, q, BH, s.N, s.D) || !make_bf16_map(&m.k, k, BH, s.N, s.D) ||
      !make_bf16_map(&m.v, v, BH, s.N, s.M) || !make_bf16_map(&m.g, dout, BH, s.N, s.M) ||
      !make_bf16_map(&m.o, out, BH, s.N, s.M) || !make_bf16_map(&m.fq, w.fq, BH, s.N) ||
      !make_bf16_map(&m.fk, w.fk, BH, s.N) || !make_bf16_map(&m.gt, w.gt, BH, s.N) ||
      !make_bf16_map(&m.dq, dq, BH, s.N, s.D) || !make_bf16_map(&m.dk, dk, BH, s.N, s.D) ||
      !make_bf16_map(&m.dv, dv, BH, s.N, s.M))
    return cudaErrorInvalidValue;
  StateMaps smap;
  smap.q = m.q;
  smap.k = m.k;
  smap.v = m.v;
  smap.g = m.g;
  smap.o = m.o;
  smap.fq = m.fq;
  smap.fk = m.fk;
  smap.gt = m.gt;
  cudaError_t e;
  const float lg = gamma == 1.f ? 0.f : log2f(gamma);
  auto kstate = lg != 0.f ? k_tc_bwd_state<true> : k_tc_bwd_state<false>;
  auto kmain = lg != 0.f ? k_tc_bwd_main<true> : k_tc_bwd_main<false>;
  if ((e = cudaFuncSetAttribute(kstate, cudaFuncAttributeMaxDynamicSharedMemorySize, SS_SMEM)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(kmain, cudaFuncAttributeMaxDynamicSharedMemorySize, M_SMEM)) !=
      cudaSuccess)
    return e;
  const int nstate = (pl.nsub + pl.spc - 1) / pl.spc;
  if ((e = launch_pdl(kstate, dim3(nstate, BH), dim3(NTHR), SS_SMEM, st, smap, den, w.gam,
                      w.gt, w.fq, w.fk, w.rec, s.N, pl.sub_len, pl.nsub, pl.spc, s.D / 8,
                      feat ? 1 : 0, lg, status_word())) != cudaSuccess)
    return e;
  if ((e = launch_pdl(kmain, dim3(pl.n0 + pl.n1), dim3(NTHR), M_SMEM, st, m,
                      static_cast<const float*>(w.rec), static_cast<const float*>(w.gam), s.N,
                      pl.nchh, pl.g, pl.nsub, BH, pl.n0, pl.upc0, pl.upc1, feat ? 1 : 0, lg,
                      status_word())) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace la
