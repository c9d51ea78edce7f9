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
//   S += phi(K)^T V, z += phi(K)^T 1;  R += phi(Q)^T gt, r += phi(Q)^T gam
// with P = bf16(mask(phi(Q) phi(K)^T)) and dP = bf16(mask(dA)); then
// dq = grad_phiQ * phi'(Q), dk = grad_phiK * phi'(K), and phi'(x) = min(phi(x), 1).
//
// Two passes.  MODE 0 (one CTA per sub-segment of whole 128-token chunks)
// reads q, k, v, dout, out and den once; it stores phi(Q), phi(K) and
// gt = dout / den (bf16) and gam (fp32) in the workspace, and the
// sub-segment's partial S, z, R, r.  MODE 1 runs two roles per segment
// (grid z): role 0 walks forward carrying S, z and writes dq; role 1 walks
// backward carrying R, r and writes dk and dv.  Each CTA first adds up the
// partial states of the sub-segments before (role 0) or after (role 1) it.
// Every product, including the vector sums z and r (against a ones column
// or the gam column), runs on tcgen05 with TMA-fed operands; dq, dk and dv
// are staged in shared memory and written with TMA stores.
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

// MODE 0 shared memory: stages of q, k, v, dout, out; two gt tiles; ones; two gam tiles
constexpr int S_STAGE = 5 * TILE;
constexpr int S_GT = NST * S_STAGE;
constexpr int S_ONES = S_GT + 2 * TILE;
constexpr int S_GAMT = S_ONES + 1024;
constexpr int S_SMEM = S_GAMT + 2 * 2048 + 1024;
// MODE 1 shared memory: stages of phi(Q), phi(K), v, gt; P; dP; two bf16
// state tiles; ones; two gam tiles
constexpr int M_STAGE = 4 * TILE;
constexpr int M_P = NST * M_STAGE;
constexpr int M_DP = M_P + 2 * TILE;
constexpr int M_RP = M_DP + 2 * TILE;
constexpr int M_ONES = M_RP + 2 * 8192;
constexpr int M_GAMT = M_ONES + 1024;
constexpr int M_SMEM = M_GAMT + 2 * 2048 + 1024;
static_assert(S_SMEM + 2048 <= 232448 && M_SMEM + 2048 <= 232448, "shared memory");

// The ones tile (1 KB, every element 1) and two zeroed gam tiles (2 KB each): B
// operands of the N = 8 products that give z = phi(K)^T 1 and r = phi(Q)^T gam.
__device__ __forceinline__ void init_vec_tiles(uint8_t* ones, uint8_t* gamt, int t) {
  for (int v = t; v < 1024 / 16; v += NCOMP)
    *reinterpret_cast<uint4*>(ones + v * 16) =
        make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
  for (int v = t; v < 2 * 2048 / 16; v += NCOMP)
    *reinterpret_cast<uint4*>(gamt + v * 16) = make_uint4(0u, 0u, 0u, 0u);
}

// gam_i into row 0, column i of the gam tile (K-major, 128-byte swizzle,
// two 64-column atoms; row 0 is not permuted by the swizzle).
__device__ __forceinline__ void put_gam(uint8_t* gamt, int i, float g) {
  *reinterpret_cast<bf16*>(gamt + (i >> 6) * 1024 + (i & 63) * 2) = __float2bfloat16_rn(g);
}

// Role 1: the masked bf16 rows of dA (+ gam) and of A for this warpgroup's
// KW keys from key0, loaded together so that one wait covers both.
__device__ __forceinline__ void mask2_cols(uint32_t tda, uint32_t ta, float add, uint8_t* ddst,
                                           uint8_t* adst, int row, int key0) {
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
    d[i] = keep ? d[i] + add : 0.f;
    a[i] = keep ? a[i] : 0.f;
  }
  tile_put_cols<KW>(ddst, row, key0 & 63, d);
  tile_put_cols<KW>(adst, row, key0 & 63, a);
}

struct BwdMaps {
  CUtensorMap q, k, v, g, o;  // MODE 0 inputs
  CUtensorMap fq, fk, gt;     // MODE 0 outputs, MODE 1 inputs
  CUtensorMap dq, dk, dv;     // MODE 1 outputs (TMA stores)
};

template <int MODE>
__global__ void __launch_bounds__(NTHR, 1)
    k_tc_bwd(const __grid_constant__ BwdMaps maps, const float* __restrict__ den,
             float* __restrict__ rec, float* __restrict__ gam, bf16* __restrict__ gt_out,
             bf16* __restrict__ fq_out, bf16* __restrict__ fk_out, int N, int seg_len, int nsub,
             int subs_per_seg, int* err) {
  const int p = blockIdx.x, bh = blockIdx.y;
  const int role = MODE == 0 ? 2 : static_cast<int>(blockIdx.z);  // 0 dq, 1 dk/dv, 2 partials
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  __shared__ uint64_t bar_full[NST], bar_empty[NST];
  __shared__ uint64_t bar_in, bar_a, bar_p, bar_rp, bar_o, bar_s, bar_s2[2];
  __shared__ uint32_t tmem_base;
  __shared__ float s_vec[2][64];    // carried z (role 0) or r (role 1) before chunk c, by c & 1
  __shared__ float s_dot[NWG][TC_C];  // MODE 0: partial dot products for gam
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p * seg_len;
  const int ne = min(N, nb + seg_len);
  const int nch = (ne - nb + TC_C - 1) / TC_C;
  const int stage_bytes = MODE == 0 ? S_STAGE : M_STAGE;
  uint8_t* ones = sm + (MODE == 0 ? S_ONES : M_ONES);
  uint8_t* gamt = sm + (MODE == 0 ? S_GAMT : M_GAMT);  // two 2 KB tiles, by chunk parity

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bar_full[s], 1);
      // MODE 0: the MMAs; MODE 1: the MMAs and every compute thread
      // (the epilogues read phi from the stage)
      mbar_init(&bar_empty[s], MODE == 0 ? 1 : 1 + NCOMP);
    }
    mbar_init(&bar_in, NCOMP);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_p, NCOMP);
    mbar_init(&bar_rp, NCOMP);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_s2[0], 1);
    mbar_init(&bar_s2[1], 1);
    fence_barrier_init();
    s_abort = 0;
  }
  if (warp == 1) tmem_alloc(&tmem_base, 512);
  if (warp >= 2) {
    init_vec_tiles(ones, gamt, threadIdx.x - 64);
    fence_proxy_async();
  }
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
  grid_dep_wait();  // the previous kernel's outputs are visible from here on
  const uint32_t tm = tmem_base;
  const uint32_t TA = tm, TDA = tm + 128, TG1 = tm + 256, TG2 = tm + 320, TST = tm + 384;
  const uint32_t TV = tm + 448, TV2 = tm + 464;  // N = 8 vector accumulators (z / r)
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
        if (MODE == 0) {
          tma_load_3d(st, &maps.q, &bar_full[s], 0, n0, bh);
          tma_load_3d(st + TILE, &maps.k, &bar_full[s], 0, n0, bh);
          tma_load_3d(st + 2 * TILE, &maps.v, &bar_full[s], 0, n0, bh);
          tma_load_3d(st + 3 * TILE, &maps.g, &bar_full[s], 0, n0, bh);
          tma_load_3d(st + 4 * TILE, &maps.o, &bar_full[s], 0, n0, bh);
        } else {
          tma_load_3d(st, &maps.fq, &bar_full[s], 0, n0, bh);
          tma_load_3d(st + TILE, &maps.fk, &bar_full[s], 0, n0, bh);
          tma_load_3d(st + 2 * TILE, &maps.v, &bar_full[s], 0, n0, bh);
          tma_load_3d(st + 3 * TILE, &maps.gt, &bar_full[s], 0, n0, bh);
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    // Per chunk: A and dA, then the carried-state update (it only needs the
    // stage and frees the compute warps to stage the next state while the
    // gradient products run), then the gradient products.
    if (lane == 0) {
      constexpr uint32_t ID_AA = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_G = idesc_bf16(128, 64, false, false);
      constexpr uint32_t ID_GMN = idesc_bf16(128, 64, false, true);
      constexpr uint32_t ID_GTT = idesc_bf16(128, 64, true, true);
      constexpr uint32_t ID_ST = idesc_bf16(64, 64, true, true);
      constexpr uint32_t ID_V = idesc_bf16(64, 8, true, false);  // phi^T x (ones | gam)
      const uint64_t dP0 = sdesc(smem_u32(sm + M_P), TILE, 1024);
      const uint64_t dDP = sdesc(smem_u32(sm + M_DP), 16, 1024);
      const uint64_t dDPT = sdesc(smem_u32(sm + M_DP), TILE, 1024);
      const uint64_t dOnes = sdesc(smem_u32(ones), 16, 1024);
      for (int c = 0; c < nch; ++c) {
        const int s = c % NST;
        const uint32_t qs = smem_u32(sm + s * stage_bytes);
        const uint32_t gs = MODE == 0 ? smem_u32(sm + S_GT + (c & 1) * TILE) : qs + 3 * TILE;
        const uint64_t dQ = sdesc(qs, 16, 1024), dK = sdesc(qs + TILE, 16, 1024);
        const uint64_t dV = sdesc(qs + 2 * TILE, 16, 1024), dG = sdesc(gs, 16, 1024);
        const uint64_t dGam = sdesc(smem_u32(gamt + (c & 1) * 2048), 16, 1024);
        const uint64_t dRP = sdesc(smem_u32(sm + M_RP + (c & 1) * 8192), 16, 1024);
        if (!wt(&bar_in, c & 1, 22)) break;
        tc_fence_after();
        if (MODE == 0) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // S += phi(K)^T V, z += phi(K)^T 1
            mma_bf16(TG1, dadd(dK, kk * 2048), dadd(dV, kk * 2048), ID_ST, 1);
            mma_bf16(TV, dadd(dK, kk * 2048), dadd(dOnes, 32 * (kk & 3)), ID_V, 1);
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // R += phi(Q)^T gt, r += phi(Q)^T gam
            mma_bf16(TST, dadd(dQ, kk * 2048), dadd(dG, kk * 2048), ID_ST, 1);
            mma_bf16(TV2, dadd(dQ, kk * 2048), dadd(dGam, (kk >> 2) * 1024 + 32 * (kk & 3)), ID_V, 1);
          }
          mma_commit(&bar_s2[c & 1]);
          mma_commit(&bar_empty[s]);
          continue;
        }
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
        if (role == 0) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // S += phi(K)^T V, z += phi(K)^T 1
            mma_bf16(TST, dadd(dK, kk * 2048), dadd(dV, kk * 2048), ID_ST, 1);
            mma_bf16(TV, dadd(dK, kk * 2048), dadd(dOnes, 32 * (kk & 3)), ID_V, 1);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // R += phi(Q)^T gt, r += phi(Q)^T gam
            mma_bf16(TST, dadd(dQ, kk * 2048), dadd(dG, kk * 2048), ID_ST, 1);
            mma_bf16(TV, dadd(dQ, kk * 2048), dadd(dGam, (kk >> 2) * 1024 + 32 * (kk & 3)), ID_V, 1);
          }
        }
        mma_commit(&bar_s);
        if (!wt(&bar_p, c & 1, 23)) break;
        tc_fence_after();
        if (role == 0) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dP phi(K)
            mma_bf16(TG1, dadd(dDP, (kk >> 2) * TILE + (kk & 3) * 32), dadd(sdesc(qs + TILE, 16, 1024), kk * 2048),
                     ID_GMN, kk > 0);
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
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // P^T gt
            mma_bf16(TG2, dadd(dP0, kk * 2048), dadd(dG, kk * 2048), ID_GTT, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // + phi(K) R
            mma_bf16(TG2, dadd(dK, 32 * kk), dadd(dRP, kk * 2048), ID_GMN, 1);
        }
        mma_commit(&bar_o);
        mma_commit(&bar_empty[s]);
      }
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
    const long hb = static_cast<long>(bh) * N;
    auto gam_at = [&](int c) {     // gam of this thread's row in chunk c
      const int n0 = nb + chunk_at(c) * TC_C;
      return row < min(TC_C, ne - n0) ? gam[hb + n0 + row] : 0.f;
    };
    if (MODE == 1) {
      // carried state: role 0 sums the records of the sub-segments before this
      // segment (S, z), role 1 those after it (R, r); warpgroup 0 loads it
      if (wg == 0) {
        const int lo = role == 0 ? 0 : (p + 1) * subs_per_seg;
        const int hi = role == 0 ? p * subs_per_seg : nsub;
        const int off = role == 0 ? 0 : DM + 64;
        float sv[64], vv[16];
        for (int j = 0; j < 64; ++j) sv[j] = 0.f;
        for (int j = 0; j < 16; ++j) vv[j] = 0.f;
        for (int pp = lo; pp < hi; ++pp) {
          const float* r0 = rec + (static_cast<long>(bh) * nsub + pp) * REC + off;
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
            vv[0] += r0[DM + srow];
          }
        }
        for (int j = 0; j < 64; j += 16) tmem_st16(TST + lq + j, sv + j);
        for (int j = 1; j < 8; ++j) vv[j] = vv[0];
        tmem_st16(TV + lq, vv);
        tmem_st_wait();
        if (has_s) {
          tile_put_cols<64>(sm + M_RP, srow, 0, sv);
          s_vec[0][srow] = vv[0];
        }
      }
      fence_proxy_async();
      compute_sync();
      tc_fence_before();
      mbar_arrive(&bar_rp);
      // chunk 0 inputs
      const float g0 = gam_at(0);
      wt(&bar_full[0], 0, 25);
      if (role == 1 && wg == 0) {
        put_gam(gamt, row, g0);
        fence_proxy_async();
      }
      mbar_arrive(&bar_in);
    } else {
      if (wg == 0) {
        float zero[16];
        for (int j = 0; j < 16; ++j) zero[j] = 0.f;
        for (int j = 0; j < 64; j += 16) {
          tmem_st16(TG1 + lq + j, zero);
          tmem_st16(TST + lq + j, zero);
        }
        tmem_st16(TV + lq, zero);
        tmem_st16(TV2 + lq, zero);
        tmem_st_wait();
      }
      tc_fence_before();
    }
    float gm = MODE == 1 ? gam_at(0) : 0.f;
    for (int c = 0; c < nch; ++c) {
      const int s = c % NST;
      const int n0 = nb + chunk_at(c) * TC_C;
      const int valid = min(TC_C, ne - n0);
      const bool rv = row < valid;
      uint8_t* st = sm + s * stage_bytes;
      if (MODE == 0) {
        const float dn = rv ? den[hb + n0 + row] : 1.f;
        if (c > 1) {  // gt / gam tiles of parity c & 1 are free once chunk c-2's MMAs finished
          wt(&bar_s2[c & 1], ((c - 2) >> 1) & 1, 24);
          tc_fence_after();
        }
        compute_sync();
        wt(&bar_full[s], (c / NST) & 1, 25);
        uint8_t* gtile = sm + S_GT + (c & 1) * TILE;
        // gt = dout / den on this warpgroup's columns; gam = -(gt . out)
        float g[OW], o[OW];
        tile_row_cols<OW>(st + 3 * TILE, row, c0, g);
        tile_row_cols<OW>(st + 4 * TILE, row, c0, o);
        const float inv = 1.f / dn;
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < OW; ++i) {
          g[i] = rv ? g[i] * inv : 0.f;
          acc = fmaf(g[i], o[i], acc);
        }
        s_dot[wg][row] = acc;
        tile_put_cols<OW>(gtile, row, c0, g);
        if (rv) store_bf16<OW>(gt_out + (hb + n0 + row) * 64 + c0, g);
        phi_tile_store(st, valid, t, fq_out + (hb + n0) * 64);
        phi_tile_store(st + TILE, valid, t, fk_out + (hb + n0) * 64);
        compute_sync();
        if (wg == 0) {
          float dot = 0.f;
#pragma unroll
          for (int w = 0; w < NWG; ++w) dot += s_dot[w][row];
          const float gmv = rv ? -dot : 0.f;
          put_gam(gamt + (c & 1) * 2048, row, gmv);
          if (rv) gam[hb + n0 + row] = gmv;
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_in);
        continue;
      }
      // ------------------------------------------------------------- MODE 1
      // P, dP of chunk c
      wt(&bar_a, c & 1, 26);
      tc_fence_after();
      if (t == 0) bulk_wait_read();  // the previous chunk's output tiles have left P / dP
      compute_sync();
      if (role == 1)
        mask2_cols(TDA + lq + k0, TA + lq + k0, gm, sm + M_DP + (k0 >> 6) * TILE,
                   sm + M_P + (k0 >> 6) * TILE, row, k0);
      else
        mask_cols<KW>(TDA + lq + k0, gm, sm + M_DP + (k0 >> 6) * TILE, row, k0);
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_p);
      // inputs of chunk c+1 (the tensor cores may start on it)
      float gm_next = 0.f;
      if (c + 1 < nch) {
        gm_next = gam_at(c + 1);
        wt(&bar_full[(c + 1) % NST], ((c + 1) / NST) & 1, 25);
        if (role == 1 && wg == 0) {
          put_gam(gamt + ((c + 1) & 1) * 2048, row, gm_next);
          fence_proxy_async();
        }
        mbar_arrive(&bar_in);
      }
      // carried state for chunk c+1 (after this chunk's update)
      if (c + 1 < nch) {
        wt(&bar_s, c & 1, 28);
        tc_fence_after();
        float sv[OW], vv[16];
        tmem_ldn<OW / 16>(TST + lq + c0, sv);
        tmem_ldn<1>(TV + lq, vv);
        if (has_s) {
          tile_put_cols<OW>(sm + M_RP + ((c + 1) & 1) * 8192, srow, c0, sv);
          if (wg == 0) s_vec[(c + 1) & 1][srow] = vv[0];
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_rp);
      }
      // gradients of chunk c, staged in the free P / dP tiles and TMA-stored
      wt(&bar_o, c & 1, 27);
      tc_fence_after();
      {
        const float* vec = s_vec[c & 1];
        float gv[OW], x[OW];
        tmem_ldn<OW / 16>(TG1 + lq + c0, gv);
        if (role == 0) {  // dq = (grad_phiQ + gam z_prev) * phi'(Q)
          tile_row_cols<OW>(st, row, c0, x);
#pragma unroll
          for (int i = 0; i < OW; ++i) gv[i] = (gv[i] + gm * vec[c0 + i]) * fminf(x[i], 1.f);
          tile_put_cols<OW>(sm + M_DP, row, c0, gv);
        } else {          // dk = (grad_phiK + r_next) * phi'(K), dv
          tile_row_cols<OW>(st + TILE, row, c0, x);
#pragma unroll
          for (int i = 0; i < OW; ++i) gv[i] = (gv[i] + vec[c0 + i]) * fminf(x[i], 1.f);
          tile_put_cols<OW>(sm + M_P, row, c0, gv);
          tmem_ldn<OW / 16>(TG2 + lq + c0, gv);
          tile_put_cols<OW>(sm + M_P + TILE, row, c0, gv);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_empty[s]);  // this thread is done with the stage
      compute_sync();              // s_vec[c & 1] is free again; the output tiles are complete
      if (t == 0) {
        if (role == 0) {
          tma_store_3d(&maps.dq, sm + M_DP, 0, n0, bh);
        } else {
          tma_store_3d(&maps.dk, sm + M_P, 0, n0, bh);
          tma_store_3d(&maps.dv, sm + M_P + TILE, 0, n0, bh);
        }
        bulk_commit();
      }
      gm = gm_next;
    }
    if (MODE == 1 && t == 0) bulk_wait_all();
    if (MODE == 0) {
      bool done = true;
      for (int c = max(0, nch - 2); c < nch; ++c)  // the last two state updates, in order
        done = wt(&bar_s2[c & 1], (c >> 1) & 1, 29) && done;
      if (done) {
        tc_fence_after();
        float* r0 = rec + (static_cast<long>(bh) * nsub + p) * REC;
        float sv[OW], vv[16];
        tmem_ldn<OW / 16>(TG1 + lq + c0, sv);
        if (has_s)
          for (int j = 0; j < OW; ++j) r0[srow * 64 + c0 + j] = sv[j];
        tmem_ldn<OW / 16>(TST + lq + c0, sv);
        if (has_s)
          for (int j = 0; j < OW; ++j) r0[DM + 64 + srow * 64 + c0 + j] = sv[j];
        if (wg < 2) {
          tmem_ldn<1>((wg == 0 ? TV : TV2) + lq, vv);
          if (has_s) r0[(wg == 0 ? DM : 2 * DM + 64) + srow] = vv[0];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tm, 512);
}

struct BwdPlan {
  SegPlan main;   // segments of the second pass (two roles each)
  int subs;       // sub-segments per segment in the first pass
  int sub_len;    // tokens per sub-segment
  int nsub;       // sub-segments per (b, h)
};

BwdPlan bwd_plan(int BH, int N) {
  BwdPlan b;
  b.main = tc_plan(2 * BH, N);
  const int per = b.main.seg_len / TC_C;
  b.subs = 1;
  for (int f = per; f >= 1; --f)
    if (per % f == 0 && static_cast<long>(b.main.nseg) * f * BH <= 152) {
      b.subs = f;
      break;
    }
  b.sub_len = b.main.seg_len / b.subs;
  b.nsub = (N + b.sub_len - 1) / b.sub_len;
  return b;
}

struct BwdWs {
  float* rec;
  bf16 *gt, *fq, *fk;
  float* gam;
  int* err;
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
  off += tok;
  w.err = reinterpret_cast<int*>(ws + off);
  w.floats = off + 4;
  return w;
}

}  // namespace

// workspace: records [BH][nsub][REC] | gt, phi(Q), phi(K) bf16 [BH][N][64] |
// gam fp32 [BH][N] | status word
size_t causal_bwd_tc_ws_floats(const Shape& s) {
  const int BH = s.B * s.H;
  return bwd_ws(nullptr, BH, s.N, bwd_plan(BH, s.N)).floats;
}

int causal_bwd_tc_launches(const Shape&) { return 2; }

cudaError_t causal_bwd_tc(const void* q, const void* k, const void* v, const void* out,
                          const float* den, const void* dout, void* dq, void* dk, void* dv,
                          float* ws, const Shape& s, cudaStream_t st) {
  const int BH = s.B * s.H;
  const BwdPlan pl = bwd_plan(BH, s.N);
  const BwdWs w = bwd_ws(ws, BH, s.N, pl);
  BwdMaps m;
  if (!make_bf16_map(&m.q, q, BH, s.N) || !make_bf16_map(&m.k, k, BH, s.N) ||
      !make_bf16_map(&m.v, v, BH, s.N) || !make_bf16_map(&m.g, dout, BH, s.N) ||
      !make_bf16_map(&m.o, out, BH, s.N) || !make_bf16_map(&m.fq, w.fq, BH, s.N) ||
      !make_bf16_map(&m.fk, w.fk, BH, s.N) || !make_bf16_map(&m.gt, w.gt, BH, s.N) ||
      !make_bf16_map(&m.dq, dq, BH, s.N) || !make_bf16_map(&m.dk, dk, BH, s.N) ||
      !make_bf16_map(&m.dv, dv, BH, s.N))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_tc_bwd<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                S_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_tc_bwd<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                M_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaMemsetAsync(w.err, 0, sizeof(int), st)) != cudaSuccess) return e;
  if ((e = launch_pdl(k_tc_bwd<0>, dim3(pl.nsub, BH, 1), dim3(NTHR), S_SMEM, st, m, den, w.rec,
                      w.gam, w.gt, w.fq, w.fk, s.N, pl.sub_len, pl.nsub, pl.subs, w.err)) !=
      cudaSuccess)
    return e;
  if ((e = launch_pdl(k_tc_bwd<1>, dim3(pl.main.nseg, BH, 2), dim3(NTHR), M_SMEM, st, m, den,
                      w.rec, w.gam, w.gt, w.fq, w.fk, s.N, pl.main.seg_len, pl.nsub, pl.subs,
                      w.err)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace la
