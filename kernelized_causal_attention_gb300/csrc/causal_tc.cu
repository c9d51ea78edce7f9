// Causal linear attention on the 5th-generation tensor cores (tcgen05), for
// bf16 inputs with D, M in {16, 32, 64} and fp32 accumulation in tensor
// memory.  Heads narrower than 64 use the same 64-wide tiles: the loads fill
// the missing columns with zeros and phi is zeroed on those features.
//
// Method: "Transformers are RNNs" (part 2/3), §3.3 eq. 9-12.
//
// GB300 design (not the pages'): each (b, h) sequence is cut into segments of
// whole 128-token chunks, one CTA per segment (one CTA per SM).  The value
// matrix is augmented with a column of ones, V~ = [V | 1], so one accumulator
// carries both the state and the normaliser, S~ = [S | z] = sum phi(K_j) V~_j^T,
// and every product that yields a numerator yields its denominator in column 64:
//   A    = phi(Q) phi(K)^T                        (128 x 128, K = 64)
//   P    = bf16(mask(A))                           (written over A in TMEM)
//   O~   = P V~ + phi(Q) bf16(S~_prev)            (128 x 80)  -> out = O~[:, :64] / O~[:, 64]
//   S~  += phi(K)^T V~                             (64 x 80, carried across chunks)
// Two kernels.  The state pass (one CTA per segment but the last) streams the
// segment's K and V through a ring deep enough to hold all of it and leaves
// the segment's partial S~ in the workspace.  The main pass starts each
// segment from the sum of the partial states before it and runs the chunks
// as a software pipeline over warp-specialised roles:
//   warp 0       TMA producer (K, V per chunk in a four-stage ring, Q in a
//                three-slot ring that turns over as soon as phi(Q) is taken)
//   warp 1       MMA issuer: A(c+1) may be issued before O~(c) and S~(c), so
//                the tensor cores compute the next chunk's scores while the
//                mask warpgroup works on the current one
//   warps 2-9    phi of the chunks ahead: phi(Q) into tensor memory (the A
//                operand of both Q products), phi(K) in place in shared memory
//   warps 10-13  mask: P(c) over A(c) in TMEM (two A/P buffers; O~(c) then
//                takes the upper columns of the same buffer)
//   warps 14-17  epilogue of O~(c) straight to global memory, then
//                S~_prev(c+1) in bf16 for the next chunk's read-out
// and the issuer polls for whichever product can go next, so a late phi never
// holds back a read-out.
//
// Variants on the same kernels.  feat: q and k already hold features (the
// degree-2 polynomial map), so no phi is applied.  DECAY (the RetNet decay
// gamma of "Linear Attention/zh", variants; a template flag, so the plain
// kernels keep their code): key j' of a chunk is scaled by gamma^(127-j') as
// phi is applied, the mask multiplies by the constant gamma^-128, so
// P_ij = gamma^-(j'+1) A_ij and output row i' comes out gamma^-(i'+1) times
// the decayed one -- out's quotient cancels that and den takes it back -- and
// the epilogue writes gamma^128 S~ back to tensor memory before the next
// chunk's keys; the state pass scales key j by gamma^(segment end - 1 - j)
// and the record sum weights each record by its distance.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tc_chunk.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcc;

constexpr int TC_MA = 80;  // augmented value width [V | 1 | 0 ...]

// shared memory of the main pass (offsets from a 1024-aligned base): a ring
// of K, V stages and a shorter ring of Q tiles (a Q tile is free once phi(Q)
// is in tensor memory), the ones tile and two bf16 S~_prev tiles
constexpr int KNS = 4;                     // K, V ring stages
constexpr int QNS = 3;                     // Q ring slots
constexpr int F_KV = 0;                    // [KNS][K | V]
constexpr int F_Q = F_KV + KNS * 2 * TILE;
constexpr int F_ONES = F_Q + QNS * TILE;   // [128][64], column 0 = 1
constexpr int F_SP = F_ONES + TILE;        // two bf16 S~_prev (by chunk parity), each
                                           // [64 d][64] then [64 d][z, 0...]
constexpr int F_SCR = F_KV + (KNS - 1) * 2 * TILE;  // fp32 [64][80] initial state, in the last
                                                    // K, V stage before its first load
constexpr int F_SMEM = F_SP + 4 * 8192 + 1024;
// shared memory of the state pass: a ring of K, V stages and the ones tile;
// the fp32 partial state is staged in stage 0 once every product is done
constexpr int SNST = 6;
constexpr int S_STAGE = 2 * TILE;
constexpr int S_ONES = SNST * S_STAGE;
constexpr int S_REC = 0;
constexpr int S_SMEM = S_ONES + TILE + 1024;
static_assert(F_SMEM <= 232448 && S_SMEM <= 232448, "shared memory");

// tensor-memory columns of the main pass
constexpr uint32_t T_BUF = 144;  // per A buffer: A (128 columns), later P (0-63) and O~ (64-143)
constexpr uint32_t T_S = 288;    // the carried S~ (M = 64 layout), 80 columns
constexpr uint32_t T_Q = 368;    // bf16 phi(Q) per K, V stage, 32 columns each

// Warp roles of the main pass (warp indices).
constexpr int W_PHI0 = 2, W_MASK0 = 10, W_EPI0 = 14;

// ------------------------------------------------------------- state pass
// Partial state dS~ = sum over the segment of phi(K) V~^T, written to
// ws[bh][p] ([64][80] fp32) for every segment p but the last.
template <bool DECAY>
__global__ void __launch_bounds__(NTHR, 1)
    k_tc_fwd_state(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   float* __restrict__ ws, int N, int nseg, int seg_len, int dch, int feat,
                   float lg, int* err) {
  const int p = blockIdx.x, bh = blockIdx.y;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  __shared__ uint64_t bar_full[SNST], bar_empty[SNST], bar_phi[SNST], bar_done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p * seg_len;
  const int ne = min(N, nb + seg_len);
  const int nch = (ne - nb + TC_C - 1) / TC_C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SNST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
      mbar_init(&bar_phi[s], NCOMP);
    }
    mbar_init(&bar_done, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    s_abort = 0;
  }
  if (warp == 1) tmem_alloc(&tmem_base, 128);
  if (warp >= 2) {
    init_ones(sm + S_ONES, threadIdx.x - 64, NCOMP);
    fence_proxy_async();
  }
  auto wt = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
    if (*reinterpret_cast<volatile int*>(&s_abort)) return false;
    if (mbar_wait(bar, parity, WAIT_NS)) return true;
    *reinterpret_cast<volatile int*>(&s_abort) = 1;
    fail(err, code);
    return false;
  };
  // the same, agreed by the whole warp (the tcgen05 loads and stores that
  // follow are warp-collective)
  auto wtu = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
    return __all_sync(0xffffffffu, wt(bar, parity, code));
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();
  // dependents start only once every earlier kernel has completed: the main
  // pass then reads q, k and v without waiting for this grid
  grid_dep_launch();
  const uint32_t TS = tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nch; ++c) {
        const int s = c % SNST;
        if (c >= SNST && !wt(&bar_empty[s], ((c / SNST) - 1) & 1, 31)) break;
        uint8_t* st = sm + s * S_STAGE;
        mbar_arrive_expect_tx(&bar_full[s], 2 * TILE);
        const int n0 = nb + c * TC_C;
        tma_load_3d(st, &tmK, &bar_full[s], 0, n0, bh);
        tma_load_3d(st + TILE, &tmV, &bar_full[s], 0, n0, bh);
        ++issued;
      }
      drain_loads<SNST>(bar_full, issued);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16(64, TC_MA, true, true);
      const uint32_t ones = smem_u32(sm + S_ONES);
      for (int c = 0; c < nch; ++c) {
        const int s = c % SNST;
        const uint32_t k = smem_u32(sm + s * S_STAGE), v = k + TILE;
        const uint64_t dK = sdesc(k, 16, 1024), dVt = sdesc(v, ones - v, 1024);
        if (!wt(&bar_phi[s], (c / SNST) & 1, 32)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // S~ += phi(K)^T V~
          mma_bf16(TS, dadd(dK, kk * 2048), dadd(dVt, kk * 2048), ID_S, c > 0 || kk > 0);
        mma_commit(&bar_empty[s]);
      }
      mma_commit(&bar_done);  // also covers an early exit: every issued MMA has finished
    }
  } else {
    const int t = threadIdx.x - 64;
    for (int c = 0; c < nch; ++c) {
      const int s = c % SNST;
      if (wt(&bar_full[s], (c / SNST) & 1, 33))
        phi_tiles<NCOMP, 1>(sm + s * S_STAGE, 0, min(TC_C, ne - (nb + c * TC_C)), t, dch, feat != 0,
                            DECAY ? lg : 0.f, (ne - 1) - (nb + c * TC_C));  // decay: phi(K_j) gamma^(ne-1-j)
      fence_proxy_async();
      mbar_arrive(&bar_phi[s]);
    }
    // the partial state: TMEM -> shared memory (fp32 [64][80]) -> one bulk copy
    const int wg = t >> 7, qd = warp & 3;
    const uint32_t lq = static_cast<uint32_t>(32 * qd) << 16;
    const int srow = 16 * qd + lane;
    float* rec = reinterpret_cast<float*>(sm + S_REC);
    if (wtu(&bar_done, 0, 34)) {
      tc_fence_after();
      float sv[16], zz[16];
      tmem_ld16(TS + lq + 16 * wg, sv);
      if (wg == 0) tmem_ld16(TS + lq + 64, zz);
      tmem_ld_wait();
      if (lane < 16) {
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4*>(rec + srow * TC_MA + 16 * wg + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
        if (wg == 0)
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(rec + srow * TC_MA + 64 + j) = make_float4(zz[j], zz[j + 1], zz[j + 2], zz[j + 3]);
      }
    }
    fence_proxy_async();
    compute_sync();
    if (t == 0 && !*reinterpret_cast<volatile int*>(&s_abort)) {
      bulk_store(ws + (static_cast<long>(bh) * nseg + p) * 64 * TC_MA, rec, 64 * TC_MA * 4);
      bulk_commit();
      bulk_wait_all();
    }
  }
  if (warp == 1 && lane == 0) mbar_wait(&bar_done, 0, WAIT_NS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(TS, 128);
}

// -------------------------------------------------------------- main pass
template <bool DECAY>
__global__ void __launch_bounds__(NTHR, 1)
    k_tc_fwd_main(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, bf16* __restrict__ out,
                  float* __restrict__ den, const float* __restrict__ ws, int N, int nseg,
                  int seg_len, int out_v8, int dch, int M, int feat, float lg, int* err,
                  const float* __restrict__ S0,
                  const float* __restrict__ Z0, int early) {
  const int p = blockIdx.x, bh = blockIdx.y;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  __shared__ uint64_t bar_kv[KNS], bar_empty[KNS], bar_phi[KNS], bar_q[QNS];
  __shared__ uint64_t bar_a[2], bar_o[2], bar_oe[2], bar_p[2], bar_sp, bar_s, bar_scr, bar_fin;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p * seg_len;
  const int ne = min(N, nb + seg_len);
  const int nch = (ne - nb + TC_C - 1) / TC_C;

  grid_dep_launch();
  if (threadIdx.x == 0) {
    for (int s = 0; s < KNS; ++s) {
      mbar_init(&bar_kv[s], 1);
      mbar_init(&bar_empty[s], 1);
      mbar_init(&bar_phi[s], 32 * (W_MASK0 - W_PHI0));
    }
    for (int s = 0; s < QNS; ++s) mbar_init(&bar_q[s], 1);
    mbar_init(&bar_scr, 128);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_a[b], 1);
      mbar_init(&bar_o[b], 1);
      mbar_init(&bar_oe[b], 128);
      mbar_init(&bar_p[b], 128);
    }
    mbar_init(&bar_sp, 128);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_fin, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    s_abort = 0;
  }
  if (warp == 1) tmem_alloc(&tmem_base, 512);
  if (warp >= W_PHI0 && warp < W_MASK0) {  // the ones tile
    init_ones(sm + F_ONES, threadIdx.x - 32 * W_PHI0, 32 * (W_MASK0 - W_PHI0));
    fence_proxy_async();
  }
  auto wt = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
    if (*reinterpret_cast<volatile int*>(&s_abort)) return false;
    if (mbar_wait(bar, parity, WAIT_NS)) return true;
    *reinterpret_cast<volatile int*>(&s_abort) = 1;
    fail(err, code);
    return false;
  };
  // the same, agreed by the whole warp (the tcgen05 loads and stores that
  // follow are warp-collective)
  auto wtu = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
    return __all_sync(0xffffffffu, wt(bar, parity, code));
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // With a state pass before it (early), this kernel starts only after every
  // kernel before that pass has completed, so only the warps that read the
  // pass's records or write out and den wait for it: the loads, phi and the
  // score products of the first chunks overlap the pass's last CTAs.
  if (!early || warp >= W_MASK0) grid_dep_wait();
  const uint32_t tm = tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    // Chunk c: Q into slot c % QNS once phi(Q) of chunk c - QNS has been taken,
    // K and V into stage c % KNS once the products of chunk c - KNS are done
    // (the last stage also waits until the initial state has left it).
    if (lane == 0) {
      int issued_q = 0, issued_kv = 0;
      for (int c = 0; c < nch; ++c) {
        const int s = c % KNS, sq = c % QNS;
        const int n0 = nb + c * TC_C;
        if (c >= QNS && !wt(&bar_phi[(c - QNS) % KNS], ((c - QNS) / KNS) & 1, 11)) break;
        mbar_arrive_expect_tx(&bar_q[sq], TILE);
        tma_load_3d(sm + F_Q + sq * TILE, &tmQ, &bar_q[sq], 0, n0, bh);
        ++issued_q;
        if (c >= KNS && !wt(&bar_empty[s], ((c / KNS) - 1) & 1, 11)) break;
        if (c == KNS - 1 && !wt(&bar_scr, 0, 11)) break;
        uint8_t* st = sm + F_KV + s * 2 * TILE;
        mbar_arrive_expect_tx(&bar_kv[s], 2 * TILE);
        tma_load_3d(st, &tmK, &bar_kv[s], 0, n0, bh);
        tma_load_3d(st + TILE, &tmV, &bar_kv[s], 0, n0, bh);
        ++issued_kv;
      }
      drain_loads<QNS>(bar_q, issued_q);
      drain_loads<KNS>(bar_kv, issued_kv);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Polls for whichever product can go next: the state update S~(cs) once
    // S~_prev(cs) has been read out (it then fills the tensor pipe while the
    // mask warps work), the read-out O~(co) once P(co) is ready, or A(ca) once
    // phi is on its stage (at most one chunk ahead of the read-out, into a
    // buffer whose O~ has been read).
    if (lane == 0) {
      constexpr uint32_t ID_A = idesc_bf16(128, 128, false, false);
      constexpr uint32_t ID_O = idesc_bf16(128, TC_MA, false, true);
      constexpr uint32_t ID_S = idesc_bf16(64, TC_MA, true, true);
      const uint32_t ones = smem_u32(sm + F_ONES);
      int ca = 0, cs = 0, co = 0;  // next A, next S~ update, next read-out
      uint32_t idle = 0;
      uint64_t t_idle = 0;
      while (co < nch) {
        bool prog = false;
        // S~(cs) needs phi on its stage (A(cs) issued) and S~ after cs-1 read out
        if (cs < ca && cs <= co && cs + 1 < nch && mbar_poll(&bar_sp, cs & 1)) {
          tc_fence_after();
          const uint32_t k = smem_u32(sm + F_KV + (cs % KNS) * 2 * TILE), v = k + TILE;
          const uint64_t dK = sdesc(k, 16, 1024);
          const uint64_t dVt = sdesc(v, ones - v, 1024);  // [V | ones] as an MN-major operand
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // S~ += phi(K)^T V~
            mma_bf16(tm + T_S, dadd(dK, kk * 2048), dadd(dVt, kk * 2048), ID_S, 1);
          mma_commit(&bar_s);
          ++cs;
          prog = true;
        }
        // O~(co) after S~(co), once P(co) is in tensor memory
        // (S~(co) issued implies S~_prev(co) is ready; only the last chunk, which
        // has no update, polls for it -- no later read-out can complete meanwhile)
        if (co < ca && (co < cs || co + 1 == nch) && mbar_poll(&bar_p[co & 1], (co >> 1) & 1) &&
            (co < cs || mbar_poll(&bar_sp, co & 1))) {
          tc_fence_after();
          const int s = co % KNS;
          const uint32_t v = smem_u32(sm + F_KV + s * 2 * TILE) + TILE;
          const uint64_t dVt = sdesc(v, ones - v, 1024);
          const uint64_t dSP = sdesc(smem_u32(sm + F_SP + (co & 1) * 16384), 8192, 1024);
          const uint32_t tp = tm + (co & 1) * T_BUF, tq = tm + T_Q + s * 32;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // O~ = P V~, P in tensor memory
            mma_bf16_ts(tp + 64, tp + 8 * kk, dadd(dVt, kk * 2048), ID_O, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // O~ += phi(Q) S~_prev, phi(Q) in tensor memory
            mma_bf16_ts(tp + 64, tq + 8 * kk, dadd(dSP, kk * 2048), ID_O, 1);
          mma_commit(&bar_o[co & 1]);
          mma_commit(&bar_empty[s]);
          ++co;
          prog = true;
        }
        if (ca < nch && ca <= co + 1 && mbar_poll(&bar_phi[ca % KNS], (ca / KNS) & 1) &&
            (ca < 2 || mbar_poll(&bar_oe[ca & 1], ((ca - 2) >> 1) & 1))) {
          tc_fence_after();
          const int s = ca % KNS;
          const uint64_t dK = sdesc(smem_u32(sm + F_KV + s * 2 * TILE), 16, 1024);
          const uint32_t tq = tm + T_Q + s * 32;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // A = phi(Q) phi(K)^T, phi(Q) in tensor memory
            mma_bf16_ts(tm + (ca & 1) * T_BUF, tq + 8 * kk, dadd(dK, 32 * kk), ID_A, kk > 0);
          mma_commit(&bar_a[ca & 1]);
          ++ca;
          prog = true;
        }
        // bounded: the clock is read once every 1024 idle polls
        if (prog) {
          idle = 0;
        } else if ((++idle & 1023u) != 0) {
          __nanosleep(32);  // leave the issue slots to the other warps of this SM quarter
        } else {
          const uint64_t now = globaltimer_ns();
          if (idle == 1024) t_idle = now;
          if (*reinterpret_cast<volatile int*>(&s_abort) || now - t_idle > WAIT_NS) {
            *reinterpret_cast<volatile int*>(&s_abort) = 1;
            fail(err, 13);
            break;
          }
        }
      }
      mma_commit(&bar_fin);
    }
  } else if (warp < W_MASK0) {
    // ----------------------------------------------------- phi on every chunk
    // phi(Q) goes to tensor memory (the A operand of both Q products): the
    // thread of row r (a warp of lane quarter r / 32) writes d 32h .. 32h+31.
    // phi(K) is applied in place in shared memory.
    const int tt = threadIdx.x - 32 * W_PHI0;  // 0 .. 255
    const int qd = warp & 3, row = 32 * qd + lane;
    const int h = (warp - W_PHI0) >> 2;
    const uint32_t lq = static_cast<uint32_t>(32 * qd) << 16;
    constexpr int NT = 32 * (W_MASK0 - W_PHI0);
    for (int c = 0; c < nch; ++c) {
      const int s = c % KNS;
      // full K, V stage c % KNS also means chunk c - KNS is done with phi(Q) slot s
      if (wtu(&bar_kv[s], (c / KNS) & 1, 14) && wtu(&bar_q[c % QNS], (c / QNS) & 1, 14)) {
        const int valid = min(TC_C, ne - (nb + c * TC_C));
        uint8_t* st = sm + F_KV + s * 2 * TILE;
        const uint8_t* qt = sm + F_Q + (c % QNS) * TILE;
        uint4 qv[4], kv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          qv[i] = *reinterpret_cast<const uint4*>(qt + row * 128 + (((4 * h + i) ^ (row & 7)) << 4));
#pragma unroll
        for (int i = 0; i < 4; ++i)
          kv[i] = *reinterpret_cast<const uint4*>(st + (tt + i * NT) * 16);
        uint32_t pq[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 r = row < valid && 4 * h + i < dch ? (feat ? qv[i] : phi_vec(qv[i]))
                                                         : make_uint4(0u, 0u, 0u, 0u);
          pq[4 * i] = r.x;
          pq[4 * i + 1] = r.y;
          pq[4 * i + 2] = r.z;
          pq[4 * i + 3] = r.w;
        }
        tmem_st16u(tm + T_Q + s * 32 + lq + 16 * h, pq);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int v = tt + i * NT;
          const bool pad = (v >> 3) >= valid || (((v & 7) ^ ((v >> 3) & 7)) >= dch);
          uint4 fk = pad ? make_uint4(0u, 0u, 0u, 0u) : (feat ? kv[i] : phi_vec(kv[i]));
          // decay: key j' of the chunk enters both products scaled by gamma^(127-j')
          if (DECAY && !pad) fk = scale_vec(fk, exp2f(lg * static_cast<float>(127 - (v >> 3))));
          *reinterpret_cast<uint4*>(st + v * 16) = fk;
        }
        tmem_st_wait();
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bar_phi[s]);
    }
  } else {
    // Warps 10-17: the initial state first (all 256 threads), then the mask
    // (10-13) and epilogue (14-17) roles.
    const int tr = threadIdx.x - 32 * W_MASK0;  // 0 .. 255
    const int qd = warp & 3, row = 32 * qd + lane;
    const uint32_t lq = static_cast<uint32_t>(32 * qd) << 16;
    const bool epi = warp >= W_EPI0;
    {
      // initial state: the sum of the earlier segments' partial states; each
      // thread adds up 20 of the 64 x 80 values of every record
      float acc[20];
#pragma unroll
      for (int j = 0; j < 20; ++j) acc[j] = 0.f;
      const float4* rec = reinterpret_cast<const float4*>(ws + static_cast<long>(bh) * nseg * 64 * TC_MA) + tr * 5;
      int pp = 0;
      for (; pp + 1 < p; pp += 2) {  // two records per round trip
        // decay: record pp (summed to its segment's end) reaches this segment's start
        // through gamma^((p-1-pp) seg_len); 1 exactly without decay
        const float f0 = DECAY ? exp2f(lg * static_cast<float>((p - 1 - pp) * seg_len)) : 1.f;
        const float f1 = DECAY ? exp2f(lg * static_cast<float>((p - 2 - pp) * seg_len)) : 1.f;
        float4 x[10];
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          x[j] = rec[pp * (64 * TC_MA / 4) + j];
          x[5 + j] = rec[(pp + 1) * (64 * TC_MA / 4) + j];
        }
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          acc[4 * j] += f0 * x[j].x + f1 * x[5 + j].x;
          acc[4 * j + 1] += f0 * x[j].y + f1 * x[5 + j].y;
          acc[4 * j + 2] += f0 * x[j].z + f1 * x[5 + j].z;
          acc[4 * j + 3] += f0 * x[j].w + f1 * x[5 + j].w;
        }
      }
      if (pp < p) {
        const float f0 = DECAY ? exp2f(lg * static_cast<float>((p - 1 - pp) * seg_len)) : 1.f;
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          const float4 x = rec[pp * (64 * TC_MA / 4) + j];
          acc[4 * j] += f0 * x.x;
          acc[4 * j + 1] += f0 * x.y;
          acc[4 * j + 2] += f0 * x.z;
          acc[4 * j + 3] += f0 * x.w;
        }
      }
      if (S0 != nullptr) {  // a state the sums start from (eq. 16-19 over a prompt)
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          const int f = 4 * (tr * 5 + j), row = f / TC_MA, col = f % TC_MA;
          if (col < 64) {
            const float4 x = *reinterpret_cast<const float4*>(S0 + (static_cast<long>(bh) * 64 + row) * 64 + col);
            acc[4 * j] += x.x;
            acc[4 * j + 1] += x.y;
            acc[4 * j + 2] += x.z;
            acc[4 * j + 3] += x.w;
          } else if (col == 64) {
            acc[4 * j] += Z0[static_cast<long>(bh) * 64 + row];
          }
        }
      }
      float4* scr = reinterpret_cast<float4*>(sm + F_SCR) + tr * 5;
#pragma unroll
      for (int j = 0; j < 5; ++j) scr[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
      asm volatile("bar.sync 4, 256;" ::: "memory");
    }
    if (!epi) {
      // ---------------------------------------- mask: P(c) written over A(c)
      // Row i keeps keys j <= i.  Key group g (32 keys) is fully kept for
      // g < qd, masked on its diagonal for g == qd and zero for g > qd, where
      // qd = i / 32 is the same for the whole warp.
      // decay: A'_ij = gamma^(127-j') A_ij, and P_ij = gamma^-128 A'_ij = gamma^-(j'+1) A_ij is
      // gamma^(i'-j') A_ij in a row frame scaled by gamma^-(i'+1), which out's quotient cancels
      const float cm = DECAY ? exp2f(-128.f * lg) : 1.f;
      for (int c = 0; c < nch; ++c) {
        const uint32_t ta = tm + (c & 1) * T_BUF + lq;
        if (wtu(&bar_a[c & 1], (c >> 1) & 1, 15)) {
          tc_fence_after();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t pk[16];
            if (g <= qd) {
              float a[32];
              tmem_ldn<2>(ta + 32 * g, a);
              if (g < qd) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  pk[i] = DECAY ? pack_bf16(a[2 * i] * cm, a[2 * i + 1] * cm) : pack_bf16(a[2 * i], a[2 * i + 1]);
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float x0 = DECAY ? a[2 * i] * cm : a[2 * i], x1 = DECAY ? a[2 * i + 1] * cm : a[2 * i + 1];
                  pk[i] = pack_bf16(2 * i <= lane ? x0 : 0.f, 2 * i + 1 <= lane ? x1 : 0.f);
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) pk[i] = 0u;
            }
            tmem_st16u(ta + 16 * g, pk);  // over A columns already read
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bar_p[c & 1]);
      }
    } else {
      // ---------- epilogue of O~(c), then S~_prev(c+1) in bf16 for the next chunk
      const int te = threadIdx.x - 32 * W_EPI0;  // 0 .. 127
      const bool has_s = lane < 16;  // M=64 accumulators: row 16*qd + lane in lane 32*qd + lane
      const int srow = 16 * qd + lane;
      // decay: the state the next chunk's keys add to is gamma^128 times the last one
      // (a full chunk); the read-out operand S~_prev stays unscaled
      const float g128 = DECAY ? exp2f(128.f * lg) : 1.f;
      {
        const float4* src = reinterpret_cast<const float4*>(sm + F_SCR) + srow * (TC_MA / 4);
#pragma unroll
        for (int j = 0; j < TC_MA / 16; ++j) {  // 16 columns at a time
          float sv[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 x = has_s ? src[4 * j + i] : make_float4(0.f, 0.f, 0.f, 0.f);
            sv[4 * i] = x.x;
            sv[4 * i + 1] = x.y;
            sv[4 * i + 2] = x.z;
            sv[4 * i + 3] = x.w;
          }
          if (DECAY) {
            float sc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) sc[i] = sv[i] * g128;
            tmem_st16(tm + T_S + lq + 16 * j, sc);
          } else {
            tmem_st16(tm + T_S + lq + 16 * j, sv);
          }
          if (has_s) {
            if (j < 4) {
              tile_put_cols<16>(sm + F_SP, srow, 16 * j, sv);
            } else {
              const float z8[8] = {sv[0], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
              st_row_chunk(sm + F_SP + 8192, srow, 0, z8);
            }
          }
        }
        for (int v = te; v < 2 * 8192 / 16; v += 128) {  // the rest of both z atoms is zero
          const int r = (v >> 3) & 63;
          if ((v & 7) != (r & 7))
            *reinterpret_cast<uint4*>(sm + F_SP + 8192 + (v >> 9) * 16384 + (v & 511) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        tmem_st_wait();
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&bar_scr);  // the initial state has left the last K, V stage
        mbar_arrive(&bar_sp);
      }
      for (int c = 0; c < nch; ++c) {
        const int n0 = nb + c * TC_C;
        if (c + 1 < nch) {  // S~ after chunk c -> S~_prev(c+1), in the buffer O~(c-1) read
          uint8_t* sp = sm + F_SP + ((c + 1) & 1) * 16384;
          if (wtu(&bar_s, c & 1, 18)) {
            tc_fence_after();
            if (DECAY) {
              // 16 columns at a time: to the tile, then S~ <- gamma^128 S~ in place for
              // the next chunk's keys (few registers live: this role shares the kernel's)
#pragma unroll 1
              for (int j = 0; j < TC_MA / 16; ++j) {
                float sv[16];
                tmem_ldn<1>(tm + T_S + lq + 16 * j, sv);
                if (has_s) {
                  if (j < 4) {
                    tile_put_cols<16>(sp, srow, 16 * j, sv);
                  } else {
                    const float z8[8] = {sv[0], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    st_row_chunk(sp + 8192, srow, 0, z8);
                  }
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) sv[i] *= g128;
                tmem_st16(tm + T_S + lq + 16 * j, sv);
                tmem_st_wait();
              }
            } else {
              float sv[48];
              tmem_ldn<3>(tm + T_S + lq, sv);  // columns 0-47
              if (has_s) tile_put_cols<48>(sp, srow, 0, sv);
              tmem_ldn<2>(tm + T_S + lq + 48, sv);  // columns 48-79: S and z
              if (has_s) {
                tile_put_cols<16>(sp, srow, 48, sv);
                const float z8[8] = {sv[16], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                st_row_chunk(sp + 8192, srow, 0, z8);
              }
            }
          }
          fence_proxy_async();
          tc_fence_before();
          mbar_arrive(&bar_sp);
        }
        // out = O~[:, :64] / O~[:, 64], straight from registers to global memory
        if (wtu(&bar_o[c & 1], (c >> 1) & 1, 17)) {
          tc_fence_after();
          const uint32_t to = tm + (c & 1) * T_BUF + 64 + lq;
          float o[32], dd[16];
          uint32_t w[32];
          tmem_ld16(to + 64, dd);
          tmem_ldn<2>(to, o);  // columns 0-31 (one wait covers both loads)
          const float d = dd[0];
          const float inv = 1.f / d;
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = pack_bf16(o[2 * i] * inv, o[2 * i + 1] * inv);
          tmem_ldn<2>(to + 32, o);  // columns 32-63
          tc_fence_before();
          mbar_arrive(&bar_oe[c & 1]);  // the buffer may take A(c+2)
#pragma unroll
          for (int i = 0; i < 16; ++i) w[16 + i] = pack_bf16(o[2 * i] * inv, o[2 * i + 1] * inv);
          if (n0 + row < ne) {
            const long r = static_cast<long>(bh) * N + n0 + row;
            store_row_bf16(out + r * M, w, out_v8 != 0, M);
            // decay: the row came out scaled by gamma^-(row+1), which out's quotient cancels
            if (den != nullptr) den[r] = DECAY ? d * exp2f(lg * static_cast<float>(row + 1)) : d;
          }
        } else {
          tc_fence_before();
          mbar_arrive(&bar_oe[c & 1]);
        }
      }
    }
  }
  if (warp == 1 && lane == 0) mbar_wait(&bar_fin, 0, WAIT_NS);  // no MMA in flight at exit
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

// [BH][N][W] bf16 viewed as a 3-D tensor, 64 x 128 x 1 boxes, 128-byte
// swizzle; for W < 64 the box reaches past the row and the load fills the
// rest with zeros (a store writes only the W columns).
bool make_bf16_map(CUtensorMap* m, const void* base, int BH, int N, int W) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(W) * 2, static_cast<cuuint64_t>(N) * W * 2};
  cuuint32_t box[3] = {64, TC_C, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [rows][cols] row-major bf16 matrix viewed as a 3-D TMA tensor with
// 64 x box_rows x 1 boxes and the 128-byte swizzle.
bool make_bf16_map_2d(CUtensorMap* m, const void* base, long cols, long rows, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, static_cast<cuuint64_t>(rows * cols) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


SegPlan tc_plan(int BH, int N) {
  const int nch = (N + TC_C - 1) / TC_C;
  int want = sm_count() / BH;  // whole segments per head so that all CTAs fit one wave
  if (want < 1) want = 1;
  if (want > nch) want = nch;
  const int per = (nch + want - 1) / want;
  SegPlan pl;
  pl.seg_len = per * TC_C;
  pl.nseg = (N + pl.seg_len - 1) / pl.seg_len;
  return pl;
}

// bf16 with D, M in {16, 32, 64}: narrower heads ride in the 64-wide tiles,
// zero-filled by the loads, with phi zeroed on the padded features.
bool tc_eligible(const Shape& s) {
  return s.dtype == 1 && (s.D == 16 || s.D == 32 || s.D == 64) && (s.M == 16 || s.M == 32 || s.M == 64);
}

// The prefill adds and returns the caller's [D][M] state, laid out for 64.
bool tc_prefill_eligible(const Shape& s) { return s.dtype == 1 && s.D == 64 && s.M == 64; }

size_t causal_fwd_tc_ws_floats(const Shape& s) {
  const SegPlan pl = tc_plan(s.B * s.H, s.N);
  return static_cast<size_t>(s.B) * s.H * pl.nseg * 64 * TC_MA;
}

int causal_fwd_tc_launches(const Shape& s) { return tc_plan(s.B * s.H, s.N).nseg > 1 ? 2 : 1; }

namespace {

// The forward's launches: the state pass over the first nrec segments (all
// of them when the state after the sequence is wanted), then the main pass,
// whose sums start from (S0, Z0) when S0 is not null.
cudaError_t fwd_tc_launch(const void* q, const void* k, const void* v, void* out, float* den,
                          float* ws, const Shape& s, cudaStream_t st, const float* S0,
                          const float* Z0, bool all_records, bool feat = false, float gamma = 1.f) {
  const float lg = gamma == 1.f ? 0.f : log2f(gamma);
  const int BH = s.B * s.H;
  const SegPlan pl = tc_plan(BH, s.N);
  CUtensorMap mq, mk, mv;
  if (!make_bf16_map(&mq, q, BH, s.N, s.D) || !make_bf16_map(&mk, k, BH, s.N, s.D) ||
      !make_bf16_map(&mv, v, BH, s.N, s.M))
    return cudaErrorInvalidValue;
  const int out_v8 = (reinterpret_cast<uintptr_t>(out) & 31) == 0;
  int* err = status_word();
  cudaError_t e;
  auto kstate = lg != 0.f ? k_tc_fwd_state<true> : k_tc_fwd_state<false>;
  auto kmain = lg != 0.f ? k_tc_fwd_main<true> : k_tc_fwd_main<false>;
  if ((e = cudaFuncSetAttribute(kstate, cudaFuncAttributeMaxDynamicSharedMemorySize, S_SMEM)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(kmain, cudaFuncAttributeMaxDynamicSharedMemorySize, F_SMEM)) !=
      cudaSuccess)
    return e;
  const int nrec = all_records ? pl.nseg : pl.nseg - 1;
  if (nrec > 0) {
    if ((e = launch_pdl(kstate, dim3(nrec, BH), dim3(NTHR), S_SMEM, st, mk, mv, ws,
                        s.N, pl.nseg, pl.seg_len, s.D / 8, feat ? 1 : 0, lg, err)) != cudaSuccess)
      return e;
  }
  if ((e = launch_pdl(kmain, dim3(pl.nseg, BH), dim3(NTHR), F_SMEM, st, mq, mk, mv,
                      static_cast<bf16*>(out), den, static_cast<const float*>(ws), s.N, pl.nseg,
                      pl.seg_len, out_v8, s.D / 8, s.M, feat ? 1 : 0, lg, err, S0, Z0,
                      nrec > 0 ? 1 : 0)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t causal_fwd_tc(const void* q, const void* k, const void* v, void* out, float* den,
                          float* ws, const Shape& s, cudaStream_t st, bool feat, float gamma) {
  return fwd_tc_launch(q, k, v, out, den, ws, s, st, nullptr, nullptr, false, feat, gamma);
}

// The state pass writes every segment's record, the main pass adds (S, Z) to
// each segment's starting state, and after it (S, Z) += the sum of the
// records ([64][80] each: S~ in columns 0-63, z in column 64).
cudaError_t causal_prefill_tc(const void* q, const void* k, const void* v, void* out, float* den,
                              float* S, float* Z, float* ws, const Shape& s, cudaStream_t st) {
  cudaError_t e = fwd_tc_launch(q, k, v, out, den, ws, s, st, S, Z, true);
  if (e != cudaSuccess) return e;
  const int nseg = tc_plan(s.B * s.H, s.N).nseg;
  return state_add_records(ws, s.B * s.H, nseg, 64 * TC_MA, 0, nseg, 64, 64, TC_MA, 64, TC_MA, S, Z,
                           st);
}

}  // namespace la
