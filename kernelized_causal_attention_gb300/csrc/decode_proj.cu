// One RNN decode step fed by its own query/key/value projection, for many
// independent streams in one launch: "Transformers are RNNs" (part 2/3) §3.4
// eq. 18-20 without the layer's f_l and residual,
//   [q | k | v] = x W_h  (per head h),
//   s <- s + phi(k) v^T,  z <- z + phi(k),  y = phi(q)^T s / phi(q)^T z,
// the batched-generation setting of §4.2.1 (thousands of images decoded at
// once, one token per step).
//
// GB300 design: one CTA per (block of SB <= 64 streams, head).  The block's
// projection is a tcgen05 product (M = 64 rows = streams, rows past the block
// are don't-care; N = the head's 2D+M columns rounded up to whole 64-column
// atoms; K = d_model in slabs of 64), its operands brought in by TMA through a
// three-stage ring (x as K-major tiles, the head's contiguous columns of W as
// MN-major atoms, both with the 128-byte swizzle) and its accumulator in
// tensor memory.  The CTA then applies phi and streams the block's fp32
// states through a ring of ~32 KB groups in the freed stages (16-byte
// cp.async, each thread copying and reading back its own pieces), updates
// them (each read and written once) and reads y out, so q, k and v never
// leave the SM.
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tc_chunk.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tcc;

constexpr int P_NT = 256;    // threads
constexpr int P_NW = P_NT / 32;
constexpr int P_KS = 64;     // d_model per slab
constexpr int P_SBMAX = 64;  // streams per CTA at most (the MMA's M)

// NS: stages of the slab ring.
template <int D, int M, int NS>
struct ProjGeom {
  static constexpr int NQKV = 2 * D + M;            // one head's q | k | v columns
  static constexpr int NP = (NQKV + 63) / 64 * 64;  // whole 64-column atoms (the MMA's N)
  static constexpr int NAT = NP / 64;
  static constexpr int SQ = NQKV + 4;               // row stride of phi(q) | phi(k) | v in smem
  static constexpr int A_BYTES = P_SBMAX * 128;     // [64 streams][64 of d_model] bf16
  static constexpr int STAGE = A_BYTES + NAT * P_KS * 128;
  static constexpr uint32_t TCOLS = NP <= 64 ? 64u : (NP <= 128 ? 128u : 256u);
  static constexpr int M4 = M / 4;                  // float4 columns of a state row
  static constexpr int RG = P_NT / M4;              // row groups of the state
  static constexpr int RPT = (D + RG - 1) / RG;     // state rows per thread
  // the states stream through a ring of NG groups of NSTR streams (about
  // 32 KB a group) in the projection's stages, free once the product is done
  static constexpr int NSTR_RAW = 8192 / (D * M);
  static constexpr int NSTR_FIT = NS * STAGE / (2 * D * M * 4);  // the ring holds two groups at least
  static constexpr int NSTR_MIN = NSTR_RAW < NSTR_FIT ? NSTR_RAW : NSTR_FIT;
  static constexpr int NSTR = NSTR_MIN > 16 ? 16 : (NSTR_MIN < 1 ? 1 : NSTR_MIN);
  static constexpr int GROUP = NSTR * D * M * 4;
  static constexpr int NG_RAW = NS * STAGE / GROUP;
  static constexpr int NG = NG_RAW > 8 ? 8 : NG_RAW;
  // the cross-warp sums of a group, [NSTR][NW][M4] float4, two buffers: the
  // second in the ring's spare bytes where they suffice
  static constexpr int RED = NSTR * (P_NT / 32) * (M / 4) * 16;
  static constexpr bool RED_IN_RING = NS * STAGE - NG * GROUP >= RED;
  static_assert(NG >= 2, "the ring needs two groups");
};

template <int D, int M, int NS>
size_t proj_smem_bytes(int SB) {
  using G = ProjGeom<D, M, NS>;
  return 1024 + static_cast<size_t>(NS) * G::STAGE + static_cast<size_t>(SB) * G::SQ * 4 +
         (G::RED_IN_RING ? 1 : 2) * static_cast<size_t>(G::RED) + static_cast<size_t>(G::NG) * G::NSTR * D * 4 +
         2 * G::NSTR * 4;
}

// phi(x) = elu(x) + 1 (eq. 7) with the exponential evaluated on both sides
// of the select, so that a run of these has no branch: the same value as
// phi() in every case.
__device__ __forceinline__ float phi_select(float x) {
  const float e = expf(fminf(x, 0.f));
  return x > 0.f ? x + 1.f : e;
}

// 16-byte asynchronous copy global -> shared (bypassing L1), and its groups.
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sdst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float comp(const float4& a, int i) {
  return i == 0 ? a.x : (i == 1 ? a.y : (i == 2 ? a.z : a.w));
}

template <int D, int M, int NS>
__global__ void __launch_bounds__(P_NT, NS <= 3 ? 2 : 1)
    k_decode_proj(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  float* __restrict__ S, float* __restrict__ Z, bf16* __restrict__ y, int B, int H,
                  int dm, int SB, int* err) {
  using G = ProjGeom<D, M, NS>;
  const int b0 = blockIdx.x * SB, h = blockIdx.y;
  const int nb = min(SB, B - b0);  // streams of this CTA
  const int nslab = dm / P_KS;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  float* sqkv = reinterpret_cast<float*>(sm + NS * G::STAGE);  // [SB][SQ]
  // the cross-warp sums of a group, double-buffered by group parity: a thread
  // is at most one group ahead of the slowest (the next group's barrier holds
  // it), so one barrier a group suffices
  float4* sred = reinterpret_cast<float4*>(sqkv + SB * G::SQ);     // [NSTR][NW][M4]
  float4* sred1 = G::RED_IN_RING ? reinterpret_cast<float4*>(sm + G::NG * G::GROUP)
                                 : sred + G::NSTR * P_NW * G::M4;  // the second buffer
  float4* zring = sred + (G::RED_IN_RING ? 1 : 2) * G::NSTR * P_NW * G::M4;  // [NG][NSTR][D/4]
  float* sden = reinterpret_cast<float*>(zring + G::NG * G::NSTR * (D / 4));  // [2][NSTR]
  float4* ring = reinterpret_cast<float4*>(sm);                    // [NG][NSTR][D*M/4]
  __shared__ uint64_t bar_full[NS], bar_empty[NS], bar_done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;

  if (t == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_done, 1);
    fence_barrier_init();
    s_abort = 0;
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(&tmem_base, G::TCOLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tacc = tmem_base;

  // ------------------------- projection: [q | k | v] = x W_h (lane 0 of warp 0)
  // The other lanes of warp 0 wait for it at __syncwarp, not on an mbarrier:
  // a sibling path suspended in try_wait could hold back the issuing lane.
  if (t == 0) {
    const uint32_t tx = static_cast<uint32_t>(SB) * 128u + G::NAT * P_KS * 128u;
    auto issue = [&](int ks) {
      const int s = ks % NS;
      uint8_t* A = sm + s * G::STAGE;
      mbar_arrive_expect_tx(&bar_full[s], tx);
      tma_load_3d(A, &tmX, &bar_full[s], ks * P_KS, b0, 0);
#pragma unroll
      for (int a = 0; a < G::NAT; ++a)
        tma_load_3d(A + G::A_BYTES + a * (P_KS * 128), &tmW, &bar_full[s], h * G::NQKV + 64 * a,
                    ks * P_KS, 0);
    };
    int issued = 0;
    for (; issued < NS && issued < nslab; ++issued) issue(issued);
    constexpr uint32_t ID = idesc_bf16(P_SBMAX, G::NP, false, true);
    bool good = true;
    for (int ks = 0; ks < nslab; ++ks) {
      const int s = ks % NS;
      if (!mbar_wait(&bar_full[s], (ks / NS) & 1, WAIT_NS)) {
        fail(err, 61);
        good = false;
        break;
      }
      tc_fence_after();
      const uint32_t a = smem_u32(sm + s * G::STAGE), b = a + G::A_BYTES;
      const uint64_t dA = sdesc(a, 16, 1024), dB = sdesc(b, P_KS * 128, 1024);
#pragma unroll
      for (int kk = 0; kk < P_KS / 16; ++kk)
        mma_bf16(tacc, dadd(dA, 32 * kk), dadd(dB, 2048 * kk), ID, (ks > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&bar_empty[s]);
      if (ks + NS < nslab) {  // refill the stage once its products have read it
        if (!mbar_wait(&bar_empty[s], (ks / NS) & 1, WAIT_NS)) {
          fail(err, 62);
          good = false;
          break;
        }
        issue(ks + NS);
        ++issued;
      }
    }
    mma_commit(&bar_done);  // every product issued so far has completed
    if (!good) {
      *reinterpret_cast<volatile int*>(&s_abort) = 1;
      drain_loads<NS>(bar_full, issued);
    }
  }
  __syncwarp();
  bool done = mbar_wait(&bar_done, 0, WAIT_NS);
  if (!done) fail(err, 63);
  const bool ok = __syncthreads_and(done && !*reinterpret_cast<volatile int*>(&s_abort));
  tc_fence_after();

  // q, k and v of the block's streams into shared memory (row r of the M = 64
  // accumulator sits in TMEM lane 32 (r / 16) + r % 16), then phi over the q
  // and k columns by all threads, element by element
  if (ok && warp < 4) {
    const uint32_t lq = static_cast<uint32_t>(32 * warp) << 16;
    const int r = 16 * warp + lane;
    const bool mine = lane < 16 && r < nb;
#pragma unroll
    for (int c0 = 0; c0 < G::NQKV; c0 += 16) {
      float f[16];
      tmem_ldn<1>(tacc + lq + c0, f);
      if (mine) {
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(sqkv + r * G::SQ + c0 + i) =
              make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  for (int e = t; ok && e < nb * 2 * D; e += P_NT) {
    float* p = sqkv + (e / (2 * D)) * G::SQ + e % (2 * D);
    *p = phi_select(*p);
  }
  __syncthreads();

  // ------------------------------------------- state update and read-out
  // Thread t owns float4 column c4 of state rows rg, rg + RG, ... of every
  // stream, and warp j % NW lanes 0 .. D/4-1 own stream j's z (j within a
  // group): each thread copies its own pieces into the ring with 16-byte
  // cp.async and reads back only those, so a wait_group is all it needs.
  const int c4 = t % G::M4, rg = t / G::M4;
  const int ngroups = (nb + G::NSTR - 1) / G::NSTR;
  auto issue = [&](int g) {
    if (g < ngroups) {
      float4* slot = ring + (g % G::NG) * (G::NSTR * D * M / 4);
      float4* zslot = zring + (g % G::NG) * (G::NSTR * D / 4);
#pragma unroll
      for (int j = 0; j < G::NSTR; ++j) {
        const int js = g * G::NSTR + j;
        if (js < nb) {
          const long sh = static_cast<long>(b0 + js) * H + h;
          const float4* Sh = reinterpret_cast<const float4*>(S) + sh * (D * M / 4);
#pragma unroll
          for (int r = 0; r < G::RPT; ++r) {
            const int d = rg + r * G::RG;
            if (d < D) cp_async16(slot + j * (D * M / 4) + d * G::M4 + c4, Sh + d * G::M4 + c4);
          }
          if (warp == j % P_NW && lane < D / 4)
            cp_async16(zslot + j * (D / 4) + lane, reinterpret_cast<const float4*>(Z) + sh * (D / 4) + lane);
        }
      }
    }
    cp_async_commit();  // one group per call, empty or not, to keep the count
  };
  auto process = [&](int g) {
    float4* red = (g & 1) ? sred1 : sred;
    float* dn = sden + (g & 1) * G::NSTR;
    const float4* slot = ring + (g % G::NG) * (G::NSTR * D * M / 4);
    const float4* zslot = zring + (g % G::NG) * (G::NSTR * D / 4);
    const int j0 = g * G::NSTR;
#pragma unroll
    for (int j = 0; j < G::NSTR; ++j) {
      if (j0 + j < nb) {
        const float* qkv = sqkv + (j0 + j) * G::SQ;
        const float4 v4 = *reinterpret_cast<const float4*>(qkv + 2 * D + 4 * c4);
        float4* Sh = reinterpret_cast<float4*>(S) + (static_cast<long>(b0 + j0 + j) * H + h) * (D * M / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < G::RPT; ++r) {
          const int d = rg + r * G::RG;
          if (d < D) {
            const float fk = qkv[D + d], fq = qkv[d];
            float4 s4 = slot[j * (D * M / 4) + d * G::M4 + c4];
            s4.x = fmaf(fk, v4.x, s4.x);
            s4.y = fmaf(fk, v4.y, s4.y);
            s4.z = fmaf(fk, v4.z, s4.z);
            s4.w = fmaf(fk, v4.w, s4.w);
            Sh[d * G::M4 + c4] = s4;
            acc.x = fmaf(fq, s4.x, acc.x);
            acc.y = fmaf(fq, s4.y, acc.y);
            acc.z = fmaf(fq, s4.z, acc.z);
            acc.w = fmaf(fq, s4.w, acc.w);
          }
        }
        // sum over the lanes of this warp that hold the same columns
#pragma unroll
        for (int off = 16; off >= G::M4; off >>= 1) {
          acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
          acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
          acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
          acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
        }
        if (lane < G::M4) red[(j * P_NW + warp) * G::M4 + lane] = acc;
      }
    }
    // z <- z + phi(k) and den = phi(q) . z: warp j % NW, four entries a lane
    for (int j = warp; j < G::NSTR; j += P_NW) {
      if (j0 + j < nb) {
        float dp = 0.f;
        if (lane < D / 4) {
          const float* qkv = sqkv + (j0 + j) * G::SQ + 4 * lane;
          const float4 z0 = zslot[j * (D / 4) + lane];
          const float4 z = make_float4(z0.x + qkv[D], z0.y + qkv[D + 1], z0.z + qkv[D + 2],
                                       z0.w + qkv[D + 3]);
          reinterpret_cast<float4*>(Z)[(static_cast<long>(b0 + j0 + j) * H + h) * (D / 4) + lane] = z;
          dp = qkv[0] * z.x + qkv[1] * z.y + qkv[2] * z.z + qkv[3] * z.w;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dp += __shfl_xor_sync(0xffffffffu, dp, off);
        if (lane == 0) dn[j] = dp;
      }
    }
    __syncthreads();
    for (int i = t; i < G::NSTR * M; i += P_NT) {
      const int j = i / M, m = i % M;
      if (j0 + j < nb) {
        float num = 0.f;
#pragma unroll
        for (int w = 0; w < P_NW; ++w) num += comp(red[(j * P_NW + w) * G::M4 + m / 4], m & 3);
        y[(static_cast<long>(b0 + j0 + j) * H + h) * M + m] = __float2bfloat16_rn(num / dn[j]);
      }
    }
  };
  if (ok) {
    fence_proxy_async();  // the ring reuses stages last touched by TMA and the tensor cores
    for (int g = 0; g < G::NG - 1; ++g) issue(g);
    for (int g = 0; g < ngroups; ++g) {
      issue(g + G::NG - 1);  // into the slot that group g - 1 has left
      cp_async_wait<G::NG - 1>();
      process(g);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tacc, G::TCOLS);
}

}  // namespace

// Streams per CTA: the largest block that still gives two CTAs per SM, with
// three stages.  (Six stages at one CTA per SM, for grids that fit one wave,
// measured slower at 256 streams: 25.0 against 23.4 us.)
ProjPlan decode_proj_plan(int B, int H) {
  const long sms = sm_count();
  auto ctas = [&](int sb) { return static_cast<long>((B + sb - 1) / sb) * H; };
  for (int sb : {64, 32, 16})
    if (ctas(sb) >= 2 * sms) return ProjPlan{sb, 3};
  return ProjPlan{8, 3};
}

int decode_proj_block(int B, int H) { return decode_proj_plan(B, H).SB; }

namespace {

template <int D, int M, int NS>
cudaError_t launch_proj_ns(const CUtensorMap& mx, const CUtensorMap& mw, float* S, float* Z, void* y,
                           int B, int H, int dm, int SB, cudaStream_t st) {
  const size_t smem = proj_smem_bytes<D, M, NS>(SB);
  cudaError_t e = cudaFuncSetAttribute(k_decode_proj<D, M, NS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k_decode_proj<D, M, NS><<<dim3((B + SB - 1) / SB, H), P_NT, smem, st>>>(
      mx, mw, S, Z, static_cast<bf16*>(y), B, H, dm, SB, status_word());
  return cudaGetLastError();
}

template <int D, int M>
cudaError_t launch_proj(const CUtensorMap& mx, const CUtensorMap& mw, float* S, float* Z, void* y,
                        int B, int H, int dm, const ProjPlan& pl, cudaStream_t st) {
  return launch_proj_ns<D, M, 3>(mx, mw, S, Z, y, B, H, dm, pl.SB, st);
}

}  // namespace

cudaError_t decode_step_proj(const void* x, const void* W, float* S, float* Z, void* y, int B,
                             int H, int dm, int D, int M, cudaStream_t st) {
  const ProjPlan pl = decode_proj_plan(B, H);
  const long wcols = static_cast<long>(H) * (2 * D + M);
  CUtensorMap mx, mw;
  if (!make_bf16_map_2d(&mx, x, dm, B, pl.SB) || !make_bf16_map_2d(&mw, W, wcols, dm, P_KS))
    return cudaErrorInvalidValue;
  LA_DISPATCH_DM(D, M, return (launch_proj<D_, M_>(mx, mw, S, Z, y, B, H, dm, pl, st)));
  return cudaErrorInvalidValue;
}

}  // namespace la
