// Shared pieces of the tcgen05 causal kernels: chunk geometry, the phi
// transform of a swizzled tile, bf16 packing into 128-byte-swizzled operand
// tiles and TMEM row loads.
#pragma once

#include <cuda_bf16.h>

#include "tc.cuh"

namespace la {
namespace tcc {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int TC_C = 128;                  // tokens per chunk (MMA M)
constexpr int NST = 2;                     // TMA ring stages
constexpr int TILE = TC_C * 64 * 2;        // one [128][64] bf16 tile
constexpr int NTHR = 192;                  // warp 0 TMA, warp 1 MMA, warps 2-5 compute
constexpr uint64_t WAIT_NS = 2000000000ull;  // bound on every wait

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

}  // namespace tcc

// [BH][N][64] bf16 viewed as a 3-D TMA tensor with 64 x 128 x 1 boxes and the
// 128-byte swizzle (defined in causal_tc.cu).
bool make_bf16_map(CUtensorMap* m, const void* base, int BH, int N);

}  // namespace la
