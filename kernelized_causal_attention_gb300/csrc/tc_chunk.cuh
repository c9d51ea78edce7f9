// Shared pieces of the tcgen05 causal kernels: chunk geometry, the phi
// transform of a swizzled tile, bf16 packing into 128-byte-swizzled operand
// tiles and TMEM row loads.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <utility>

#include "tc.cuh"

namespace la {
namespace tcc {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int TC_C = 128;                  // tokens per chunk (MMA M)
constexpr int NST = 2;                     // TMA ring stages
constexpr int TILE = TC_C * 64 * 2;        // one [128][64] bf16 tile
constexpr int NWG = 4;                     // compute warpgroups
constexpr int NCOMP = 128 * NWG;           // compute threads
constexpr int NTHR = 64 + NCOMP;           // warp 0 TMA, warp 1 MMA, the rest compute
constexpr int KW = TC_C / NWG;             // key columns of a 128-wide accumulator per warpgroup
constexpr int OW = 64 / NWG;               // columns of a 64-wide output per warpgroup
constexpr uint64_t WAIT_NS = 2000000000ull;  // bound on every wait

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// 16-byte shared-memory store / load through an explicit shared-window
// address.  The tiles are addressed through pointers aligned at run time, from
// which the compiler cannot always tell that they point into shared memory;
// these keep such accesses on the shared-memory path.
__device__ __forceinline__ void sts128(const void* p, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p))
               : "memory");
  return v;
}

__device__ __forceinline__ float lds32f(const void* p) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ float4 lds128f(const void* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(p))
               : "memory");
  return v;
}
__device__ __forceinline__ void sts16(const void* p, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(smem_u32(p)), "h"(v) : "memory");
}

__device__ __forceinline__ void fail(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// phi(x) = elu(x) + 1 (eq. 7) on a pair of bf16 values, written as
// max(x, 0) + 2^min(x log2 e, 0): x + 1 for x > 0 and exp(x) otherwise.  All
// arithmetic is packed bf16: x log2 e is formed as x c_hi + (x c_lo) with
// c_hi + c_lo = log2 e to 2^-17 (one rounding of the fused multiply-add, so
// the product is the correctly rounded bf16 value up to that residual), and
// the exponential is the hardware base-2 exponential on bf16 pairs.
__device__ __forceinline__ uint32_t phi_bf16x2(uint32_t w) {
  const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w);
  const __nv_bfloat162 c_hi = __halves2bfloat162(__ushort_as_bfloat16(0x3fb9),
                                                 __ushort_as_bfloat16(0x3fb9));  // 1.4453125
  const __nv_bfloat162 c_lo = __halves2bfloat162(__ushort_as_bfloat16(0xbb2c),
                                                 __ushort_as_bfloat16(0xbb2c));  // -0.0026245
  const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
  const __nv_bfloat162 t = __hmin2(__hfma2(x, c_hi, __hmul2(x, c_lo)), zero);
  uint32_t e;
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(*reinterpret_cast<const uint32_t*>(&t)));
  const __nv_bfloat162 r = __hadd2(__hmax2(x, zero), *reinterpret_cast<const __nv_bfloat162*>(&e));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint4 phi_vec(uint4 u) {
  return make_uint4(phi_bf16x2(u.x), phi_bf16x2(u.y), phi_bf16x2(u.z), phi_bf16x2(u.w));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Eight packed bf16 values times an fp32 factor, rounded once.
__device__ __forceinline__ uint4 scale_vec(uint4 u, float f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    r[i] = pack_bf16(__uint_as_float(w[i] << 16) * f, __uint_as_float(w[i] & 0xffff0000u) * f);
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// phi applied in place to NTL swizzled [128][64] bf16 tiles spaced `stride`
// bytes apart, by NT threads (t = 0 .. NT-1; elementwise, so the swizzle does
// not matter).  Every thread first loads all of its vectors, then transforms
// and stores them, so the loads and the exponentials overlap.  Rows at or past
// `valid` are zeroed: a zero phi row adds nothing to any sum.  So are the
// columns at or past 8 dch (a head narrower than 64 whose tile the load
// filled with zeros: phi(0) = 1, but a padded feature must add nothing).
// ident: the tiles already hold features (a feature map applied before the
// call); only the masking applies.  lg != 0: row r is also scaled by
// 2^(lg (e0 - r)), i.e. gamma^(e0 - r) with lg = log2 gamma (the decay).
template <int NT, int NTL>
__device__ __forceinline__ void phi_tiles(uint8_t* tile, int stride, int valid, int t, int dch = 8,
                                          bool ident = false, float lg = 0.f, int e0 = 0) {
  constexpr int PER = TILE / 16 / NT;  // vectors per thread and tile
  static_assert(PER * NT * 16 == TILE, "threads must divide the tile");
  uint4 u[NTL][PER];
#pragma unroll
  for (int k = 0; k < NTL; ++k)
#pragma unroll
    for (int i = 0; i < PER; ++i)
      u[k][i] = lds128(tile + k * stride + (t + i * NT) * 16);
#pragma unroll
  for (int k = 0; k < NTL; ++k)
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int v = t + i * NT;
      const bool pad = (v >> 3) >= valid || (((v & 7) ^ ((v >> 3) & 7)) >= dch);
      uint4 r = pad ? make_uint4(0u, 0u, 0u, 0u) : (ident ? u[k][i] : phi_vec(u[k][i]));
      if (lg != 0.f && !pad) r = scale_vec(r, exp2f(lg * static_cast<float>(e0 - (v >> 3))));
      sts128(tile + k * stride + v * 16, r);
    }
}

// phi applied in place to a swizzled [128][64] bf16 tile by `nthr` threads.
__device__ __forceinline__ void phi_tile(uint8_t* tile, int valid, int t, int nthr = NCOMP) {
  for (int v = t; v < TILE / 16; v += nthr) {
    uint4* ptr = reinterpret_cast<uint4*>(tile + v * 16);
    *ptr = (v >> 3) >= valid ? make_uint4(0u, 0u, 0u, 0u) : phi_vec(*ptr);
  }
}

// phi_tile that also writes the transformed rows below `valid` to the
// row-major [*][64] bf16 global rows starting at `g` (16-byte stores; the
// eight vectors of a row are written by consecutive threads).
__device__ __forceinline__ void phi_tile_store(uint8_t* tile, int valid, int t, bf16* g) {
  for (int v = t; v < TILE / 16; v += NCOMP) {
    uint4* ptr = reinterpret_cast<uint4*>(tile + v * 16);
    const int r = v >> 3;
    uint4 u = *ptr;
    if (r >= valid) {
      u = make_uint4(0u, 0u, 0u, 0u);
    } else {
      u = phi_vec(u);
      const int lc = (v & 7) ^ (r & 7);  // logical 16-byte chunk of this vector
      *reinterpret_cast<uint4*>(g + r * 64 + lc * 8) = u;
    }
    *ptr = u;
  }
}

// A shared-memory descriptor advanced by `bytes` (the start-address field is
// the low 14 bits in 16-byte units; shared addresses stay below 256 KB).
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its memory is visible.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


// Writes 8 consecutive values (columns 8c .. 8c+7) of row r of a swizzled
// [rows][64] bf16 tile.
__device__ __forceinline__ void st_row_chunk(uint8_t* tile, int r, int c, const float* x) {
  const uint32_t off = static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(c) ^ (r & 7u)) << 4);
  sts128(tile + off, make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                                pack_bf16(x[6], x[7])));
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

// 16 * n fp32 columns of this thread's TMEM lane (n = 1..4), one wait.
template <int n>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, float* v) {
#pragma unroll
  for (int i = 0; i < n; ++i) tmem_ld16(taddr + 16 * i, v + 16 * i);
  tmem_ld_wait();
}

// NC columns (a multiple of 8) from column col0 of row r of a swizzled
// [128][64] bf16 tile, as floats.
template <int NC>
__device__ __forceinline__ void tile_row_cols(const uint8_t* tile, int r, int col0, float* x) {
#pragma unroll
  for (int c = 0; c < NC / 8; ++c) {
    const int c8 = (col0 >> 3) + c;
    const uint4 u = lds128(tile + r * 128 + ((c8 ^ (r & 7)) << 4));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
      x[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

// NC floats (a multiple of 8) as bf16 columns col0 .. of row r of a
// swizzled [128][64] bf16 tile.
template <int NC>
__device__ __forceinline__ void tile_put_cols(uint8_t* tile, int r, int col0, const float* x) {
#pragma unroll
  for (int c = 0; c < NC / 8; ++c) st_row_chunk(tile, r, (col0 >> 3) + c, x + 8 * c);
}

// NC floats (a multiple of 8) as bf16 to global memory (16-byte aligned).
template <int NC>
__device__ __forceinline__ void store_bf16(bf16* dst, const float* f) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < NC / 8; ++c)
    d[c] = make_uint4(pack_bf16(f[8 * c], f[8 * c + 1]), pack_bf16(f[8 * c + 2], f[8 * c + 3]),
                      pack_bf16(f[8 * c + 4], f[8 * c + 5]), pack_bf16(f[8 * c + 6], f[8 * c + 7]));
}

// Reads NC fp32 columns of this thread's TMEM lane from `taddr` (keys key0 ..
// of row `row`), adds `add`, keeps keys j <= row and stores them as bf16
// columns (key0 & 63) .. of row `row` of the swizzled tile `dst`.
template <int NC>
__device__ __forceinline__ void mask_cols(uint32_t taddr, float add, uint8_t* dst, int row,
                                          int key0, float scale = 1.f) {
  float a[NC];
  tmem_ldn<NC / 16>(taddr, a);
#pragma unroll
  for (int i = 0; i < NC; ++i) a[i] = (key0 + i <= row) ? (a[i] + add) * scale : 0.f;
  tile_put_cols<NC>(dst, row, key0 & 63, a);
}

// Lets the next kernel in the stream start its prologue on free SMs; its
// griddepcontrol.wait still waits for this whole grid and its memory.
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Producer epilogue: wait (bounded) for the last loads issued into each stage,
// so that no TMA write into shared memory is still in flight at exit.
template <int NS>
__device__ __forceinline__ void drain_loads(uint64_t* full, int issued) {
  for (int i = issued > NS ? issued - NS : 0; i < issued; ++i)
    mbar_wait(&full[i % NS], (i / NS) & 1, WAIT_NS);
}

// The first `ncols` (16, 32 or 64) of 64 bf16 (32 packed words) to a global
// row: 32-byte stores when the row is 32-byte aligned, else 16-byte stores.
__device__ __forceinline__ void store_row_bf16(bf16* dst, const uint32_t* w, bool v8, int ncols = 64) {
  if (v8) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (16 * i < ncols)
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 16 * i),
                     "r"(w[8 * i]), "r"(w[8 * i + 1]), "r"(w[8 * i + 2]), "r"(w[8 * i + 3]),
                     "r"(w[8 * i + 4]), "r"(w[8 * i + 5]), "r"(w[8 * i + 6]), "r"(w[8 * i + 7])
                     : "memory");
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (8 * i < ncols)
        *reinterpret_cast<uint4*>(dst + 8 * i) = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

// The constant ones tile: a [128][64] bf16 K-major tile whose column 0 is 1;
// read as the second 64-wide N atom of the MN-major operand [V | 1].
__device__ __forceinline__ void init_ones(uint8_t* tile, int t, int nthr) {
  for (int v = t; v < TILE / 16; v += nthr) {
    const int r = v >> 3, c = (v & 7) ^ (r & 7);  // logical 16-byte chunk of this vector
    *reinterpret_cast<uint4*>(tile + v * 16) =
        c == 0 ? make_uint4(0x3f80u, 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// An [80]-wide fp32 state in tensor memory (M = 64 layout: row r of the
// state in lane 32 * (r / 16) + r % 16) as a bf16 operand tile: row r, columns
// 0-63 into `tile` ([64][64], 128-byte swizzle) and column 64 into column 0 of
// the second atom at tile + 8192 (whose other columns stay zero).  Called by
// all four warps of a warpgroup (one per lane quarter); `lq` is the lane-quarter
// field of this warp.
__device__ __forceinline__ void state_to_tile(uint32_t tstate, uint32_t lq, int lane, int qd,
                                              uint8_t* tile) {
  const bool has_s = lane < 16;
  const int srow = 16 * qd + lane;
  float sv[48];
  tmem_ldn<3>(tstate + lq, sv);  // columns 0-47
  if (has_s) tile_put_cols<48>(tile, srow, 0, sv);
  tmem_ldn<2>(tstate + lq + 48, sv);  // columns 48-79: the rest and the vector column
  if (has_s) {
    tile_put_cols<16>(tile, srow, 48, sv);
    const float z8[8] = {sv[16], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    st_row_chunk(tile + 8192, srow, 0, z8);
  }
}

// Zeroes the second atoms (tile + 8192, [64][64]) of `n` state tiles spaced
// `stride` bytes apart, except their column 0 which state_to_tile writes.
__device__ __forceinline__ void zero_state_atoms(uint8_t* tile, int stride, int n, int t, int nthr) {
  for (int v = t; v < n * 512; v += nthr) {
    const int r = (v >> 3) & 63;
    if ((v & 7) != (r & 7))
      *reinterpret_cast<uint4*>(tile + (v >> 9) * stride + 8192 + (v & 511) * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Sum of records [lo, hi) of an [64][80] fp32 state spaced `stride` floats
// apart, by 256 threads (t = 0 .. 255, 20 values each), into the fp32
// [64][80] scratch `scr`.  Two records per round trip.
__device__ __forceinline__ void sum_records(const float* rec0, long stride, int lo, int hi, int t,
                                            float* scr) {
  float acc[20];
#pragma unroll
  for (int j = 0; j < 20; ++j) acc[j] = 0.f;
  int pp = lo;
  for (; pp + 1 < hi; pp += 2) {
    const float4* r0 = reinterpret_cast<const float4*>(rec0 + pp * stride) + t * 5;
    const float4* r1 = reinterpret_cast<const float4*>(rec0 + (pp + 1) * stride) + t * 5;
    float4 x[10];
#pragma unroll
    for (int j = 0; j < 5; ++j) {
      x[j] = r0[j];
      x[5 + j] = r1[j];
    }
#pragma unroll
    for (int j = 0; j < 5; ++j) {
      acc[4 * j] += x[j].x + x[5 + j].x;
      acc[4 * j + 1] += x[j].y + x[5 + j].y;
      acc[4 * j + 2] += x[j].z + x[5 + j].z;
      acc[4 * j + 3] += x[j].w + x[5 + j].w;
    }
  }
  if (pp < hi) {
    const float4* r0 = reinterpret_cast<const float4*>(rec0 + pp * stride) + t * 5;
#pragma unroll
    for (int j = 0; j < 5; ++j) {
      const float4 x = r0[j];
      acc[4 * j] += x.x;
      acc[4 * j + 1] += x.y;
      acc[4 * j + 2] += x.z;
      acc[4 * j + 3] += x.w;
    }
  }
  float4* d = reinterpret_cast<float4*>(scr) + t * 5;
#pragma unroll
  for (int j = 0; j < 5; ++j) d[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
}

// The initial carried state from the fp32 scratch written by sum_records:
// into tensor memory (80 columns at tstate) and, as bf16, into the operand
// tile (see state_to_tile).  Called by one warpgroup.
__device__ __forceinline__ void scratch_to_state(const float* scr, uint32_t tstate, uint32_t lq,
                                                 int lane, int qd, uint8_t* tile) {
  const bool has_s = lane < 16;
  const int srow = 16 * qd + lane;
  const float4* src = reinterpret_cast<const float4*>(scr) + srow * 20;
#pragma unroll
  for (int j = 0; j < 5; ++j) {  // 16 columns at a time
    float sv[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 x = has_s ? src[4 * j + i] : make_float4(0.f, 0.f, 0.f, 0.f);
      sv[4 * i] = x.x;
      sv[4 * i + 1] = x.y;
      sv[4 * i + 2] = x.z;
      sv[4 * i + 3] = x.w;
    }
    tmem_st16(tstate + lq + 16 * j, sv);
    if (has_s) {
      if (j < 4) {
        tile_put_cols<16>(tile, srow, 16 * j, sv);
      } else {
        const float z8[8] = {sv[0], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        st_row_chunk(tile + 8192, srow, 0, z8);
      }
    }
  }
  tmem_st_wait();
}

// min(phi(x), 1) = phi'(x) on 8 bf16 values (one 16-byte vector), as floats.
__device__ __forceinline__ void dphi8(uint4 u, float* f) {
  const uint4 r = phi_vec(u);
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = fminf(__uint_as_float(w[i] << 16), 1.f);
    f[2 * i + 1] = fminf(__uint_as_float(w[i] & 0xffff0000u), 1.f);
  }
}

// Idle accounting of a polling loop: returns false once `limit_ns` have
// passed without progress (the clock is read every 1024 idle polls), else
// sleeps briefly so the other warps of this SM quarter keep the issue slots.
struct PollIdle {
  uint32_t idle = 0;
  uint64_t t0 = 0;
  __device__ __forceinline__ void progress() { idle = 0; }
  __device__ __forceinline__ bool wait(uint64_t limit_ns) {
    if ((++idle & 1023u) != 0) {
      __nanosleep(32);
      return true;
    }
    const uint64_t now = globaltimer_ns();
    if (idle == 1024) t0 = now;
    return now - t0 <= limit_ns;
  }
};

__device__ __forceinline__ void compute_sync() {  // the compute warps only
  asm volatile("bar.sync 1, %0;" ::"n"(NCOMP) : "memory");
}

// Named barrier over the first NCOMP / 2 compute threads (the consumer
// warpgroups of a specialised kernel).
__device__ __forceinline__ void half_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(NCOMP / 2) : "memory");
}

}  // namespace tcc

// Launches `kernel` with programmatic stream serialisation, so that its CTAs
// may start (and run their prologue) while the previous kernel drains.  The
// kernel must call grid_dep_wait() before touching memory the previous
// kernel writes.
template <typename... Exp, typename... Act>
cudaError_t launch_pdl(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

// [BH][N][W] bf16 (W = 16, 32 or 64) viewed as a 3-D TMA tensor with
// 64 x 128 x 1 boxes and the 128-byte swizzle (defined in causal_tc.cu): a
// narrower row arrives zero-filled to 64 columns, and a store writes only
// its W columns.
bool make_bf16_map(CUtensorMap* m, const void* base, int BH, int N, int W = 64);

// [rows][cols] row-major bf16 as a 3-D TMA tensor with 64 x box_rows x 1 boxes
// and the 128-byte swizzle (defined in causal_tc.cu).
bool make_bf16_map_2d(CUtensorMap* m, const void* base, long cols, long rows, int box_rows);

}  // namespace la
