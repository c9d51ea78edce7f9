// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace la {

// The device address of the library's status word on the current device
// (nullptr if it cannot be had): kernels whose bounded waits run out store
// a nonzero code there; la_device_status reads it.
int* status_word();

// Streaming multiprocessors of the current device (cudaDevAttrMultiProcessorCount,
// cached per device); 152, GB300's count, when no device can be queried (so
// workspace sizes can be computed on a machine without one).
int sm_count();

constexpr int kChunk = 64;  // tokens per chunk in the CUDA-core kernels

// Split of each (b, h) sequence into segments of whole chunks.
struct SegPlan {
  int nseg;     // segments per (b, h)
  int seg_len;  // tokens per segment (a multiple of the chunk length)
};

// Segments are sized to fill the SMs twice unless `target` says otherwise.
inline SegPlan plan_segments(int BH, int N, int chunk = kChunk, int target = 0) {
  if (target <= 0) target = 2 * sm_count();
  const int nch = (N + chunk - 1) / chunk;
  int want = (target + BH - 1) / BH;
  if (want < 1) want = 1;
  if (want > nch) want = nch;
  const int per = (nch + want - 1) / want;  // chunks per segment
  SegPlan p;
  p.seg_len = per * chunk;
  p.nseg = (N + p.seg_len - 1) / p.seg_len;
  return p;
}

// The argument checks of la_causal_fwd other than the workspace (shape,
// dtype, pointers): LA_OK or the error code that call would return.
int causal_fwd_check(const void* q, const void* k, const void* v, const void* out,
                     const float* den, int B, int H, int N, int D, int M, int dtype);

struct Shape {
  int B, H, N, D, M;
  int dtype;  // 0 = fp32, 1 = bf16
};

// Workspace (floats) each path needs.
size_t causal_fwd_ws_floats(const Shape& s);
size_t causal_bwd_ws_floats(const Shape& s);
size_t noncausal_fwd_ws_floats(const Shape& s);
size_t noncausal_bwd_ws_floats(const Shape& s);

// Kernel launches per call (must match the launchers below).
int causal_fwd_launches(const Shape& s);
int causal_bwd_launches(const Shape& s);
int noncausal_fwd_launches(const Shape& s);
int noncausal_bwd_launches(const Shape& s);

// In-place exclusive scans over the nseg records (stride floats each) of
// every (b, h) in ws: entries [0, wf) become prefix sums over earlier
// records, entries [ro, ro + wr) suffix sums over later records.
void k_seg_scan_ext(float* ws, int BH, int nseg, int stride, int wf, int ro, int wr,
                    cudaStream_t st);

// (S, Z)[bh] += the sum of records r0 .. r1 - 1 of ws[bh] (nrec records of
// rstride floats per (b, h)); a record holds S[d][m] at d * srow + m and z[d]
// at zoff + d * zstride.  One launch.
cudaError_t state_add_records(const float* ws, int BH, int nrec, int rstride, int r0, int r1, int D,
                              int M, int srow, int zoff, int zstride, float* S, float* Z,
                              cudaStream_t st);

// The causal forward from the state (S, Z), which then holds the state after
// the sequence (eq. 16-19 over a prompt).  CUDA cores: four launches;
// tcgen05: three.
size_t causal_prefill_ws_floats(const Shape& s);
cudaError_t causal_prefill_cc(const void* q, const void* k, const void* v, void* out, float* den,
                              float* S, float* Z, float* ws, const Shape& s, cudaStream_t st);
cudaError_t causal_prefill_tc(const void* q, const void* k, const void* v, void* out, float* den,
                              float* S, float* Z, float* ws, const Shape& s, cudaStream_t st);

// tcgen05 path (bf16, D and M in {16, 32, 64}).
SegPlan tc_plan(int BH, int N);
bool tc_eligible(const Shape& s);          // causal fwd / bwd on the tensor cores
bool tc_prefill_eligible(const Shape& s);  // the prefill on the tensor cores (D = M = 64)
size_t causal_fwd_tc_ws_floats(const Shape& s);
int causal_fwd_tc_launches(const Shape& s);
// feat: q and k already hold features (a feature map applied before the call,
// e.g. the degree-2 polynomial one); the kernels then apply no phi.
// gamma: the RetNet decay (1 = none); the tensor-core forward takes gamma in
// [TC_DECAY_MIN, 1] (its row and column factors stay inside fp32 and bf16).
constexpr float TC_DECAY_MIN = 0.75f;
cudaError_t causal_fwd_tc(const void* q, const void* k, const void* v, void* out, float* den,
                          float* ws, const Shape& s, cudaStream_t st, bool feat = false,
                          float gamma = 1.f);
size_t causal_bwd_tc_ws_floats(const Shape& s);
int causal_bwd_tc_launches(const Shape& s);
cudaError_t causal_bwd_tc(const void* q, const void* k, const void* v, const void* out,
                          const float* den, const void* dout, void* dq, void* dk, void* dv,
                          float* ws, const Shape& s, cudaStream_t st, bool feat = false,
                          float gamma = 1.f);

// The degree-2 polynomial kernel (poly.cu): features f(x) = [x_a^2, sqrt(2)
// x_a x_b (a < b)] zero-padded to 64, then the tensor-core kernels with
// feat = true; D in [1, 10], bf16.  Workspace: the feature tensors (and
// their gradients) followed by the tensor-core workspace.
constexpr int POLY_MAX_D = 10;
size_t causal_poly_ws_bytes(const Shape& s, bool bwd);
int causal_poly_launches(const Shape& s, bool bwd);
cudaError_t causal_fwd_poly(const void* q, const void* k, const void* v, void* out, float* den,
                            void* ws, const Shape& s, cudaStream_t st);
cudaError_t causal_bwd_poly(const void* q, const void* k, const void* v, const void* out,
                            const float* den, const void* dout, void* dq, void* dk, void* dv,
                            void* ws, const Shape& s, cudaStream_t st);

// CUDA-core (FFMA) paths; every kernel of the library is launched from these.
// gamma: the RetNet decay in [0, 1] (1 = the undecayed method).
cudaError_t causal_fwd_cc(const void* q, const void* k, const void* v, void* out, float* den,
                          float* ws, const Shape& s, cudaStream_t st, float gamma = 1.f);
cudaError_t causal_bwd_cc(const void* q, const void* k, const void* v, const void* out,
                          const float* den, const void* dout, void* dq, void* dk, void* dv,
                          float* ws, const Shape& s, cudaStream_t st, float gamma = 1.f);
cudaError_t noncausal_fwd_cc(const void* q, const void* k, const void* v, const int* lengths,
                             void* out, float* den, float* S, float* Z, float* ws, const Shape& s,
                             cudaStream_t st);
cudaError_t noncausal_bwd_cc(const void* q, const void* k, const void* v, const int* lengths,
                             const void* out, const float* den, const float* S, const float* Z,
                             const void* dout, void* dq, void* dk, void* dv, float* ws,
                             const Shape& s, cudaStream_t st);
// Non-causal path for D = M = 64 (fp32 or bf16) on the tensor cores: one
// cluster launch per direction, no workspace.
int noncausal_tc_nseg(int BH, int N);
cudaError_t noncausal_tc_fwd(const void* q, const void* k, const void* v, const int* lengths,
                             void* out, float* den, float* S, float* Z, const Shape& s,
                             cudaStream_t st);
cudaError_t noncausal_tc_bwd(const void* q, const void* k, const void* v, const int* lengths,
                             const float* den, const float* S, const float* Z, const void* dout,
                             void* dq, void* dk, void* dv, const Shape& s, cudaStream_t st);
// gamma: the RetNet decay (1 = the undecayed step).
cudaError_t decode_step(const void* q, const void* k, const void* v, float* S, float* Z, void* y,
                        const Shape& s, cudaStream_t st, float gamma = 1.f);
// The decode step fed by its projection (decode_proj.cu): x [B][dm] and W
// [dm][H (2D+M)] in bf16, d_model dm a multiple of 64; streams per CTA.
cudaError_t decode_step_proj(const void* x, const void* W, float* S, float* Z, void* y, int B,
                             int H, int dm, int D, int M, cudaStream_t st);
struct ProjPlan {
  int SB;  // streams per CTA
  int NS;  // stages of the slab ring
};
ProjPlan decode_proj_plan(int B, int H);
int decode_proj_block(int B, int H);

}  // namespace la

// Expands BODY once per supported (D, M) pair with constexpr D_ and M_ in scope.
#define LA_DISPATCH_DM(Dv, Mv, BODY)                         \
  switch ((Dv) * 1000 + (Mv)) {                              \
    case 16016: { constexpr int D_ = 16, M_ = 16; BODY; } break; \
    case 16032: { constexpr int D_ = 16, M_ = 32; BODY; } break; \
    case 16064: { constexpr int D_ = 16, M_ = 64; BODY; } break; \
    case 32016: { constexpr int D_ = 32, M_ = 16; BODY; } break; \
    case 32032: { constexpr int D_ = 32, M_ = 32; BODY; } break; \
    case 32064: { constexpr int D_ = 32, M_ = 64; BODY; } break; \
    case 64016: { constexpr int D_ = 64, M_ = 16; BODY; } break; \
    case 64032: { constexpr int D_ = 64, M_ = 32; BODY; } break; \
    case 64064: { constexpr int D_ = 64, M_ = 64; BODY; } break; \
    default: return cudaErrorInvalidValue;                   \
  }
