// C ABI of the library (declared in include/linattn.h): argument checks,
// workspace sizing and dispatch to the kernel launchers.  Nothing here
// allocates device memory, prints or aborts.
#include <stdint.h>

#include <algorithm>
#include <initializer_list>

#include "../../include/linattn.h"
#include "launch.h"

namespace {

using la::Shape;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dim(int x) { return x == 16 || x == 32 || x == 64; }

// Checks shared by all calls; returns LA_OK or the error code.  max_bh is
// the largest B*H the call's grids take (65535 grid rows for the sequence
// calls, 2^20 streams for the decode step).
int check_shape(int B, int H, int N, int D, int M, int dtype, long long max_bh = 65535) {
  if (B < 1 || H < 1 || N < 1) return LA_ERR_INVALID_ARG;
  if ((long long)B * H > max_bh || N > (1 << 24)) return LA_ERR_INVALID_ARG;
  if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
  if (D < 1 || M < 1) return LA_ERR_INVALID_ARG;
  if (!supported_dim(D) || !supported_dim(M)) return LA_ERR_UNSUPPORTED;
  return LA_OK;
}

// Every listed pointer must be non-null and 16-byte aligned.
int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr || !aligned16(p)) return LA_ERR_INVALID_ARG;
  return LA_OK;
}

int check_opt_ptr(const void* p) { return (p == nullptr || aligned16(p)) ? LA_OK : LA_ERR_INVALID_ARG; }

size_t ws_bytes(int op, const Shape& s) {
  switch (op) {
    case LA_OP_CAUSAL_FWD:
      return 4 * (la::tc_eligible(s) ? la::causal_fwd_tc_ws_floats(s) : la::causal_fwd_ws_floats(s));
    case LA_OP_CAUSAL_BWD:
      return 4 * (la::tc_eligible(s) ? la::causal_bwd_tc_ws_floats(s) : la::causal_bwd_ws_floats(s));
    case LA_OP_CAUSAL_PREFILL:
      return 4 * (la::tc_prefill_eligible(s) ? la::causal_fwd_tc_ws_floats(s) : la::causal_prefill_ws_floats(s));
    case LA_OP_CAUSAL_FWD_DECAY:  // either path, whichever gamma picks
      return 4 * (la::tc_eligible(s) ? std::max(la::causal_fwd_tc_ws_floats(s), la::causal_fwd_ws_floats(s))
                                     : la::causal_fwd_ws_floats(s));
    case LA_OP_CAUSAL_BWD_DECAY:  // either path, whichever gamma picks
      return 4 * (la::tc_eligible(s) ? std::max(la::causal_bwd_tc_ws_floats(s), la::causal_bwd_ws_floats(s))
                                     : la::causal_bwd_ws_floats(s));
    case LA_OP_NONCAUSAL_FWD: return 4 * la::noncausal_fwd_ws_floats(s);
    case LA_OP_NONCAUSAL_BWD: return 4 * la::noncausal_bwd_ws_floats(s);
    default: return 0;
  }
}

int check_ws(int op, const Shape& s, const void* ws, size_t bytes) {
  const size_t need = ws_bytes(op, s);
  if (need == 0) return LA_OK;
  if (ws == nullptr || bytes < need) return LA_ERR_WORKSPACE;
  if (!aligned16(ws)) return LA_ERR_INVALID_ARG;
  return LA_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

// The RetNet decay must lie in [0, 1] (a NaN fails both comparisons).
int check_gamma(float gamma) { return (gamma >= 0.f && gamma <= 1.f) ? LA_OK : LA_ERR_INVALID_ARG; }

// Workspace of the polynomial calls (their own op ids: the features live there).
int check_ws_poly(int op, const Shape& s, const void* ws, size_t bytes) {
  const size_t need = la::causal_poly_ws_bytes(s, op == LA_OP_CAUSAL_BWD_POLY);
  if (ws == nullptr || bytes < need) return LA_ERR_WORKSPACE;
  if (!aligned16(ws)) return LA_ERR_INVALID_ARG;
  return LA_OK;
}

// The degree-2 polynomial kernel: D in [1, 10] (its D (D + 1) / 2 features fit
// a 64-wide row), M as elsewhere, bf16 (the tensor-core path).
int check_poly(int B, int H, int N, int D, int M, int dtype) {
  if (B < 1 || H < 1 || N < 1 || D < 1 || M < 1) return LA_ERR_INVALID_ARG;
  if ((long long)B * H > 65535 || N > (1 << 24)) return LA_ERR_INVALID_ARG;
  if ((long long)B * H * N > (1ll << 31)) return LA_ERR_INVALID_ARG;  // the feature kernels' grids
  if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
  if (D > la::POLY_MAX_D || !supported_dim(M) || dtype != LA_BF16) return LA_ERR_UNSUPPORTED;
  return LA_OK;
}

// The projected decode step: B*H streams as for the decode step, H grid rows,
// d_model whole slabs of 64, bf16 only.
int check_proj(int B, int H, int dm, int D, int M, int dtype) {
  const int rc = check_shape(B, H, 1, D, M, dtype, 1ll << 20);
  if (rc != LA_OK) return rc;
  if (H > 65535 || dm < 1) return LA_ERR_INVALID_ARG;
  if (dtype != LA_BF16 || dm % 64 != 0 || dm > 16384) return LA_ERR_UNSUPPORTED;
  return LA_OK;
}

}  // namespace

namespace la {

int causal_fwd_check(const void* q, const void* k, const void* v, const void* out,
                     const float* den, int B, int H, int N, int D, int M, int dtype) {
  int rc = check_shape(B, H, N, D, M, dtype);
  if (rc == LA_OK) rc = check_ptrs({q, k, v, out});
  if (rc == LA_OK) rc = check_opt_ptr(den);
  return rc;
}

}  // namespace la

#define LA_TRY(x)              \
  do {                         \
    const int rc_ = (x);       \
    if (rc_ != LA_OK) return rc_; \
  } while (0)

extern "C" {

const char* la_status_string(int status) {
  switch (status) {
    case LA_OK: return "ok";
    case LA_ERR_INVALID_ARG: return "invalid argument";
    case LA_ERR_UNSUPPORTED: return "unsupported head size";
    case LA_ERR_CUDA: return "CUDA error";
    case LA_ERR_WORKSPACE: return "workspace missing or too small";
    case LA_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    default: return "unknown status";
  }
}

int la_version(void) { return 200; }

size_t la_workspace_bytes(int op, int B, int H, int N, int D, int M, int dtype) {
  if (op == LA_OP_DECODE || op == LA_OP_DECODE_PROJ) return 0;
  if (op == LA_OP_CAUSAL_FWD_POLY || op == LA_OP_CAUSAL_BWD_POLY) {
    if (check_poly(B, H, N, D, M, dtype) != LA_OK) return 0;
    return la::causal_poly_ws_bytes(Shape{B, H, N, D, M, dtype}, op == LA_OP_CAUSAL_BWD_POLY);
  }
  if (check_shape(B, H, N, D, M, dtype) != LA_OK) return 0;
  return ws_bytes(op, Shape{B, H, N, D, M, dtype});
}

int la_kernel_launches(int op, int B, int H, int N, int D, int M, int dtype) {
  if (op == LA_OP_DECODE_PROJ) return check_proj(B, H, N, D, M, dtype) == LA_OK ? 1 : 0;
  if (op == LA_OP_CAUSAL_FWD_POLY || op == LA_OP_CAUSAL_BWD_POLY)
    return check_poly(B, H, N, D, M, dtype) == LA_OK
               ? la::causal_poly_launches(Shape{B, H, N, D, M, dtype}, op == LA_OP_CAUSAL_BWD_POLY)
               : 0;
  if (check_shape(B, H, op == LA_OP_DECODE ? 1 : N, D, M, dtype,
                  op == LA_OP_DECODE ? (1ll << 20) : 65535) != LA_OK)
    return 0;
  const Shape s{B, H, N, D, M, dtype};
  switch (op) {
    case LA_OP_CAUSAL_FWD:
      return la::tc_eligible(s) ? la::causal_fwd_tc_launches(s) : la::causal_fwd_launches(s);
    case LA_OP_CAUSAL_BWD:
      return la::tc_eligible(s) ? la::causal_bwd_tc_launches(s) : la::causal_bwd_launches(s);
    case LA_OP_CAUSAL_PREFILL: return la::tc_prefill_eligible(s) ? 3 : 4;
    case LA_OP_CAUSAL_FWD_DECAY:  // gamma in [0.75, 1] on the tensor-core path
      return la::tc_eligible(s) ? la::causal_fwd_tc_launches(s) : la::causal_fwd_launches(s);
    case LA_OP_CAUSAL_BWD_DECAY:  // gamma in [0.75, 1] on the tensor-core path
      return la::tc_eligible(s) ? la::causal_bwd_tc_launches(s) : la::causal_bwd_launches(s);
    case LA_OP_NONCAUSAL_FWD: return la::noncausal_fwd_launches(s);
    case LA_OP_NONCAUSAL_BWD: return la::noncausal_bwd_launches(s);
    case LA_OP_DECODE: return 1;
    default: return 0;
  }
}

int la_causal_fwd(const void* q, const void* k, const void* v, void* out, float* den,
                  void* workspace, size_t workspace_bytes, int B, int H, int N, int D, int M,
                  int dtype, void* stream) {
  LA_TRY(la::causal_fwd_check(q, k, v, out, den, B, H, N, D, M, dtype));
  const Shape s{B, H, N, D, M, dtype};
  LA_TRY(check_ws(LA_OP_CAUSAL_FWD, s, workspace, workspace_bytes));
  if (la::tc_eligible(s))
    return from_cuda(la::causal_fwd_tc(q, k, v, out, den, static_cast<float*>(workspace), s,
                                       static_cast<cudaStream_t>(stream)));
  return from_cuda(la::causal_fwd_cc(q, k, v, out, den, static_cast<float*>(workspace), s,
                                     static_cast<cudaStream_t>(stream)));
}

int la_causal_prefill(const void* q, const void* k, const void* v, void* out, float* den, float* S,
                      float* Z, void* workspace, size_t workspace_bytes, int B, int H, int N,
                      int D, int M, int dtype, void* stream) {
  LA_TRY(check_shape(B, H, N, D, M, dtype));
  LA_TRY(check_ptrs({q, k, v, out, S, Z}));
  LA_TRY(check_opt_ptr(den));
  const Shape s{B, H, N, D, M, dtype};
  LA_TRY(check_ws(LA_OP_CAUSAL_PREFILL, s, workspace, workspace_bytes));
  if (la::tc_prefill_eligible(s))
    return from_cuda(la::causal_prefill_tc(q, k, v, out, den, S, Z, static_cast<float*>(workspace),
                                           s, static_cast<cudaStream_t>(stream)));
  return from_cuda(la::causal_prefill_cc(q, k, v, out, den, S, Z, static_cast<float*>(workspace), s,
                                         static_cast<cudaStream_t>(stream)));
}

int la_causal_bwd(const void* q, const void* k, const void* v, const void* out, const float* den,
                  const void* dout, void* dq, void* dk, void* dv, void* workspace,
                  size_t workspace_bytes, int B, int H, int N, int D, int M, int dtype,
                  void* stream) {
  LA_TRY(check_shape(B, H, N, D, M, dtype));
  LA_TRY(check_ptrs({q, k, v, out, den, dout, dq, dk, dv}));
  const Shape s{B, H, N, D, M, dtype};
  LA_TRY(check_ws(LA_OP_CAUSAL_BWD, s, workspace, workspace_bytes));
  if (la::tc_eligible(s))
    return from_cuda(la::causal_bwd_tc(q, k, v, out, den, dout, dq, dk, dv,
                                       static_cast<float*>(workspace), s,
                                       static_cast<cudaStream_t>(stream)));
  return from_cuda(la::causal_bwd_cc(q, k, v, out, den, dout, dq, dk, dv,
                                     static_cast<float*>(workspace), s,
                                     static_cast<cudaStream_t>(stream)));
}

int la_noncausal_fwd(const void* q, const void* k, const void* v, const int* lengths, void* out,
                     float* den, float* S, float* Z, void* workspace, size_t workspace_bytes,
                     int B, int H, int N, int D, int M, int dtype, void* stream) {
  LA_TRY(check_shape(B, H, N, D, M, dtype));
  LA_TRY(check_ptrs({q, k, v, out, S, Z}));
  LA_TRY(check_opt_ptr(den));
  LA_TRY(check_opt_ptr(lengths));
  const Shape s{B, H, N, D, M, dtype};
  LA_TRY(check_ws(LA_OP_NONCAUSAL_FWD, s, workspace, workspace_bytes));
  return from_cuda(la::noncausal_fwd_cc(q, k, v, lengths, out, den, S, Z,
                                        static_cast<float*>(workspace), s,
                                        static_cast<cudaStream_t>(stream)));
}

int la_noncausal_bwd(const void* q, const void* k, const void* v, const int* lengths,
                     const void* out, const float* den, const float* S, const float* Z,
                     const void* dout, void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, int B, int H, int N, int D, int M, int dtype,
                     void* stream) {
  LA_TRY(check_shape(B, H, N, D, M, dtype));
  LA_TRY(check_ptrs({q, k, v, out, den, S, Z, dout, dq, dk, dv}));
  LA_TRY(check_opt_ptr(lengths));
  const Shape s{B, H, N, D, M, dtype};
  LA_TRY(check_ws(LA_OP_NONCAUSAL_BWD, s, workspace, workspace_bytes));
  return from_cuda(la::noncausal_bwd_cc(q, k, v, lengths, out, den, S, Z, dout, dq, dk, dv,
                                        static_cast<float*>(workspace), s,
                                        static_cast<cudaStream_t>(stream)));
}

int la_causal_fwd_decay(const void* q, const void* k, const void* v, void* out, float* den,
                        float gamma, void* workspace, size_t workspace_bytes, int B, int H, int N,
                        int D, int M, int dtype, void* stream) {
  LA_TRY(la::causal_fwd_check(q, k, v, out, den, B, H, N, D, M, dtype));
  LA_TRY(check_gamma(gamma));
  const Shape s{B, H, N, D, M, dtype};
  LA_TRY(check_ws(LA_OP_CAUSAL_FWD_DECAY, s, workspace, workspace_bytes));
  if (la::tc_eligible(s) && gamma >= la::TC_DECAY_MIN)
    return from_cuda(la::causal_fwd_tc(q, k, v, out, den, static_cast<float*>(workspace), s,
                                       static_cast<cudaStream_t>(stream), false, gamma));
  return from_cuda(la::causal_fwd_cc(q, k, v, out, den, static_cast<float*>(workspace), s,
                                     static_cast<cudaStream_t>(stream), gamma));
}

int la_causal_bwd_decay(const void* q, const void* k, const void* v, const void* out,
                        const float* den, const void* dout, void* dq, void* dk, void* dv,
                        float gamma, void* workspace, size_t workspace_bytes, int B, int H, int N,
                        int D, int M, int dtype, void* stream) {
  LA_TRY(check_shape(B, H, N, D, M, dtype));
  LA_TRY(check_ptrs({q, k, v, out, den, dout, dq, dk, dv}));
  LA_TRY(check_gamma(gamma));
  const Shape s{B, H, N, D, M, dtype};
  LA_TRY(check_ws(LA_OP_CAUSAL_BWD_DECAY, s, workspace, workspace_bytes));
  if (la::tc_eligible(s) && gamma >= la::TC_DECAY_MIN)
    return from_cuda(la::causal_bwd_tc(q, k, v, out, den, dout, dq, dk, dv,
                                       static_cast<float*>(workspace), s,
                                       static_cast<cudaStream_t>(stream), false, gamma));
  return from_cuda(la::causal_bwd_cc(q, k, v, out, den, dout, dq, dk, dv,
                                     static_cast<float*>(workspace), s,
                                     static_cast<cudaStream_t>(stream), gamma));
}

int la_decode_step_decay(const void* q, const void* k, const void* v, float* S, float* Z, void* y,
                         float gamma, int B, int H, int D, int M, int dtype, void* stream) {
  LA_TRY(check_shape(B, H, 1, D, M, dtype, 1ll << 20));
  LA_TRY(check_ptrs({q, k, v, S, Z, y}));
  LA_TRY(check_gamma(gamma));
  const Shape s{B, H, 1, D, M, dtype};
  return from_cuda(la::decode_step(q, k, v, S, Z, y, s, static_cast<cudaStream_t>(stream), gamma));
}

int la_decode_step_proj(const void* x, const void* W, float* S, float* Z, void* y, int B, int H,
                        int d_model, int D, int M, int dtype, void* stream) {
  LA_TRY(check_proj(B, H, d_model, D, M, dtype));
  LA_TRY(check_ptrs({x, W, S, Z, y}));
  return from_cuda(la::decode_step_proj(x, W, S, Z, y, B, H, d_model, D, M,
                                        static_cast<cudaStream_t>(stream)));
}

int la_causal_fwd_poly(const void* q, const void* k, const void* v, void* out, float* den,
                       void* workspace, size_t workspace_bytes, int B, int H, int N, int D, int M,
                       int dtype, void* stream) {
  LA_TRY(check_poly(B, H, N, D, M, dtype));
  LA_TRY(check_ptrs({q, k, v, out}));
  LA_TRY(check_opt_ptr(den));
  const Shape s{B, H, N, D, M, dtype};
  LA_TRY(check_ws_poly(LA_OP_CAUSAL_FWD_POLY, s, workspace, workspace_bytes));
  return from_cuda(la::causal_fwd_poly(q, k, v, out, den, workspace, s, static_cast<cudaStream_t>(stream)));
}

int la_causal_bwd_poly(const void* q, const void* k, const void* v, const void* out, const float* den,
                       const void* dout, void* dq, void* dk, void* dv, void* workspace,
                       size_t workspace_bytes, int B, int H, int N, int D, int M, int dtype,
                       void* stream) {
  LA_TRY(check_poly(B, H, N, D, M, dtype));
  LA_TRY(check_ptrs({q, k, v, out, den, dout, dq, dk, dv}));
  const Shape s{B, H, N, D, M, dtype};
  LA_TRY(check_ws_poly(LA_OP_CAUSAL_BWD_POLY, s, workspace, workspace_bytes));
  return from_cuda(la::causal_bwd_poly(q, k, v, out, den, dout, dq, dk, dv, workspace, s,
                                       static_cast<cudaStream_t>(stream)));
}

int la_decode_step(const void* q, const void* k, const void* v, float* S, float* Z, void* y,
                   int B, int H, int D, int M, int dtype, void* stream) {
  LA_TRY(check_shape(B, H, 1, D, M, dtype, 1ll << 20));
  LA_TRY(check_ptrs({q, k, v, S, Z, y}));
  const Shape s{B, H, 1, D, M, dtype};
  return from_cuda(la::decode_step(q, k, v, S, Z, y, s, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
