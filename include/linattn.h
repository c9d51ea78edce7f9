/*
 * linattn.h -- C ABI of the GB300 (sm_103a) elu(x)+1 linear-attention library.
 *
 * The operations are those of Katharopoulos et al., "Transformers are RNNs:
 * Fast Autoregressive Transformers with Linear Attention" (part 2/3 of the
 * paper text): the feature map phi(x) = elu(x) + 1 (eq. 7), causal linear
 * attention (§3.3, eq. 9-12), its cumulative-sum gradients (§3.3.1,
 * eq. 13-15, completed with the denominator by the quotient rule), the
 * non-causal form with one shared S and Z ("Linear Attention/zh", kernel
 * reformulation), the RNN-form decode step (§3.4, eq. 16-19), and the
 * prefill that joins the two (the causal form started from a state, which
 * hands its final state to the decode step).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers named q, k, v, out, dout, dq, dk, dv, den, S, Z, x, W, y,
 *    lengths and workspace are DEVICE pointers (or managed memory) of the current CUDA
 *    device.  The caller owns every buffer; the library never allocates,
 *    frees or retains memory and keeps no state between calls other than
 *    one device status word per GPU (see la_device_status).
 *  - Layouts are dense row-major: q, k, dq, dk [B][H][N][D]; v, out, dout, dv
 *    [B][H][N][M]; den [B][H][N]; S [B][H][D][M]; Z [B][H][D]; lengths [B].
 *    Decode tensors drop N: q, k [B][H][D], v, y [B][H][M].
 *  - dtype selects the element type of q, k, v, out, dout, dq, dk, dv and y:
 *    LA_F32 (float) or LA_BF16 (bfloat16).  den, S and Z are always float.
 *    Arithmetic accumulates in fp32.  The feature map uses no 1/sqrt(D)
 *    temperature and the denominator no epsilon.
 *  - Every pointer must be 16-byte aligned.  Supported head sizes: D and M in
 *    {16, 32, 64}.  Limits: 1 <= N <= 2^24; 1 <= B*H <= 65535 for the
 *    sequence calls (causal and non-causal; one grid row per (b, h)) and
 *    1 <= B*H <= 2^20 for la_decode_step.  Larger B*H is refused with
 *    LA_ERR_INVALID_ARG before anything is launched.
 *  - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls are asynchronous on it; results are ready when the
 *    stream reaches them.  Calls that share a workspace must be ordered.
 *  - Return value: LA_OK, or an error code.  Argument errors are detected on
 *    the host before anything is launched, so nothing was written.
 *    LA_ERR_CUDA reports a launch failure (cudaGetLastError after the
 *    launch).  The library never prints, exits or aborts.
 *  - Device-side failures: every wait inside a kernel (on a shared-memory
 *    barrier, a bulk copy or a tensor-core product) is bounded (2 s).  A
 *    wait that runs out stores a nonzero code in the library's status word
 *    on that GPU (the first code sticks), and the kernel unwinds: it drains
 *    its own copies and products with bounded waits, frees its tensor
 *    memory and returns, leaving its outputs undefined and the CUDA context
 *    usable.  la_device_status reports and clears it.
 *  - Workspace: calls that take `workspace` need at least
 *    la_workspace_bytes(op, ...) bytes of device scratch (may be NULL when
 *    that size is 0).  Its contents on entry do not matter and are garbage on
 *    return.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  la_status is an int in the ABI (every call returns one);
 * the values are fixed. */
typedef int la_status;
enum {
  LA_OK = 0,
  LA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, bad dtype */
  LA_ERR_UNSUPPORTED = 2, /* valid but unsupported (D or M not in the set) */
  LA_ERR_CUDA = 3,        /* a CUDA launch or runtime call failed */
  LA_ERR_TIMEOUT = 4,     /* a bounded wait inside a kernel ran out (la_device_status) */
  LA_ERR_WORKSPACE = 5    /* workspace missing or smaller than required */
};

/* Element types.  la_dtype is an int in the ABI. */
typedef int la_dtype;
enum { LA_F32 = 0, LA_BF16 = 1 };

/* operation ids for la_workspace_bytes */
#define LA_OP_CAUSAL_FWD 0
#define LA_OP_CAUSAL_BWD 1
#define LA_OP_NONCAUSAL_FWD 2
#define LA_OP_NONCAUSAL_BWD 3
#define LA_OP_DECODE 4
#define LA_OP_CAUSAL_PREFILL 5
#define LA_OP_CAUSAL_FWD_DECAY 6
#define LA_OP_CAUSAL_BWD_DECAY 7
#define LA_OP_DECODE_PROJ 8 /* the N argument is d_model */
#define LA_OP_CAUSAL_FWD_POLY 9
#define LA_OP_CAUSAL_BWD_POLY 10

/* Human-readable name of a status code (static string, never NULL). */
const char* la_status_string(la_status status);

/* ABI version of this header (major * 100 + minor). */
int la_version(void);

/* Bytes of device workspace the operation needs for these sizes; 0 when it
 * needs none or when the arguments are invalid. */
size_t la_workspace_bytes(int op, int B, int H, int N, int D, int M, la_dtype dtype);

/* Number of kernel launches one call of `op` makes for these sizes (for
 * launch accounting by callers and benchmarks); 0 for invalid arguments. */
int la_kernel_launches(int op, int B, int H, int N, int D, int M, la_dtype dtype);

/*
 * Causal forward, eq. 9-12:
 *   S_i = sum_{j<=i} phi(K_j) V_j^T,  Z_i = sum_{j<=i} phi(K_j),
 *   out_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i,   den_i = phi(Q_i)^T Z_i.
 * Inputs q, k, v; outputs out (dtype) and den (float, may be NULL when no
 * backward pass follows; la_causal_bwd needs it).
 */
la_status la_causal_fwd(const void* q, const void* k, const void* v, void* out, float* den,
                  void* workspace, size_t workspace_bytes, int B, int H, int N, int D,
                  int M, la_dtype dtype, void* stream);

/*
 * Causal backward: gradients of L = sum_i dout_i . out_i with respect to q, k
 * and v, by the cumulative sums of eq. 13-15 (forward sum of S for dq,
 * reverse sums of phi(Q) (dout/den)^T for dk and dv) plus the denominator
 * terms.  No S_i is stored.  out and den are the forward's outputs.
 * Outputs dq, dk (dtype, [B][H][N][D]) and dv ([B][H][N][M]).
 */
la_status la_causal_bwd(const void* q, const void* k, const void* v, const void* out,
                  const float* den, const void* dout, void* dq, void* dk, void* dv,
                  void* workspace, size_t workspace_bytes, int B, int H, int N, int D,
                  int M, la_dtype dtype, void* stream);

/*
 * Prefill: the causal forward started from the state (S, Z) instead of zero,
 * i.e. the RNN form of §3.4 eq. 16-19 run over a whole prompt:
 *   S_i = S + sum_{j<=i} phi(k_j) v_j^T,   Z_i = Z + sum_{j<=i} phi(k_j),
 *   out_i = phi(q_i)^T S_i / phi(q_i)^T Z_i,   den_i = phi(q_i)^T Z_i.
 * On return S and Z hold S_N and Z_N, the state after the last token, from
 * which la_decode_step continues (the two compose: prefill of a prompt, then
 * decode steps, equals prefill of the whole sequence).  S [B][H][D][M] and
 * Z [B][H][D] are fp32, read and updated in place; zeros give la_causal_fwd
 * plus the final state.  den may be NULL.  Needs la_workspace_bytes(
 * LA_OP_CAUSAL_PREFILL, ...) bytes of workspace; other arguments and errors
 * as la_causal_fwd.
 */
la_status la_causal_prefill(const void* q, const void* k, const void* v, void* out, float* den,
                      float* S, float* Z, void* workspace, size_t workspace_bytes, int B, int H,
                      int N, int D, int M, la_dtype dtype, void* stream);

/*
 * la_causal_fwd for callers that cannot allocate device memory: the same
 * operation and arguments minus the workspace, which is taken from a fixed
 * scratch array built into the library (LA_NOALLOC_SCRATCH_BYTES per GPU that
 * loads the library, held until the process exits).  The paper has no
 * counterpart; this exists for code that runs inside a host application that
 * owns all device memory (e.g. a plug-in with a fixed memory budget) or in
 * loops where a cudaMalloc, which may synchronise the device, is not allowed.
 *  - Returns LA_ERR_WORKSPACE, launching nothing, when the problem needs more
 *    scratch than the array holds (la_workspace_bytes(LA_OP_CAUSAL_FWD, ...) >
 *    LA_NOALLOC_SCRATCH_BYTES); other errors as la_causal_fwd.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and keeps it for later calls; make that first call
 *    before any stream capture, and do not reset the device (cudaDeviceReset)
 *    after it, since the kept address would then be stale.
 *  - Argument errors are reported exactly as la_causal_fwd reports them, and
 *    before anything touches the device.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents; calls that overlap on the GPU (other streams, other threads)
 *    race on it, so order them on one stream or serialise them.
 */
#define LA_NOALLOC_SCRATCH_BYTES (4u << 20)
la_status la_causal_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* den,
                          int B, int H, int N, int D, int M, la_dtype dtype, void* stream);

/*
 * Non-causal forward with one shared state per (b, h):
 *   S = sum_{j<L_b} phi(K_j) V_j^T,  Z = sum_{j<L_b} phi(K_j),
 *   out_i = phi(Q_i)^T S / phi(Q_i)^T Z  for i < L_b, and 0 for i >= L_b.
 * lengths: device int32 [B] of valid lengths (values are clamped to [0, N]),
 * or NULL for "all N".  Outputs out, den (0 on padded rows), S and Z (both
 * required: the backward pass reads them).
 */
la_status la_noncausal_fwd(const void* q, const void* k, const void* v, const int* lengths,
                     void* out, float* den, float* S, float* Z, void* workspace,
                     size_t workspace_bytes, int B, int H, int N, int D, int M, la_dtype dtype,
                     void* stream);

/*
 * Non-causal backward: gradients of L = sum_i dout_i . out_i over the valid
 * rows; eq. 13-15 with full sums in place of cumulative ones.  Padded rows
 * of dq, dk, dv are written as 0.  out, den, S, Z come from la_noncausal_fwd.
 */
la_status la_noncausal_bwd(const void* q, const void* k, const void* v, const int* lengths,
                     const void* out, const float* den, const float* S, const float* Z,
                     const void* dout, void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, int B, int H, int N, int D, int M, la_dtype dtype,
                     void* stream);

/*
 * One RNN decode step for B*H independent streams, eq. 16-19 (state update,
 * then read-out; the layer's f_l and residual of eq. 20 are not applied):
 *   S <- S + phi(k) v^T,  Z <- Z + phi(k),  y = phi(q)^T S / phi(q)^T Z.
 * S [B][H][D][M] and Z [B][H][D] are read and updated in place (start from
 * zeros for eq. 16-17).  q, k [B][H][D], v and y [B][H][M] in dtype.
 * Needs no workspace.
 */
la_status la_decode_step(const void* q, const void* k, const void* v, float* S, float* Z,
                   void* y, int B, int H, int D, int M, la_dtype dtype, void* stream);

/*
 * The RetNet decay ("Linear Attention/zh", variants and extensions): the
 * causal sums become S_i = gamma S_{i-1} + phi(K_i) V_i^T and, so that the
 * output stays a weighted mean of the values, Z_i = gamma Z_{i-1} + phi(K_i):
 *   out_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i
 *         = sum_{j<=i} gamma^(i-j) phi(Q_i).phi(K_j) V_j / sum_{j<=i} gamma^(i-j) phi(Q_i).phi(K_j),
 * den_i = phi(Q_i)^T Z_i.  gamma must lie in [0, 1] (else LA_ERR_INVALID_ARG);
 * gamma = 1 is la_causal_fwd's operation and gamma = 0 returns V.  Both
 * calls run on the tensor cores for the shapes la_causal_fwd runs there (bf16,
 * D and M in {16, 32, 64}) when gamma >= 0.75, else on the CUDA cores.  They
 * take the workspace of
 * la_workspace_bytes(LA_OP_CAUSAL_FWD_DECAY / _BWD_DECAY, ...) (enough for
 * either path; la_kernel_launches counts the tensor-core path where it applies);
 * other arguments and errors as la_causal_fwd / la_causal_bwd.
 * la_causal_bwd_decay's out and den are la_causal_fwd_decay's, with the same
 * gamma.
 */
la_status la_causal_fwd_decay(const void* q, const void* k, const void* v, void* out, float* den,
                              float gamma, void* workspace, size_t workspace_bytes, int B, int H,
                              int N, int D, int M, la_dtype dtype, void* stream);
la_status la_causal_bwd_decay(const void* q, const void* k, const void* v, const void* out,
                              const float* den, const void* dout, void* dq, void* dk, void* dv,
                              float gamma, void* workspace, size_t workspace_bytes, int B, int H,
                              int N, int D, int M, la_dtype dtype, void* stream);

/*
 * One decayed RNN step (the decode step of the decayed causal form):
 *   S <- gamma S + phi(k) v^T,  Z <- gamma Z + phi(k),  y = phi(q)^T S / phi(q)^T Z.
 * gamma in [0, 1]; arguments otherwise as la_decode_step.
 */
la_status la_decode_step_decay(const void* q, const void* k, const void* v, float* S, float* Z,
                               void* y, float gamma, int B, int H, int D, int M, la_dtype dtype,
                               void* stream);

/*
 * Causal linear attention with the degree-2 polynomial kernel ("Transformers
 * are RNNs", part 2/3, the feature-map discussion before eq. 7: an exact finite
 * feature map, O(N D^2 M) at degree 2), read as sim(q, k) = (q . k)^2 in
 * eq. 8-12 with no elu feature map:
 *   out_i = sum_{j<=i} (Q_i . K_j)^2 V_j / den_i,  den_i = sum_{j<=i} (Q_i . K_j)^2,
 * and its gradients.  bf16 only (LA_F32 gives LA_ERR_UNSUPPORTED); D in [1, 10]
 * (the D (D + 1) / 2 features fill at most a 64-wide row; larger D gives
 * LA_ERR_UNSUPPORTED); M in {16, 32, 64}; q, k [B][H][N][D], v, out, dout, dv
 * [B][H][N][M], den [B][H][N] float (may be NULL in the forward).  A
 * denominator of zero (every Q_i . K_j = 0 for j <= i) gives a non-finite row.
 * Workspace: la_workspace_bytes(LA_OP_CAUSAL_FWD_POLY / _BWD_POLY, ...) bytes
 * (it holds the feature rows); errors and the rest as la_causal_fwd / _bwd.
 */
la_status la_causal_fwd_poly(const void* q, const void* k, const void* v, void* out, float* den,
                             void* workspace, size_t workspace_bytes, int B, int H, int N, int D,
                             int M, la_dtype dtype, void* stream);
la_status la_causal_bwd_poly(const void* q, const void* k, const void* v, const void* out,
                             const float* den, const void* dout, void* dq, void* dk, void* dv,
                             void* workspace, size_t workspace_bytes, int B, int H, int N, int D,
                             int M, la_dtype dtype, void* stream);

/*
 * One RNN decode step fed by its own projection: "Transformers are RNNs"
 * (part 2/3) §3.4 eq. 18-20 without the layer's f_l and residual, for B
 * streams of H heads.  Per stream b and head h,
 *   [q | k | v] = x_b W[:, h (2D+M) : (h+1) (2D+M)]   (q, k: D columns; v: M),
 *   S <- S + phi(k) v^T,  Z <- Z + phi(k),  y = phi(q)^T S / phi(q)^T Z.
 * x [B][d_model] and W [d_model][H (2D+M)] are bf16 (row-major; the columns of
 * W hold head 0's q, k, v side by side, then head 1's, ...); y [B][H][M] is
 * bf16; S [B][H][D][M] and Z [B][H][D] are float, updated in place.  The
 * projection accumulates in fp32 on the tensor cores; phi and the step are
 * fp32.  dtype must be LA_BF16 (LA_F32 gives LA_ERR_UNSUPPORTED); d_model a
 * multiple of 64 in [64, 16384] (else LA_ERR_UNSUPPORTED when positive,
 * LA_ERR_INVALID_ARG when not); 1 <= B*H <= 2^20, H <= 65535; D, M in {16,
 * 32, 64}.  Needs no workspace; one kernel launch.
 */
la_status la_decode_step_proj(const void* x, const void* W, float* S, float* Z, void* y, int B,
                              int H, int d_model, int D, int M, la_dtype dtype, void* stream);

/*
 * Reads the status word of the current GPU after all work queued on
 * `stream` so far (the call synchronises `stream`; other streams' work is
 * covered once it has finished).  Returns LA_OK when no bounded wait has
 * run out since the word was last cleared, LA_ERR_TIMEOUT when one has, and
 * LA_ERR_CUDA when the stream or the copy fails.  *code (if code is not
 * NULL) receives the word: 0, or the code of the first wait that ran out
 * (a small integer naming the kernel and the wait).  clear != 0 resets the
 * word to 0 after reading it.  The first call on a device (this one or any
 * compute call) looks up the word's device address with that device
 * current.
 */
la_status la_device_status(void* stream, int clear, int* code);

/*
 * Diagnostic: launches on `stream` one kernel that waits, with the bounded
 * wait every kernel uses, on a shared-memory barrier that nothing arrives
 * at, for limit_ns nanoseconds (1 .. 10^9), and then records code 99 in the
 * status word and returns.  It shows that a wait which runs out reaches the
 * host as LA_ERR_TIMEOUT and that the context stays usable.  Returns
 * LA_ERR_INVALID_ARG for a limit outside the range (nothing launched).
 */
la_status la_selftest_wait(void* stream, unsigned long long limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
