"""GB300 (sm_103a) elu(x)+1 linear attention: Python binding of the C ABI.

This module only marshals arguments: it loads ``_lib/liblinattn.so`` (built by
``_build.py``), passes tensor data pointers and the current CUDA stream to the
C entry points declared in ``include/linattn.h``, and turns error codes into
exceptions.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback of any kind, and using any entry point without
the built library raises.

Raw entry points (same names and argument order as the C ABI, tensors in
place of pointers): ``la_causal_fwd``, ``la_causal_bwd``, ``la_causal_prefill``,
``la_noncausal_fwd``, ``la_noncausal_bwd``, ``la_decode_step``, the decayed
``la_causal_fwd_decay``, ``la_causal_bwd_decay``, ``la_decode_step_decay``, the projected
``la_decode_step_proj``, the degree-2 polynomial ``la_causal_fwd_poly``,
``la_causal_bwd_poly``, ``la_workspace_bytes``, ``la_device_status``.
Convenience wrappers that allocate outputs with torch: ``causal_fwd``,
``causal_bwd``, ``causal_prefill``, ``noncausal_fwd``, ``noncausal_bwd``, ``decode_step``, ``decode_step_proj``,
``causal_fwd_poly``, ``causal_bwd_poly`` and the
autograd functions ``causal_linear_attention`` / ``noncausal_linear_attention``.

The method is Katharopoulos et al., "Transformers are RNNs" (part 2/3):
eq. 7 (phi), §3.3 eq. 9-12, §3.3.1 eq. 13-15, §3.4 eq. 16-20.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "liblinattn.so")

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT, LA_ERR_WORKSPACE = range(6)
LA_F32, LA_BF16 = 0, 1
(LA_OP_CAUSAL_FWD, LA_OP_CAUSAL_BWD, LA_OP_NONCAUSAL_FWD, LA_OP_NONCAUSAL_BWD, LA_OP_DECODE,
 LA_OP_CAUSAL_PREFILL, LA_OP_CAUSAL_FWD_DECAY, LA_OP_CAUSAL_BWD_DECAY, LA_OP_DECODE_PROJ,
 LA_OP_CAUSAL_FWD_POLY, LA_OP_CAUSAL_BWD_POLY) = range(11)

# exported symbols and their ctypes signatures ("p" pointer, "i" int, "z" size_t,
# "u" unsigned long long)
_SIGS = {
    "la_status_string": ("i", ctypes.c_char_p),
    "la_version": ("", ctypes.c_int),
    "la_workspace_bytes": ("i i i i i i i", ctypes.c_size_t),
    "la_kernel_launches": ("i i i i i i i", ctypes.c_int),
    "la_causal_fwd": ("p p p p p p z i i i i i i p", ctypes.c_int),
    "la_causal_bwd": ("p p p p p p p p p p z i i i i i i p", ctypes.c_int),
    "la_causal_prefill": ("p p p p p p p p z i i i i i i p", ctypes.c_int),
    "la_noncausal_fwd": ("p p p p p p p p p z i i i i i i p", ctypes.c_int),
    "la_noncausal_bwd": ("p p p p p p p p p p p p p z i i i i i i p", ctypes.c_int),
    "la_decode_step": ("p p p p p p i i i i i p", ctypes.c_int),
    "la_causal_fwd_decay": ("p p p p p f p z i i i i i i p", ctypes.c_int),
    "la_causal_bwd_decay": ("p p p p p p p p p f p z i i i i i i p", ctypes.c_int),
    "la_decode_step_decay": ("p p p p p p f i i i i i p", ctypes.c_int),
    "la_decode_step_proj": ("p p p p p i i i i i i p", ctypes.c_int),
    "la_causal_fwd_poly": ("p p p p p p z i i i i i i p", ctypes.c_int),
    "la_causal_bwd_poly": ("p p p p p p p p p p z i i i i i i p", ctypes.c_int),
    "la_causal_fwd_noalloc": ("p p p p p i i i i i i p", ctypes.c_int),
    "la_device_status": ("p i p", ctypes.c_int),
    "la_selftest_wait": ("p u", ctypes.c_int),
}
EXPORTED = tuple(_SIGS)

_lock = threading.Lock()
_lib = None


class LinAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (code {code})")


def library_path() -> str:
    return LIB_PATH


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library not built: {LIB_PATH} is missing. Build it with "
                    "`python -m kernelized_causal_attention_gb300._build` (needs nvcc).")
            h = ctypes.CDLL(LIB_PATH)
            kinds = {"p": ctypes.c_void_p, "i": ctypes.c_int, "z": ctypes.c_size_t,
                     "u": ctypes.c_ulonglong, "f": ctypes.c_float}
            for name, (sig, res) in _SIGS.items():
                fn = getattr(h, name)
                fn.argtypes = [kinds[c] for c in sig.split()]
                fn.restype = res
            _lib = h
    return _lib


def status_string(code: int) -> str:
    return lib().la_status_string(int(code)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LA_F32
    if t.dtype == torch.bfloat16:
        return LA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return int(t)  # a raw address
    if not t.is_cuda:
        # the library takes device pointers; a host address would reach a kernel
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(rc: int, where: str):
    if rc != LA_OK:
        raise LinAttnError(rc, where)


def _nbytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


# ------------------------------------------------------------------ raw C ABI

def la_workspace_bytes(op, B, H, N, D, M, dtype) -> int:
    return int(lib().la_workspace_bytes(op, B, H, N, D, M, dtype))


def la_kernel_launches(op, B, H, N, D, M, dtype) -> int:
    return int(lib().la_kernel_launches(op, B, H, N, D, M, dtype))


def la_causal_fwd(q, k, v, out, den, workspace, B, H, N, D, M, dtype, stream=None):
    _check(lib().la_causal_fwd(_p(q), _p(k), _p(v), _p(out), _p(den), _p(workspace),
                               _nbytes(workspace), B, H, N, D, M, dtype, _stream(stream)),
           "la_causal_fwd")


def la_causal_bwd(q, k, v, out, den, dout, dq, dk, dv, workspace, B, H, N, D, M, dtype,
                  stream=None):
    _check(lib().la_causal_bwd(_p(q), _p(k), _p(v), _p(out), _p(den), _p(dout), _p(dq), _p(dk),
                               _p(dv), _p(workspace), _nbytes(workspace), B, H, N, D, M, dtype,
                               _stream(stream)), "la_causal_bwd")


def la_causal_prefill(q, k, v, out, den, S, Z, workspace, B, H, N, D, M, dtype, stream=None):
    _check(lib().la_causal_prefill(_p(q), _p(k), _p(v), _p(out), _p(den), _p(S), _p(Z),
                                   _p(workspace), _nbytes(workspace), B, H, N, D, M, dtype,
                                   _stream(stream)), "la_causal_prefill")


def la_noncausal_fwd(q, k, v, lengths, out, den, S, Z, workspace, B, H, N, D, M, dtype,
                     stream=None):
    _check(lib().la_noncausal_fwd(_p(q), _p(k), _p(v), _p(lengths), _p(out), _p(den), _p(S),
                                  _p(Z), _p(workspace), _nbytes(workspace), B, H, N, D, M, dtype,
                                  _stream(stream)), "la_noncausal_fwd")


def la_noncausal_bwd(q, k, v, lengths, out, den, S, Z, dout, dq, dk, dv, workspace, B, H, N, D,
                     M, dtype, stream=None):
    _check(lib().la_noncausal_bwd(_p(q), _p(k), _p(v), _p(lengths), _p(out), _p(den), _p(S),
                                  _p(Z), _p(dout), _p(dq), _p(dk), _p(dv), _p(workspace),
                                  _nbytes(workspace), B, H, N, D, M, dtype, _stream(stream)),
           "la_noncausal_bwd")


def la_decode_step(q, k, v, S, Z, y, B, H, D, M, dtype, stream=None):
    _check(lib().la_decode_step(_p(q), _p(k), _p(v), _p(S), _p(Z), _p(y), B, H, D, M, dtype,
                                _stream(stream)), "la_decode_step")


def la_causal_fwd_decay(q, k, v, out, den, gamma, workspace, B, H, N, D, M, dtype, stream=None):
    _check(lib().la_causal_fwd_decay(_p(q), _p(k), _p(v), _p(out), _p(den), float(gamma),
                                     _p(workspace), _nbytes(workspace), B, H, N, D, M, dtype,
                                     _stream(stream)), "la_causal_fwd_decay")


def la_causal_bwd_decay(q, k, v, out, den, dout, dq, dk, dv, gamma, workspace, B, H, N, D, M,
                        dtype, stream=None):
    _check(lib().la_causal_bwd_decay(_p(q), _p(k), _p(v), _p(out), _p(den), _p(dout), _p(dq),
                                     _p(dk), _p(dv), float(gamma), _p(workspace),
                                     _nbytes(workspace), B, H, N, D, M, dtype, _stream(stream)),
           "la_causal_bwd_decay")


def la_decode_step_decay(q, k, v, S, Z, y, gamma, B, H, D, M, dtype, stream=None):
    _check(lib().la_decode_step_decay(_p(q), _p(k), _p(v), _p(S), _p(Z), _p(y), float(gamma), B,
                                      H, D, M, dtype, _stream(stream)), "la_decode_step_decay")


def la_causal_fwd_poly(q, k, v, out, den, workspace, B, H, N, D, M, dtype, stream=None):
    _check(lib().la_causal_fwd_poly(_p(q), _p(k), _p(v), _p(out), _p(den), _p(workspace),
                                    _nbytes(workspace), B, H, N, D, M, dtype, _stream(stream)),
           "la_causal_fwd_poly")


def la_causal_bwd_poly(q, k, v, out, den, dout, dq, dk, dv, workspace, B, H, N, D, M, dtype,
                       stream=None):
    _check(lib().la_causal_bwd_poly(_p(q), _p(k), _p(v), _p(out), _p(den), _p(dout), _p(dq), _p(dk),
                                    _p(dv), _p(workspace), _nbytes(workspace), B, H, N, D, M, dtype,
                                    _stream(stream)), "la_causal_bwd_poly")


def la_decode_step_proj(x, W, S, Z, y, B, H, d_model, D, M, dtype, stream=None):
    _check(lib().la_decode_step_proj(_p(x), _p(W), _p(S), _p(Z), _p(y), B, H, d_model, D, M, dtype,
                                     _stream(stream)), "la_decode_step_proj")


def la_causal_fwd_noalloc(q, k, v, out, den, B, H, N, D, M, dtype, stream=None):
    """la_causal_fwd with the library's built-in scratch instead of a workspace
    (for callers that may not allocate device memory)."""
    _check(lib().la_causal_fwd_noalloc(_p(q), _p(k), _p(v), _p(out), _p(den), B, H, N, D, M,
                                       dtype, _stream(stream)), "la_causal_fwd_noalloc")


def la_device_status(clear=True, stream=None):
    """(status, code): LA_OK and 0, or LA_ERR_TIMEOUT and the code of the first
    bounded wait inside a kernel that ran out (after the stream's queued work);
    clear resets the status word."""
    code = ctypes.c_int(0)
    rc = lib().la_device_status(_stream(stream), int(bool(clear)), ctypes.byref(code))
    if rc not in (LA_OK, LA_ERR_TIMEOUT):
        raise LinAttnError(rc, "la_device_status")
    return rc, code.value


def la_selftest_wait(limit_ns, stream=None):
    """Launches the diagnostic kernel whose bounded wait runs out after limit_ns."""
    _check(lib().la_selftest_wait(_stream(stream), int(limit_ns)), "la_selftest_wait")


def check_device_status(stream=None):
    """Raises LinAttnError(LA_ERR_TIMEOUT) if a kernel's bounded wait ran out
    (and clears the status word); returns None otherwise."""
    rc, code = la_device_status(True, stream)
    if rc != LA_OK:
        raise LinAttnError(rc, f"device status (wait code {code})")


# --------------------------------------------------- allocating convenience API

def workspace(op, B, H, N, D, M, dtype, device):
    n = la_workspace_bytes(op, B, H, N, D, M, dtype)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=device)


def causal_fwd(q, k, v, stream=None):
    """(out, den) of the causal form; q, k [B,H,N,D], v [B,H,N,M] on the GPU."""
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    out = torch.empty(B, H, N, M, dtype=q.dtype, device=q.device)
    den = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    ws = workspace(LA_OP_CAUSAL_FWD, B, H, N, D, M, dt, q.device)
    la_causal_fwd(q, k, v, out, den, ws, B, H, N, D, M, dt, stream)
    return out, den


def causal_fwd_decay(q, k, v, gamma, stream=None):
    """(out, den) of the causal form with the RetNet decay gamma in [0, 1]."""
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    out = torch.empty(B, H, N, M, dtype=q.dtype, device=q.device)
    den = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    ws = workspace(LA_OP_CAUSAL_FWD_DECAY, B, H, N, D, M, dt, q.device)
    la_causal_fwd_decay(q, k, v, out, den, gamma, ws, B, H, N, D, M, dt, stream)
    return out, den


def causal_bwd_decay(q, k, v, out, den, dout, gamma, stream=None):
    """(dq, dk, dv) of sum(dout * out) for the decayed causal form."""
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = workspace(LA_OP_CAUSAL_BWD_DECAY, B, H, N, D, M, dt, q.device)
    la_causal_bwd_decay(q, k, v, out, den, dout, dq, dk, dv, gamma, ws, B, H, N, D, M, dt, stream)
    return dq, dk, dv


def causal_fwd_poly(q, k, v, stream=None):
    """(out, den) of causal attention with the degree-2 polynomial kernel
    sim = (q . k)^2 (bf16, D <= 10)."""
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    out = torch.empty(B, H, N, M, dtype=q.dtype, device=q.device)
    den = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    ws = workspace(LA_OP_CAUSAL_FWD_POLY, B, H, N, D, M, dt, q.device)
    la_causal_fwd_poly(q, k, v, out, den, ws, B, H, N, D, M, dt, stream)
    return out, den


def causal_bwd_poly(q, k, v, out, den, dout, stream=None):
    """(dq, dk, dv) of sum(dout * out) with the degree-2 polynomial kernel."""
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = workspace(LA_OP_CAUSAL_BWD_POLY, B, H, N, D, M, dt, q.device)
    la_causal_bwd_poly(q, k, v, out, den, dout, dq, dk, dv, ws, B, H, N, D, M, dt, stream)
    return dq, dk, dv


def decode_step_decay(q, k, v, S, Z, gamma, stream=None):
    """One decayed RNN step; S, Z updated in place.  Returns y [B,H,M]."""
    B, H, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    y = torch.empty(B, H, M, dtype=q.dtype, device=q.device)
    la_decode_step_decay(q, k, v, S, Z, y, gamma, B, H, D, M, dt, stream)
    return y


def causal_prefill(q, k, v, S=None, Z=None, stream=None):
    """(out, den, S, Z): the causal form started from the state (S, Z) (zeros
    if None), which is updated in place to the state after the sequence and
    returned; la_decode_step continues from it."""
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    out = torch.empty_like(v)
    den = torch.empty(B, H, N, device=q.device, dtype=torch.float32)
    if S is None:
        S = torch.zeros(B, H, D, M, device=q.device, dtype=torch.float32)
    if Z is None:
        Z = torch.zeros(B, H, D, device=q.device, dtype=torch.float32)
    ws = workspace(LA_OP_CAUSAL_PREFILL, B, H, N, D, M, dt, q.device)
    la_causal_prefill(q, k, v, out, den, S, Z, ws, B, H, N, D, M, dt, stream)
    return out, den, S, Z


def causal_bwd(q, k, v, out, den, dout, stream=None):
    """(dq, dk, dv) of sum(dout * out) for the causal form."""
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = workspace(LA_OP_CAUSAL_BWD, B, H, N, D, M, dt, q.device)
    la_causal_bwd(q, k, v, out, den, dout, dq, dk, dv, ws, B, H, N, D, M, dt, stream)
    return dq, dk, dv


def noncausal_fwd(q, k, v, lengths=None, stream=None):
    """(out, den, S, Z) of the non-causal form; lengths: int32 [B] on the GPU or None."""
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    out = torch.empty(B, H, N, M, dtype=q.dtype, device=q.device)
    den = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    S = torch.empty(B, H, D, M, dtype=torch.float32, device=q.device)
    Z = torch.empty(B, H, D, dtype=torch.float32, device=q.device)
    ws = workspace(LA_OP_NONCAUSAL_FWD, B, H, N, D, M, dt, q.device)
    la_noncausal_fwd(q, k, v, lengths, out, den, S, Z, ws, B, H, N, D, M, dt, stream)
    return out, den, S, Z


def noncausal_bwd(q, k, v, lengths, out, den, S, Z, dout, stream=None):
    B, H, N, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = workspace(LA_OP_NONCAUSAL_BWD, B, H, N, D, M, dt, q.device)
    la_noncausal_bwd(q, k, v, lengths, out, den, S, Z, dout, dq, dk, dv, ws, B, H, N, D, M, dt,
                     stream)
    return dq, dk, dv


def decode_step(q, k, v, S, Z, stream=None):
    """One RNN step; S [B,H,D,M] and Z [B,H,D] (float32) are updated in place.
    Returns y [B,H,M]."""
    B, H, D = q.shape
    M = v.shape[-1]
    dt = _dtype_code(q)
    y = torch.empty(B, H, M, dtype=q.dtype, device=q.device)
    la_decode_step(q, k, v, S, Z, y, B, H, D, M, dt, stream)
    return y


def decode_step_proj(x, W, S, Z, H, D, M, stream=None):
    """One RNN step whose q, k, v are the projection x W (bf16): x [B, d_model],
    W [d_model, H*(2D+M)] with each head's W_Q | W_K | W_V columns side by side,
    head after head.  S [B,H,D,M] and Z [B,H,D] (float32) are updated in place.
    Returns y [B,H,M] (bf16)."""
    B, dm = x.shape
    y = torch.empty(B, H, M, dtype=x.dtype, device=x.device)
    la_decode_step_proj(x, W, S, Z, y, B, H, dm, D, M, _dtype_code(x), stream)
    return y


class _Causal(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        out, den = causal_fwd(q, k, v)
        ctx.save_for_backward(q, k, v, out, den)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, den = ctx.saved_tensors
        return causal_bwd(q, k, v, out, den, dout.contiguous())


class _NonCausal(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, lengths):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        out, den, S, Z = noncausal_fwd(q, k, v, lengths)
        ctx.save_for_backward(q, k, v, out, den, S, Z)
        ctx.lengths = lengths
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, den, S, Z = ctx.saved_tensors
        dq, dk, dv = noncausal_bwd(q, k, v, ctx.lengths, out, den, S, Z, dout.contiguous())
        return dq, dk, dv, None


def causal_linear_attention(q, k, v):
    """Causal elu+1 linear attention with the constant-memory backward."""
    return _Causal.apply(q, k, v)


def noncausal_linear_attention(q, k, v, lengths=None):
    """Non-causal elu+1 linear attention (shared S, Z per sequence)."""
    return _NonCausal.apply(q, k, v, lengths)
