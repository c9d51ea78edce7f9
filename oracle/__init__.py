"""fp64 CPU oracle for elu(x)+1 linear attention -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
compiles it with gcc and wraps it with ctypes and numpy.  Only the test suite,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import this
package.  The CUDA library never imports it and it imports nothing from the
CUDA library.

Sources: "Transformers are RNNs: Fast Autoregressive Transformers with Linear
Attention -- part 2/3" (eq. 7, §3.3 eq. 8-12, §3.3.1 eq. 13-15, §3.4 eq. 16-19)
and "Linear Attention/zh" (kernel reformulation; recurrent form; the RetNet
decay of "variants and extensions", taken with gamma in [0, 1]).  Each C
function cites the passage it follows.

Every function takes arrays of any float dtype (a bf16 input is passed already
widened, so the oracle sees exactly the values the kernel sees) and returns
float64 numpy arrays.  Layouts: q, k [B, H, N, D]; v, g [B, H, N, M]; decode
inputs [T, B, H, D|M]; state S [B, H, D, M], Z [B, H, D].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_default = None

_SIGS = {
    "orc_phi": "l p p p",
    "orc_causal_fwd_quadratic": "i i i i p p p p p i",
    "orc_causal_fwd_recurrent": "i i i i p p p p p i",
    "orc_causal_bwd_recurrent": "i i i i p p p p p p p i",
    "orc_causal_bwd_quadratic": "i i i i p p p p p p p i",
    "orc_noncausal_fwd": "i i i i i p p p p p p p p i",
    "orc_noncausal_fwd_quadratic": "i i i i i p p p p p p i",
    "orc_noncausal_bwd": "i i i i i p p p p p p p p i",
    "orc_noncausal_bwd_quadratic": "i i i i i p p p p p p p p i",
    "orc_decode": "i i i i p p p p p p i",
    "orc_causal_fwd_quadratic_decay": "i i i i p p p d p p i",
    "orc_causal_fwd_recurrent_decay": "i i i i p p p d p p i",
    "orc_causal_bwd_recurrent_decay": "i i i i p p p p d p p p i",
    "orc_causal_bwd_quadratic_decay": "i i i i p p p p d p p p i",
    "orc_decode_decay": "i i i i p p p d p p p i",
    "orc_causal_prefill": "i i i i p p p p p p p i",
    "orc_causal_fwd_poly": "i i i i p p p p p i",
    "orc_causal_bwd_poly": "i i i i p p p p p p p i",
}


def compile_c(src: str, out: str) -> str:
    """gcc -O2 (OpenMP when available, no FMA contraction) into a shared library."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC",
            src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_lib/liboracle.so."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    return compile_c(_SRC, _LIB)


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor (possibly bf16): widen exactly
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _lengths(lengths, B):
    if lengths is None:
        return None
    if hasattr(lengths, "cpu"):
        lengths = lengths.cpu().numpy()
    lens = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32))
    assert lens.shape == (B,)
    return lens


def default_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return len(os.sched_getaffinity(0))
    return os.cpu_count() or 1


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        kinds = {"i": ctypes.c_int, "l": ctypes.c_long, "p": ctypes.c_void_p, "d": ctypes.c_double}
        for name, sig in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = [kinds[c] for c in sig.split()]
            fn.restype = None
        lib.orc_openmp_enabled.argtypes = []
        lib.orc_openmp_enabled.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def openmp_enabled(self) -> bool:
        return bool(self.lib.orc_openmp_enabled())

    def phi(self, x):
        """Feature map of eq. 7 and its derivative: returns (phi(x), phi'(x))."""
        x = _f64(x)
        y, dy = np.empty_like(x), np.empty_like(x)
        self.lib.orc_phi(x.size, _ptr(x), _ptr(y), _ptr(dy))
        return y, dy

    def causal_fwd(self, q, k, v, form="recurrent", nthreads=0, gamma=None):
        """Causal forward: (out [B,H,N,M], den [B,H,N]).  form = 'recurrent'
        (eq. 10-12) or 'quadratic' (eq. 8 with sim = phi(q)^T phi(k)).  gamma:
        the RetNet decay in [0, 1] (None: the undecayed entry points)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, D = q.shape
        M = v.shape[-1]
        out, den = np.empty((B, H, N, M)), np.empty((B, H, N))
        if gamma is None:
            fn = {"recurrent": self.lib.orc_causal_fwd_recurrent,
                  "quadratic": self.lib.orc_causal_fwd_quadratic}[form]
            fn(B * H, N, D, M, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(den), nthreads)
        else:
            fn = {"recurrent": self.lib.orc_causal_fwd_recurrent_decay,
                  "quadratic": self.lib.orc_causal_fwd_quadratic_decay}[form]
            fn(B * H, N, D, M, _ptr(q), _ptr(k), _ptr(v), float(gamma), _ptr(out), _ptr(den),
               nthreads)
        return out, den

    def causal_bwd(self, q, k, v, g, form="recurrent", nthreads=0, gamma=None):
        """Gradients (dq, dk, dv) of sum(g * V') for the causal form (gamma:
        the RetNet decay, None for the undecayed entry points)."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
        B, H, N, D = q.shape
        M = v.shape[-1]
        dq, dk, dv = np.empty((B, H, N, D)), np.empty((B, H, N, D)), np.empty((B, H, N, M))
        if gamma is None:
            fn = {"recurrent": self.lib.orc_causal_bwd_recurrent,
                  "quadratic": self.lib.orc_causal_bwd_quadratic}[form]
            fn(B * H, N, D, M, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
               _ptr(dq), _ptr(dk), _ptr(dv), nthreads)
        else:
            fn = {"recurrent": self.lib.orc_causal_bwd_recurrent_decay,
                  "quadratic": self.lib.orc_causal_bwd_quadratic_decay}[form]
            fn(B * H, N, D, M, _ptr(q), _ptr(k), _ptr(v), _ptr(g), float(gamma),
               _ptr(dq), _ptr(dk), _ptr(dv), nthreads)
        return dq, dk, dv

    def causal_fwd_poly(self, q, k, v, nthreads=0):
        """Causal forward with the degree-2 polynomial kernel sim = (q . k)^2
        (the quadratic form, every pair): (out [B,H,N,M], den [B,H,N])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, D = q.shape
        M = v.shape[-1]
        out, den = np.empty((B, H, N, M)), np.empty((B, H, N))
        self.lib.orc_causal_fwd_poly(B * H, N, D, M, _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                     _ptr(den), nthreads)
        return out, den

    def causal_bwd_poly(self, q, k, v, g, nthreads=0):
        """Gradients (dq, dk, dv) of sum(g * V') with the degree-2 polynomial
        kernel, by the pairwise rule."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
        B, H, N, D = q.shape
        M = v.shape[-1]
        dq, dk, dv = np.empty((B, H, N, D)), np.empty((B, H, N, D)), np.empty((B, H, N, M))
        self.lib.orc_causal_bwd_poly(B * H, N, D, M, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                     _ptr(dq), _ptr(dk), _ptr(dv), nthreads)
        return dq, dk, dv

    def noncausal_fwd(self, q, k, v, lengths=None, form="recurrent", nthreads=0):
        """Non-causal forward with a shared S, Z: (out, den, S, Z); the
        quadratic form returns S = Z = None."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, D = q.shape
        M = v.shape[-1]
        lens = _lengths(lengths, B)
        out, den = np.empty((B, H, N, M)), np.empty((B, H, N))
        if form == "quadratic":
            self.lib.orc_noncausal_fwd_quadratic(B, H, N, D, M, _ptr(lens), _ptr(q), _ptr(k),
                                                 _ptr(v), _ptr(out), _ptr(den), nthreads)
            return out, den, None, None
        S, Z = np.empty((B, H, D, M)), np.empty((B, H, D))
        self.lib.orc_noncausal_fwd(B, H, N, D, M, _ptr(lens), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(out), _ptr(den), _ptr(S), _ptr(Z), nthreads)
        return out, den, S, Z

    def noncausal_bwd(self, q, k, v, g, lengths=None, form="recurrent", nthreads=0):
        """Gradients (dq, dk, dv) of sum(g * V') for the non-causal form."""
        q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
        B, H, N, D = q.shape
        M = v.shape[-1]
        lens = _lengths(lengths, B)
        dq, dk, dv = np.empty((B, H, N, D)), np.empty((B, H, N, D)), np.empty((B, H, N, M))
        fn = {"recurrent": self.lib.orc_noncausal_bwd,
              "quadratic": self.lib.orc_noncausal_bwd_quadratic}[form]
        fn(B, H, N, D, M, _ptr(lens), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
           _ptr(dq), _ptr(dk), _ptr(dv), nthreads)
        return dq, dk, dv

    def decode(self, q, k, v, S=None, Z=None, nthreads=0, gamma=None):
        """T RNN steps (eq. 16-19) over independent streams.  q, k: [T,B,H,D];
        v: [T,B,H,M]; S, Z: initial state (zeros if None); gamma: the RetNet
        decay (None: undecayed).  Returns (y [T,B,H,M], S_T [B,H,D,M], Z_T [B,H,D])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        T, B, H, D = q.shape
        M = v.shape[-1]
        S = np.zeros((B, H, D, M)) if S is None else _f64(S).copy()
        Z = np.zeros((B, H, D)) if Z is None else _f64(Z).copy()
        y = np.empty((T, B, H, M))
        if gamma is None:
            self.lib.orc_decode(T, B * H, D, M, _ptr(q), _ptr(k), _ptr(v), _ptr(S), _ptr(Z),
                                _ptr(y), nthreads)
        else:
            self.lib.orc_decode_decay(T, B * H, D, M, _ptr(q), _ptr(k), _ptr(v), float(gamma),
                                      _ptr(S), _ptr(Z), _ptr(y), nthreads)
        return y, S, Z

    def decode_proj(self, x, W, H, D, M, S=None, Z=None, nthreads=0):
        """One RNN step (eq. 16-19) whose q_t, k_t, v_t are the projections
        x_t W of the layer input (eq. 18-20 write phi(x_i W_Q), x_i W_K,
        x_i W_V); f_l and the residual of eq. 20 are not applied.  x: [B,
        d_model]; W: [d_model, H*(2D+M)] whose columns hold, head after head,
        that head's W_Q (D columns), W_K (D) and W_V (M) side by side; S, Z:
        state (zeros if None).  The projection is a plain fp64 matmul (numpy);
        the step is orc_decode.  Returns (y [B,H,M], S_1 [B,H,D,M], Z_1
        [B,H,D])."""
        x, W = _f64(x), _f64(W)
        B = x.shape[0]
        assert W.shape == (x.shape[1], H * (2 * D + M))
        p = (x @ W).reshape(B, H, 2 * D + M)  # [B, H, q | k | v]
        q = p[:, :, :D].reshape(1, B, H, D)
        k = p[:, :, D:2 * D].reshape(1, B, H, D)
        v = p[:, :, 2 * D:].reshape(1, B, H, M)
        y, S1, Z1 = self.decode(q, k, v, S, Z, nthreads)
        return y[0], S1, Z1

    def causal_prefill(self, q, k, v, S=None, Z=None, nthreads=0):
        """The causal form started from the state (S, Z) (zeros if None):
        eq. 16-19 over a prompt.  q, k: [B,H,N,D]; v: [B,H,N,M].
        Returns (out [B,H,N,M], den [B,H,N], S_N [B,H,D,M], Z_N [B,H,D])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, D = q.shape
        M = v.shape[-1]
        S = np.zeros((B, H, D, M)) if S is None else _f64(S).copy()
        Z = np.zeros((B, H, D)) if Z is None else _f64(Z).copy()
        out = np.empty((B, H, N, M))
        den = np.empty((B, H, N))
        self.lib.orc_causal_prefill(B * H, N, D, M, _ptr(q), _ptr(k), _ptr(v), _ptr(S), _ptr(Z),
                                    _ptr(out), _ptr(den), nthreads)
        return out, den, S, Z


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def openmp_enabled():
    return default().openmp_enabled()


def phi(x):
    return default().phi(x)


def causal_fwd(q, k, v, form="recurrent", nthreads=0, gamma=None):
    return default().causal_fwd(q, k, v, form, nthreads, gamma)


def causal_bwd(q, k, v, g, form="recurrent", nthreads=0, gamma=None):
    return default().causal_bwd(q, k, v, g, form, nthreads, gamma)


def noncausal_fwd(q, k, v, lengths=None, form="recurrent", nthreads=0):
    return default().noncausal_fwd(q, k, v, lengths, form, nthreads)


def noncausal_bwd(q, k, v, g, lengths=None, form="recurrent", nthreads=0):
    return default().noncausal_bwd(q, k, v, g, lengths, form, nthreads)


def decode(q, k, v, S=None, Z=None, nthreads=0, gamma=None):
    return default().decode(q, k, v, S, Z, nthreads, gamma)


def causal_fwd_poly(q, k, v, nthreads=0):
    return default().causal_fwd_poly(q, k, v, nthreads)


def causal_bwd_poly(q, k, v, g, nthreads=0):
    return default().causal_bwd_poly(q, k, v, g, nthreads)


def causal_prefill(q, k, v, S=None, Z=None, nthreads=0):
    return default().causal_prefill(q, k, v, S, Z, nthreads)


def decode_proj(x, W, H, D, M, S=None, Z=None, nthreads=0):
    return default().decode_proj(x, W, H, D, M, S, Z, nthreads)
