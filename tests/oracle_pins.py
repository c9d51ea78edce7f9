"""Checks that pin the fp64 oracle to facts that do not come from the oracle.

Each ``pin_*`` function takes an oracle instance and raises AssertionError when
the oracle disagrees with something the pages or the mathematics fix: a second,
independent form of the same quantity, a closed form, an invariant, a library
routine (torch's ELU, numpy matmul), or central finite differences.  The
mutation tests run the same pins against deliberately broken builds of the
oracle to show that each plausible slip is caught.

Sources: "Transformers are RNNs -- part 2/3": eq. 7 (phi = elu + 1), §3.3
eq. 8 (masked quadratic form) and eq. 10-12 (recurrence), §3.3.1 eq. 13-15
(gradients), §3.4 eq. 16-19 (RNN form, also run over a prompt from a given
state); "Linear Attention/zh": kernel
reformulation (shared S, z for the non-causal form) and the RetNet decay of
"variants and extensions" (S_t = gamma S_{t-1} + phi(k_t) v_t^T, read with z
decaying alongside S).
"""
from __future__ import annotations

import numpy as np
import scipy.signal
import torch

RNG_SHAPES = [  # (B, H, N, D, M): D != M catches transposed operands
    (1, 1, 1, 3, 5),
    (1, 2, 7, 3, 5),
    (2, 1, 13, 4, 2),
]


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def phi_lib(x):
    """elu(x) + 1 through torch's own ELU (alpha = 1)."""
    return torch.nn.functional.elu(torch.as_tensor(x, dtype=torch.float64)).numpy() + 1.0


def rel(a, b, floor=1e-300):
    """max |a - b| / max |b| (normwise-max), with max |b| floored at ``floor``
    for quantities whose exact value is zero."""
    a, b = np.asarray(a), np.asarray(b)
    scale = max(np.max(np.abs(b)), floor)
    return float(np.max(np.abs(a - b)) / scale)


# ---------------------------------------------------------------- feature map

def pin_phi(orc):
    """eq. 7 against torch's ELU + 1, and phi' against autograd through it."""
    x = np.concatenate([rand(200, 1, 3.0), [0.0, -0.0, 1e-300, -1e-300, 50.0, -50.0]])
    y, dy = orc.phi(x)
    assert rel(y, phi_lib(x)) < 1e-15, "phi != elu + 1"
    xt = torch.tensor(x, requires_grad=True)
    (torch.nn.functional.elu(xt) + 1.0).sum().backward()
    assert rel(dy, xt.grad.numpy()) < 1e-15, "phi' != d(elu + 1)/dx"
    assert np.all(y > 0), "phi must be positive"


# ------------------------------------------------------------ causal forward

def pin_causal_forms_agree(orc):
    """eq. 8 (explicit masked matrix) and eq. 10-12 (recurrence) are the same
    function: two independent algorithms must agree."""
    for i, (B, H, N, D, M) in enumerate(RNG_SHAPES + [(1, 1, 64, 16, 16)]):
        q, k, v = rand((B, H, N, D), 10 + i), rand((B, H, N, D), 20 + i), rand((B, H, N, M), 30 + i)
        o1, d1 = orc.causal_fwd(q, k, v, "quadratic")
        o2, d2 = orc.causal_fwd(q, k, v, "recurrent")
        assert rel(o1, o2) < 1e-12 and rel(d1, d2) < 1e-12, "causal forms disagree"


def pin_causal_closed_forms(orc):
    """Closed forms of eq. 8:
      * Q = K = 0 gives phi = 1, every weight equals D, so V'_i is the running
        mean of V_1..V_i and den_i = D * i;
      * V'_1 = V_1 (only one key is visible);
      * constant value rows are reproduced exactly;
      * V'_i lies in the per-coordinate hull of V_1..V_i (positive weights);
      * den > 0."""
    B, H, N, D, M = 2, 3, 9, 4, 6
    v = rand((B, H, N, M), 1)
    zeros = np.zeros((B, H, N, D))
    for form in ("quadratic", "recurrent"):
        o, den = orc.causal_fwd(zeros, zeros, v, form)
        mean = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
        assert rel(o, mean) < 1e-14, "Q=K=0 must give the running mean"
        assert rel(den, D * np.broadcast_to(np.arange(1, N + 1), den.shape)) < 1e-15
        q, k = rand((B, H, N, D), 2, 2.0), rand((B, H, N, D), 3, 2.0)
        o, den = orc.causal_fwd(q, k, v, form)
        assert np.array_equal(o[:, :, 0], v[:, :, 0]) or rel(o[:, :, 0], v[:, :, 0]) < 1e-15, \
            "V'_1 must equal V_1"
        assert np.all(den > 0), "den must be positive"
        lo = np.minimum.accumulate(v, axis=2)
        hi = np.maximum.accumulate(v, axis=2)
        assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12), "V' outside the hull"
        c = rand((B, H, 1, M), 4)
        oc, _ = orc.causal_fwd(q, k, np.broadcast_to(c, (B, H, N, M)), form)
        assert rel(oc, np.broadcast_to(c, oc.shape)) < 1e-14, "constant V not reproduced"


def pin_grad_single_token(orc):
    """N = 1: V'_1 = V_1 whatever Q and K are, so dQ = dK = 0 and dV = G."""
    q, k, v, g = rand((2, 2, 1, 3), 15), rand((2, 2, 1, 3), 16), rand((2, 2, 1, 4), 17), rand((2, 2, 1, 4), 18)
    for form in ("recurrent", "quadratic"):
        dq, dk, dv = orc.causal_bwd(q, k, v, g, form)
        assert np.max(np.abs(dq)) < 1e-14 and np.max(np.abs(dk)) < 1e-14, "N=1 gradient not zero"
        assert rel(dv, g) < 1e-15, "N=1: dV != G"


# --------------------------------------------------------------- non-causal

def pin_noncausal_gemm(orc):
    """Non-causal form = two textbook products (kernel reformulation of
    "Linear Attention/zh"): S = phi(K)^T V, z = phi(K)^T 1, V' = phi(Q) S / phi(Q) z,
    computed with numpy matmul and torch's ELU."""
    B, H, N, D, M = 2, 2, 11, 3, 5
    q, k, v = rand((B, H, N, D), 5), rand((B, H, N, D), 6), rand((B, H, N, M), 7)
    fq, fk = phi_lib(q), phi_lib(k)
    S = np.matmul(np.swapaxes(fk, -1, -2), v)
    Z = fk.sum(axis=2)
    den = np.matmul(fq, Z[..., None])[..., 0]
    ref = np.matmul(fq, S) / den[..., None]
    for form in ("recurrent", "quadratic"):
        o, d, S2, Z2 = orc.noncausal_fwd(q, k, v, None, form)
        assert rel(o, ref) < 1e-13 and rel(d, den) < 1e-13, "non-causal != GEMM form"
        if S2 is not None:
            assert rel(S2, S) < 1e-13 and rel(Z2, Z) < 1e-13, "S, Z != phi(K)^T [V, 1]"


def pin_noncausal_last_row(orc):
    """With every position valid, the non-causal output equals the causal one at
    the last position (both read S_N, Z_N)."""
    B, H, N, D, M = 1, 2, 10, 3, 4
    q, k, v = rand((B, H, N, D), 8), rand((B, H, N, D), 9), rand((B, H, N, M), 10)
    oc, dc = orc.causal_fwd(q, k, v, "quadratic")
    on, dn, _, _ = orc.noncausal_fwd(q, k, v, None, "recurrent")
    assert rel(on[:, :, -1], oc[:, :, -1]) < 1e-13 and rel(dn[:, :, -1], dc[:, :, -1]) < 1e-13


def pin_noncausal_lengths(orc):
    """Padding: a batch entry of valid length L gives the same result as the
    unpadded sequence truncated to L, zeros beyond it, and no dependence on the
    padded contents."""
    B, H, N, D, M = 3, 2, 12, 3, 4
    lengths = np.array([12, 5, 1], dtype=np.int32)
    q, k, v, g = (rand((B, H, N, D), 11), rand((B, H, N, D), 12), rand((B, H, N, M), 13),
                  rand((B, H, N, M), 14))
    for form in ("recurrent", "quadratic"):
        o, den, _, _ = orc.noncausal_fwd(q, k, v, lengths, form)
        dq, dk, dv = orc.noncausal_bwd(q, k, v, g, lengths, form)
        for b, L in enumerate(lengths):
            sl = (slice(b, b + 1), slice(None), slice(0, L))
            ot, dt, _, _ = orc.noncausal_fwd(q[sl], k[sl], v[sl], None, form)
            gq, gk, gv = orc.noncausal_bwd(q[sl], k[sl], v[sl], g[sl], None, form)
            assert rel(o[sl], ot) < 1e-13 and rel(den[sl], dt) < 1e-13, "length mask wrong"
            for a, r in ((dq, gq), (dk, gk), (dv, gv)):
                assert rel(a[sl], r) < 1e-12, "length mask wrong in gradients"
            pad = (b, slice(None), slice(L, None))
            for a in (o, den, dq, dk, dv):
                assert np.all(a[pad] == 0), "padded rows must be zero"
        # scramble the padding: nothing may change
        q2, k2, v2, g2 = q.copy(), k.copy(), v.copy(), g.copy()
        for b, L in enumerate(lengths):
            for a in (q2, k2, v2, g2):
                a[b, :, L:] = 1e3 * np.sign(a[b, :, L:]) + 7.0
        o2, _, _, _ = orc.noncausal_fwd(q2, k2, v2, lengths, form)
        d2 = orc.noncausal_bwd(q2, k2, v2, g2, lengths, form)
        assert np.array_equal(o, o2), "output depends on padding"
        for a, r in zip((dq, dk, dv), d2):
            assert np.array_equal(a, r), "gradient depends on padding"


# ------------------------------------------------------------------ gradients

def _loss(orc, kind, q, k, v, g, lengths):
    if kind == "causal":
        o, _ = orc.causal_fwd(q, k, v, "quadratic")
    else:
        o, _, _, _ = orc.noncausal_fwd(q, k, v, lengths, "quadratic")
    return float(np.sum(g * o))


def fd_grads(orc, kind, q, k, v, g, lengths=None, h=1e-6):
    """Central finite differences of L = sum(G * V') through the quadratic
    forward (no gradient code involved)."""
    out = []
    for x in (q, k, v):
        d = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = x[idx]
            x[idx] = x0 + h
            lp = _loss(orc, kind, q, k, v, g, lengths)
            x[idx] = x0 - h
            lm = _loss(orc, kind, q, k, v, g, lengths)
            x[idx] = x0
            d[idx] = (lp - lm) / (2 * h)
        out.append(d)
    return out


def pin_grad_fd(orc):
    """Both gradient forms (cumulative sums, eq. 13-15 with the quotient rule;
    and the explicit pairwise form) match central finite differences."""
    cases = [("causal", (1, 1, 6, 3, 4), None), ("causal", (1, 2, 5, 2, 3), None),
             ("noncausal", (2, 1, 6, 3, 2), np.array([6, 4], dtype=np.int32))]
    for n, (kind, (B, H, N, D, M), lengths) in enumerate(cases):
        q, k = rand((B, H, N, D), 40 + n), rand((B, H, N, D), 50 + n)
        v, g = rand((B, H, N, M), 60 + n), rand((B, H, N, M), 70 + n)
        ref = fd_grads(orc, kind, q, k, v, g, lengths)
        for form in ("recurrent", "quadratic"):
            if kind == "causal":
                got = orc.causal_bwd(q, k, v, g, form)
            else:
                got = orc.noncausal_bwd(q, k, v, g, lengths, form)
            for name, a, r in zip("qkv", got, ref):
                assert rel(a, r) < 1e-7, f"{kind} d{name} ({form}) != finite differences"


def pin_grad_forms_agree(orc):
    """Cumulative-sum gradients (eq. 13-15) equal the pairwise gradients on
    larger inputs than finite differences can afford."""
    for i, (B, H, N, D, M) in enumerate(RNG_SHAPES + [(1, 1, 64, 16, 16)]):
        q, k = rand((B, H, N, D), 80 + i), rand((B, H, N, D), 81 + i)
        v, g = rand((B, H, N, M), 82 + i), rand((B, H, N, M), 83 + i)
        a = orc.causal_bwd(q, k, v, g, "recurrent")
        b = orc.causal_bwd(q, k, v, g, "quadratic")
        for x, y in zip(a, b):
            assert rel(x, y, floor=1.0) < 1e-11, "causal gradient forms disagree"
        lengths = np.full(B, max(N - 2, 0), dtype=np.int32)
        a = orc.noncausal_bwd(q, k, v, g, lengths, "recurrent")
        b = orc.noncausal_bwd(q, k, v, g, lengths, "quadratic")
        for x, y in zip(a, b):
            assert rel(x, y, floor=1.0) < 1e-11, "non-causal gradient forms disagree"


def pin_grad_invariants(orc):
    """Symmetries of the quotient, exact in exact arithmetic:
      * V'_i is unchanged by scaling phi(Q_i), so phi(Q_i) . grad_phi(Q_i) = 0;
      * V' is unchanged by scaling every phi(K_j) by one factor, so
        sum_j phi(K_j) . grad_phi(K_j) = 0;
      * adding one row c to every V_j adds c to every V'_i, so
        sum_j grad V_j = sum_i G_i."""
    B, H, N, D, M = 2, 2, 33, 5, 7
    q, k = rand((B, H, N, D), 90), rand((B, H, N, D), 91)
    v, g = rand((B, H, N, M), 92), rand((B, H, N, M), 93)
    fq, dfq = orc.phi(q)
    fk, dfk = orc.phi(k)
    for form in ("recurrent", "quadratic"):
        dq, dk, dv = orc.causal_bwd(q, k, v, g, form)
        gq, gk = dq / dfq, dk / dfk
        scale = np.max(np.abs(gq * fq))
        assert np.max(np.abs(np.sum(fq * gq, axis=-1))) < 1e-12 * scale * D
        assert np.max(np.abs(np.sum(fk * gk, axis=(-1, -2)))) < 1e-11 * np.max(np.abs(fk * gk)) * N
        assert rel(dv.sum(axis=2), g.sum(axis=2)) < 1e-12


# --------------------------------------------------------------------- decode

def pin_decode(orc):
    """RNN form (eq. 16-19) against the causal quadratic form on the stacked
    sequence (the "transformers are RNNs" equivalence), the final state against
    numpy products S_T = phi(K)^T V and Z_T = sum phi(K), and resuming from a
    saved state against one uninterrupted run."""
    T, B, H, D, M = 9, 2, 3, 4, 5
    q, k, v = rand((T, B, H, D), 94), rand((T, B, H, D), 95), rand((T, B, H, M), 96)
    y, S, Z = orc.decode(q, k, v)
    perm = lambda x: np.ascontiguousarray(np.transpose(x, (1, 2, 0, 3)))  # -> [B,H,T,.]
    oc, _ = orc.causal_fwd(perm(q), perm(k), perm(v), "quadratic")
    assert rel(perm(y), oc) < 1e-13, "decode != causal forward"
    fk = phi_lib(perm(k))
    assert rel(S, np.matmul(np.swapaxes(fk, -1, -2), perm(v))) < 1e-13, "S_T != phi(K)^T V"
    assert rel(Z, fk.sum(axis=2)) < 1e-14, "Z_T != sum phi(K)"
    y1, S1, Z1 = orc.decode(q[:4], k[:4], v[:4])
    y2, S2, Z2 = orc.decode(q[4:], k[4:], v[4:], S1, Z1)
    assert np.array_equal(np.concatenate([y1, y2]), y), "resumed decode differs"
    assert np.array_equal(S2, S) and np.array_equal(Z2, Z)


# -------------------------------------------------------------------- prefill

def pin_prefill(orc):
    """The causal form started from a state (eq. 16-19 run over a prompt):
    from a zero state it is the masked quadratic form of eq. 8; its final state
    is S_0 + phi(K)^T V and Z_0 + sum phi(K) (numpy products); with phi(K) ~ 0
    (K = -60) only the state speaks, out = phi(Q) S_0 / phi(Q) Z_0 and
    den = phi(Q) Z_0 (numpy products); a prompt cut in two, the second part
    started from the first part's state, gives the outputs and state of one
    call, and so does the first part followed by RNN steps (the decode
    function) over the rest."""
    B, H, N, D, M = 2, 3, 11, 4, 5
    q, k, v = rand((B, H, N, D), 101), rand((B, H, N, D), 102), rand((B, H, N, M), 103)
    out0, den0, _, _ = orc.causal_prefill(q, k, v)
    oc, dc = orc.causal_fwd(q, k, v, "quadratic")
    assert rel(out0, oc) < 1e-13 and rel(den0, dc) < 1e-13, "prefill from zero != eq. 8"
    # a state as an earlier prompt leaves it: S of either sign, Z positive
    S_init = rand((B, H, D, M), 104)
    Z_init = 3.0 * phi_lib(rand((B, H, D), 105))
    out, den, S_N, Z_N = orc.causal_prefill(q, k, v, S_init, Z_init)
    fk = phi_lib(k)
    assert rel(S_N, S_init + np.matmul(np.swapaxes(fk, -1, -2), v)) < 1e-13, "S_N != S_0 + phi(K)^T V"
    assert rel(Z_N, Z_init + fk.sum(axis=2)) < 1e-14, "Z_N != Z_0 + sum phi(K)"
    fq = phi_lib(q)
    outz, denz, _, _ = orc.causal_prefill(q, np.full_like(k, -60.0), v, S_init, Z_init)
    dz = np.einsum("bhnd,bhd->bhn", fq, Z_init)
    assert rel(denz, dz) < 1e-12, "den != phi(Q) Z_0 when phi(K) ~ 0"
    assert rel(outz, np.matmul(fq, S_init) / dz[..., None]) < 1e-12, "out != phi(Q) S_0 / phi(Q) Z_0"
    n1 = 4
    cut = lambda x, a, b: np.ascontiguousarray(x[:, :, a:b])
    o1, d1, S1, Z1 = orc.causal_prefill(cut(q, 0, n1), cut(k, 0, n1), cut(v, 0, n1), S_init, Z_init)
    o2, d2, S2, Z2 = orc.causal_prefill(cut(q, n1, N), cut(k, n1, N), cut(v, n1, N), S1, Z1)
    assert rel(np.concatenate([o1, o2], axis=2), out) < 1e-13, "prefill cut in two differs"
    assert rel(np.concatenate([d1, d2], axis=2), den) < 1e-13
    assert rel(S2, S_N) < 1e-13 and rel(Z2, Z_N) < 1e-13
    steps = lambda x: np.ascontiguousarray(np.transpose(x[:, :, n1:], (2, 0, 1, 3)))  # [T,B,H,.]
    y, Sd, Zd = orc.decode(steps(q), steps(k), steps(v), S1, Z1)
    assert rel(np.transpose(y, (1, 2, 0, 3)), out[:, :, n1:]) < 1e-13, "prompt + RNN steps != one prefill"
    assert rel(Sd, S_N) < 1e-13 and rel(Zd, Z_N) < 1e-13


# ------------------------------------------------------------- RetNet decay

DECAYS = (0.0, 0.5, 0.9, 0.99)


def pin_decay_gamma_one(orc):
    """gamma = 1 is the undecayed method itself: the decayed entry points give
    the same bits as the (separately pinned) undecayed ones."""
    B, H, N, D, M = 2, 2, 9, 3, 5
    q, k, v, g = rand((B, H, N, D), 201), rand((B, H, N, D), 202), rand((B, H, N, M), 203), rand((B, H, N, M), 204)
    for form in ("recurrent", "quadratic"):
        a = orc.causal_fwd(q, k, v, form)
        b = orc.causal_fwd(q, k, v, form, gamma=1.0)
        assert all(np.array_equal(x, y) for x, y in zip(a, b)), f"{form} forward: gamma = 1 changed it"
        a = orc.causal_bwd(q, k, v, g, form)
        b = orc.causal_bwd(q, k, v, g, form, gamma=1.0)
        assert all(np.array_equal(x, y) for x, y in zip(a, b)), f"{form} gradients: gamma = 1 changed them"
    st = lambda x: np.ascontiguousarray(np.transpose(x, (2, 0, 1, 3)))
    a = orc.decode(st(q), st(k), st(v))
    b = orc.decode(st(q), st(k), st(v), gamma=1.0)
    assert all(np.array_equal(x, y) for x, y in zip(a, b)), "decode: gamma = 1 changed it"


def pin_decay_gamma_zero(orc):
    """gamma = 0 keeps only the pair i = j (gamma^0 = 1): V'_i = V_i,
    den_i = phi(Q_i) . phi(K_i) (numpy), dV = G and dQ = dK = 0; the decode
    state is the last token's phi(k) v^T."""
    B, H, N, D, M = 1, 2, 8, 3, 4
    q, k, v, g = rand((B, H, N, D), 211), rand((B, H, N, D), 212), rand((B, H, N, M), 213), rand((B, H, N, M), 214)
    for form in ("recurrent", "quadratic"):
        out, den = orc.causal_fwd(q, k, v, form, gamma=0.0)
        assert rel(out, v) < 1e-14, f"{form}: gamma = 0 must return V"
        assert rel(den, np.einsum("bhnd,bhnd->bhn", phi_lib(q), phi_lib(k))) < 1e-14
        dq, dk, dv = orc.causal_bwd(q, k, v, g, form, gamma=0.0)
        assert rel(dv, g) < 1e-14 and np.max(np.abs(dq)) < 1e-13 and np.max(np.abs(dk)) < 1e-13
    st = lambda x: np.ascontiguousarray(np.transpose(x, (2, 0, 1, 3)))
    y, S, Z = orc.decode(st(q), st(k), st(v), gamma=0.0)
    assert rel(y, st(v)) < 1e-14
    assert rel(S, np.einsum("bhd,bhm->bhdm", phi_lib(k[:, :, -1]), v[:, :, -1])) < 1e-14
    assert rel(Z, phi_lib(k[:, :, -1])) < 1e-14


def pin_decay_closed_form(orc):
    """Q = K = 0 makes phi = 1, so every pair weighs D gamma^(i-j): V'_i is
    the exponentially weighted mean of V_1..V_i and den_i = D sum_j gamma^(i-j),
    both by scipy's IIR filter y_i = x_i + gamma y_{i-1}; constant V rows are
    reproduced for any gamma."""
    B, H, N, D, M = 1, 2, 17, 3, 4
    z = np.zeros((B, H, N, D))
    v = rand((B, H, N, M), 221)
    for gm in DECAYS[1:]:
        num = scipy.signal.lfilter([1.0], [1.0, -gm], v, axis=2)
        cnt = scipy.signal.lfilter([1.0], [1.0, -gm], np.ones((B, H, N)), axis=2)
        for form in ("recurrent", "quadratic"):
            out, den = orc.causal_fwd(z, z, v, form, gamma=gm)
            assert rel(out, num / cnt[..., None]) < 1e-13, f"{form} gamma={gm}: not the weighted mean"
            assert rel(den, D * cnt) < 1e-13
            c = np.broadcast_to(rand((1, 1, 1, M), 222), v.shape).copy()
            outc, _ = orc.causal_fwd(rand((B, H, N, D), 223), rand((B, H, N, D), 224), c, form, gamma=gm)
            assert rel(outc, c) < 1e-13, "constant V not reproduced"


def pin_decay_forms_agree(orc):
    """The decayed quadratic form (every pair weighted gamma^(i-j)) and the
    decayed recurrence agree, forward and gradients."""
    for gm in DECAYS:
        for shp in RNG_SHAPES:
            B, H, N, D, M = shp
            q, k, v, g = rand((B, H, N, D), 231), rand((B, H, N, D), 232), rand((B, H, N, M), 233), rand((B, H, N, M), 234)
            o1, d1 = orc.causal_fwd(q, k, v, "recurrent", gamma=gm)
            o2, d2 = orc.causal_fwd(q, k, v, "quadratic", gamma=gm)
            assert rel(o1, o2) < 1e-12 and rel(d1, d2) < 1e-12, f"forward forms differ at gamma={gm}"
            if gm == 0.0:
                continue  # dq = dk = 0 exactly there (pin_decay_gamma_zero); only rounding is left
            a = orc.causal_bwd(q, k, v, g, "recurrent", gamma=gm)
            b = orc.causal_bwd(q, k, v, g, "quadratic", gamma=gm)
            for x, y, nm in zip(a, b, ("dq", "dk", "dv")):
                assert rel(x, y, 1e-3) < 1e-11, f"{nm} forms differ at gamma={gm}"  # N = 1: exact zeros


def pin_decay_grad_fd(orc):
    """Both decayed gradient forms against central finite differences of the
    decayed loss sum(G * V')."""
    B, H, N, D, M = 1, 1, 9, 3, 4
    q, k, v, g = rand((B, H, N, D), 241), rand((B, H, N, D), 242), rand((B, H, N, M), 243), rand((B, H, N, M), 244)
    for gm in (0.5, 0.9):
        loss = lambda q_, k_, v_: float(np.sum(g * orc.causal_fwd(q_, k_, v_, "recurrent", gamma=gm)[0]))
        h = 1e-6
        num = []
        for x, idx in ((q, 0), (k, 1), (v, 2)):
            gr = np.zeros_like(x)
            for e in np.ndindex(x.shape):
                args = [q.copy(), k.copy(), v.copy()]
                args[idx][e] += h
                up = loss(*args)
                args[idx][e] -= 2 * h
                gr[e] = (up - loss(*args)) / (2 * h)
            num.append(gr)
        for form in ("recurrent", "quadratic"):
            an = orc.causal_bwd(q, k, v, g, form, gamma=gm)
            for a_, n_, nm in zip(an, num, ("dq", "dk", "dv")):
                assert rel(a_, n_) < 1e-6, f"{form} {nm} != finite differences at gamma={gm}"


def pin_decay_invariants(orc):
    """The decayed output is still a normalised weighted mean per row, so
    phi(Q_i) . grad phi(Q_i) = 0, sum_j phi(K_j) . grad phi(K_j) = 0 and
    sum_j dV_j = sum_i G_i (checked through dq / phi' and dk / phi')."""
    B, H, N, D, M = 2, 1, 11, 3, 5
    q, k, v, g = rand((B, H, N, D), 251), rand((B, H, N, D), 252), rand((B, H, N, M), 253), rand((B, H, N, M), 254)
    fq, fk = phi_lib(q), phi_lib(k)
    dfq = np.where(q > 0, 1.0, np.exp(q))
    dfk = np.where(k > 0, 1.0, np.exp(k))
    for gm in (0.3, 0.9):
        dq, dk, dv = orc.causal_bwd(q, k, v, g, "recurrent", gamma=gm)
        gq, gk = dq / dfq, dk / dfk
        assert np.max(np.abs(np.sum(fq * gq, axis=-1))) < 1e-12, "phi(Q_i) . grad phi(Q_i) != 0"
        assert np.max(np.abs(np.sum(fk * gk, axis=(2, 3)))) < 1e-11, "sum phi(K) . grad phi(K) != 0"
        assert rel(dv.sum(axis=2), g.sum(axis=2)) < 1e-12, "sum dV != sum G"


def pin_decay_decode(orc):
    """Decayed RNN steps = the decayed causal form on the stacked sequence;
    the final state is sum_t gamma^(T-1-t) phi(k_t) v_t^T (numpy einsum)."""
    T, B, H, D, M = 10, 2, 2, 3, 4
    q, k, v = rand((T, B, H, D), 261), rand((T, B, H, D), 262), rand((T, B, H, M), 263)
    seq = lambda x: np.ascontiguousarray(np.transpose(x, (1, 2, 0, 3)))
    for gm in (0.4, 0.95):
        y, S, Z = orc.decode(q, k, v, gamma=gm)
        o, _ = orc.causal_fwd(seq(q), seq(k), seq(v), "quadratic", gamma=gm)
        assert rel(np.transpose(y, (1, 2, 0, 3)), o) < 1e-13, f"decode != decayed causal form at gamma={gm}"
        w = gm ** np.arange(T - 1, -1, -1.0)
        fk = phi_lib(k)
        assert rel(S, np.einsum("t,tbhd,tbhm->bhdm", w, fk, v)) < 1e-13
        assert rel(Z, np.einsum("t,tbhd->bhd", w, fk)) < 1e-13


# --------------------------------------------- decode with the projection

def pin_decode_proj(orc):
    """The projected step against things fixed outside it: with x = [q_h |
    k_h | v_h] of every head h in turn and W the identity, it is the plain
    decode step (orc_decode) on those q, k, v; for general W (columns grouped
    per head: W_Q, W_K, W_V of head 0, then head 1, ...) its state is S_0 +
    phi(k) v^T with k, v taken from numpy's x @ W by column slices, and its
    output is the quotient phi(q)^T S_1 / phi(q)^T Z_1 formed with numpy."""
    B, H, D, M = 5, 3, 4, 6
    q, k, v = rand((B, H, D), 301), rand((B, H, D), 302), rand((B, H, M), 303)
    S0, Z0 = rand((B, H, D, M), 304), 2.0 * phi_lib(rand((B, H, D), 305))
    x = np.concatenate([q, k, v], axis=2).reshape(B, -1)
    W = np.eye(x.shape[1])
    y, S1, Z1 = orc.decode_proj(x, W, H, D, M, S0, Z0)
    yd, Sd, Zd = orc.decode(q[None], k[None], v[None], S0, Z0)
    assert np.array_equal(y, yd[0]) and np.array_equal(S1, Sd) and np.array_equal(Z1, Zd), \
        "block-identity projection != the plain decode step"
    dm = 7
    x, W = rand((B, dm), 306), rand((dm, H * (2 * D + M)), 307, 0.5)
    y, S1, Z1 = orc.decode_proj(x, W, H, D, M, S0, Z0)
    p, n = x @ W, 2 * D + M
    pq = np.stack([p[:, h * n:h * n + D] for h in range(H)], axis=1)
    pk = np.stack([p[:, h * n + D:h * n + 2 * D] for h in range(H)], axis=1)
    pv = np.stack([p[:, h * n + 2 * D:(h + 1) * n] for h in range(H)], axis=1)
    fk, fq = phi_lib(pk), phi_lib(pq)
    assert rel(S1, S0 + np.einsum("bhd,bhm->bhdm", fk, pv)) < 1e-13, "S_1 != S_0 + phi(k) v^T"
    assert rel(Z1, Z0 + fk) < 1e-13
    num = np.einsum("bhd,bhdm->bhm", fq, S1)
    den = np.einsum("bhd,bhd->bh", fq, Z1)
    assert rel(y, num / den[..., None]) < 1e-13, "y != phi(q)^T S_1 / phi(q)^T Z_1"


# ------------------------------------------- degree-2 polynomial kernel

def _poly_features_full(x):
    """All D^2 products x_a x_b (numpy outer product, flattened): an exact
    feature map of (q . k)^2, independent of any packing the GPU uses."""
    return np.einsum("...a,...b->...ab", x, x).reshape(*x.shape[:-1], x.shape[-1] ** 2)


def pin_poly_feature_form(orc):
    """The pairwise form of sim = (q . k)^2 equals linear attention on the
    explicit D^2 features: S_i, Z_i as numpy cumulative sums of
    f(K_j) V_j^T and f(K_j), out_i = f(Q_i)^T S_i / f(Q_i)^T Z_i."""
    for B, H, N, D, M in ((1, 2, 11, 3, 5), (2, 1, 7, 4, 2)):
        q, k, v = rand((B, H, N, D), 501), rand((B, H, N, D), 502), rand((B, H, N, M), 503)
        out, den = orc.causal_fwd_poly(q, k, v)
        fq, fk = _poly_features_full(q), _poly_features_full(k)
        S = np.cumsum(np.einsum("bhnc,bhnm->bhncm", fk, v), axis=2)
        Z = np.cumsum(fk, axis=2)
        num = np.einsum("bhnc,bhncm->bhnm", fq, S)
        dn = np.einsum("bhnc,bhnc->bhn", fq, Z)
        assert rel(den, dn) < 1e-12, "den != f(Q) . Z"
        assert rel(out, num / dn[..., None]) < 1e-12, "out != f(Q)^T S / f(Q)^T Z"


def pin_poly_closed_forms(orc):
    """out_1 = V_1; constant V rows come back unchanged; with D = 1 the
    weights q_i^2 k_j^2 lose q_i in the quotient, so out_i is the k^2-weighted
    running mean of V (numpy) and dq = 0 (its terms cancel, to rounding)."""
    B, H, N, M = 1, 2, 9, 3
    q, k, v, g = rand((B, H, N, 1), 511), rand((B, H, N, 1), 512), rand((B, H, N, M), 513), rand((B, H, N, M), 514)
    out, _ = orc.causal_fwd_poly(q, k, v)
    w = k[..., 0] ** 2
    ref = np.cumsum(w[..., None] * v, axis=2) / np.cumsum(w, axis=2)[..., None]
    assert rel(out, ref) < 1e-12, "D = 1 is not the k^2-weighted running mean"
    dq, dk, _ = orc.causal_bwd_poly(q, k, v, g)
    assert np.max(np.abs(dq)) < 1e-12 * np.max(np.abs(dk)), "D = 1: the output depends on q"
    q, k = rand((B, H, N, 4), 515), rand((B, H, N, 4), 516)
    out, _ = orc.causal_fwd_poly(q, k, v)
    assert rel(out[:, :, 0], v[:, :, 0]) < 1e-13, "out_1 != V_1"
    c = np.broadcast_to(rand((B, H, 1, M), 517), v.shape).copy()
    out, _ = orc.causal_fwd_poly(q, k, c)
    assert rel(out, c) < 1e-12, "a constant V is not reproduced"


def pin_poly_grad_fd(orc):
    """dq, dk, dv against central finite differences of sum(G * V')."""
    B, H, N, D, M = 1, 2, 7, 3, 4
    q, k, v, g = rand((B, H, N, D), 521), rand((B, H, N, D), 522), rand((B, H, N, M), 523), rand((B, H, N, M), 524)
    loss = lambda q_, k_, v_: float(np.sum(g * orc.causal_fwd_poly(q_, k_, v_)[0]))
    h = 1e-6
    an = orc.causal_bwd_poly(q, k, v, g)
    for x, idx, nm in ((q, 0, "dq"), (k, 1, "dk"), (v, 2, "dv")):
        gr = np.zeros_like(x)
        for e in np.ndindex(x.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[idx][e] += h
            up = loss(*args)
            args[idx][e] -= 2 * h
            gr[e] = (up - loss(*args)) / (2 * h)
        assert rel(an[idx], gr) < 1e-6, f"{nm} != finite differences"


def pin_poly_invariants(orc):
    """sim(c q_i, k) = c^2 sim(q_i, k) leaves out_i unchanged, so
    q_i . dq_i = 0 for every i; a common scale of all k gives
    sum_j k_j . dk_j = 0; a constant row added to V gives sum_j dV_j =
    sum_i G_i."""
    B, H, N, D, M = 2, 1, 10, 3, 4
    q, k, v, g = rand((B, H, N, D), 531), rand((B, H, N, D), 532), rand((B, H, N, M), 533), rand((B, H, N, M), 534)
    dq, dk, dv = orc.causal_bwd_poly(q, k, v, g)
    scale = np.max(np.abs(dq)) * np.max(np.abs(q))
    assert np.max(np.abs(np.sum(q * dq, axis=-1))) < 1e-12 * scale * D, "q_i . dq_i != 0"
    assert np.max(np.abs(np.sum(k * dk, axis=(-2, -1)))) < 1e-11 * np.max(np.abs(dk)) * np.max(np.abs(k)) * N * D
    assert rel(np.sum(dv, axis=2), np.sum(g, axis=2)) < 1e-12, "sum dV != sum G"


ALL_PINS = [pin_phi, pin_causal_forms_agree, pin_causal_closed_forms, pin_grad_single_token, pin_noncausal_gemm,
            pin_noncausal_last_row, pin_noncausal_lengths, pin_grad_fd, pin_grad_forms_agree,
            pin_grad_invariants, pin_decode, pin_prefill, pin_decay_gamma_one, pin_decay_gamma_zero,
            pin_decay_closed_form, pin_decay_forms_agree, pin_decay_grad_fd, pin_decay_invariants,
            pin_decay_decode, pin_decode_proj, pin_poly_feature_form, pin_poly_closed_forms,
            pin_poly_grad_fd, pin_poly_invariants]
