"""Causal linear attention with the degree-2 polynomial kernel sim = (q . k)^2
("Transformers are RNNs", part 2/3, the feature-map discussion before eq. 7)
through the C ABI, against the fp64 oracle's pairwise form on the same seeded
bf16 inputs: max |gpu - oracle| / max |oracle| <= 2e-2 for out, den and dv
(bf16 inputs and features, fp32 accumulation), <= 4e-2 for dq and dk.  The
gradient bound comes from the arithmetic: fp64 emulations (features only
rounded to bf16; feature gradients only rounded to bf16) put those two
roundings at <= 1.3e-2 and <= 0.4e-2 of dq, dk at these shapes, and the bf16
scores, score gradients and gt of the tensor-core backward add about 1e-2
with elu + 1 and up to 2e-2 with the squared, wider-spread scores (measured
2.2-2.8e-2 in all).  Where the exact gradient is 0 (a one-token sequence; dq
at D = 1, where the output does not depend on q) its size is checked
instead, against the size of the terms that cancel in it.
"""
import numpy as np
import pytest
import torch

import oracle
from errstats import rel_err
from kernelized_causal_attention_gb300.workloads import causal_inputs

TOL = 2e-2
TOL_GRAD = 4e-2


def check_poly(la, dev, B, H, N, D, M, seed):
    q, k, v, g = causal_inputs(B, H, N, D, M, "bf16", seed)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    out, den = la.causal_fwd_poly(qd, kd, vd)
    dq, dk, dv = la.causal_bwd_poly(qd, kd, vd, out, den, gd)
    torch.cuda.synchronize()
    la.check_device_status()
    o_ref, den_ref = oracle.causal_fwd_poly(q, k, v)
    dq_ref, dk_ref, dv_ref = oracle.causal_bwd_poly(q, k, v, g)
    errs = {"out": rel_err(out, o_ref), "den": rel_err(den, den_ref), "dv": rel_err(dv, dv_ref)}
    if N == 1:
        # dq = dk = 0 only through gam + gt . V = 0; the kernels form gt in bf16,
        # so the cancellation leaves an error relative to the cancelling terms'
        # size, |gt| |V| d sim / d q = |G| |V| / den * 2 |q . k| |k| (and |q| for dk)
        qf, kf, vf, gf = (t.double().numpy() for t in (q, k, v, g))
        qk = np.abs(np.sum(qf * kf, axis=-1))
        tq = np.linalg.norm(gf, axis=-1) * np.linalg.norm(vf, axis=-1) / den_ref * 2 * qk
        errs["dq_abs"] = float(np.max(np.abs(dq.double().cpu().numpy())) / np.max(tq * np.linalg.norm(kf, axis=-1)))
        errs["dk_abs"] = float(np.max(np.abs(dk.double().cpu().numpy())) / np.max(tq * np.linalg.norm(qf, axis=-1)))
    else:
        errs["dk"] = rel_err(dk, dk_ref)
        if D == 1:
            # the terms that cancel in dq_i have size 2 |G_i| max |V_j| / |q_i|
            qf, vf, gf = (t.double().numpy() for t in (q, v, g))
            vmax = np.max(np.linalg.norm(vf, axis=-1), axis=-1)[..., None]
            scale = 2 * np.linalg.norm(gf, axis=-1) * vmax / np.maximum(np.abs(qf[..., 0]), 1e-30)
            errs["dq_abs"] = float(np.max(np.abs(dq.double().cpu().numpy()[..., 0]) / scale))
        else:
            errs["dq"] = rel_err(dq, dq_ref)
    bound = {"dq": TOL_GRAD, "dk": TOL_GRAD}
    bad = {n: e for n, e in errs.items() if not e <= bound.get(n, TOL)}
    assert not bad, f"poly B={B} H={H} N={N} D={D} M={M}: {errs}"
    return errs


CASES = [
    (1, 1, 1, 8, 64),      # one token: out = v, dq = dk = 0
    (1, 2, 200, 8, 64),    # two partial chunks
    (2, 1, 1000, 4, 32),   # several segments, ragged tail
    (1, 3, 3001, 10, 16),  # the widest map: 55 features
    (2, 2, 777, 1, 64),    # D = 1: the k^2-weighted running mean
    (3, 2, 129, 5, 32),
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,D,M", CASES)
def test_poly_small(cuda, linattn, B, H, N, D, M):
    check_poly(linattn, cuda, B, H, N, D, M, seed=9000 + N + D)


@pytest.mark.gpu
def test_poly_image_workload(cuda, linattn):
    """The 3072-token image shape with 8-wide heads (36 features)."""
    print(check_poly(linattn, cuda, 4, 8, 3072, 8, 64, seed=91))


# ------------------------------------------------------------- host checks

FAKE = 1 << 20


@pytest.mark.parametrize("kw,code", [
    (dict(D=11), "LA_ERR_UNSUPPORTED"),   # more than 64 features
    (dict(M=48), "LA_ERR_UNSUPPORTED"),
    (dict(dt=0), "LA_ERR_UNSUPPORTED"),   # fp32
    (dict(D=0), "LA_ERR_INVALID_ARG"),
    (dict(N=0), "LA_ERR_INVALID_ARG"),
    (dict(q=None), "LA_ERR_INVALID_ARG"),
    (dict(ws=None), "LA_ERR_WORKSPACE"),
])
def test_poly_argument_errors(linattn, kw, code):
    """Checked on the host before anything is launched (no GPU needed)."""
    la = linattn
    a = dict(q=FAKE, ws=FAKE, B=2, H=2, N=300, D=8, M=64, dt=la.LA_BF16)
    a.update(kw)
    L = la.lib()
    rc = L.la_causal_fwd_poly(a["q"], FAKE, FAKE, FAKE, FAKE, a["ws"], 1 << 40, a["B"], a["H"], a["N"],
                              a["D"], a["M"], a["dt"], None)
    assert rc == getattr(la, code)
    rc = L.la_causal_bwd_poly(a["q"], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["ws"], 1 << 40,
                              a["B"], a["H"], a["N"], a["D"], a["M"], a["dt"], None)
    assert rc == getattr(la, code)


def test_poly_workspace_and_launches(linattn):
    la = linattn
    f = la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD_POLY, 4, 8, 3072, 8, 64, la.LA_BF16)
    b = la.la_workspace_bytes(la.LA_OP_CAUSAL_BWD_POLY, 4, 8, 3072, 8, 64, la.LA_BF16)
    rows = 4 * 8 * 3072
    assert f >= 2 * rows * 64 * 2 and b >= 4 * rows * 64 * 2 and f % 16 == 0 and b % 16 == 0
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD_POLY, 4, 8, 3072, 11, 64, la.LA_BF16) == 0
    # one feature launch (q and k) + the tensor-core forward; + one gradient launch backward
    assert la.la_kernel_launches(la.LA_OP_CAUSAL_FWD_POLY, 4, 8, 3072, 8, 64, la.LA_BF16) == \
        1 + la.la_kernel_launches(la.LA_OP_CAUSAL_FWD, 4, 8, 3072, 64, 64, la.LA_BF16)
    assert la.la_kernel_launches(la.LA_OP_CAUSAL_BWD_POLY, 4, 8, 3072, 8, 64, la.LA_BF16) == \
        2 + la.la_kernel_launches(la.LA_OP_CAUSAL_BWD, 4, 8, 3072, 64, 64, la.LA_BF16)
    # a short workspace is refused before launching
    assert la.lib().la_causal_fwd_poly(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, f - 16, 4, 8, 3072, 8, 64,
                                       la.LA_BF16, None) == la.LA_ERR_WORKSPACE
