"""The RetNet decay ("Linear Attention/zh", variants and extensions): the causal
form with S_i = gamma S_{i-1} + phi(K_i) V_i^T and Z decaying alongside, its
gradients and the decayed RNN step, through the C ABI against the fp64 oracle
on the same seeded inputs.  Tolerances as for the undecayed calls:
max |gpu - oracle| / max |oracle| <= 1e-4 (fp32 inputs), 2e-2 (bf16 inputs).
"""
import numpy as np
import pytest
import torch

import oracle
from kernelized_causal_attention_gb300.workloads import WORKLOADS, DecodeStream, causal_inputs

TOL = {"f32": 1e-4, "bf16": 2e-2}


from errstats import rel_err  # noqa: E402  (normwise; records the elementwise figure)


def check_decay(la, dev, B, H, N, D, M, dtype, gamma, seed):
    q, k, v, g = causal_inputs(B, H, N, D, M, dtype, seed)
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    out, den = la.causal_fwd_decay(qd, kd, vd, gamma)
    dq, dk, dv = la.causal_bwd_decay(qd, kd, vd, out, den, gd, gamma)
    torch.cuda.synchronize()
    o_ref, den_ref = oracle.causal_fwd(q, k, v, gamma=gamma)
    dq_ref, dk_ref, dv_ref = oracle.causal_bwd(q, k, v, g, gamma=gamma)
    errs = {"out": rel_err(out, o_ref), "den": rel_err(den, den_ref), "dv": rel_err(dv, dv_ref)}
    if N == 1 or gamma == 0.0:
        # each output depends on its own token only: dq = dk = 0 exactly
        errs["dq_abs"] = float(dq.float().abs().max())
        errs["dk_abs"] = float(dk.float().abs().max())
    else:
        errs["dq"] = rel_err(dq, dq_ref)
        errs["dk"] = rel_err(dk, dk_ref)
    bad = {n: e for n, e in errs.items() if not e <= TOL[dtype]}
    assert not bad, f"decay B={B} H={H} N={N} D={D} M={M} {dtype} gamma={gamma}: {errs}"
    return errs


SMALL = [
    (1, 1, 1, 16, 16, "f32", 0.9),
    (1, 1, 70, 16, 32, "f32", 0.5),      # one segment, ragged second chunk
    (1, 2, 1000, 64, 64, "f32", 0.9),    # several segments: the decayed scan
    (2, 1, 3001, 32, 16, "f32", 0.99),
    (1, 3, 777, 64, 32, "bf16", 0.9),
    (2, 2, 2049, 64, 64, "bf16", 0.99),
    (1, 1, 500, 32, 64, "f32", 0.0),     # gamma = 0: out = v
    (1, 2, 300, 16, 16, "f32", 0.3),
    # bf16 forwards on the tensor cores for gamma >= 0.75, on the CUDA cores below
    (1, 2, 1000, 64, 64, "bf16", 0.75),
    (2, 1, 3001, 32, 32, "bf16", 0.95),
    (1, 2, 777, 64, 64, "bf16", 0.5),
    (1, 1, 1, 64, 64, "bf16", 0.9),
    # backward runs that cross heads with record sums at both ends
    (3, 7, 777, 64, 64, "bf16", 0.95),
    (1, 17, 2500, 64, 64, "bf16", 0.9),
    # long sequences: many segments, records weighted over long distances
    (1, 2, 65536, 64, 64, "bf16", 0.999),
    (1, 1, 20000, 32, 32, "bf16", 0.9),
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,D,M,dtype,gamma", SMALL)
def test_decay_small(cuda, linattn, B, H, N, D, M, dtype, gamma):
    check_decay(linattn, cuda, B, H, N, D, M, dtype, gamma, seed=7000 + N)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["causal_mnist_bf16", "causal_cifar_bf16"])
@pytest.mark.parametrize("gamma", [0.9, 0.99])
def test_decay_image_workloads(cuda, linattn, name, gamma):
    """The 784-token and 3072-token image workloads with the decay."""
    w = WORKLOADS[name]
    print(name, gamma, check_decay(linattn, cuda, w.B, w.H, w.N, w.D, w.M, w.dtype, gamma, w.seed))


@pytest.mark.gpu
def test_decay_gamma_zero_returns_v(cuda, linattn):
    q, k, v, _ = causal_inputs(2, 2, 333, 64, 64, "f32", 31)
    out, _ = linattn.causal_fwd_decay(q.to(cuda), k.to(cuda), v.to(cuda), 0.0)
    torch.cuda.synchronize()
    assert rel_err(out, v.double().numpy()) <= 1e-6


@pytest.mark.gpu
def test_decay_gamma_one_is_the_undecayed_call(cuda, linattn):
    """For shapes on the CUDA-core path the decayed entry point with gamma = 1
    runs the undecayed kernels: the same bits as la_causal_fwd / _bwd."""
    q, k, v, g = (t.to(cuda) for t in causal_inputs(1, 2, 1000, 32, 64, "f32", 32))
    a = linattn.causal_fwd(q, k, v)
    b = linattn.causal_fwd_decay(q, k, v, 1.0)
    ga = linattn.causal_bwd(q, k, v, a[0], a[1], g)
    gb = linattn.causal_bwd_decay(q, k, v, b[0], b[1], g, 1.0)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert all(torch.equal(x, y) for x, y in zip(ga, gb))


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,D,M,dtype,T,gamma", [
    (4, 2, 64, 64, "f32", 64, 0.9),
    (3, 3, 32, 16, "f32", 100, 0.5),
    (8, 8, 64, 64, "bf16", 40, 0.99),
])
def test_decay_decode(cuda, linattn, B, H, D, M, dtype, T, gamma):
    """T decayed RNN steps against the oracle: every y_t and the final S, Z."""
    ds = DecodeStream(B, H, D, M, dtype, seed=71)
    qs, ks, vs = ds.steps(T)
    S = torch.zeros(B, H, D, M, device=cuda)
    Z = torch.zeros(B, H, D, device=cuda)
    ys = torch.stack([linattn.decode_step_decay(qs[t].to(cuda), ks[t].to(cuda), vs[t].to(cuda), S, Z,
                                                gamma) for t in range(T)])
    torch.cuda.synchronize()
    y_ref, S_ref, Z_ref = oracle.decode(qs, ks, vs, gamma=gamma)
    tol = TOL[dtype] if dtype == "bf16" else 1e-4
    errs = [rel_err(ys, y_ref), rel_err(S, S_ref), rel_err(Z, Z_ref)]
    assert max(errs) <= tol, errs


@pytest.mark.gpu
def test_decay_decode_matches_decayed_causal(cuda, linattn):
    """The decayed RNN steps and the decayed causal form are the same
    operation: y_t = out_t of the causal call on the stacked sequence."""
    B, H, T, D, M, gamma = 2, 3, 150, 64, 64, 0.95
    q, k, v, _ = causal_inputs(B, H, T, D, M, "f32", 72)
    qd, kd, vd = (t.to(cuda) for t in (q, k, v))
    out, _ = linattn.causal_fwd_decay(qd, kd, vd, gamma)
    S = torch.zeros(B, H, D, M, device=cuda)
    Z = torch.zeros(B, H, D, device=cuda)
    ys = torch.stack([linattn.decode_step_decay(qd[:, :, t].contiguous(), kd[:, :, t].contiguous(),
                                                vd[:, :, t].contiguous(), S, Z, gamma)
                      for t in range(T)], dim=2)
    torch.cuda.synchronize()
    assert rel_err(ys, out.double().cpu().numpy()) <= 1e-5


# ------------------------------------------------------------- host checks

FAKE = 1 << 20


@pytest.mark.parametrize("gamma", [-0.1, 1.5, float("nan"), float("inf")])
def test_decay_rejects_gamma_outside_0_1(linattn, gamma):
    """Checked on the host before anything is launched (no GPU needed)."""
    la = linattn
    L = la.lib()
    assert L.la_causal_fwd_decay(FAKE, FAKE, FAKE, FAKE, FAKE, gamma, None, 0, 1, 1, 64, 16, 16,
                                 la.LA_F32, None) == la.LA_ERR_INVALID_ARG
    assert L.la_causal_bwd_decay(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, gamma, None, 0,
                                 1, 1, 64, 16, 16, la.LA_F32, None) == la.LA_ERR_INVALID_ARG
    assert L.la_decode_step_decay(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, gamma, 1, 1, 64, 64, la.LA_F32,
                                  None) == la.LA_ERR_INVALID_ARG


def test_decay_workspace_and_launches(linattn):
    la = linattn
    # the decayed forward's workspace covers both paths
    n = la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD_DECAY, 4, 8, 3072, 64, 64, la.LA_BF16)
    assert n >= la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD, 4, 8, 3072, 64, 64, la.LA_BF16)
    assert n > 0 and n % 16 == 0
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL_BWD_DECAY, 4, 8, 3072, 64, 64, la.LA_BF16) > n
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL_BWD_DECAY, 4, 8, 3072, 64, 64, la.LA_BF16) >= \
        la.la_workspace_bytes(la.LA_OP_CAUSAL_BWD, 4, 8, 3072, 64, 64, la.LA_BF16)
    assert la.la_kernel_launches(la.LA_OP_CAUSAL_FWD_DECAY, 4, 8, 3072, 64, 64, la.LA_BF16) == \
        la.la_kernel_launches(la.LA_OP_CAUSAL_FWD, 4, 8, 3072, 64, 64, la.LA_BF16)  # tensor cores
    assert la.la_kernel_launches(la.LA_OP_CAUSAL_FWD_DECAY, 4, 8, 3072, 64, 64, la.LA_F32) == 3
    assert la.la_kernel_launches(la.LA_OP_CAUSAL_BWD_DECAY, 1, 1, 64, 16, 16, la.LA_F32) == 1
    assert la.la_kernel_launches(la.LA_OP_CAUSAL_BWD_DECAY, 4, 8, 3072, 64, 64, la.LA_BF16) == \
        la.la_kernel_launches(la.LA_OP_CAUSAL_BWD, 4, 8, 3072, 64, 64, la.LA_BF16)  # tensor cores
    # a missing workspace is reported before launching
    assert la.lib().la_causal_fwd_decay(FAKE, FAKE, FAKE, FAKE, FAKE, 0.9, None, 0, 4, 8, 3072, 64, 64,
                                        la.LA_BF16, None) == la.LA_ERR_WORKSPACE
