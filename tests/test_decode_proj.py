"""The decode step fed by its own projection ("Transformers are RNNs" §3.4,
eq. 18-20 without f_l and the residual) through the C ABI, against the fp64
oracle (numpy x @ W, then the plain RNN step) on the same seeded bf16 inputs.

Tolerances, written as max |gpu - oracle| / max |oracle| per output: the
states S and Z are fp32 on both sides of the kernel (the projection
accumulates bf16 products in fp32 over d_model terms: relative error about
d_model * 2^-24, far below 1e-4); y is rounded to bf16 on output (half an ulp
of bf16 is 2^-9 of the value), so 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from kernelized_causal_attention_gb300.workloads import WORKLOADS, proj_inputs

TOL_STATE = 1e-4
TOL_Y = 1e-2


def errs(gpu, ref):
    """(normwise max relative error, largest elementwise relative error over
    entries above 1e-3 of the largest); only the first is asserted."""
    g = gpu.detach().double().cpu().numpy()
    assert np.all(np.isfinite(g)), "non-finite values in the GPU result"
    scale = max(np.max(np.abs(ref)), 1e-30)
    big = np.abs(ref) > 1e-3 * scale
    elem = float(np.max(np.abs(g - ref)[big] / np.abs(ref)[big])) if big.any() else 0.0
    return float(np.max(np.abs(g - ref)) / scale), elem


def run_step(la, dev, x, W, S, Z, H, D, M):
    Sd, Zd = S.to(dev), Z.to(dev)
    y = la.decode_step_proj(x.to(dev), W.to(dev), Sd, Zd, H, D, M)
    torch.cuda.synchronize()
    return y, Sd, Zd


def check(la, dev, B, dm, H, D, M, seed, t=100, rows=None):
    """One step on all B streams; compared on all of them, or on `rows` (the
    oracle takes the same rows of x, S, Z: the streams are independent)."""
    x, W, S, Z = proj_inputs(B, dm, H, D, M, t=t, seed=seed)
    y, S1, Z1 = run_step(la, dev, x, W, S, Z, H, D, M)
    if rows is None:
        rows = torch.arange(B)
    y_ref, S_ref, Z_ref = oracle.decode_proj(x[rows], W, H, D, M, S[rows], Z[rows])
    e = {"y": errs(y[rows.to(dev)], y_ref), "S": errs(S1[rows.to(dev)], S_ref),
         "Z": errs(Z1[rows.to(dev)], Z_ref)}
    bad = [n for n, tol in (("y", TOL_Y), ("S", TOL_STATE), ("Z", TOL_STATE)) if not e[n][0] <= tol]
    assert not bad, f"B={B} d_model={dm} H={H} D={D} M={M}: {e}"
    return e


SMALL = [
    (1, 64, 1, 16, 16),      # one stream, one slab
    (7, 128, 3, 32, 64),     # ragged block, two slabs
    (100, 320, 2, 64, 64),   # five slabs: the three-stage ring wraps
    (130, 192, 5, 64, 32),   # several blocks, last one ragged
    (64, 256, 4, 32, 32),
    (33, 64, 2, 16, 64),
    (90, 128, 3, 64, 16),
    (65, 512, 1, 32, 16),
    (300, 128, 2, 16, 32),
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,dm,H,D,M", SMALL)
def test_decode_proj_small(cuda, linattn, B, dm, H, D, M):
    check(linattn, cuda, B, dm, H, D, M, seed=8000 + B)


@pytest.mark.gpu
def test_decode_proj_256_streams(cuda, linattn):
    """256 streams, d_model = 512, 8 heads of 64: every output."""
    w = WORKLOADS["decode_proj_bf16"]
    print(check(linattn, cuda, w.B, w.d_model, w.H, w.D, w.M, w.seed, t=w.N))


@pytest.mark.gpu
def test_decode_proj_10000_streams(cuda, linattn):
    """10,000 streams (the MNIST batch of §4.2.1), d_model = 256, 8 heads of
    32: 1,500 sampled streams, among them the last, partly filled block."""
    w = WORKLOADS["decode_proj_mnist_bf16"]
    gen = torch.Generator().manual_seed(99)
    rows = torch.cat([torch.randperm(w.B - 64, generator=gen)[:1436], torch.arange(w.B - 64, w.B)])
    print(check(linattn, cuda, w.B, w.d_model, w.H, w.D, w.M, w.seed, t=w.N, rows=rows))


@pytest.mark.gpu
def test_decode_proj_steps_carry_the_state(cuda, linattn):
    """Six steps in a row, each with a fresh x: the states carried on the GPU
    against the oracle's."""
    B, dm, H, D, M = 100, 128, 3, 32, 64
    x, W, S, Z = proj_inputs(B, dm, H, D, M, t=0, seed=81)
    S, Z = S * 0, Z * 0  # from the start of a sequence (eq. 16-17)
    Sd, Zd, Wd = S.to(cuda), Z.to(cuda), W.to(cuda)
    S_ref, Z_ref = S.double().numpy(), Z.double().numpy()
    for step in range(6):
        xs = proj_inputs(B, dm, H, D, M, seed=900 + step)[0]
        y = linattn.decode_step_proj(xs.to(cuda), Wd, Sd, Zd, H, D, M)
        y_ref, S_ref, Z_ref = oracle.decode_proj(xs, W, H, D, M, S_ref, Z_ref)
        torch.cuda.synchronize()
        assert errs(y, y_ref)[0] <= TOL_Y, step
    assert errs(Sd, S_ref)[0] <= TOL_STATE and errs(Zd, Z_ref)[0] <= TOL_STATE


@pytest.mark.gpu
def test_decode_proj_matches_the_plain_step(cuda, linattn):
    """The fused step and la_decode_step fed with the same q, k, v (the
    projection formed here with torch in fp32, rounded to bf16 for the plain
    step's inputs) agree to bf16 rounding of q, k, v."""
    B, dm, H, D, M = 200, 256, 4, 64, 64
    x, W, S, Z = proj_inputs(B, dm, H, D, M, seed=82)
    y, S1, _ = run_step(linattn, cuda, x, W, S, Z, H, D, M)
    p = (x.float() @ W.float()).view(B, H, 2 * D + M)
    q, k, v = (p[..., :D], p[..., D:2 * D], p[..., 2 * D:])
    S2, Z2 = S.to(cuda), Z.to(cuda)
    y2 = linattn.decode_step(q.bfloat16().contiguous().to(cuda), k.bfloat16().contiguous().to(cuda),
                             v.bfloat16().contiguous().to(cuda), S2, Z2)
    torch.cuda.synchronize()
    assert errs(y, y2.double().cpu().numpy())[0] <= 2e-2
    assert errs(S1, S2.double().cpu().numpy())[0] <= 2e-2


# ------------------------------------------------------------- host checks

FAKE = 1 << 20


@pytest.mark.parametrize("kw,code", [
    (dict(dt=0), "LA_ERR_UNSUPPORTED"),        # fp32 x and W
    (dict(dm=96), "LA_ERR_UNSUPPORTED"),       # not whole slabs of 64
    (dict(dm=16448), "LA_ERR_UNSUPPORTED"),    # above 16384
    (dict(dm=0), "LA_ERR_INVALID_ARG"),
    (dict(D=48), "LA_ERR_UNSUPPORTED"),
    (dict(B=0), "LA_ERR_INVALID_ARG"),
    (dict(B=1 << 18, H=8), "LA_ERR_INVALID_ARG"),  # B*H above 2^20
    (dict(B=1, H=70000), "LA_ERR_INVALID_ARG"),    # more heads than grid rows
    (dict(x=None), "LA_ERR_INVALID_ARG"),
    (dict(W=FAKE + 8), "LA_ERR_INVALID_ARG"),      # misaligned
    (dict(dt=5), "LA_ERR_INVALID_ARG"),
])
def test_decode_proj_argument_errors(linattn, kw, code):
    """Checked on the host before anything is launched (no GPU needed)."""
    la = linattn
    a = dict(x=FAKE, W=FAKE, S=FAKE, Z=FAKE, y=FAKE, B=4, H=2, dm=128, D=64, M=64, dt=la.LA_BF16)
    a.update(kw)
    rc = la.lib().la_decode_step_proj(a["x"], a["W"], a["S"], a["Z"], a["y"], a["B"], a["H"],
                                      a["dm"], a["D"], a["M"], a["dt"], None)
    assert rc == getattr(la, code)


def test_decode_proj_workspace_and_launches(linattn):
    la = linattn
    assert la.la_workspace_bytes(la.LA_OP_DECODE_PROJ, 10000, 8, 256, 32, 32, la.LA_BF16) == 0
    assert la.la_kernel_launches(la.LA_OP_DECODE_PROJ, 10000, 8, 256, 32, 32, la.LA_BF16) == 1
    assert la.la_kernel_launches(la.LA_OP_DECODE_PROJ, 10000, 8, 100, 32, 32, la.LA_BF16) == 0
    assert la.la_kernel_launches(la.LA_OP_DECODE_PROJ, 10000, 8, 256, 32, 32, la.LA_F32) == 0


@pytest.mark.gpu
def test_decode_proj_limits(cuda, linattn):
    """The largest stream count (B*H = 2^20, 16-wide heads) on sampled streams,
    and the widest layer input (d_model = 16384: 256 slabs through the ring)."""
    B, H, D, M, dm = (1 << 20) // 8, 8, 16, 16, 64
    gen = torch.Generator().manual_seed(5)
    rows = torch.cat([torch.randperm(B - 64, generator=gen)[:400], torch.arange(B - 64, B)])
    print(check(linattn, cuda, B, dm, H, D, M, seed=96, rows=rows))
    print(check(linattn, cuda, 100, 16384, 2, 64, 64, seed=97))
