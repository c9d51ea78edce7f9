"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs, element by element.

Tolerance: max |gpu - oracle| / max |oracle| per tensor (normwise-max
relative error), <= 1e-4 for fp32 inputs and <= 2e-2 for bf16 inputs with
fp32 accumulation.  For bf16 the oracle receives exactly the bf16-rounded
inputs, widened to fp64.
"""
import numpy as np
import pytest
import torch

import oracle
from kernelized_causal_attention_gb300.workloads import (WORKLOADS, DecodeStream, causal_inputs,
                                                         noncausal_inputs)

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


from errstats import rel_err  # noqa: E402  (normwise; records the elementwise figure)


def _to(dev, *ts):
    return [t.to(dev).contiguous() for t in ts]


def check_causal(la, dev, B, H, N, D, M, dtype, seed):
    q, k, v, g = causal_inputs(B, H, N, D, M, dtype, seed)
    qd, kd, vd, gd = _to(dev, q, k, v, g)
    out, den = la.causal_fwd(qd, kd, vd)
    dq, dk, dv = la.causal_bwd(qd, kd, vd, out, den, gd)
    torch.cuda.synchronize()
    o_ref, den_ref = oracle.causal_fwd(q, k, v)
    dq_ref, dk_ref, dv_ref = oracle.causal_bwd(q, k, v, g)
    tol = TOL[dtype]
    errs = {"out": rel_err(out, o_ref), "den": rel_err(den, den_ref), "dv": rel_err(dv, dv_ref)}
    if N == 1:
        # a single token: out = v whatever q and k are, so dq = dk = 0 exactly;
        # a relative error against zero is meaningless, check the absolute size
        errs["dq_abs"] = float(dq.abs().max())
        errs["dk_abs"] = float(dk.abs().max())
    else:
        errs["dq"] = rel_err(dq, dq_ref)
        errs["dk"] = rel_err(dk, dk_ref)
    bad = {k_: e for k_, e in errs.items() if not e <= tol}
    assert not bad, f"causal B={B} H={H} N={N} D={D} M={M} {dtype}: {errs}"
    return errs


# small and ragged cases first: N=1, N below one chunk, ragged tails, many
# segments per head (small B*H), D != M, every supported head size
SMALL = [
    (1, 1, 1, 16, 16, "f32"),
    (1, 1, 5, 32, 16, "f32"),
    (1, 1, 64, 16, 16, "f32"),
    (2, 3, 100, 32, 64, "f32"),
    (1, 2, 333, 64, 32, "f32"),
    (1, 1, 1000, 64, 64, "f32"),
    (3, 1, 129, 16, 64, "f32"),
    (1, 2, 200, 64, 32, "bf16"),
    (2, 2, 257, 64, 64, "bf16"),
    (1, 1, 2049, 32, 32, "bf16"),
    (2, 1, 77, 16, 16, "bf16"),
    # bf16 heads narrower than 64 also run on the tensor cores (tiles zero-filled
    # to 64 columns, phi zeroed on the padded features)
    (1, 1, 1, 32, 32, "bf16"),
    (2, 2, 1000, 32, 64, "bf16"),
    (1, 3, 3001, 16, 32, "bf16"),
    (3, 2, 129, 64, 16, "bf16"),
    (1, 1, 4097, 32, 32, "bf16"),
    (8, 8, 784, 32, 32, "bf16"),
    # bf16 with D = M = 64 runs on the tensor cores: 128-token chunks, segments
    (1, 1, 1, 64, 64, "bf16"),
    (1, 1, 100, 64, 64, "bf16"),
    (1, 3, 128, 64, 64, "bf16"),
    (3, 1, 1000, 64, 64, "bf16"),
    (40, 4, 300, 64, 64, "bf16"),
    (1, 1, 4097, 64, 64, "bf16"),
    # backward runs over whole sub-segments that cross from one (b, h) into the
    # next, start or end mid-head (record sums at both ends), ragged last chunks
    (3, 7, 777, 64, 64, "bf16"),     # both roles cross heads
    (2, 5, 2000, 64, 64, "bf16"),    # two sub-segments per state-pass CTA
    (1, 17, 2500, 32, 64, "bf16"),   # 2-chunk sub-segments, dq runs cross heads
    (1, 2, 6000, 64, 64, "bf16"),    # a one-chunk last sub-segment
    (64, 64, 100, 64, 64, "bf16"),   # one-chunk heads: each run crosses ~28 heads
    (32, 64, 129, 64, 64, "bf16"),   # two-chunk heads, a one-token last chunk
]


@pytest.mark.parametrize("B,H,N,D,M,dtype", SMALL)
def test_causal_small(cuda, linattn, B, H, N, D, M, dtype):
    check_causal(linattn, cuda, B, H, N, D, M, dtype, seed=1000 + N)


@pytest.mark.parametrize("B,H,N,D,M,dtype", [
    (1, 2, 65536, 64, 64, "bf16"),   # the sweep's longest sequence, tensor cores (74 segments)
    (1, 1, 16384, 32, 32, "f32"),    # CUDA cores, 256 chunks
])
def test_causal_long(cuda, linattn, B, H, N, D, M, dtype):
    check_causal(linattn, cuda, B, H, N, D, M, dtype, 5000 + N)


def test_causal_beyond_2_31_elements(cuda, linattn):
    """Tensors of 1 x 160 x 2^18 x 64 = 2.7e9 elements (5.4 GB each in bf16):
    the last head starts past element 2^31, so its reads and writes need
    64-bit offsets.  Inputs are drawn on the GPU from a seeded generator; out,
    den and dq of a token depend only on the tokens up to it, so the last
    head's first 2048 tokens are checked against the oracle on that prefix."""
    if torch.cuda.get_device_properties(cuda).total_memory < 120 * 2**30:
        pytest.skip("needs about 60 GB of device memory")
    B, H, N, D, M, P = 1, 160, 1 << 18, 64, 64, 2048
    gen = torch.Generator(device=cuda).manual_seed(2031)
    q, k, v, g = (torch.randn(B, H, N, D, generator=gen, device=cuda, dtype=torch.bfloat16)
                  for _ in range(4))
    out, den = linattn.causal_fwd(q, k, v)
    dq, dk, dv = linattn.causal_bwd(q, k, v, out, den, g)
    torch.cuda.synchronize()
    h = H - 1
    assert (h * N * D) > 2**31
    pre = lambda t: t[:, h:h + 1, :P].cpu()
    o_ref, den_ref = oracle.causal_fwd(pre(q), pre(k), pre(v))
    dq_ref, _, _ = oracle.causal_bwd(pre(q), pre(k), pre(v), pre(g))
    errs = {"out": rel_err(out[:, h:h + 1, :P], o_ref), "den": rel_err(den[:, h:h + 1, :P], den_ref),
            "dq": rel_err(dq[:, h:h + 1, :P], dq_ref)}
    assert all(e <= TOL["bf16"] for e in errs.values()), errs
    # every element written: finite outputs and gradients at the far end too
    for t in (out, dq, dk, dv):
        assert torch.isfinite(t[:, h, -P:].float()).all()
    linattn.check_device_status()


@pytest.mark.parametrize("name", ["causal_tiny_f32", "causal_mnist_bf16", "causal_cifar_bf16", "causal_cifar_d32_bf16",
                                  "causal_cifar_f32"])
def test_causal_workloads(cuda, linattn, name):
    w = WORKLOADS[name]
    errs = check_causal(linattn, cuda, w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed)
    print(name, errs)


# ------------------------------------------------------------------ prefill

def earlier_state(B, H, D, M, dtype, seed, P=37):
    """(S, Z) as an earlier prompt of P tokens leaves them (oracle, fp64,
    rounded to fp32 -- the GPU and the oracle both start from these values)."""
    q, k, v, _ = causal_inputs(B, H, P, D, M, dtype, seed)
    _, _, S, Z = oracle.causal_prefill(q, k, v)
    return torch.from_numpy(S).float(), torch.from_numpy(Z).float()


PREFILL = [
    (1, 1, 1, 16, 16, "f32"),
    (2, 3, 100, 32, 64, "f32"),
    (1, 2, 1000, 64, 64, "f32"),     # several segments on the CUDA cores
    (2, 1, 77, 16, 16, "bf16"),
    # bf16, D = M = 64: the tensor cores
    (1, 1, 1, 64, 64, "bf16"),
    (1, 1, 100, 64, 64, "bf16"),     # one partial chunk, one segment
    (3, 1, 1000, 64, 64, "bf16"),    # several segments, ragged tail
    (40, 4, 300, 64, 64, "bf16"),    # more heads than SMs: one segment each
    (4, 8, 3072, 64, 64, "bf16"),    # the 3072-token image workload's size
]


@pytest.mark.parametrize("B,H,N,D,M,dtype", PREFILL)
def test_causal_prefill(cuda, linattn, B, H, N, D, M, dtype):
    """The causal form from a state (eq. 16-19 over a prompt): out, den and
    the state after the sequence against the oracle, from the state an
    earlier prompt left."""
    q, k, v, _ = causal_inputs(B, H, N, D, M, dtype, 3100 + N)
    S0, Z0 = earlier_state(B, H, D, M, dtype, 3200 + N)
    qd, kd, vd, S, Z = _to(cuda, q, k, v, S0, Z0)
    out, den, S, Z = linattn.causal_prefill(qd, kd, vd, S, Z)
    torch.cuda.synchronize()
    o_ref, den_ref, S_ref, Z_ref = oracle.causal_prefill(q, k, v, S0, Z0)
    errs = {"out": rel_err(out, o_ref), "den": rel_err(den, den_ref), "S": rel_err(S, S_ref),
            "Z": rel_err(Z, Z_ref)}
    bad = {k_: e for k_, e in errs.items() if not e <= TOL[dtype]}
    assert not bad, f"prefill B={B} H={H} N={N} D={D} M={M} {dtype}: {errs}"


@pytest.mark.parametrize("D,M,dtype", [(64, 64, "bf16"), (32, 64, "f32")])
def test_prefill_then_decode(cuda, linattn, D, M, dtype):
    """A prompt through la_causal_prefill, the rest of the sequence token by
    token through la_decode_step from the state it leaves: outputs and final
    state are those of one pass over the whole sequence (oracle)."""
    B, H, N, n1 = 2, 3, 300, 211
    q, k, v, _ = causal_inputs(B, H, N, D, M, dtype, 77)
    qd, kd, vd = _to(cuda, q, k, v)
    head = lambda x: x[:, :, :n1].contiguous()
    out1, _, S, Z = linattn.causal_prefill(head(qd), head(kd), head(vd))
    ys = [linattn.decode_step(qd[:, :, t].contiguous(), kd[:, :, t].contiguous(),
                              vd[:, :, t].contiguous(), S, Z) for t in range(n1, N)]
    y = torch.stack(ys, dim=2)
    torch.cuda.synchronize()
    o_ref, _, S_ref, Z_ref = oracle.causal_prefill(q, k, v)
    errs = {"prompt": rel_err(out1, o_ref[:, :, :n1]), "steps": rel_err(y, o_ref[:, :, n1:]),
            "S": rel_err(S, S_ref), "Z": rel_err(Z, Z_ref)}
    bad = {k_: e for k_, e in errs.items() if not e <= TOL[dtype]}
    assert not bad, f"prefill + decode D={D} M={M} {dtype}: {errs}"


def check_noncausal(la, dev, B, H, N, D, M, dtype, seed, len_range):
    lengths, q, k, v, g = noncausal_inputs(B, H, N, D, M, dtype, seed, len_range)
    qd, kd, vd, gd = _to(dev, q, k, v, g)
    ld = lengths.to(dev) if len_range is not None else None
    out, den, S, Z = la.noncausal_fwd(qd, kd, vd, ld)
    dq, dk, dv = la.noncausal_bwd(qd, kd, vd, ld, out, den, S, Z, gd)
    torch.cuda.synchronize()
    lens = lengths if len_range is not None else None
    o_ref, den_ref, S_ref, Z_ref = oracle.noncausal_fwd(q, k, v, lens)
    dq_ref, dk_ref, dv_ref = oracle.noncausal_bwd(q, k, v, g, lens)
    tol = TOL[dtype]
    errs = {"out": rel_err(out, o_ref), "den": rel_err(den, den_ref), "S": rel_err(S, S_ref),
            "Z": rel_err(Z, Z_ref), "dv": rel_err(dv, dv_ref)}
    if N == 1:  # one valid token: dq = dk = 0 exactly (see the causal case)
        errs["dq_abs"] = float(dq.abs().max())
        errs["dk_abs"] = float(dk.abs().max())
    else:
        errs["dq"] = rel_err(dq, dq_ref)
        errs["dk"] = rel_err(dk, dk_ref)
    bad = {k_: e for k_, e in errs.items() if not e <= tol}
    assert not bad, f"non-causal B={B} H={H} N={N} D={D} M={M} {dtype}: {errs}"
    # padded rows are exactly zero
    for b, L in enumerate(lengths.tolist() if len_range is not None else [N] * B):
        for t in (out, den, dq, dk, dv):
            assert torch.all(t[b, :, L:] == 0)
    return errs


@pytest.mark.parametrize("B,H,N,D,M,dtype,lr", [
    (1, 1, 1, 16, 16, "f32", None),
    (2, 3, 100, 32, 64, "f32", (1, 100)),
    (4, 2, 300, 64, 64, "f32", (0, 300)),
    (3, 2, 513, 64, 32, "bf16", (200, 513)),
    (2, 1, 64, 16, 16, "f32", (64, 64)),
    # D = M = 64: several 128-token chunks and segments, ragged tails,
    # empty sequences, no lengths, one token, forty partial records
    (2, 3, 1000, 64, 64, "bf16", (0, 1000)),
    (1, 2, 777, 64, 64, "f32", None),
    (1, 1, 1, 64, 64, "f32", None),
    (5, 1, 2500, 64, 64, "f32", (1, 2500)),
    (100, 10, 100, 64, 64, "f32", (0, 100)),  # enough heads for one CTA per head
])
def test_noncausal_small(cuda, linattn, B, H, N, D, M, dtype, lr):
    check_noncausal(linattn, cuda, B, H, N, D, M, dtype, 2000 + N, lr)


@pytest.mark.parametrize("D,M,dtype", [(64, 64, "f32"), (64, 64, "bf16"), (32, 32, "f32")])
@pytest.mark.parametrize("raw", [(0, 0, 0, 0), (-5, 0, 301, 1000), (300, -1, 1, 299)])
def test_noncausal_length_edges(cuda, linattn, D, M, dtype, raw):
    """Every sequence empty, and lengths outside [0, N], which the ABI clamps:
    the GPU gets the raw lengths, the oracle the clamped ones."""
    B, H, N = 4, 2, 300
    _, q, k, v, g = noncausal_inputs(B, H, N, D, M, dtype, 4242, None)
    raw_l = torch.tensor(raw, dtype=torch.int32)
    lens = raw_l.clamp(0, N)
    qd, kd, vd, gd = _to(cuda, q, k, v, g)
    out, den, S, Z = linattn.noncausal_fwd(qd, kd, vd, raw_l.to(cuda))
    dq, dk, dv = linattn.noncausal_bwd(qd, kd, vd, raw_l.to(cuda), out, den, S, Z, gd)
    torch.cuda.synchronize()
    o_ref, den_ref, S_ref, Z_ref = oracle.noncausal_fwd(q, k, v, lens)
    dq_ref, dk_ref, dv_ref = oracle.noncausal_bwd(q, k, v, g, lens)
    tol = TOL[dtype]
    errs = {"out": rel_err(out, o_ref), "den": rel_err(den, den_ref), "S": rel_err(S, S_ref),
            "Z": rel_err(Z, Z_ref), "dq": rel_err(dq, dq_ref), "dk": rel_err(dk, dk_ref),
            "dv": rel_err(dv, dv_ref)}
    bad = {k_: e for k_, e in errs.items() if not e <= tol}
    assert not bad, f"lengths {raw}, D={D} M={M} {dtype}: {errs}"
    for b, L in enumerate(lens.tolist()):
        for t in (out, den, dq, dk, dv):
            assert torch.all(t[b, :, L:] == 0)
        if L == 0:
            assert torch.all(S[b] == 0) and torch.all(Z[b] == 0)


def test_noncausal_workload(cuda, linattn):
    w = WORKLOADS["noncausal_speech_f32"]
    errs = check_noncausal(linattn, cuda, w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.len_range)
    print(w.name, errs)


def test_noncausal_beyond_2_31_elements(cuda, linattn):
    """fp32 tensors of 2 x 80 x 2^18 x 64 = 2.7e9 elements (10.7 GB each): the
    second batch entry lies past element 2^31.  Its valid length is 2048, so
    all of its outputs and gradients depend on its first 2048 tokens only:
    its last head is checked against the oracle on those, and its padded
    rows must be zero; the first entry runs all 2^18 tokens."""
    if torch.cuda.get_device_properties(cuda).total_memory < 160 * 2**30:
        pytest.skip("needs about 90 GB of device memory")
    B, H, N, D, M, P = 2, 80, 1 << 18, 64, 64, 2048
    gen = torch.Generator(device=cuda).manual_seed(2032)
    q, k, v, g = (torch.randn(B, H, N, D, generator=gen, device=cuda) for _ in range(4))
    lengths = torch.tensor([N, P], dtype=torch.int32, device=cuda)
    out, den, S, Z = linattn.noncausal_fwd(q, k, v, lengths)
    dq, dk, dv = linattn.noncausal_bwd(q, k, v, lengths, out, den, S, Z, g)
    torch.cuda.synchronize()
    b, h = 1, H - 1
    assert (b * H + h) * N * D > 2**31
    pre = lambda t: t[b:b + 1, h:h + 1, :P].cpu()
    o_ref, den_ref, S_ref, Z_ref = oracle.noncausal_fwd(pre(q), pre(k), pre(v))
    dq_ref, dk_ref, dv_ref = oracle.noncausal_bwd(pre(q), pre(k), pre(v), pre(g))
    got = lambda t: t[b:b + 1, h:h + 1, :P]
    errs = {"out": rel_err(got(out), o_ref), "den": rel_err(got(den), den_ref),
            "S": rel_err(S[b:b + 1, h:h + 1], S_ref), "Z": rel_err(Z[b:b + 1, h:h + 1], Z_ref),
            "dq": rel_err(got(dq), dq_ref), "dk": rel_err(got(dk), dk_ref), "dv": rel_err(got(dv), dv_ref)}
    assert all(e <= TOL["f32"] for e in errs.values()), errs
    for t in (out, den, dq, dk, dv):
        assert torch.all(t[b, :, P:] == 0)
    linattn.check_device_status()


def test_every_output_written_launch_after_launch(cuda, linattn):
    """Outputs are filled with NaN before every call, over a sequence of
    non-causal, causal, prefill and decode calls in both dtypes and several
    cluster and segment counts: every element must come back finite (written by the
    kernels, and nothing one launch leaves in shared or tensor memory leaks
    into the next)."""
    la, nan = linattn, float("nan")
    nc_cases = [(2, 3, 1000, "bf16", (0, 1000), 3000), (2, 3, 1000, "f32", (0, 1000), 3000),
                (4, 2, 300, "f32", None, 0), (4, 2, 300, "bf16", None, 0),
                (5, 1, 2500, "f32", (1, 2500), 4500), (100, 10, 100, "f32", (0, 100), 2100),
                (2, 3, 1000, "bf16", (0, 1000), 77), (3, 2, 700, "bf16", (0, 20), 5)]
    for B, H, N, dt, lr, seed in nc_cases:
        D = M = 64
        lengths, q, k, v, g = noncausal_inputs(B, H, N, D, M, dt, seed, lr)
        qd, kd, vd, gd, ld = _to(cuda, q, k, v, g, lengths)
        code = la.LA_F32 if dt == "f32" else la.LA_BF16
        out, dq, dk, dv = (torch.full_like(x, nan) for x in (vd, qd, kd, vd))
        den = torch.full((B, H, N), nan, device=cuda)
        S = torch.full((B, H, D, M), nan, device=cuda)
        Z = torch.full((B, H, D), nan, device=cuda)
        la.la_noncausal_fwd(qd, kd, vd, ld, out, den, S, Z, None, B, H, N, D, M, code)
        la.la_noncausal_bwd(qd, kd, vd, ld, out, den, S, Z, gd, dq, dk, dv, None, B, H, N, D, M,
                            code)
        torch.cuda.synchronize()
        for name, t in (("out", out), ("den", den), ("S", S), ("Z", Z), ("dq", dq), ("dk", dk),
                        ("dv", dv)):
            assert torch.isfinite(t.float()).all(), f"non-causal {B}x{H}x{N} {dt} seed {seed}: {name}"
    for B, H, N, D, M, dt in [(2, 3, 1000, 64, 64, "bf16"), (1, 2, 333, 64, 32, "f32"),
                              (4, 8, 3072, 64, 64, "bf16"), (3, 1, 129, 16, 64, "f32")]:
        q, k, v, g = causal_inputs(B, H, N, D, M, dt, 6000 + N)
        qd, kd, vd, gd = _to(cuda, q, k, v, g)
        code = la.LA_F32 if dt == "f32" else la.LA_BF16
        out, dq, dk, dv = (torch.full_like(x, nan) for x in (vd, qd, kd, vd))
        den = torch.full((B, H, N), nan, device=cuda)
        wf = la.workspace(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, code, cuda)
        wb = la.workspace(la.LA_OP_CAUSAL_BWD, B, H, N, D, M, code, cuda)
        la.la_causal_fwd(qd, kd, vd, out, den, wf, B, H, N, D, M, code)
        la.la_causal_bwd(qd, kd, vd, out, den, gd, dq, dk, dv, wb, B, H, N, D, M, code)
        torch.cuda.synchronize()
        for name, t in (("out", out), ("den", den), ("dq", dq), ("dk", dk), ("dv", dv)):
            assert torch.isfinite(t.float()).all(), f"causal {B}x{H}x{N} {dt}: {name}"
        # the same inputs through the prefill (from a finite state) and one decode step
        S0 = torch.rand(B, H, D, M, device=cuda)
        Z0 = torch.rand(B, H, D, device=cuda) + 1.0
        wp = la.workspace(la.LA_OP_CAUSAL_PREFILL, B, H, N, D, M, code, cuda)
        out.fill_(nan)
        den.fill_(nan)
        la.la_causal_prefill(qd, kd, vd, out, den, S0, Z0, wp, B, H, N, D, M, code)
        y = torch.full_like(vd[:, :, 0], nan)
        la.la_decode_step(qd[:, :, 0].contiguous(), kd[:, :, 0].contiguous(), vd[:, :, 0].contiguous(),
                          S0, Z0, y, B, H, D, M, code)
        torch.cuda.synchronize()
        for name, t in (("prefill out", out), ("prefill den", den), ("S_N", S0), ("Z_N", Z0),
                        ("decode y", y)):
            assert torch.isfinite(t.float()).all(), f"causal {B}x{H}x{N} {dt}: {name}"
    la.check_device_status()


@pytest.mark.parametrize("D,M,dtype", [(64, 64, "bf16"), (32, 64, "f32")])
def test_den_is_optional(cuda, linattn, D, M, dtype):
    """den may be NULL for the causal forward, the prefill and the non-causal
    forward: the other outputs are the same bits as with den."""
    la = linattn
    B, H, N = 2, 3, 700
    q, k, v, _ = causal_inputs(B, H, N, D, M, dtype, 8800)
    qd, kd, vd = _to(cuda, q, k, v)
    code = la.LA_F32 if dtype == "f32" else la.LA_BF16
    ws = la.workspace(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, code, cuda)
    o1, o2 = torch.empty_like(vd), torch.empty_like(vd)
    den = torch.empty(B, H, N, device=cuda)
    la.la_causal_fwd(qd, kd, vd, o1, den, ws, B, H, N, D, M, code)
    la.la_causal_fwd(qd, kd, vd, o2, None, ws, B, H, N, D, M, code)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    wp = la.workspace(la.LA_OP_CAUSAL_PREFILL, B, H, N, D, M, code, cuda)
    S1, Z1 = torch.rand(B, H, D, M, device=cuda), torch.rand(B, H, D, device=cuda) + 1.0
    S2, Z2 = S1.clone(), Z1.clone()
    la.la_causal_prefill(qd, kd, vd, o1, den, S1, Z1, wp, B, H, N, D, M, code)
    la.la_causal_prefill(qd, kd, vd, o2, None, S2, Z2, wp, B, H, N, D, M, code)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2) and torch.equal(Z1, Z2)
    if D == M:
        wn = la.workspace(la.LA_OP_NONCAUSAL_FWD, B, H, N, D, M, code, cuda)
        Sa, Za = torch.empty(B, H, D, M, device=cuda), torch.empty(B, H, D, device=cuda)
        Sb, Zb = torch.empty_like(Sa), torch.empty_like(Za)
        la.la_noncausal_fwd(qd, kd, vd, None, o1, den, Sa, Za, wn, B, H, N, D, M, code)
        la.la_noncausal_fwd(qd, kd, vd, None, o2, None, Sb, Zb, wn, B, H, N, D, M, code)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(Sa, Sb) and torch.equal(Za, Zb)


def run_decode(la, dev, B, H, D, M, dtype, seed, T, sample_heads=None, chunk=64):
    """Runs T steps on the GPU; checks y_t for every step and the final
    state against the oracle on a sample of heads (all heads if None)."""
    stream = DecodeStream(B, H, D, M, dtype, seed)
    S = torch.zeros(B, H, D, M, dtype=torch.float32, device=dev)
    Z = torch.zeros(B, H, D, dtype=torch.float32, device=dev)
    flat = lambda t: t.reshape(t.shape[0], B * H, -1)
    heads = np.arange(B * H) if sample_heads is None else np.asarray(sample_heads)
    S_ref = np.zeros((1, len(heads), D, M))
    Z_ref = np.zeros((1, len(heads), D))
    worst = 0.0
    for t0 in range(0, T, chunk):
        n = min(chunk, T - t0)
        qs, ks, vs = stream.steps(n)
        ys = []
        for t in range(n):
            qd, kd, vd = _to(dev, qs[t], ks[t], vs[t])
            ys.append(la.decode_step(qd, kd, vd, S, Z))
        y = torch.stack(ys)
        qh, kh, vh = (flat(x)[:, heads][:, None] for x in (qs, ks, vs))
        y_ref, S_ref, Z_ref = oracle.decode(qh, kh, vh, S_ref, Z_ref)
        worst = max(worst, rel_err(flat(y)[:, heads][:, None], y_ref))
    s_err = rel_err(S.reshape(B * H, D, M)[heads][None], S_ref)
    z_err = rel_err(Z.reshape(B * H, D)[heads][None], Z_ref)
    return worst, s_err, z_err


@pytest.mark.parametrize("B,H,D,M,dtype,T", [
    (2, 3, 16, 16, "f32", 40), (1, 4, 64, 32, "f32", 70), (3, 1, 32, 64, "bf16", 33),
    (2, 2, 64, 64, "f32", 130)])
def test_decode_small(cuda, linattn, B, H, D, M, dtype, T):
    y_err, s_err, z_err = run_decode(linattn, cuda, B, H, D, M, dtype, 3000 + T, T)
    tol = TOL[dtype]
    assert y_err <= tol and s_err <= 1e-4 and z_err <= 1e-4, (y_err, s_err, z_err)


def test_decode_matches_causal(cuda, linattn):
    """T decode steps reproduce the causal forward on the stacked sequence."""
    B, H, D, M, T = 2, 2, 64, 64, 200
    q, k, v, _ = causal_inputs(B, H, T, D, M, "f32", 77)
    out, _ = linattn.causal_fwd(*_to(cuda, q, k, v))
    S = torch.zeros(B, H, D, M, device=cuda)
    Z = torch.zeros(B, H, D, device=cuda)
    ys = [linattn.decode_step(*_to(cuda, q[:, :, t], k[:, :, t], v[:, :, t]), S, Z) for t in range(T)]
    y = torch.stack(ys, dim=2)
    assert rel_err(y, out.double().cpu().numpy()) < 1e-5


def test_decode_workload(cuda, linattn):
    """256 streams x 8 heads, 3072 steps; every step's y and the final S, Z on
    64 sampled heads against the oracle."""
    w = WORKLOADS["decode_f32"]
    heads = np.random.default_rng(0).choice(w.B * w.H, size=64, replace=False)
    y_err, s_err, z_err = run_decode(linattn, cuda, w.B, w.H, w.D, w.M, w.dtype, w.seed, w.N,
                                     sample_heads=np.sort(heads), chunk=256)
    print(w.name, y_err, s_err, z_err)
    assert y_err <= 1e-4 and s_err <= 1e-4 and z_err <= 1e-4, (y_err, s_err, z_err)
