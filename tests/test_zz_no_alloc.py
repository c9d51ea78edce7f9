"""la_causal_fwd_noalloc: the causal forward for callers that may not allocate
device memory (plug-ins inside an application that owns all GPU memory, or
loops where a cudaMalloc and the device synchronisation it can cause are not
allowed).  It takes its scratch from an array built into the library.

Checked through the C ABI against la_causal_fwd (caller-provided workspace) on
two calls in a row, so that the second call starts from the first call's
leftovers in the shared scratch array.  This file is collected last on
purpose.
"""
import pytest
import torch

from kernelized_causal_attention_gb300.workloads import causal_inputs

LIMIT = 4 << 20  # LA_NOALLOC_SCRATCH_BYTES in include/linattn.h
TOL = {"f32": 1e-4, "bf16": 2e-2}


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


def _reference(la, q, k, v, B, H, N, D, M, dt):
    out = torch.empty(B, H, N, M, dtype=q.dtype, device=q.device)
    den = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    ws = la.workspace(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, dt, q.device)
    la.la_causal_fwd(q, k, v, out, den, ws, B, H, N, D, M, dt)
    return out, den


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,D,M,dtype", [
    (4, 8, 3072, 64, 64, "bf16"),   # tensor-core path, several segments per head
    (2, 3, 777, 32, 64, "f32"),     # CUDA-core path
])
def test_noalloc_matches_workspace_entry_point(cuda, linattn, B, H, N, D, M, dtype):
    la = linattn
    dt = la.LA_BF16 if dtype == "bf16" else la.LA_F32
    assert 0 < la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, dt) <= LIMIT
    for call, seed in enumerate((11, 12)):  # two calls in a row on the shared scratch
        q, k, v, _ = (t.to(cuda) for t in causal_inputs(B, H, N, D, M, dtype, seed))
        out_ref, den_ref = _reference(la, q, k, v, B, H, N, D, M, dt)
        out = torch.full_like(out_ref, float("nan"))
        den = torch.full_like(den_ref, float("nan"))
        la.la_causal_fwd_noalloc(q, k, v, out, den, B, H, N, D, M, dt)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all() and torch.isfinite(den).all()
        assert _rel(out, out_ref) <= TOL[dtype], f"call {call}: out differs"
        assert _rel(den, den_ref) <= TOL[dtype], f"call {call}: den differs"


def test_noalloc_rejects_problems_beyond_the_scratch(linattn):
    """A problem whose workspace exceeds the built-in array is refused before
    anything is launched (so this runs without a GPU)."""
    la = linattn
    B, H, N, D, M = 64, 16, 1 << 16, 64, 64
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, la.LA_BF16) > LIMIT
    fake = 1 << 20
    rc = la.lib().la_causal_fwd_noalloc(fake, fake, fake, fake, fake, B, H, N, D, M, la.LA_BF16,
                                        None)
    assert rc == la.LA_ERR_WORKSPACE
