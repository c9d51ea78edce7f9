"""la_causal_fwd_noalloc: the causal forward for callers that may not allocate
device memory (plug-ins inside an application that owns all GPU memory, or
loops where a cudaMalloc and the device synchronisation it can cause are not
allowed).  It takes its scratch from an array built into the library.

Checked through the C ABI against la_causal_fwd (caller-provided workspace) on
two calls in a row, so that the second call starts from the first call's
leftovers in the shared scratch array.  Both calls run the same kernels on the
same inputs, and those kernels are deterministic, so the outputs must be equal
bit for bit.  This file is collected last on purpose.
"""
import pytest
import torch

from kernelized_causal_attention_gb300.workloads import causal_inputs

LIMIT = 4 << 20  # LA_NOALLOC_SCRATCH_BYTES in include/linattn.h


def _reference(la, q, k, v, B, H, N, D, M, dt):
    out = torch.empty(B, H, N, M, dtype=q.dtype, device=q.device)
    den = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    ws = la.workspace(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, dt, q.device)
    la.la_causal_fwd(q, k, v, out, den, ws, B, H, N, D, M, dt)
    return out, den


def _largest_fitting_shape(la):
    """A bf16 D = M = 64 shape whose forward workspace is as close to the
    scratch size as the candidates allow, without exceeding it."""
    best = None
    for H in (1, 2, 3, 4, 6, 8, 12, 16, 24, 32):
        for N in range(128, 1 << 16, 128):
            n = la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD, 1, H, N, 64, 64, la.LA_BF16)
            if n > LIMIT:
                break
            if best is None or n > best[0]:
                best = (n, (1, H, N, 64, 64, "bf16"))
    return best


def _run_pair(la, cuda, B, H, N, D, M, dtype):
    dt = la.LA_BF16 if dtype == "bf16" else la.LA_F32
    assert 0 < la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, dt) <= LIMIT
    for call, seed in enumerate((11, 12)):  # two calls in a row on the shared scratch
        q, k, v, _ = (t.to(cuda) for t in causal_inputs(B, H, N, D, M, dtype, seed))
        out_ref, den_ref = _reference(la, q, k, v, B, H, N, D, M, dt)
        out = torch.full_like(out_ref, float("nan"))
        den = torch.full_like(den_ref, float("nan"))
        la.la_causal_fwd_noalloc(q, k, v, out, den, B, H, N, D, M, dt)
        torch.cuda.synchronize()
        assert torch.equal(out, out_ref), f"call {call}: out differs"
        assert torch.equal(den, den_ref), f"call {call}: den differs"


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,D,M,dtype", [
    (4, 8, 3072, 64, 64, "bf16"),   # tensor-core path, several segments per head
    (2, 3, 777, 32, 64, "f32"),     # CUDA-core path, fp32
    (2, 4, 1000, 32, 32, "bf16"),   # bf16 with D, M below 64
])
def test_noalloc_matches_workspace_entry_point(cuda, linattn, B, H, N, D, M, dtype):
    _run_pair(linattn, cuda, B, H, N, D, M, dtype)


@pytest.mark.gpu
def test_noalloc_at_the_scratch_limit(cuda, linattn):
    """The largest problem of the candidates whose workspace still fits."""
    n, shape = _largest_fitting_shape(linattn)
    assert n > LIMIT // 2
    _run_pair(linattn, cuda, *shape)


@pytest.mark.gpu
def test_noalloc_allocates_nothing(cuda, linattn):
    """After a warm-up call (which may load kernel modules), a call leaves the
    device's free memory and torch's allocator exactly as they were."""
    la = linattn
    B, H, N, D, M = 4, 8, 3072, 64, 64
    q, k, v, _ = (t.to(cuda) for t in causal_inputs(B, H, N, D, M, "bf16", 5))
    out = torch.empty(B, H, N, M, dtype=q.dtype, device=cuda)
    den = torch.empty(B, H, N, dtype=torch.float32, device=cuda)
    la.la_causal_fwd_noalloc(q, k, v, out, den, B, H, N, D, M, la.LA_BF16)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        la.la_causal_fwd_noalloc(q, k, v, out, den, B, H, N, D, M, la.LA_BF16)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0


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


@pytest.mark.parametrize("kw,code", [
    (dict(D=48), "LA_ERR_UNSUPPORTED"), (dict(M=128), "LA_ERR_UNSUPPORTED"),
    (dict(N=0), "LA_ERR_INVALID_ARG"), (dict(q=None), "LA_ERR_INVALID_ARG"),
    (dict(den=(1 << 20) + 8), "LA_ERR_INVALID_ARG"), (dict(dt=7), "LA_ERR_INVALID_ARG"),
])
def test_noalloc_argument_errors_match_the_forward(linattn, kw, code):
    """Bad arguments give the code la_causal_fwd gives, checked before the
    scratch array's address is looked up (so this runs without a GPU)."""
    la = linattn
    fake = 1 << 20
    a = dict(q=fake, k=fake, v=fake, out=fake, den=fake, B=1, H=1, N=64, D=64, M=64, dt=la.LA_BF16)
    a.update(kw)
    rc = la.lib().la_causal_fwd_noalloc(a["q"], a["k"], a["v"], a["out"], a["den"], a["B"], a["H"],
                                        a["N"], a["D"], a["M"], a["dt"], None)
    assert rc == getattr(la, code)
    rc_fwd = la.lib().la_causal_fwd(a["q"], a["k"], a["v"], a["out"], a["den"], None, 0, a["B"],
                                    a["H"], a["N"], a["D"], a["M"], a["dt"], None)
    assert rc_fwd == rc
