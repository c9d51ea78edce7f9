"""Device-side failure reporting: a bounded wait inside a kernel that runs out
reaches the host as LA_ERR_TIMEOUT through the library's status word, and the
CUDA context stays usable.  The wait is made to run out on purpose only by
the diagnostic kernel, whose barrier nothing arrives at; no kernel is made
to fault or hang."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_survives(cuda, linattn):
    la = linattn
    la.la_device_status(clear=True)  # whatever earlier tests left
    assert la.la_device_status(clear=False) == (la.LA_OK, 0)

    la.la_selftest_wait(2_000_000)  # 2 ms
    assert la.la_device_status(clear=False) == (la.LA_ERR_TIMEOUT, 99)
    # the word sticks until it is cleared
    assert la.la_device_status(clear=True) == (la.LA_ERR_TIMEOUT, 99)
    assert la.la_device_status(clear=False) == (la.LA_OK, 0)

    # the same context still computes: constant V comes back as V from the
    # tensor-core causal and non-causal paths (weights that sum to one)
    g = torch.Generator().manual_seed(7)
    q = torch.randn(1, 2, 300, 64, generator=g).to(cuda, torch.bfloat16)
    k = torch.randn(1, 2, 300, 64, generator=g).to(cuda, torch.bfloat16)
    v = torch.full((1, 2, 300, 64), 0.5, device=cuda, dtype=torch.bfloat16)
    out, den = la.causal_fwd(q, k, v)
    assert torch.all(den > 0)
    assert torch.allclose(out.float(), v.float(), atol=1e-2)
    out, den, S, Z = la.noncausal_fwd(q.float(), k.float(), v.float())
    assert torch.allclose(out, v.float(), rtol=1e-5, atol=1e-6)
    assert la.la_device_status(clear=False) == (la.LA_OK, 0)

    # the raising form
    la.la_selftest_wait(1_000_000)
    with pytest.raises(la.LinAttnError) as e:
        la.check_device_status()
    assert e.value.code == la.LA_ERR_TIMEOUT
    la.check_device_status()  # cleared by the call above


def test_compute_calls_leave_the_status_clear(cuda, linattn):
    la = linattn
    la.la_device_status(clear=True)
    g = torch.Generator().manual_seed(11)
    q, k, v, do = (torch.randn(2, 4, 1000, 64, generator=g).to(cuda, torch.bfloat16) for _ in range(4))
    out, den = la.causal_fwd(q, k, v)
    la.causal_bwd(q, k, v, out, den, do)
    lengths = torch.tensor([1000, 17], dtype=torch.int32, device=cuda)
    out, den, S, Z = la.noncausal_fwd(q.float(), k.float(), v.float(), lengths)
    la.noncausal_bwd(q.float(), k.float(), v.float(), lengths, out, den, S, Z, do.float())
    la.check_device_status()
