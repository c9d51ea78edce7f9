"""The library's calls inside a CUDA graph: every call enqueues its kernels on
the caller's stream and does no host-side synchronisation, so fwd + bwd
captured once and replayed give the same bits as the same calls run eagerly
(the kernels are deterministic)."""
import pytest
import torch

from kernelized_causal_attention_gb300.workloads import causal_inputs


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,D,M,dtype", [(2, 4, 3072, 64, 64, "bf16"), (2, 2, 1000, 32, 32, "f32")])
def test_fwd_bwd_in_a_cuda_graph(cuda, linattn, B, H, N, D, M, dtype):
    la = linattn
    dt = la.LA_BF16 if dtype == "bf16" else la.LA_F32
    q, k, v, g = (t.to(cuda) for t in causal_inputs(B, H, N, D, M, dtype, 55))
    out = torch.empty(B, H, N, M, dtype=q.dtype, device=cuda)
    den = torch.empty(B, H, N, device=cuda)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wf = la.workspace(la.LA_OP_CAUSAL_FWD, B, H, N, D, M, dt, cuda)
    wb = la.workspace(la.LA_OP_CAUSAL_BWD, B, H, N, D, M, dt, cuda)

    def step():
        la.la_causal_fwd(q, k, v, out, den, wf, B, H, N, D, M, dt)
        la.la_causal_bwd(q, k, v, out, den, g, dq, dk, dv, wb, B, H, N, D, M, dt)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, den, dq, dk, dv)]
    for t in (out, den, dq, dk, dv):
        t.fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    la.check_device_status()
    for a, b in zip((out, den, dq, dk, dv), eager):
        assert torch.equal(a, b)
