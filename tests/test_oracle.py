"""The fp64 oracle against what the pages and the mathematics fix (no GPU).

See tests/oracle_pins.py for what each pin compares against."""
import numpy as np
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_threads_do_not_change_results(orc):
    """OpenMP over heads must not change any value (heads are independent)."""
    q, k = P.rand((2, 3, 40, 8), 1), P.rand((2, 3, 40, 8), 2)
    v, g = P.rand((2, 3, 40, 6), 3), P.rand((2, 3, 40, 6), 4)
    a = orc.causal_bwd(q, k, v, g, "recurrent", nthreads=1)
    b = orc.causal_bwd(q, k, v, g, "recurrent", nthreads=4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    S0, Z0 = P.rand((2, 3, 8, 6), 5), 1.0 + np.abs(P.rand((2, 3, 8), 6))
    a = orc.causal_prefill(q, k, v, S0, Z0, nthreads=1)
    b = orc.causal_prefill(q, k, v, S0, Z0, nthreads=4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_fd_at_tiny_workload_size(orc):
    """Gradients at the size of the smallest parity workload (N=64, D=M=16)
    against finite differences on a sample of entries."""
    from kernelized_causal_attention_gb300.workloads import causal_inputs
    q, k, v, g = (t.double().numpy() for t in causal_inputs(1, 1, 64, 16, 16, "f32", 1))
    dq, dk, dv = orc.causal_bwd(q, k, v, g)
    rng = np.random.default_rng(0)
    h = 1e-6
    for x, dx in ((q, dq), (k, dk), (v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)
            x0 = x[idx]
            x[idx] = x0 + h
            lp = float(np.sum(g * orc.causal_fwd(q, k, v)[0]))
            x[idx] = x0 - h
            lm = float(np.sum(g * orc.causal_fwd(q, k, v)[0]))
            x[idx] = x0
            fd = (lp - lm) / (2 * h)
            assert abs(fd - dx[idx]) <= 1e-6 * max(1.0, np.max(np.abs(dx)))


def test_golden_regression(orc):
    """The oracle still reproduces its committed regression record
    (tests/golden/causal_tiny_f32.json, written by tests/golden/make_golden.py)."""
    import json
    import os
    from kernelized_causal_attention_gb300.workloads import causal_inputs
    rec = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "causal_tiny_f32.json")))
    B, H, N, D, M = rec["shape"]
    q, k, v, g = causal_inputs(B, H, N, D, M, "f32", rec["seed"])
    out, den = orc.causal_fwd(q, k, v)
    dq, dk, dv = orc.causal_bwd(q, k, v, g)
    rows = rec["rows"]
    for name, arr in (("out", out), ("den", den), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert np.allclose(arr[0, 0, rows], np.array(rec[name]), rtol=1e-12, atol=1e-13), name
