"""The C ABI on the host: the library loads, exports every symbol that
include/linattn.h declares, sizes workspaces, and rejects bad arguments before
launching anything (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_symbols()
    for n in ("la_causal_fwd", "la_causal_bwd", "la_noncausal_fwd", "la_noncausal_bwd",
              "la_decode_step", "la_causal_prefill", "la_workspace_bytes", "la_status_string",
              "la_version", "la_device_status", "la_selftest_wait"):
        assert n in names


def test_library_exports_every_declared_symbol(linattn):
    h = ctypes.CDLL(linattn.library_path())
    for name in declared_symbols():
        assert hasattr(h, name), f"{name} declared in linattn.h but not exported"
    assert set(declared_symbols()) <= set(linattn.EXPORTED) | {"la_workspace_bytes"}


def header_constants():
    """name -> value of every LA_* constant the header's enums define."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", text, flags=re.S):
        for name, val in re.findall(r"(LA_\w+)\s*=\s*(\d+)", body):
            out[name] = int(val)
    return out


def test_status_and_dtype_values_match_the_header(linattn):
    """The fixed numbering (LA_ERR_TIMEOUT = 4, LA_ERR_WORKSPACE = 5; LA_F32 = 0,
    LA_BF16 = 1) is what the header states and what the binding uses."""
    h = header_constants()
    want = {"LA_OK": 0, "LA_ERR_INVALID_ARG": 1, "LA_ERR_UNSUPPORTED": 2, "LA_ERR_CUDA": 3,
            "LA_ERR_TIMEOUT": 4, "LA_ERR_WORKSPACE": 5, "LA_F32": 0, "LA_BF16": 1}
    for name, val in want.items():
        assert h[name] == val, name
        assert getattr(linattn, name) == val, name
    text = open(HEADER).read()
    assert re.search(r"typedef\s+int\s+la_status\s*;", text)
    assert re.search(r"typedef\s+int\s+la_dtype\s*;", text)
    assert linattn.status_string(4) == "a bounded wait inside a kernel ran out"
    assert linattn.status_string(5) == "workspace missing or too small"


def test_version_and_status_strings(linattn):
    assert linattn.lib().la_version() == 200
    for code in range(6):
        assert linattn.status_string(code) != "unknown status"
    assert linattn.status_string(99) == "unknown status"


def test_selftest_wait_rejects_limits_before_launching(linattn):
    # checked on the host: no GPU is touched for a limit outside 1 ns .. 1 s
    for limit in (0, 1_000_000_001, 1 << 63):
        assert linattn.lib().la_selftest_wait(None, limit) == linattn.LA_ERR_INVALID_ARG


def test_workspace_sizes(linattn):
    la = linattn
    # one segment per sequence needs no workspace for the causal path
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD, 1, 1, 64, 16, 16, la.LA_F32) == 0
    n = la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD, 4, 8, 3072, 64, 64, la.LA_BF16)
    assert n > 0 and n % 16 == 0
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL_BWD, 4, 8, 3072, 64, 64, la.LA_BF16) > 0
    assert la.la_workspace_bytes(la.LA_OP_DECODE, 256, 8, 1, 64, 64, la.LA_F32) == 0
    # the non-causal path for D = M = 64 reduces its partial states within a
    # cluster and needs none (either dtype); other head sizes need some
    for dt in (la.LA_F32, la.LA_BF16):
        assert la.la_workspace_bytes(la.LA_OP_NONCAUSAL_FWD, 16, 6, 2048, 64, 64, dt) == 0
        assert la.la_workspace_bytes(la.LA_OP_NONCAUSAL_BWD, 16, 6, 2048, 64, 64, dt) == 0
    assert la.la_workspace_bytes(la.LA_OP_NONCAUSAL_BWD, 16, 6, 2048, 32, 64, la.LA_F32) > 0
    # the forward from a state keeps every segment's sums (and the CUDA-core
    # path one more record), so it always needs a workspace
    for shape in ((4, 8, 3072, 64, 64, la.LA_BF16), (1, 1, 64, 16, 16, la.LA_F32),
                  (1, 1, 1, 64, 64, la.LA_BF16)):
        assert la.la_workspace_bytes(la.LA_OP_CAUSAL_PREFILL, *shape) > 0
    assert la.la_kernel_launches(la.LA_OP_CAUSAL_PREFILL, 4, 8, 3072, 64, 64, la.LA_BF16) == 3
    assert la.la_kernel_launches(la.LA_OP_CAUSAL_PREFILL, 4, 8, 3072, 64, 64, la.LA_F32) == 4
    # invalid arguments size to 0
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD, 0, 8, 3072, 64, 64, la.LA_BF16) == 0
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL_FWD, 1, 8, 3072, 48, 64, la.LA_BF16) == 0


FAKE = 1 << 20  # an aligned, never-dereferenced address: every call below fails its checks first


def _fwd(la, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, den=FAKE, ws=None, wsb=0, B=1, H=1, N=64, D=16, M=16,
             dt=la.LA_F32)
    a.update(kw)
    return la.lib().la_causal_fwd(a["q"], a["k"], a["v"], a["out"], a["den"], a["ws"], a["wsb"],
                                  a["B"], a["H"], a["N"], a["D"], a["M"], a["dt"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(out=None), 1),
    (dict(q=FAKE + 4), 1), (dict(den=FAKE + 8), 1),
    (dict(N=0), 1), (dict(B=0), 1), (dict(H=-1), 1), (dict(N=(1 << 24) + 1), 1),
    (dict(dt=7), 1), (dict(D=48), 2), (dict(M=128), 2), (dict(D=0), 1),
    (dict(B=65536), 1), (dict(B=256, H=256), 1),     # B*H above the 65535 grid rows
    (dict(B=4, H=8, N=3072, D=64, M=64), 5),          # needs workspace, none given
    (dict(B=4, H=8, N=3072, D=64, M=64, ws=FAKE, wsb=16), 5),
    (dict(B=4, H=8, N=3072, D=64, M=64, ws=FAKE + 4, wsb=1 << 30), 1),
])
def test_causal_fwd_rejects(linattn, kw, code):
    assert _fwd(linattn, **kw) == code


def test_other_calls_reject(linattn):
    L = linattn.lib()
    F = FAKE
    # causal bwd: den is required
    assert L.la_causal_bwd(F, F, F, F, None, F, F, F, F, None, 0, 1, 1, 64, 16, 16, 0, None) == 1
    # non-causal: S and Z required, lengths optional but aligned
    assert L.la_noncausal_fwd(F, F, F, None, F, F, None, F, F, 1 << 30, 1, 1, 64, 16, 16, 0, None) == 1
    assert L.la_noncausal_fwd(F, F, F, F + 4, F, F, F, F, F, 1 << 30, 1, 1, 64, 16, 16, 0, None) == 1
    assert L.la_noncausal_fwd(F, F, F, None, F, F, F, F, None, 0, 1, 1, 64, 16, 16, 0, None) == 5
    assert L.la_noncausal_bwd(F, F, F, None, F, F, F, F, F, F, F, None, F, 1 << 30, 1, 1, 64, 16,
                              16, 0, None) == 1
    # decode
    assert L.la_decode_step(F, F, None, F, F, F, 1, 1, 64, 64, 0, None) == 1
    assert L.la_decode_step(F, F, F, F, F, F, 1, 1, 64, 96, 0, None) == 2
    assert L.la_decode_step(F, F, F, F, F, F, 0, 1, 64, 64, 0, None) == 1
    assert L.la_decode_step(F, F, F, F, F, F, (1 << 20) + 1, 1, 64, 64, 0, None) == 1


def test_prefill_rejects(linattn):
    la = linattn
    call = lambda S, Z, ws=None, wsb=0, N=64: la.lib().la_causal_prefill(
        FAKE, FAKE, FAKE, FAKE, None, S, Z, ws, wsb, 1, 1, N, 16, 16, la.LA_F32, None)
    assert call(None, FAKE) == la.LA_ERR_INVALID_ARG      # the state is required
    assert call(FAKE, None) == la.LA_ERR_INVALID_ARG
    assert call(FAKE + 4, FAKE) == la.LA_ERR_INVALID_ARG  # misaligned
    assert call(FAKE, FAKE) == la.LA_ERR_WORKSPACE        # needs a workspace
    assert call(FAKE, FAKE, N=0) == la.LA_ERR_INVALID_ARG


def test_head_count_limits(linattn):
    """B*H limits: 65535 for the sequence calls, 2^20 streams for decode
    (sizes only: nothing is launched)."""
    la = linattn
    for op in (la.LA_OP_CAUSAL_FWD, la.LA_OP_CAUSAL_BWD, la.LA_OP_NONCAUSAL_FWD,
               la.LA_OP_NONCAUSAL_BWD):
        assert la.la_kernel_launches(op, 65535, 1, 64, 16, 16, la.LA_F32) > 0
        assert la.la_kernel_launches(op, 65536, 1, 64, 16, 16, la.LA_F32) == 0
        assert la.la_workspace_bytes(op, 65536, 1, 64, 16, 16, la.LA_F32) == 0
    assert la.la_kernel_launches(la.LA_OP_DECODE, 1 << 20, 1, 1, 64, 64, la.LA_F32) == 1
    assert la.la_kernel_launches(la.LA_OP_DECODE, (1 << 20) + 1, 1, 1, 64, 64, la.LA_F32) == 0


def test_binding_requires_library(monkeypatch, tmp_path):
    """Without the built library the binding raises instead of falling back."""
    import kernelized_causal_attention_gb300 as la
    monkeypatch.setattr(la, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(la, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        la.lib()


def test_binding_refuses_host_tensors(linattn):
    """The binding passes device pointers only: a CPU tensor is refused before
    anything reaches the library (no GPU needed)."""
    import torch
    q = torch.zeros(1, 1, 64, 16)
    with pytest.raises(ValueError, match="CUDA device"):
        linattn.la_causal_fwd(q, q, q, q, None, None, 1, 1, 64, 16, 16, linattn.LA_F32)
    with pytest.raises(ValueError, match="CUDA device"):
        linattn.la_decode_step(q[0, 0, 0], q[0, 0, 0], q[0, 0, 0], q, q, q, 1, 1, 16, 16, linattn.LA_F32)


def test_kernel_launch_counts(linattn):
    """The launch accounting behind bench.py's gpu_launches, per path."""
    la = linattn
    n = la.la_kernel_launches
    # causal, tensor cores: a state pass only when a head has several segments
    assert n(la.LA_OP_CAUSAL_FWD, 4, 8, 3072, 64, 64, la.LA_BF16) == 2
    assert n(la.LA_OP_CAUSAL_FWD, 1, 160, 3072, 64, 64, la.LA_BF16) == 1   # one segment per head
    assert n(la.LA_OP_CAUSAL_BWD, 4, 8, 3072, 64, 64, la.LA_BF16) == 2
    # causal, CUDA cores: partial sums + scan + main with several segments
    assert n(la.LA_OP_CAUSAL_FWD, 1, 1, 4096, 64, 64, la.LA_F32) == 3
    assert n(la.LA_OP_CAUSAL_FWD, 1, 1, 64, 16, 16, la.LA_F32) == 1
    # non-causal: one launch per direction on the tensor cores
    for dt in (la.LA_F32, la.LA_BF16):
        assert n(la.LA_OP_NONCAUSAL_FWD, 16, 6, 2048, 64, 64, dt) == 1
        assert n(la.LA_OP_NONCAUSAL_BWD, 16, 6, 2048, 64, 64, dt) == 1
    assert n(la.LA_OP_DECODE, 256, 8, 1, 64, 64, la.LA_F32) == 1
    # invalid sizes count no launches
    assert n(la.LA_OP_CAUSAL_FWD, 0, 8, 3072, 64, 64, la.LA_BF16) == 0
