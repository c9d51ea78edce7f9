"""bench.py's JSON line on the CPU: the reference arm (the fp64 oracle timed on
the host cores) prints one complete line, and our arm without a GPU fails
loudly instead of printing a number (there is no CPU fallback)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, env=None):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=600, env=env)


def test_reference_arm_prints_one_complete_line():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == "causal_cifar_bf16"
    assert d["config"]["N"] == 3072 and d["config"]["D"] == 64
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert abs(d["ms_per_step"] * 1e-3 * d["value"] - 4 * 3072) / (4 * 3072) < 1e-3


def test_our_arm_without_a_gpu_fails_loudly():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = _run("--steps", "1", "--warmup", "3", "--no-secondary", "--no-cpu", env=env)
    assert r.returncode != 0
    assert r.stdout.strip() == ""


def _bench():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    return bench


def test_algorithmic_bytes_per_token_head():
    """Every input read once, every output written once: bf16, D = M = 64 gives
    516 B (fwd: q, k, v, out, den) and 1028 B (bwd: q, k, v, out, dout, den,
    dq, dk, dv) per token-head."""
    fwd, bwd = _bench().causal_bytes(4, 8, 3072, 64, 64, 2)
    th = 4 * 8 * 3072
    assert fwd == 516 * th and bwd == 1028 * th


def test_stored_traffic_only_for_the_sources_it_was_taken_on(monkeypatch):
    b = _bench()
    stored = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    monkeypatch.setattr(b, "kernel_source_hash", lambda: stored["source_hash"])
    assert b.stored_traffic("la_causal_bwd") == stored["per_call_dram_bytes"]["la_causal_bwd"]
    monkeypatch.setattr(b, "kernel_source_hash", lambda: "0000000000000000")
    assert b.stored_traffic("la_causal_bwd") is None


def test_fp32_algorithmic_bytes_per_token_head():
    """fp32 inputs and outputs, D = M = 64: 1028 B forward and 2052 B backward
    per token-head (the same tensors at four bytes an element)."""
    fwd, bwd = _bench().causal_bytes(4, 8, 3072, 64, 64, 4)
    th = 4 * 8 * 3072
    assert fwd == 1028 * th and bwd == 2052 * th


class _FakeCuda:
    """A device clock for time_calls on the CPU: a call advances it by its
    cost; an event records the clock when the 'stream' reaches it."""

    def __init__(self):
        self.t = 0.0

    def make_torch(self):
        clock = self

        class FakeEvent:
            def __init__(self, enable_timing=False):
                self.at = None

            def record(self, stream=None):
                self.at = clock.t

            def elapsed_time(self, other):
                return other.at - self.at

        class Cuda:
            Event = FakeEvent

            @staticmethod
            def synchronize():
                pass

            @staticmethod
            def _sleep(cycles):
                pass

        class Torch:
            cuda = Cuda

        return Torch


def test_time_calls_with_and_without_events_between_calls():
    b = _bench()
    fake = _FakeCuda()
    torch = fake.make_torch()

    def call(ms):
        def f():
            fake.t += ms
        return f

    fns = [call(0.25), call(0.5)]
    per_call, step = b.time_calls(fns, 4, lambda: None, torch, None, None)
    assert per_call == [0.25, 0.5] and abs(step - 0.75) < 1e-12
    none, step2, median = b.time_calls(fns, 4, lambda: None, torch, None, None, with_median=True,
                                       split=False)
    assert none is None and abs(step2 - 0.75) < 1e-12 and abs(median - 0.75) < 1e-12
    per_call3, step3 = b.step_and_calls(fns, 3, lambda: None, torch, None)
    assert per_call3 == [0.25, 0.5] and abs(step3 - 0.75) < 1e-12
