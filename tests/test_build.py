"""The in-tree build's staleness check (no GPU, no compiler): the library is
rebuilt when it is missing, older than a source, or built from a different
set of translation units (an added or removed file)."""
import os
import time

from kernelized_causal_attention_gb300 import _build as b


def _tree(tmp_path, monkeypatch, names=("a.cu", "b.cu")):
    csrc = tmp_path / "csrc"
    lib = tmp_path / "_lib"
    csrc.mkdir()
    lib.mkdir()
    for n in names:
        (csrc / n).write_text("// unit\n")
    (csrc / "k.cuh").write_text("// header\n")
    header = tmp_path / "linattn.h"
    header.write_text("/* abi */\n")
    monkeypatch.setattr(b, "CSRC", str(csrc))
    monkeypatch.setattr(b, "LIB", str(lib / "liblinattn.so"))
    monkeypatch.setattr(b, "MANIFEST", str(lib / "sources.txt"))
    # the inputs: the tree's units and headers and the ABI header
    monkeypatch.setattr(b, "_deps", lambda: b.sources() + [str(csrc / "k.cuh"), str(header)])
    return csrc, lib


def _build_now(lib):
    old = time.time() - 100
    (lib / "liblinattn.so").write_bytes(b"\0")
    (lib / "sources.txt").write_text(b._manifest())
    return old


def test_fresh_build_is_up_to_date(tmp_path, monkeypatch):
    csrc, lib = _tree(tmp_path, monkeypatch)
    assert not b.up_to_date()                      # nothing built yet
    old = _build_now(lib)
    for f in list(csrc.iterdir()) + [tmp_path / "linattn.h"]:
        os.utime(f, (old, old))                    # every input older than the library
    assert b.up_to_date()


def test_a_newer_source_forces_a_rebuild(tmp_path, monkeypatch):
    csrc, lib = _tree(tmp_path, monkeypatch)
    old = _build_now(lib)
    os.utime(lib / "liblinattn.so", (old, old))
    (csrc / "a.cu").write_text("// changed\n")     # newer than the library
    assert not b.up_to_date()


def test_an_added_or_removed_unit_forces_a_rebuild(tmp_path, monkeypatch):
    csrc, lib = _tree(tmp_path, monkeypatch)
    _build_now(lib)
    (csrc / "c.cu").write_text("// new unit\n")
    assert not b.up_to_date()
    (csrc / "c.cu").unlink()
    (csrc / "b.cu").unlink()
    assert not b.up_to_date()
