"""Host-side logic of bench.py that needs no GPU: the roofline `traffic` figure is taken from a
committed ncu summary only while the kernel source still has the hash recorded there."""
import hashlib
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
bench = pytest.importorskip("bench")


def _write(root, rel, text):
    p = os.path.join(root, rel)
    os.makedirs(os.path.dirname(p), exist_ok=True)
    with open(p, "w") as f:
        f.write(text)
    return p


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    root = str(tmp_path)
    src = _write(root, "pkg/kernel.cuh", "kernel source v1\n")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    _write(root, "profiles/k.md", f"counters-for: pkg/kernel.cuh sha256={digest}\ntraffic_per_launch_bytes: 1234\n")
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench._recorded_traffic("k.md") == 1234
    _write(root, "pkg/kernel.cuh", "kernel source v2\n")  # the kernel changed after the capture
    assert bench._recorded_traffic("k.md") is None
    assert bench._recorded_traffic("missing.md") is None

