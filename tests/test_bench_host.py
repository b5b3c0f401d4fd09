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



def _fake_smi(tmp_path, line):
    """A stand-in `nvidia-smi` on PATH that prints one CSV sample line every 20 ms."""
    d = tmp_path / "bin"
    d.mkdir()
    exe = d / "nvidia-smi"
    exe.write_text(f"#!{sys.executable}\nimport sys, time\n"
                   f"while True:\n    print({line!r}, flush=True)\n    time.sleep(0.02)\n")
    exe.chmod(0o755)
    return str(d)


@pytest.mark.parametrize("line,reasons", [
    ("0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active", ["sw_power_cap"]),
    ("0, 1500, 2070, 1390.0, 0x8, Active, Not Active, Not Active, Not Active", ["hw_slowdown"]),
])
def test_clock_sampler_waits_for_its_first_sample_and_reads_reasons(tmp_path, monkeypatch, line, reasons):
    import time
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, line) + os.pathsep + os.environ.get("PATH", ""))
    path = str(tmp_path / "clk.csv")
    c = bench.ClockSampler(0, path)
    c.wait_running(limit_s=10)
    assert os.path.getsize(path) > 0  # the timed region starts only once a sample is in
    time.sleep(0.1)
    r = c.stop()
    assert r["samples"] >= 1
    assert r["sm_max_mhz"] == 2070.0
    assert r["sm_mhz"] == float(line.split(",")[1])
    assert r["reasons"] == reasons


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # nothing named nvidia-smi there
    c = bench.ClockSampler(0, str(tmp_path / "clk.csv"))
    c.wait_running(limit_s=1)
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]
