"""Test-side access to the GPU step runner plus the element-wise tolerance check."""
import numpy as np

from paged_kv_cache_134_gb300.runner import (TORCH_DT, DecodeInputs, decode_step, dev, fill_cache,  # noqa: F401
                                             new_cache, pool_numpy, run_decode, run_prefill)


def assert_close(gpu, ref, atol, rtol, what=""):
    """Pass iff every element has |gpu - ref| <= atol + rtol * |ref|; returns (max abs, max rel)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    big = np.abs(ref) >= 0.1
    rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max abs {err.max():.3e}, max rel (|ref|>=0.1) {rel:.3e}")
    return float(err.max()), rel
