"""Test-side access to the GPU step runner plus the element-wise tolerance check."""
import os

import numpy as np

import parity_log

from paged_kv_cache_134_gb300.runner import (TORCH_DT, DecodeInputs, decode_step, dev, fill_cache,  # noqa: F401
                                             new_cache, pool_numpy, run_decode, run_prefill)


def assert_close(gpu, ref, atol, rtol, what="", out_dtype=None):
    """Pass iff every element has |gpu - ref| <= atol + rtol * |ref|; returns (max abs, max rel).

    The case's max abs error and max relative error (over |ref| >= 0.1) are recorded in
    ``parity_log.RECORDS`` together with the output dtype (``out_dtype``: "f16" or "bf16").  fp16
    outputs must also meet both bounds on their own: max abs <= atol and max rel <= rtol.  bf16
    outputs are held to the combined form only: rounding a bf16 output alone moves it by up to
    2^-9 |o| (3.9e-3 at |o| = 2), which a 2e-3 absolute bound cannot hold."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    big = np.abs(ref) >= 0.1
    rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    parity_log.RECORDS.append(dict(test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], case=what,
                                   out_dtype=out_dtype, max_abs=float(err.max()) if err.size else 0.0,
                                   max_rel=rel, atol=atol, rtol=rtol, elements=int(err.size)))
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max abs {err.max():.3e}, max rel (|ref|>=0.1) {rel:.3e}")
    if out_dtype == "f16":
        # fp16 outputs round at <= 2^-11 relative, so they are also held to the two bounds as stated:
        # max abs error <= atol and max relative error <= rtol (over |ref| >= 0.1), separately
        assert err.max() <= atol and rel <= rtol, (f"{what}: fp16 output beyond the literal bounds: max abs "
                                                   f"{err.max():.3e} (<= {atol:g}), max rel {rel:.3e} (<= {rtol:g})")
    return float(err.max()), rel


def OUT_DT(w):
    """Output dtype of a workload ("f16" or "bf16"): its model dtype (decode) or its dtype (prefill)."""
    return getattr(w, "model_dtype", None) or getattr(w, "dtype", None)
