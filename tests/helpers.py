"""Shared test helpers: tolerances and GPU plumbing (no attention arithmetic)."""
import numpy as np
import pytest


def require_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA device")
    return torch


def bf16_atol(ref, floor=1e-2):
    """Per-element bound on O: max(floor, one bf16 ulp of the reference).
    O is written as bf16, so its rounding alone is half an ulp, which exceeds
    1e-2 once |O| >= 4 (and 6e-2 once |O| >= 16, reached with the FP8
    workload's x20 outliers in V)."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ref, 1e-30)))
    return np.maximum(floor, np.exp2(e - 7))


def f16_atol(ref, floor=1e-2):
    """Per-element bound on an fp16 O: max(floor, one fp16 ulp of the reference)."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ref, 1e-30)))
    return np.maximum(floor, np.exp2(e - 10))


def assert_o_close(o_gpu, o_ref, kind="bf16"):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    assert np.isfinite(o_gpu).all(), "non-finite output"
    err = np.abs(o_gpu - o_ref)
    if kind == "f16":
        tol = f16_atol(o_ref)
    else:
        tol = bf16_atol(o_ref, 1e-2 if kind == "bf16" else 6e-2)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def assert_lse_close(l_gpu, l_ref, tol=1e-3):
    l_gpu = np.asarray(l_gpu, dtype=np.float64)
    l_ref = np.asarray(l_ref, dtype=np.float64)
    inf_ref = np.isneginf(l_ref)
    assert (np.isneginf(l_gpu) == inf_ref).all(), "-inf rows differ"
    if (~inf_ref).any():
        err = np.abs(l_gpu[~inf_ref] - l_ref[~inf_ref])
        assert err.max() <= tol, f"LSE max err {err.max():.3e}"
        return float(err.max())
    return 0.0
