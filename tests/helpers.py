"""Shared test helpers: tolerances, error reports and GPU plumbing (no
attention arithmetic)."""
import numpy as np
import pytest

# Per-case error figures recorded by the parity tests, printed at the end of
# the run (tests/conftest.py) and written as JSON when ATTN_PARITY_REPORT names
# a file.
REPORT = []


def require_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA device")
    return torch


def ulp16(ref, mant_bits):
    """One unit in the last place of a 16-bit float at |ref| (bf16: 7 stored
    mantissa bits, fp16: 10), ignoring the subnormal range (far below every
    floor used here)."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ref, 1e-30)))
    return np.exp2(e - mant_bits)


def bf16_atol(ref, floor=1e-2):
    """Per-element bound on a bf16 O: max(floor, one bf16 ulp of the reference).

    Why one ulp: O is returned in bf16, so its own rounding is up to half an
    ulp; and P enters the P.V product rounded to bf16 (unit roundoff 2^-8), so
    a row whose output is carried by one dominant key (the only way |O| gets
    large on these inputs) moves by up to 2^-8 |O| more: half an ulp at the
    bottom of a binade, a full one at its top. On inputs at scale 1/sqrt(d) a
    row's weight is spread and one ulp in all holds with room; steeper scores
    are checked against the exact bound instead (test_parity, steep cases).
    The floor (1e-2 bf16, 6e-2 FP8) is the target's stated bound; it governs
    for |O| < 2 (bf16) and |O| < 8 (FP8)."""
    return np.maximum(floor, ulp16(ref, 7))


def f16_atol(ref, floor=1e-2):
    """Per-element bound on an fp16 O: max(floor, one fp16 ulp of the reference)."""
    return np.maximum(floor, ulp16(ref, 10))


def o_error_stats(o_gpu, o_ref, kind="bf16"):
    """Strict error figures of O against the oracle: the max-abs error, how
    many elements exceed the plain floor (1e-2 bf16 / fp16, 6e-2 FP8) and so
    pass only through the ulp branch of the gate, and the largest error in
    units of the output type's ulp at the reference value."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    err = np.abs(o_gpu - o_ref)
    floor = 6e-2 if kind == "fp8" else 1e-2
    ulp = ulp16(o_ref, 10 if kind == "f16" else 7)
    over = err > floor
    return {
        "o_max_abs": float(err.max()) if err.size else 0.0,
        "o_floor": floor,
        "n_elems": int(err.size),
        "n_over_floor": int(over.sum()),
        # worst error over the elements past the floor, in ulps of the output
        # type at the reference value (0 when none is past the floor)
        "max_ulps_over_floor": float((err[over] / ulp[over]).max()) if over.any() else 0.0,
        # largest share of the per-element gate max(floor, ulp) used
        "gate_use": float((err / np.maximum(floor, ulp)).max()) if err.size else 0.0,
        "max_abs_ref": float(np.abs(o_ref).max()) if err.size else 0.0,
    }


def assert_o_close(o_gpu, o_ref, kind="bf16"):
    """Gate: |O_gpu - O_ref| <= max(floor, one ulp of O_ref) per element.
    Returns the strict error figures (o_error_stats)."""
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
    return o_error_stats(o_gpu, o_ref, kind)


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


def record(case, kind, o_stats, lse_err, rows_checked, note=""):
    """Adds one parity case's figures to the end-of-run report."""
    entry = {"case": case, "kind": kind, "lse_max_abs": lse_err, "rows_checked": rows_checked}
    entry.update(o_stats)
    if note:
        entry["note"] = note
    REPORT.append(entry)
    return entry
