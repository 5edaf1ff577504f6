"""CPU oracle for the exact attention forward pass (fp64, plain C + OpenMP).

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers. The CUDA library never imports this
package and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (see its header for the definition it
evaluates and the passages of the FlashAttention-3 deep-dive page it follows);
this module only builds that file with gcc and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_BF16 = 0
DTYPE_E4M3 = 1
DTYPE_F16 = 2
FP8_BLOCK_ROWS = 64


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so beside it (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_f16_decode.restype = ctypes.c_double
        lib.oracle_f16_decode.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_quantize_fp8_e4m3.restype = None
        lib.oracle_quantize_fp8_e4m3.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4
        lib.oracle_rmsnorm_heads.restype = None
        lib.oracle_rmsnorm_heads.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                             ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = ([ctypes.c_void_p] * 4 + [ctypes.c_int] + [ctypes.c_void_p] * 3
                                        + [ctypes.c_int] * 7 + [ctypes.c_double])
        lib.oracle_attn_bwd_sampled.restype = ctypes.c_int
        lib.oracle_attn_bwd_sampled.argtypes = (
            [ctypes.c_void_p] * 4 + [ctypes.c_int] * 8 + [ctypes.c_double]
            + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64]
            + [ctypes.c_void_p] * 3)
        lib.oracle_attn_fwd.restype = ctypes.c_int
        lib.oracle_attn_fwd.argtypes = (
            [ctypes.c_void_p] * 6 + [ctypes.c_int] + [ctypes.c_void_p] * 2
            + [ctypes.c_int] * 7 + [ctypes.c_double] + [ctypes.c_void_p, ctypes.c_int64])
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """fp64 value of each E4M3 code (OCP 'fn' variant, NaN for 0x7F/0xFF)."""
    lib = _load()
    table = np.array([lib.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def f16_decode(bits: np.ndarray) -> np.ndarray:
    """fp64 value of each IEEE binary16 bit pattern (uint16)."""
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.fromiter((lib.oracle_f16_decode(int(b)) for b in flat), dtype=np.float64,
                      count=flat.size)
    return out.reshape(np.shape(bits))


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even, saturating fp32 -> E4M3 code (elementwise)."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float32).ravel()
    out = np.fromiter((lib.oracle_e4m3_encode(float(v)) for v in flat), dtype=np.uint8,
                      count=flat.size)
    return out.reshape(np.shape(x))


def quantize_fp8_e4m3(x: np.ndarray):
    """Block-quantise fp32 x[B, S, H, d] into E4M3 codes plus fp32 scales
    [B, H, ceil(S/64)] (one scale per 64 sequence rows of one head)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    B, S, H, d = x.shape
    nblk = (S + FP8_BLOCK_ROWS - 1) // FP8_BLOCK_ROWS
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty((B, H, nblk), dtype=np.float32)
    _load().oracle_quantize_fp8_e4m3(_ptr(x), _ptr(codes), _ptr(scales), B, S, H, d)
    return codes, scales


def rmsnorm_heads(x, w, eps: float, dtype: str = "bf16"):
    """fp64 RMSNorm across heads of x [..., H, d] (16-bit bits as uint16) with
    weight w [H * d] (same type): every token's H * d values share one RMS.
    Returns fp64 with x's shape."""
    if dtype not in ("bf16", "f16"):
        raise ValueError(f"unknown dtype {dtype!r}")
    x = np.ascontiguousarray(x).view(np.uint16)
    w = np.ascontiguousarray(w).view(np.uint16)
    H, d = x.shape[-2], x.shape[-1]
    if w.size != H * d:
        raise ValueError("w must hold H * d weights")
    T = x.size // (H * d)
    y = np.empty(x.shape, dtype=np.float64)
    _load().oracle_rmsnorm_heads(_ptr(x), _ptr(w), DTYPE_F16 if dtype == "f16" else DTYPE_BF16,
                                 _ptr(y), T, H, d, float(eps))
    return y


def attn_fwd(q, k, v, causal: bool, scale: float, dtype: str = "bf16",
             q_scale=None, k_scale=None, v_scale=None, rows=None):
    """fp64 exact attention forward.

    q: [B, Sq, Hq, d], k/v: [B, Sk, Hkv, d], given as raw bits: uint16 for
    dtype 'bf16' or 'f16' (IEEE half), uint8 E4M3 codes plus fp32 block scales
    for 'e4m3'.
    Returns (o, lse): o fp64 [B, Sq, Hq, d], lse fp64 [B, Hq, Sq]; or, when
    ``rows`` lists flat indices (b*Hq + hq)*Sq + i, o [n, d] and lse [n].
    """
    lib = _load()
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    if dtype == "bf16":
        code = DTYPE_BF16
        want = np.uint16
    elif dtype == "f16":
        code = DTYPE_F16
        want = np.uint16
    elif dtype == "e4m3":
        code = DTYPE_E4M3
        want = np.uint8
    else:
        raise ValueError(f"unknown dtype {dtype!r}")
    q = np.ascontiguousarray(q).view(want)
    k = np.ascontiguousarray(k).view(want)
    v = np.ascontiguousarray(v).view(want)
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must both be [B, Sk, Hkv, d] matching q")
    scales = [None, None, None]
    if code == DTYPE_E4M3:
        scales = [np.ascontiguousarray(s, dtype=np.float32) for s in (q_scale, k_scale, v_scale)]
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        if rows.size and (rows.min() < 0 or rows.max() >= B * Hq * Sq):
            raise ValueError("row index out of range")
        o = np.empty((rows.size, d), dtype=np.float64)
        lse = np.empty(rows.size, dtype=np.float64)
    else:
        o = np.empty((B, Sq, Hq, d), dtype=np.float64)
        lse = np.empty((B, Hq, Sq), dtype=np.float64)
    rc = lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), *[_ptr(s) for s in scales], code,
                             _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk, d, int(bool(causal)),
                             float(scale), _ptr(rows), 0 if rows is None else rows.size)
    if rc != 0:
        raise ValueError("oracle rejected the dimensions")
    return o, lse


def attn_bwd(q, k, v, d_o, causal: bool, scale: float, dtype: str = "bf16"):
    """fp64 gradients (dq, dk, dv) of sum(d_o * O) for O = attn_fwd(q, k, v);
    q, d_o: [B, Sq, Hq, d], k, v: [B, Sk, Hkv, d], 16-bit bits (bf16 or f16)."""
    lib = _load()
    if dtype not in ("bf16", "f16"):
        raise ValueError(f"unknown dtype {dtype!r}")
    q, k, v, d_o = (np.ascontiguousarray(x).view(np.uint16) for x in (q, k, v, d_o))
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    dq = np.empty(q.shape, dtype=np.float64)
    dk = np.empty(k.shape, dtype=np.float64)
    dv = np.empty(v.shape, dtype=np.float64)
    rc = lib.oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(d_o),
                             DTYPE_F16 if dtype == "f16" else DTYPE_BF16,
                             _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Sk, d,
                             int(bool(causal)), float(scale))
    if rc != 0:
        raise ValueError("oracle rejected the dimensions")
    return dq, dk, dv


def attn_bwd_sampled(q, k, v, d_o, causal: bool, scale: float, qrows, krows, dtype: str = "bf16"):
    """fp64 gradients at sampled positions: dq [len(qrows), d] for the query
    rows (b*Hq + hq)*Sq + i and (dk, dv) [len(krows), d] for the keys
    (b*Hkv + hk)*Sk + j, in the order given."""
    lib = _load()
    if dtype not in ("bf16", "f16"):
        raise ValueError(f"unknown dtype {dtype!r}")
    q, k, v, d_o = (np.ascontiguousarray(x).view(np.uint16) for x in (q, k, v, d_o))
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    qrows = np.ascontiguousarray(qrows, dtype=np.int64)
    krows = np.asarray(krows, dtype=np.int64)
    order = np.argsort(krows, kind="stable")
    ks = np.ascontiguousarray(krows[order])
    dq = np.empty((qrows.size, d), dtype=np.float64)
    dk = np.empty((ks.size, d), dtype=np.float64)
    dv = np.empty((ks.size, d), dtype=np.float64)
    rc = lib.oracle_attn_bwd_sampled(_ptr(q), _ptr(k), _ptr(v), _ptr(d_o),
                                     DTYPE_F16 if dtype == "f16" else DTYPE_BF16, B, Hq, Hkv,
                                     Sq, Sk, d, int(bool(causal)), float(scale), _ptr(qrows),
                                     qrows.size, _ptr(ks), ks.size, _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError("oracle rejected the dimensions or rows")
    out_k = np.empty_like(dk)
    out_v = np.empty_like(dv)
    out_k[order] = dk
    out_v[order] = dv
    return dq, out_k, out_v
