"""Exact attention for B300 (sm_103a): Python binding of libattn_b300.

The functions named like the C ABI (``attn_fwd``, ``attn_fwd_fp8``,
``attn_fwd_splitkv``, ``attn_bwd``, ``attn_quantize_fp8_e4m3``,
``attn_device_status``, ``attn_status_string``, ...) only marshal arguments:
tensors become device pointers, a torch stream (or None = torch's current
stream) becomes a cudaStream_t; they return the C status code. ``forward``,
``forward_fp8``, ``forward_splitkv``, ``backward`` and ``quantize_fp8``
additionally allocate the outputs with torch and raise ``AttnError`` on a
non-zero status.
All compute runs in the CUDA library; there is no fallback path: if the
library is missing every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_MISALIGNED",
    "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT", "ATTN_BF16", "ATTN_FP8_E4M3", "ATTN_F16", "AttnError",
    "attn_fwd", "attn_fwd_fp8", "attn_fwd_splitkv", "attn_fwd_splitkv_noalloc",
    "attn_splitkv_plan", "attn_qk_rmsnorm", "qk_rmsnorm", "attn_bwd", "attn_bwd_workspace_size",
    "backward",
    "attn_quantize_fp8_e4m3", "attn_device_status", "attn_set_wait_limit_ns",
    "attn_get_wait_limit_ns", "attn_status_string", "forward", "forward_fp8", "forward_splitkv", "quantize_fp8",
    "library_path", "load",
]

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5
ATTN_BF16 = 0
ATTN_FP8_E4M3 = 1
ATTN_F16 = 2
FP8_BLOCK_ROWS = 64

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return os.path.join(_HERE, "libattn_b300.so")


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {attn_status_string(code)} ({code})" if what else
                         f"{attn_status_string(code)} ({code})")


def load():
    """Load libattn_b300.so (built in-tree by ``exact_attention_forward_14_b300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build it with `python -m exact_attention_forward_14_b300.build`"
                " (nvcc, sm_103a); this package has no non-CUDA fallback")
        lib = ctypes.CDLL(path)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
        lib.attn_fwd.restype = I
        lib.attn_fwd_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.attn_fwd_fp8.restype = I
        lib.attn_fwd_splitkv.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P,
                                         ctypes.c_size_t, P]
        lib.attn_fwd_splitkv.restype = I
        lib.attn_fwd_splitkv_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P]
        lib.attn_fwd_splitkv_noalloc.restype = I
        lib.attn_splitkv_plan.argtypes = [I, I, I, I, I, I, I, ctypes.POINTER(I),
                                          ctypes.POINTER(ctypes.c_size_t)]
        lib.attn_splitkv_plan.restype = I
        lib.attn_qk_rmsnorm.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, I, P]
        lib.attn_qk_rmsnorm.restype = I
        lib.attn_quantize_fp8_e4m3.argtypes = [P, P, P, I, I, I, I, P]
        lib.attn_quantize_fp8_e4m3.restype = I
        lib.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P,
                                 ctypes.c_size_t, P]
        lib.attn_bwd.restype = I
        lib.attn_bwd_workspace_size.argtypes = [I, I, I, ctypes.POINTER(ctypes.c_size_t)]
        lib.attn_bwd_workspace_size.restype = I
        lib.attn_device_status.argtypes = [P]
        lib.attn_device_status.restype = I
        lib.attn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.attn_set_wait_limit_ns.restype = I
        lib.attn_get_wait_limit_ns.argtypes = []
        lib.attn_get_wait_limit_ns.restype = ctypes.c_ulonglong
        lib.attn_status_string.argtypes = [I]
        lib.attn_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _ptr(x):
    """Device pointer of a tensor, or an int passed through (0 / None = NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


# ----------------------------------------------------------- C ABI mirror --

def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, dtype=ATTN_BF16,
             stream=None) -> int:
    return load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq),
                           int(Hkv), int(Sq), int(Sk), int(d), int(bool(causal)), float(scale),
                           int(dtype), _stream(stream))


def attn_fwd_fp8(q, k, v, q_scale, k_scale, v_scale, o, lse, B, Hq, Hkv, Sq, Sk, d, causal,
                 scale, stream=None) -> int:
    return load().attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(q_scale), _ptr(k_scale),
                               _ptr(v_scale), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv),
                               int(Sq), int(Sk), int(d), int(bool(causal)), float(scale),
                               _stream(stream))


def attn_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, dtype, num_splits,
                     workspace, workspace_bytes, stream=None) -> int:
    return load().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                   int(Hq), int(Hkv), int(Sq), int(Sk), int(d),
                                   int(bool(causal)), float(scale), int(dtype), int(num_splits),
                                   _ptr(workspace), int(workspace_bytes), _stream(stream))


def attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, dtype,
                             num_splits, stream=None) -> int:
    """attn_fwd_splitkv with the library's built-in 64 MiB workspace (no
    allocation anywhere; for callers that may not allocate device memory)."""
    return load().attn_fwd_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B),
                                           int(Hq), int(Hkv), int(Sq), int(Sk), int(d),
                                           int(bool(causal)), float(scale), int(dtype),
                                           int(num_splits), _stream(stream))


def attn_splitkv_plan(B, Hq, Sq, Sk, d, causal=False, num_sms=0):
    """Returns (status, num_splits, workspace_bytes)."""
    n = ctypes.c_int(0)
    w = ctypes.c_size_t(0)
    rc = load().attn_splitkv_plan(int(B), int(Hq), int(Sq), int(Sk), int(d), int(bool(causal)),
                                  int(num_sms), ctypes.byref(n), ctypes.byref(w))
    return rc, n.value, w.value


def attn_qk_rmsnorm(q, k, q_weight, k_weight, q_out, k_out, B, Sq, Sk, Hq, Hkv, d, eps, dtype,
                    stream=None) -> int:
    return load().attn_qk_rmsnorm(_ptr(q), _ptr(k), _ptr(q_weight), _ptr(k_weight), _ptr(q_out),
                                  _ptr(k_out), int(B), int(Sq), int(Sk), int(Hq), int(Hkv),
                                  int(d), float(eps), int(dtype), _stream(stream))


def attn_quantize_fp8_e4m3(x, codes, scale, B, S, H, d, stream=None) -> int:
    return load().attn_quantize_fp8_e4m3(_ptr(x), _ptr(codes), _ptr(scale), int(B), int(S),
                                         int(H), int(d), _stream(stream))


def attn_bwd(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale, dtype,
             workspace, workspace_bytes, stream=None) -> int:
    return load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq),
                           _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(Sq), int(Sk),
                           int(d), int(bool(causal)), float(scale), int(dtype), _ptr(workspace),
                           int(workspace_bytes), _stream(stream))


def attn_bwd_workspace_size(B, Hq, Sq):
    """Returns (status, workspace_bytes)."""
    w = ctypes.c_size_t(0)
    rc = load().attn_bwd_workspace_size(int(B), int(Hq), int(Sq), ctypes.byref(w))
    return rc, w.value


def attn_device_status(stream=None) -> int:
    return load().attn_device_status(_stream(stream))


def attn_set_wait_limit_ns(ns: int) -> int:
    return load().attn_set_wait_limit_ns(int(ns))


def attn_get_wait_limit_ns() -> int:
    return int(load().attn_get_wait_limit_ns())


def attn_status_string(code: int) -> str:
    return load().attn_status_string(int(code)).decode()


# ------------------------------------------------------ tensor conveniences --

def _check(rc, what):
    if rc != ATTN_OK:
        raise AttnError(rc, what)


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
            stream=None):
    """bf16 or fp16 attention forward. q [B,Sq,Hq,d], k/v [B,Sk,Hkv,d] (CUDA,
    contiguous, all of one dtype). Returns (o [B,Sq,Hq,d] in the inputs'
    dtype, lse fp32 [B,Hq,Sq])."""
    import torch
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    if q.dtype == torch.bfloat16:
        code = ATTN_BF16
    elif q.dtype == torch.float16:
        code = ATTN_F16
    else:
        raise TypeError(f"forward takes bf16 or fp16 tensors, not {q.dtype}")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Sq, Hq, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    for t in (q, k, v, out, lse):
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    _check(attn_fwd(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, code, stream),
           "attn_fwd")
    return out, lse


def forward_fp8(q, k, v, q_scale, k_scale, v_scale, causal: bool = False,
                scale: float | None = None, out=None, lse=None, stream=None):
    """E4M3 attention forward with per-64-row block scales. Returns (o bf16, lse fp32)."""
    import torch
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Sq, Hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check(attn_fwd_fp8(q, k, v, q_scale, k_scale, v_scale, out, lse, B, Hq, Hkv, Sq, Sk, d,
                        causal, scale, stream), "attn_fwd_fp8")
    return out, lse


def forward_splitkv(q, k, v, causal: bool = False, scale: float | None = None,
                    num_splits: int | None = None, workspace=None, out=None, lse=None,
                    stream=None):
    """Split-KV forward (bf16 or fp16). num_splits None = attn_splitkv_plan's
    choice; the fp32 workspace is allocated with torch unless given."""
    import torch
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    code = ATTN_F16 if q.dtype == torch.float16 else ATTN_BF16
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits is None:
        rc, num_splits, _ = attn_splitkv_plan(B, Hq, Sq, Sk, d, causal)
        _check(rc, "attn_splitkv_plan")
    need = num_splits * B * Hq * Sq * (d + 1) * 4
    if workspace is None:
        workspace = torch.empty(need // 4, dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty((B, Sq, Hq, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check(attn_fwd_splitkv(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, code,
                            num_splits, workspace, workspace.numel() * workspace.element_size(),
                            stream), "attn_fwd_splitkv")
    return out, lse


def backward(q, k, v, o, lse, d_o, causal: bool = False, scale: float | None = None,
             workspace=None, out=None, stream=None):
    """Gradients (dq, dk, dv) of sum(d_o * O) for the forward pass that gave
    (o, lse) on (q, k, v); bf16 or fp16, CUDA, contiguous. The fp32 workspace
    is allocated with torch unless given; out = (dq, dk, dv) or None."""
    import torch
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"backward takes bf16 or fp16 tensors, not {q.dtype}")
    if any(t.dtype != q.dtype for t in (k, v, o, d_o)):
        raise TypeError("q, k, v, o and d_o must share one dtype")
    if lse.dtype != torch.float32:
        raise TypeError("lse must be float32")
    code = ATTN_F16 if q.dtype == torch.float16 else ATTN_BF16
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc, need = attn_bwd_workspace_size(B, Hq, Sq)
    _check(rc, "attn_bwd_workspace_size")
    if workspace is None:
        workspace = torch.empty(need // 4, dtype=torch.float32, device=q.device)
    dq, dk, dv = out if out is not None else (torch.empty_like(q), torch.empty_like(k),
                                              torch.empty_like(v))
    for t in (q, k, v, o, lse, d_o, dq, dk, dv):
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    _check(attn_bwd(q, k, v, o, lse, d_o, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale, code,
                    workspace, workspace.numel() * workspace.element_size(), stream), "attn_bwd")
    return dq, dk, dv


def qk_rmsnorm(q, k, q_weight, k_weight, eps: float = 1e-6, out=None, stream=None):
    """RMSNorm across heads of q [B,Sq,Hq,d] and k [B,Sk,Hkv,d] (bf16 or fp16,
    CUDA) with weights [Hq*d] / [Hkv*d]. out = (q_out, k_out), or None for new
    tensors; pass (q, k) to normalise in place. Returns (q_out, k_out)."""
    import torch
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    code = ATTN_F16 if q.dtype == torch.float16 else ATTN_BF16
    q_out, k_out = out if out is not None else (torch.empty_like(q), torch.empty_like(k))
    _check(attn_qk_rmsnorm(q, k, q_weight, k_weight, q_out, k_out, B, Sq, Sk, Hq, Hkv, d, eps,
                           code, stream), "attn_qk_rmsnorm")
    return q_out, k_out


def quantize_fp8(x, stream=None):
    """fp32 x [B,S,H,d] (CUDA) -> (E4M3 codes as uint8 [B,S,H,d], fp32 scales [B,H,ceil(S/64)])."""
    import torch
    B, S, H, d = x.shape
    codes = torch.empty((B, S, H, d), dtype=torch.uint8, device=x.device)
    scales = torch.empty((B, H, (S + FP8_BLOCK_ROWS - 1) // FP8_BLOCK_ROWS), dtype=torch.float32,
                         device=x.device)
    _check(attn_quantize_fp8_e4m3(x, codes, scales, B, S, H, d, stream), "attn_quantize_fp8_e4m3")
    return codes, scales
