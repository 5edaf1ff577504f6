"""The kernel's watchdog on a real GPU, without faulting it.

A test-only build of the library (libattn_watchdog_test.so, built with
ATTN_TEST_NEVER_ARM_Q) never arms the Q-tile barrier, so the MMA warp waits on
a flag that nothing sets. Its bounded wait must run out after the one-second
limit, record ATTN_ERR_TIMEOUT in the device status word, drain, release the
tensor memory and return. The CUDA context must stay usable: the regular
library, loaded in the same process, still matches the oracle afterwards.
"""
import ctypes
import os
import time

import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, require_gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "exact_attention_forward_14_b300", "libattn_watchdog_test.so")


def _load_test_lib():
    lib = ctypes.CDLL(LIB)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
    lib.attn_fwd.restype = I
    lib.attn_device_status.argtypes = [P]
    lib.attn_device_status.restype = I
    return lib


@pytest.mark.gpu
def test_unarmed_barrier_times_out_and_context_survives(oracle_mod):
    torch = require_gpu()
    lib = _load_test_lib()
    B, H, S, d = 1, 4, 512, 128
    q, k, v = inputs.draw_qkv_bf16(B, H, H, S, S, d, seed=77)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty((B, S, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    t0 = time.perf_counter()
    rc = lib.attn_fwd(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, H, H, S, S, d, 1, 1.0 / np.sqrt(d), ea.ATTN_BF16, stream)
    assert rc == ea.ATTN_OK  # the launch itself is valid
    st = lib.attn_device_status(stream)
    elapsed = time.perf_counter() - t0
    assert st == ea.ATTN_ERR_TIMEOUT
    assert 0.9 < elapsed < 10.0, f"watchdog took {elapsed:.2f} s"
    # the word is cleared by the read
    assert lib.attn_device_status(stream) == ea.ATTN_OK

    # the context is intact: the regular library still computes the right answer
    o2, lse2 = ea.forward(dq, dk, dv, causal=True)
    assert ea.attn_device_status() == ea.ATTN_OK
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), True, 1.0 / np.sqrt(d))
    assert_o_close(o2.float().cpu().numpy(), o_ref)
    assert_lse_close(lse2.cpu().numpy(), lse_ref)


def _bind_bwd(lib):
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P,
                             ctypes.c_size_t, P]
    lib.attn_bwd.restype = I
    return lib


@pytest.mark.gpu
def test_backward_unarmed_barriers_time_out_and_context_survives(oracle_mod):
    """The same test build never arms the dK/dV kernel's K/V barrier nor the
    dQ kernel's Q/dO barrier: both tensor-core kernels of attn_bwd must end
    through their watchdogs, and the regular library still computes correct
    gradients afterwards."""
    torch = require_gpu()
    lib = _bind_bwd(_load_test_lib())
    B, Hq, Hkv, S, d = 1, 4, 2, 384, 128
    q, k, v = (t.cuda() for t in inputs.draw_qkv_bf16(B, Hq, Hkv, S, S, d, seed=78))
    do = inputs.draw_grad_out(B, S, Hq, d, 78).cuda()
    o, lse = ea.forward(q, k, v, causal=True)
    assert ea.attn_device_status() == ea.ATTN_OK
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc, wbytes = ea.attn_bwd_workspace_size(B, Hq, S)
    ws = torch.empty(wbytes // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    rc = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, S, S,
                      d, 1, 1.0 / np.sqrt(d), ea.ATTN_BF16, ws.data_ptr(), wbytes, stream)
    assert rc == ea.ATTN_OK
    st = lib.attn_device_status(stream)
    elapsed = time.perf_counter() - t0
    assert st == ea.ATTN_ERR_TIMEOUT
    assert 0.9 < elapsed < 20.0, f"watchdog took {elapsed:.2f} s"
    assert lib.attn_device_status(stream) == ea.ATTN_OK
    # the regular library on the same context: gradients still right
    g = ea.backward(q, k, v, o, lse, do, causal=True)
    assert ea.attn_device_status() == ea.ATTN_OK
    ref = oracle_mod.attn_bwd(*(inputs.bits16(t.cpu()) for t in (q, k, v, do)), True,
                              1.0 / np.sqrt(d))
    for got, r in zip(g, ref):
        err = np.abs(got.float().cpu().numpy() - r)
        assert (err <= 2.0 ** -7 * np.abs(r) + 0.01 * np.abs(r).max()).all()


@pytest.mark.gpu
def test_d256_unarmed_barrier_times_out_and_context_survives(oracle_mod):
    torch = require_gpu()
    lib = _load_test_lib()
    B, H, S, d = 1, 2, 300, 256
    q, k, v = inputs.draw_qkv_bf16(B, H, H, S, S, d, seed=79)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty((B, S, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    rc = lib.attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, H, H, S, S, d, 1, 1.0 / 16, ea.ATTN_BF16, stream)
    assert rc == ea.ATTN_OK
    st = lib.attn_device_status(stream)
    assert st == ea.ATTN_ERR_TIMEOUT
    assert 0.9 < time.perf_counter() - t0 < 10.0
    o2, lse2 = ea.forward(qd, kd, vd, causal=True, scale=1.0 / 16)
    assert ea.attn_device_status() == ea.ATTN_OK
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), True, 1.0 / 16)
    assert_o_close(o2.float().cpu().numpy(), o_ref)
    assert_lse_close(lse2.cpu().numpy(), lse_ref)
