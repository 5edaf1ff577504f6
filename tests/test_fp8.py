"""GPU parity for the FP8 path: the block quantiser bit for bit against the
oracle's quantiser, and E4M3 attention against the fp64 oracle evaluated on
the dequantised inputs. Each side quantises with its own code."""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, record, require_gpu


def gpu_quantise(torch, x):
    codes, scales = ea.quantize_fp8(x.cuda())
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1, 64, 1, 128), (2, 150, 3, 64), (1, 1, 2, 128),
                                   (2, 333, 4, 128)])
def test_quantiser_bit_exact_small(oracle_mod, shape):
    torch = require_gpu()
    g = torch.Generator().manual_seed(sum(shape))
    x = torch.randn(shape, generator=g) * 3
    x[0, : min(64, shape[1]), 0, :] = 0.0  # an all-zero block
    if shape[1] > 70:
        x[-1, 70, -1, 5] = 1e4  # an outlier
        x[-1, 71, -1, 6] = 1e-30  # a tiny value (flushes to a zero code)
    c_g, s_g = gpu_quantise(torch, x)
    c_o, s_o = oracle_mod.quantize_fp8_e4m3(x.numpy())
    np.testing.assert_array_equal(s_g, s_o)
    np.testing.assert_array_equal(c_g, c_o)


@pytest.mark.gpu
def test_quantiser_bit_exact_fp8_workload(oracle_mod):
    torch = require_gpu()
    w = inputs.WORKLOADS["fp8_b4h16s4096d128"]
    for x in inputs.draw_workload_f32(w):
        c_g, s_g = gpu_quantise(torch, x)
        c_o, s_o = oracle_mod.quantize_fp8_e4m3(x.numpy())
        np.testing.assert_array_equal(s_g, s_o)
        np.testing.assert_array_equal(c_g, c_o)


def _fp8_case(oracle_mod, torch, q, k, v, causal, scale, rows=None):
    qc, qs = ea.quantize_fp8(q.cuda())
    kc, ks = ea.quantize_fp8(k.cuda())
    vc, vs = ea.quantize_fp8(v.cuda())
    o, lse = ea.forward_fp8(qc, kc, vc, qs, ks, vs, causal=causal, scale=scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    oq = [oracle_mod.quantize_fp8_e4m3(t.numpy()) for t in (q, k, v)]
    o_ref, lse_ref = oracle_mod.attn_fwd(oq[0][0], oq[1][0], oq[2][0], causal, scale, dtype="e4m3",
                                         q_scale=oq[0][1], k_scale=oq[1][1], v_scale=oq[2][1],
                                         rows=rows)
    return o, lse, o_ref, lse_ref


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1, 2, 2, 128, 128, 128, False), (2, 4, 2, 300, 300, 128, True),
                                   (1, 2, 2, 200, 517, 128, False), (1, 4, 4, 513, 513, 64, True),
                                   (1, 8, 2, 700, 1100, 128, True), (2, 4, 1, 900, 333, 64, True)])
def test_fp8_attention_small(oracle_mod, shape):
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = inputs.draw_qkv_f32(B, Hq, Hkv, Sq, Sk, d, seed=sum(shape), outlier_frac=0.001)
    o, lse, o_ref, lse_ref = _fp8_case(oracle_mod, torch, q, k, v, causal, 1 / np.sqrt(d))
    st = assert_o_close(o.float().cpu().numpy(), o_ref, kind="fp8")
    record("small fp8 b{}hq{}hkv{}sq{}sk{}d{}{}".format(*shape[:6], "c" if causal else ""), "fp8",
           st, assert_lse_close(lse.cpu().numpy(), lse_ref, tol=1e-3), B * Hq * Sq)


@pytest.mark.gpu
def test_fp8_workload_full_compare(oracle_mod):
    """Every element of the FP8 workload (B4 H16 S4096, 0.1 % x20 outliers)."""
    torch = require_gpu()
    w = inputs.WORKLOADS["fp8_b4h16s4096d128"]
    q, k, v = inputs.draw_workload_f32(w)
    o, lse, o_ref, lse_ref = _fp8_case(oracle_mod, torch, q, k, v, w.causal, w.scale)
    st = assert_o_close(o.float().cpu().numpy(), o_ref, kind="fp8")
    record(w.name + " (full)", "fp8", st,
           assert_lse_close(lse.cpu().numpy(), lse_ref, tol=1e-3), w.B * w.Hq * w.Sq)
