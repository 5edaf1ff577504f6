"""GPU parity of the head-dimension-256 forward kernel against the fp64 CPU
oracle, through the C ABI (same tolerances as d = 64 / 128: bf16 O within
max(1e-2, one bf16 ulp), LSE within 1e-3)."""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, require_gpu

# (B, Hq, Hkv, Sq, Sk, causal): several 128-key steps, ragged tails, GQA,
# Sq != Sk, fully masked rows (causal with Sq > Sk), a single row / key.
SMALL = [
    (1, 1, 1, 1, 1, False),
    (1, 2, 2, 128, 128, False),
    (1, 2, 1, 300, 300, True),
    (2, 4, 2, 257, 333, True),
    (1, 2, 2, 300, 127, True),
    (1, 4, 1, 130, 1000, False),
    (1, 2, 2, 1, 700, True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}hq{}hkv{}sq{}sk{}{}".format(
    *s[:5], "c" if s[5] else ""))
def test_d256_small_full_compare(oracle_mod, shape, dtype):
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, causal = shape
    d = 256
    draw = inputs.draw_qkv_f16 if dtype == "f16" else inputs.draw_qkv_bf16
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, d, seed=sum(shape) + 61)
    scale = 1.0 / np.sqrt(d)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         causal, scale, dtype=dtype)
    assert_o_close(o.float().cpu().numpy(), o_ref, kind=dtype)
    assert_lse_close(lse.cpu().numpy(), lse_ref)


@pytest.mark.gpu
def test_d256_rescaling(oracle_mod):
    """Scores rising along the keys, so the running max is raised and O
    rescaled on later steps (the rescale waits for the previous P V). At
    scale 1/48 the 128-key steps see 131 (row, step) rescales after the first
    step. Steeper scales (1/16, 1/32) put a few elements past the bf16
    tolerance in any implementation of the method: P is rounded to bf16 at
    up to 2^8 under the stale max, and a numpy emulation of exactly that
    arithmetic reproduces the kernel's error there element for element."""
    torch = require_gpu()
    B, H, S, d = 1, 2, 700, 256
    g = torch.Generator().manual_seed(8)
    q = (torch.randn(B, S, H, d, generator=g) * 2.0).to(torch.bfloat16)
    ramp = torch.linspace(0.0, 3.0, S).view(1, S, 1, 1)
    k = (torch.randn(B, S, H, d, generator=g) * (0.5 + ramp)).to(torch.bfloat16)
    v = torch.randn(B, S, H, d, generator=g).to(torch.bfloat16)
    scale = 1.0 / 48
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=False, scale=scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         False, scale)
    assert_o_close(o.float().cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), lse_ref)


@pytest.mark.gpu
def test_d256_equals_d128_on_zero_padded_heads():
    """Property at any size: with the upper 128 columns of Q and K zero, the
    scores are those of the d = 128 problem (same scale), so LSE matches the
    d = 128 kernel and O's first 128 columns match its O on V's first half."""
    torch = require_gpu()
    B, Hq, Hkv, S = 1, 4, 2, 1500
    q, k, v = (t.cuda() for t in inputs.draw_qkv_bf16(B, Hq, Hkv, S, S, 256, seed=77))
    q[..., 128:] = 0
    k[..., 128:] = 0
    scale = 0.0883
    o2, l2 = ea.forward(q, k, v, causal=True, scale=scale)
    o1, l1 = ea.forward(q[..., :128].contiguous(), k[..., :128].contiguous(),
                        v[..., :128].contiguous(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    assert (l1 - l2).abs().max().item() <= 1e-4
    diff = (o1.float() - o2[..., :128].float()).abs()
    tol = 2.0 ** -7 * o1.float().abs() + 1e-2
    assert bool((diff <= tol).all())


@pytest.mark.gpu
def test_d256_full_size_sampled_rows(oracle_mod):
    """The benchmark's d = 256 workload in its launch configuration."""
    torch = require_gpu()
    w = inputs.WORKLOADS["d256_b2h16s8192_causal"]
    q, k, v = inputs.draw_workload_16(w)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    rows = inputs.sample_rows(w.B, w.Hq, w.Sq, 800, seed=w.seed)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         w.causal, w.scale, rows=rows)
    b, rem = np.divmod(rows, w.Hq * w.Sq)
    h, i = np.divmod(rem, w.Sq)
    o_g = o[torch.as_tensor(b), torch.as_tensor(i), torch.as_tensor(h)].float().cpu().numpy()
    assert_o_close(o_g, o_ref)
    assert_lse_close(lse.cpu().numpy()[b, h, i], lse_ref)
