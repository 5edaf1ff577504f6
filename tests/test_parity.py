"""GPU parity: the CUDA attention path against the fp64 CPU oracle, on the
same seeded inputs, through the C ABI. Small shapes are compared element by
element in full; the full-size workloads (run in the launch configuration the
benchmark times) on sampled rows."""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, bf16_atol, require_gpu

# (B, Hq, Hkv, Sq, Sk, d, causal): several tiles, ragged tails, GQA, Sq != Sk,
# fully masked rows (causal with Sq > Sk), single row / single key.
SMALL = [
    (1, 1, 1, 128, 128, 64, False),
    (1, 2, 2, 1, 1, 128, False),
    (1, 2, 2, 1, 1, 64, True),
    (1, 2, 1, 17, 17, 128, True),
    (2, 4, 2, 300, 300, 128, True),
    (1, 2, 2, 129, 127, 128, False),
    (1, 2, 2, 127, 300, 64, True),
    (1, 2, 2, 300, 127, 128, True),
    (1, 4, 4, 600, 600, 128, False),
    (2, 4, 1, 513, 513, 64, True),
    (1, 3, 3, 1000, 777, 128, True),
    (1, 2, 2, 256, 1025, 128, False),
]


def run_bf16(torch, q, k, v, causal, scale):
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    return o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}hq{}hkv{}sq{}sk{}d{}{}".format(
    *s[:6], "c" if s[6] else ""))
def test_bf16_small_full_compare(oracle_mod, shape):
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = inputs.draw_qkv_bf16(B, Hq, Hkv, Sq, Sk, d, seed=sum(shape) + 17)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_bf16(torch, q, k, v, causal, scale)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), causal, scale)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)


@pytest.mark.gpu
def test_bf16_large_scores_exercise_rescaling(oracle_mod):
    """Scores spread over many log2 units, rising along the keys, so the
    running max is raised (and O rescaled) on later tiles."""
    torch = require_gpu()
    B, H, S, d = 1, 2, 700, 128
    g = torch.Generator().manual_seed(5)
    q = (torch.randn(B, S, H, d, generator=g) * 2.0).to(torch.bfloat16)
    ramp = torch.linspace(0.0, 3.0, S).view(1, S, 1, 1)
    k = (torch.randn(B, S, H, d, generator=g) * (0.5 + ramp)).to(torch.bfloat16)
    v = torch.randn(B, S, H, d, generator=g).to(torch.bfloat16)
    vmax = float(v.float().abs().max())
    for causal in (False, True):
        o, lse = run_bf16(torch, q, k, v, causal, 0.125)
        o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                             inputs.bf16_bits(v), causal, 0.125)
        # With a few dominant keys the bf16 rounding of P (relative 2^-9 per
        # weight, the normaliser kept in fp32) moves O by up to 2^-9 * max|V|
        # on top of the output's own half-ulp rounding; a rescaling mistake
        # would be off by O(1).
        err = np.abs(o - o_ref)
        bound = 2.0 ** -9 * vmax + bf16_atol(o_ref) / 2 + 1e-3
        assert (err <= bound).all(), f"max err {err.max():.3e}"
        assert_lse_close(lse, lse_ref)


@pytest.mark.gpu
def test_repeated_calls_are_deterministic():
    torch = require_gpu()
    q, k, v = (t.cuda() for t in inputs.draw_qkv_bf16(2, 4, 2, 700, 700, 128, seed=3))
    o1, l1 = ea.forward(q, k, v, causal=True)
    o2, l2 = ea.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _full_size_rows(oracle_mod, w, n_rows):
    torch = require_gpu()
    q, k, v = inputs.draw_qkv_bf16(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.seed)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    rows = inputs.sample_rows(w.B, w.Hq, w.Sq, n_rows, seed=w.seed)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), w.causal, w.scale, rows=rows)
    b, rem = np.divmod(rows, w.Hq * w.Sq)
    h, i = np.divmod(rem, w.Sq)
    o_g = o[torch.as_tensor(b), torch.as_tensor(i), torch.as_tensor(h)].float().cpu().numpy()
    l_g = lse.cpu().numpy()[b, h, i]
    assert_o_close(o_g, o_ref)
    assert_lse_close(l_g, lse_ref)
    assert torch.isfinite(lse).all() and torch.isfinite(o.float()).all()


@pytest.mark.gpu
def test_tiny_workload_full(oracle_mod):
    w = inputs.WORKLOADS["tiny_b1h1s128d64"]
    torch = require_gpu()
    q, k, v = inputs.draw_qkv_bf16(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.seed)
    o, lse = run_bf16(torch, q, k, v, w.causal, w.scale)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), w.causal, w.scale)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("name,n_rows", [
    ("b4h16s2048d128_causal", 3000),
    ("b2h32s8192d128_causal", 1500),
    ("b2h32s8192d128", 1000),
    ("gqa_b1hq32hkv8s16384d128_causal", 800),
])
def test_full_size_workloads_sampled_rows(oracle_mod, name, n_rows):
    _full_size_rows(oracle_mod, inputs.WORKLOADS[name], n_rows)


# ------------------------------------------------------------ fp16 inputs --
# (B, Hq, Hkv, Sq, Sk, d, causal): d = 64 and 128, GQA, ragged tails, Sq != Sk
SMALL_F16 = [
    (1, 2, 2, 128, 128, 128, False),
    (2, 4, 2, 300, 300, 128, True),
    (1, 2, 2, 127, 300, 64, True),
    (1, 4, 1, 600, 513, 128, False),
    (1, 2, 2, 300, 127, 128, True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SMALL_F16, ids=lambda s: "f16_b{}hq{}hkv{}sq{}sk{}d{}{}".format(
    *s[:6], "c" if s[6] else ""))
def test_f16_small_full_compare(oracle_mod, shape):
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = inputs.draw_qkv_f16(B, Hq, Hkv, Sq, Sk, d, seed=sum(shape) + 29)
    scale = 1.0 / np.sqrt(d)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    assert o.dtype == torch.float16
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         causal, scale, dtype="f16")
    assert_o_close(o.float().cpu().numpy(), o_ref, kind="f16")
    assert_lse_close(lse.cpu().numpy(), lse_ref)


@pytest.mark.gpu
def test_f16_full_size_sampled_rows(oracle_mod):
    torch = require_gpu()
    w = inputs.WORKLOADS["f16_b2h32s8192d128_causal"]
    q, k, v = inputs.draw_workload_16(w)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    rows = inputs.sample_rows(w.B, w.Hq, w.Sq, 1200, seed=w.seed)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         w.causal, w.scale, dtype="f16", rows=rows)
    b, rem = np.divmod(rows, w.Hq * w.Sq)
    h, i = np.divmod(rem, w.Sq)
    o_g = o[torch.as_tensor(b), torch.as_tensor(i), torch.as_tensor(h)].float().cpu().numpy()
    assert_o_close(o_g, o_ref, kind="f16")
    assert_lse_close(lse.cpu().numpy()[b, h, i], lse_ref)


# ------------------------------------------------------------- large sizes --

@pytest.mark.gpu
def test_long_sequence_near_the_index_limit(oracle_mod):
    """Sq = Sk = 131072 with 16 heads: 268M elements per tensor (the 32-bit
    element-count guard allows up to 2^31 - 1), K/V tile coordinates up to
    1024 tiles, causal; sampled rows across the whole range against the
    oracle, including the first and the last row."""
    torch = require_gpu()
    B, H, S, d = 1, 16, 131072, 128
    g = torch.Generator().manual_seed(77)
    q = torch.randn(B, S, H, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, S, H, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, S, H, d, generator=g).to(torch.bfloat16)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=True)
    assert ea.attn_device_status() == ea.ATTN_OK
    rows = inputs.sample_rows(B, H, S, 120, seed=7)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         True, 1.0 / np.sqrt(d), rows=rows)
    b, rem = np.divmod(rows, H * S)
    h, i = np.divmod(rem, S)
    o_g = o[torch.as_tensor(b), torch.as_tensor(i), torch.as_tensor(h)].float().cpu().numpy()
    assert_o_close(o_g, o_ref)
    assert_lse_close(lse.cpu().numpy()[b, h, i], lse_ref)
