"""Seeded random shapes against the oracle: the forward (d = 64, 128, 256;
bf16 / fp16; GQA; causal with Sq above, equal to or below Sk) and the backward
(d = 64, 128), compared element by element in full. The draw is fixed, so every
case is reproducible by its id; it covers tile edges (sizes around multiples
of 64 and 128, single rows and keys) that the hand-picked cases may miss."""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, require_gpu
from tests.test_bwd import assert_grad_close


def _size(rng):
    """Mostly random in [1, 900], sometimes on or next to a tile edge."""
    if rng.random() < 0.4:
        return int(max(1, rng.choice([64, 128, 192, 256, 384, 512]) + rng.integers(-1, 2)))
    return int(rng.integers(1, 901))


def _forward_cases(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        d = int(rng.choice([64, 128, 256]))
        hkv = int(rng.choice([1, 2]))
        group = int(rng.choice([1, 2, 4]))
        cases.append((int(rng.integers(1, 3)), hkv * group, hkv, _size(rng), _size(rng), d,
                      bool(rng.random() < 0.6), str(rng.choice(["bf16", "f16"])), 3000 + i))
    return cases


def _backward_cases(n=12, seed=2025):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        d = int(rng.choice([64, 128]))
        hkv = int(rng.choice([1, 2]))
        group = int(rng.choice([1, 2, 4]))
        cases.append((1, hkv * group, hkv, _size(rng), _size(rng), d, bool(rng.random() < 0.6),
                      str(rng.choice(["bf16", "f16"])), 4000 + i))
    return cases


def _id(c):
    return "b{}hq{}hkv{}sq{}sk{}d{}{}_{}".format(*c[:6], "c" if c[6] else "", c[7])


@pytest.mark.gpu
@pytest.mark.parametrize("case", _forward_cases(), ids=_id)
def test_forward_random_shapes(oracle_mod, case):
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d, causal, dtype, seed = case
    draw = inputs.draw_qkv_f16 if dtype == "f16" else inputs.draw_qkv_bf16
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, d, seed=seed)
    scale = 1.0 / np.sqrt(d)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         causal, scale, dtype=dtype)
    assert_o_close(o.float().cpu().numpy(), o_ref, kind=dtype)
    assert_lse_close(lse.cpu().numpy(), lse_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("case", _backward_cases(), ids=_id)
def test_backward_random_shapes(oracle_mod, case):
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d, causal, dtype, seed = case
    draw = inputs.draw_qkv_f16 if dtype == "f16" else inputs.draw_qkv_bf16
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, d, seed=seed)
    do = inputs.draw_grad_out(B, Sq, Hq, d, seed, dtype=dtype)
    scale = 1.0 / np.sqrt(d)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = ea.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    rq, rk, rv = oracle_mod.attn_bwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                     inputs.bits16(do), causal, scale, dtype=dtype)
    assert_grad_close("dq", dq.float().cpu().numpy(), rq)
    assert_grad_close("dk", dk.float().cpu().numpy(), rk)
    assert_grad_close("dv", dv.float().cpu().numpy(), rv)
