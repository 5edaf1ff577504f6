"""GPU parity of the QK-RMSNorm prologue (RMSNorm across heads) against the
fp64 oracle, and of the prologue followed by attention."""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, require_gpu


def _ulp(ref, dtype):
    """Spacing of the storage type at |ref|: 2^(e - mantissa bits) in the
    normal range; fixed below it (fp16 subnormals are multiples of 2^-24,
    bf16 ones of 2^-133)."""
    mant, tiny = (10, 2.0 ** -24) if dtype == "f16" else (7, 2.0 ** -133)
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-300)))
    return np.maximum(np.exp2(e - mant), tiny)


def _draw_weights(torch, n, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    w = 1.0 + 0.25 * torch.randn(n, generator=g)
    return w.to(torch.float16 if dtype == "f16" else torch.bfloat16)


def _check_norm(got, x_bits, w_bits, eps, dtype, oracle_mod):
    ref = oracle_mod.rmsnorm_heads(x_bits, w_bits, eps, dtype)
    err = np.abs(got.astype(np.float64) - ref)
    # fp32 arithmetic then one rounding: within one ulp of the storage type
    assert (err <= _ulp(ref, dtype) + 1e-30).all(), f"max err {err.max():.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(2, 37, 53, 4, 2, 64), (1, 130, 7, 8, 8, 128),
                                   (3, 1, 1, 2, 1, 128)])
def test_qk_rmsnorm_matches_oracle(oracle_mod, dtype, shape):
    torch = require_gpu()
    B, Sq, Sk, Hq, Hkv, d = shape
    draw = inputs.draw_qkv_f16 if dtype == "f16" else inputs.draw_qkv_bf16
    q, k, _ = draw(B, Hq, Hkv, Sq, Sk, d, seed=sum(shape) + 3)
    q = q * 3  # keep the data away from unit RMS
    wq, wk = _draw_weights(torch, Hq * d, dtype, 1), _draw_weights(torch, Hkv * d, dtype, 2)
    qo, ko = ea.qk_rmsnorm(q.cuda(), k.cuda(), wq.cuda(), wk.cuda(), eps=1e-6)
    assert ea.attn_device_status() == ea.ATTN_OK
    _check_norm(qo.float().cpu().numpy(), inputs.bits16(q), inputs.bits16(wq), 1e-6, dtype,
                oracle_mod)
    _check_norm(ko.float().cpu().numpy(), inputs.bits16(k), inputs.bits16(wk), 1e-6, dtype,
                oracle_mod)


@pytest.mark.gpu
def test_qk_rmsnorm_in_place(oracle_mod):
    torch = require_gpu()
    q, k, _ = inputs.draw_qkv_bf16(1, 4, 4, 100, 100, 64, seed=8)
    wq, wk = _draw_weights(torch, 256, "bf16", 3), _draw_weights(torch, 256, "bf16", 4)
    dq, dk = q.cuda(), k.cuda()
    ea.qk_rmsnorm(dq, dk, wq.cuda(), wk.cuda(), eps=0.0, out=(dq, dk))
    assert ea.attn_device_status() == ea.ATTN_OK
    _check_norm(dq.float().cpu().numpy(), inputs.bits16(q), inputs.bits16(wq), 0.0, "bf16",
                oracle_mod)
    _check_norm(dk.float().cpu().numpy(), inputs.bits16(k), inputs.bits16(wk), 0.0, "bf16",
                oracle_mod)


@pytest.mark.gpu
def test_qk_rmsnorm_full_size_sampled_tokens(oracle_mod):
    torch = require_gpu()
    w = inputs.WORKLOADS["b2h32s8192d128_causal"]
    q, k, _ = inputs.draw_qkv_bf16(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.seed)
    wq, wk = _draw_weights(torch, w.Hq * w.d, "bf16", 5), _draw_weights(torch, w.Hkv * w.d, "bf16", 6)
    qo, ko = ea.qk_rmsnorm(q.cuda(), k.cuda(), wq.cuda(), wk.cuda())
    assert ea.attn_device_status() == ea.ATTN_OK
    rng = np.random.default_rng(0)
    toks = rng.choice(w.B * w.Sq, 400, replace=False)
    b, s = np.divmod(toks, w.Sq)
    for x, xo, wt in ((q, qo, wq), (k, ko, wk)):
        xs = x[torch.as_tensor(b), torch.as_tensor(s)]
        got = xo[torch.as_tensor(b), torch.as_tensor(s)].float().cpu().numpy()
        _check_norm(got, inputs.bits16(xs), inputs.bits16(wt), 1e-6, "bf16", oracle_mod)


@pytest.mark.gpu
def test_prologue_then_attention(oracle_mod):
    """qk_rmsnorm -> attention on the GPU against the oracle's own
    rmsnorm -> round to bf16 -> attention."""
    torch = require_gpu()
    B, Hq, Hkv, S, d = 1, 4, 2, 300, 128
    q, k, v = inputs.draw_qkv_bf16(B, Hq, Hkv, S, S, d, seed=12)
    wq, wk = _draw_weights(torch, Hq * d, "bf16", 7), _draw_weights(torch, Hkv * d, "bf16", 8)
    qn, kn = ea.qk_rmsnorm(q.cuda(), k.cuda(), wq.cuda(), wk.cuda())
    o, lse = ea.forward(qn, kn, v.cuda(), causal=True)
    assert ea.attn_device_status() == ea.ATTN_OK
    rq = oracle_mod.rmsnorm_heads(inputs.bits16(q), inputs.bits16(wq), 1e-6)
    rk = oracle_mod.rmsnorm_heads(inputs.bits16(k), inputs.bits16(wk), 1e-6)
    qb = inputs.bits16(torch.from_numpy(rq).to(torch.bfloat16))
    kb = inputs.bits16(torch.from_numpy(rk).to(torch.bfloat16))
    o_ref, lse_ref = oracle_mod.attn_fwd(qb, kb, inputs.bits16(v), True, 1.0 / np.sqrt(d))
    # a normalised value can differ from the oracle's rounding of it only when
    # the fp32 result falls within ~1e-7 of a bf16 rounding boundary (a few in
    # 10^5 elements, one ulp each); the attention tolerances stand
    assert_o_close(o.float().cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), lse_ref)
