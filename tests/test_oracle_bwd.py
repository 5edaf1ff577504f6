"""Pins for the oracle's backward pass (dQ, dK, dV of sum(dO * O)), checked
against things other than its own formula: central finite differences of the
oracle's forward pass, torch autograd through a materialised fp64 softmax, the
closed form of a single key, and the invariants that follow from the softmax
being shift-invariant and summing to one. CPU only."""
import numpy as np
import pytest
import torch

from exact_attention_forward_14_b300 import inputs

H_STEP = 2.0 ** -8  # grid spacing of the test inputs


def grid_bits(rng, shape, lim=200):
    """Values k / 256 with |k| <= lim: exact in bf16 (at most 8 significant
    bits), and so are the values two grid steps away, which the finite
    differences need. Returns (uint16 bf16 bits, float64 values)."""
    vals = rng.integers(-lim, lim + 1, size=shape).astype(np.float64) * H_STEP
    t = torch.as_tensor(vals).to(torch.bfloat16)
    assert np.array_equal(t.to(torch.float64).numpy(), vals)
    return inputs.bf16_bits(t), vals


def to_bits(vals):
    t = torch.as_tensor(vals).to(torch.bfloat16)
    assert np.array_equal(t.to(torch.float64).numpy(), vals)
    return inputs.bf16_bits(t)


def make_case(seed, B, Hq, Hkv, Sq, Sk, d):
    rng = np.random.default_rng(seed)
    q = grid_bits(rng, (B, Sq, Hq, d))
    k = grid_bits(rng, (B, Sk, Hkv, d))
    v = grid_bits(rng, (B, Sk, Hkv, d))
    do = grid_bits(rng, (B, Sq, Hq, d))
    return q, k, v, do


def loss(oracle_mod, qv, kv, vv, do_vals, causal, scale):
    o, _ = oracle_mod.attn_fwd(to_bits(qv), to_bits(kv), to_bits(vv), causal, scale)
    return float(np.sum(o * do_vals))


@pytest.mark.parametrize("causal,shape", [
    (True, (1, 4, 2, 9, 13, 8)),    # GQA, Sq < Sk
    (True, (1, 2, 1, 11, 6, 8)),    # Sq > Sk: the first rows see no key
    (False, (2, 2, 2, 7, 10, 8)),
])
def test_gradients_match_finite_differences_of_the_forward(oracle_mod, causal, shape):
    """Richardson-extrapolated central differences, error O(h^4) ~ 1e-10,
    of the oracle's forward loss at a sample of elements of q, k and v."""
    B, Hq, Hkv, Sq, Sk, d = shape
    scale = 0.5
    (qb, qv), (kb, kv), (vb, vv), (dob, dov) = make_case(7, *shape)
    dq, dk, dv = oracle_mod.attn_bwd(qb, kb, vb, dob, causal, scale)
    rng = np.random.default_rng(11)
    for name, vals, grad in (("q", qv, dq), ("k", kv, dk), ("v", vv, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in vals.shape)

            def at(delta):
                x = vals.copy()
                x[idx] += delta
                args = {"q": qv, "k": kv, "v": vv}
                args[name] = x
                return loss(oracle_mod, args["q"], args["k"], args["v"], dov, causal, scale)

            d1 = (at(H_STEP) - at(-H_STEP)) / (2 * H_STEP)
            d2 = (at(2 * H_STEP) - at(-2 * H_STEP)) / (4 * H_STEP)
            fd = (4 * d1 - d2) / 3
            assert abs(grad[idx] - fd) <= 1e-7 + 1e-6 * abs(fd), (name, idx, grad[idx], fd)


def torch_reference_grads(qv, kv, vv, dov, causal, scale):
    """Autograd through a materialised fp64 softmax (every row has a key)."""
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (qv, kv, vv))
    Hq, Hkv = q.shape[2], k.shape[2]
    kr = k.repeat_interleave(Hq // Hkv, dim=2)
    vr = v.repeat_interleave(Hq // Hkv, dim=2)
    s = torch.einsum("bihc,bjhc->bhij", q, kr) * scale
    Sq, Sk = s.shape[-2], s.shape[-1]
    if causal:
        i = torch.arange(Sq)[:, None]
        j = torch.arange(Sk)[None, :]
        s = s.masked_fill(j > i + Sk - Sq, float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.einsum("bhij,bjhc->bihc", p, vr)
    o.backward(torch.tensor(dov))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal,shape", [
    (True, (2, 6, 2, 33, 47, 16)),
    (True, (1, 4, 4, 40, 40, 32)),
    (False, (1, 8, 1, 19, 70, 16)),
])
def test_gradients_match_torch_autograd_fp64(oracle_mod, causal, shape):
    (qb, qv), (kb, kv), (vb, vv), (dob, dov) = make_case(3, *shape)
    scale = shape[-1] ** -0.5
    dq, dk, dv = oracle_mod.attn_bwd(qb, kb, vb, dob, causal, scale)
    rq, rk, rv = torch_reference_grads(qv, kv, vv, dov, causal, scale)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-12)


def test_single_key_closed_form(oracle_mod):
    """One key: O_i = v_0 whatever q and k are, so dQ = dK = 0 and dV_0 is the
    sum of dO over rows and over the query heads sharing the KV head."""
    (qb, _), (kb, _), (vb, _), (dob, dov) = make_case(5, 1, 4, 2, 6, 1, 8)
    dq, dk, dv = oracle_mod.attn_bwd(qb, kb, vb, dob, False, 0.7)
    assert np.all(dq == 0) and np.all(dk == 0)
    want = dov.reshape(1, 6, 2, 2, 8).sum(axis=(1, 3))  # [B, Hkv, d]
    np.testing.assert_allclose(dv[:, 0], want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_shift_and_normalisation_invariants(oracle_mod, causal):
    """Adding one vector to every key leaves O unchanged, so dK sums to zero
    over the keys of each (b, kv head); the weights of a row sum to one, so
    dV summed over the keys equals dO summed over the rows that see a key."""
    B, Hq, Hkv, Sq, Sk, d = 2, 4, 2, 21, 15, 16
    (qb, _), (kb, _), (vb, _), (dob, dov) = make_case(9, B, Hq, Hkv, Sq, Sk, d)
    dq, dk, dv = oracle_mod.attn_bwd(qb, kb, vb, dob, causal, 0.3)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-10)
    rows = np.arange(Sq)
    seen = (rows + Sk - Sq >= 0) if causal else np.ones(Sq, bool)
    want = dov[:, seen].reshape(B, -1, Hkv, Hq // Hkv, d).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), want, atol=1e-10)
    if causal:  # rows with no visible key get no gradient
        assert np.all(dq[:, ~seen] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_gradients_equal_the_whole(oracle_mod, causal):
    """The sampled form (used at sizes the whole oracle cannot finish) gives
    the whole computation's values at the sampled rows and keys."""
    B, Hq, Hkv, Sq, Sk, d = 2, 4, 2, 37, 53, 16
    (qb, _), (kb, _), (vb, _), (dob, _) = make_case(13, B, Hq, Hkv, Sq, Sk, d)
    dq, dk, dv = oracle_mod.attn_bwd(qb, kb, vb, dob, causal, 0.25)
    rng = np.random.default_rng(2)
    qrows = rng.choice(B * Hq * Sq, size=40, replace=False)
    krows = rng.choice(B * Hkv * Sk, size=30, replace=False)  # unsorted on purpose
    sq, sk, sv = oracle_mod.attn_bwd_sampled(qb, kb, vb, dob, causal, 0.25, qrows, krows)
    dq_flat = dq.transpose(0, 2, 1, 3).reshape(-1, d)  # (b, hq, i) order
    dk_flat = dk.transpose(0, 2, 1, 3).reshape(-1, d)
    dv_flat = dv.transpose(0, 2, 1, 3).reshape(-1, d)
    np.testing.assert_allclose(sq, dq_flat[qrows], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(sk, dk_flat[krows], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(sv, dv_flat[krows], rtol=1e-12, atol=1e-14)


def test_f16_gradients_equal_bf16_gradients_on_shared_values(oracle_mod):
    """Multiples of 1/256 up to +-200/256 are exact in both bf16 and fp16, so
    the backward pass's two 16-bit input paths (whole and sampled) must give
    identical gradients on them: the input type only changes the decoding."""
    B, Hq, Hkv, Sq, Sk, d = 1, 4, 2, 19, 23, 8
    (qb, qv), (kb, kv), (vb, vv), (dob, dov) = make_case(21, B, Hq, Hkv, Sq, Sk, d)
    as_f16 = [torch.tensor(x, dtype=torch.float16).view(torch.int16).numpy().view(np.uint16)
              for x in (qv, kv, vv, dov)]
    qrows = np.array([0, 5, B * Hq * Sq - 1])
    krows = np.array([1, 7, B * Hkv * Sk - 1])
    for causal in (False, True):
        got = oracle_mod.attn_bwd(*as_f16, causal, 0.4, dtype="f16")
        want = oracle_mod.attn_bwd(qb, kb, vb, dob, causal, 0.4, dtype="bf16")
        for g, w in zip(got, want):
            np.testing.assert_array_equal(g, w)
        got = oracle_mod.attn_bwd_sampled(*as_f16, causal, 0.4, qrows, krows, dtype="f16")
        want = oracle_mod.attn_bwd_sampled(qb, kb, vb, dob, causal, 0.4, qrows, krows,
                                           dtype="bf16")
        for g, w in zip(got, want):
            np.testing.assert_array_equal(g, w)
