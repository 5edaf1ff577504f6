"""Pins for the CPU oracle, checked against things other than itself:
hand-worked cases, closed forms, invariants, brute force on tiny inputs and
library routines. CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from exact_attention_forward_14_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    """Round an array to bf16 and return (uint16 bits, float64 values)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return inputs.bf16_bits(t), t.to(torch.float64).numpy()


def rand_case(rng, B, Hq, Hkv, Sq, Sk, d, scale_mag=1.0):
    q = rng.standard_normal((B, Sq, Hq, d)) * scale_mag
    k = rng.standard_normal((B, Sk, Hkv, d)) * scale_mag
    v = rng.standard_normal((B, Sk, Hkv, d))
    return bf16(q), bf16(k), bf16(v)


def brute_force(q, k, v, causal, scale):
    """Materialised softmax in plain Python floats: exp of the raw scores (no
    max subtraction, inputs are tiny), normalised after the fact."""
    B, Sq, Hq, d = q.shape
    _, Sk, Hkv, _ = k.shape
    g = Hq // Hkv
    o = np.zeros((B, Sq, Hq, d))
    lse = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            for i in range(Sq):
                weights = []
                for j in range(Sk):
                    if causal and j > i + Sk - Sq:
                        weights.append(0.0)
                        continue
                    s = sum(float(q[b, i, h, c]) * float(k[b, j, hk, c]) for c in range(d))
                    weights.append(math.exp(scale * s))
                z = sum(weights)
                if z == 0.0:
                    lse[b, h, i] = -math.inf
                    continue
                lse[b, h, i] = math.log(z)
                for c in range(d):
                    o[b, i, h, c] = sum(weights[j] * float(v[b, j, hk, c]) for j in range(Sk)) / z
    return o, lse


def test_hand_worked_golden(oracle_mod):
    with open(os.path.join(GOLDEN, "hand_worked_attention.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        shp_q = (c["B"], c["Sq"], c["Hq"], c["d"])
        shp_k = (c["B"], c["Sk"], c["Hkv"], c["d"])
        (qb, _), (kb, _), (vb, _) = (bf16(np.reshape(c["q"], shp_q)),
                                     bf16(np.reshape(c["k"], shp_k)),
                                     bf16(np.reshape(c["v"], shp_k)))
        o, lse = oracle_mod.attn_fwd(qb, kb, vb, c["causal"], c["scale"])
        np.testing.assert_allclose(o.ravel(), c["o"], rtol=0, atol=1e-12, err_msg=c["name"])
        want = np.array([-np.inf if x is None else x for x in c["lse"]])
        np.testing.assert_allclose(lse.ravel(), want, rtol=0, atol=1e-12, err_msg=c["name"])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 1, 1), (1, 2, 1, 3, 5, 2), (2, 4, 2, 8, 8, 4),
                                   (1, 3, 3, 7, 4, 3), (2, 2, 1, 4, 7, 4)])
def test_brute_force_tiny(oracle_mod, shape, causal):
    B, Hq, Hkv, Sq, Sk, d = shape
    rng = np.random.default_rng(7 + sum(shape))
    (qb, q), (kb, k), (vb, v) = rand_case(rng, B, Hq, Hkv, Sq, Sk, d)
    scale = 0.7
    o, lse = oracle_mod.attn_fwd(qb, kb, vb, causal, scale)
    o_ref, lse_ref = brute_force(q, k, v, causal, scale)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_single_key_gives_value_and_score(oracle_mod):
    rng = np.random.default_rng(1)
    (qb, q), (kb, k), (vb, v) = rand_case(rng, 2, 4, 2, 5, 1, 8)
    o, lse = oracle_mod.attn_fwd(qb, kb, vb, False, 0.3)
    for h in range(4):
        np.testing.assert_array_equal(o[:, :, h, :], v[:, 0:1, h // 2, :].repeat(5, axis=1))
        s = 0.3 * np.einsum("bid,bd->bi", q[:, :, h, :], k[:, 0, h // 2, :])
        np.testing.assert_allclose(lse[:, h, :], s, rtol=0, atol=1e-13)


def test_causal_first_row_is_first_value(oracle_mod):
    rng = np.random.default_rng(2)
    (qb, q), (kb, k), (vb, v) = rand_case(rng, 1, 2, 2, 33, 33, 16, scale_mag=3.0)
    o, lse = oracle_mod.attn_fwd(qb, kb, vb, True, 0.25)
    np.testing.assert_array_equal(o[:, 0], v[:, 0])
    np.testing.assert_allclose(lse[:, :, 0], 0.25 * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]),
                               rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_visible_values(oracle_mod, causal):
    rng = np.random.default_rng(3)
    Sq, Sk, d = 6, 9, 8
    (qb, q), _, (vb, v) = rand_case(rng, 1, 1, 1, Sq, Sk, d)
    krow = rng.standard_normal(d)
    kb, k = bf16(np.broadcast_to(krow, (1, Sk, 1, d)))
    o, lse = oracle_mod.attn_fwd(qb, kb, vb, causal, 0.5)
    for i in range(Sq):
        n = min(Sk, i + Sk - Sq + 1) if causal else Sk
        np.testing.assert_allclose(o[0, i, 0], v[0, :n, 0].mean(axis=0), rtol=0, atol=1e-13)
        s = 0.5 * float(q[0, i, 0] @ k[0, 0, 0])
        np.testing.assert_allclose(lse[0, 0, i], s + math.log(n), rtol=0, atol=1e-13)


def test_zero_query_gives_uniform_weights(oracle_mod):
    rng = np.random.default_rng(4)
    _, (kb, k), (vb, v) = rand_case(rng, 1, 1, 1, 4, 11, 8)
    qb, _ = bf16(np.zeros((1, 4, 1, 8)))
    o, lse = oracle_mod.attn_fwd(qb, kb, vb, False, 1.0)
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(v[0, :, 0].mean(0), (4, 8)), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(11), atol=1e-13)


def test_joint_permutation_of_keys_and_values(oracle_mod):
    rng = np.random.default_rng(5)
    (qb, q), (kb, k), (vb, v) = rand_case(rng, 2, 2, 1, 7, 19, 8)
    perm = rng.permutation(19)
    o1, l1 = oracle_mod.attn_fwd(qb, kb, vb, False, 0.4)
    o2, l2 = oracle_mod.attn_fwd(qb, kb[:, perm], vb[:, perm], False, 0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
    # ...and a permutation of K alone changes the result (the pin can fail).
    o3, _ = oracle_mod.attn_fwd(qb, kb[:, perm], vb, False, 0.4)
    assert np.abs(o3 - o1).max() > 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_on_duplicated_kv_heads(oracle_mod, causal):
    rng = np.random.default_rng(6)
    (qb, q), (kb, k), (vb, v) = rand_case(rng, 2, 8, 2, 10, 12, 8)
    o1, l1 = oracle_mod.attn_fwd(qb, kb, vb, causal, 0.35)
    kdup = np.repeat(kb, 4, axis=2)  # head h of the copy = KV head h // 4
    vdup = np.repeat(vb, 4, axis=2)
    o2, l2 = oracle_mod.attn_fwd(qb, kdup, vdup, causal, 0.35)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_scaling_q_equals_scaling_scale(oracle_mod):
    rng = np.random.default_rng(8)
    (qb, q), (kb, k), (vb, v) = rand_case(rng, 1, 2, 2, 9, 9, 8)
    q2b, _ = bf16(q * 2.0)  # power of two: exact in bf16
    o1, l1 = oracle_mod.attn_fwd(qb, kb, vb, True, 0.6)
    o2, l2 = oracle_mod.attn_fwd(q2b, kb, vb, True, 0.3)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("sq_sk", [(33, 33), (17, 40), (40, 17)])
def test_matches_torch_sdpa_fp64(oracle_mod, causal, sq_sk):
    """Library cross-check: torch's scaled_dot_product_attention in fp64 on the
    CPU, with an explicit bottom-right causal mask, plus torch.logsumexp."""
    Sq, Sk = sq_sk
    rng = np.random.default_rng(9)
    (qb, q), (kb, k), (vb, v) = rand_case(rng, 2, 4, 2, Sq, Sk, 16)
    scale = 1 / 4
    o, lse = oracle_mod.attn_fwd(qb, kb, vb, causal, scale)
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(np.repeat(k, 2, axis=2)).permute(0, 2, 1, 3)
    tv = torch.from_numpy(np.repeat(v, 2, axis=2)).permute(0, 2, 1, 3)
    i = torch.arange(Sq)[:, None]
    j = torch.arange(Sk)[None, :]
    mask = (j <= i + Sk - Sq) if causal else torch.ones(Sq, Sk, dtype=torch.bool)
    scores = (tq @ tk.transpose(-1, -2)) * scale
    scores = scores.masked_fill(~mask, -math.inf)
    ref_lse = torch.logsumexp(scores, dim=-1)
    visible = mask.any(dim=-1)
    ref_o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=mask | ~visible[:, None], scale=scale)
    ref_o = ref_o.masked_fill(~visible[None, None, :, None], 0.0).permute(0, 2, 1, 3)
    np.testing.assert_allclose(o, ref_o.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


def test_row_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(10)
    (qb, _), (kb, _), (vb, _) = rand_case(rng, 2, 4, 2, 21, 21, 8)
    o, lse = oracle_mod.attn_fwd(qb, kb, vb, True, 0.5)
    rows = inputs.sample_rows(2, 4, 21, 25, seed=0)
    o_s, lse_s = oracle_mod.attn_fwd(qb, kb, vb, True, 0.5, rows=rows)
    b, rem = np.divmod(rows, 4 * 21)
    h, i = np.divmod(rem, 21)
    np.testing.assert_array_equal(o_s, o[b, i, h])
    np.testing.assert_array_equal(lse_s, lse[b, h, i])


# ------------------------------------------------------------- E4M3 codec --

def test_e4m3_decode_known_codes(oracle_mod):
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0, 0x80: -0.0}
    got = oracle_mod.e4m3_decode(np.array(list(table), dtype=np.uint8))
    np.testing.assert_array_equal(got, np.array(list(table.values())))
    assert np.isnan(oracle_mod.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_decode_matches_torch(oracle_mod):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle_mod.e4m3_decode(codes), ref)


def _nearest_even_brute(x):
    """Nearest finite E4M3 value by exhaustive search; ties to the even code."""
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    vals = {c: (-1.0 if c & 0x80 else 1.0) * (
        (c & 7) * 2.0 ** -9 if (c >> 3) & 15 == 0 else (1 + (c & 7) / 8) * 2.0 ** (((c >> 3) & 15) - 7))
        for c in codes}
    if abs(x) >= 448:
        return 0x7E | (0x80 if x < 0 else 0)
    best = min(codes, key=lambda c: (abs(vals[c] - x), c & 1, -(c & 0x80 == (0x80 if x < 0 else 0))))
    return best


def test_e4m3_encode_matches_brute_force_and_torch(oracle_mod):
    rng = np.random.default_rng(11)
    finite = oracle_mod.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (finite[1:] + finite[:-1]) / 2  # exact ties (all representable in fp32)
    x = np.concatenate([finite, mids, -mids, rng.standard_normal(2000) * 40,
                        rng.standard_normal(500) * 0.01, [0.0, 447.9, 448.0, 460.0, 470.0, 1e6]])
    x = x.astype(np.float32)
    got = oracle_mod.e4m3_encode(x)
    brute = np.array([_nearest_even_brute(float(v)) for v in x], dtype=np.uint8)
    # compare values (the sign of zero aside)
    np.testing.assert_array_equal(oracle_mod.e4m3_decode(got), oracle_mod.e4m3_decode(brute))
    inrange = np.abs(x) <= 448
    ref = torch.from_numpy(x[inrange]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got[inrange], ref)
    assert oracle_mod.e4m3_decode(got[~inrange]).tolist() == [448.0] * int((~inrange).sum())


# -------------------------------------------------------- FP8 quantiser --

def test_quantiser_block_scales_and_codes(oracle_mod):
    rng = np.random.default_rng(12)
    B, S, H, d = 2, 150, 3, 16  # 3 blocks of 64 rows, the last one ragged (22 rows)
    x = rng.standard_normal((B, S, H, d)).astype(np.float32)
    x[1, 64:128, 2, :] = 0.0  # an all-zero block
    codes, scales = oracle_mod.quantize_fp8_e4m3(x)
    assert scales.shape == (B, H, 3)
    for b in range(B):
        for h in range(H):
            for blk in range(3):
                xs = x[b, blk * 64:(blk + 1) * 64, h, :]
                amax = np.float32(np.abs(xs).max())
                s = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))
                assert scales[b, h, blk] == s
                cs = codes[b, blk * 64:(blk + 1) * 64, h, :]
                if amax == 0:
                    assert (cs == 0).all()
                    continue
                # the block maximum lands on the largest code (|x|/s rounds to 448)
                at = np.unravel_index(np.abs(xs).argmax(), xs.shape)
                assert cs[at] & 0x7F == 0x7E
                deq = oracle_mod.e4m3_decode(cs) * float(s)
                err = np.abs(deq - xs)
                # half a unit in the last place: 2^-4 relative for normals,
                # 2^-10 * s absolute in the subnormal range
                bound = np.maximum(np.abs(xs) * 2.0 ** -4, 2.0 ** -10 * float(s))
                assert (err <= bound * (1 + 1e-6)).all()


def test_fp8_attention_equals_bf16_attention_on_dequantised_values(oracle_mod):
    """With power-of-two block scales, every dequantised value is exact in
    bf16, so the E4M3 input path must agree with the bf16 input path."""
    rng = np.random.default_rng(13)
    B, H, S, d = 1, 2, 130, 8
    nblk = 3
    codes = [rng.integers(0, 0x7E, size=(B, S, H, d), dtype=np.uint8) |
             (rng.integers(0, 2, size=(B, S, H, d), dtype=np.uint8) << 7) for _ in range(3)]
    scales = [np.exp2(rng.integers(-4, 3, size=(B, H, nblk))).astype(np.float32) for _ in range(3)]
    deq = []
    for c, s in zip(codes, scales):
        rows_blk = np.arange(S) // 64
        val = oracle_mod.e4m3_decode(c) * s[:, :, rows_blk].transpose(0, 2, 1)[..., None]
        deq.append(bf16(val))
    for causal in (False, True):
        o8, l8 = oracle_mod.attn_fwd(*codes, causal, 0.2, dtype="e4m3", q_scale=scales[0],
                                     k_scale=scales[1], v_scale=scales[2])
        o16, l16 = oracle_mod.attn_fwd(deq[0][0], deq[1][0], deq[2][0], causal, 0.2)
        np.testing.assert_array_equal(deq[0][1], oracle_mod.e4m3_decode(codes[0]) *
                                      scales[0][:, :, np.arange(S) // 64].transpose(0, 2, 1)[..., None])
        np.testing.assert_allclose(o8, o16, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l8, l16, rtol=0, atol=1e-12)


# ------------------------------------------------------------ fp16 inputs --

def test_f16_decode_known_values(oracle_mod):
    """Values fixed by the binary16 definition: 1, the smallest subnormal
    2^-24, the largest finite 65504, signed zero and infinity."""
    table = {0x3C00: 1.0, 0x0001: 2.0 ** -24, 0x0400: 2.0 ** -14, 0x7BFF: 65504.0,
             0xC000: -2.0, 0x8000: -0.0, 0x3555: 1365 / 4096, 0x7C00: np.inf, 0xFC00: -np.inf}
    got = oracle_mod.f16_decode(np.array(list(table), dtype=np.uint16))
    np.testing.assert_array_equal(got, np.array(list(table.values())))
    assert np.isnan(oracle_mod.f16_decode(np.array([0x7E00, 0xFC01], dtype=np.uint16))).all()


def test_f16_decode_matches_torch_on_every_pattern(oracle_mod):
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    got = oracle_mod.f16_decode(bits)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_f16_attention_equals_bf16_attention_on_shared_values(oracle_mod):
    """Multiples of 1/16 up to +-7.9375 are exact in both bf16 and fp16, so the
    two 16-bit input paths must give identical results on them."""
    rng = np.random.default_rng(17)
    B, Hq, Hkv, S, d = 2, 4, 2, 37, 8
    vals = [rng.integers(-127, 128, size=(B, S, h, d)) / 16.0 for h in (Hq, Hkv, Hkv)]
    as_f16 = [torch.tensor(v, dtype=torch.float16).view(torch.int16).numpy().view(np.uint16)
              for v in vals]
    as_bf16 = [torch.tensor(v, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
               for v in vals]
    for causal in (False, True):
        o_h, l_h = oracle_mod.attn_fwd(*as_f16, causal, 0.3, dtype="f16")
        o_b, l_b = oracle_mod.attn_fwd(*as_bf16, causal, 0.3, dtype="bf16")
        np.testing.assert_array_equal(o_h, o_b)
        np.testing.assert_array_equal(l_h, l_b)


# ------------------------------------------------- merge across key ranges --

def test_merging_key_ranges_reproduces_the_whole(oracle_mod):
    """The split-KV combine formula, checked on the oracle itself: attention
    over keys [0, c) and [c, Sk) separately, merged with
    LSE = ln(e^LSE1 + e^LSE2), O = e^(LSE1 - LSE) O1 + e^(LSE2 - LSE) O2,
    equals attention over all keys (non-causal; the causal mask is a per-row
    key range, covered by the GPU tests against the unsplit oracle)."""
    rng = np.random.default_rng(23)
    B, Hq, Hkv, Sq, Sk, d = 1, 4, 2, 9, 40, 8
    q, k, v = (bf16(rng.standard_normal(s) * 2)[0] for s in
               ((B, Sq, Hq, d), (B, Sk, Hkv, d), (B, Sk, Hkv, d)))
    o, lse = oracle_mod.attn_fwd(q, k, v, False, 0.4)
    for c in (1, 13, 39):
        o1, l1 = oracle_mod.attn_fwd(q, k[:, :c], v[:, :c], False, 0.4)
        o2, l2 = oracle_mod.attn_fwd(q, k[:, c:], v[:, c:], False, 0.4)
        lm = np.logaddexp(l1, l2)
        w1 = np.exp(l1 - lm).transpose(0, 2, 1)[..., None]
        w2 = np.exp(l2 - lm).transpose(0, 2, 1)[..., None]
        np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-12)
        np.testing.assert_allclose(w1 * o1 + w2 * o2, o, rtol=0, atol=1e-12)


# ----------------------------------------------------- QK RMSNorm (heads) --

def _bits(x, dtype):
    t = torch.tensor(np.asarray(x, dtype=np.float32),
                     dtype=torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t.to(torch.float64).numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rmsnorm_heads_brute_force(oracle_mod, dtype):
    rng = np.random.default_rng(31)
    T, H, d, eps = 5, 3, 4, 1e-6
    xb, xv = _bits(rng.standard_normal((T, H, d)) * 3, dtype)
    wb, wv = _bits(rng.standard_normal(H * d), dtype)
    y = oracle_mod.rmsnorm_heads(xb, wb, eps, dtype)
    for t in range(T):
        vals = [float(v) for v in xv[t].ravel()]
        r = 1.0 / math.sqrt(eps + sum(v * v for v in vals) / len(vals))
        want = [vals[i] * r * float(wv[i]) for i in range(len(vals))]
        np.testing.assert_allclose(y[t].ravel(), want, rtol=1e-13, atol=0)


def test_rmsnorm_heads_closed_forms(oracle_mod):
    # a constant row c with unit weights and eps = 0 normalises to sign(c)
    xb, _ = _bits(np.full((2, 4, 8), -2.5), "bf16")
    wb, _ = _bits(np.ones(32), "bf16")
    np.testing.assert_array_equal(oracle_mod.rmsnorm_heads(xb, wb, 0.0), -np.ones((2, 4, 8)))
    # with unit weights and eps = 0 every row has mean square 1, whatever its scale
    rng = np.random.default_rng(5)
    for s in (1e-3, 1.0, 300.0):
        xb, _ = _bits(rng.standard_normal((3, 2, 64)) * s, "bf16")
        wb, _ = _bits(np.ones(128), "bf16")
        y = oracle_mod.rmsnorm_heads(xb, wb, 0.0)
        np.testing.assert_allclose((y ** 2).mean(axis=(1, 2)), 1.0, rtol=1e-12)


def test_rmsnorm_heads_spans_all_heads(oracle_mod):
    """Across heads, not per head: scaling one head's values changes the
    normalisation of every head in the token."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((1, 4, 16))
    wb, _ = _bits(np.ones(64), "bf16")
    y0 = oracle_mod.rmsnorm_heads(_bits(x, "bf16")[0], wb, 1e-6)
    x2 = x.copy()
    x2[0, 0] *= 4.0  # exact in bf16
    y1 = oracle_mod.rmsnorm_heads(_bits(x2, "bf16")[0], wb, 1e-6)
    ratio = y1[0, 1:] / y0[0, 1:]
    assert np.allclose(ratio, ratio.flat[0]) and ratio.flat[0] < 0.9
