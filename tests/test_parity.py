"""GPU parity: the CUDA attention path against the fp64 CPU oracle, on the
same seeded inputs, through the C ABI. Small shapes, the B4 H16 S2048 causal
workload and a medium shape that takes the kernel's default pair-order
schedule are compared element by element in full; the long-context workloads
(run in the launch configuration the benchmark times) on three rows of every
(batch, head, 128-row query tile): its first, its last and one at random, so
every work item the kernel runs is checked. Every case records its strict
error figures for the end-of-run report."""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import (assert_lse_close, assert_o_close, bf16_atol, o_error_stats, record,
                           require_gpu, ulp16)

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
    st = assert_o_close(o, o_ref)
    record("small b{}hq{}hkv{}sq{}sk{}d{}{}".format(*shape[:6], "c" if causal else ""), "bf16",
           st, assert_lse_close(lse, lse_ref), B * Hq * Sq)


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


def _compare_rows(oracle_mod, torch, w, q, k, v, o, lse, rows, case, kind="bf16"):
    """O and LSE of the listed flat rows (b*Hq + hq)*Sq + i against the oracle."""
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         w.causal, w.scale, dtype="f16" if kind == "f16" else "bf16",
                                         rows=rows)
    b, rem = np.divmod(rows, w.Hq * w.Sq)
    h, i = np.divmod(rem, w.Sq)
    o_g = o[torch.as_tensor(b), torch.as_tensor(i), torch.as_tensor(h)].float().cpu().numpy()
    l_g = lse.cpu().numpy()[b, h, i]
    st = assert_o_close(o_g, o_ref, kind=kind)
    record(case, kind, st, assert_lse_close(l_g, lse_ref), len(rows))


def _run_workload(w):
    torch = require_gpu()
    q, k, v = inputs.draw_workload_16(w)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    assert torch.isfinite(lse[lse != float("-inf")]).all() and torch.isfinite(o.float()).all()
    return torch, q, k, v, o, lse


@pytest.mark.gpu
def test_tiny_workload_full(oracle_mod):
    w = inputs.WORKLOADS["tiny_b1h1s128d64"]
    torch = require_gpu()
    q, k, v = inputs.draw_qkv_bf16(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.seed)
    o, lse = run_bf16(torch, q, k, v, w.causal, w.scale)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), w.causal, w.scale)
    st = assert_o_close(o, o_ref)
    record(w.name + " (full)", "bf16", st, assert_lse_close(lse, lse_ref), w.B * w.Hq * w.Sq)


@pytest.mark.gpu
def test_b4h16s2048_causal_full_compare(oracle_mod):
    """Every element of the B4 H16 S2048 causal workload (single-unit snake
    order: 512 units on the SMs)."""
    w = inputs.WORKLOADS["b4h16s2048d128_causal"]
    torch, q, k, v, o, lse = _run_workload(w)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), w.causal, w.scale)
    st = assert_o_close(o.float().cpu().numpy(), o_ref)
    record(w.name + " (full)", "bf16", st, assert_lse_close(lse.cpu().numpy(), lse_ref),
           w.B * w.Hq * w.Sq)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["b2h32s8192d128_causal", "b2h32s8192d128",
                                  "gqa_b1hq32hkv8s16384d128_causal", "d64_b2h64s8192_causal"])
def test_full_size_workloads_every_tile(oracle_mod, name):
    """The long-context workloads in the benchmark's launch configuration
    (pair-order schedule): the first, the last and one random row of every
    (b, hq, 128-row Q tile)."""
    w = inputs.WORKLOADS[name]
    torch, q, k, v, o, lse = _run_workload(w)
    rows = inputs.stratified_rows(w.B, w.Hq, w.Sq, 128, seed=w.seed)
    _compare_rows(oracle_mod, torch, w, q, k, v, o, lse, rows, w.name + " (every Q tile)")


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [True, False])
def test_pair_order_schedule_medium_shape_full(oracle_mod, causal):
    """A shape with exactly 4 work items per SM, so the host picks the
    default pair order (heavy level + its mirror per item) rather than the
    single-unit order small problems get; S = 640 gives an odd number of
    256-row levels (3), so one item per head runs the middle level alone;
    GQA with 4 query heads per KV head. Compared in full."""
    torch = require_gpu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hkv = sms // 2 if sms % 2 == 0 else sms
    Hq, S, d = 2 * sms, 640, 128
    n_qp = -(-S // 256)
    items = Hq * ((n_qp + 1) // 2)
    assert n_qp % 2 == 1 and items >= 4 * sms  # the pair-order branch of the launch
    q, k, v = inputs.draw_qkv_bf16(1, Hq, Hkv, S, S, d, seed=640 + causal)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_bf16(torch, q, k, v, causal, scale)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), causal, scale)
    st = assert_o_close(o, o_ref)
    record(f"pair order b1hq{Hq}hkv{Hkv}s{S}{'c' if causal else ''} (full)", "bf16", st,
           assert_lse_close(lse, lse_ref), Hq * S)


# ----------------------------------------- steep scores: P's bf16 rounding --
# (B, Hq, Hkv, Sq, Sk, d, causal) at scale 0.3, several times 1/sqrt(d): rows
# are nearly one-hot, the regime where rounding P to bf16 shows most.
STEEP = [
    (1, 4, 2, 640, 640, 256, False),
    (1, 4, 1, 1000, 1000, 128, True),
    (2, 2, 2, 700, 900, 64, True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", STEEP, ids=lambda s: "steep_b{}hq{}hkv{}sq{}sk{}d{}{}".format(
    *s[:6], "c" if s[6] else ""))
def test_bf16_steep_scores_within_the_p_rounding_bound(oracle_mod, shape):
    """P enters P.V rounded to bf16 (relative error |delta_j| <= 2^-8) while
    the normaliser l sums the unrounded p, so before its own rounding the
    kernel's O is O + sum_j w_j delta_j v_j, with w_j = p_j / l. That moves O
    by at most 2^-8 A, A = sum_j w_j |v_j| (the attention of |V|, which the
    oracle computes exactly from |V|, itself exact in bf16); O's rounding to
    bf16 adds half an ulp. The bound checked is exactly that sum (plus 1e-5
    for the fp32 accumulations): it can exceed both the plain 1e-2 floor and
    one ulp when a row is carried by one key with |v| near the top of its
    binade. The strict figures are recorded; the plain gate is not applied."""
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = inputs.draw_qkv_bf16(B, Hq, Hkv, Sq, Sk, d, seed=sum(shape) + 53)
    scale = 0.3
    o, lse = run_bf16(torch, q, k, v, causal, scale)
    qb, kb = inputs.bf16_bits(q), inputs.bf16_bits(k)
    o_ref, lse_ref = oracle_mod.attn_fwd(qb, kb, inputs.bf16_bits(v), causal, scale)
    a_ref, _ = oracle_mod.attn_fwd(qb, kb, inputs.bf16_bits(v.abs()), causal, scale)
    drift = 2.0 ** -8 * np.asarray(a_ref, dtype=np.float64)
    bound = drift + 0.5 * ulp16(np.abs(o_ref) + drift, 7) + 1e-5
    err = np.abs(np.asarray(o, dtype=np.float64) - o_ref)
    bad = err > bound
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} past the P-rounding bound; max err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    record("steep scale 0.3 b{}hq{}hkv{}sq{}sk{}d{}{}".format(*shape[:6], "c" if causal else ""),
           "bf16", o_error_stats(o, o_ref), assert_lse_close(lse, lse_ref), B * Hq * Sq,
           note="gate: 2^-8 A + half an ulp (P rounding bound), not max(1e-2, 1 ulp)")


# ------------------------------------------------- d = 64, medium shapes --
# (B, Hq, Hkv, Sq, Sk, d, causal): several 256-row units per head, Q and K/V
# tails inside a unit, causal Sq > Sk (rows with no visible key) and Sq < Sk,
# GQA, and one head long enough for the causal tile skip to matter.
D64_SHAPES = [
    (1, 2, 2, 1100, 1100, 64, True),
    (2, 3, 1, 700, 1000, 64, False),
    (1, 2, 2, 1000, 700, 64, True),
    (1, 2, 2, 600, 1500, 64, True),
    (1, 1, 1, 2048, 2048, 64, True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", D64_SHAPES, ids=lambda s: "d64_b{}hq{}hkv{}sq{}sk{}{}".format(
    *s[:5], "c" if s[6] else ""))
def test_d64_medium_shapes_full_compare(oracle_mod, shape):
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d, causal = shape
    q, k, v = inputs.draw_qkv_bf16(B, Hq, Hkv, Sq, Sk, d, seed=sum(shape) + 41)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_bf16(torch, q, k, v, causal, scale)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), causal, scale)
    st = assert_o_close(o, o_ref)
    record("d64 units b{}hq{}hkv{}sq{}sk{}{}".format(*shape[:5], "c" if causal else ""), "bf16",
           st, assert_lse_close(lse, lse_ref), B * Hq * Sq)


@pytest.mark.gpu
def test_d64_pair_order_schedule_full(oracle_mod):
    """d = 64 with at least 4 work items per SM, so the host picks the pair
    order; S = 1100 gives an odd number of 256-row levels (5), so one item
    per head runs the middle level alone. Compared in full."""
    torch = require_gpu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hq, S, d = 2 * sms, 1100, 64
    Hkv = Hq // 2
    n_qp = -(-S // 256)
    assert n_qp % 2 == 1 and Hq * ((n_qp + 1) // 2) >= 4 * sms
    q, k, v = inputs.draw_qkv_bf16(1, Hq, Hkv, S, S, d, seed=1100)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_bf16(torch, q, k, v, True, scale)
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bf16_bits(q), inputs.bf16_bits(k),
                                         inputs.bf16_bits(v), True, scale)
    st = assert_o_close(o, o_ref)
    record(f"d64 pair order b1hq{Hq}hkv{Hkv}s{S}c (full)", "bf16", st,
           assert_lse_close(lse, lse_ref), Hq * S)


# ------------------------------------------------------------ fp16 inputs --
# (B, Hq, Hkv, Sq, Sk, d, causal): d = 64 and 128, GQA, ragged tails, Sq != Sk
SMALL_F16 = [
    (1, 2, 2, 128, 128, 128, False),
    (1, 2, 2, 1100, 900, 64, True),
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
    st = assert_o_close(o.float().cpu().numpy(), o_ref, kind="f16")
    record("small f16 b{}hq{}hkv{}sq{}sk{}d{}{}".format(*shape[:6], "c" if causal else ""), "f16",
           st, assert_lse_close(lse.cpu().numpy(), lse_ref), B * Hq * Sq)


@pytest.mark.gpu
def test_f16_full_size_every_tile(oracle_mod):
    w = inputs.WORKLOADS["f16_b2h32s8192d128_causal"]
    torch, q, k, v, o, lse = _run_workload(w)
    assert o.dtype == torch.float16
    rows = inputs.stratified_rows(w.B, w.Hq, w.Sq, 128, seed=w.seed)
    _compare_rows(oracle_mod, torch, w, q, k, v, o, lse, rows, w.name + " (every Q tile)",
                  kind="f16")


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
