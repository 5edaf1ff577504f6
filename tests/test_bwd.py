"""GPU parity of the attention backward pass (dQ, dK, dV) against the fp64
oracle, through the C ABI.

Tolerance, per gradient tensor (derived from the arithmetic: the kernels
round P and dS to the input type before the tensor cores, accumulate in
fp32 and round the gradients to the input type; a numpy emulation of exactly
those roundings on these inputs stays below a quarter of both bounds):
  element-wise   |got - ref| <= 2^-7 |ref| + 0.01 max|ref|
                 (half an ulp of bf16 output rounding is <= 2^-8 |ref|; the
                 emulated residual beyond it is <= 0.0036 max|ref|)
  aggregate      ||got - ref||_2 <= 0.01 ||ref||_2
                 (the emulation gives 0.0024, the level of output rounding;
                 a skipped tile or a wrong mask raises it well above 0.01)
The upstream gradient dO is N(0, 1); O and LSE come from this library's own
forward pass, as they would in training."""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import require_gpu

REL = 2.0 ** -7
ABS_OF_MAX = 0.01
AGG = 0.01


def assert_grad_close(name, got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), f"{name}: non-finite gradient"
    err = np.abs(got - ref)
    mx = float(np.abs(ref).max()) if ref.size else 0.0
    tol = REL * np.abs(ref) + ABS_OF_MAX * mx
    bad = err > tol
    assert not bad.any(), (f"{name}: {int(bad.sum())} of {bad.size} outside tolerance; max err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}, "
                           f"max|ref| {mx:.3e}")
    nref = float(np.sqrt(np.sum(ref * ref)))
    if nref > 0:
        agg = float(np.sqrt(np.sum(err * err))) / nref
        assert agg <= AGG, f"{name}: relative 2-norm error {agg:.3e}"


def run_case(torch, B, Hq, Hkv, Sq, Sk, d, causal, dtype, seed):
    draw = inputs.draw_qkv_f16 if dtype == "f16" else inputs.draw_qkv_bf16
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, d, seed=seed)
    do = inputs.draw_grad_out(B, Sq, Hq, d, seed, dtype=dtype)
    scale = 1.0 / np.sqrt(d)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = ea.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    return (q, k, v, do, scale), (dq.float().cpu().numpy(), dk.float().cpu().numpy(),
                                  dv.float().cpu().numpy())


# (B, Hq, Hkv, Sq, Sk, d, causal, dtype)
CASES = [
    (1, 2, 2, 300, 300, 128, True, "bf16"),     # ragged last tiles, diagonal masks
    (2, 2, 2, 256, 256, 128, False, "bf16"),    # whole tiles, two batches
    (1, 4, 1, 700, 1100, 64, True, "bf16"),     # GQA 4:1, Sq < Sk, d = 64
    (1, 2, 1, 1100, 700, 128, True, "bf16"),    # Sq > Sk: early rows see no key
    (1, 2, 2, 129, 257, 128, False, "bf16"),    # one row / key past a tile edge
    (1, 8, 2, 520, 520, 128, True, "bf16"),     # GQA 4:1, several units per CTA row
    (1, 2, 2, 300, 300, 128, True, "f16"),      # fp16
    (1, 4, 2, 200, 333, 64, False, "f16"),      # fp16, d = 64, GQA
    (1, 1, 1, 1, 1, 64, False, "bf16"),         # one query, one key
    (1, 1, 1, 1, 1000, 128, True, "bf16"),      # one query row (decode), causal
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}hq{}hkv{}sq{}sk{}d{}{}_{}".format(
    *c[:6], "c" if c[6] else "", c[7]))
def test_backward_matches_oracle(oracle_mod, case):
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d, causal, dtype = case
    (q, k, v, do, scale), (dq, dk, dv) = run_case(torch, *case, seed=sum(case[:6]) + 77)
    rq, rk, rv = oracle_mod.attn_bwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                     inputs.bits16(do), causal, scale, dtype=dtype)
    assert_grad_close("dq", dq, rq)
    assert_grad_close("dk", dk, rk)
    assert_grad_close("dv", dv, rv)


@pytest.mark.gpu
def test_backward_is_deterministic():
    """Every output element is written once by one thread (no atomics): two
    calls give identical bits."""
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d = 1, 8, 2, 1000, 1000, 128
    q, k, v = (t.cuda() for t in inputs.draw_qkv_bf16(B, Hq, Hkv, Sq, Sk, d, seed=3))
    do = inputs.draw_grad_out(B, Sq, Hq, d, 3).cuda()
    o, lse = ea.forward(q, k, v, causal=True)
    g1 = ea.backward(q, k, v, o, lse, do, causal=True)
    g2 = ea.backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


@pytest.mark.gpu
def test_backward_results_are_complete_on_the_callers_stream():
    """dK/dV and dQ run side by side, dQ on a second stream of the library's
    that is forked from the caller's stream and joined back into it. Work
    enqueued on the caller's stream right after the call, with no host
    synchronisation in between, must see all three gradients complete: the
    outputs start as NaN, the call is queued behind a long fill so that it
    runs while the host has already enqueued the copies, and the copies must
    equal a separately synchronised call bit for bit."""
    torch = require_gpu()
    B, Hq, Hkv, S, d = 1, 16, 4, 4096, 128
    q, k, v = (t.cuda() for t in inputs.draw_qkv_bf16(B, Hq, Hkv, S, S, d, seed=17))
    do = inputs.draw_grad_out(B, S, Hq, d, 17).cuda()
    o, lse = ea.forward(q, k, v, causal=True)
    ref = ea.backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        out = tuple(torch.full_like(t, float("nan")) for t in ref)
        busy = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
        busy.fill_(1)
        g = ea.backward(q, k, v, o, lse, do, causal=True, out=out, stream=side)
        copies = tuple(t.clone() for t in g)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    for name, got, want in zip(("dq", "dk", "dv"), copies, ref):
        assert torch.equal(got, want), name


@pytest.mark.gpu
def test_gqa_equals_mha_on_repeated_kv_heads():
    """Property at any size: with each KV head repeated for its query heads,
    MHA's dK / dV summed over each group equal the GQA gradients (up to the
    rounding of the sum), and dQ is the same."""
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d = 1, 8, 2, 640, 640, 128
    q, k, v = (t.cuda() for t in inputs.draw_qkv_bf16(B, Hq, Hkv, Sq, Sk, d, seed=21))
    do = inputs.draw_grad_out(B, Sq, Hq, d, 21).cuda()
    g = Hq // Hkv
    kr, vr = (t.repeat_interleave(g, dim=2).contiguous() for t in (k, v))
    o1, l1 = ea.forward(q, k, v, causal=True)
    o2, l2 = ea.forward(q, kr, vr, causal=True)
    dq1, dk1, dv1 = ea.backward(q, k, v, o1, l1, do, causal=True)
    dq2, dk2, dv2 = ea.backward(q, kr, vr, o2, l2, do, causal=True)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    assert torch.equal(dq1, dq2)
    dk2s = dk2.float().view(B, Sk, Hkv, g, d).sum(3)
    dv2s = dv2.float().view(B, Sk, Hkv, g, d).sum(3)
    for a, b in ((dk1.float(), dk2s), (dv1.float(), dv2s)):
        tol = 2.0 ** -7 * b.abs() + 0.01 * b.abs().max()
        assert bool(((a - b).abs() <= tol).all())


@pytest.mark.gpu
@pytest.mark.parametrize("name,nkv", [("bwd_b2h32s8192d128_causal", 2),
                                      ("bwd_gqa_b1hq32hkv8s16384d128_causal", 1)])
def test_backward_full_size_sampled(oracle_mod, name, nkv):
    """The bench's workloads at full size, in the bench's launch configuration:
    dQ at sampled query rows (the first and last rows of the first and last
    heads included) and dK, dV at sampled keys of nkv (batch, KV head) pairs
    (the first and last keys included), against the sampled oracle. The
    tolerance's max|ref| is taken over the sample, which holds the largest
    gradients (the first rows and keys under the causal mask)."""
    torch = require_gpu()
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.draw_workload_16(w)
    do = inputs.draw_grad_out(w.B, w.Sq, w.Hq, w.d, w.seed, w.dtype)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = ea.forward(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, causal=w.causal, scale=w.scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    del o, lse, qd, kd, vd, dod
    qrows = inputs.sample_rows(w.B, w.Hq, w.Sq, 48, seed=w.seed + 7)
    rng = np.random.default_rng(w.seed + 8)
    pairs = [0, w.B * w.Hkv - 1][:nkv]
    krows = []
    for bhk in pairs:
        keys = set(int(x) for x in rng.choice(w.Sk, size=22, replace=False)) | {0, w.Sk - 1}
        krows += [bhk * w.Sk + j for j in sorted(keys)]
    krows = np.array(krows, dtype=np.int64)
    rq, rk, rv = oracle_mod.attn_bwd_sampled(inputs.bits16(q), inputs.bits16(k),
                                             inputs.bits16(v), inputs.bits16(do), w.causal,
                                             w.scale, qrows, krows, dtype=w.dtype)

    def gather(t, rows, H, S):  # flat (b*H + h)*S + s -> [n, d]
        bh, s = rows // S, rows % S
        b, h = bh // H, bh % H
        return t[torch.as_tensor(b), torch.as_tensor(s), torch.as_tensor(h)].float().cpu().numpy()

    assert_grad_close("dq", gather(dq, qrows, w.Hq, w.Sq), rq)
    assert_grad_close("dk", gather(dk, krows, w.Hkv, w.Sk), rk)
    assert_grad_close("dv", gather(dv, krows, w.Hkv, w.Sk), rv)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_backward_long_key_side(oracle_mod, causal):
    """Sq = 256 against Sk = 131072 (1024 key tiles, GQA 4:1): dQ at sampled
    rows and dK, dV at sampled keys (the first and last keys included; under
    the bottom-right causal mask every key is seen by some row)."""
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d = 1, 4, 1, 256, 131072, 128
    q, k, v = inputs.draw_qkv_bf16(B, Hq, Hkv, Sq, Sk, d, seed=31)
    do = inputs.draw_grad_out(B, Sq, Hq, d, 31)
    scale = d ** -0.5
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = ea.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = ea.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    assert ea.attn_device_status() == ea.ATTN_OK
    qrows = inputs.sample_rows(B, Hq, Sq, 24, seed=5)
    rng = np.random.default_rng(6)
    krows = np.array(sorted(set(int(x) for x in rng.choice(Sk, size=30, replace=False)) |
                            {0, Sk - 1, Sk - Sq, Sk - 1 - Sq}), dtype=np.int64)
    rq, rk, rv = oracle_mod.attn_bwd_sampled(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                             inputs.bits16(do), causal, scale, qrows, krows)
    b, rem = np.divmod(qrows, Hq * Sq)
    h, i = np.divmod(rem, Sq)
    gq = dq[torch.as_tensor(b), torch.as_tensor(i), torch.as_tensor(h)].float().cpu().numpy()
    gk = dk[0, torch.as_tensor(krows), 0].float().cpu().numpy()
    gv = dv[0, torch.as_tensor(krows), 0].float().cpu().numpy()
    assert_grad_close("dq", gq, rq)
    assert_grad_close("dk", gk, rk)
    assert_grad_close("dv", gv, rv)
