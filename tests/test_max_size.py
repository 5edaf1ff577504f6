"""Keys at the largest size the 32-bit element-count guard admits.

K and V hold 2^31 - 128 elements each at d = 128 (16,777,215 keys), so K/V
tile coordinates run past 131,000 and the last tile has 127 keys. With random
keys alone the softmax over 16.7M keys is nearly flat, and no sampled output
would notice a skipped tile or a shifted mask. So the inputs plant "needle"
keys along a direction u that every query shares. Their scores (about 27-31)
dominate each row's softmax, so every sampled output depends on finding the
needles at their exact positions:
  - 16 needles spread over the whole key range (tile indices up to ~123,000);
  - one 200 keys before the end, visible (bottom-right causal) from query
    row 56 on;
  - one on the very last key, in the ragged last tile, visible to the last
    query row only.
V is K shifted by one row, so each needle carries its own random value row.
The background (scores ~N(0, 0.5^2)) weighs below 2e-6 of the total, so the
fp32 accumulation over 131k tiles cannot move the result past the
tolerances. A CPU test checks this design's power on a smaller key range:
an off-by-one mask or a skipped needle tile moves the oracle's outputs by
more than twice the tolerance."""
import numpy as np
import pytest
import torch

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, require_gpu

D, SQ, HQ = 128, 256, 2
SK_MAX = (2 ** 31 - 1) // D  # largest key count with Sk * d below 2^31


def needle_positions(Sk):
    """Key index -> gamma (the needle is gamma * u)."""
    pos = {m * ((Sk + 1) // 16) + 61 * m + 7: 2.4 for m in range(16)}
    pos[Sk - 200] = 2.6
    pos[Sk - 1] = 2.7
    return pos


def needle_inputs(Sk, seed=91, drop=None, move_last=False):
    """q [1, SQ, HQ, D], k and v [1, Sk, 1, D] in bf16. `drop` leaves one
    needle out; `move_last` puts the last needle one key earlier (as a mask
    shifted by one would see it). Both exist only for the power test."""
    g = torch.Generator().manual_seed(seed)
    u = torch.where(torch.rand(D, generator=g) < 0.5, -1.0, 1.0)
    q = (u + 0.25 * torch.randn(1, SQ, HQ, D, generator=g)).to(torch.bfloat16)
    k = torch.empty(1, Sk, 1, D, dtype=torch.bfloat16)
    flat = k.view(-1)
    step = 1 << 26
    for s0 in range(0, flat.numel(), step):
        n = min(step, flat.numel() - s0)
        flat[s0:s0 + n] = 0.5 * torch.randn(n, generator=g)
    v = torch.roll(k, shifts=-1, dims=1)  # v[j] = k[j + 1], taken before the needles
    for j, gamma in needle_positions(Sk).items():
        if j == drop:
            continue
        if move_last and j == Sk - 1:
            j = Sk - 2
        k[0, j, 0] = (gamma * u).to(torch.bfloat16)
    return q, k, v


# query rows at the mask boundaries of the late needles, in both heads
ROWS = np.array([0, 55, 56, 130, 254, 255, SQ + 0, SQ + 56, SQ + 254, SQ + 255], dtype=np.int64)


def oracle_rows(oracle_mod, q, k, v):
    return oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v), True,
                               D ** -0.5, rows=ROWS)


def test_needle_design_has_the_power_to_fail(oracle_mod):
    """On 2^16 - 1 keys: the needles dominate (LSE well above the background's
    ln Sk), a one-key mask shift changes the last row's output by far more
    than the tolerance, and so does skipping any one needle's tile."""
    Sk = 2 ** 16 - 1
    o, lse = oracle_rows(oracle_mod, *needle_inputs(Sk))
    assert lse.min() > np.log(Sk) + 9.0
    o_moved, _ = oracle_rows(oracle_mod, *needle_inputs(Sk, move_last=True))
    assert np.abs(o_moved - o).max() > 0.2
    for j in needle_positions(Sk):
        o_drop, _ = oracle_rows(oracle_mod, *needle_inputs(Sk, drop=j))
        assert np.abs(o_drop - o).max() > 2e-2, j


@pytest.mark.gpu
def test_keys_at_the_element_count_limit(oracle_mod):
    require_gpu()
    assert SK_MAX * D < 2 ** 31 <= (SK_MAX + 1) * D and SK_MAX % 128 == 127
    q, k, v = needle_inputs(SK_MAX)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_ref, lse_ref = oracle_rows(oracle_mod, q, k, v)
    h, i = np.divmod(ROWS, SQ)
    hi, ii = torch.as_tensor(h), torch.as_tensor(i)
    for name, run in (("attn_fwd", ea.forward), ("attn_fwd_splitkv", ea.forward_splitkv)):
        o, lse = run(qd, kd, vd, causal=True)
        assert ea.attn_device_status() == ea.ATTN_OK, name
        assert_o_close(o[0, ii, hi].float().cpu().numpy(), o_ref)
        assert_lse_close(lse[0, hi, ii].cpu().numpy(), lse_ref)
