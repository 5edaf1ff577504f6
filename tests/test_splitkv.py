"""GPU parity of the split-KV path (per-range partial attention + LSE merge)
against the fp64 oracle on the whole key set, through the C ABI."""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, require_gpu

# (B, Hq, Hkv, Sq, Sk, d, causal, dtype, num_splits)
CASES = [
    (1, 8, 2, 64, 5000, 128, False, "bf16", 7),      # GQA, ragged last range and tile
    (2, 4, 4, 300, 3000, 128, True, "bf16", 5),      # causal: late ranges empty for early rows
    (1, 4, 4, 1, 4096, 64, False, "bf16", 16),       # decode: one query row
    (1, 4, 2, 200, 2000, 128, True, "f16", 3),       # fp16, Sq < Sk bottom-right causal
    (1, 2, 2, 129, 700, 128, False, "bf16", 1),      # one range
    (1, 2, 2, 40, 1000, 64, False, "f16", 200),      # more ranges asked than K/V tiles
    (1, 2, 2, 300, 127, 128, True, "bf16", 2),       # Sq > Sk: fully masked rows
]


def _run(torch, oracle_mod, B, Hq, Hkv, Sq, Sk, d, causal, dtype, num_splits, seed):
    draw = inputs.draw_qkv_f16 if dtype == "f16" else inputs.draw_qkv_bf16
    q, k, v = draw(B, Hq, Hkv, Sq, Sk, d, seed=seed)
    scale = 1.0 / np.sqrt(d)
    o, lse = ea.forward_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                                num_splits=num_splits)
    assert ea.attn_device_status() == ea.ATTN_OK
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         causal, scale, dtype=dtype)
    assert_o_close(o.float().cpu().numpy(), o_ref, kind=dtype)
    assert_lse_close(lse.cpu().numpy(), lse_ref)
    return o, lse


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}hq{}hkv{}sq{}sk{}d{}{}_{}_s{}".format(
    *c[:6], "c" if c[6] else "", c[7], c[8]))
def test_splitkv_matches_oracle(oracle_mod, case):
    torch = require_gpu()
    _run(torch, oracle_mod, *case, seed=sum(case[:6]) + 41)


@pytest.mark.gpu
def test_planned_split_on_long_keys(oracle_mod):
    """The plan's own split count on a query side too small for the GPU."""
    torch = require_gpu()
    B, Hq, Hkv, Sq, Sk, d = 1, 8, 2, 16, 16384, 128
    rc, n, wbytes = ea.attn_splitkv_plan(B, Hq, Sq, Sk, d, False)
    assert rc == ea.ATTN_OK and n > 1
    q, k, v = inputs.draw_qkv_bf16(B, Hq, Hkv, Sq, Sk, d, seed=5)
    ws = torch.empty(wbytes // 4, dtype=torch.float32, device="cuda")
    o, lse = ea.forward_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=False, workspace=ws,
                                num_splits=n)
    assert ea.attn_device_status() == ea.ATTN_OK
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(q), inputs.bits16(k), inputs.bits16(v),
                                         False, 1.0 / np.sqrt(d))
    assert_o_close(o.float().cpu().numpy(), o_ref)
    assert_lse_close(lse.cpu().numpy(), lse_ref)


@pytest.mark.gpu
def test_split_and_unsplit_agree():
    """Both paths on the same inputs: equal up to the rounding of the merge."""
    torch = require_gpu()
    q, k, v = (t.cuda() for t in inputs.draw_qkv_bf16(1, 4, 4, 256, 4096, 128, seed=9))
    o1, l1 = ea.forward(q, k, v, causal=True)
    o2, l2 = ea.forward_splitkv(q, k, v, causal=True, num_splits=6)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-4
