"""The split-KV entry point that allocates nothing (attn_fwd_splitkv_noalloc).

It exists for callers that may not allocate device memory themselves (a
plugin inside an application that owns all device buffers, or a loop that must
not call cudaMalloc / cudaFree). Its workspace is a fixed 64 MiB array inside
the library. Here it is called through the C ABI, several times in a row, and
each result is checked twice:
  * bit for bit against the regular attn_fwd_splitkv given a workspace the test
    allocates: both run the same kernels with the same split on the same
    inputs, so any difference is a fault of the built-in array (a wrong offset,
    or stale data a call read instead of writing);
  * element by element against the fp64 oracle.
The first two calls have the same shape, non-causal then causal, so the causal
call uses exactly the array entries the non-causal one filled; under the
causal mask the later key ranges are empty for the early query rows, and the
merge is right only if the call wrote those ranges' entries itself. This file
is collected last, so a run stopping at its first failure has already run
every other test. It also passes on its own in a fresh process: the first
call does the per-device set-up.
"""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, require_gpu

# (B, Hq, Hkv, Sq, Sk, d, causal, dtype, num_splits)
CALLS = [
    (1, 4, 2, 1000, 1024, 128, False, "bf16", 8),
    (1, 4, 2, 1000, 1024, 128, True, "bf16", 8),
    (2, 4, 4, 300, 3000, 64, True, "f16", 5),
    (1, 8, 2, 64, 5000, 128, False, "bf16", 7),
]


def _call(oracle_mod, torch, B, Hq, Hkv, Sq, Sk, d, causal, dtype, num_splits, seed):
    draw = inputs.draw_qkv_f16 if dtype == "f16" else inputs.draw_qkv_bf16
    qh, kh, vh = draw(B, Hq, Hkv, Sq, Sk, d, seed=seed)
    q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
    code = ea.ATTN_F16 if dtype == "f16" else ea.ATTN_BF16
    scale = 1.0 / np.sqrt(d)
    o = torch.empty((B, Sq, Hq, d), dtype=q.dtype, device="cuda")
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
    rc = ea.attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, code,
                                     num_splits)
    assert rc == ea.ATTN_OK, ea.attn_status_string(rc)
    assert ea.attn_device_status() == ea.ATTN_OK
    # the same request with a workspace of the test's own
    o_ws, lse_ws = ea.forward_splitkv(q, k, v, causal=causal, scale=scale, num_splits=num_splits)
    assert ea.attn_device_status() == ea.ATTN_OK
    assert torch.equal(o, o_ws), "O differs from attn_fwd_splitkv"
    assert torch.equal(lse, lse_ws), "LSE differs from attn_fwd_splitkv"
    o_ref, lse_ref = oracle_mod.attn_fwd(inputs.bits16(qh), inputs.bits16(kh), inputs.bits16(vh),
                                         causal, scale, dtype=dtype)
    assert_o_close(o.float().cpu().numpy(), o_ref, kind=dtype)
    assert_lse_close(lse.cpu().numpy(), lse_ref)


@pytest.mark.gpu
def test_noalloc_is_bit_identical_to_the_workspace_entry_point_and_matches_the_oracle(oracle_mod):
    torch = require_gpu()
    for i, call in enumerate(CALLS):
        _call(oracle_mod, torch, *call, seed=300 + i)


@pytest.mark.gpu
def test_noalloc_rejects_a_workspace_beyond_its_array():
    torch = require_gpu()
    # every size passes the 32-bit index check; only the workspace, 256 ranges
    # x 4 x 64 x 2048 rows x 129 x 4 bytes (69 GB), is beyond the 64 MiB array
    B, Hq, Sq, Sk, d = 4, 64, 2048, 32768, 128
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never read: rejected first
    lse = torch.empty(16, dtype=torch.float32, device="cuda")
    rc = ea.attn_fwd_splitkv_noalloc(x, x, x, x, lse, B, Hq, Hq, Sq, Sk, d, False, 0.1,
                                     ea.ATTN_BF16, 256)
    assert rc == ea.ATTN_ERR_INVALID_ARG
    # an E4M3 request is unsupported whatever its size, as for attn_fwd_splitkv
    rc = ea.attn_fwd_splitkv_noalloc(x, x, x, x, lse, B, Hq, Hq, Sq, Sk, d, False, 0.1,
                                     ea.ATTN_FP8_E4M3, 256)
    assert rc == ea.ATTN_ERR_UNSUPPORTED
    assert ea.attn_device_status() == ea.ATTN_OK
