"""The split-KV entry point that allocates nothing (attn_fwd_splitkv_noalloc).

It exists for callers that may not allocate device memory themselves (a
plugin inside an application that owns all device buffers, or a loop that must
not call cudaMalloc / cudaFree). Its workspace is a fixed 64 MiB array inside
the library. Here it is called through the C ABI and compared with the
regular attn_fwd_splitkv, which is given a workspace allocated by the test, on
two calls in a row with different shapes. The second call reuses the array
the first one filled. This file is collected last, so that a run stopping at
its first failure has already run every other test. It also passes on its
own in a fresh process: the first call does the per-device set-up.
"""
import numpy as np
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import assert_lse_close, assert_o_close, require_gpu

# (B, Hq, Hkv, Sq, Sk, d, causal, dtype, num_splits)
CALLS = [
    (1, 8, 2, 64, 5000, 128, False, "bf16", 7),
    (2, 4, 4, 300, 3000, 64, True, "f16", 5),
]


def _both(torch, B, Hq, Hkv, Sq, Sk, d, causal, dtype, num_splits, seed):
    draw = inputs.draw_qkv_f16 if dtype == "f16" else inputs.draw_qkv_bf16
    q, k, v = (t.cuda() for t in draw(B, Hq, Hkv, Sq, Sk, d, seed=seed))
    code = ea.ATTN_F16 if dtype == "f16" else ea.ATTN_BF16
    scale = 1.0 / np.sqrt(d)
    o = torch.empty((B, Sq, Hq, d), dtype=q.dtype, device="cuda")
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
    rc = ea.attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, code,
                                     num_splits)
    assert rc == ea.ATTN_OK, ea.attn_status_string(rc)
    assert ea.attn_device_status() == ea.ATTN_OK
    o_ref, lse_ref = ea.forward_splitkv(q, k, v, causal=causal, scale=scale,
                                        num_splits=num_splits)
    assert ea.attn_device_status() == ea.ATTN_OK
    return o, lse, o_ref, lse_ref


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    torch = require_gpu()
    for i, call in enumerate(CALLS):
        o, lse, o_ref, lse_ref = _both(torch, *call, seed=300 + i)
        kind = call[7]
        assert_o_close(o.float().cpu().numpy(), o_ref.float().cpu().numpy(), kind=kind)
        assert_lse_close(lse.cpu().numpy(), lse_ref.cpu().numpy())


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
    assert ea.attn_device_status() == ea.ATTN_OK
