"""The entry points only enqueue work (no host synchronisation, no allocation
inside the call), so a sequence of them can be captured into a CUDA graph and
replayed. Replays must reproduce the eager results bit for bit."""
import pytest

import exact_attention_forward_14_b300 as ea
from exact_attention_forward_14_b300 import inputs
from tests.helpers import require_gpu


@pytest.mark.gpu
def test_forward_backward_and_splitkv_replay_from_a_cuda_graph():
    torch = require_gpu()
    B, Hq, Hkv, S, d = 1, 8, 2, 1000, 128
    q, k, v = (t.cuda() for t in inputs.draw_qkv_bf16(B, Hq, Hkv, S, S, d, seed=91))
    do = inputs.draw_grad_out(B, S, Hq, d, 91).cuda()
    scale = d ** -0.5
    rc, wbytes = ea.attn_bwd_workspace_size(B, Hq, S)
    ws = torch.empty(wbytes // 4, dtype=torch.float32, device="cuda")
    nsplit = 3
    skv_ws = torch.empty(nsplit * B * Hq * S * (d + 1), dtype=torch.float32, device="cuda")
    o, lse = torch.empty_like(q), torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def work(stream):
        assert ea.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, S, S, d, True, scale, ea.ATTN_BF16,
                           stream) == ea.ATTN_OK
        assert ea.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, S, S, d, True, scale,
                           ea.ATTN_BF16, ws, wbytes, stream) == ea.ATTN_OK
        assert ea.attn_fwd_splitkv(q, k, v, o2, lse2, B, Hq, Hkv, S, S, d, True, scale,
                                   ea.ATTN_BF16, nsplit, skv_ws, skv_ws.numel() * 4,
                                   stream) == ea.ATTN_OK

    side = torch.cuda.Stream()
    with torch.cuda.stream(side):  # eager run (also sets the kernels' attributes once)
        work(side)
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    eager = [t.clone() for t in (o, lse, dq, dk, dv, o2, lse2)]
    for t in (o, lse, dq, dk, dv, o2, lse2):
        t.zero_()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        work(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert ea.attn_device_status() == ea.ATTN_OK
    for got, want in zip((o, lse, dq, dk, dv, o2, lse2), eager):
        assert torch.equal(got, want)
