"""Single-tile checks of the two tcgen05 contraction forms the kernel uses
(S = Q K^T with both operands K-major in shared memory; O = P V with P in
tensor memory and V d-contiguous; for E4M3 inputs, P in fp16 and the E4M3 V
tile widened to fp16 in shared memory as the kernel does), against torch
matmul in fp32."""
import ctypes
import os

import pytest

from tests.helpers import require_gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "exact_attention_forward_14_b300", "libattn_selftest.so")


def _single_tile(form, fp8):
    torch = require_gpu()
    lib = ctypes.CDLL(LIB)
    lib.attn_selftest_umma.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5
    lib.attn_selftest_umma.restype = ctypes.c_int
    g = torch.Generator().manual_seed(100 + 2 * form + fp8)
    a32 = torch.randn(128, 128, generator=g)
    b32 = torch.randn(128, 128, generator=g)
    if form == 1:
        a32 = a32.abs()  # P is non-negative
    if fp8:
        a = a32.to(torch.float8_e4m3fn)
        b = b32.to(torch.float8_e4m3fn)
    else:
        a = a32.to(torch.bfloat16)
        b = b32.to(torch.bfloat16)
    af, bf = a.float(), b.float()
    if fp8 and form == 1:
        # the FP8 path keeps P in fp16 and widens the E4M3 V tile to fp16
        a = a32.to(torch.float16)
        af = a.float()
    ref = af @ bf.T if form == 0 else af @ bf
    if fp8 and form == 1:
        da = a.cuda()
    else:
        da = a.view(torch.uint8).cuda() if fp8 else a.cuda()
    db = b.view(torch.uint8).cuda() if fp8 else b.cuda()
    out = torch.full((128, 128), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.attn_selftest_umma(form, fp8, da.data_ptr(), db.data_ptr(), out.data_ptr(),
                                err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(err.item()) == 0, "a wait timed out"
    got = out.cpu()
    diff = (got - ref).abs().max().item()
    assert diff < 1e-3 * max(1.0, ref.abs().max().item()), f"max diff {diff}"


@pytest.mark.gpu
@pytest.mark.parametrize("form", [0, 1], ids=["qk", "pv"])
def test_umma_bf16(form):
    _single_tile(form, 0)


@pytest.mark.gpu
@pytest.mark.parametrize("form", [0, 1], ids=["qk", "pv"])
def test_umma_fp8(form):
    _single_tile(form, 1)


@pytest.mark.gpu
def test_mufu_ex2_rate_is_measured():
    """The exp2 throughput microbenchmark runs on every SM and reports a
    plausible per-SM rate (the SFU issues a warp's ex2 over a few cycles per
    scheduler: between 8 and 128 results per clock per SM)."""
    torch = require_gpu()
    lib = ctypes.CDLL(LIB)
    lib.attn_selftest_ex2_rate.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 3
    lib.attn_selftest_ex2_rate.restype = ctypes.c_int
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    sink = torch.zeros(1024, dtype=torch.float32, device="cuda")
    for _ in range(2):
        assert lib.attn_selftest_ex2_rate(1024, sms, cyc.data_ptr(), sink.data_ptr(), None) == 0
    rates = [1024 * 8 * 1024 / c for c in cyc.cpu().tolist()]
    assert all(c > 0 for c in cyc.cpu().tolist())
    med = sorted(rates)[len(rates) // 2]
    print(f"ex2 per clock per SM: median {med:.2f}, min {min(rates):.2f}, max {max(rates):.2f}")
    assert 8.0 <= med <= 128.0
