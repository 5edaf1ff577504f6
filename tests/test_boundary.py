"""C-ABI boundary checks that need no GPU: the library loads, exports every
entry point the header declares, and rejects bad arguments on the host with
the documented status codes before touching CUDA."""
import os
import re

import pytest

import exact_attention_forward_14_b300 as ea

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_b300.h")
PKG = os.path.join(ROOT, "exact_attention_forward_14_b300")

# fake, never dereferenced device addresses (16-byte aligned)
Q, K, V, O, L = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000


@pytest.fixture(scope="module")
def lib():
    from exact_attention_forward_14_b300 import build
    build.build()
    return ea.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|const char\s*\*|unsigned long long)\s*(\w+)\s*\(", text,
                      flags=re.M)


def test_header_declares_the_boundary():
    assert set(declared_functions()) >= {"attn_fwd", "attn_fwd_fp8", "attn_quantize_fp8_e4m3",
                                         "attn_device_status", "attn_status_string"}


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_watchdog_test_library_exports_the_same_boundary(lib):
    import ctypes
    wd = ctypes.CDLL(os.path.join(PKG, "libattn_watchdog_test.so"))
    for name in declared_functions():
        assert hasattr(wd, name), name


def test_wait_limit_is_settable_within_its_range(lib):
    default = ea.attn_get_wait_limit_ns()
    assert default == 1_000_000_000
    try:
        assert ea.attn_set_wait_limit_ns(5_000_000_000) == ea.ATTN_OK
        assert ea.attn_get_wait_limit_ns() == 5_000_000_000
        # out of range: rejected, limit unchanged
        assert ea.attn_set_wait_limit_ns(999_999) == ea.ATTN_ERR_INVALID_ARG
        assert ea.attn_set_wait_limit_ns(3_600_000_000_001) == ea.ATTN_ERR_INVALID_ARG
        assert ea.attn_set_wait_limit_ns(0) == ea.ATTN_ERR_INVALID_ARG
        assert ea.attn_get_wait_limit_ns() == 5_000_000_000
        assert ea.attn_set_wait_limit_ns(1_000_000) == ea.ATTN_OK
        assert ea.attn_set_wait_limit_ns(3_600_000_000_000) == ea.ATTN_OK
    finally:
        assert ea.attn_set_wait_limit_ns(default) == ea.ATTN_OK


def test_status_strings(lib):
    names = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
             3: "ATTN_ERR_MISALIGNED", 4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_TIMEOUT"}
    for code, name in names.items():
        assert ea.attn_status_string(code) == name
    assert ea.attn_status_string(99) == "ATTN_ERR_UNKNOWN"


def fwd(**kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, Hq=2, Hkv=2, Sq=128, Sk=128, d=128, causal=0,
             scale=0.1, dtype=ea.ATTN_BF16, stream=0)
    a.update(kw)
    return ea.attn_fwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(lse=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(B=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(Sk=-1), ea.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), ea.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), ea.ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.5), ea.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), ea.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), ea.ATTN_ERR_INVALID_ARG),
    (dict(B=1, Sq=1 << 20, Hq=32, Hkv=32, d=128), ea.ATTN_ERR_INVALID_ARG),  # 2^32 elements
    (dict(d=96), ea.ATTN_ERR_UNSUPPORTED),
    (dict(d=192), ea.ATTN_ERR_UNSUPPORTED),
    (dict(d=256, dtype=ea.ATTN_FP8_E4M3), ea.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=7), ea.ATTN_ERR_UNSUPPORTED),
    (dict(q=Q + 8), ea.ATTN_ERR_MISALIGNED),
    (dict(v=V + 2), ea.ATTN_ERR_MISALIGNED),
    (dict(o=O + 4), ea.ATTN_ERR_MISALIGNED),
    (dict(lse=L + 2), ea.ATTN_ERR_MISALIGNED),
])
def test_attn_fwd_rejects_bad_arguments(lib, kw, code):
    assert fwd(**kw) == code


def test_attn_fwd_fp8_requires_scales(lib):
    args = [Q, K, V, 0x60000, 0x70000, 0x80000, O, L, 1, 2, 2, 128, 128, 128, 0, 0.1]
    bad = list(args)
    bad[4] = 0
    assert ea.attn_fwd_fp8(*bad, stream=0) == ea.ATTN_ERR_INVALID_ARG
    bad = list(args)
    bad[3] = 0x60002
    assert ea.attn_fwd_fp8(*bad, stream=0) == ea.ATTN_ERR_MISALIGNED
    bad = list(args)
    bad[13] = 80
    assert ea.attn_fwd_fp8(*bad, stream=0) == ea.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("args,code", [
    ((0, Q, L, 1, 64, 2, 128), ea.ATTN_ERR_INVALID_ARG),
    ((Q, Q, L, 1, 0, 2, 128), ea.ATTN_ERR_INVALID_ARG),
    ((Q, Q, L, 1, 64, 2, 32), ea.ATTN_ERR_UNSUPPORTED),
    ((Q + 4, K, L, 1, 64, 2, 128), ea.ATTN_ERR_MISALIGNED),
])
def test_quantiser_rejects_bad_arguments(lib, args, code):
    assert ea.attn_quantize_fp8_e4m3(*args, stream=0) == code


def test_valid_call_without_a_gpu_fails_loudly(lib):
    """With no CUDA device the library returns an error: there is no CPU path."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd() in (ea.ATTN_ERR_CUDA, ea.ATTN_ERR_UNSUPPORTED)
    with pytest.raises(ea.AttnError):
        ea._check(fwd(), "attn_fwd")


def test_product_package_never_touches_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "attn_oracle" not in text and "liboracle" not in text, f


# ------------------------------------------------------------------ split-KV --

def _plan_by_hand(B, Hq, Sq, Sk, causal, sms):
    """The documented cost model, restated: argmin over s of
    ceil(items * s / sms) * (ceil(tiles / s) + 2), smallest s on ties."""
    nkv, nqt, nqp = -(-Sk // 128), -(-Sq // 128), -(-Sq // 256)
    items = B * Hq * ((nqp + 1) // 2)
    tiles = max(1, nkv - nqt // 2) if causal else nkv
    smax = min(max(1, nkv // 4), 256)
    costs = [(-(-items * s // sms) * (-(-tiles // s) + 2), s) for s in range(1, smax + 1)]
    s = min(costs)[1]
    kps = -(-nkv // min(s, nkv))
    return -(-nkv // kps)


@pytest.mark.parametrize("shape", [
    (1, 32, 256, 65536, False),   # 32 items: 9 ranges make two full rounds
    (1, 8, 64, 65536, False),
    (2, 32, 8192, 8192, True),    # the query side fills the GPU
    (4, 16, 2048, 2048, True),
    (1, 1, 1, 1024, False),
    (1, 4, 300, 3000, True),
])
def test_splitkv_plan_follows_the_cost_model(shape):
    B, Hq, Sq, Sk, causal = shape
    rc, n, w = ea.attn_splitkv_plan(B, Hq, Sq, Sk, 128, causal, num_sms=148)
    assert rc == ea.ATTN_OK
    assert n == _plan_by_hand(B, Hq, Sq, Sk, causal, 148)
    assert w == n * B * Hq * Sq * 129 * 4


def test_splitkv_plan_examples_and_errors():
    assert ea.attn_splitkv_plan(1, 32, 256, 65536, 128, False, num_sms=148)[1] == 9
    assert ea.attn_splitkv_plan(2, 32, 8192, 8192, 128, True, num_sms=148)[1] == 1
    assert ea.attn_splitkv_plan(1, 1, 1, 100, 96, False, num_sms=148)[0] == ea.ATTN_ERR_UNSUPPORTED
    assert ea.attn_splitkv_plan(0, 1, 1, 100, 64, False, num_sms=148)[0] == ea.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(num_splits=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(num_splits=257), ea.ATTN_ERR_INVALID_ARG),
    (dict(workspace=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(workspace_bytes=16), ea.ATTN_ERR_INVALID_ARG),
    (dict(workspace=0x60008), ea.ATTN_ERR_MISALIGNED),
    (dict(dtype=ea.ATTN_FP8_E4M3), ea.ATTN_ERR_UNSUPPORTED),
    (dict(d=96), ea.ATTN_ERR_UNSUPPORTED),
    (dict(Hkv=3), ea.ATTN_ERR_INVALID_ARG),
])
def test_splitkv_rejects_bad_arguments(lib, kw, code):
    a = dict(B=1, Hq=4, Hkv=2, Sq=64, Sk=1000, d=128, causal=0, scale=0.1, dtype=ea.ATTN_BF16,
             num_splits=4, workspace=0x60000, workspace_bytes=1 << 30)
    a.update(kw)
    rc = ea.attn_fwd_splitkv(Q, K, V, O, L, a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["d"],
                             a["causal"], a["scale"], a["dtype"], a["num_splits"], a["workspace"],
                             a["workspace_bytes"], stream=0)
    assert rc == code


# --------------------------------------------------------------- QK RMSNorm --

@pytest.mark.parametrize("kw,code", [
    (dict(q=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(k_out=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(B=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(eps=-1.0), ea.ATTN_ERR_INVALID_ARG),
    (dict(eps=float("nan")), ea.ATTN_ERR_INVALID_ARG),
    (dict(d=96), ea.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=ea.ATTN_FP8_E4M3), ea.ATTN_ERR_UNSUPPORTED),
    (dict(q_weight=0x70004), ea.ATTN_ERR_MISALIGNED),
])
def test_qk_rmsnorm_rejects_bad_arguments(lib, kw, code):
    a = dict(q=Q, k=K, q_weight=0x70000, k_weight=0x80000, q_out=O, k_out=0x90000, B=1, Sq=8,
             Sk=8, Hq=2, Hkv=2, d=64, eps=1e-6, dtype=ea.ATTN_BF16)
    a.update(kw)
    rc = ea.attn_qk_rmsnorm(a["q"], a["k"], a["q_weight"], a["k_weight"], a["q_out"], a["k_out"],
                            a["B"], a["Sq"], a["Sk"], a["Hq"], a["Hkv"], a["d"], a["eps"],
                            a["dtype"], stream=0)
    assert rc == code


# ----------------------------------------------------------------- backward --

def test_bwd_workspace_size():
    # 2 fp32 per query row padded to whole 128-row tiles
    assert ea.attn_bwd_workspace_size(2, 32, 8192) == (ea.ATTN_OK, 2 * 2 * 32 * 8192 * 4)
    assert ea.attn_bwd_workspace_size(1, 3, 300) == (ea.ATTN_OK, 2 * 3 * 384 * 4)
    assert ea.attn_bwd_workspace_size(1, 1, 1) == (ea.ATTN_OK, 2 * 128 * 4)
    assert ea.attn_bwd_workspace_size(0, 1, 1)[0] == ea.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(d_o=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(dk=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(o=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(lse=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(workspace=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(workspace_bytes=2 * 4 * 128 * 4 - 4), ea.ATTN_ERR_INVALID_ARG),
    (dict(workspace=0xC0008), ea.ATTN_ERR_MISALIGNED),
    (dict(dq=0xA0004), ea.ATTN_ERR_MISALIGNED),
    (dict(d_o=0x70002), ea.ATTN_ERR_MISALIGNED),
    (dict(dtype=ea.ATTN_FP8_E4M3), ea.ATTN_ERR_UNSUPPORTED),
    (dict(d=96), ea.ATTN_ERR_UNSUPPORTED),
    (dict(Hkv=3), ea.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), ea.ATTN_ERR_INVALID_ARG),
    (dict(Sk=0), ea.ATTN_ERR_INVALID_ARG),
])
def test_bwd_rejects_bad_arguments(lib, kw, code):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, d_o=0x70000, dq=0xA0000, dk=0xB0000, dv=0xD0000, B=1,
             Hq=4, Hkv=2, Sq=100, Sk=100, d=128, causal=1, scale=0.1, dtype=ea.ATTN_BF16,
             workspace=0xC0000, workspace_bytes=2 * 4 * 128 * 4)
    a.update(kw)
    rc = ea.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["d_o"], a["dq"], a["dk"],
                     a["dv"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["d"], a["causal"],
                     a["scale"], a["dtype"], a["workspace"], a["workspace_bytes"], stream=0)
    assert rc == code


def test_d256_is_forward_only(lib):
    """Head dimension 256 is served by attn_fwd (bf16 / fp16) only."""
    assert ea.attn_fwd(Q, K, V, O, L, 1, 2, 2, 64, 64, 256, 1, 0.1, ea.ATTN_FP8_E4M3,
                       stream=0) == ea.ATTN_ERR_UNSUPPORTED
    assert ea.attn_fwd_fp8(Q, K, V, 0x60000, 0x60100, 0x60200, O, L, 1, 2, 2, 64, 64, 256, 1,
                           0.1, stream=0) == ea.ATTN_ERR_UNSUPPORTED
    assert ea.attn_fwd_splitkv(Q, K, V, O, L, 1, 2, 2, 64, 1000, 256, 0, 0.1, ea.ATTN_BF16, 2,
                               0x60000, 1 << 30, stream=0) == ea.ATTN_ERR_UNSUPPORTED
    assert ea.attn_bwd(Q, K, V, O, L, 0x70000, 0xA0000, 0xB0000, 0xD0000, 1, 2, 2, 64, 64, 256,
                       1, 0.1, ea.ATTN_BF16, 0xC0000, 1 << 20, stream=0) == ea.ATTN_ERR_UNSUPPORTED
    assert ea.attn_fwd(Q, K, V, O, L, 1, 2, 2, 64, 64, 192, 1, 0.1, ea.ATTN_BF16,
                       stream=0) == ea.ATTN_ERR_UNSUPPORTED


def test_noalloc_checks_match_the_workspace_entry_point(lib):
    """attn_fwd_splitkv_noalloc returns the codes attn_fwd_splitkv returns for
    the same request, and checks the type before its array's size (an
    oversized E4M3 request is unsupported, not too large); all on the host."""
    big = dict(B=4, Hq=64, Sq=2048, Sk=32768)  # 69 GB of workspace at 256 ranges
    for dtype, d, splits, code in [(ea.ATTN_FP8_E4M3, 128, 256, ea.ATTN_ERR_UNSUPPORTED),
                                   (7, 128, 2, ea.ATTN_ERR_UNSUPPORTED),
                                   (ea.ATTN_BF16, 256, 2, ea.ATTN_ERR_UNSUPPORTED),
                                   (ea.ATTN_BF16, 128, 0, ea.ATTN_ERR_INVALID_ARG),
                                   (ea.ATTN_BF16, 128, 257, ea.ATTN_ERR_INVALID_ARG),
                                   (ea.ATTN_BF16, 128, 256, ea.ATTN_ERR_INVALID_ARG)]:
        Sk = big["Sk"] if d == 128 else 1024  # d = 256: every tensor below 2^31 elements
        rc = ea.attn_fwd_splitkv_noalloc(Q, K, V, O, L, big["B"], big["Hq"], big["Hq"],
                                         big["Sq"], Sk, d, 0, 0.1, dtype, splits, stream=0)
        assert rc == code, (dtype, d, splits, rc)
        if splits != 256 or dtype != ea.ATTN_BF16:  # the workspace form has no size to refuse
            rc2 = ea.attn_fwd_splitkv(Q, K, V, O, L, big["B"], big["Hq"], big["Hq"], big["Sq"],
                                      Sk, d, 0, 0.1, dtype, splits, 0x60000, 1 << 62,
                                      stream=0)
            assert rc2 == code, (dtype, d, splits, rc2)


def test_bwd_rejects_padded_row_statistics_past_32_bits(lib):
    """Sq = 1 pads to a 128-row tile: 20M (b, hq) pairs keep every tensor below
    2^31 elements (20M x 64) but the padded statistics (20M x 128 rows) past
    it, so the call is refused on the host."""
    B, Hq = 2, 10_000_000
    assert B * 1 * Hq * 64 < 2 ** 31 < B * Hq * 128
    rc = ea.attn_bwd(Q, K, V, O, L, 0x70000, 0xA0000, 0xB0000, 0xD0000, B, Hq, Hq, 1, 1, 64, 0,
                     0.1, ea.ATTN_BF16, 0xC0000, 1 << 40, stream=0)
    assert rc == ea.ATTN_ERR_INVALID_ARG


def test_backward_wrapper_checks_dtypes():
    """The tensor convenience refuses mixed or unsupported dtypes on the host."""
    import torch
    q = torch.zeros(1, 4, 1, 64, dtype=torch.bfloat16)
    f = torch.zeros(1, 4, 1, 64, dtype=torch.float16)
    lse = torch.zeros(1, 1, 4, dtype=torch.float32)
    with pytest.raises(TypeError):
        ea.backward(q, q, q, q, lse, f)
    with pytest.raises(TypeError):
        ea.backward(q, q, q, q, lse.double(), q)
    with pytest.raises(TypeError):
        ea.backward(q.float(), q.float(), q.float(), q.float(), lse, q.float())


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every entry point raises: there is no
    non-CUDA fallback for a caller to land on silently."""
    monkeypatch.setattr(ea, "_lib", None)
    monkeypatch.setattr(ea, "library_path", lambda: str(tmp_path / "libattn_b300.so"))
    with pytest.raises(ImportError, match="no non-CUDA fallback"):
        ea.load()
    with pytest.raises(ImportError):
        ea.attn_fwd(Q, K, V, O, L, 1, 1, 1, 64, 64, 64, 0, 0.1, stream=0)
    with pytest.raises(ImportError):
        ea.attn_bwd_workspace_size(1, 1, 1)
