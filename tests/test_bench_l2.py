"""bench.py's L2 policy, host-side: the per-step byte counts that decide it
match the compulsory traffic computed by hand for the five workload shapes
(Q, K, V read and O, LSE written once), and only workloads whose inputs fit
in the 126 MiB L2 get the flush."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_attention_forward_14_b300 import inputs  # noqa: E402

W = inputs.WORKLOADS


@pytest.mark.parametrize("name,total", [
    ("tiny_b1h1s128d64", 66_048),                    # 4 x 128 x 64 x 2 B + 128 x 4 B
    ("b4h16s2048d128_causal", 134_742_016),          # 4 x 2^24 x 2 B + 2^17 x 4 B
    ("b2h32s8192d128_causal", 538_968_064),          # 4 x 2^26 x 2 B + 2^19 x 4 B
    ("gqa_b1hq32hkv8s16384d128_causal", 337_641_472),  # (2^26 + 2 x 2^24 + 2^26) x 2 B + 2^19 x 4 B
    ("fp8_b4h16s4096d128", 168_869_888),             # 3 x 2^25 x 1 B + 2^25 x 2 B + 2^18 x 4 B + scales
])
def test_step_bytes_match_the_compulsory_traffic(name, total):
    inb, outb = bench.step_bytes(W[name])
    assert inb + outb == total


def test_fp8_scales_are_counted():
    # one fp32 scale per 64 rows of each head of Q, K and V
    inb, _ = bench.step_bytes(W["fp8_b4h16s4096d128"])
    assert inb == 3 * 4 * 4096 * 16 * 128 + 4 * 3 * 4 * 16 * (4096 // 64)


def test_backward_bytes():
    # in: Q, K, V, O, dO (bf16) and LSE; out: dQ, dK, dV
    w = W["bwd_b2h32s8192d128_causal"]
    n = 2 * 8192 * 32 * 128
    assert bench.step_bytes(w) == (5 * n * 2 + 2 * 32 * 8192 * 4, 3 * n * 2)


@pytest.mark.parametrize("name,flushed", [
    ("tiny_b1h1s128d64", True),
    ("b4h16s2048d128_causal", True),
    ("fp8_b4h16s4096d128", True),
    ("b2h32s8192d128_causal", False),
    ("gqa_b1hq32hkv8s16384d128_causal", False),
    ("longkv_b1hq32hkv8sq256sk65536d128_splitkv", False),
    ("bwd_b2h32s8192d128_causal", False),
])
def test_only_workloads_that_fit_in_l2_are_flushed(name, flushed):
    n = bench.l2_flush_bytes(W[name])
    assert (n > 0) == flushed
    if flushed:
        assert n >= 2 * bench.L2_BYTES
        assert "fit in L2" in bench.workload_config(W[name])["l2"]
    else:
        assert bench.workload_config(W[name])["l2"] == "inputs larger than L2 (no flush)"


def test_flush_follows_the_device_l2_size():
    w = W["b4h16s2048d128_causal"]
    assert bench.l2_flush_bytes(w, 64 * 2 ** 20) == 0      # would not fit a 64 MiB L2
    assert bench.l2_flush_bytes(w, 200 * 2 ** 20) == 400 * 2 ** 20
