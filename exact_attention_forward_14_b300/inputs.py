"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

Holds no attention arithmetic: it only draws random numbers and names the
workload shapes. Both the CUDA path and the CPU oracle consume what it makes.

Recipe (all on the CPU, one ``torch.Generator`` per workload):
  * Q, K, V are drawn in that order as fp32 N(0, 1) of shape [B, S, H, d];
  * for the FP8 workload, after each tensor's values a Bernoulli(0.001) mask is
    drawn from the same generator and the selected entries are multiplied by 20
    (outliers);
  * bf16 / fp16 workloads round the fp32 draw to that type (round-to-nearest-
    even, torch's cast); the FP8 workload hands the fp32 draw to the block
    quantiser.
The pages' own benchmark shape is "sequence length 8K, head dim 128"; no public
dataset is involved.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    d: int
    causal: bool
    dtype: str = "bf16"          # "bf16", "f16" or "e4m3"
    outlier_frac: float = 0.0
    seed: int = 1000
    splits: int = 0              # split-KV ranges: 0 = plain forward, -1 = the plan's choice
    qknorm: bool = False         # RMSNorm across heads of Q and K before the attention
    backward: bool = False       # the step is the backward pass (dQ, dK, dV) instead

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self) -> float:
        """Metric FLOP count of the forward pass: 4*B*H*Sq*Sk*d, halved for
        causal; the backward pass counts 2.5 times that (its five matrix
        products against the forward's two)."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.d
        f = f / 2 if self.causal else f
        return 2.5 * f if self.backward else f


# The five reference workloads (long-context prefill shapes); the seed is
# 1000 + the workload's position in this list.
WORKLOADS = {
    "tiny_b1h1s128d64": Workload("tiny_b1h1s128d64", 1, 1, 1, 128, 128, 64, False, seed=1000),
    "b4h16s2048d128_causal": Workload("b4h16s2048d128_causal", 4, 16, 16, 2048, 2048, 128, True,
                                      seed=1001),
    "b2h32s8192d128_causal": Workload("b2h32s8192d128_causal", 2, 32, 32, 8192, 8192, 128, True,
                                      seed=1002),
    "b2h32s8192d128": Workload("b2h32s8192d128", 2, 32, 32, 8192, 8192, 128, False, seed=1002),
    "gqa_b1hq32hkv8s16384d128_causal": Workload("gqa_b1hq32hkv8s16384d128_causal", 1, 32, 8,
                                                16384, 16384, 128, True, seed=1003),
    "fp8_b4h16s4096d128": Workload("fp8_b4h16s4096d128", 4, 16, 16, 4096, 4096, 128, False,
                                   dtype="e4m3", outlier_frac=0.001, seed=1004),
    # the FP8 workload's shape in bf16 (N(0, 1), no outliers), to compare the two input
    # types on one shape
    "b4h16s4096d128": Workload("b4h16s4096d128", 4, 16, 16, 4096, 4096, 128, False, seed=1004),
    # long key side, short query side (the last 256 rows of a 64K context, GQA):
    # 32 work items alone leave most SMs idle; the split-KV form fills them
    "longkv_b1hq32hkv8sq256sk65536d128": Workload("longkv_b1hq32hkv8sq256sk65536d128", 1, 32, 8,
                                                  256, 65536, 128, False, seed=1006),
    "longkv_b1hq32hkv8sq256sk65536d128_splitkv": Workload(
        "longkv_b1hq32hkv8sq256sk65536d128_splitkv", 1, 32, 8, 256, 65536, 128, False,
        seed=1006, splits=-1),
    # the long-context prefill shape behind the QK-RMSNorm prologue
    "qknorm_b2h32s8192d128_causal": Workload("qknorm_b2h32s8192d128_causal", 2, 32, 32, 8192,
                                             8192, 128, True, seed=1002, qknorm=True),
    # backward pass of the long-context prefill shape (same inputs, dO drawn
    # from its own generator)
    "bwd_b2h32s8192d128_causal": Workload("bwd_b2h32s8192d128_causal", 2, 32, 32, 8192, 8192,
                                          128, True, seed=1002, backward=True),
    "bwd_gqa_b1hq32hkv8s16384d128_causal": Workload("bwd_gqa_b1hq32hkv8s16384d128_causal", 1, 32,
                                                    8, 16384, 16384, 128, True, seed=1003,
                                                    backward=True),
    # head dimension 256 (the same FLOPs as the d = 128 prefill shape: half the heads)
    "d256_b2h16s8192_causal": Workload("d256_b2h16s8192_causal", 2, 16, 16, 8192, 8192, 256,
                                       True, seed=1007),
    # head dimension 64 at long context (twice the heads of the d = 128 prefill shape,
    # the same FLOPs): the d = 64 instantiation of the forward kernel
    "d64_b2h64s8192_causal": Workload("d64_b2h64s8192_causal", 2, 64, 64, 8192, 8192, 64, True,
                                      seed=1008),
    # fp16 variant of the long-context prefill shape (the FA3 page benchmarks FP16)
    "f16_b2h32s8192d128_causal": Workload("f16_b2h32s8192d128_causal", 2, 32, 32, 8192, 8192, 128,
                                          True, dtype="f16", seed=1005),
}


def draw_qkv_f32(B, Hq, Hkv, Sq, Sk, d, seed, outlier_frac=0.0, outlier_mult=20.0):
    """fp32 CPU tensors q [B,Sq,Hq,d], k/v [B,Sk,Hkv,d], N(0,1) with optional outliers."""
    g = torch.Generator().manual_seed(int(seed))
    out = []
    for shape in ((B, Sq, Hq, d), (B, Sk, Hkv, d), (B, Sk, Hkv, d)):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if outlier_frac > 0:
            hit = torch.rand(shape, generator=g) < outlier_frac
            x = torch.where(hit, x * outlier_mult, x)
        out.append(x)
    return tuple(out)


def draw_workload_f32(w: Workload):
    return draw_qkv_f32(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.seed, w.outlier_frac)


def draw_qkv_bf16(B, Hq, Hkv, Sq, Sk, d, seed, outlier_frac=0.0):
    """bf16 CPU tensors (the fp32 draw rounded to bf16)."""
    return tuple(t.to(torch.bfloat16) for t in
                 draw_qkv_f32(B, Hq, Hkv, Sq, Sk, d, seed, outlier_frac))


def draw_qkv_f16(B, Hq, Hkv, Sq, Sk, d, seed, outlier_frac=0.0):
    """fp16 CPU tensors (the fp32 draw rounded to fp16)."""
    return tuple(t.to(torch.float16) for t in
                 draw_qkv_f32(B, Hq, Hkv, Sq, Sk, d, seed, outlier_frac))


def draw_workload_16(w: Workload):
    """The workload's q, k, v in its 16-bit type (bf16 or f16)."""
    f = draw_qkv_f16 if w.dtype == "f16" else draw_qkv_bf16
    return f(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.seed)


def draw_grad_out(B, Sq, Hq, d, seed, dtype="bf16"):
    """Upstream gradient dO [B, Sq, Hq, d] for the backward pass: fp32 N(0, 1)
    from its own generator (seed + 500), rounded to the 16-bit type."""
    g = torch.Generator().manual_seed(int(seed) + 500)
    x = torch.randn((B, Sq, Hq, d), generator=g, dtype=torch.float32)
    return x.to(torch.float16 if dtype == "f16" else torch.bfloat16)


def draw_norm_weights(n, seed, dtype="bf16"):
    """RMSNorm weights ~ 1 + 0.25 N(0, 1), rounded to the 16-bit type."""
    g = torch.Generator().manual_seed(int(seed))
    w = 1.0 + 0.25 * torch.randn(n, generator=g)
    return w.to(torch.float16 if dtype == "f16" else torch.bfloat16)


def bits16(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bits of a bf16 or fp16 CPU tensor, as numpy (for the oracle)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bits of a bf16 CPU tensor, as numpy (for the oracle)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(B, H, Sq, n, seed):
    """n distinct flat row indices (b*H + h)*Sq + i, always including the first
    and last row of the first and last (b, h) so edge rows are covered."""
    total = B * H * Sq
    g = np.random.default_rng(seed)
    pick = set(int(x) for x in g.choice(total, size=min(n, total), replace=False))
    pick.update({0, Sq - 1, total - Sq, total - 1})
    return np.array(sorted(pick), dtype=np.int64)


def stratified_rows(B, H, Sq, tile, seed):
    """Flat row indices (b*H + h)*Sq + i covering every (b, h, tile of `tile`
    consecutive query rows): the tile's first and last row and one more drawn
    at random inside it, so every work item of the kernel is checked."""
    g = np.random.default_rng(seed)
    ntile = -(-Sq // tile)
    first = np.arange(ntile, dtype=np.int64) * tile
    last = np.minimum(first + tile, Sq) - 1
    pick = []
    for bh in range(B * H):
        mid = first + (g.random(ntile) * (last - first + 1)).astype(np.int64)
        pick.append(bh * Sq + np.unique(np.concatenate([first, last, mid])))
    return np.unique(np.concatenate(pick))
