"""Seeded synthetic inputs and workload shapes for the fused-dequant linear layer.

This module is shared by the oracle tests, the CUDA-path tests and the
benchmark.  It holds no arithmetic of the quantization method: only shapes,
per-layer bit-width tables and seeded random draws.

Shapes and widths come from the pages this project follows:

* single 4096x4096 layer, 4-bit, group 128 ("a 4096x4096 weight tensor",
  "Mixed-width quantization" page, section 1.2);
* mixed 2/3/5/6-bit widths with a 2-bit share of about half the layers,
  3-bit at most 8 %, 5-bit in attention/middle layers, 6-bit at the ends
  ("Mixed-width quantization" page, section 2.2, width-allocation table);
* a 70B-shaped stack kept at INT4 group 128 with FP16 outliers
  ("70B on one GPU" page, section 2);
* an MoE layer with 16 experts and top-2 routing over a skewed expert
  popularity ("On-device MoE" page, sections 1-2).

Value distributions: weights ~ N(0, 0.02) drawn in fp32 and cast to fp16;
planted outliers of magnitude U(3, 6) with a random sign (the "70B on one GPU" page,
section 2, reports outliers above 3.0 on a distribution concentrated near 0);
activations ~ N(0, 1) drawn in fp32 and cast to bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_W = 1234
SEED_X = 4321
SEED_OUTLIER = 777
SEED_ROUTE = 99


# --------------------------------------------------------------------------
# workload tables
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Linear:
    name: str
    N: int          # output features (rows of W)
    K: int          # input features
    bits: int
    group: int
    frac: float     # outlier fraction


def single_layer():
    """4096x4096, 4-bit, group 128, no outliers; decode M=1."""
    return Linear("single", 4096, 4096, 4, 128, 0.0)


def mixed_sweep():
    """Mixed-width sweep: two shapes x widths {2,3,5,6} x groups {64,128}.

    Every layer carries 0.1 % planted outliers; decode M in {1, 8, 32}.
    """
    out = []
    for (N, K) in ((4096, 4096), (11008, 4096)):
        for bits in (2, 3, 5, 6):
            for group in (64, 128):
                out.append(Linear(f"sweep_{N}x{K}_b{bits}_g{group}", N, K, bits, group, 0.001))
    return out


MIXED_SWEEP_M = (1, 8, 32)


def stack_7b():
    """32-layer 7B-shaped stack with per-layer widths.

    Layers 0, 1, 30, 31: every projection 6-bit.  Layers 2-29: q, k, o 5-bit;
    v 6-bit; gate/up 2-bit (codebook); down 2-bit in layers 6-23, 3-bit in
    24-29 and 5-bit in 2-5.  Group 128, 0.1 % outliers.
    """
    hid, ffn = 4096, 11008
    layers = []
    for L in range(32):
        if L in (0, 1, 30, 31):
            w = dict(q=6, k=6, v=6, o=6, gate=6, up=6, down=6)
        else:
            down = 2 if 6 <= L <= 23 else (3 if L >= 24 else 5)
            w = dict(q=5, k=5, v=6, o=5, gate=2, up=2, down=down)
        shapes = dict(q=(hid, hid), k=(hid, hid), v=(hid, hid), o=(hid, hid),
                      gate=(ffn, hid), up=(ffn, hid), down=(hid, ffn))
        for p in ("q", "k", "v", "o", "gate", "up", "down"):
            N, K = shapes[p]
            layers.append(Linear(f"L{L}.{p}", N, K, w[p], 128, 0.001))
    return layers


STACK_7B_M = (1, 8, 32)


def stack_70b(n_layers: int = 80):
    """80-layer 70B-shaped stack, INT4 group 128, 0.1 % outliers.

    hidden 8192, q/o 8192x8192, k/v 1024x8192 (8 KV heads), gate/up
    28672x8192, down 8192x28672.
    """
    hid, ffn, kv = 8192, 28672, 1024
    shapes = dict(q=(hid, hid), k=(kv, hid), v=(kv, hid), o=(hid, hid),
                  gate=(ffn, hid), up=(ffn, hid), down=(hid, ffn))
    out = []
    for L in range(n_layers):
        for p in ("q", "k", "v", "o", "gate", "up", "down"):
            N, K = shapes[p]
            out.append(Linear(f"L{L}.{p}", N, K, 4, 128, 0.001))
    return out


STACK_70B_DECODE_M = (1, 16, 64)
STACK_70B_PREFILL_M = 2048


@dataclass(frozen=True)
class MoE:
    hidden: int = 4096
    ffn: int = 3072
    n_experts: int = 16
    tokens: int = 256
    top_k: int = 2
    zipf_s: float = 1.1
    bits: int = 4
    group: int = 128
    frac: float = 0.0

    def projections(self):
        """(name, N, K) of the three expert matrices."""
        return (("gate", self.ffn, self.hidden), ("up", self.ffn, self.hidden),
                ("down", self.hidden, self.ffn))


# --------------------------------------------------------------------------
# seeded generators
# --------------------------------------------------------------------------
def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def planted_count(N: int, K: int, frac: float) -> int:
    """How many outliers the generator plants: floor(frac * N * K) in float64."""
    return int(math.floor(float(np.float32(frac)) * float(N) * float(K)))


def gen_weight(N: int, K: int, seed: int = SEED_W, std: float = 0.02,
               outlier_frac: float = 0.0, outlier_seed: int = SEED_OUTLIER,
               device="cpu", distinct_positions: bool = True) -> torch.Tensor:
    """W [N, K] fp16 ~ N(0, std) plus planted outliers of magnitude U(3, 6).

    Positions are distinct (a seeded permutation) unless
    ``distinct_positions`` is False, in which case they are drawn with
    replacement (cheaper for very large matrices; duplicates simply plant
    fewer outliers).
    """
    g = _gen(seed, device)
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32).mul_(std)
    n_out = planted_count(N, K, outlier_frac) if outlier_frac > 0 else 0
    if n_out > 0:
        go = _gen(outlier_seed, device)
        if distinct_positions:
            pos = torch.randperm(N * K, generator=go, device=device)[:n_out]
        else:
            pos = torch.randint(0, N * K, (n_out,), generator=go, device=device)
        mag = torch.rand((n_out,), generator=go, device=device).mul_(3.0).add_(3.0)
        sgn = torch.randint(0, 2, (n_out,), generator=go, device=device).float().mul_(2.0).sub_(1.0)
        w.view(-1)[pos] = mag * sgn
    return w.to(torch.float16)


def gen_extreme_weight(N: int, K: int, group: int, seed: int = SEED_W) -> torch.Tensor:
    """W [N, K] fp16 ~ N(0, 0.02) whose first rows hold groups at the edges of
    fp16's range, in group 0 of each row:

    row 0: a ramp over [0, 65504]; row 1: alternating +-65504;
    row 2: a ramp over [-2256, 65504] (a range whose 4-bit scale puts the top
    grid point past 65504); row 3: one value 65504 among zeros;
    row 4: all zero; row 5: all -1.0 (one-signed); row 6: a ramp over
    [-65504, 0]; row 7: 6.0e4 and -6.0e4 at both ends of a small group.
    The other groups and rows stay ~ N(0, 0.02).  N >= 8, K >= group.
    """
    w = gen_weight(N, K, seed=seed).float()
    g = group
    w[0, :g] = torch.linspace(0.0, 65504.0, g)
    w[1, :g] = torch.tensor([65504.0, -65504.0]).repeat(g // 2)
    w[2, :g] = torch.linspace(-2256.0, 65504.0, g)
    w[3, :g] = 0.0
    w[3, g // 3] = 65504.0
    w[4, :] = 0.0
    w[5, :] = -1.0
    w[6, :g] = torch.linspace(-65504.0, 0.0, g)
    w[7, 0], w[7, g - 1] = 6.0e4, -6.0e4
    return w.to(torch.float16)


def gen_spread_scale_weight(N: int, K: int, group: int, seed: int = SEED_W, tiny: float = 0.05,
                            huge: float = 0.03) -> torch.Tensor:
    """W [N, K] fp16 ~ N(0, 0.02) with a seeded share of its groups scaled by
    2^-11 (``tiny``) and by 2^9 (``huge``): group scales spread over about
    twenty binades."""
    w = gen_weight(N, K, seed=seed).float().reshape(N, K // group, group)
    g = _gen(seed + 7, "cpu")
    u = torch.rand((N, K // group), generator=g)
    f = torch.where(u < tiny, 2.0 ** -11, torch.where(u > 1.0 - huge, 2.0 ** 9, 1.0))
    return (w * f[..., None]).reshape(N, K).to(torch.float16)


def gen_x(M: int, K: int, seed: int = SEED_X, device="cpu") -> torch.Tensor:
    """x [M, K] bf16 ~ N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn((M, K), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def gen_topk(T: int, k: int, n_experts: int, s: float = 1.1, seed: int = SEED_ROUTE) -> torch.Tensor:
    """topk_ids [T, k] int32: k distinct experts per token.

    Expert popularity follows Zipf(s) over ranks 1..E (p_r proportional to
    r^-s); ranks map to experts through a seeded permutation.  Each token
    draws k experts without replacement.
    """
    rng = np.random.default_rng(seed)
    ranks = np.arange(1, n_experts + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    rank_to_expert = rng.permutation(n_experts)
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        r = rng.choice(n_experts, size=k, replace=False, p=p)
        out[t] = rank_to_expert[r]
    return torch.from_numpy(out)


def gen_group_values(n_groups: int, group: int, seed: int, std: float = 1.0) -> np.ndarray:
    """Float16 rows of ``group`` N(0, std) values, for statistical pins."""
    g = _gen(seed)
    w = torch.randn((n_groups, group), generator=g, dtype=torch.float32).mul_(std)
    return w.to(torch.float16).numpy()
