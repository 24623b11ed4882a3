"""Seeded synthetic inputs for the INT8 linear layer.

This module draws random numbers and nothing else: no quantization, no rotation, no
GEMM.  Both the CUDA path and the CPU oracle are fed from it, so it must not hold any
of the method's arithmetic.  Every draw comes from a ``torch.Generator`` seeded with
an explicit integer, on the device the caller names (the CPU for the sizes the oracle
checks in full; the GPU for the multi-GB shapes, whose sampled rows are copied back).

Workload shapes follow the comfy-kitchen pages: the repro of issue #136 ("Minimal
reproduction": x bf16 ~N(0,1) [m,k], w int8 uniform [n,k], w_scale fp32 U(0,1)*0.01),
the A6000 sweep of PR #142 ("Numbers from the sweep"), the 4096^3 shape of issue #278
("What happens") and the ConvRot layout of issue #278 ("Suggested fix").
"""
from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch

TENSORWISE, PER_ROW, CONVROT = 0, 1, 2
MODE_NAMES = {TENSORWISE: "tensorwise", PER_ROW: "per_row", CONVROT: "convrot"}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed, std=1.0, device="cpu", outlier_channels=None, outlier_scale=20.0,
                chunk_rows=8192):
    """bf16 tensor of N(0, std^2) draws (fp32 draw rounded to bf16, round-to-nearest-even).

    ``outlier_channels``: optional 1-D index tensor of columns whose fp32 draw is
    multiplied by ``outlier_scale`` before rounding (the 1% x20 outlier recipe).
    Rows are drawn in chunks so multi-GB tensors need no fp32 copy of the whole.
    """
    rows, cols = shape
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    g = generator(seed, device)
    scale_vec = None
    if outlier_channels is not None and len(outlier_channels) > 0:
        scale_vec = torch.ones(cols, dtype=torch.float32, device=device)
        scale_vec[outlier_channels.to(device)] = float(outlier_scale)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        f = torch.randn((r1 - r0, cols), generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            f.mul_(std)
        if scale_vec is not None:
            f.mul_(scale_vec)
        out[r0:r1].copy_(f)
    return out


def normal_f32(shape, seed, std=1.0, device="cpu"):
    g = generator(seed, device)
    f = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    return f.mul_(std) if std != 1.0 else f


def int8_uniform(shape, seed, lo=-127, hi=127, device="cpu"):
    """int8 tensor uniform on the inclusive range [lo, hi]."""
    g = generator(seed, device)
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int8, device=device)


def scale_uniform(n, seed, mul=0.01, device="cpu"):
    """fp32 scales U(0,1) * mul."""
    g = generator(seed, device)
    return torch.rand((n,), generator=g, dtype=torch.float32, device=device).mul_(mul)


def outlier_columns(K, frac, seed):
    """floor(frac*K) distinct column indices from a seeded permutation."""
    n = int(frac * K)
    g = generator(seed, "cpu")
    return torch.randperm(K, generator=g)[:n]


@dataclass
class Case:
    """One linear-layer problem.  ``w`` is None for ConvRot cases, whose int8 weight is
    derived from ``w_float`` by the caller (the pre-rotation is not a random draw)."""
    name: str
    M: int
    N: int
    K: int
    mode: int
    x: torch.Tensor
    w: Optional[torch.Tensor]
    w_scale: Optional[torch.Tensor]
    bias: Optional[torch.Tensor]
    w_float: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)


def make_case(name, M, N, K, mode, *, bias=False, seed=1, device="cpu", outlier_frac=0.0,
              w_device=None) -> Case:
    """Draw the inputs of one problem.  Sub-seeds are fixed offsets of ``seed`` so
    every tensor has its own stream:  x: seed, w: seed+101, w_scale: seed+202,
    bias: seed+303, outlier columns: seed+404, ConvRot float weight: seed+505."""
    w_device = device if w_device is None else w_device
    oc = outlier_columns(K, outlier_frac, seed + 404) if outlier_frac > 0 else None
    x = normal_bf16((M, K), seed, device=device, outlier_channels=oc)
    b = normal_bf16((1, N), seed + 303, std=0.02, device=w_device).reshape(N) if bias else None
    if mode == CONVROT:
        wf = normal_f32((N, K), seed + 505, std=0.02, device=w_device)
        return Case(name, M, N, K, mode, x, None, None, b, w_float=wf,
                    meta={"outlier_columns": None if oc is None else oc.tolist()})
    w = int8_uniform((N, K), seed + 101, device=w_device)
    ws = scale_uniform(1 if mode == TENSORWISE else N, seed + 202, device=w_device)
    return Case(name, M, N, K, mode, x, w, ws, b)


# The workloads: (name, M, N, K, mode, bias, outlier_frac, seed)
PER_ROW_SMALL = ("per_row_256x512x512", 256, 512, 512, PER_ROW, False, 0.0, 1)
TENSORWISE_4096 = ("tensorwise_4096x4096x4096_bias", 4096, 4096, 4096, TENSORWISE, True, 0.0, 2)
SWEEP = [
    ("per_row_274x2048x2048", 274, 2048, 2048, PER_ROW, False, 0.0, 3),
    ("per_row_1024x4096x4096", 1024, 4096, 4096, PER_ROW, False, 0.0, 3),
    ("per_row_8192x16384x4096", 8192, 16384, 4096, PER_ROW, False, 0.0, 3),
    ("per_row_25900x16384x4096", 25900, 16384, 4096, PER_ROW, False, 0.0, 3),
    ("per_row_80666x28672x5376", 80666, 28672, 5376, PER_ROW, False, 0.0, 3),
]
LARGE_INDEX = [
    ("per_row_99864x21504x5376", 99864, 21504, 5376, PER_ROW, False, 0.0, 4),
    ("per_row_99865x21504x5376", 99865, 21504, 5376, PER_ROW, False, 0.0, 4),
    ("per_row_100000x21504x5376", 100000, 21504, 5376, PER_ROW, False, 0.0, 4),
]
CONVROT_4096 = ("convrot_4096x12288x3072_bias", 4096, 12288, 3072, CONVROT, True, 0.01, 5)

ALL_WORKLOADS = [PER_ROW_SMALL, TENSORWISE_4096, *SWEEP, *LARGE_INDEX, CONVROT_4096]


def case_from_spec(spec: Tuple, device="cpu", w_device=None) -> Case:
    name, M, N, K, mode, bias, outlier_frac, seed = spec
    return make_case(name, M, N, K, mode, bias=bias, seed=seed, device=device,
                     outlier_frac=outlier_frac, w_device=w_device)


def sample_rows(M, n_random=64, n_first=16, n_last=16, seed=1000):
    """Seeded row sample for shapes the oracle cannot finish in full: n_random rows
    drawn without replacement plus the first and last rows, sorted and unique."""
    g = generator(seed, "cpu")
    r = torch.randperm(M, generator=g)[:min(n_random, M)]
    rows = set(r.tolist()) | set(range(min(n_first, M))) | set(range(max(0, M - n_last), M))
    return sorted(rows)
