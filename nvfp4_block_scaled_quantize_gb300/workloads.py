"""Seeded synthetic inputs shaped like LLM/MoE training tensors.

This module only draws random inputs (numpy PCG64 streams, rounded to BF16 by torch's
round-to-nearest-even cast). It holds none of the quantizer's arithmetic, and it is the one
module that both the CUDA path's tests/benchmark and the CPU oracle's tests take inputs from.

The pages measure on DeepSeek-V3 671B FFN tensors (hidden 7168, four local experts; page
"[nvfp4_training] Optimize CuteDSL kernels for NVFP4 training", section "Performance"). No
dataset or checkpoint is used: these synthetic tensors stand in for those activations,
weights and gradients.
"""
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One benchmark/parity configuration: the tensor's shape and distribution and the
    quantizer options it is run with."""
    name: str
    rows: int
    cols: int
    dist: str                 # "normal", "normal_outliers", "laplace"
    scale: float              # standard deviation (normal) or diversity b (laplace)
    seed: int
    rowwise: bool = True
    columnwise: bool = False
    block2d: bool = False
    round_row_sr: bool = False
    round_col_sr: bool = False
    rht_col: bool = False
    experts: int = 0          # > 0: grouped (MoE) input with that many experts
    zero_experts: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def grouped(self) -> bool:
        return self.experts > 0


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tensor_256x512_row_rtne", 256, 512, "normal", 1.0, 1),
        Workload("activation_8192x4096_rowcol_rtne", 8192, 4096, "normal_outliers", 1.0, 2,
                 columnwise=True, extra={"outlier_fraction": 0.001, "outlier_gain": 100.0}),
        Workload("weight_4096x14336_2d_rtne", 4096, 14336, "normal", 0.02, 3,
                 columnwise=True, block2d=True),
        Workload("gradient_16384x8192_row_rtne_col_rht_sr", 16384, 8192, "laplace", 1e-3, 4,
                 columnwise=True, rht_col=True, round_col_sr=True),
        Workload("moe_64experts_32768x7168_row_rtne_col_rht_sr", 32768, 7168, "normal", 1.0, 5,
                 columnwise=True, rht_col=True, round_col_sr=True, experts=64, zero_experts=4),
        # four local experts' gate/up weights stacked along the rows (the pages' grouped 2D
        # weight quantize, DeepSeek-V3 hidden 7168), equal row counts
        Workload("moe_weights_4experts_16384x7168_2d_rtne", 16384, 7168, "normal", 0.02, 6,
                 columnwise=True, block2d=True, experts=4, extra={"equal_experts": True}),
    ]
}


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 numpy array -> CPU torch.bfloat16 tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal(rows, cols, std, seed) -> torch.Tensor:
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((rows, cols), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return to_bf16(a)


def normal_with_outliers(rows, cols, seed, fraction=0.001, gain=100.0) -> torch.Tensor:
    """N(0,1) with ``fraction`` of the positions (a seeded sample without replacement)
    multiplied by ``gain``."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((rows, cols), dtype=np.float32)
    n_out = int(round(fraction * rows * cols))
    pos = rng.choice(rows * cols, size=n_out, replace=False)
    a.reshape(-1)[pos] *= np.float32(gain)
    return to_bf16(a)


def laplace(rows, cols, b, seed) -> torch.Tensor:
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.laplace(0.0, b, size=(rows, cols)).astype(np.float32)
    return to_bf16(a)


def expert_offsets(tokens, experts, zero_experts, seed) -> np.ndarray:
    """Cumulative int32 expert ends: counts ~ Multinomial(tokens, p) with p proportional to
    exp(N(0,1)) and a seeded subset of ``zero_experts`` experts given p = 0."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    w = np.exp(rng.standard_normal(experts))
    if zero_experts:
        w[rng.choice(experts, size=zero_experts, replace=False)] = 0.0
    p = w / w.sum()
    counts = rng.multinomial(tokens, p)
    return np.cumsum(counts).astype(np.int32)


def sign_mask(seed) -> int:
    """The 16 random signs of the Hadamard transform, bit i set meaning d_i = -1."""
    rng = np.random.Generator(np.random.PCG64(seed + 2000))
    return int(rng.integers(0, 1 << 16))


def make_input(w: Workload, rows: int = None) -> dict:
    """The workload's seeded input. ``rows`` overrides the row count (a smaller case of the same
    distribution; grouped inputs then keep the expert count with proportionally fewer tokens)."""
    rows = w.rows if rows is None else rows
    if w.dist == "normal":
        x = normal(rows, w.cols, w.scale, w.seed)
    elif w.dist == "normal_outliers":
        x = normal_with_outliers(rows, w.cols, w.seed, w.extra["outlier_fraction"],
                                 w.extra["outlier_gain"])
    elif w.dist == "laplace":
        x = laplace(rows, w.cols, w.scale, w.seed)
    else:
        raise ValueError(w.dist)
    out = {"x": x, "seed": w.seed, "offset": 0,
           "sign_mask": sign_mask(w.seed) if w.rht_col else 0}
    if w.grouped and w.extra.get("equal_experts"):
        out["offsets"] = (np.arange(1, w.experts + 1) * (rows // w.experts)).astype(np.int32)
    elif w.grouped:
        out["offsets"] = expert_offsets(rows, w.experts, w.zero_experts, w.seed)
    return out


def random_bf16_bits(shape, seed, finite_only=True) -> np.ndarray:
    """Uniformly random BF16 bit patterns (every exponent, both signs), as uint16."""
    rng = np.random.Generator(np.random.PCG64(seed))
    bits = rng.integers(0, 1 << 16, size=shape, dtype=np.uint32).astype(np.uint16)
    if finite_only:
        bad = (bits & 0x7F80) == 0x7F80
        bits[bad] &= 0xBFFF  # clear the top exponent bit: a finite pattern
    return bits
