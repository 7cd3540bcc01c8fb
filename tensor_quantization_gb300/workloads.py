"""Seeded synthetic inputs for the quantizer's workloads.

This module only draws random numbers (torch CPU ``Generator``) and records
each workload's settings; it holds none of the quantizer's arithmetic, so both
the CUDA path and the CPU oracle can consume the same tensors.

The five workloads follow the training recipe's operands:

* ``randn_rne_256x1024`` -- N(0,1), per-tensor scale, 1x16 blocks, RNE, rowwise,
  linear scales (small case).
* ``act_rht_sr_8192x4096`` -- activation with 0.1% outlier columns (x50),
  per-tensor scale, 16-point RHT then Philox stochastic rounding, rowwise,
  32x4x4-swizzled scales.
* ``weight_2d_rne_14336x4096`` -- N(0, 0.02^2) weight, one scale per 16x16 tile,
  RNE, rowwise and columnwise outputs from one read.
* ``grad_col_rht_sr_16384x8192`` -- Student-t (nu=3) x 1e-3 gradient, RHT + SR
  along M (columnwise), swizzled scales.
* ``rowscaled_4o6_8192x8192`` -- rows with log-uniform std in [1e-3, 10],
  per-row global scales, four-over-six, rowwise.

Two more measure follow-up forms on the activation input:

* ``act_rht_sr_given_8192x4096`` -- quantized with its amax given
  (``NVFP4_AMAX_GIVEN``, e.g. from delayed scaling), so the call is the encode
  pass alone.
* ``act_rht_sr_rowcol_8192x4096`` -- RHT + SR in both orientations (the wgrad
  operand: rowwise and columnwise codes, one amax and global scale each).
* ``act_rht_sr_groups_8192x4096`` -- RHT + SR over 8 row groups of uneven
  sizes (one empty, one of a single row), each with its own amax and global
  scale (grouped MoE-style quantize).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    cols: int
    seed: int
    mode: str  # "rne" | "sr" | "4o6"
    rht: bool = False
    block2d: bool = False
    per_row: bool = False
    swizzled: bool = False
    rowwise: bool = True
    colwise: bool = False
    philox_seed: int = 0
    philox_offset: int = 0
    recipe: str = "randn"  # randn | outlier_cols | weight | student_t | rowscaled
    amax_given: bool = False  # the call gets the per-tensor amax (NVFP4_AMAX_GIVEN): no amax pass
    groups: tuple = ()  # row offsets of the groups of a grouped call (n_groups + 1), else empty

    def resized(self, rows: int, cols: int) -> "Workload":
        return replace(self, rows=rows, cols=cols, name=f"{self.name}@{rows}x{cols}")

    @property
    def numel(self) -> int:
        return self.rows * self.cols


WORKLOADS = {
    w.name: w
    for w in [
        Workload("randn_rne_256x1024", 256, 1024, 0, "rne", recipe="randn"),
        Workload("act_rht_sr_8192x4096", 8192, 4096, 1, "sr", rht=True, swizzled=True,
                 philox_seed=1, philox_offset=0, recipe="outlier_cols"),
        Workload("weight_2d_rne_14336x4096", 14336, 4096, 2, "rne", block2d=True, rowwise=True,
                 colwise=True, recipe="weight"),
        Workload("grad_col_rht_sr_16384x8192", 16384, 8192, 3, "sr", rht=True, swizzled=True,
                 rowwise=False, colwise=True, philox_seed=3, philox_offset=0, recipe="student_t"),
        Workload("rowscaled_4o6_8192x8192", 8192, 8192, 4, "4o6", per_row=True, recipe="rowscaled"),
        Workload("act_rht_sr_given_8192x4096", 8192, 4096, 1, "sr", rht=True, swizzled=True,
                 philox_seed=1, philox_offset=0, recipe="outlier_cols", amax_given=True),
        Workload("act_rht_sr_rowcol_8192x4096", 8192, 4096, 1, "sr", rht=True, swizzled=True, colwise=True,
                 philox_seed=1, philox_offset=0, recipe="outlier_cols"),
        Workload("act_rht_sr_groups_8192x4096", 8192, 4096, 1, "sr", rht=True, swizzled=True,
                 philox_seed=1, philox_offset=0, recipe="outlier_cols",
                 groups=(0, 100, 1124, 1124, 4000, 4001, 6000, 7999, 8192)),
    ]
}

# The configuration the headline throughput is quoted on.
HEADLINE = "act_rht_sr_8192x4096"


def _sign_mask(g: torch.Generator) -> int:
    bits = torch.randint(0, 2, (16,), generator=g)
    return int(sum(int(b) << j for j, b in enumerate(bits.tolist())))


def make_input(w: Workload) -> tuple[torch.Tensor, int]:
    """Return (bf16 CPU tensor [rows, cols], 16-bit RHT sign mask) for ``w``.

    The sign mask is 0 for workloads without RHT.
    """
    g = torch.Generator().manual_seed(w.seed)
    R, C = w.rows, w.cols
    mask = 0
    if w.recipe == "randn":
        x = torch.randn(R, C, generator=g)
    elif w.recipe == "outlier_cols":
        x = torch.randn(R, C, generator=g)
        n_out = max(1, round(0.001 * C))
        cols = torch.randperm(C, generator=g)[:n_out]
        x[:, cols] *= 50.0
        mask = _sign_mask(g)
    elif w.recipe == "weight":
        x = torch.randn(R, C, generator=g) * 0.02
    elif w.recipe == "student_t":
        z = torch.randn(R, C, generator=g)
        chi2 = torch.zeros(R, C)
        for _ in range(3):
            chi2 += torch.randn(R, C, generator=g).square_()
        x = z.div_(chi2.div_(3.0).sqrt_()).mul_(1e-3)
        del chi2
        mask = _sign_mask(g)
    elif w.recipe == "rowscaled":
        sigma = torch.exp(math.log(1e-3) + torch.rand(R, generator=g) * math.log(1e4))
        x = torch.randn(R, C, generator=g) * sigma[:, None]
    else:
        raise ValueError(f"unknown recipe {w.recipe}")
    return x.to(torch.bfloat16).contiguous(), mask
