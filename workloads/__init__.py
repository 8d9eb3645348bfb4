"""Seeded synthetic workloads for fused residual-add + RMSNorm + FP4 quantization.

This module only draws random numbers and names shapes: it holds none of the
method's arithmetic (no add, no normalisation, no rounding to FP4), so both the
CUDA path and the CPU oracle can take their inputs from it without sharing any
of the computation.

Recipe (all configurations):
  * input ``x`` and ``residual`` are N(mean 0, std sigma) drawn in fp32 with a
    torch generator seeded per (seed, tensor, row block), then rounded to the
    storage dtype (bf16 or fp16) by torch's round-to-nearest-even cast;
  * ``weight`` = 1 + 0.1 * N(0, 1), rounded to the same dtype;
  * optional outlier columns: a seeded permutation picks round(0.01 * H)
    columns of ``x`` which are multiplied by 50 before the rounding.

Row blocks of 4096 rows are drawn with their own generator, so a tensor is the
same whatever device memory is available, and rows of a large tensor can be
generated without materialising all of it in fp32.
"""
from __future__ import annotations

import dataclasses
import itertools
from typing import Dict, List, Optional

import torch

NVFP4 = "nvfp4"   # 16-element blocks, E4M3 scales
MXFP4 = "mxfp4"   # 32-element blocks, UE8M0 scales

ROWMAJOR = "rowmajor"
SWIZZLED = "swizzled"
BOTH = "both"

E4M3_B32 = "e4m3b32"  # 32-element blocks, E4M3 scales
BLOCK_SIZE = {NVFP4: 16, MXFP4: 32, E4M3_B32: 32}

_ROW_BLOCK = 4096


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    H: int
    dtype: str            # "bf16" or "fp16"
    fmt: str              # NVFP4 or MXFP4
    sf_layout: str        # ROWMAJOR, SWIZZLED or BOTH
    eps: float
    x_std: float = 1.0
    r_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_gain: float = 50.0
    seed: int = 0

    @property
    def block(self) -> int:
        return BLOCK_SIZE[self.fmt]

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def algorithmic_bytes(self, op: str = "fused") -> int:
        """HBM bytes one call must move.  Fused op: read x and r, write r,
        write the packed codes and every scale layout asked for, read the
        weight once.  Standalone quantize: read x, write codes and scales.
        Swizzle padding is not counted."""
        nb = self.H // self.block
        n_layouts = 2 if self.sf_layout == BOTH else 1
        if op == "quantize":
            return self.M * (2 * self.H + self.H // 2 + n_layouts * nb)
        return self.M * (6 * self.H + self.H // 2 + n_layouts * nb) + 2 * self.H

    def with_shape(self, M: int, H: Optional[int] = None) -> "Workload":
        return dataclasses.replace(self, M=M, H=self.H if H is None else H)


# The five workload families.  C1..C4 are single shapes; C5 is a sweep.
C1 = Workload("C1_M4_H256_bf16_nvfp4_rowmajor", 4, 256, "bf16", NVFP4, ROWMAJOR, 1e-6, seed=1)
C2 = Workload("C2_M128_H4096_bf16_nvfp4_swizzled", 128, 4096, "bf16", NVFP4, SWIZZLED, 1e-6,
              r_std=2.0, seed=2)
C3 = Workload("C3_M8192_H7168_bf16_mxfp4_swizzled_outliers", 8192, 7168, "bf16", MXFP4, SWIZZLED,
              1e-6, outlier_frac=0.01, seed=3)
C4 = Workload("C4_M16384_H5120_fp16_nvfp4_both", 16384, 5120, "fp16", NVFP4, BOTH, 1e-5, seed=4)

SWEEP_M = (1, 41, 512, 32768)
SWEEP_H = (1536, 6144, 17408, 32768)


def sweep() -> List[Workload]:
    out = []
    for fmt, M, H in itertools.product((NVFP4, MXFP4), SWEEP_M, SWEEP_H):
        out.append(Workload(f"C5_M{M}_H{H}_bf16_{fmt}_swizzled", M, H, "bf16", fmt, SWIZZLED,
                            1e-6, seed=5))
    return out


CONFIGS: Dict[str, Workload] = {w.name: w for w in (C1, C2, C3, C4, *sweep())}


def _gen(seed: int, tensor_id: int, block_idx: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tensor_id * 7_919 + block_idx * 104_729) & 0x7FFF_FFFF_FFFF)
    return g


def outlier_columns(wl: Workload) -> torch.Tensor:
    """The seeded set of outlier columns of ``x`` (CPU int64 tensor, sorted)."""
    n = int(round(wl.outlier_frac * wl.H))
    if n == 0:
        return torch.zeros(0, dtype=torch.int64)
    g = _gen(wl.seed, 99, 0, "cpu")
    return torch.sort(torch.randperm(wl.H, generator=g)[:n]).values


def make_rows(wl: Workload, which: str, row0: int, row1: int, device="cpu") -> torch.Tensor:
    """Rows [row0, row1) of tensor ``which`` ("x" or "r"), in the storage dtype.

    Row blocks are aligned to multiples of 4096 rows so any row range gives
    the same values as the full tensor.
    """
    tid, std = {"x": (1, wl.x_std), "r": (2, wl.r_std)}[which]
    cols = outlier_columns(wl).to(device) if which == "x" else None
    parts = []
    b0 = row0 // _ROW_BLOCK
    b1 = (row1 + _ROW_BLOCK - 1) // _ROW_BLOCK
    for b in range(b0, b1):
        lo = b * _ROW_BLOCK
        hi = min(lo + _ROW_BLOCK, wl.M)
        blk = torch.randn(hi - lo, wl.H, generator=_gen(wl.seed, tid, b, device),
                          device=device, dtype=torch.float32)
        if std != 1.0:
            blk.mul_(std)
        if cols is not None and cols.numel():
            blk[:, cols] *= wl.outlier_gain
        s0 = max(row0, lo) - lo
        s1 = min(row1, hi) - lo
        parts.append(blk[s0:s1].to(wl.torch_dtype))
    if not parts:
        return torch.empty(0, wl.H, dtype=wl.torch_dtype, device=device)
    return torch.cat(parts, 0)


def make_weight(wl: Workload, device="cpu") -> torch.Tensor:
    g = _gen(wl.seed, 3, 0, device)
    w = 1.0 + 0.1 * torch.randn(wl.H, generator=g, device=device, dtype=torch.float32)
    return w.to(wl.torch_dtype)


def make_inputs(wl: Workload, device="cpu"):
    """(x, residual, weight) for the whole workload on ``device``."""
    x = make_rows(wl, "x", 0, wl.M, device)
    r = make_rows(wl, "r", 0, wl.M, device)
    w = make_weight(wl, device)
    return x, r, w


# ---------------------------------------------------------------------------
# Consumer GEMM: operand bytes are drawn directly (packed codes and scale
# bytes), never computed, so the oracle and the kernel read identical bytes.
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class GemmWorkload:
    name: str
    M: int
    N: int
    K: int
    seed: int = 0

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def algorithmic_bytes(self) -> int:
        """Operands (codes + tiled scales, padding excluded) read once, bf16
        output written once."""
        return (self.M + self.N) * (self.K // 2 + self.K // 16) + 2 * self.M * self.N


# The FlashRT fp4-gemm README's release-gate shapes (M = 41 decode rows against
# 1536 / 6144 wide weights) and a prefill-sized product: the 8192 x 7168
# activations of the MXFP4 workload above times a square 7168 weight.
GEMM_CONFIGS: Dict[str, GemmWorkload] = {w.name: w for w in (
    GemmWorkload("G1_M41_N4608_K1536", 41, 4608, 1536, seed=11),
    GemmWorkload("G2_M41_N6144_K1536", 41, 6144, 1536, seed=12),
    GemmWorkload("G3_M41_N1536_K6144", 41, 1536, 6144, seed=13),
    GemmWorkload("G4_M8192_N7168_K7168", 8192, 7168, 7168, seed=14),
)}


def random_bytes(n: int, seed: int, tensor_id: int, alphabet=None, device="cpu") -> torch.Tensor:
    """n seeded bytes (uint8), uniform over 0..255 or over `alphabet` (a list of
    byte values).  Drawn on the CPU, so the bytes do not depend on the device."""
    g = _gen(seed, 100 + tensor_id, 0, "cpu")
    if alphabet is None:
        out = torch.randint(0, 256, (n,), generator=g, dtype=torch.int32)
    else:
        table = torch.tensor(list(alphabet), dtype=torch.int32)
        out = table[torch.randint(0, len(table), (n,), generator=g)]
    return out.to(torch.uint8).to(device)
