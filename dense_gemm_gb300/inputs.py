"""Seeded synthetic operands and the workload catalogue.

This module draws random numbers and lays them out in memory; it contains none
of the GEMM's arithmetic. Tests feed the same tensors to the CUDA path and to
the oracle, and bench.py uses it for its inputs.

Recipe: values are drawn in fp32 on the host from ``torch.Generator`` seeded
per operand, then rounded to fp16 with round-to-nearest-even (``.half()``).
Distributions: ``uniform`` = U[-1, 1), ``normal`` = N(0, 1), ``int`` = integers
in [-4, 4] (every partial sum of a K <= 4096 product is an integer below 2^24,
so an fp32 accumulation is exact in any order).
"""
from dataclasses import dataclass, field

import torch


def draw(rows: int, cols: int, dist: str, seed: int) -> torch.Tensor:
    """A dense row-major [rows, cols] fp16 CPU tensor."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (rows, cols)
    if dist == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32)
    elif dist == "int":
        x = torch.randint(-4, 5, shape, generator=g, dtype=torch.int32).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.half()


def relayout(x: torch.Tensor, layout: str = "row", pad: int = 0, offset: int = 0) -> torch.Tensor:
    """The same logical matrix in another memory layout.

    layout ``row``: unit stride along columns, leading dimension cols + pad.
    layout ``col``: unit stride along rows, leading dimension rows + pad.
    ``offset`` shifts the first element by that many elements inside a larger
    buffer (an offset of 1 makes the base address only 2-byte aligned).
    """
    rows, cols = x.shape
    if layout == "row":
        ld = cols + pad
        buf = torch.zeros(offset + rows * ld, dtype=x.dtype, device=x.device)
        view = buf.as_strided((rows, cols), (ld, 1), offset)
    elif layout == "col":
        ld = rows + pad
        buf = torch.zeros(offset + cols * ld, dtype=x.dtype, device=x.device)
        view = buf.as_strided((rows, cols), (1, ld), offset)
    else:
        raise ValueError(f"unknown layout {layout!r}")
    view.copy_(x)
    return view


@dataclass(frozen=True)
class Workload:
    """One GEMM problem: shapes, value distribution, layouts, seeds."""
    name: str
    M: int
    N: int
    K: int
    dist: str
    a_layout: str = "row"
    b_layout: str = "row"
    seed: int = 1000
    notes: str = ""
    tags: tuple = field(default_factory=tuple)

    def operands(self):
        """(A [M,K], B [K,N]) fp16 host tensors in the workload's layouts."""
        A = draw(self.M, self.K, self.dist, self.seed)
        B = draw(self.K, self.N, self.dist, self.seed + 1)
        if self.a_layout != "row":
            A = relayout(A, self.a_layout)
        if self.b_layout != "row":
            B = relayout(B, self.b_layout)
        return A, B

    def describe(self) -> str:
        return (f"gemm_f16 M={self.M} N={self.N} K={self.K} fp16 in, fp32 acc+out; "
                f"A {self.a_layout}-major, B {self.b_layout}-major; {self.dist} values")


def _k_sweep():
    return {f"ksweep_16384x16384x{k}": Workload(f"ksweep_16384x16384x{k}", 16384, 16384, k,
                                                "uniform", seed=1040 + 2 * i, tags=("ksweep",))
            for i, k in enumerate((128, 512, 1024, 2048, 4096))}


WORKLOADS = {
    "square_512": Workload("square_512", 512, 512, 512, "uniform", seed=1010),
    "square_8192x8192x4096": Workload("square_8192x8192x4096", 8192, 8192, 4096, "uniform",
                                      seed=1020),
    "square_16384x16384x4096": Workload("square_16384x16384x4096", 16384, 16384, 4096,
                                        "normal", seed=1030, tags=("headline",)),
    **_k_sweep(),
    "ragged_4000x5000x3000": Workload("ragged_4000x5000x3000", 4000, 5000, 3000, "uniform",
                                      b_layout="col", seed=1050, tags=("ragged",)),
    "ragged_8191x8191x257": Workload("ragged_8191x8191x257", 8191, 8191, 257, "uniform",
                                     b_layout="col", seed=1060, tags=("ragged",)),
    # the headline's B operand (16384 columns: one grouped band of B panels larger
    # than L2) with half its rows: the case for multi-pass profiler captures of the
    # headline's L2 behaviour (not one of the pages' shapes)
    "half_8192x16384x4096": Workload("half_8192x16384x4096", 8192, 16384, 4096, "normal", seed=1080,
                                     tags=("study",)),
    # long K with 8200-byte rows of A and B (not 16-byte multiples): the case operand
    # copies (gemm_f16_packed) are for (not one of the pages' shapes)
    "unaligned_8192x8192x4100": Workload("unaligned_8192x8192x4100", 8192, 8192, 4100, "uniform",
                                         b_layout="col", seed=1090, tags=("study",)),
    # few output tiles, long K: the case split-K is for (not one of the pages' shapes)
    "longk_1024x1024x32768": Workload("longk_1024x1024x32768", 1024, 1024, 32768, "uniform",
                                      seed=1070, tags=("study",)),
}

HEADLINE = "square_16384x16384x4096"
