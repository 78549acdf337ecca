"""GPU parity of gemm_f16_packed: operands copied onto 128-byte lines in a
caller workspace, then the GEMM. Same bar as the other parity tests: integer
inputs bit-exact against the oracle, random inputs within the stated bound;
and C bit-identical to gemm_f16 on the caller's layout (the same products,
summed in the same order)."""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_gb300 import gemm, gemm_packed, packed_workspace_size, sync_status
from dense_gemm_gb300.inputs import WORKLOADS, draw
from gpu_util import check_row_col_sums, check_sampled_rows, check_sampled_tiles, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    from dense_gemm_gb300 import build
    build.build()
    torch.cuda.init()
    yield
    assert sync_status() == 0


def nan_layout(x: torch.Tensor, layout: str, pad: int, offset: int) -> torch.Tensor:
    """`x` in a row- or column-major view with leading dimension (+pad) and a
    storage offset, inside a buffer whose other elements are NaN: a copy that
    took a neighbouring element into the product would show it."""
    rows, cols = x.shape
    ld = (cols if layout == "row" else rows) + pad
    n = offset + (rows if layout == "row" else cols) * ld
    buf = torch.full((n,), float("nan"), dtype=x.dtype)
    view = buf.as_strided((rows, cols), (ld, 1) if layout == "row" else (1, ld), offset)
    view.copy_(x)
    return view


def both(A_host, B_host, ws=None):
    """(gemm_f16_packed C, gemm_f16 C) on the same device operands."""
    A, B = to_dev(A_host), to_dev(B_host)
    Cp = gemm_packed(A, B, workspace=ws)
    Cd = gemm(A, B)
    torch.cuda.synchronize()
    assert sync_status() == 0
    return Cp.cpu().numpy().astype(np.float64), Cd.cpu().numpy().astype(np.float64)


CASES = [
    # (M, N, K, a_layout, a_pad, a_off, b_layout, b_pad, b_off)
    (300, 500, 257, "row", 0, 0, "col", 0, 0),     # K-major rows of 514 bytes (not 16-byte aligned)
    (300, 500, 257, "row", 3, 1, "col", 5, 3),     # odd leading dimensions, 2-byte-aligned bases
    (256, 256, 200, "row", 8, 8, "row", 8, 0),     # 16-byte aligned, not on 128-byte lines
    (130, 270, 136, "col", 2, 1, "row", 6, 5),     # M-major A, N-major B
    (129, 257, 65, "col", 0, 0, "col", 1, 7),
    (1, 1, 1, "row", 0, 1, "row", 0, 1),
    (7, 1000, 33, "row", 1, 0, "row", 3, 2),
    (512, 384, 128, "row", 0, 0, "row", 0, 0),     # already on 128-byte lines: read in place
]


@pytest.mark.parametrize("case", CASES)
def test_packed_integer_exact_and_identical(case):
    M, N, K, al, ap, ao, bl, bp, bo = case
    A = draw(M, K, "int", 40 + M)
    B = draw(K, N, "int", 41 + N)
    Cp, Cd = both(nan_layout(A, al, ap, ao), nan_layout(B, bl, bp, bo))
    assert np.array_equal(Cp, oracle.gemm(A, B))
    assert np.array_equal(Cp, Cd)


@pytest.mark.parametrize("case", CASES[:5])
def test_packed_random_within_bound_and_identical(case):
    M, N, K, al, ap, ao, bl, bp, bo = case
    A = draw(M, K, "uniform", 50 + M)
    B = draw(K, N, "uniform", 51 + N)
    Cp, Cd = both(nan_layout(A, al, ap, ao), nan_layout(B, bl, bp, bo))
    from gpu_util import assert_within_bound
    assert_within_bound(Cp, oracle.gemm(A, B), A, B, "packed")
    assert np.array_equal(Cp, Cd)


def test_packed_workspace_reused_across_calls():
    """One workspace, consecutive calls with different shapes and layouts on one
    stream: each result is exact."""
    shapes = [(300, 500, 257), (640, 200, 1000), (100, 700, 130)]
    need = max(packed_workspace_size(M, N, K, K + 1, 1, 1, K + 3) for (M, N, K) in shapes)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for i, (M, N, K) in enumerate(shapes):
        A = draw(M, K, "int", 60 + i)
        B = draw(K, N, "int", 70 + i)
        Cp, _ = both(nan_layout(A, "row", 1, 0), nan_layout(B, "col", 3, 1), ws=ws)
        assert np.array_equal(Cp, oracle.gemm(A, B)), (M, N, K)


def test_packed_small_workspace_raises():
    from dense_gemm_gb300 import GemmError
    A = to_dev(nan_layout(draw(64, 100, "int", 1), "row", 1, 0))
    B = to_dev(draw(100, 64, "int", 2))
    need = packed_workspace_size(64, 64, 100, 101, 1, 64, 1)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(GemmError, match="INVALID_ARG"):
        gemm_packed(A, B, workspace=ws)


def _full_packed(name, exact_dist=False, count=64):
    w = WORKLOADS[name]
    A, B = w.operands()
    if exact_dist:
        from dense_gemm_gb300.inputs import relayout
        A = draw(w.M, w.K, "int", w.seed)
        B = draw(w.K, w.N, "int", w.seed + 1)
        if w.b_layout != "row":
            B = relayout(B, w.b_layout)
    Ad, Bd = to_dev(A), to_dev(B)
    C = gemm_packed(Ad, Bd)
    Cd = gemm(Ad, Bd)
    torch.cuda.synchronize()
    assert sync_status() == 0
    assert torch.equal(C, Cd), f"{name}: gemm_f16_packed differs from gemm_f16"
    Ch = C.cpu().numpy().astype(np.float64)
    check_sampled_tiles(Ch, A, B, count=count, seed=w.seed, exact=exact_dist, what=name)
    assert check_sampled_rows(Ch, A, B, count=4096, seed=w.seed, exact=exact_dist, what=name) >= min(4096, w.M)
    check_row_col_sums(Ch, A, B, what=name)


def test_packed_full_ragged_4000x5000x3000():
    _full_packed("ragged_4000x5000x3000")


def test_packed_full_ragged_8191x8191x257():
    _full_packed("ragged_8191x8191x257")


def test_packed_full_ragged_8191x8191x257_integer_exact():
    _full_packed("ragged_8191x8191x257", exact_dist=True, count=32)


def test_packed_full_unaligned_8192x8192x4100():
    """8200-byte rows of A and B (the alignment-class loader's case in gemm_f16);
    sampled tiles and rows against the oracle, and bit-identical to gemm_f16."""
    _full_packed("unaligned_8192x8192x4100", count=16)
