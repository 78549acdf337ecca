"""The allocation-free split-K entry point (gemm_f16_splitk_noalloc).

It exists for callers that must not allocate device memory where they
multiply (memory owned by another allocator or a fixed arena; no room for the
synchronisation or the out-of-memory failure of cudaMalloc on that path). It
uses a 32 MiB array built into the library instead of a caller workspace.
These tests call it through the C ABI and check it against the existing
split-K entry point (with a caller workspace), within the parity tolerance,
on two calls in a row (the shared array keeps the previous call's contents).
This file runs last so that a failure here comes after every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_gb300.inputs import draw
from gpu_util import assert_within_bound, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    from dense_gemm_gb300 import build
    build.build()


@pytest.mark.parametrize("M,N,K,splits", [(512, 512, 512, 0), (1024, 768, 8192, 4), (300, 304, 2000, 3)])
def test_noalloc_matches_splitk_on_two_calls_in_a_row(M, N, K, splits):
    from dense_gemm_gb300 import gemm_splitk, gemm_splitk_noalloc, splitk_workspace_size, sync_status
    need, used = splitk_workspace_size(M, N, K, splits)
    assert used > 1 and 0 < need <= 32 << 20
    A = draw(M, K, "normal", 300 + M)
    B = draw(K, N, "normal", 301 + N)
    Ad, Bd = to_dev(A), to_dev(B)
    ref = gemm_splitk(Ad, Bd, splits=splits)  # existing entry point, caller workspace
    torch.cuda.synchronize()
    ref_h = ref.cpu().numpy().astype(np.float64)
    exact = oracle.gemm(A, B)
    for call in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        gemm_splitk_noalloc(Ad, Bd, C, splits=splits)
        assert sync_status() == 0
        got = C.cpu().numpy().astype(np.float64)
        assert_within_bound(got, ref_h, A, B, f"no-alloc call {call} vs gemm_f16_splitk")
        assert_within_bound(got, exact, A, B, f"no-alloc call {call} vs oracle")


def test_noalloc_rejects_problems_larger_than_its_scratch():
    from dense_gemm_gb300 import GemmError, gemm_splitk_noalloc, splitk_workspace_size
    need, used = splitk_workspace_size(4096, 4096, 4096, 8)
    assert need > 32 << 20
    A = torch.zeros(4096, 4096, dtype=torch.float16, device="cuda")
    C = torch.zeros(4096, 4096, device="cuda")
    with pytest.raises(GemmError) as e:
        gemm_splitk_noalloc(A, A, C, splits=8)
    assert e.value.status == 2  # GEMM_ERR_UNSUPPORTED
