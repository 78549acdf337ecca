"""Helpers shared by the GPU parity tests (comparison rules and sampling)."""
import math

import numpy as np
import torch

import oracle
from dense_gemm_gb300 import gemm, get_config


def require_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def to_dev(x: torch.Tensor) -> torch.Tensor:
    """Copy a host tensor to cuda:0 keeping its strides (and storage offset)."""
    storage = x.untyped_storage()
    base = torch.empty(0, dtype=x.dtype).set_(storage, 0, (storage.nbytes() // x.element_size(),), (1,))
    dev = base.to("cuda")
    return dev.as_strided(x.shape, x.stride(), x.storage_offset())


def error_bound(A: torch.Tensor, B: torch.Tensor) -> float:
    """max |C_gpu - C_ref| <= 2e-3 * sqrt(K) * max|A| * max|B| (stated tolerance)."""
    K = A.shape[1]
    amax = float(A.float().abs().max()) if A.numel() else 0.0
    bmax = float(B.float().abs().max()) if B.numel() else 0.0
    return 2e-3 * math.sqrt(max(K, 1)) * amax * bmax


def assert_within_bound(got: np.ndarray, ref: np.ndarray, A, B, what=""):
    got = np.asarray(got, dtype=np.float64)
    diff = np.abs(got - ref)
    bound = error_bound(A, B)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert diff.max(initial=0.0) <= bound, f"{what}: max|d|={diff.max():.3e} > {bound:.3e}"
    nref = np.linalg.norm(ref)
    if nref > 0:
        rel = np.linalg.norm(got - ref) / nref
        assert rel <= 1e-3, f"{what}: relative Frobenius error {rel:.3e} > 1e-3"


def run(A_host, B_host, grouped=True, cross_tile=True, G=8, out_layout=None, single_cta=False,
        persistent=True, dynamic=False, tail_split=False):
    """C = A @ B through the C ABI; returns (C_device_fp32, C_host_numpy)."""
    A = to_dev(A_host)
    B = to_dev(B_host)
    M, N = A.shape[0], B.shape[1]
    out = None
    if out_layout is not None:
        ld, off = out_layout
        buf = torch.full((off + M * ld,), float("nan"), dtype=torch.float32, device="cuda")
        out = buf.as_strided((M, N), (ld, 1), off)
    C = gemm(A, B, out, group_size_m=G, grouped=grouped, cross_tile=cross_tile,
             single_cta=single_cta, persistent=persistent, dynamic=dynamic, tail_split=tail_split)
    torch.cuda.synchronize()
    return C, C.cpu().numpy().astype(np.float64)


def sample_tiles(M, N, count, seed):
    """(row0, rows, col0, cols) of `count` output tiles of the kernel's tile
    shape, always including the first, the last and ragged-edge tiles."""
    cfg = get_config(M, N)
    bm, bn = cfg["bm"], cfg["bn"]
    nm, nn = -(-M // bm), -(-N // bn)
    rng = np.random.default_rng(seed)
    ids = {0, nm * nn - 1, (nm - 1) * nn, nn - 1}
    while len(ids) < min(count, nm * nn):
        ids.add(int(rng.integers(0, nm * nn)))
    out = []
    for t in sorted(ids):
        tm, tn = divmod(t, nn)
        r0, c0 = tm * bm, tn * bn
        out.append((r0, min(bm, M - r0), c0, min(bn, N - c0)))
    return out


def check_sampled_tiles(C_host, A, B, count=64, seed=0, exact=False, what=""):
    for (r0, nr, c0, nc) in sample_tiles(A.shape[0], B.shape[1], count, seed):
        ref = oracle.gemm_rows(A, B, rows=np.arange(r0, r0 + nr), col0=c0, ncols=nc)
        got = C_host[r0:r0 + nr, c0:c0 + nc]
        if exact:
            assert np.array_equal(got, ref), f"{what}: tile at ({r0},{c0}) differs"
        else:
            assert_within_bound(got, ref, A, B, f"{what} tile ({r0},{c0})")


def check_sampled_rows(C_host, A, B, count=4096, seed=0, exact=False, what=""):
    """`count` whole rows of C (always the first and the last), every column,
    against the oracle; `exact` for integer inputs, else the error bound."""
    M = A.shape[0]
    if M <= count:
        rows = np.arange(M)
    else:
        rng = np.random.default_rng(seed + 7)
        inner = rng.choice(np.arange(1, M - 1), size=count - 2, replace=False)
        rows = np.sort(np.concatenate([[0, M - 1], inner]))
    ref = oracle.gemm_rows(A, B, rows=rows)
    got = C_host[rows]
    if exact:
        assert np.array_equal(got, ref), f"{what}: sampled rows differ"
    else:
        assert_within_bound(got, ref, A, B, f"{what}: {rows.size} sampled rows")
    return rows.size


def check_row_col_sums(C_host, A, B, what=""):
    """Every row sum of C equals A @ (B @ 1) and every column sum equals
    (1^T A) @ B (float64, numpy); a tile written to the wrong place or left
    unwritten moves a whole row/column sum far outside the tolerance."""
    Af = A.double().numpy() if isinstance(A, torch.Tensor) else A
    Bf = B.double().numpy() if isinstance(B, torch.Tensor) else B
    rs_ref = Af @ Bf.sum(axis=1)
    cs_ref = Af.sum(axis=0) @ Bf
    absC = np.abs(C_host)
    tol_r = 1e-5 * absC.sum(axis=1) + 1e-3
    tol_c = 1e-5 * absC.sum(axis=0) + 1e-3
    assert np.all(np.abs(C_host.sum(axis=1) - rs_ref) <= tol_r), f"{what}: row sums"
    assert np.all(np.abs(C_host.sum(axis=0) - cs_ref) <= tol_c), f"{what}: column sums"
