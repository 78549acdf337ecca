"""GPU: calls launched back to back on one stream, each reading the previous
call's output, with no host synchronisation in between.

Every kernel of a call is launched with programmatic stream serialization
allowed: its CTAs may be scheduled while the kernel before it is finishing,
and they wait (griddepcontrol.wait) before their first global-memory access.
The chains below check that each link reads only its predecessor's finished
output and writes nothing the predecessor still reads. With grids of 24-32
CTA pairs on a 76-pair device, the next kernel's CTAs find free SMs at once,
so a read taken before that wait would see the buffer's previous contents.

B is a signed permutation (B[perm[n], n] = s_n, zero elsewhere), so every
product is exact in any accumulation order and C[:, n] = s_n * A[:, perm[n]]:
the expected result of a whole chain is known in closed form.
"""
import pytest
import torch

from dense_gemm_gb300 import gemm, gemm_packed, gemm_splitk, gemm_splitk_noalloc, sync_status
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    from dense_gemm_gb300 import build
    build.build()
    torch.cuda.init()
    yield
    assert sync_status() == 0


def signed_permutation(n: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n, generator=g)
    sign = torch.where(torch.rand(n, generator=g) < 0.5, -1.0, 1.0)
    P = torch.zeros(n, n, dtype=torch.float16)
    P[perm, torch.arange(n)] = sign.half()
    return P, perm, sign


def apply(X: torch.Tensor, perm, sign, times: int) -> torch.Tensor:
    """X (fp16, CPU) after `times` multiplications by the signed permutation."""
    Y = X.float()
    for _ in range(times):
        Y = Y[:, perm] * sign
    return Y


def padded_view(M: int, K: int, dtype, pad: int = 3, offset: int = 1) -> torch.Tensor:
    """An [M, K] view whose rows are not 16-byte aligned (row stride K + pad)."""
    buf = torch.full((offset + M * (K + pad),), float("nan"), dtype=dtype, device="cuda")
    return buf.as_strided((M, K), (K + pad, 1), offset)


@pytest.mark.parametrize("M,K", [(2048, 1024), (4096, 512)])
def test_chain_of_dependent_calls_is_exact(M, K):
    X0 = torch.empty(M, K, dtype=torch.float16).uniform_(-4, 4, generator=torch.Generator().manual_seed(M + K))
    P, perm, sign = signed_permutation(K, seed=K)
    Pd = P.cuda()
    ping = X0.cuda()
    pong = torch.empty_like(ping)
    odd_a = padded_view(M, K, torch.float16)   # predicated loads / plain 16-bit stores
    f32 = torch.empty(M, K, device="cuda")
    steps = 0
    for _ in range(2):
        gemm(ping, Pd, pong)                                   # CTA pairs, TMA loads and stores
        gemm(pong, Pd, ping, single_cta=True)                  # one CTA per tile
        gemm(ping, Pd, pong, tail_split=True)                  # split tail (+ its reduction kernel)
        gemm(pong, Pd, ping, dynamic=True)                     # cluster launch control
        gemm(ping, Pd, odd_a)                                  # C rows off 16-byte boundaries
        gemm(odd_a, Pd, pong)                                  # operands through the predicated loader
        gemm_splitk(pong, Pd, f32, splits=4)                   # split-K (+ reduction kernel), fp32 C
        ping.copy_(f32)                                        # a library kernel between calls
        gemm_splitk_noalloc(ping, Pd, f32, splits=3)           # built-in scratch
        odd_a.copy_(f32)
        gemm_packed(odd_a, Pd, f32)                            # operand copy kernel, then the GEMM
        pong.copy_(f32)
        gemm(pong, Pd, ping, persistent=False)                 # one program per tile
        steps += 10
    torch.cuda.synchronize()
    assert sync_status() == 0
    expected = apply(X0, perm, sign, steps)
    assert torch.equal(ping.float().cpu(), expected)


def test_write_after_read_between_consecutive_calls():
    """Each call overwrites the operand the call before it reads: a store issued
    before the predecessor has finished reading would change its result."""
    M, K = 2048, 768
    X0 = torch.empty(M, K, dtype=torch.float16).uniform_(-2, 2, generator=torch.Generator().manual_seed(7))
    P, perm, sign = signed_permutation(K, seed=3)
    Pd = P.cuda()
    a = X0.cuda()
    b = torch.empty_like(a)
    outs = []
    for i in range(12):
        src, dst = (a, b) if i % 2 == 0 else (b, a)
        gemm(src, Pd, dst)
        if i % 4 == 3:
            outs.append((i + 1, dst.clone()))
    torch.cuda.synchronize()
    assert sync_status() == 0
    for n, o in outs:
        assert torch.equal(o.float().cpu(), apply(X0, perm, sign, n)), f"after {n} calls"
