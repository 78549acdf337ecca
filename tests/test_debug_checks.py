"""The checked library (GEMM_DEBUG) on the GPU: device-side bounds and alignment
checks stand in for a sanitizer run. Every TMA copy's coordinates, every shared
memory access of the wrappers, every TMEM load's columns and every plain store
of C are checked; a failed check records GEMM_ERR_CHECK and skips the access.
The cases cover every store path, both kernels, the alignment-class loader,
split-K, the split tail, 16-bit C, the dynamic schedule, the operand copies of
gemm_f16_packed and the degenerate sizes, on integer inputs (exact)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu

CHILD = r'''
import json, numpy as np, torch
import oracle
from dense_gemm_gb300 import (gemm, gemm_splitk, splitk_workspace_size, sync_status,
                              selftest_check, library_path)
from dense_gemm_gb300.inputs import draw, relayout

def dev(x):
    st = x.untyped_storage()
    base = torch.empty(0, dtype=x.dtype).set_(st, 0, (st.nbytes() // x.element_size(),), (1,)).cuda()
    return base.as_strided(x.shape, x.stride(), x.storage_offset())

out = {"library": library_path(), "cases": []}
def case(name, M, N, K, la=("row", 0, 0), lb=("row", 0, 0), c=None, dtype=torch.float32, **kw):
    A0 = draw(M, K, "int", 7 + M)
    B0 = draw(K, N, "int", 8 + N)
    want = oracle.round_output(oracle.gemm(A0, B0), {torch.float32: "f32", torch.float16: "f16",
                                                     torch.bfloat16: "bf16"}[dtype], 1.0)
    if K == 0:
        A = torch.zeros((M, 0), dtype=torch.float16, device="cuda")
        B = torch.zeros((0, N), dtype=torch.float16, device="cuda")
    else:
        A = dev(relayout(A0, la[0], pad=la[1], offset=la[2]))
        B = dev(relayout(B0, lb[0], pad=lb[1], offset=lb[2]))
    if c is None:
        C = torch.empty((M, N), dtype=dtype, device="cuda")
    else:
        ld, off = c
        C = torch.full((off + M * ld,), float("nan"), dtype=dtype, device="cuda").as_strided((M, N), (ld, 1), off)
    gemm(A, B, C, **kw)
    st = sync_status()
    got = C.double().cpu().numpy()
    out["cases"].append({"name": name, "status": st, "exact": bool(np.array_equal(got, want))})

for single in (False, True):
    s = "single" if single else "pair"
    case(f"1x1x1 {s}", 1, 1, 1, single_cta=single)
    case(f"ragged tiles {s}", 257, 513, 72, single_cta=single)
    case(f"odd K, col-major B {s}", 260, 513, 257, lb=("col", 0, 0), single_cta=single)
    case(f"padded odd strides {s}", 130, 270, 100, la=("row", 3, 0), lb=("row", 5, 0), single_cta=single)
    case(f"unaligned everything {s}", 131, 259, 67, la=("col", 1, 1), lb=("col", 3, 1), c=(263, 3),
         single_cta=single)
    case(f"C view, N % 4 != 0 {s}", 260, 513, 64, c=(520, 0), single_cta=single)
    case(f"fp16 C, odd stride {s}", 257, 301, 130, c=(311, 3), dtype=torch.float16, single_cta=single)
    case(f"bf16 C {s}", 300, 600, 200, dtype=torch.bfloat16, single_cta=single)
    case(f"K = 0 {s}", 100, 300, 0, single_cta=single)
case("non-persistent", 513, 770, 128, persistent=False)
case("row-major order", 600, 700, 256, grouped=False)
case("cross-tile off", 600, 700, 256, cross_tile=False)
case("dynamic units", 2304, 2560, 640, dynamic=True)
case("dynamic units, C view", 700, 513, 128, c=(520, 0), dynamic=True)
case("split tail", 2304, 2560, 1280, tail_split=True)
case("split tail, fp16 C", 700, 1200, 1100, dtype=torch.float16, tail_split=True)

A0 = draw(512, 2048, "int", 90)
B0 = draw(2048, 304, "int", 91)
need, used = splitk_workspace_size(512, 304, 2048, 4)
ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
C = torch.empty((512, 304), device="cuda")
gemm_splitk(dev(A0), dev(B0), C, splits=4, workspace=ws)
st = sync_status()
out["cases"].append({"name": "split-K", "status": st,
                     "exact": bool(np.array_equal(C.double().cpu().numpy(), oracle.gemm(A0, B0)))})

from dense_gemm_gb300 import gemm_packed
for (M, N, K, la, lb) in [(300, 500, 257, ("row", 3, 1), ("col", 5, 3)), (130, 270, 136, ("col", 2, 1), ("row", 6, 5))]:
    A0 = draw(M, K, "int", 92 + M)
    B0 = draw(K, N, "int", 93 + N)
    C = gemm_packed(dev(relayout(A0, la[0], pad=la[1], offset=la[2])), dev(relayout(B0, lb[0], pad=lb[1], offset=lb[2])))
    st = sync_status()
    out["cases"].append({"name": f"packed operands {M}x{N}x{K}", "status": st,
                         "exact": bool(np.array_equal(C.double().cpu().numpy(), oracle.gemm(A0, B0)))})

out["selftest_entry"] = selftest_check()
out["selftest_status"] = sync_status()
out["status_after"] = sync_status()
print(json.dumps(out))
'''


def test_checked_library_finds_no_bad_access_and_reports_a_failed_check():
    subprocess.run([sys.executable, "-m", "dense_gemm_gb300.build", "--debug"], cwd=ROOT, check=True)
    env = dict(os.environ, GEMM_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=1200)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["library"].endswith("libgemm_f16_debug.so")
    bad = [c for c in res["cases"] if c["status"] != 0 or not c["exact"]]
    assert not bad, (bad, r.stderr[-2000:])
    assert len(res["cases"]) == 28
    # the reporting path works: one failing check -> GEMM_ERR_CHECK, cleared by the read
    assert res["selftest_entry"] == 0
    assert res["selftest_status"] == 5
    assert res["status_after"] == 0
    assert "device check failed at source line" in r.stderr
