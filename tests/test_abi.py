"""The C-ABI library builds, loads and exports every symbol the header declares;
argument validation runs on the host without touching a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gemm_f16.h")


@pytest.fixture(scope="module")
def lib():
    from dense_gemm_gb300 import build as b
    b.build()
    from dense_gemm_gb300 import binding
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_f16\w*)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert "gemm_f16" in names and "gemm_f16_tile_map" in names
    assert len(names) == 16, names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    from dense_gemm_gb300 import status_str
    assert status_str(0) == "GEMM_OK"
    assert status_str(1) == "GEMM_ERR_INVALID_ARG"
    assert status_str(2) == "GEMM_ERR_UNSUPPORTED"
    assert status_str(3) == "GEMM_ERR_CUDA"
    assert status_str(4) == "GEMM_ERR_TIMEOUT"
    assert status_str(5) == "GEMM_ERR_CHECK"


def _call(lib, **kw):
    a = dict(A=16, B=16, C=16, M=4, N=4, K=4, sam=4, sak=1, sbk=4, sbn=1, scm=4, scn=1, G=8,
             flags=3, stream=0)
    a.update(kw)
    return lib.gemm_f16(a["A"], a["B"], a["C"], a["M"], a["N"], a["K"], a["sam"], a["sak"],
                        a["sbk"], a["sbn"], a["scm"], a["scn"], a["G"], a["flags"], a["stream"])


@pytest.mark.parametrize("kw", [dict(M=-1), dict(N=-5), dict(K=-1), dict(M=2 ** 31),
                                dict(sam=0), dict(sak=-1), dict(sbk=0), dict(sbn=0), dict(scm=0),
                                dict(scn=0), dict(G=0), dict(G=-3), dict(flags=64),
                                dict(flags=0x80000000), dict(C=0), dict(A=0), dict(B=0),
                                dict(scm=3)])
def test_invalid_arguments(lib, kw):
    assert _call(lib, **kw) == 1


@pytest.mark.parametrize("kw", [dict(sak=2, sam=3), dict(sbn=2, sbk=3), dict(scn=2, scm=8)])
def test_unsupported_layouts(lib, kw):
    assert _call(lib, **kw) == 2


def test_group_size_ignored_without_grouping(lib):
    # G < 1 is only an error when the grouped order is asked for; M == 0 is a no-op
    assert _call(lib, G=0, flags=2, M=0) == 0


def test_empty_problems_are_noops(lib):
    assert _call(lib, M=0) == 0
    assert _call(lib, N=0) == 0
    assert _call(lib, M=0, A=0, B=0, C=0) == 0


def test_tile_map_validation(lib):
    assert lib.gemm_f16_tile_map(0, 4, 8, 1, 4, 16, 0) == 1
    assert lib.gemm_f16_tile_map(4, 0, 8, 1, 4, 16, 0) == 1
    assert lib.gemm_f16_tile_map(4, 4, 8, 1, 0, 16, 0) == 1
    assert lib.gemm_f16_tile_map(4, 4, 0, 1, 4, 16, 0) == 1
    assert lib.gemm_f16_tile_map(4, 4, 8, 1, 4, 0, 0) == 1
    assert lib.gemm_f16_tile_map(65536, 65536, 8, 1, 4, 16, 0) == 1


def test_config_without_device(lib):
    from dense_gemm_gb300 import get_config
    cfg = get_config(0, 0)
    assert (cfg["bm"], cfg["bn"], cfg["bk"]) == (256, 256, 64)
    assert cfg["stages"] >= 2 and cfg["grid"] == 0
    cfg = get_config(0, 0, single_cta=True)
    assert (cfg["bm"], cfg["bn"], cfg["bk"]) == (128, 256, 64)
    assert lib.gemm_f16_get_config(-1, 4, 0, None, None, None, None, None) == 1
    assert lib.gemm_f16_get_config(4, 4, 64, None, None, None, None, None) == 1


def test_wait_timeout_validation(lib):
    assert lib.gemm_f16_set_wait_timeout(999) == 1
    assert lib.gemm_f16_set_wait_timeout(2_000_000_000) == 0
    assert lib.gemm_f16_selftest_wait_timeout(999, 0) == 1
    assert lib.gemm_f16_selftest_wait_timeout(10 ** 11, 0) == 1


def test_product_library_has_no_device_checks(lib):
    assert lib.gemm_f16_selftest_check(None) == 2  # GEMM_ERR_UNSUPPORTED


def test_kernel_info_rejects_unknown_variant(lib):
    i32 = ctypes.POINTER(ctypes.c_int32)
    assert lib.gemm_f16_kernel_info(13, i32(), i32(), i32(), i32()) == 1
    assert lib.gemm_f16_kernel_info(-1, i32(), i32(), i32(), i32()) == 1


def test_binding_raises_when_library_missing(monkeypatch, tmp_path):
    from dense_gemm_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "nope.so"))
    with pytest.raises(binding.GemmError):
        binding.load_library()


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "dense_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle_gemm" not in text, f


def test_splitk_host_validation(lib):
    import ctypes as C
    b, sp = C.c_uint64(), C.c_int32()
    assert lib.gemm_f16_splitk_workspace_size(512, 512, 512, 4, C.byref(b), C.byref(sp)) == 0
    assert sp.value == 4 and b.value == 4 * 512 * 512 * 4
    # never an empty slice: 5 k-blocks asked for 4 slices -> 2 per slice -> 3 slices
    assert lib.gemm_f16_splitk_workspace_size(300, 301, 320, 4, C.byref(b), C.byref(sp)) == 0
    assert sp.value == 3 and b.value == 3 * 300 * 304 * 4
    assert lib.gemm_f16_splitk_workspace_size(512, 512, 64, 8, C.byref(b), C.byref(sp)) == 0
    assert sp.value == 1 and b.value == 0
    assert lib.gemm_f16_splitk_workspace_size(-1, 512, 64, 8, None, None) == 1
    assert lib.gemm_f16_splitk_workspace_size(4, 512, 64, -1, None, None) == 1
    a = dict(A=16, B=16, C=16, M=4, N=4, K=4, sam=4, sak=1, sbk=4, sbn=1, scm=4, scn=1)
    args = [a[k] for k in ("A", "B", "C", "M", "N", "K", "sam", "sak", "sbk", "sbn", "scm", "scn")]
    assert lib.gemm_f16_splitk(*args, -1, None, 0, 8, 3, None) == 1
    assert lib.gemm_f16_splitk(*args[:3], 0, *args[4:], 4, None, 0, 8, 3, None) == 0  # M == 0


def test_out_dtype_validation(lib):
    import ctypes as C
    args = (16, 16, 16)
    # unknown element type -> INVALID_ARG before any GPU work
    assert lib.gemm_f16_out(*args, 3, C.c_float(1.0), 4, 4, 4, 4, 1, 4, 1, 4, 1, 8, 3, None) == 1
    assert lib.gemm_f16_out(*args, -1, C.c_float(1.0), 4, 4, 4, 4, 1, 4, 1, 4, 1, 8, 3, None) == 1
    assert lib.gemm_f16_out(*args, 1, C.c_float(2.0), 0, 4, 4, 4, 1, 4, 1, 4, 1, 8, 3, None) == 0


def test_binding_rejects_operands_on_different_devices():
    """The C entry points act on the current device (status words, scratch,
    stream); the binding therefore requires A, B and out on one device and makes
    the call with that device current."""
    import torch
    from dense_gemm_gb300.binding import _common_device
    a = torch.empty(2, 2, dtype=torch.float16)
    assert _common_device(a, a, torch.empty(2, 2)) == torch.device("cpu")
    with pytest.raises(ValueError, match="one CUDA device"):
        _common_device(a, torch.empty(2, 2, dtype=torch.float16, device="meta"), a)


def test_packed_host_validation(lib):
    """gemm_f16_packed checks its workspace before any GPU work; the size query
    needs no device."""
    import ctypes as C
    b = C.c_uint64()
    # A K-major 300 x 257 (rows of 320 once copied), B K-major 500 x 257
    assert lib.gemm_f16_packed_workspace_size(300, 500, 257, 257, 1, 1, 257, C.byref(b)) == 0
    a_bytes = (300 * 320 * 2 + 255) // 256 * 256
    assert b.value == a_bytes + 500 * 320 * 2
    # A M-major (rows are K = 64 rows of M = 100 -> 128), B N-major (64 rows of 70 -> 128)
    assert lib.gemm_f16_packed_workspace_size(100, 70, 64, 1, 100, 70, 1, C.byref(b)) == 0
    assert b.value == (64 * 128 * 2 + 255) // 256 * 256 + 64 * 128 * 2
    assert lib.gemm_f16_packed_workspace_size(0, 70, 64, 1, 100, 70, 1, C.byref(b)) == 0 and b.value == 0
    assert lib.gemm_f16_packed_workspace_size(-1, 70, 64, 1, 100, 70, 1, None) == 1
    assert lib.gemm_f16_packed_workspace_size(4, 70, 64, 0, 100, 70, 1, None) == 1
    args = (16, 16, 16, 4, 4, 4, 4, 1, 4, 1, 4, 1, 8, 3)
    need = (4 * 64 * 2 + 255) // 256 * 256 + 4 * 64 * 2
    assert lib.gemm_f16_packed(*args, None, need, None) == 1        # no workspace
    assert lib.gemm_f16_packed(*args, 256 + 16, need, None) == 1    # not 128-byte aligned
    assert lib.gemm_f16_packed(*args, 256, need - 1, None) == 1     # too small
    assert lib.gemm_f16_packed(16, 16, 16, 0, 4, 4, 4, 1, 4, 1, 4, 1, 8, 3, None, 0, None) == 0  # M == 0


def test_element_alignment_validation(lib):
    # fp16 operands at odd addresses, fp32 C not 4-byte aligned -> INVALID_ARG before any GPU work
    assert _call(lib, A=17) == 1
    assert _call(lib, B=33) == 1
    assert _call(lib, C=18) == 1
