"""ctypes binding of ``include/gemm_f16.h`` (argument marshalling only).

Every function here forwards to the C-ABI library ``libgemm_f16.so``; the
arithmetic runs in its CUDA kernels. Torch is used for device memory and the
current stream. If the library has not been built, every call raises
``GemmError`` — there is no fallback path. ``GEMM_LIBRARY=debug`` selects
``libgemm_f16_debug.so`` (device-side bounds checks, ``GEMM_ERR_CHECK``).
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libgemm_f16.so"

SCHED_GROUPED = 0x1
SCHED_CROSS_TILE = 0x2
SCHED_SINGLE_CTA = 0x4
SCHED_NON_PERSISTENT = 0x8
SCHED_DYNAMIC = 0x10
SCHED_TAIL_SPLIT = 0x20

_STATUS = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_UNSUPPORTED",
           3: "GEMM_ERR_CUDA", 4: "GEMM_ERR_TIMEOUT", 5: "GEMM_ERR_CHECK"}


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        name = _STATUS.get(self.status, f"status {status}")
        super().__init__(f"{what}: {name}" if what else name)


_lib = None


def library_path() -> str:
    if os.environ.get("GEMM_LIBRARY", "") == "debug":
        return os.path.join(_HERE, "libgemm_f16_debug.so")
    return os.path.join(_HERE, _LIB_NAME)


def load_library():
    """Load (once) and return the ctypes handle of libgemm_f16.so."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise GemmError(3, f"{path} is missing: build it with "
                           "`python -m dense_gemm_gb300.build` (`--debug` for the checked "
                           "library; no fallback path exists)")
    lib = ctypes.CDLL(path)
    i64, i32, u32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_void_p
    pi32 = ctypes.POINTER(ctypes.c_int32)
    lib.gemm_f16.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                             i32, u32, vp]
    lib.gemm_f16.restype = ctypes.c_int
    u64 = ctypes.c_uint64
    lib.gemm_f16_splitk.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                                    i32, vp, u64, i32, u32, vp]
    lib.gemm_f16_splitk.restype = ctypes.c_int
    lib.gemm_f16_splitk_workspace_size.argtypes = [i64, i64, i64, i32, ctypes.POINTER(u64),
                                                   ctypes.POINTER(i32)]
    lib.gemm_f16_splitk_workspace_size.restype = ctypes.c_int
    lib.gemm_f16_splitk_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64,
                                            i64, i32, i32, u32, vp]
    lib.gemm_f16_splitk_noalloc.restype = ctypes.c_int
    lib.gemm_f16_packed.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                                    i32, u32, vp, u64, vp]
    lib.gemm_f16_packed.restype = ctypes.c_int
    lib.gemm_f16_packed_workspace_size.argtypes = [i64, i64, i64, i64, i64, i64, i64,
                                                   ctypes.POINTER(u64)]
    lib.gemm_f16_packed_workspace_size.restype = ctypes.c_int
    lib.gemm_f16_out.argtypes = [vp, vp, vp, i32, ctypes.c_float, i64, i64, i64, i64, i64, i64,
                                 i64, i64, i64, i32, u32, vp]
    lib.gemm_f16_out.restype = ctypes.c_int
    lib.gemm_f16_tile_map.argtypes = [i32, i32, i32, u32, i32, vp, vp]
    lib.gemm_f16_tile_map.restype = ctypes.c_int
    lib.gemm_f16_get_config.argtypes = [i64, i64, u32, pi32, pi32, pi32, pi32, pi32]
    lib.gemm_f16_get_config.restype = ctypes.c_int
    lib.gemm_f16_kernel_info.argtypes = [i32, pi32, pi32, pi32, pi32]
    lib.gemm_f16_kernel_info.restype = ctypes.c_int
    lib.gemm_f16_sync_status.argtypes = [vp]
    lib.gemm_f16_sync_status.restype = ctypes.c_int
    lib.gemm_f16_set_wait_timeout.argtypes = [ctypes.c_uint64]
    lib.gemm_f16_set_wait_timeout.restype = ctypes.c_int
    lib.gemm_f16_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.gemm_f16_selftest_wait_timeout.restype = ctypes.c_int
    lib.gemm_f16_selftest_pair_abort.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
    lib.gemm_f16_selftest_pair_abort.restype = ctypes.c_int
    lib.gemm_f16_selftest_check.argtypes = [vp]
    lib.gemm_f16_selftest_check.restype = ctypes.c_int
    lib.gemm_f16_status_str.argtypes = [ctypes.c_int]
    lib.gemm_f16_status_str.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        raise GemmError(status, what)


def _stream_handle(stream=None, device=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return int(stream.cuda_stream)


def _common_device(*tensors) -> torch.device:
    """The one CUDA device all `tensors` live on. The C entry points work on the
    current device (its status words, its scratch and its stream), so every
    call is made with this device current."""
    devs = {t.device for t in tensors}
    if len(devs) != 1:
        raise ValueError(f"A, B and out must be on one CUDA device, got {sorted(map(str, devs))}")
    return devs.pop()


def status_str(status: int) -> str:
    return load_library().gemm_f16_status_str(int(status)).decode()


def gemm_raw(A_ptr: int, B_ptr: int, C_ptr: int, M: int, N: int, K: int,
             stride_am: int, stride_ak: int, stride_bk: int, stride_bn: int,
             stride_cm: int, stride_cn: int, group_size_m: int = 8,
             schedule_flags: int = SCHED_GROUPED | SCHED_CROSS_TILE, stream: int = 0) -> int:
    """The C call with raw integers; returns the status code (no raise)."""
    return load_library().gemm_f16(A_ptr, B_ptr, C_ptr, M, N, K, stride_am, stride_ak,
                                   stride_bk, stride_bn, stride_cm, stride_cn,
                                   group_size_m, schedule_flags, stream)


def sched_flags(grouped: bool = True, cross_tile: bool = True, single_cta: bool = False,
                persistent: bool = True, dynamic: bool = False, tail_split: bool = False) -> int:
    return ((SCHED_GROUPED if grouped else 0) | (SCHED_CROSS_TILE if cross_tile else 0)
            | (SCHED_SINGLE_CTA if single_cta else 0) | (0 if persistent else SCHED_NON_PERSISTENT)
            | (SCHED_DYNAMIC if dynamic else 0) | (SCHED_TAIL_SPLIT if tail_split else 0))


_OUT_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}


def gemm(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor = None, *,
         group_size_m: int = 8, grouped: bool = True, cross_tile: bool = True,
         single_cta: bool = False, persistent: bool = True, dynamic: bool = False,
         tail_split: bool = False, alpha: float = 1.0,
         out_dtype: torch.dtype = torch.float32, stream=None) -> torch.Tensor:
    """C = alpha * (A @ B) with A [M,K], B [K,N] fp16 CUDA tensors.

    The keywords map to the GEMM_SCHED_* flags (``tail_split`` to
    GEMM_SCHED_TAIL_SPLIT).

    ``out`` ([M,N], unit column stride, float32 / float16 / bfloat16) is
    written if given, else allocated with ``out_dtype``. fp32 output with
    alpha == 1 goes through gemm_f16, everything else through gemm_f16_out.
    Strided views are passed through as strides.
    """
    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("A and B must be float16")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shapes {tuple(A.shape)} @ {tuple(B.shape)} do not chain")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    if out.dtype not in _OUT_CODES or tuple(out.shape) != (M, N) or not out.is_cuda:
        raise ValueError("out must be a float32/float16/bfloat16 CUDA tensor of shape [M, N]")
    dev = _common_device(A, B, out)
    flags = sched_flags(grouped, cross_tile, single_cta, persistent, dynamic, tail_split)
    sam, sak = A.stride()
    sbk, sbn = B.stride()
    scm, scn = out.stride()
    # torch gives stride 1 to size-1 dims' neighbours freely; keep them >= 1
    strides = (max(sam, 1), max(sak, 1), max(sbk, 1), max(sbn, 1), max(scm, 1), max(scn, 1))
    with torch.cuda.device(dev):
        if out.dtype == torch.float32 and alpha == 1.0:
            st = gemm_raw(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, *strides,
                          group_size_m, flags, _stream_handle(stream, dev))
            _check(st, "gemm_f16")
        else:
            st = load_library().gemm_f16_out(A.data_ptr(), B.data_ptr(), out.data_ptr(),
                                             _OUT_CODES[out.dtype], float(alpha), M, N, K, *strides,
                                             group_size_m, flags, _stream_handle(stream, dev))
            _check(st, "gemm_f16_out")
    return out


def packed_workspace_size(M: int, N: int, K: int, stride_am: int, stride_ak: int,
                          stride_bk: int, stride_bn: int) -> int:
    """Workspace bytes of gemm_f16_packed for these sizes and operand strides."""
    b = ctypes.c_uint64()
    _check(load_library().gemm_f16_packed_workspace_size(M, N, K, stride_am, stride_ak, stride_bk,
                                                         stride_bn, ctypes.byref(b)),
           "gemm_f16_packed_workspace_size")
    return int(b.value)


def gemm_packed(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor = None, *,
                workspace: torch.Tensor = None, group_size_m: int = 8, grouped: bool = True,
                cross_tile: bool = True, tail_split: bool = False, stream=None) -> torch.Tensor:
    """C = A @ B through gemm_f16_packed: operands whose rows do not start on
    128-byte boundaries are first copied into ``workspace`` (a CUDA tensor of at
    least packed_workspace_size() bytes, allocated when omitted)."""
    out = _check_operands(A, B, out)
    M, K = A.shape
    N = B.shape[1]
    dev = A.device
    sam, sak = (max(x, 1) for x in A.stride())
    sbk, sbn = (max(x, 1) for x in B.stride())
    scm, scn = (max(x, 1) for x in out.stride())
    with torch.cuda.device(dev):
        need = packed_workspace_size(M, N, K, sam, sak, sbk, sbn)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        _common_device(A, workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
        st = load_library().gemm_f16_packed(
            A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, sam, sak, sbk, sbn, scm, scn,
            group_size_m, sched_flags(grouped, cross_tile, tail_split=tail_split), workspace.data_ptr(),
            ws_bytes, _stream_handle(stream, dev))
    _check(st, "gemm_f16_packed")
    return out


def _check_operands(A, B, out):
    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("A and B must be float16")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shapes {tuple(A.shape)} @ {tuple(B.shape)} do not chain")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    M, N = A.shape[0], B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if out.dtype != torch.float32 or tuple(out.shape) != (M, N) or not out.is_cuda:
        raise ValueError("out must be a float32 CUDA tensor of shape [M, N]")
    _common_device(A, B, out)
    return out


def splitk_workspace_size(M: int, N: int, K: int, splits: int = 0):
    """(bytes, splits used) of gemm_f16_splitk for these sizes."""
    b, sp = ctypes.c_uint64(), ctypes.c_int32()
    _check(load_library().gemm_f16_splitk_workspace_size(M, N, K, splits, ctypes.byref(b),
                                                         ctypes.byref(sp)),
           "gemm_f16_splitk_workspace_size")
    return int(b.value), int(sp.value)


def gemm_splitk(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor = None, *, splits: int = 0,
                workspace: torch.Tensor = None, group_size_m: int = 8, grouped: bool = True,
                cross_tile: bool = True, stream=None) -> torch.Tensor:
    """C = A @ B with K split across CTA pairs (gemm_f16_splitk). ``workspace``
    (a CUDA tensor of at least splitk_workspace_size() bytes) is allocated
    when omitted."""
    out = _check_operands(A, B, out)
    M, K = A.shape
    N = B.shape[1]
    dev = A.device
    with torch.cuda.device(dev):
        need, _ = splitk_workspace_size(M, N, K, splits)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        _common_device(A, workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
        sam, sak = A.stride()
        sbk, sbn = B.stride()
        scm, scn = out.stride()
        st = load_library().gemm_f16_splitk(
            A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, max(sam, 1), max(sak, 1), max(sbk, 1),
            max(sbn, 1), max(scm, 1), max(scn, 1), splits, workspace.data_ptr(), ws_bytes, group_size_m,
            sched_flags(grouped, cross_tile), _stream_handle(stream, dev))
    _check(st, "gemm_f16_splitk")
    return out


def gemm_splitk_noalloc(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor, *, splits: int = 0,
                        group_size_m: int = 8, grouped: bool = True, cross_tile: bool = True,
                        stream=None) -> torch.Tensor:
    """gemm_f16_splitk_noalloc: split-K through the library's built-in 32 MiB
    scratch, for callers that cannot allocate device memory at this point
    (``out`` must be given; nothing is allocated)."""
    out = _check_operands(A, B, out)
    M, K = A.shape
    N = B.shape[1]
    sam, sak = A.stride()
    sbk, sbn = B.stride()
    scm, scn = out.stride()
    dev = A.device
    with torch.cuda.device(dev):  # the entry point uses the current device's scratch
        st = load_library().gemm_f16_splitk_noalloc(
            A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, max(sam, 1), max(sak, 1),
            max(sbk, 1), max(sbn, 1), max(scm, 1), max(scn, 1), splits, group_size_m,
            sched_flags(grouped, cross_tile), _stream_handle(stream, dev))
    _check(st, "gemm_f16_splitk_noalloc")
    return out


def tile_map(num_m_tiles: int, num_n_tiles: int, group_size_m: int, grouped: bool,
             grid: int, device=None, stream=None) -> torch.Tensor:
    """[T, 3] int32 CUDA tensor from the kernel's scheduler: row tile_id =
    (program id, tile_m, tile_n)."""
    device = device or torch.device("cuda")
    out = torch.full((num_m_tiles * num_n_tiles, 3), -1, dtype=torch.int32, device=device)
    with torch.cuda.device(out.device):
        st = load_library().gemm_f16_tile_map(num_m_tiles, num_n_tiles, group_size_m,
                                              SCHED_GROUPED if grouped else 0, grid,
                                              out.data_ptr(), _stream_handle(stream, out.device))
    _check(st, "gemm_f16_tile_map")
    return out


def get_config(M: int = 0, N: int = 0, single_cta: bool = False, persistent: bool = True,
               dynamic: bool = False) -> dict:
    v = [ctypes.c_int32() for _ in range(5)]
    flags = sched_flags(single_cta=single_cta, persistent=persistent, dynamic=dynamic)
    _check(load_library().gemm_f16_get_config(M, N, flags, *[ctypes.byref(x) for x in v]),
           "gemm_f16_get_config")
    return dict(zip(("bm", "bn", "bk", "stages", "grid"), (x.value for x in v)))


def kernel_info(variant: int = 0) -> dict:
    v = [ctypes.c_int32() for _ in range(4)]
    _check(load_library().gemm_f16_kernel_info(variant, *[ctypes.byref(x) for x in v]),
           "gemm_f16_kernel_info")
    return dict(zip(("regs_per_thread", "static_smem", "dynamic_smem", "threads_per_cta"),
                    (x.value for x in v)))


def sync_status(stream=None) -> int:
    """Synchronize and return (and clear) the device status code."""
    return int(load_library().gemm_f16_sync_status(_stream_handle(stream)))


def selftest_check(stream=None) -> int:
    """Debug library only: one device-side check that fails (no access behind
    it); returns the entry point's status (GEMM_ERR_UNSUPPORTED = 2 in the
    product library)."""
    return int(load_library().gemm_f16_selftest_check(_stream_handle(stream)))


def selftest_wait_timeout(timeout_ns: int = 1_000_000, stream=None):
    """Enqueue the bounded-wait self-test kernel (see the header)."""
    _check(load_library().gemm_f16_selftest_wait_timeout(int(timeout_ns), _stream_handle(stream)),
           "gemm_f16_selftest_wait_timeout")


def selftest_pair_abort(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, stop_after: int, stream=None):
    """Enqueue the CTA-pair abort self-test (see the header): row-major fp16 A,
    B and fp32 C on one device; the kernel's wait runs out and it returns."""
    dev = _common_device(A, B, C)
    M, K = A.shape
    N = B.shape[1]
    if not (A.is_contiguous() and B.is_contiguous() and C.is_contiguous()):
        raise ValueError("the abort self-test takes contiguous row-major A, B and C")
    with torch.cuda.device(dev):
        _check(load_library().gemm_f16_selftest_pair_abort(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                                           int(stop_after), _stream_handle(stream, dev)),
               "gemm_f16_selftest_pair_abort")


def set_wait_timeout(ns: int):
    _check(load_library().gemm_f16_set_wait_timeout(int(ns)), "gemm_f16_set_wait_timeout")


def gemm_from_host(A_host: torch.Tensor, B_host: torch.Tensor, C_host: torch.Tensor = None, *,
                   workspace=None, group_size_m: int = 8, grouped: bool = True,
                   cross_tile: bool = True, single_cta: bool = False, stream=None) -> torch.Tensor:
    """End-to-end call on HOST operands: copy A and B (pinned host fp16) to the
    device, run gemm_f16, copy C back into ``C_host`` (pinned fp32).

    ``workspace`` = (A_dev, B_dev, C_dev) device buffers of matching shapes to
    reuse across calls; allocated when omitted. Copies and the kernel are
    enqueued on one stream; the call returns after the device-to-host copy has
    been enqueued (synchronize the stream before reading ``C_host``).
    """
    M, K = A_host.shape
    N = B_host.shape[1]
    if C_host is None:
        C_host = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    if workspace is None:
        workspace = (torch.empty_like(A_host, device="cuda"), torch.empty_like(B_host, device="cuda"),
                     torch.empty((M, N), dtype=torch.float32, device="cuda"))
    A_dev, B_dev, C_dev = workspace
    s = stream if stream is not None else torch.cuda.current_stream()
    with torch.cuda.stream(s):
        A_dev.copy_(A_host, non_blocking=True)
        B_dev.copy_(B_host, non_blocking=True)
        gemm(A_dev, B_dev, C_dev, group_size_m=group_size_m, grouped=grouped,
             cross_tile=cross_tile, single_cta=single_cta, stream=s)
        C_host.copy_(C_dev, non_blocking=True)
    return C_host


class HostPipeline:
    """Back-to-back GEMMs on host operands with the copies of consecutive calls
    overlapped.

    Each ``submit(A_host, B_host, C_host)`` copies A and B (pinned host fp16) to
    one of ``depth`` device buffer sets, runs gemm_f16 there, and copies C back
    into ``C_host`` (pinned fp32). Uploads and the GEMM run on one stream,
    downloads on another, so the download of call i overlaps the upload and
    GEMM of call i+1 (the host link carries both directions at once). A buffer
    set is reused only after its previous download has finished. Call
    ``synchronize()`` before reading the last ``C_host``.
    """

    def __init__(self, A_like: torch.Tensor, B_like: torch.Tensor, depth: int = 2, *,
                 group_size_m: int = 8, grouped: bool = True, cross_tile: bool = True,
                 single_cta: bool = False, device=None):
        device = torch.device(device or "cuda")
        M, N = A_like.shape[0], B_like.shape[1]
        self.kw = dict(group_size_m=group_size_m, grouped=grouped, cross_tile=cross_tile,
                       single_cta=single_cta)
        self.sets = [(torch.empty_strided(A_like.shape, A_like.stride(), dtype=A_like.dtype, device=device),
                      torch.empty_strided(B_like.shape, B_like.stride(), dtype=B_like.dtype, device=device),
                      torch.empty((M, N), dtype=torch.float32, device=device)) for _ in range(depth)]
        self.s_in = torch.cuda.Stream(device=device)
        self.s_out = torch.cuda.Stream(device=device)
        self.gemm_done = [torch.cuda.Event() for _ in range(depth)]
        self.out_done = [torch.cuda.Event() for _ in range(depth)]
        self.used = [False] * depth
        self.calls = 0

    def submit(self, A_host: torch.Tensor, B_host: torch.Tensor, C_host: torch.Tensor):
        j = self.calls % len(self.sets)
        A_dev, B_dev, C_dev = self.sets[j]
        with torch.cuda.stream(self.s_in):
            if self.used[j]:
                self.s_in.wait_event(self.out_done[j])  # C_dev[j] has been downloaded
            A_dev.copy_(A_host, non_blocking=True)
            B_dev.copy_(B_host, non_blocking=True)
            gemm(A_dev, B_dev, C_dev, stream=self.s_in, **self.kw)
            self.gemm_done[j].record(self.s_in)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.gemm_done[j])
            C_host.copy_(C_dev, non_blocking=True)
            self.out_done[j].record(self.s_out)
        self.used[j] = True
        self.calls += 1
        return C_host

    def synchronize(self):
        self.s_in.synchronize()
        self.s_out.synchronize()
