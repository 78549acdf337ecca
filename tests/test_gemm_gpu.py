"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Bar: tile map and integer-valued inputs bit-exact; random fp16 inputs within
max|C - C_ref| <= 2e-3 sqrt(K) max|A| max|B| and relative Frobenius error
<= 1e-3, on every element at small sizes and on sampled tiles plus row/column
sum identities at the full workload sizes.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_gb300 import GemmError, gemm, get_config, sync_status, tile_map, kernel_info
from dense_gemm_gb300.inputs import WORKLOADS, draw, relayout
from gpu_util import (assert_within_bound, check_row_col_sums, check_sampled_rows, check_sampled_tiles,
                      require_gpu,
                      run, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    from dense_gemm_gb300 import build
    build.build()
    torch.cuda.init()
    yield
    assert sync_status() == 0


ORDERS = [(True, True), (True, False), (False, True), (False, False)]  # (grouped, cross_tile)
# (grouped, cross_tile, single_cta): CTA-pair 256x256 tiles and one-CTA 128x256 tiles
VARIANTS = [(g, c, False) for (g, c) in ORDERS] + [(True, True, True), (False, False, True)]


# ------------------------------------------------------------------ tile map

@pytest.mark.parametrize("nm,nn,G,grid", [(1, 1, 8, 1), (3, 2, 2, 4), (64, 32, 8, 152),
                                          (128, 64, 8, 152), (65, 63, 8, 152), (37, 13, 5, 7),
                                          (7, 40, 12, 300), (1, 1000, 8, 152), (1000, 1, 8, 152),
                                          (64, 64, 1, 152), (9, 9, 100, 2)])
@pytest.mark.parametrize("grouped", [True, False])
def test_tile_map_bit_exact(nm, nn, G, grid, grouped):
    got = tile_map(nm, nn, G, grouped, grid).cpu().numpy()
    want = oracle.schedule(nm, nn, G, grouped, grid)
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ exact (integer) parity

SMALL_SHAPES = [(1, 1, 1), (128, 256, 64), (129, 257, 65), (300, 600, 200), (64, 100, 1000),
                (256, 512, 128), (7, 1000, 33), (1000, 9, 70), (640, 640, 640)]


@pytest.mark.parametrize("shape", SMALL_SHAPES)
@pytest.mark.parametrize("grouped,cross,single", VARIANTS)
def test_integer_inputs_bit_exact(shape, grouped, cross, single):
    M, N, K = shape
    A = draw(M, K, "int", 7 + M)
    B = draw(K, N, "int", 8 + N)
    _, C = run(A, B, grouped=grouped, cross_tile=cross, G=3, single_cta=single)
    assert np.array_equal(C, oracle.gemm(A, B))


@pytest.mark.parametrize("a_layout,b_layout", [("row", "row"), ("row", "col"), ("col", "row"),
                                               ("col", "col")])
@pytest.mark.parametrize("shape", [(200, 300, 136), (384, 512, 256), (130, 260, 72)])
@pytest.mark.parametrize("single", [False, True])
def test_operand_layouts_bit_exact(a_layout, b_layout, shape, single):
    M, N, K = shape
    A = draw(M, K, "int", 11)
    B = draw(K, N, "int", 12)
    ref = oracle.gemm(A, B)
    _, C = run(relayout(A, a_layout), relayout(B, b_layout), single_cta=single)
    assert np.array_equal(C, ref)


# ------------------------------------------------------------------ random parity, every element

@pytest.mark.parametrize("shape", [(512, 512, 512), (300, 600, 200), (1000, 1000, 1000),
                                   (128, 2048, 4096), (2176, 384, 320)])
@pytest.mark.parametrize("dist", ["uniform", "normal"])
def test_random_inputs_within_bound(shape, dist):
    M, N, K = shape
    A = draw(M, K, dist, 21)
    B = draw(K, N, dist, 22)
    ref = oracle.gemm(A, B)
    for grouped, cross, single in VARIANTS:
        _, C = run(A, B, grouped=grouped, cross_tile=cross, single_cta=single)
        assert_within_bound(C, ref, A, B,
                            f"{shape} {dist} grouped={grouped} cross={cross} single={single}")


def test_orders_give_identical_results():
    # tile order and cross-tile change only which CTA computes a tile and when;
    # each tile's arithmetic is the same, so the outputs are bit-identical
    A = draw(1000, 1200, "normal", 31)
    B = draw(1200, 1500, "normal", 32)
    for single in (False, True):
        outs = [run(A, B, grouped=g, cross_tile=c, G=G, single_cta=single)[1]
                for (g, c) in ORDERS for G in (1, 8)]
        for o in outs[1:]:
            assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("single", [False, True])
@pytest.mark.parametrize("grouped", [False, True])
@pytest.mark.parametrize("shape", [(640, 640, 640), (1000, 1200, 300), (129, 257, 65)])
def test_non_persistent_grid_bit_exact(shape, grouped, single):
    M, N, K = shape
    A = draw(M, K, "int", 33)
    B = draw(K, N, "int", 34)
    _, C = run(A, B, grouped=grouped, single_cta=single, persistent=False, G=3)
    assert np.array_equal(C, oracle.gemm(A, B))
    cfg = get_config(M, N, single_cta=single, persistent=False)
    assert cfg["grid"] == -(-M // cfg["bm"]) * -(-N // cfg["bn"])


# ------------------------------------------------------------------ predicated (non-TMA) paths

@pytest.mark.parametrize("case", [
    # name, M, N, K, A layout/pad/offset, B layout/pad/offset, C (ld, offset)
    ("odd K rows", 300, 300, 257, ("row", 0, 0), ("row", 0, 0), None),
    ("odd K col-major B", 260, 513, 257, ("row", 0, 0), ("col", 0, 0), None),
    ("misaligned A base", 200, 300, 128, ("row", 0, 1), ("row", 0, 0), None),
    ("misaligned B base", 200, 300, 128, ("row", 0, 0), ("col", 0, 3), None),
    ("padded odd strides", 130, 270, 100, ("row", 3, 0), ("row", 5, 0), None),
    ("odd C stride", 257, 300, 64, ("row", 0, 0), ("row", 0, 0), (301, 0)),
    ("misaligned C base", 129, 256, 64, ("row", 0, 0), ("row", 0, 0), (256, 1)),
    ("all predicated", 131, 259, 67, ("col", 1, 1), ("col", 3, 1), (263, 3)),
    ("pair tiles, predicated store", 300, 520, 128, ("row", 0, 0), ("col", 0, 0), (523, 1)),
    # alignment classes with no rows: K < 8 rows of M/N-major operands, M < 8 rows of K-major A
    ("tiny K, M- and N-major odd strides", 70, 90, 3, ("col", 1, 0), ("row", 1, 1), None),
    ("tiny M, odd K", 3, 300, 101, ("row", 0, 0), ("row", 0, 0), None),
    ("N-major B, stride 4 mod 8", 150, 200, 70, ("row", 2, 0), ("row", 4, 0), None),
])
def test_predicated_paths_bit_exact(case):
    name, M, N, K, la, lb, lc = case
    A0 = draw(M, K, "int", 41)
    B0 = draw(K, N, "int", 42)
    ref = oracle.gemm(A0, B0)
    A = relayout(A0, la[0], pad=la[1], offset=la[2])
    B = relayout(B0, lb[0], pad=lb[1], offset=lb[2])
    for grouped, cross, single in VARIANTS:
        Cd, C = run(A, B, grouped=grouped, cross_tile=cross, out_layout=lc, single_cta=single)
        assert np.array_equal(C, ref), f"{name} grouped={grouped} cross={cross} single={single}"
        if lc is not None:
            # nothing outside the logical C was written
            ld, off = lc
            buf = Cd.as_strided((Cd.untyped_storage().nbytes() // 4,), (1,), 0).cpu().numpy()
            mask = np.ones(buf.size, bool)
            for i in range(M):
                mask[off + i * ld: off + i * ld + N] = False
            assert np.isnan(buf[mask]).all(), name


@pytest.mark.parametrize("M,ld,off,N", [(300, 1027, 0, 1027), (300, 1027, 3, 1025), (300, 1026, 1, 1026),
                                        (300, 1025, 2, 1024), (300, 1028, 0, 1027), (300, 1028, 1, 1028),
                                        (70, 8191, 0, 8191), (2600, 2051, 1, 2051), (2600, 2054, 2, 2053)])
@pytest.mark.parametrize("K", [64, 800])
def test_c_row_classes_bit_exact(M, ld, off, N, K):
    """fp32 C whose rows are not all 16-byte aligned goes out per row class
    (rows sharing their offset in a granule, one tensor map each) with the
    values of each row shifted across chunk boundaries: every element exact,
    every element outside C (row padding, before and after) keeps its NaN.
    K = 64 splits a row block's chunks between two epilogue warps, K = 800
    leaves them to one; M is not a multiple of 32. At 2600 rows there are more
    tiles than CTA pairs, so warps go from class-stored tiles to the last tile
    column (plain stores) and back."""
    A = draw(M, K, "int", 470 + ld % 7)
    B = draw(K, N, "int", 471 + N % 5)
    want = oracle.gemm(A, B)
    n = off + M * ld + 37
    buf = torch.full((n,), float("nan"), device="cuda")
    C = buf.as_strided((M, N), (ld, 1), off)
    gemm(to_dev(A), to_dev(B), C)
    torch.cuda.synchronize()
    assert sync_status() == 0
    assert np.array_equal(C.double().cpu().numpy(), want)
    host = buf.cpu().numpy()
    mask = np.ones(n, bool)
    for i in range(M):
        mask[off + i * ld: off + i * ld + N] = False
    assert np.isnan(host[mask]).all(), f"{int((~np.isnan(host[mask])).sum())} values written outside C"


OUT_TYPES = [(torch.float32, "f32"), (torch.float16, "f16"), (torch.bfloat16, "bf16")]


@pytest.mark.parametrize("dtype,name", OUT_TYPES)
@pytest.mark.parametrize("N", [513, 509, 4, 3, 1])
@pytest.mark.parametrize("single", [False, True])
def test_c_views_keep_their_padding_columns(dtype, name, N, single):
    """C a view of a wider buffer (aligned rows, N not a multiple of the 16-byte
    granule): a TMA store clipped inside a granule writes the whole granule, so
    the kernel must end C's map on the last granule boundary and store the rest
    itself. Every column past N keeps its NaN."""
    M, K, ld = 260, 64, 520
    A = draw(M, K, "int", 450 + N)
    B = draw(K, N, "int", 451 + N)
    want = oracle.round_output(oracle.gemm(A, B), name, 1.0)
    buf = torch.full((M * ld,), float("nan"), dtype=dtype, device="cuda")
    C = buf.as_strided((M, N), (ld, 1), 0)
    gemm(to_dev(A), to_dev(B), C, single_cta=single)
    torch.cuda.synchronize()
    assert np.array_equal(C.double().cpu().numpy(), want)
    pad = buf.view(M, ld)[:, N:].float().cpu().numpy()
    assert np.isnan(pad).all(), f"{int((~np.isnan(pad)).sum())} padding values written"


def test_operand_padding_at_the_k_edge_is_not_read():
    """K = 250 inside rows of 256 (TMA loads): the padding holds NaN, and TMA
    zero-fills per element, so the product is exact."""
    M, N, K = 300, 400, 250
    A0 = draw(M, K, "int", 460)
    B0 = draw(K, N, "int", 461)
    ref = oracle.gemm(A0, B0)
    Ab = torch.full((M, 256), float("nan"), dtype=torch.float16)
    Ab[:, :K] = A0
    Bc = torch.full((N, 256), float("nan"), dtype=torch.float16)
    Bc[:, :K] = B0.t()
    for single in (False, True):
        _, C = run(Ab[:, :K], B0, single_cta=single)
        assert np.array_equal(C, ref)
        _, C = run(A0, Bc[:, :K].t(), single_cta=single)
        assert np.array_equal(C, ref)


def test_predicated_random_within_bound():
    A = relayout(draw(600, 257, "uniform", 51), "row")
    B = relayout(draw(257, 700, "uniform", 52), "col")
    ref = oracle.gemm(A, B)
    _, C = run(A, B)
    assert_within_bound(C, ref, A, B, "K=257 predicated")


# ------------------------------------------------------------------ degenerate sizes

def test_k_zero_sets_c_to_zero():
    A = torch.zeros(100, 0, dtype=torch.float16, device="cuda")
    B = torch.zeros(0, 300, dtype=torch.float16, device="cuda")
    C = torch.full((100, 300), 7.0, device="cuda")
    gemm(A, B, C)
    torch.cuda.synchronize()
    assert (C == 0).all()


def test_empty_outputs_are_noops():
    A = torch.ones(0, 64, dtype=torch.float16, device="cuda")
    B = torch.ones(64, 30, dtype=torch.float16, device="cuda")
    assert gemm(A, B).shape == (0, 30)
    B = torch.ones(64, 0, dtype=torch.float16, device="cuda")
    assert gemm(torch.ones(5, 64, dtype=torch.float16, device="cuda"), B).shape == (5, 0)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 4096, 64), (4096, 1, 64), (2, 3, 4),
                                   (127, 255, 63), (128, 256, 64), (129, 257, 65),
                                   (255, 255, 8), (256, 256, 64), (257, 513, 72), (384, 128, 16)])
@pytest.mark.parametrize("single", [False, True])
def test_edge_shapes_bit_exact(M, N, K, single):
    A = draw(M, K, "int", 61)
    B = draw(K, N, "int", 62)
    _, C = run(A, B, single_cta=single)
    assert np.array_equal(C, oracle.gemm(A, B))


def test_overwrites_and_never_reads_c():
    A = draw(256, 128, "int", 71)
    B = draw(128, 512, "int", 72)
    ref = oracle.gemm(A, B)
    for fill in (float("nan"), float("inf"), 1e30):
        Cd = torch.full((256, 512), fill, device="cuda")
        gemm(to_dev(A), to_dev(B), Cd)
        torch.cuda.synchronize()
        assert np.array_equal(Cd.cpu().numpy().astype(np.float64), ref)


def test_group_size_above_m_tiles_is_one_group():
    A = draw(700, 300, "int", 81)
    B = draw(300, 900, "int", 82)
    ref = oracle.gemm(A, B)
    for G in (5, 6, 1000, 2 ** 31 - 1):
        assert np.array_equal(run(A, B, G=G)[1], ref)


def test_invalid_arguments_raise():
    A = torch.ones(8, 8, dtype=torch.float16, device="cuda")
    with pytest.raises(GemmError):
        gemm(A, A, group_size_m=0)
    with pytest.raises(GemmError):
        gemm(A, A, torch.empty(8, 16, device="cuda")[:, ::2])  # stride_cn = 2


def test_kernel_resources():
    # warps: producer (1; predicated loads: 3 for one CTA, 4 + 1 issuer per CTA of a pair) + MMA + 8 epilogue
    threads = {0: 320, 1: 320, 2: 384, 3: 384, 4: 320, 5: 320, 6: 448, 7: 448, 8: 320, 9: 320, 10: 320,
               11: 320, 12: 448}
    for v in range(13):
        info = kernel_info(v)
        assert info["dynamic_smem"] <= 232448 and info["regs_per_thread"] <= 255
        assert info["threads_per_cta"] == threads[v]
        assert info["threads_per_cta"] * info["regs_per_thread"] <= 65536  # one CTA per SM fits
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert get_config(16384, 16384, single_cta=True)["grid"] == sms
    pairs = get_config(16384, 16384)["grid"]
    assert sms // 2 - 8 <= pairs <= sms // 2
    assert get_config(512, 512)["grid"] == 4


def test_repeated_calls_and_streams():
    A = draw(512, 512, "int", 91)
    B = draw(512, 512, "int", 92)
    ref = oracle.gemm(A, B)
    Ad, Bd = to_dev(A), to_dev(B)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(20):
            outs.append(gemm(Ad, Bd))
    s.synchronize()
    for o in outs:
        assert np.array_equal(o.cpu().numpy().astype(np.float64), ref)


def test_calls_captured_in_a_cuda_graph():
    """The entry points only enqueue work (no host synchronisation, no
    allocation), so calls can be captured into a CUDA graph and replayed:
    TMA and predicated paths, fp32 and 16-bit outputs."""
    A = draw(700, 520, "int", 93)
    B = draw(520, 900, "int", 94)
    ref = oracle.gemm(A, B)
    Ad, Bd = to_dev(A), to_dev(B)
    Au = to_dev(relayout(A, "row", pad=3, offset=1))  # predicated loads
    outs = [torch.full((700, 900), float("nan"), device="cuda") for _ in range(2)]
    out16 = torch.full((700, 900), float("nan"), device="cuda", dtype=torch.float16)
    for o, a in zip(outs, (Ad, Au)):  # first calls (library set-up) outside the capture
        gemm(a, Bd, o)
    gemm(Ad, Bd, out16)
    torch.cuda.synchronize()
    for o in outs + [out16]:
        o.fill_(float("nan"))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gemm(Ad, Bd, outs[0])
        gemm(Au, Bd, outs[1])
        gemm(Ad, Bd, out16)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert sync_status() == 0
    for o in outs:
        assert np.array_equal(o.cpu().numpy().astype(np.float64), ref)
    np.testing.assert_array_equal(out16.cpu().numpy().astype(np.float64),
                                  oracle.round_output(ref, "f16"))


@pytest.mark.parametrize("shape", [(256, 256, 64), (512, 512, 512), (1000, 1200, 320),
                                   (2304, 2560, 640), (4096, 4096, 256),
                                   (16384, 16384, 64)])  # ~54 tiles per CTA pair: the unit ring wraps
@pytest.mark.parametrize("grouped,cross", [(True, True), (False, True), (True, False)])
def test_dynamic_units_bit_exact(shape, grouped, cross):
    """GEMM_SCHED_DYNAMIC: every tile computed exactly once whichever cluster
    takes it (fewer tiles than CTA pairs, ragged edges, many tiles per pair)."""
    M, N, K = shape
    A = draw(M, K, "int", 95)
    B = draw(K, N, "int", 96)
    _, C = run(A, B, grouped=grouped, cross_tile=cross, G=3, dynamic=True)
    assert np.array_equal(C, oracle.gemm(A, B))
    assert sync_status() == 0
    cfg = get_config(M, N, dynamic=True)
    assert cfg["grid"] == -(-M // cfg["bm"]) * -(-N // cfg["bn"])


def test_dynamic_units_match_static_bitwise():
    """A tile's arithmetic does not depend on which cluster computes it, so the
    dynamic and the static orders give identical bits on random operands."""
    A = draw(2304, 640, "normal", 99)
    B = draw(640, 2560, "normal", 100)
    _, Cs = run(A, B, G=8)
    _, Cd = run(A, B, G=8, dynamic=True)
    assert np.array_equal(Cs, Cd)
    assert_within_bound(Cd, oracle.gemm(A, B), A, B, "dynamic 2304x2560x640")


def test_dynamic_units_ignored_on_predicated_and_single_cta_paths():
    A = draw(300, 257, "int", 97)
    B = draw(257, 520, "int", 98)
    ref = oracle.gemm(A, B)
    for single in (False, True):
        _, C = run(A, B, single_cta=single, dynamic=True)
        assert np.array_equal(C, ref)


# ------------------------------------------------------------------ full workload sizes

def _full(name, grouped=True, cross=True, exact_dist=False, count=64, single=False, dynamic=False):
    w = WORKLOADS[name]
    A, B = w.operands()
    if exact_dist:
        A = draw(w.M, w.K, "int", w.seed)
        B = draw(w.K, w.N, "int", w.seed + 1)
        if w.b_layout != "row":
            B = relayout(B, w.b_layout)
    _, C = run(A, B, grouped=grouped, cross_tile=cross, single_cta=single, dynamic=dynamic)
    check_sampled_tiles(C, A, B, count=count, seed=w.seed, exact=exact_dist, what=name)
    assert check_sampled_rows(C, A, B, count=4096, seed=w.seed, exact=exact_dist, what=name) >= min(4096, w.M)
    check_row_col_sums(C, A, B, what=name)
    return C


@pytest.mark.parametrize("grouped", [True, False])
def test_full_square_512(grouped):
    w = WORKLOADS["square_512"]
    A, B = w.operands()
    _, C = run(A, B, grouped=grouped)
    assert_within_bound(C, oracle.gemm(A, B), A, B, "512^3")


@pytest.mark.parametrize("grouped", [True, False])
def test_full_8192x8192x4096(grouped):
    _full("square_8192x8192x4096", grouped=grouped)


def test_full_8192x8192x4096_dynamic():
    _full("square_8192x8192x4096", grouped=True, dynamic=True, count=16)


def test_full_16384x16384x4096_headline():
    _full("square_16384x16384x4096", grouped=True, cross=True)


def test_full_16384x16384x4096_row_major_no_cross():
    _full("square_16384x16384x4096", grouped=False, cross=False, count=16)


def test_full_16384x16384x4096_single_cta():
    _full("square_16384x16384x4096", grouped=True, cross=True, count=16, single=True)


@pytest.mark.parametrize("K", [128, 512, 1024, 2048, 4096])
@pytest.mark.parametrize("cross", [True, False])
def test_full_k_sweep(K, cross):
    _full(f"ksweep_16384x16384x{K}", grouped=True, cross=cross, count=32)


def test_full_ragged_4000x5000x3000():
    _full("ragged_4000x5000x3000")


def test_full_ragged_8191x8191x257():
    _full("ragged_8191x8191x257")


def test_full_ragged_8191x8191x257_integer_exact():
    _full("ragged_8191x8191x257", exact_dist=True, count=32)


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_times_out_and_context_survives():
    from dense_gemm_gb300 import selftest_wait_timeout
    assert sync_status() == 0
    selftest_wait_timeout(2_000_000)  # 2 ms: an mbarrier nothing arrives on
    assert sync_status() == 4          # GEMM_ERR_TIMEOUT, read and cleared
    assert sync_status() == 0
    # the next GEMM on the same context is correct
    A = draw(300, 200, "int", 99)
    B = draw(200, 400, "int", 98)
    assert np.array_equal(run(A, B)[1], oracle.gemm(A, B))


# stages per pair: 16 (one tile each); 20 for the pairs with two tiles, 10 for the others
# (those finish normally while the rest abort in their second tile); 4
@pytest.mark.parametrize("M,N,K,stop_after", [(512, 512, 1024, 3), (2304, 2560, 640, 15), (300, 520, 256, 2)])
def test_pair_kernel_abort_returns_and_context_survives(M, N, K, stop_after):
    """Both CTAs of every pair stop issuing copies after `stop_after` stages:
    the MMA warp's wait runs out, the launch records GEMM_ERR_TIMEOUT and every
    CTA (the second of each pair included) returns; the next GEMM is exact."""
    from dense_gemm_gb300 import selftest_pair_abort, set_wait_timeout
    assert sync_status() == 0
    A = to_dev(draw(M, K, "int", 700))
    B = to_dev(draw(K, N, "int", 701))
    C = torch.empty(M, N, device="cuda")
    set_wait_timeout(5_000_000)  # 5 ms
    try:
        selftest_pair_abort(A, B, C, stop_after)
        assert sync_status() == 4  # GEMM_ERR_TIMEOUT, read and cleared
        assert sync_status() == 0
    finally:
        set_wait_timeout(2_000_000_000)
    Ah = draw(700, 300, "int", 702)
    Bh = draw(300, 900, "int", 703)
    assert np.array_equal(run(Ah, Bh)[1], oracle.gemm(Ah, Bh))
    assert sync_status() == 0


# ------------------------------------------------------------------ host-operand APIs

def test_gemm_from_host_matches_oracle():
    from dense_gemm_gb300 import gemm_from_host
    A = draw(300, 200, "int", 111).pin_memory()
    B = draw(200, 500, "int", 112).pin_memory()
    C = gemm_from_host(A, B)
    torch.cuda.synchronize()
    assert np.array_equal(C.numpy().astype(np.float64), oracle.gemm(A, B))


def test_host_pipeline_overlapped_calls_match_oracle():
    from dense_gemm_gb300 import HostPipeline
    inputs = [(draw(384, 256, "int", 120 + i).pin_memory(), draw(256, 640, "int", 140 + i).pin_memory())
              for i in range(5)]
    outs = [torch.empty((384, 640), dtype=torch.float32, pin_memory=True) for _ in inputs]
    pipe = HostPipeline(inputs[0][0], inputs[0][1], depth=2)
    for (A, B), C in zip(inputs, outs):
        pipe.submit(A, B, C)
    pipe.synchronize()
    for (A, B), C in zip(inputs, outs):
        assert np.array_equal(C.numpy().astype(np.float64), oracle.gemm(A, B))


# ------------------------------------------------------------------ split-K (scratch workspace)

@pytest.mark.parametrize("shape", [(512, 512, 512), (300, 304, 320), (256, 256, 64), (129, 704, 1000),
                                   (1024, 512, 4096)])
@pytest.mark.parametrize("splits", [0, 1, 2, 3, 7])
def test_splitk_integer_bit_exact(shape, splits):
    from dense_gemm_gb300 import gemm_splitk
    M, N, K = shape
    A = draw(M, K, "int", 200 + M)
    B = draw(K, N, "int", 201 + N)
    C = gemm_splitk(to_dev(A), to_dev(B), splits=splits)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy().astype(np.float64), oracle.gemm(A, B))


@pytest.mark.parametrize("grouped,cross", ORDERS)
def test_splitk_random_within_bound_and_strided_c(grouped, cross):
    from dense_gemm_gb300 import gemm_splitk
    M, N, K = 384, 520, 2000
    A = draw(M, K, "normal", 210)
    B = relayout(draw(K, N, "normal", 211), "col")
    ref = oracle.gemm(A, B)
    buf = torch.full((M * 531 + 1,), float("nan"), device="cuda")
    C = buf.as_strided((M, N), (531, 1), 1)  # odd stride, misaligned base
    gemm_splitk(to_dev(A), to_dev(B), C, splits=5, grouped=grouped, cross_tile=cross)
    torch.cuda.synchronize()
    assert_within_bound(C.cpu().numpy().astype(np.float64), ref, A, B, "split-K")


def test_splitk_matches_unsplit_on_integers_full_512():
    from dense_gemm_gb300 import gemm_splitk, splitk_workspace_size
    w = WORKLOADS["square_512"]
    A, B = w.operands()
    ref = oracle.gemm(A, B)
    need, used = splitk_workspace_size(512, 512, 512, 0)
    assert used > 1 and need == used * 512 * 512 * 4
    C = gemm_splitk(to_dev(A), to_dev(B))
    torch.cuda.synchronize()
    assert_within_bound(C.cpu().numpy().astype(np.float64), ref, A, B, "512^3 split-K")


def test_splitk_rejects_small_workspace_and_unaligned_operands():
    from dense_gemm_gb300 import gemm_splitk
    A = torch.ones(512, 512, dtype=torch.float16, device="cuda")
    with pytest.raises(GemmError) as e:
        gemm_splitk(A, A, splits=4, workspace=torch.empty(1024, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 1
    A2 = to_dev(relayout(draw(300, 257, "int", 5), "row"))  # 514-byte rows: no TMA
    B2 = to_dev(draw(257, 300, "int", 6))
    with pytest.raises(GemmError) as e:
        gemm_splitk(A2, B2, splits=2)
    assert e.value.status == 2


# ------------------------------------------------------------------ split tail (GEMM_SCHED_TAIL_SPLIT)

def _tail_plan(M, N, K):
    """(first, tiles, slices) the library plans for the split tail, restated from
    the header's rule with the current device's pair count."""
    cfg = get_config(M, N)
    T = -(-M // cfg["bm"]) * -(-N // cfg["bn"])
    P = get_config(16384, 16384)["grid"]
    nkb = -(-K // cfg["bk"])
    rest = T % P
    if rest == 0 or 4 * rest > P:
        return None
    S = min(P // rest, 96 // rest, nkb // 8)
    if S < 2:
        return None
    kps = -(-nkb // S)
    S = -(-nkb // kps)
    return (T - rest, rest, S) if S >= 2 else None


@pytest.mark.parametrize("shape", [(512, 512, 1024), (700, 1200, 1100), (2304, 2560, 1280), (4000, 5000, 1200),
                                   (300, 304, 4096), (2176, 384, 1000)])
@pytest.mark.parametrize("grouped,cross", [(True, True), (False, True), (True, False)])
def test_tail_split_integer_bit_exact(shape, grouped, cross):
    """The split tail's slices of a tile are summed in a fixed order; with
    integer inputs every partial sum is exact, so C equals the oracle."""
    M, N, K = shape
    assert _tail_plan(M, N, K) is not None  # these shapes do split their tail
    A = draw(M, K, "int", 600 + M)
    B = draw(K, N, "int", 601 + N)
    ref = oracle.gemm(A, B)
    for _ in range(2):  # the second call reuses the scratch
        _, C = run(A, B, grouped=grouped, cross_tile=cross, G=3, tail_split=True)
        assert np.array_equal(C, ref)


@pytest.mark.parametrize("dtype,name", OUT_TYPES)
@pytest.mark.parametrize("alpha", [1.0, 0.5, -2.0])
def test_tail_split_out_dtype_alpha_bit_exact(dtype, name, alpha):
    M, N, K = 2304, 2560, 1280
    A = draw(M, K, "int", 610)
    B = relayout(draw(K, N, "int", 611), "col")
    want = oracle.round_output(oracle.gemm(A, B), name, alpha)
    C = gemm(to_dev(A), to_dev(B), out_dtype=dtype, alpha=alpha, tail_split=True)
    torch.cuda.synchronize()
    assert np.array_equal(C.double().cpu().numpy(), want)


def test_tail_split_random_within_bound_and_unsplit_tiles_identical():
    """Random operands: within the stated bound; the tiles outside the tail are
    computed exactly as without the flag (same bits), the tail tiles differ at
    most by the bound."""
    M, N, K = 2304, 2560, 4096
    A = draw(M, K, "normal", 620)
    B = draw(K, N, "normal", 621)
    ref = oracle.gemm(A, B)
    _, C0 = run(A, B)
    _, C1 = run(A, B, tail_split=True)
    assert_within_bound(C1, ref, A, B, "tail split")
    first, tiles, S = _tail_plan(M, N, K)
    cfg = get_config(M, N)
    nm, nn = -(-M // cfg["bm"]), -(-N // cfg["bn"])
    sched = oracle.schedule(nm, nn, 8, True, 1)
    tail = np.zeros((M, N), bool)
    for t in range(first, first + tiles):
        tm, tn = int(sched[t, 1]), int(sched[t, 2])
        tail[tm * cfg["bm"]:(tm + 1) * cfg["bm"], tn * cfg["bn"]:(tn + 1) * cfg["bn"]] = True
    assert np.array_equal(C1[~tail], C0[~tail])


def test_tail_split_without_effect_where_it_does_not_apply():
    """No partial last round, predicated operands, a predicated C store, one-CTA
    tiles: the flag changes nothing (bit-identical)."""
    P = get_config(16384, 16384)["grid"]
    cases = [((256, 256 * (P - 1), 256), {}),  # P - 1 tiles: the last round is nearly full
             ((512, 512, 512), {}),  # 8 k-blocks: too short to split
             ((300, 300, 257), {}), ((512, 509, 1024), {}), ((1000, 1200, 1100), {"single_cta": True})]
    for (M, N, K), kw in cases:
        A = draw(M, K, "normal", 630 + M)
        B = draw(K, N, "normal", 631 + N)
        _, C0 = run(A, B, **kw)
        _, C1 = run(A, B, tail_split=True, **kw)
        assert np.array_equal(C0, C1), (M, N, K, kw)


def test_full_ragged_4000x5000x3000_tail_split():
    w = WORKLOADS["ragged_4000x5000x3000"]
    A, B = w.operands()
    _, C = run(A, B, tail_split=True)
    check_sampled_tiles(C, A, B, count=64, seed=w.seed, what="4000x5000x3000 tail split")
    check_sampled_rows(C, A, B, count=4000, seed=w.seed, what="4000x5000x3000 tail split")
    check_row_col_sums(C, A, B, what="4000x5000x3000 tail split")


# ------------------------------------------------------------------ 16-bit C and alpha



@pytest.mark.parametrize("dtype,name", OUT_TYPES)
@pytest.mark.parametrize("alpha", [1.0, 0.5, -2.0])
@pytest.mark.parametrize("shape,single", [((300, 600, 200), False), ((512, 512, 4096), False),
                                          ((129, 257, 65), True), ((640, 384, 1000), False)])
def test_out_dtype_alpha_integer_bit_exact(dtype, name, alpha, shape, single):
    # integer inputs: the fp32 accumulator and alpha * acc are exact (alpha a power
    # of two), so both sides round the same value to the output type
    M, N, K = shape
    A = draw(M, K, "int", 400 + M)
    B = draw(K, N, "int", 401 + N)
    want = oracle.round_output(oracle.gemm(A, B), name, alpha)
    C = gemm(to_dev(A), to_dev(B), out_dtype=dtype, alpha=alpha, single_cta=single)
    torch.cuda.synchronize()
    assert C.dtype == dtype
    assert np.array_equal(C.double().cpu().numpy(), want)


@pytest.mark.parametrize("dtype,name,ulp", [(torch.float16, "f16", 2.0 ** -10),
                                            (torch.bfloat16, "bf16", 2.0 ** -7)])
def test_out_dtype_random_within_bound(dtype, name, ulp):
    M, N, K = 1000, 1200, 1500
    A = draw(M, K, "normal", 420)
    B = relayout(draw(K, N, "normal", 421), "col")
    exact = oracle.gemm(A, B)
    alpha = 0.75
    C = gemm(to_dev(A), to_dev(B), out_dtype=dtype, alpha=alpha)
    torch.cuda.synchronize()
    got = C.double().cpu().numpy()
    ref = alpha * exact
    # stated bound (scaled by |alpha|) plus one unit in the last place of the output type
    from gpu_util import error_bound
    tol = abs(alpha) * error_bound(A, B) + ulp * np.abs(ref)
    assert np.all(np.abs(got - ref) <= tol)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-3 + ulp


@pytest.mark.parametrize("dtype,name", OUT_TYPES[1:])
def test_out_dtype_predicated_store_and_k0(dtype, name):
    M, N, K = 257, 301, 130
    A = draw(M, K, "int", 430)
    B = draw(K, N, "int", 431)
    want = oracle.round_output(oracle.gemm(A, B), name, 1.0)
    buf = torch.full((M * 311 + 3,), float("nan"), dtype=dtype, device="cuda")
    C = buf.as_strided((M, N), (311, 1), 3)  # odd stride, misaligned base: predicated stores
    gemm(to_dev(A), to_dev(B), C)
    torch.cuda.synchronize()
    assert np.array_equal(C.double().cpu().numpy(), want)
    Z = torch.full((M, N), 3.0, dtype=dtype, device="cuda")
    gemm(torch.zeros(M, 0, dtype=torch.float16, device="cuda"),
         torch.zeros(0, N, dtype=torch.float16, device="cuda"), Z)
    torch.cuda.synchronize()
    assert (Z == 0).all()


def test_out_dtype_split_k_applies_alpha_once():
    from dense_gemm_gb300 import gemm_splitk
    A = draw(512, 2048, "int", 440)
    B = draw(2048, 512, "int", 441)
    exact = oracle.gemm(A, B)
    C = gemm_splitk(to_dev(A), to_dev(B), splits=4)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy().astype(np.float64), exact)
