"""Pins for the oracle's counting formulas against the pages' printed figures
(fixtures under tests/golden/, each with its citation)."""
from decimal import Decimal
from fractions import Fraction as F

import pytest

from oracle import counts as C

GB = 10 ** 9
KB = 1024
MIB = 1024 * 1024


def rounds_to(value, printed: str) -> bool:
    """True when ``value`` rounds to the printed digits (half a unit in the
    last printed place), or to the printed significand for e-notation."""
    d = Decimal(printed)
    exp = d.as_tuple().exponent
    half = Decimal(5) * Decimal(10) ** (exp - 1)
    return abs(Decimal(float(value)) - d) <= half


def test_worked_example(golden):
    g = golden("worked_example_4x4.json")
    M, N, K, BM, BN, BK, e = g["M"], g["N"], g["K"], g["BM"], g["BN"], g["BK"], g["elem_bytes"]
    assert C.reads_no_reuse(M, N, K) == g["reads_elems"]["no_reuse"]
    assert C.reads_tiled(M, N, K, BM, BN) == g["reads_elems"]["tiled_2x2"]
    assert C.reads_once(M, N, K) == g["reads_elems"]["all_onchip"]
    assert C.flops(M, N, K) == g["flops"]
    assert C.per_step_reads(BM, BN, BK) == g["per_step"]["reads_elems"]
    assert C.per_step_flops(BM, BN, BK) == g["per_step"]["flops"]
    assert C.per_step_flops(BM, BN, BK) * (K // BK) == g["per_tile_flops"]
    assert (M // BM) * (N // BN) == g["tiles"]
    assert C.writes(M, N) * e == g["c_write_bytes"]
    nr = C.traffic_bytes(C.reads_no_reuse(M, N, K), C.writes(M, N), e, e)
    tl = C.tile_traffic_bytes(M, N, K, BM, BN, e, e)
    assert nr == g["total_bytes"]["no_reuse"]
    assert tl == g["total_bytes"]["tiled_2x2"]
    assert C.reads_no_reuse(M, N, K) * e == g["read_bytes"]["no_reuse"]
    assert C.reads_tiled(M, N, K, BM, BN) * e == g["read_bytes"]["tiled_2x2"]
    assert C.intensity(C.flops(M, N, K), nr) == F(g["intensity_exact"]["no_reuse"])
    assert C.intensity(C.flops(M, N, K), tl) == F(g["intensity_exact"]["tiled_2x2"])
    assert rounds_to(C.intensity(C.flops(M, N, K), nr), g["intensity_printed"]["no_reuse"])
    # uses per input element = outputs it feeds inside one tile
    total_uses = M * N * 2 * K
    for case in ("no_reuse", "tiled_2x2", "all_onchip"):
        assert total_uses // g["reads_elems"][case] == g["outputs_per_input"][case]


def test_roofline_4096_table(golden):
    g = golden("roofline_4096_fp32.json")
    M, N, K, e = g["M"], g["N"], g["K"], g["elem_bytes"]
    P, BW = g["P_flops_per_s"], g["BW_bytes_per_s"]
    fl = C.flops(M, N, K)
    assert rounds_to(fl, g["flops_printed"])
    assert rounds_to(F(fl, int(P)) * 1000, g["compute_ms_printed"])
    assert rounds_to(F(C.writes(M, N) * e, GB), g["c_write_gb_printed"])
    assert C.ridge_point(P, BW) == int(g["ridge_printed"])
    for row in g["rows"]:
        if row["case"] == "no_reuse":
            b = C.traffic_bytes(C.reads_no_reuse(M, N, K), C.writes(M, N), e, e)
        elif row["case"] == "read_once":
            b = C.traffic_bytes(C.reads_once(M, N, K), C.writes(M, N), e, e)
        else:
            T = row["tile"]
            b = C.tile_traffic_bytes(M, N, K, T, T, e, e)
        I = C.intensity(fl, b)
        bound = C.roofline_bound(P, BW, I)
        t = C.ideal_time(fl, P, BW, b)
        assert rounds_to(b / GB, row["traffic_gb"]), row
        assert rounds_to(I, row["intensity"]), row
        assert rounds_to(bound / 10 ** 12, row["bound_tflops"]), row
        assert rounds_to(t * 1000, row["time_ms"]), row
        assert (bound < P) == (row["bottleneck"] == "memory"), row
        assert t == fl / bound


def test_tile_intensity_approximation():
    # "I ≈ BM·BN / (2(BM + BN))" for 4-byte elements; = T/4 when BM = BN = T,
    # and the exact value (with the C write) stays just below it
    for T in (32, 64, 128):
        assert C.intensity_tile_approx(T, T) == F(T, 4)
        exact = C.intensity(C.flops(4096, 4096, 4096), C.tile_traffic_bytes(4096, 4096, 4096, T, T))
        assert exact < F(T, 4)
    assert C.intensity_tile_approx(128, 64) == F(128 * 64, 2 * 192)


def test_bk_cancels():
    # BK changes neither FLOPs nor reads: per tile (K/BK steps) x per step
    M, N, K, BM, BN = 256, 512, 1024, 128, 64
    for BK in (16, 32, 64, 128):
        per_tile_reads = (K // BK) * C.per_step_reads(BM, BN, BK)
        per_tile_flops = (K // BK) * C.per_step_flops(BM, BN, BK)
        tiles = (M // BM) * (N // BN)
        assert tiles * per_tile_reads == C.reads_tiled(M, N, K, BM, BN)
        assert tiles * per_tile_flops == C.flops(M, N, K)


def test_padded_reads_equal_exact_when_divisible():
    assert C.reads_tiled_padded(512, 1024, 64, 128, 256) == C.reads_tiled(512, 1024, 64, 128, 256)
    assert C.reads_tiled_padded(513, 1024, 64, 128, 256) > C.reads_tiled(513, 1024, 64, 128, 256)


def _enumerate_tile_loads(M, N, K, BM, BN, BK):
    """Walk the tiled loop nest of "4주차 정리: Roofline과 Tiling" section 5 ("일반
    공식") on a ragged grid: every output tile, every K step, one BM x BK piece of
    A and one BK x BN piece of B, a piece cut by an edge still moved whole (the
    zero-filled box of a TMA load). Returns (moved, useful) element counts, the
    useful ones being the in-bounds elements of each piece."""
    moved = useful = 0
    for m0 in range(0, M, BM):
        for n0 in range(0, N, BN):
            for k0 in range(0, K, BK):
                moved += BM * BK + BK * BN
                rows, cols, ks = min(BM, M - m0), min(BN, N - n0), min(BK, K - k0)
                useful += rows * ks + ks * cols
    return moved, useful


@pytest.mark.parametrize("M,N,K,BM,BN,BK", [(300, 520, 192, 128, 256, 64), (257, 513, 64, 128, 256, 64),
                                           (1000, 90, 320, 64, 32, 32), (8, 8, 8, 4, 4, 4), (5, 7, 3, 2, 2, 1)])
def test_padded_reads_match_an_enumeration_of_tile_loads(M, N, K, BM, BN, BK):
    """reads_tiled_padded counts whole tiles on the cdiv grid. The enumeration
    moves whole pieces along K too, so it equals the formula when BK divides K
    (every case here) and exceeds the useful reads exactly on ragged grids."""
    assert K % BK == 0
    moved, useful = _enumerate_tile_loads(M, N, K, BM, BN, BK)
    assert C.reads_tiled_padded(M, N, K, BM, BN) == moved
    nm, nn = C.cdiv(M, BM), C.cdiv(N, BN)
    # useful reads: each tile row re-reads its A rows once per tile column, and vice versa
    assert useful == nn * M * K + nm * K * N
    assert (moved == useful) == (M % BM == 0 and N % BN == 0)


def test_compulsory_bytes_is_the_single_tile_limit_and_a_brute_force_count():
    """Each input element read once and C written once: the page's tile traffic
    HBM bytes = in * MNK(1/BM + 1/BN) + out * MN with one tile covering all of C
    (BM = M, BN = N), and the number of distinct A, B and C elements a direct
    triple loop touches."""
    for M, N, K in [(512, 512, 512), (16384, 16384, 4096), (8191, 8191, 257), (4000, 5000, 3000)]:
        assert C.compulsory_bytes(M, N, K) == C.tile_traffic_bytes(M, N, K, M, N, in_bytes=2, out_bytes=4)
    for M, N, K in [(3, 4, 5), (6, 2, 7), (1, 1, 1)]:
        a, b, c = set(), set(), set()
        for i in range(M):
            for j in range(N):
                for k in range(K):
                    a.add((i, k))
                    b.add((k, j))
                c.add((i, j))
        assert C.compulsory_bytes(M, N, K) == 2 * len(a) + 2 * len(b) + 4 * len(c)
        assert C.compulsory_bytes(M, N, K, in_bytes=4, out_bytes=4) == 4 * (len(a) + len(b) + len(c))


def test_onchip_table(golden):
    g = golden("onchip_memory.json")
    e = g["elem_bytes"]
    for row in g["rows"]:
        T = row["T"]
        assert C.onchip_input_bytes(T, T, T, e) == row["input_kb"] * KB
        assert C.onchip_acc_bytes(T, T, e) == row["acc_kb"] * KB
        assert C.onchip_input_bytes(T, T, T, e) + C.onchip_acc_bytes(T, T, e) == row["total_kb"] * KB
    s = g["small_bk_example"]
    assert C.onchip_input_bytes(s["BM"], s["BN"], s["BK"], e) == s["input_kb"] * KB
    exact = C.intensity(C.flops(4096, 4096, 4096),
                        C.tile_traffic_bytes(4096, 4096, 4096, s["BM"], s["BN"], e, e))
    assert rounds_to(exact, s["intensity_approx_printed"])
    r = g["acc_registers"]
    assert C.onchip_acc_bytes(r["T"], r["T"], e) // 4 == r["regs_32bit"]
    assert r["regs_32bit"] // r["threads"] == r["regs_per_thread"]


def test_cta_swizzle_panels(golden):
    g = golden("cta_swizzle_panels.json")
    e, BM, BN, K, G = g["elem_bytes"], g["BLOCK_M"], g["BLOCK_N"], g["K"], g["GROUP_SIZE_M"]
    for n, want in g["num_n_tiles"].items():
        assert C.cdiv(int(n), BN) == want
        assert C.row_major_tile_id_gap(C.cdiv(int(n), BN)) == want
    assert F(C.a_panel_bytes(BM, K, e), MIB) == F(g["a_panel_mib"])
    assert F(C.b_panel_bytes(K, BN, e), MIB) == F(g["b_panel_mib"])
    for n, want in g["row_major_sweep_mib"].items():
        assert F(C.row_major_sweep_bytes(int(n), K, BM, BN, e), MIB) == F(want)
    assert F(C.grouped_working_set_bytes(G, K, BM, BN, e), MIB) == F(g["grouped_working_set_mib"])
    # the page's capacity argument: the 8192 sweep fits in 96 MiB, the 16384 one does not
    l2 = g["l2_mib_of_measured_gpu"] * MIB
    assert C.row_major_sweep_bytes(8192, K, BM, BN, e) < l2 < C.row_major_sweep_bytes(16384, K, BM, BN, e)


def test_persistent_kernel_counts(golden):
    g = golden("persistent_kernel_counts.json")
    assert C.hmma_m16n8k16_count(g["M"], g["N"], g["K"]) == g["hmma_m16n8k16"]
    s = g["stage_bytes"]
    stage = C.onchip_input_bytes(s["BLOCK_M"], s["BLOCK_N"], s["BLOCK_K"], s["elem_bytes"])
    assert stage == s["bytes"]
    assert g["shared_per_cta_bytes"] == g["stages_resident"] * stage


def test_tflops_definition_matches_printed_measurements(golden):
    g = golden("timings_tflops.json")
    for row in g["rows"]:
        tf = C.tflops(row["M"], row["N"], row["K"], row["ms"])
        # ms printed to 4 decimals: allow its rounding plus the 2-decimal TFLOPS rounding
        slack = tf * 0.5e-4 / row["ms"] + 0.005
        assert abs(tf - row["tflops"]) <= slack, row


@pytest.mark.parametrize("M,N,K", [(512, 512, 512), (16384, 16384, 4096), (8191, 8191, 257)])
def test_compulsory_bytes_fp16_in_fp32_out(M, N, K):
    assert C.compulsory_bytes(M, N, K) == 2 * (M * K + K * N) + 4 * M * N
