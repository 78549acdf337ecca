"""Pins for the oracle's GEMM and tile maps (CPU only).

Each test checks the oracle against something other than itself: the fp16
format as numpy decodes it, closed forms (identity, permutation, rank-1),
brute force in exact Python integers, numpy's float64 matmul, the 4x4 worked
example of "4주차 정리: Roofline과 Tiling" (section 5, "작은 예"), and the
statements of "(2/n) Triton matmul 커널 탐험 - grouped ordering(CTA swizzle)"
(sections "구현" and "타일 배정 순서 비교") about the tile orders.
"""
import itertools
import random

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_gb300.inputs import draw, relayout


def f64(x):
    return x.float().double().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float64)


# ---------------------------------------------------------------- fp16 decode

def test_fp16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    ours = np.array([oracle.fp16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_fp16_decode_landmarks():
    assert oracle.fp16_to_f64(0x3C00) == 1.0
    assert oracle.fp16_to_f64(0xC000) == -2.0
    assert oracle.fp16_to_f64(0x7BFF) == 65504.0
    assert oracle.fp16_to_f64(0x0400) == 2.0 ** -14   # smallest normal
    assert oracle.fp16_to_f64(0x0001) == 2.0 ** -24   # smallest subnormal
    assert oracle.fp16_to_f64(0x3555) == 1365 / 4096  # 0.333251953125
    assert oracle.fp16_to_f64(0x8000) == 0.0 and np.signbit(oracle.fp16_to_f64(0x8000))
    assert np.isinf(oracle.fp16_to_f64(0x7C00))


# ---------------------------------------------------------------- closed forms

def test_identity_left_and_right():
    B = draw(37, 45, "uniform", 11)
    I = torch.eye(37, dtype=torch.float16)
    assert np.array_equal(oracle.gemm(I, B), f64(B))
    A = draw(29, 37, "normal", 12)
    assert np.array_equal(oracle.gemm(A, I), f64(A))


def test_permutation_left_and_right():
    rng = np.random.default_rng(5)
    n = 23
    perm = rng.permutation(n)
    P = torch.zeros(n, n, dtype=torch.float16)
    P[np.arange(n), perm] = 1          # (P @ B)[i, :] = B[perm[i], :]
    B = draw(n, 31, "uniform", 13)
    assert np.array_equal(oracle.gemm(P, B), f64(B)[perm, :])
    Q = torch.zeros(n, n, dtype=torch.float16)
    Q[perm, np.arange(n)] = 1          # (A @ Q)[:, j] = A[:, perm[j]]
    A = draw(19, n, "uniform", 14)
    assert np.array_equal(oracle.gemm(A, Q), f64(A)[:, perm])


def test_rank_one_closed_form():
    # A[i, k] = u_i, B[k, j] = v_j  =>  C[i, j] = K * u_i * v_j (exact here)
    rng = np.random.default_rng(6)
    M, N, K = 13, 17, 100
    u = rng.integers(-16, 17, M) / 8.0
    v = rng.integers(-16, 17, N) / 8.0
    A = torch.tensor(np.repeat(u[:, None], K, axis=1), dtype=torch.float16)
    B = torch.tensor(np.repeat(v[None, :], K, axis=0), dtype=torch.float16)
    assert np.array_equal(oracle.gemm(A, B), K * np.outer(u, v))


def test_k_zero_gives_zero():
    A = torch.zeros(5, 0, dtype=torch.float16)
    B = torch.zeros(0, 7, dtype=torch.float16)
    assert np.array_equal(oracle.gemm(A, B), np.zeros((5, 7)))


# ---------------------------------------------------------------- brute force

def _py_matmul(A, B):
    a = [[int(v) for v in row] for row in A.float().tolist()]
    b = [[int(v) for v in row] for row in B.float().tolist()]
    M, K, N = len(a), len(b), len(b[0]) if b else 0
    return [[sum(a[i][k] * b[k][j] for k in range(K)) for j in range(N)] for i in range(M)]


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 1, 4), (5, 7, 9), (8, 3, 2), (16, 24, 40)])
@pytest.mark.parametrize("layouts", [("row", "row"), ("col", "row"), ("row", "col"), ("col", "col")])
def test_integer_bruteforce(shape, layouts):
    M, N, K = shape
    A = draw(M, K, "int", 100 + M)
    B = draw(K, N, "int", 200 + N)
    ref = np.array(_py_matmul(A, B), dtype=np.float64).reshape(M, N)
    A2 = relayout(A, layouts[0], pad=3, offset=1)
    B2 = relayout(B, layouts[1], pad=5, offset=3)
    assert np.array_equal(oracle.gemm(A2, B2), ref)


def test_random_matches_numpy_float64():
    for (M, N, K, seed) in [(17, 33, 65, 1), (64, 64, 64, 2), (3, 130, 257, 3)]:
        A = draw(M, K, "uniform", seed)
        B = draw(K, N, "normal", seed + 50)
        ref = f64(A) @ f64(B)
        got = oracle.gemm(A, B)
        # both are double sums of exactly representable products; only the
        # summation order can differ
        bound = K * np.abs(f64(A)).max() * np.abs(f64(B)).max() * K * 2.0 ** -52
        assert np.abs(got - ref).max() <= bound


# ------------------------------------------------- the pages' 4x4 worked example

def test_worked_example_4x4_tiled_accumulation(golden):
    """C tiles of 2x2 built from K/BK = 2 steps of (2x2)@(2x2) products equal the
    direct definition ("4주차 정리", section 5, 작은 예)."""
    g = golden("worked_example_4x4.json")
    M, N, K, BM, BN, BK = g["M"], g["N"], g["K"], g["BM"], g["BN"], g["BK"]
    A = draw(M, K, "int", 44)
    B = draw(K, N, "int", 45)
    Af, Bf = f64(A), f64(B)
    full = oracle.gemm(A, B)
    steps = 0
    for tm in range(M // BM):
        for tn in range(N // BN):
            acc = np.zeros((BM, BN))
            for s in range(K // BK):
                acc += Af[tm * BM:(tm + 1) * BM, s * BK:(s + 1) * BK] @ \
                       Bf[s * BK:(s + 1) * BK, tn * BN:(tn + 1) * BN]
                steps += 1
            assert np.array_equal(acc, full[tm * BM:(tm + 1) * BM, tn * BN:(tn + 1) * BN])
    assert steps == g["tiles"] * g["steps_per_tile"]


# ---------------------------------------------------------------- API shape

def test_layouts_give_identical_results():
    A = draw(33, 70, "uniform", 7)
    B = draw(70, 41, "uniform", 8)
    ref = oracle.gemm(A, B)
    for la, lb in itertools.product(["row", "col"], repeat=2):
        got = oracle.gemm(relayout(A, la, pad=2, offset=1), relayout(B, lb, pad=1))
        assert np.array_equal(got, ref)


def test_row_subset_and_column_window():
    A = draw(50, 40, "uniform", 9)
    B = draw(40, 60, "uniform", 10)
    full = oracle.gemm(A, B)
    rows = [49, 0, 17, 17, 3]
    got = oracle.gemm_rows(A, B, rows=rows, col0=13, ncols=29)
    assert np.array_equal(got, full[rows][:, 13:42])


def test_thread_count_does_not_change_result():
    A = draw(40, 300, "normal", 21)
    B = draw(300, 50, "normal", 22)
    assert np.array_equal(oracle.gemm(A, B, threads=1), oracle.gemm(A, B, threads=4))


def test_rejects_bad_arguments():
    A = draw(4, 5, "uniform", 1)
    B = draw(6, 4, "uniform", 2)
    with pytest.raises(ValueError):
        oracle.gemm(A, B)
    B = draw(5, 4, "uniform", 2)
    with pytest.raises(ValueError):
        oracle.gemm_rows(A, B, rows=[4])
    with pytest.raises(ValueError):
        oracle.gemm_rows(A, B, col0=2, ncols=3)


# ================================================================ tile maps

def _check_bijection(sched, nm, nn):
    cover = np.zeros((nm, nn), dtype=np.int64)
    np.add.at(cover, (sched[:, 1], sched[:, 2]), 1)
    return bool((cover == 1).all())


def test_grouped_map_is_bijection_exhaustive():
    for nm in range(1, 41):
        for nn in range(1, 41, 3):
            for G in range(1, 13):
                s = oracle.schedule(nm, nn, G, True, 7)
                assert _check_bijection(s, nm, nn), (nm, nn, G)


@pytest.mark.parametrize("nm,nn,G", [(512, 64, 8), (128, 64, 8), (64, 32, 8), (128, 128, 8),
                                     (65, 63, 8), (64, 64, 8), (32, 32, 8), (4, 2, 8),
                                     (63, 33, 5), (1, 1000, 8), (1000, 1, 8)])
def test_grouped_map_is_bijection_large(nm, nn, G):
    assert _check_bijection(oracle.schedule(nm, nn, G, True, 152), nm, nn)
    assert _check_bijection(oracle.schedule(nm, nn, G, False, 152), nm, nn)


def test_row_major_formula():
    nm, nn = 7, 11
    for t in range(nm * nn):
        assert oracle.tile_coord(t, nm, nn, 8, False) == (t // nn, t % nn)


def test_g1_is_row_major():
    for nm, nn in [(1, 1), (5, 9), (16, 3), (33, 40)]:
        a = oracle.schedule(nm, nn, 1, True, 11)
        b = oracle.schedule(nm, nn, 1, False, 11)
        assert np.array_equal(a, b)


def test_g_at_least_nm_is_column_major():
    # one group holds every m-tile: m moves first over the whole grid
    for nm, nn, G in [(3, 5, 3), (3, 5, 8), (8, 8, 8), (1, 7, 8)]:
        for t in range(nm * nn):
            assert oracle.tile_coord(t, nm, nn, G, True) == (t % nm, t // nm)


def test_grouped_hand_case_short_last_group():
    # nm = 3, nn = 2, G = 2: groups {m0, m1} then a short group {m2}
    want = [(0, 0), (1, 0), (0, 1), (1, 1), (2, 0), (2, 1)]
    got = [oracle.tile_coord(t, 3, 2, 2, True) for t in range(6)]
    assert got == want


def test_grouped_neighbours_share_b_panel():
    """Inside a group, C(m, n) and C(m+1, n) get consecutive tile ids
    ("타일 배정 순서 비교"); each group walks the B panels one at a time."""
    nm, nn, G = 37, 13, 8
    for t in range(nm * nn - 1):
        m0, n0 = oracle.tile_coord(t, nm, nn, G, True)
        m1, n1 = oracle.tile_coord(t + 1, nm, nn, G, True)
        first = (m0 // G) * G
        gs = min(G, nm - first)
        if m0 - first < gs - 1:
            assert (m1, n1) == (m0 + 1, n0)
        elif n0 < nn - 1:
            assert (m1, n1) == (first, n0 + 1)
        else:
            assert (m1, n1) == (first + gs, 0)


def test_row_major_gap_is_num_n_tiles():
    nm, nn = 9, 128
    for m in range(nm - 1):
        for n in (0, 5, nn - 1):
            t0 = m * nn + n
            assert oracle.tile_coord(t0, nm, nn, 8, False) == (m, n)
            assert oracle.tile_coord(t0 + nn, nm, nn, 8, False) == (m + 1, n)


def test_persistent_schedule_order():
    nm, nn, G, grid = 13, 9, 4, 10
    s = oracle.schedule(nm, nn, G, True, grid)
    T = nm * nn
    assert np.array_equal(s[:, 0], np.arange(T) % grid)
    for t in range(T):
        assert tuple(s[t, 1:]) == oracle.tile_coord(t, nm, nn, G, True)


def test_tile_map_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.tile_coord(0, 4, 4, 0, True)
    with pytest.raises(ValueError):
        oracle.tile_coord(16, 4, 4, 2, True)
    with pytest.raises(ValueError):
        oracle.schedule(4, 4, 0, True, 3)
    assert oracle.tile_coord(3, 4, 4, 0, False) == (0, 3)


# ------------------------------------------- the pins catch planted mistakes

def _mapping_variant(t, nm, nn, G, bug):
    nig = G * nn
    g, r = t // nig, t % nig
    fm = g * G
    gs = G if bug == "no_short_group" else min(G, nm - fm)
    if bug == "swapped_div_mod":
        return fm + r // gs, r % gs
    return fm + r % gs, r // gs


@pytest.mark.parametrize("bug", ["no_short_group", "swapped_div_mod"])
def test_planted_mapping_mistakes_fail_the_pins(bug):
    caught = False
    for nm, nn, G in [(3, 2, 2), (37, 13, 8), (10, 4, 3)]:
        coords = [_mapping_variant(t, nm, nn, G, bug) for t in range(nm * nn)]
        ok = sorted(coords) == [(m, n) for m in range(nm) for n in range(nn)]
        consecutive = all(coords[t + 1] == (coords[t][0] + 1, coords[t][1])
                          for t in range(G - 1))
        caught |= (not ok) or (not consecutive)
    assert caught
    # and the oracle itself passes the same checks
    for nm, nn, G in [(3, 2, 2), (37, 13, 8), (10, 4, 3)]:
        assert _check_bijection(oracle.schedule(nm, nn, G, True, 5), nm, nn)


def test_random_shapes_schedule_consistency():
    rng = random.Random(3)
    for _ in range(200):
        nm, nn, G, grid = rng.randint(1, 60), rng.randint(1, 60), rng.randint(1, 16), rng.randint(1, 200)
        s = oracle.schedule(nm, nn, G, True, grid)
        assert _check_bijection(s, nm, nn)


# ------------------------------------------------ 16-bit output rounding (C as fp16 / bf16)

def _special_values():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -24, 2.0 ** -25,
            3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11,
            3.0e38, 3.4e38, 2.0 ** -126, 2.0 ** -133, 2.0 ** -134, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]
    return vals + [-v for v in vals]


def test_bf16_decode_exhaustive_vs_torch():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double().numpy()
    ours = np.array([oracle.bf16_to_f64(int(b) & 0xFFFF) for b in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000),
                         np.array(_special_values())])
    # exact ties: midpoints between neighbouring binary16 values
    b = rng.integers(0, 0x7BFF, 3000).astype(np.uint16)
    lo = b.view(np.float16).astype(np.float64)
    hi = (b + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    xs = np.concatenate([xs, (lo + hi) / 2, -(lo + hi) / 2])
    with np.errstate(over="ignore"):  # values past the fp16 range round to infinity, as intended
        ref = xs.astype(np.float16).view(np.uint16)
    ours = np.array([oracle.f64_to_f16_bits(x) for x in xs], dtype=np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_rounding_is_nearest_ties_to_even_brute_force(fmt):
    enc = oracle.f64_to_f16_bits if fmt == "f16" else oracle.f64_to_bf16_bits
    dec = oracle.fp16_to_f64 if fmt == "f16" else oracle.bf16_to_f64
    top = 0x7BFF if fmt == "f16" else 0x7F7F  # largest finite
    rng = np.random.default_rng(8)
    xs = list(rng.standard_normal(3000) * 10.0 ** rng.uniform(-45 if fmt == "bf16" else -9,
                                                              38 if fmt == "bf16" else 4.8, 3000))
    xs += [v for v in _special_values() if np.isfinite(v)]
    for x in xs:
        r = enc(x)
        mag = r & 0x7FFF
        if mag > top:  # infinity: only beyond the last finite value's half-ulp
            assert abs(x) > dec(top)
            continue
        got = abs(dec(r))
        for nb in (mag - 1, mag + 1):
            if 0 <= nb <= top:
                d_nb, d_r = abs(abs(x) - dec(nb)), abs(abs(x) - got)
                assert d_r <= d_nb, (fmt, x, hex(r), hex(nb))
                if d_r == d_nb:  # a tie goes to the even fraction
                    assert mag % 2 == 0, (fmt, x, hex(r))
        if x != 0:
            assert (r >> 15) == (1 if x < 0 else 0)


def test_rounding_landmarks():
    f = oracle.f64_to_f16_bits
    assert f(65504.0) == 0x7BFF and f(65519.99) == 0x7BFF and f(65520.0) == 0x7C00
    assert f(2.0 ** -24) == 0x0001 and f(2.0 ** -25) == 0x0000 and f(3 * 2.0 ** -26) == 0x0001
    assert f(1 + 2.0 ** -11) == 0x3C00 and f(1 + 3 * 2.0 ** -11) == 0x3C02
    assert f(-0.0) == 0x8000 and (f(float("nan")) & 0x7C00) == 0x7C00
    g = oracle.f64_to_bf16_bits
    assert g(1.0) == 0x3F80 and g(1 + 2.0 ** -8) == 0x3F80 and g(1 + 3 * 2.0 ** -8) == 0x3F82
    assert g(2.0 ** -133) == 0x0001 and g(2.0 ** -134) == 0x0000
    assert g(3.4e38) == 0x7F80  # past the midpoint between 0x7F7F (3.3895e38) and 2^128
    assert g(3.0e38) == 0x7F62  # 3.0e38 = 1.7633 * 2^127 -> fraction 0x62
    assert g(-2.0) == 0xC000


def test_round_output_alpha_and_formats():
    C = np.array([[1.0, -3.0], [65519.0, 1e-8]])
    assert np.array_equal(oracle.round_output(C, "f32", 0.5), np.float32(C * 0.5).astype(np.float64))
    r16 = oracle.round_output(C, "f16", 2.0)
    assert r16[0, 0] == 2.0 and r16[0, 1] == -6.0 and np.isinf(r16[1, 0]) and r16[1, 1] == 0.0
    rb = oracle.round_output(C, "bf16", 1.0)
    assert rb[0, 0] == 1.0 and rb[1, 0] == 65536.0
