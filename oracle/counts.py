"""FLOP, HBM-traffic, intensity and panel-size counts of the tiled GEMM.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``); also read by
``bench.py`` for the algorithmic FLOPs and bytes of the roofline.

Exact rational arithmetic (``fractions.Fraction``) so the pins can compare
with the pages' printed figures at any precision.

Sources:
  * "4주차 정리: Roofline과 Tiling", section 1 (arithmetic intensity
    I = FLOPs / HBM bytes; a GEMM does 2MNK FLOPs), section 2 (roofline bound
    min(P, BW * I), ridge point P / BW), section 5 "작은 예" (the 4x4 example
    with 2x2 tiles, BK = 2), section 5 "일반 공식" (per-tile and whole-problem
    FLOPs / reads / writes table; reads = MNK(1/BM + 1/BN) elements,
    writes = MN), section 5 "4096 × 4096 FP32 행렬곱" (the hypothetical
    roofline table) and "필요한 온칩 메모리" (on-chip bytes per tile).
  * "(2/n) Triton matmul 커널 탐험 - grouped ordering(CTA swizzle)...",
    sections "타일 배정 순서 비교" and "재사용 거리와 캐시 용량" (A / B panel
    sizes, the row-major B sweep and the grouped working set).
  * "(1/n) ... persistent kernel", section "나머지 3.1%" (the HMMA count table;
    one m16n8k16 HMMA does 2*16*8*16 FLOPs).
"""
from fractions import Fraction as F


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def flops(M: int, N: int, K: int) -> int:
    """2MNK: one multiply and one add per (i, j, k)."""
    return 2 * M * N * K


# ---- reads / writes in ELEMENTS ------------------------------------------

def reads_no_reuse(M: int, N: int, K: int) -> int:
    """Every output element reads its whole A row and B column: MN * 2K."""
    return M * N * 2 * K


def reads_tiled(M: int, N: int, K: int, BM: int, BN: int) -> F:
    """MNK(1/BM + 1/BN): the tile table's whole-problem read row.

    Assumes BM | M and BN | N, as the page does; BK cancels.
    """
    return F(M * N * K) * (F(1, BM) + F(1, BN))


def reads_tiled_padded(M: int, N: int, K: int, BM: int, BN: int) -> int:
    """Ragged-shape version: cdiv(M,BM)*cdiv(N,BN) tiles, each reading
    K*(BM + BN) elements (edge tiles counted as full tiles)."""
    return cdiv(M, BM) * cdiv(N, BN) * K * (BM + BN)


def reads_once(M: int, N: int, K: int) -> int:
    """Each input element read exactly once: MK + KN."""
    return M * K + K * N


def writes(M: int, N: int) -> int:
    """C written once, never read: MN elements."""
    return M * N


def per_step_reads(BM: int, BN: int, BK: int) -> int:
    """One K step of one tile: A piece BM*BK plus B piece BK*BN."""
    return BM * BK + BK * BN


def per_step_flops(BM: int, BN: int, BK: int) -> int:
    return 2 * BM * BN * BK


# ---- bytes and intensity --------------------------------------------------

def traffic_bytes(read_elems, write_elems, in_bytes: int, out_bytes: int) -> F:
    return F(read_elems) * in_bytes + F(write_elems) * out_bytes


def tile_traffic_bytes(M, N, K, BM, BN, in_bytes=4, out_bytes=4) -> F:
    """in_bytes * MNK(1/BM + 1/BN) + out_bytes * MN (the page uses 4 B for all)."""
    return traffic_bytes(reads_tiled(M, N, K, BM, BN), writes(M, N), in_bytes, out_bytes)


def compulsory_bytes(M, N, K, in_bytes=2, out_bytes=4) -> int:
    """Each input element read once and C written once."""
    return in_bytes * reads_once(M, N, K) + out_bytes * writes(M, N)


def intensity(flop_count, byte_count) -> F:
    return F(flop_count) / F(byte_count)


def intensity_tile_approx(BM: int, BN: int, elem_bytes: int = 4) -> F:
    """BM*BN / (2(BM+BN)) for 4-byte elements, C write ignored.

    Generalised to other element sizes as 2*BM*BN / (elem_bytes*(BM+BN)).
    """
    return F(2 * BM * BN, elem_bytes * (BM + BN))


def roofline_bound(P, BW, I):
    """Attainable FLOP/s = min(P, BW * I)."""
    return min(F(P), F(BW) * F(I))


def ridge_point(P, BW) -> F:
    return F(P) / F(BW)


def ideal_time(flop_count, P, BW, byte_count) -> F:
    """FLOPs / bound = max(compute time, memory time)."""
    return max(F(flop_count) / F(P), F(byte_count) / F(BW))


# ---- on-chip memory per tile (section "필요한 온칩 메모리") ---------------

def onchip_input_bytes(BM: int, BN: int, BK: int, elem_bytes: int = 4) -> int:
    return (BM * BK + BK * BN) * elem_bytes


def onchip_acc_bytes(BM: int, BN: int, elem_bytes: int = 4) -> int:
    return BM * BN * elem_bytes


# ---- panels and reuse (CTA-swizzle page) ----------------------------------

def a_panel_bytes(BM: int, K: int, elem_bytes: int = 2) -> int:
    return BM * K * elem_bytes


def b_panel_bytes(K: int, BN: int, elem_bytes: int = 2) -> int:
    return K * BN * elem_bytes


def row_major_sweep_bytes(N: int, K: int, BM: int, BN: int, elem_bytes: int = 2) -> int:
    """One output-tile row under row-major order walks every B panel once
    while reusing one A panel: num_n_tiles * B panel + A panel."""
    return cdiv(N, BN) * b_panel_bytes(K, BN, elem_bytes) + a_panel_bytes(BM, K, elem_bytes)


def grouped_working_set_bytes(G: int, K: int, BM: int, BN: int, elem_bytes: int = 2) -> int:
    """Tiles of one group that share a B panel: G distinct A panels + 1 B panel."""
    return G * a_panel_bytes(BM, K, elem_bytes) + b_panel_bytes(K, BN, elem_bytes)


def row_major_tile_id_gap(num_n_tiles: int) -> int:
    """tile_id distance between C(m, n) and C(m+1, n) under row-major order."""
    return num_n_tiles


def hmma_m16n8k16_count(M: int, N: int, K: int) -> int:
    """Instructions of shape m16n8k16 needed for 2MNK FLOPs."""
    per = 2 * 16 * 8 * 16
    assert flops(M, N, K) % per == 0
    return flops(M, N, K) // per


def tflops(M: int, N: int, K: int, ms: float) -> float:
    """Throughput in TFLOP/s of a GEMM that took ``ms`` milliseconds."""
    return flops(M, N, K) / (ms * 1e-3) / 1e12
