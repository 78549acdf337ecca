/*
 * Oracle for the dense FP16 GEMM: plain CPU reference code.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the CPU
 * baseline / reference arm of bench.py may load this library. The product path
 * (the CUDA library under dense_gemm_gb300/) never includes, links or calls it,
 * and this file includes nothing from there.
 *
 * What is computed, and where the pages define it:
 *
 *  - oracle_gemm_block: C[i,j] = sum_k A[i,k] * B[k,j], the dense product the
 *    pages' kernels compute ("(1/n) Triton matmul ... persistent kernel",
 *    section "naive tiled matmul": loads masked with zero fill, an FP32
 *    accumulator started from zero, C stored, never read). Tiling and ordering
 *    change only the order of the same multiply-adds ("4주차 정리: Roofline과
 *    Tiling", section 5 "일반 공식", the FLOP row of the tile table), so the
 *    oracle is the definition itself: every fp16 input widened exactly to
 *    double, products and sums in double, k ascending.
 *
 *  - oracle_tile_coord / oracle_schedule: the tile_id -> (tile_m, tile_n) maps.
 *    Row-major: "(1/n) ... persistent kernel", section "naive tiled matmul"
 *    (tile_m = tile_id // num_n_tiles, tile_n = tile_id % num_n_tiles).
 *    Grouped ("CTA swizzle"): "(2/n) Triton matmul ... grouped ordering(CTA
 *    swizzle)", section "구현" (implementation), steps SWIZZLE 1-3, including
 *    the short last group clipped by a minimum. The persistent visiting order
 *    (program pid takes tile_id = pid, pid + P, pid + 2P, ...) is from
 *    "(1/n) ...", section "naive persistent matmul".
 *
 *  - oracle_fp16_to_f64: IEEE 754 binary16 decoding written from the format's
 *    definition (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits).
 *
 * Parity pins: every function here is pinned by -m "not gpu" tests against
 * closed forms, brute force and library routines (tests/test_oracle.py).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------
 * IEEE binary16 -> double, from the format definition.
 *   e == 0        : subnormal, value = (-1)^s * 2^-14 * (f / 1024)
 *   1 <= e <= 30  : normal,    value = (-1)^s * 2^(e-15) * (1 + f / 1024)
 *   e == 31       : f == 0 -> infinity, else NaN
 * ------------------------------------------------------------------------- */
double oracle_fp16_to_f64(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* 2^-14 * f / 2^10 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp(1024.0 + (double)f, e - 25); /* 2^(e-15) * (1024+f) / 2^10 */
    }
    return s ? -v : v;
}

/* Decode table: one entry per 16-bit pattern, filled from the function above. */
static double g_h2d[65536];
static int g_h2d_ready = 0;

static void h2d_init(void) {
    if (g_h2d_ready) return;
    for (int i = 0; i < 65536; ++i) g_h2d[i] = oracle_fp16_to_f64((uint16_t)i);
    g_h2d_ready = 1;
}

void oracle_init(void) { h2d_init(); }

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * out[r][c] = sum_{k=0}^{K-1} A(rows[r], k) * B(k, col0 + c)
 *   for r < n_rows, c < n_cols, in double.
 * A(i,k) = A[i*sam + k*sak], B(k,j) = B[k*sbk + j*sbn] (strides in elements,
 * like the pages' stride arguments). out is dense row-major [n_rows][n_cols].
 * Rows run in parallel when the library is built with OpenMP; each output
 * element is still summed by one thread with k ascending, so the result does
 * not depend on the thread count. K == 0 gives zeros.
 * Returns 0, or -1 for invalid arguments.
 * ------------------------------------------------------------------------- */
int oracle_gemm_block(const uint16_t *A, const uint16_t *B,
                      int64_t M, int64_t N, int64_t K,
                      int64_t sam, int64_t sak, int64_t sbk, int64_t sbn,
                      const int64_t *rows, int64_t n_rows,
                      int64_t col0, int64_t n_cols,
                      double *out, int n_threads) {
    if (M < 0 || N < 0 || K < 0 || n_rows < 0 || n_cols < 0 || col0 < 0) return -1;
    if (col0 + n_cols > N) return -1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    h2d_init();
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int64_t r;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (r = 0; r < n_rows; ++r) {
        const int64_t i = rows[r];
        double *c = out + r * n_cols;
        for (int64_t j = 0; j < n_cols; ++j) c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = g_h2d[A[i * sam + k * sak]];
            const uint16_t *brow = B + k * sbk + col0 * sbn;
            for (int64_t j = 0; j < n_cols; ++j) c[j] += a * g_h2d[brow[j * sbn]];
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Tile maps.
 * grouped == 0: row-major order over the nm x nn tile grid.
 * grouped != 0: groups of G m-tiles; inside a group the m index moves first;
 *               the last group holds min(G, nm - first_tile_m) m-tiles.
 * Returns 0, or -1 for invalid arguments (G < 1 only matters when grouped).
 * ------------------------------------------------------------------------- */
int oracle_tile_coord(int64_t tile_id, int64_t nm, int64_t nn, int64_t G, int grouped,
                      int64_t *tile_m, int64_t *tile_n) {
    if (nm < 1 || nn < 1 || tile_id < 0 || tile_id >= nm * nn) return -1;
    if (!grouped) {
        *tile_m = tile_id / nn;
        *tile_n = tile_id % nn;
        return 0;
    }
    if (G < 1) return -1;
    /* SWIZZLE 1: which group, where it starts */
    const int64_t num_tiles_in_group = G * nn;
    const int64_t group_id = tile_id / num_tiles_in_group;
    const int64_t tile_id_in_group = tile_id % num_tiles_in_group;
    const int64_t first_tile_m = group_id * G;
    /* SWIZZLE 2: the last group may be shorter than G */
    int64_t group_size_m = nm - first_tile_m;
    if (G < group_size_m) group_size_m = G;
    /* SWIZZLE 3: m moves first inside the group */
    *tile_m = first_tile_m + tile_id_in_group % group_size_m;
    *tile_n = tile_id_in_group / group_size_m;
    return 0;
}

/* Persistent schedule: program pid (0 <= pid < grid) visits
 * tile_id = pid, pid + grid, pid + 2*grid, ... while tile_id < nm*nn.
 * out[3*tile_id + 0..2] = {pid, tile_m, tile_n}. */
int oracle_schedule(int64_t nm, int64_t nn, int64_t G, int grouped, int64_t grid,
                    int32_t *out) {
    if (nm < 1 || nn < 1 || grid < 1) return -1;
    if (grouped && G < 1) return -1;
    const int64_t T = nm * nn;
    for (int64_t pid = 0; pid < grid; ++pid) {
        for (int64_t t = pid; t < T; t += grid) {
            int64_t tm, tn;
            if (oracle_tile_coord(t, nm, nn, G, grouped, &tm, &tn) != 0) return -1;
            out[3 * t + 0] = (int32_t)pid;
            out[3 * t + 1] = (int32_t)tm;
            out[3 * t + 2] = (int32_t)tn;
        }
    }
    return 0;
}
