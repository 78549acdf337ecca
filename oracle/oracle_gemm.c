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

/* ---------------------------------------------------------------------------
 * Rounding to a 16-bit IEEE-style format, from the formats' definitions:
 * sign bit, `ebits` exponent bits with bias 2^(ebits-1) - 1, `mbits` fraction
 * bits; binary16 is (5, 10), bfloat16 is (8, 7). Round to nearest, ties to the
 * even fraction (nearbyint in the default rounding mode); values at or beyond
 * the midpoint between the largest finite value and 2^(emax+1) become
 * infinity; NaN -> quiet NaN. Returns the bit pattern.
 * ------------------------------------------------------------------------- */
static uint16_t round_ieee16(double x, int ebits, int mbits) {
    const int bias = (1 << (ebits - 1)) - 1;
    const int emax = bias, emin = 1 - bias;
    const uint16_t sign = signbit(x) ? (uint16_t)(1u << 15) : 0;
    const uint16_t inf = (uint16_t)(((1u << ebits) - 1u) << mbits);
    if (isnan(x)) return (uint16_t)(inf | (1u << (mbits - 1)));
    double a = fabs(x);
    if (a == 0.0) return sign;
    /* largest finite: (2 - 2^-mbits) * 2^emax; overflow from the midpoint up */
    const double limit = ldexp(2.0 - ldexp(1.0, -(mbits + 1)), emax);
    if (a >= limit) return (uint16_t)(sign | inf);
    int e2;
    frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1): a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    if (E < emin) E = emin; /* subnormal range shares the smallest normal's quantum */
    const double q = ldexp(1.0, E - mbits);
    double n = nearbyint(a / q); /* exact scaling by a power of two, then RNE */
    /* n in [0, 2^(mbits+1)]; 2^(mbits+1) carries into the next binade */
    uint32_t bits;
    if (E == emin && n < ldexp(1.0, mbits)) {
        bits = (uint32_t)n; /* subnormal (or the smallest normal when n reaches 2^mbits) */
    } else {
        if (n >= ldexp(1.0, mbits + 1)) {
            n = ldexp(1.0, mbits);
            E += 1;
        }
        if (E > emax) return (uint16_t)(sign | inf);
        bits = ((uint32_t)(E + bias) << mbits) | (uint32_t)(n - ldexp(1.0, mbits));
    }
    return (uint16_t)(sign | bits);
}

uint16_t oracle_f64_to_f16(double x) { return round_ieee16(x, 5, 10); }
uint16_t oracle_f64_to_bf16(double x) { return round_ieee16(x, 8, 7); }

/* bfloat16 -> double from the format (8 exponent bits, bias 127, 7 fraction bits). */
double oracle_bf16_to_f64(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133); /* 2^-126 * f / 2^7 */
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp(128.0 + (double)f, e - 134); /* 2^(e-127) * (128+f) / 2^7 */
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
