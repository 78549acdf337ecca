// Persistent FP16 GEMM kernel for sm_103a: C[M,N] = A[M,K] @ B[K,N], fp32 accumulate.
//
// What each part implements, and the page it comes from:
//  * tile GEMM body (masked/zero-filled loads, accumulator started from zero, C
//    overwritten): "(1/n) Triton matmul 커널 탐험 - persistent kernel은 그 자체로
//    빠르지 않다", section "naive tiled matmul";
//  * persistent grid and visiting order tile_id = pid, pid + grid, ...: same page,
//    section "naive persistent matmul";
//  * grouped ("CTA swizzle") tile order with the clipped last group:
//    "(2/n) Triton matmul 커널 탐험 - grouped ordering(CTA swizzle)...", section "구현";
//  * cross-tile pipelining (the next tile's loads run while the current tile is
//    stored): "(3/n) Triton matmul 커널 탐험 - cross tile pipelining 적용".
//
// GB300 design (not the pages' Triton/mma.sync design): one CTA per SM with
// warp-specialised roles that all walk the same static tile sequence:
//   producer warp(s)  TMA (or predicated loads) of A/B K-blocks into a
//                     STAGES-deep shared-memory ring guarded by mbarriers;
//   MMA warp          one thread issues tcgen05.mma (128x256x16, fp16 -> fp32)
//                     into one of two TMEM accumulators (2 x 256 columns);
//   4 epilogue warps  TMEM -> registers -> swizzled smem -> TMA store (or
//                     predicated coalesced stores) of the fp32 C tile.
// With cross-tile on, the producer and MMA move on to the next tile while the
// epilogue drains the other accumulator (the flattened loop of the "(3/n)"
// page); with it off, the producer waits for the previous tile's epilogue
// before loading the next tile.
//
// Every wait is bounded (GPU global timer); a wait that runs out records
// GEMM_ERR_TIMEOUT, tells the other CTAs of the same launch to stop, waits
// (bounded) for its own copies in flight, and the CTA frees its TMEM and exits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace g16 {

// ------------------------------------------------------------------ tile config
constexpr int BM = 128;           // rows of C per tile (TMEM lanes)
constexpr int BN = 256;           // columns of C per tile (TMEM columns per accumulator)
constexpr int BK = 64;            // K per stage: one 128-byte swizzle row of fp16
constexpr int STAGES = 4;         // shared-memory ring depth
constexpr int UMMA_K = 16;        // K of one tcgen05.mma kind::f16
constexpr int NUM_ACC = 2;        // TMEM accumulators (cross-tile double buffer)
constexpr int TMEM_COLS = NUM_ACC * BN;  // 512 = all of TMEM
constexpr int A_STAGE_BYTES = BM * BK * 2;  // 16 KiB
constexpr int B_STAGE_BYTES = BN * BK * 2;  // 32 KiB
constexpr int MN_CHUNK = 64;                // MN elements per 128-byte swizzle row
constexpr int MN_CHUNK_BYTES = MN_CHUNK * BK * 2;  // 8 KiB: one MN-major TMA box
constexpr int EPI_WARPS = 4;
constexpr int EPI_COLS = 32;                       // fp32 columns per epilogue chunk
constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 4;   // 32 rows x 128 B
constexpr int EPI_BUFS = 2;

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
constexpr int OFF_EPI = OFF_B + STAGES * B_STAGE_BYTES;
constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 2 * NUM_ACC + 1;
constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = OFF_TMEM_SLOT + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024 B

static_assert(OFF_B % 1024 == 0 && OFF_EPI % 1024 == 0, "swizzled buffers need 1 KiB alignment");
static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KiB per-CTA shared memory limit");

__host__ __device__ constexpr int load_warps(bool tma_load) { return tma_load ? 1 : 4; }
__host__ __device__ constexpr int cta_threads(bool tma_load) {
    return (load_warps(tma_load) + 1 + EPI_WARPS) * 32;
}

// ------------------------------------------------------------------ status words
// Sticky status (first error wins) and the launch epoch that must stop early.
// One copy per device in the module image; no allocation.
__device__ unsigned int g_status;
__device__ unsigned int g_abort_epoch;

constexpr unsigned int kStatusTimeout = 4;  // == GEMM_ERR_TIMEOUT

struct WaitCtl {
    uint64_t timeout_ns;
    uint32_t epoch;
};

__device__ __forceinline__ bool launch_aborted(uint32_t epoch) {
    return *reinterpret_cast<volatile unsigned int *>(&g_abort_epoch) == epoch;
}

// Slow path of a bounded wait. `bail` = also stop when another CTA of this
// launch gave up. kCluster: acquire at cluster scope (the barrier receives
// arrivals from the peer CTA). Returns false when the wait did not complete.
// The loop polls the barrier tightly: the clock and the launch-wide abort flag
// (a global-memory load) are consulted only every 1024 polls, so that a
// completed phase is noticed within one poll; these waits sit on the
// producer -> MMA -> producer hand-off that feeds the tensor pipe.
template <bool kCluster = false>
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, WaitCtl w, bool bail) {
    uint64_t t0 = 0;
    for (uint32_t n = 1;; ++n) {
        if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((n & 1023u) == 0) {
            const uint64_t t = global_timer_ns();
            if (t0 == 0) {
                t0 = t;
                continue;
            }
            if (bail && launch_aborted(w.epoch)) return false;
            if (t - t0 > w.timeout_ns) {
                atomicCAS(&g_status, 0u, kStatusTimeout);
                atomicExch(&g_abort_epoch, w.epoch);
                return false;
            }
        }
    }
}

// Waits made while cleaning up after an abort (copies or MMAs still in flight)
// use at least this bound, so that a very short user timeout cannot free TMEM
// or shared memory that asynchronous work is still using.
constexpr uint64_t kCleanupFloorNs = 100000000ull;  // 100 ms

__device__ __forceinline__ WaitCtl cleanup_wait(WaitCtl w) {
    if (w.timeout_ns < kCleanupFloorNs) w.timeout_ns = kCleanupFloorNs;
    return w;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, WaitCtl w) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow<false>(bar, parity, w, true);
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, WaitCtl w) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    return mbar_wait_slow<true>(bar, parity, w, true);
}

// ------------------------------------------------------------------ scheduler
struct Sched {
    int32_t nm;        // m-tiles
    int32_t nn;        // n-tiles
    int32_t group_m;   // GROUP_SIZE_M (>= 1 when grouped)
    int32_t grouped;   // 0: row-major order
};

// tile_id -> (tile_m, tile_n). Row-major: m = id / nn, n = id % nn. Grouped:
// groups of G m-tiles, m moving first inside a group, last group clipped to the
// m-tiles that remain. G >= nm gives the same map as G = nm (one group), so G is
// clipped first, which also keeps G * nn inside int32 (it is <= nm * nn).
__device__ __forceinline__ void tile_coords(int32_t tile_id, const Sched &s, int32_t &tm,
                                            int32_t &tn) {
    if (!s.grouped) {
        tm = tile_id / s.nn;
        tn = tile_id - tm * s.nn;
        return;
    }
    const int32_t G = s.group_m < s.nm ? s.group_m : s.nm;
    const int32_t per_group = G * s.nn;
    const int32_t group = tile_id / per_group;
    const int32_t in_group = tile_id - group * per_group;
    const int32_t first_m = group * G;
    const int32_t rest = s.nm - first_m;
    const int32_t gsize = G < rest ? G : rest;
    const int32_t q = in_group / gsize;
    tm = first_m + (in_group - q * gsize);
    tn = q;
}

// ------------------------------------------------------------------ parameters
struct Params {
    const uint16_t *A;  // used by the predicated load path
    const uint16_t *B;
    float *C;           // used by the predicated store path
    int64_t M, N, K;
    int64_t sam, sak, sbk, sbn, scm;  // element strides (stride_cn == 1)
    Sched sched;
    int32_t num_tiles;
    int32_t num_kb;     // cdiv(K, BK) >= 1
    // Split-K (CTA-pair kernel only): work unit u covers tile u % num_tiles and
    // k-blocks [s * kb_per_split, min(num_kb, (s + 1) * kb_per_split)) with
    // s = u / num_tiles; with splits > 1 the epilogue stores the partial tile into
    // slice s of the workspace (3-D tensor map in place of C's) instead of C.
    int32_t splits;     // >= 1
    int32_t kb_per_split;
    int32_t num_units;  // num_tiles * splits
    uint32_t a_mn;      // 1: A is M-major in memory (and in shared memory)
    uint32_t b_mn;      // 1: B is N-major
    uint32_t idesc;     // tcgen05 instruction descriptor
    uint32_t cross_tile;
    uint32_t l2_mode;   // bit 0: C stores evict-first; bit 1: A/B loads evict-last (pair kernel)
    uint32_t out_dtype; // C element type: 0 fp32, 1 fp16, 2 bf16 (nearest-even)
    float alpha;        // C = alpha * (A @ B)
    WaitCtl wait;
};

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A/B fp16, dense,
// per-operand major-ness, MMA shape M x N (M = 128 for one CTA, 256 for a pair).
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_mn, uint32_t b_mn, uint32_t m,
                                                  uint32_t n) {
    return (1u << 4)                 // D format: f32
           | (0u << 7) | (0u << 10)  // A, B format: f16
           | (a_mn << 15) | (b_mn << 16)
           | ((n >> 3) << 17)   // N / 8
           | ((m >> 4) << 24);  // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family layout):
// start address, leading / stride byte offsets (all >> 4), version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Operand tile in shared memory (R = 128 rows of A or 256 columns of B, BK = 64):
//  K-major : R rows of 128 B (64 k), 8-row swizzle atoms 1 KiB apart
//            -> LBO unused (16), SBO = 1024, next k16 slice at +32 B;
//  MN-major: R/64 chunks of [64 k rows x 128 B (64 mn)], 8 KiB apart
//            -> LBO = 8 KiB (next 64 mn), SBO = 1024 (next 8 k), next k16 at +2 KiB.
__device__ __forceinline__ uint64_t operand_desc(uint32_t tile_addr, uint32_t mn_major, int k16) {
    if (mn_major) return smem_desc(tile_addr + uint32_t(k16) * (UMMA_K * 128), MN_CHUNK_BYTES, 1024);
    return smem_desc(tile_addr + uint32_t(k16) * (UMMA_K * 2), 16, 1024);
}

// Descriptor stepping without rebuilding: the start address sits in the low
// 14 bits in units of 16 bytes, and every shared-memory address here is below
// 256 KiB, so adding (byte offset >> 4) to a descriptor moves its start address
// without carrying into the other fields. The MMA-issuing thread is on the
// critical path of the tensor pipe, so it only adds precomputed steps.
struct DescStep {
    uint64_t base;       // descriptor of stage 0, k16 slice 0
    uint32_t stage;      // (stage bytes) >> 4
    uint32_t k16;        // (bytes between consecutive k16 slices) >> 4
};

__device__ __forceinline__ DescStep make_desc_step(uint32_t tile_addr, uint32_t mn_major,
                                                   uint32_t stage_bytes) {
    DescStep d;
    d.base = operand_desc(tile_addr, mn_major, 0);
    d.stage = stage_bytes >> 4;
    d.k16 = (mn_major ? UMMA_K * 128u : UMMA_K * 2u) >> 4;
    return d;
}

// Byte offset of 16-byte unit `unit` (0..7) of 128-byte row `row` after the
// 128-byte swizzle (unit index XOR row mod 8).
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t unit) {
    return row * 128u + ((unit ^ (row & 7u)) << 4);
}

// Predicated copy of one operand tile into the swizzled layout the descriptors
// above describe; elements outside [0, mn_ext) x [0, K) read as zero.
// X(mn, k) = X[mn * s_mn + k * s_k].
template <int R>
__device__ __forceinline__ void load_operand_tile(uint32_t dst, const uint16_t *X, int64_t mn0,
                                                  int64_t mn_ext, int64_t k0, int64_t K,
                                                  int64_t s_mn, int64_t s_k, uint32_t mn_major,
                                                  int tid, int nthreads) {
    constexpr int CHUNKS = R * BK / 8;  // 8 contiguous elements per chunk
    for (int c = tid; c < CHUNKS; c += nthreads) {
        uint32_t off;
        int64_t mn, k;
        if (!mn_major) {  // chunk = 8 consecutive k of one mn
            const int r = c >> 3, u = c & 7;
            off = swz128(r, u);
            mn = mn0 + r;
            k = k0 + u * 8;
        } else {  // chunk = 8 consecutive mn of one k
            const int kk = c / (R / 8), mc = c % (R / 8);
            off = uint32_t(mc >> 3) * MN_CHUNK_BYTES + swz128(kk, mc & 7);
            mn = mn0 + mc * 8;
            k = k0 + kk;
        }
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            uint32_t lo = 0, hi = 0;
            const int64_t mn_a = mn_major ? mn + e : mn, k_a = mn_major ? k : k + e;
            const int64_t mn_b = mn_major ? mn + e + 1 : mn, k_b = mn_major ? k : k + e + 1;
            if (mn_a < mn_ext && k_a < K) lo = __ldg(X + mn_a * s_mn + k_a * s_k);
            if (mn_b < mn_ext && k_b < K) hi = __ldg(X + mn_b * s_mn + k_b * s_k);
            w[e >> 1] = lo | (hi << 16);
        }
        st_shared_v4(dst + off, w[0], w[1], w[2], w[3]);
    }
}

// ------------------------------------------------------------------ epilogue
// Drains one accumulator of this CTA to C: the calling warp reads TMEM lanes
// t_row.lane .. +31 (tile rows row0 .. row0+31) across BN columns in chunks of
// 32, and writes C[row0 + r][col_base + c] for rows < M and columns < N.
// TMA store: 128-byte-swizzled staging (two buffers per warp) + bulk tensor
// store, which clips the M/N edges. Otherwise: transpose through the staging
// buffer so each store instruction writes 32 consecutive floats of one row.
// `drained()` runs on every lane right after the last TMEM load of the tile.
//
// Pacing: every program walks the same tile sequence in step, so without it all
// epilogues would write their C tiles in the same few microseconds, a burst that
// saturates HBM and stalls the next tile's operand loads. For long work units
// the chunks are spread over the next unit's main loop (the accumulator is only
// needed again two units later). Measured at 16384^2 x 4096: tensor-pipe
// activity 89 % -> 92 %.
// Without cross-tile overlap the producer waits for the epilogue, so there is
// nothing to spread the stores over.
__device__ __forceinline__ uint32_t epilogue_pace_ns(int32_t unit_kblocks, uint32_t cross_tile) {
    return (cross_tile && unit_kblocks >= 32) ? uint32_t(unit_kblocks) * 20u : 0u;
}

template <bool kTmaStore, typename Drained>
__device__ __forceinline__ void epilogue_tile(uint32_t t_row, int64_t row0, int64_t col_base,
                                              const Params &p, const CUtensorMap *tmC, uint32_t stg,
                                              uint32_t &buf, int lane, Drained drained,
                                              int32_t split = 0, uint32_t pace_ns = 0) {
#pragma unroll 1
    for (int c = 0; c < BN / EPI_COLS; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_row + c * EPI_COLS, v);
        tmem_ld_wait();
        if (c == BN / EPI_COLS - 1) drained();
        if (p.alpha != 1.0f) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(p.alpha * __uint_as_float(v[i]));
        }
        const int64_t col0 = col_base + c * EPI_COLS;
        if (kTmaStore) {
            const uint32_t dst = stg + buf * EPI_BUF_BYTES;
            if (lane == 0) bulk_wait_group_read<EPI_BUFS - 1>();  // buffer free again
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u)
                st_shared_v4(dst + swz128(lane, u), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (row0 < p.M && col0 < p.N) {
                    if (p.splits > 1)  // partial tile -> workspace slice `split`, read once by the reduction
                        tma_store_3d_hint(tmC, dst, int32_t(col0), int32_t(row0), split,
                                          l2_policy_evict_normal());
                    else if (p.l2_mode & 1u)  // C is never read again: do not keep it in L2
                        tma_store_2d_hint(tmC, dst, int32_t(col0), int32_t(row0), l2_policy_evict_first());
                    else
                        tma_store_2d(tmC, dst, int32_t(col0), int32_t(row0));
                }
                bulk_commit_group();
            }
            buf ^= 1u;
            if (pace_ns != 0 && c < BN / EPI_COLS - 1) __nanosleep(pace_ns);
        } else {
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u)
                st_shared_v4(stg + swz128(lane, u), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            __syncwarp();
            const int64_t col = col0 + lane;
#pragma unroll 4
            for (int r = 0; r < 32; ++r) {
                const uint32_t bits = ld_shared_b32(stg + swz128(r, lane >> 2) + (lane & 3) * 4);
                const int64_t row = row0 + r;
                if (row < p.M && col < p.N) p.C[row * p.scm + col] = __uint_as_float(bits);
            }
        }
    }
}

// Two fp32 values -> one 32-bit word of two 16-bit values (lo in the low half),
// each round-to-nearest-even to fp16 (dtype 1) or bf16 (dtype 2).
__device__ __forceinline__ uint32_t pack_16x2(float lo, float hi, uint32_t dtype) {
    if (dtype == 1) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

// 16-bit C: like epilogue_tile, but 64 columns per chunk (two 32-column TMEM
// loads), scaled by alpha and rounded, so that each staging row is again 128
// bytes; the TMA store box is 64 x 32 elements of the 16-bit type.
template <bool kTmaStore, typename Drained>
__device__ __forceinline__ void epilogue_tile16(uint32_t t_row, int64_t row0, int64_t col_base,
                                                const Params &p, const CUtensorMap *tmC, uint32_t stg,
                                                uint32_t &buf, int lane, Drained drained,
                                                uint32_t pace_ns = 0) {
    const float alpha = p.alpha;
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
        uint32_t v[32], w[32];
        tmem_ld_32x32b_x32(t_row + c * 64, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[i] = pack_16x2(alpha * __uint_as_float(v[2 * i]), alpha * __uint_as_float(v[2 * i + 1]),
                             p.out_dtype);
        tmem_ld_32x32b_x32(t_row + c * 64 + 32, v);
        tmem_ld_wait();
        if (c == BN / 64 - 1) drained();
#pragma unroll
        for (int i = 0; i < 16; ++i)
            w[16 + i] = pack_16x2(alpha * __uint_as_float(v[2 * i]),
                                  alpha * __uint_as_float(v[2 * i + 1]), p.out_dtype);
        const int64_t col0 = col_base + c * 64;
        if (kTmaStore) {
            const uint32_t dst = stg + buf * EPI_BUF_BYTES;
            if (lane == 0) bulk_wait_group_read<EPI_BUFS - 1>();
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u)
                st_shared_v4(dst + swz128(lane, u), w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (row0 < p.M && col0 < p.N)
                    tma_store_2d_hint(tmC, dst, int32_t(col0), int32_t(row0), l2_policy_evict_first());
                bulk_commit_group();
            }
            buf ^= 1u;
            if (pace_ns != 0 && c < BN / 64 - 1) __nanosleep(pace_ns);
        } else {
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u)
                st_shared_v4(stg + swz128(lane, u), w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
            __syncwarp();
            const int64_t col = col0 + 2 * lane;  // this lane: columns col, col + 1
            uint16_t *C16 = reinterpret_cast<uint16_t *>(p.C);
#pragma unroll 4
            for (int r = 0; r < 32; ++r) {
                const uint32_t word = ld_shared_b32(stg + swz128(r, lane >> 2) + (lane & 3) * 4);
                const int64_t row = row0 + r;
                if (row < p.M) {
                    if (col < p.N) C16[row * p.scm + col] = uint16_t(word & 0xffffu);
                    if (col + 1 < p.N) C16[row * p.scm + col + 1] = uint16_t(word >> 16);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ the kernel
template <bool kTmaLoad, bool kTmaStore>
__global__ void __launch_bounds__(cta_threads(kTmaLoad), 1)
    gemm_f16_persistent(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const Params p) {
    constexpr int LOAD_WARPS = load_warps(kTmaLoad);
    constexpr int MMA_WARP = LOAD_WARPS;
    constexpr int EPI_WARP0 = LOAD_WARPS + 1;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);

    const uint32_t sA = base + OFF_A;
    const uint32_t sB = base + OFF_B;
    const uint32_t bar0 = base + OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + NUM_ACC + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * NUM_ACC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM_SLOT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), kTmaLoad ? 1 : LOAD_WARPS * 32);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EPI_WARPS * 32);
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (kTmaLoad && warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (kTmaStore && warp == EPI_WARP0 && lane == 0) prefetch_tensormap(&tmC);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int32_t grid = gridDim.x;
    const int32_t num_kb = p.num_kb;

    if (warp < LOAD_WARPS) {
        // ============================================================ producer
        if (kTmaLoad) {
            if (lane == 0) {
                uint32_t stage = 0, phase = 0;
                uint32_t issued = 0;
                bool ok = true;
                int32_t it = 0;
                for (int32_t tile = blockIdx.x; ok && tile < p.num_tiles; tile += grid, ++it) {
                    int32_t tm, tn;
                    tile_coords(tile, p.sched, tm, tn);
                    if (!p.cross_tile && it > 0) {
                        const int32_t j = it - 1;  // wait until tile j's accumulator is drained
                        if (!mbar_wait(tempty_bar(j & 1), (j >> 1) & 1, p.wait)) { ok = false; break; }
                    }
                    const int32_t m0 = tm * BM, n0 = tn * BN;
                    for (int32_t kb = 0; kb < num_kb; ++kb) {
                        if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.wait)) { ok = false; break; }
                        const uint32_t fb = full_bar(stage);
                        mbar_arrive_expect_tx(fb, A_STAGE_BYTES + B_STAGE_BYTES);
                        const int32_t k0 = kb * BK;
                        const uint32_t a_dst = sA + stage * A_STAGE_BYTES;
                        const uint32_t b_dst = sB + stage * B_STAGE_BYTES;
                        if (!p.a_mn) {
                            tma_load_2d(a_dst, &tmA, k0, m0, fb);
                        } else {
#pragma unroll
                            for (int c = 0; c < BM / MN_CHUNK; ++c)
                                tma_load_2d(a_dst + c * MN_CHUNK_BYTES, &tmA, m0 + c * MN_CHUNK, k0, fb);
                        }
                        if (!p.b_mn) {
                            tma_load_2d(b_dst, &tmB, k0, n0, fb);
                        } else {
#pragma unroll
                            for (int c = 0; c < BN / MN_CHUNK; ++c)
                                tma_load_2d(b_dst + c * MN_CHUNK_BYTES, &tmB, n0 + c * MN_CHUNK, k0, fb);
                        }
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                }
                if (!ok) {
                    // Let the copies this thread started land before the CTA exits.
                    const uint32_t n = issued < STAGES ? issued : STAGES;
                    for (uint32_t q = issued - n; q < issued; ++q)
                        mbar_wait_slow(full_bar(q % STAGES), (q / STAGES) & 1u, cleanup_wait(p.wait),
                                       false);
                }
            }
            __syncwarp();
        } else {
            const int tid = threadIdx.x;  // 0 .. LOAD_WARPS*32-1
            constexpr int NT = LOAD_WARPS * 32;
            uint32_t stage = 0, phase = 0;
            int32_t it = 0;
            bool ok = true;
            for (int32_t tile = blockIdx.x; ok && tile < p.num_tiles; tile += grid, ++it) {
                int32_t tm, tn;
                tile_coords(tile, p.sched, tm, tn);
                if (!p.cross_tile && it > 0) {
                    const int32_t j = it - 1;
                    if (!mbar_wait(tempty_bar(j & 1), (j >> 1) & 1, p.wait)) { ok = false; break; }
                }
                const int64_t m0 = int64_t(tm) * BM, n0 = int64_t(tn) * BN;
                for (int32_t kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.wait)) { ok = false; break; }
                    const int64_t k0 = int64_t(kb) * BK;
                    load_operand_tile<BM>(sA + stage * A_STAGE_BYTES, p.A, m0, p.M, k0, p.K, p.sam,
                                          p.sak, p.a_mn, tid, NT);
                    load_operand_tile<BN>(sB + stage * B_STAGE_BYTES, p.B, n0, p.N, k0, p.K, p.sbn,
                                          p.sbk, p.b_mn, tid, NT);
                    fence_proxy_async_smem();
                    mbar_arrive(full_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == MMA_WARP) {
        // ============================================================ MMA issuer
        // The whole warp runs this loop with warp-uniform values; every lane
        // waits on the barriers (votes keep the outcome uniform) and one
        // elected lane issues each MMA and commit.
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        int32_t it = 0;
        const DescStep da = make_desc_step(sA, p.a_mn, A_STAGE_BYTES);
        const DescStep db = make_desc_step(sB, p.b_mn, B_STAGE_BYTES);
        const uint32_t idesc = p.idesc;
        for (int32_t tile = blockIdx.x; ok && tile < p.num_tiles; tile += grid, ++it) {
            const uint32_t acc = it & 1, use = it >> 1;
            if (!__all_sync(0xffffffffu, mbar_wait(tempty_bar(acc), (use & 1u) ^ 1u, p.wait))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int32_t kb = 0; kb < num_kb; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(full_bar(stage), phase, p.wait))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t a0 = da.base + stage * da.stage;
                const uint64_t b0 = db.base + stage * db.stage;
#pragma unroll
                for (int k16 = 0; k16 < BK / UMMA_K; ++k16)
                    mma_f16_elect(d_tmem, a0 + k16 * da.k16, b0 + k16 * db.k16, idesc,
                                  (kb | k16) != 0 ? 1u : 0u);
                mma_commit_elect(empty_bar(stage));  // slot reusable once these MMAs finish
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            mma_commit_elect(tfull_bar(acc));  // accumulator complete
        }
        // No MMA may still be writing TMEM when it is freed.
        mma_commit_elect(drain_bar);
        __all_sync(0xffffffffu, mbar_wait_slow(drain_bar, 0, cleanup_wait(p.wait), false));
    } else {
        // ============================================================ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access = tile rows q*32..q*32+31
        const int ew = warp - EPI_WARP0;
        const uint32_t stg = base + OFF_EPI + uint32_t(ew) * (EPI_BUFS * EPI_BUF_BYTES);
        uint32_t buf = 0;
        int32_t it = 0;
        for (int32_t tile = blockIdx.x; tile < p.num_tiles; tile += grid, ++it) {
            int32_t tm, tn;
            tile_coords(tile, p.sched, tm, tn);
            const uint32_t acc = it & 1, use = it >> 1;
            // every lane waits (acquire), then the decision is made warp-uniform so
            // the .sync.aligned TMEM loads below run converged
            const bool ready = __all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), use & 1u, p.wait));
            if (!ready) break;
            tc_fence_after();
            const int64_t row0 = int64_t(tm) * BM + q * 32;
            const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + acc * BN;
            auto release = [&] {
                tc_fence_before();
                mbar_arrive(tempty_bar(acc));  // accumulator may be overwritten
            };
            if (p.out_dtype == 0)
                epilogue_tile<kTmaStore>(t_row, row0, int64_t(tn) * BN, p, &tmC, stg, buf, lane, release,
                                         0, epilogue_pace_ns(num_kb, p.cross_tile));
            else
                epilogue_tile16<kTmaStore>(t_row, row0, int64_t(tn) * BN, p, &tmC, stg, buf, lane,
                                           release, epilogue_pace_ns(num_kb, p.cross_tile));
        }
        if (kTmaStore && lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ helpers
// Failure-detection self-test: one thread waits, through the same bounded wait
// the GEMM roles use, on an mbarrier that nothing ever arrives on. The wait runs
// out after `timeout_ns`, records GEMM_ERR_TIMEOUT in the sticky status and
// returns; the context stays usable.
__global__ void wait_timeout_selftest_kernel(WaitCtl w) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    mbar_wait(b, 0, w);  // phase 0 never completes
}

__global__ void tile_map_kernel(Sched s, int32_t num_tiles, int32_t *out) {
    if (threadIdx.x != 0) return;
    for (int32_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int32_t tm, tn;
        tile_coords(t, s, tm, tn);
        out[3 * int64_t(t) + 0] = int32_t(blockIdx.x);
        out[3 * int64_t(t) + 1] = tm;
        out[3 * int64_t(t) + 2] = tn;
    }
}

// Split-K reduction: C[i][j] = sum over s = 0 .. S-1, in that order, of
// W[s][i][j] (W dense [S][M][ldw] fp32). Fixed order: the result does not
// depend on scheduling. Four consecutive columns per thread.
__global__ void splitk_reduce_kernel(const float *__restrict__ W, void *__restrict__ Cv, int64_t M,
                                     int64_t N, int64_t ldw, int64_t scm, int32_t S,
                                     uint32_t out_dtype, float alpha) {
    const int64_t nq = (N + 3) / 4;
    const int64_t total = M * nq;
    const int64_t slice = M * ldw;
    float *C = static_cast<float *>(Cv);
    const bool vec_c = (scm % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0);
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = e / nq, j = (e - i * nq) * 4;
        const float *w = W + i * ldw + j;
        float4 acc = *reinterpret_cast<const float4 *>(w);  // ldw % 4 == 0, W 16-byte aligned
        for (int32_t s = 1; s < S; ++s) {
            const float4 v = *reinterpret_cast<const float4 *>(w + s * slice);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        if (alpha != 1.0f) {
            acc.x *= alpha;
            acc.y *= alpha;
            acc.z *= alpha;
            acc.w *= alpha;
        }
        if (out_dtype != 0) {
            uint16_t *c16 = static_cast<uint16_t *>(Cv) + i * scm + j;
            const uint32_t w01 = pack_16x2(acc.x, acc.y, out_dtype);
            const uint32_t w23 = pack_16x2(acc.z, acc.w, out_dtype);
            c16[0] = uint16_t(w01 & 0xffffu);
            if (j + 1 < N) c16[1] = uint16_t(w01 >> 16);
            if (j + 2 < N) c16[2] = uint16_t(w23 & 0xffffu);
            if (j + 3 < N) c16[3] = uint16_t(w23 >> 16);
            continue;
        }
        float *c = C + i * scm + j;
        if (vec_c && j + 3 < N) {
            *reinterpret_cast<float4 *>(c) = acc;
        } else {
            c[0] = acc.x;
            if (j + 1 < N) c[1] = acc.y;
            if (j + 2 < N) c[2] = acc.z;
            if (j + 3 < N) c[3] = acc.w;
        }
    }
}

// K == 0: C := 0 (the accumulator starts at zero and no K step adds to it).
__global__ void zero_c_kernel(void *C, int64_t M, int64_t N, int64_t scm, int32_t esize) {
    const int64_t total = M * N;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e - i * N;
        if (esize == 4)
            static_cast<float *>(C)[i * scm + j] = 0.0f;
        else
            static_cast<uint16_t *>(C)[i * scm + j] = 0;
    }
}

}  // namespace g16
