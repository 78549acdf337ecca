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
constexpr int EPI_WARPS = 8;                       // two per TMEM lane quarter
constexpr int EPI_COLS = 32;                       // fp32 columns per epilogue chunk
constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 4;   // 32 rows x 128 B
constexpr int EPI_BUFS = 1;

// Predicated-load path: for operands that one tensor map cannot describe (a
// row stride or a base address that is not a multiple of 16 bytes).
// Terms: a "row" of an operand runs along its unit stride (K for a K-major
// operand, M or N for an M/N-major one); S is the element distance between
// rows. A "line" is 64 elements of one row: one 128-byte swizzle row of a
// stage. Rows rho with rho mod P == c (P = 16 / gcd(2S mod 16, 16) <= 8) form
// alignment class c: they all start m_c bytes into a 16-byte granule, and two
// consecutive rows of a class are 2*S*P bytes apart, a multiple of 16. Each
// class gets its own tensor map whose rows begin at those granule boundaries,
// so TMA copies boxes of h class rows x 72 elements (a line plus up to 7
// leading elements; h = 16, or 8 for an M/N-major operand with 8 classes)
// into a staging ring, with zero fill past the matrix edges, and loader warps
// shift each line by m_c bytes into the stage. A loader warp handles copy
// groups of 64 lines.
constexpr int MAX_CLASSES = 8;
constexpr int BOX_W = 72;                           // elements per staged line
constexpr int LINE_PITCH = BOX_W * 2;               // 144 bytes
constexpr int GROUP_LINES = 64;
constexpr int GROUP_BYTES = GROUP_LINES * LINE_PITCH;  // 9216 = 72 x 128
constexpr int COPY_DEPTH = 3;                       // copy groups in flight per loader warp
// one-CTA kernel: three loader warps, two groups each per K-block
constexpr int PRED_LOAD_WARPS = 3;
constexpr int A_GROUPS = BM / GROUP_LINES, B_GROUPS = BN / GROUP_LINES;
constexpr int GROUPS_PER_KB = A_GROUPS + B_GROUPS;  // 6
constexpr int WARP_GROUPS = GROUPS_PER_KB / PRED_LOAD_WARPS;
static_assert(GROUPS_PER_KB % PRED_LOAD_WARPS == 0, "equal loader shares");

// log2 of the box height for an operand with 2^lp classes (host and device).
__host__ __device__ constexpr int class_box_lh(bool mn_major, int lp) {
    // rows per class in one 64-deep k-block tile: 64 / P (M/N-major) or >= 128 / P
    return mn_major ? (6 - lp < 4 ? 6 - lp : 4) : 4;
}

// Shared-memory map of the one-CTA kernel. The predicated-load variant keeps
// two operand stages and holds the loader warps' staging rings (with one
// mbarrier per ring slot) in the space of the others.
template <bool kTmaLoad>
struct Layout {
    static constexpr int stages = kTmaLoad ? STAGES : 2;
    static constexpr int off_a = 0;
    static constexpr int off_b = off_a + stages * A_STAGE_BYTES;
    static constexpr int off_epi = off_b + stages * B_STAGE_BYTES;
    static constexpr int off_copy = off_epi + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
    static constexpr int copy_slots = kTmaLoad ? 0 : PRED_LOAD_WARPS * COPY_DEPTH;
    static constexpr int off_bar = off_copy + copy_slots * GROUP_BYTES;
    static constexpr int copy_bar0 = 2 * stages + 2 * NUM_ACC + 1;  // index of the first slot barrier
    static constexpr int num_bars = copy_bar0 + copy_slots;
    static constexpr int off_tmem_slot = off_bar + num_bars * 8;
    static constexpr int smem_bytes = off_tmem_slot + 16 + 1024;  // slack to align the base to 1 KiB
    static_assert(off_b % 1024 == 0 && off_epi % 1024 == 0, "swizzled buffers need 1 KiB alignment");
    static_assert(off_copy % 128 == 0 && GROUP_BYTES % 128 == 0 && (8 * LINE_PITCH) % 128 == 0,
                  "TMA box destinations (multiples of 8 lines) need 128-byte alignment");
    static_assert(smem_bytes <= 232448, "exceeds the 227 KiB per-CTA shared memory limit");
};

// Tensor maps of the alignment classes of A and B (predicated-load variant).
struct ClassMaps {
    CUtensorMap a[MAX_CLASSES];
    CUtensorMap b[MAX_CLASSES];
};
struct NoClassMaps {
    uint32_t unused;
};
template <bool kTmaLoad>
struct ClassMapsFor {
    using type = ClassMaps;
};
template <>
struct ClassMapsFor<true> {
    using type = NoClassMaps;
};

// CTA-pair kernel with C stored per row class (see epilogue_tile_class): the
// maps of C's classes, beside those of A and B for predicated loads.
constexpr int MAX_C_CLASSES = 4;
struct CClassMaps {
    CUtensorMap c[MAX_C_CLASSES];
};
struct ClassMapsAndC {
    CUtensorMap a[MAX_CLASSES];
    CUtensorMap b[MAX_CLASSES];
    CUtensorMap c[MAX_C_CLASSES];
};
template <bool kTmaLoad, bool kClassStore>
struct PairMapsFor {
    using type = typename ClassMapsFor<kTmaLoad>::type;
};
template <>
struct PairMapsFor<true, true> {
    using type = CClassMaps;
};
template <>
struct PairMapsFor<false, true> {
    using type = ClassMapsAndC;
};

__host__ __device__ constexpr int load_warps(bool tma_load) { return tma_load ? 1 : PRED_LOAD_WARPS; }
__host__ __device__ constexpr int cta_threads(bool tma_load) {
    return (load_warps(tma_load) + 1 + EPI_WARPS) * 32;
}

// ------------------------------------------------------------------ status words
// Sticky status (first error wins) and the launch epoch that must stop early.
// One copy per device in the module image; no allocation.
__device__ unsigned int g_status;
__device__ unsigned int g_abort_epoch;

constexpr unsigned int kStatusTimeout = 4;  // == GEMM_ERR_TIMEOUT
constexpr unsigned int kStatusCheck = 5;    // == GEMM_ERR_CHECK (debug build)

#ifdef GEMM_DEBUG
// Source line of the first failed debug check (read by gemm_f16_sync_status).
__device__ unsigned int g_check_line;

__device__ __noinline__ bool check_failed(int line) {
    if (atomicCAS(&g_status, 0u, kStatusCheck) == 0u) atomicExch(&g_check_line, unsigned(line));
    return false;
}
#endif

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
    int32_t num_units;  // num_tiles * splits, or with a split tail tail_first + tail_splits * tail_tiles
    // Split tail (CTA-pair kernel, GEMM_SCHED_TAIL_SPLIT): units below tail_first
    // are whole tiles; the last tail_tiles tiles (fewer than one round of
    // programs) are split along K into slices of tail_kps k-blocks. Unit
    // tail_first + v covers tile tail_first + v % tail_tiles and slice
    // v / tail_tiles, and stores its fp32 partial tile into slot v of the scratch.
    int32_t tail_first;
    int32_t tail_tiles;
    int32_t tail_kps;
    uint32_t a_mn;      // 1: A is M-major in memory (and in shared memory)
    uint32_t b_mn;      // 1: B is N-major
    uint32_t idesc;     // tcgen05 instruction descriptor
    uint32_t cross_tile;
    uint32_t l2_mode;   // bit 0: C stores evict-first; bit 1: A/B loads evict-last (pair kernel)
    uint32_t out_dtype; // C element type: 0 fp32, 1 fp16, 2 bf16 (nearest-even)
    uint32_t dynamic;   // units taken by cluster launch control (logged; the kernel instantiation decides)
    uint32_t relay;     // CTA pairs with TMA loads: CTA 1's drained tiles reach CTA 0 through one relay arrive
    // predicated loads, per operand (0 = A, 1 = B): log2 of the class count P
    // and of the box height, each class's byte offset in its first granule (4
    // bits per class), and the classes that hold rows
    uint32_t cls_lp[2];
    uint32_t cls_lh[2];
    uint32_t cls_mis[2];
    uint32_t cls_live[2];
    uint32_t c_classes; // C stored per row class: number of classes P (1, 2 or 4), 0 otherwise
    float alpha;        // C = alpha * (A @ B)
    // Failure-detection self-test only (0 otherwise): the CTA-pair producers
    // issue no copies once they have issued this many stages, and keep waiting
    // for stages to be freed, so that the MMA warp's wait runs out.
    int32_t stop_after;
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

// ------------------------------------------------------------------ predicated loads
// Position of a predicated loader warp in the static work sequence: tile
// (it-th of this CTA), K-block, and which of the warp's copy groups of that
// K-block (group index warp + PRED_LOAD_WARPS * g of GROUPS_PER_KB).
struct LineCursor {
    int32_t tile, it, kb, g;
    int64_t m0, n0;

    __device__ __forceinline__ void coords(const Params &p) {
        if (tile < p.num_tiles) {
            int32_t tm, tn;
            tile_coords(tile, p.sched, tm, tn);
            m0 = int64_t(tm) * BM;
            n0 = int64_t(tn) * BN;
        }
    }
    __device__ __forceinline__ void start(int32_t first, const Params &p) {
        tile = first;
        it = kb = g = 0;
        m0 = n0 = 0;
        coords(p);
    }
    __device__ __forceinline__ bool valid(const Params &p) const { return tile < p.num_tiles; }
    __device__ __forceinline__ void next(const Params &p, int32_t grid) {
        if (++g < WARP_GROUPS) return;
        g = 0;
        if (++kb < p.num_kb) return;
        kb = 0;
        tile += grid;
        ++it;
        coords(p);
    }
};

// Copy group g of one operand's 2^lr-line tile (lines 64g .. 64g+63) of a
// K-block. Box beta of the operand covers class c, row block b (h class rows)
// and 64-element segment s, s fastest: an operand has NS = R/64 segments per
// row when M/N-major (rows are k, 64 per K-block) and 1 when K-major (rows are
// m or n, R per tile).
struct GroupShape {
    int op;                 // 0 = A, 1 = B
    int first_box;          // beta of the group's first box
    int lp, lns, lbc, lh;   // log2 of: classes P, segments per row NS, row blocks per class, box height
    uint32_t mn_major;
    int64_t mn0;            // first m (A) or n (B) of the tile

    // box beta -> class, row block, segment (all counts are powers of two)
    __device__ __forceinline__ int cls(int beta) const { return beta >> (lbc + lns); }
    __device__ __forceinline__ int blk(int beta) const { return (beta >> lns) & ((1 << lbc) - 1); }
    __device__ __forceinline__ int seg(int beta) const { return beta & ((1 << lns) - 1); }
};

__device__ __forceinline__ GroupShape group_shape(const Params &p, int op, int g, int lr, int64_t mn0) {
    GroupShape gs;
    gs.op = op;
    gs.mn_major = op == 0 ? p.a_mn : p.b_mn;
    gs.lp = int(op == 0 ? p.cls_lp[0] : p.cls_lp[1]);
    gs.lh = int(op == 0 ? p.cls_lh[0] : p.cls_lh[1]);
    gs.lns = gs.mn_major ? lr - 6 : 0;
    gs.lbc = (gs.mn_major ? 6 : lr) - gs.lp - gs.lh;  // rows per tile / (P h)
    gs.first_box = g << (6 - gs.lh);                   // 64 / h boxes per group
    gs.mn0 = mn0;
    return gs;
}

// Starts the TMA copies of one group into ring slot `slot`; they complete on
// `bar`. Lane 0 announces the byte count, then lane i < 64/h issues box i
// (boxes of classes without rows are skipped and placed as zeros). Whole warp.
template <typename Maps>
__device__ __forceinline__ void issue_class_group(const Params &p, const Maps &cm, const GroupShape &gs,
                                                  int64_t k0, uint32_t slot, uint32_t bar, int lane) {
    const uint32_t live = gs.op == 0 ? p.cls_live[0] : p.cls_live[1];
    const int nbox = GROUP_LINES >> gs.lh;
    const uint32_t box_bytes = uint32_t(LINE_PITCH) << gs.lh;
    if (lane == 0) {
        uint32_t boxes = 0;
        for (int i = 0; i < nbox; ++i) boxes += (live >> gs.cls(gs.first_box + i)) & 1u;
        fence_proxy_async_smem();  // this slot's staging reads precede the new copies
        mbar_arrive_expect_tx(bar, boxes * box_bytes);
    }
    __syncwarp();
    if (lane < nbox) {
        const int32_t xb = int32_t(gs.mn_major ? gs.mn0 : k0);              // unit-stride coordinate
        const int32_t yb = int32_t((gs.mn_major ? k0 : gs.mn0) >> gs.lp);  // class row of the tile's first row
        const int beta = gs.first_box + lane, cls = gs.cls(beta);
        const CUtensorMap *maps = gs.op == 0 ? cm.a : cm.b;
        if ((live >> cls) & 1u)
            tma_load_2d(slot + uint32_t(lane) * box_bytes, &maps[cls], xb + 64 * gs.seg(beta),
                        yb + (gs.blk(beta) << gs.lh), bar);
    }
}

// Issues the TMA copies of one group from the calling lane: `bi` is the box
// index within the group; box 0's lane announces the group's byte count on
// `bar` first (ordered before the other boxes' issue by the caller's warp
// convergence through __syncwarp). Boxes of classes without rows are skipped.
template <typename Maps>
__device__ __forceinline__ void issue_class_group_lanes(const Params &p, const Maps &cm,
                                                        const GroupShape &gs, int64_t k0, uint32_t slot,
                                                        uint32_t bar, int bi) {
    const uint32_t live = gs.op == 0 ? p.cls_live[0] : p.cls_live[1];
    const int nbox = GROUP_LINES >> gs.lh;
    const uint32_t box_bytes = uint32_t(LINE_PITCH) << gs.lh;
    if (bi == 0) {
        uint32_t boxes = 0;
        for (int i = 0; i < nbox; ++i) boxes += (live >> gs.cls(gs.first_box + i)) & 1u;
        mbar_arrive_expect_tx(bar, boxes * box_bytes);
    }
    __syncwarp();
    if (bi < nbox) {
        const int32_t xb = int32_t(gs.mn_major ? gs.mn0 : k0);
        const int32_t yb = int32_t((gs.mn_major ? k0 : gs.mn0) >> gs.lp);
        const int beta = gs.first_box + bi, cls = gs.cls(beta);
        const CUtensorMap *maps = gs.op == 0 ? cm.a : cm.b;
        if ((live >> cls) & 1u)
            tma_load_2d(slot + uint32_t(bi) * box_bytes, &maps[cls], xb + 64 * gs.seg(beta),
                        yb + (gs.blk(beta) << gs.lh), bar);
    }
}

// Bytes [m, m + 16) of the 32-byte window w[0..7] (m even, 0..14): select
// by whole words (m / 4), then shift by a half word when m % 4 == 2.
__device__ __forceinline__ void window16(const uint32_t (&w)[8], uint32_t m, uint32_t (&o)[4]) {
    uint32_t x[6], y[5];
#pragma unroll
    for (int t = 0; t < 6; ++t) x[t] = (m & 8u) ? w[t + 2] : w[t];
#pragma unroll
    for (int t = 0; t < 5; ++t) y[t] = (m & 4u) ? x[t + 1] : x[t];
    const uint32_t sel = (m & 2u) ? 0x5432u : 0x3210u;
#pragma unroll
    for (int t = 0; t < 4; ++t) o[t] = __byte_perm(y[t], y[t + 1], sel);
}

// All lanes: shift the group's 64 staged lines into the operand stage at
// `dst`. In step k (0..15) lane l moves 16 bytes: unit l % 8 of staged line
// 4k + l / 8. The four lines of a step lie in one box (h >= 8), hence share a
// class and its offset m. Staging reads of four steps are issued first.
__device__ __forceinline__ void place_class_group(const Params &p, const GroupShape &gs, uint32_t slot,
                                                  uint32_t dst, int lane) {
    const uint32_t mis = gs.op == 0 ? p.cls_mis[0] : p.cls_mis[1];
    const uint32_t live = gs.op == 0 ? p.cls_live[0] : p.cls_live[1];
    const uint32_t u = uint32_t(lane) & 7u, r4 = uint32_t(lane) >> 3;
    const uint32_t seg_bytes = gs.mn_major ? uint32_t(MN_CHUNK_BYTES) : 0u;
    const uint32_t hmask = (1u << gs.lh) - 1u;
#pragma unroll 1
    for (int k0 = 0; k0 < GROUP_LINES / 4; k0 += 4) {
        uint32_t w[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t src = slot + (uint32_t(4 * (k0 + j)) + r4) * LINE_PITCH + 16u * u;
            ld_shared_v4(src, w[j][0], w[j][1], w[j][2], w[j][3]);
            ld_shared_v4(src + 16u, w[j][4], w[j][5], w[j][6], w[j][7]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t l = uint32_t(4 * (k0 + j)) + r4;
            const int beta = gs.first_box + int(l >> gs.lh), cls = gs.cls(beta);
            const uint32_t m = (mis >> (4 * cls)) & 15u;  // where the lines start in their window
            uint32_t o[4];
            window16(w[j], m, o);
            if (!((live >> cls) & 1u)) o[0] = o[1] = o[2] = o[3] = 0u;
            const uint32_t rho = uint32_t(cls) + (((uint32_t(gs.blk(beta)) << gs.lh) + (l & hmask)) << gs.lp);
            st_shared_v4(dst + uint32_t(gs.seg(beta)) * seg_bytes + rho * 128u + ((u ^ (rho & 7u)) << 4), o[0],
                         o[1], o[2], o[3]);
        }
    }
}

// ------------------------------------------------------------------ epilogue
// Drains one accumulator of this CTA to C. Two warps share each TMEM lane
// quarter (tile rows row0 .. row0+31): warp half h takes accumulator columns
// [128h, 128h + 128). The TMEM load of the next 32 columns is issued before the
// current ones are stored, so its latency overlaps the store work.
// TMA store: 128-byte-swizzled staging (one buffer per warp) + bulk tensor
// store, which clips the M/N edges. Otherwise: transpose through the staging
// buffer so each store instruction writes 32 consecutive floats of one row.
// `drained()` runs on every lane right after the warp's last TMEM load.
// The chunks are stored as fast as they come: spacing them out over the next
// unit's main loop by a fixed sleep per k-block measured the same (device-timed
// on GB300, 16384^2 x K for K = 512 ... 4096 and 8192^2 x 4096, within 0.7 %
// both in short loops and under the power limit), so nothing here depends on
// the clock.
constexpr int EPI_CHUNKS32 = BN / EPI_COLS;  // 8 fp32 chunks of 32 columns per accumulator row block
constexpr int EPI_CHUNKS16 = BN / 64;        // 4 chunks of 64 16-bit values
// Work units shorter than this many K-blocks split each row block's chunks
// between its two epilogue warps (the drain is then on the critical path);
// longer ones leave the second warp idle, which measured faster (less
// interference with the MMA issue and the operand traffic): 16384^2 x K on
// CTA pairs, two warps vs one per row block: K = 128 184 vs 202 us, K = 512
// 258 vs 274 us, K = 1024 401 vs 380 us.
constexpr int EPI_SPLIT_MAX_KB = 12;
static_assert(EPI_WARPS == 8, "two epilogue warps per TMEM lane quarter");

// Chunk range [c0, c0 + n) of the calling warp (n even, or 0). A program's
// last unit is always split: no MMA runs beside it any more.
__device__ __forceinline__ void epilogue_chunks(int32_t unit_kblocks, bool last_unit, int half, int chunks,
                                                int &c0, int &n) {
    if (unit_kblocks < EPI_SPLIT_MAX_KB || last_unit) {
        n = chunks / 2;
        c0 = half * n;
    } else {
        n = half == 0 ? chunks : 0;
        c0 = 0;
    }
}

// Where a partial tile of a split tail unit goes: the scratch map, the row of
// the scratch that holds this warp's first tile row, and the tile's first
// column of C (scratch columns are tile-local).
struct TailStore {
    const CUtensorMap *map;
    int32_t row;
    int64_t col_base;
};

// Stores one 32 x 32 fp32 chunk (this lane's row, 32 columns from col0).
template <bool kTmaStore>
__device__ __forceinline__ void store_chunk32(uint32_t (&v)[32], int64_t row0, int64_t col0, const Params &p,
                                              const CUtensorMap *tmC, uint32_t stg, int lane, int32_t split,
                                              const TailStore *ts = nullptr) {
    if (p.alpha != 1.0f && ts == nullptr) {  // a split tail's partials are scaled once summed
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(p.alpha * __uint_as_float(v[i]));
    }
    if (kTmaStore) {
        if (lane == 0) bulk_wait_group_read<0>();  // the buffer's previous store has read it
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u)
            st_shared_v4(stg + swz128(lane, u), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (ts != nullptr) {  // split tail: partial tile -> its scratch slot (always in bounds)
                if (row0 < p.M && col0 < p.N)
                    tma_store_2d_hint(ts->map, stg, int32_t(col0 - ts->col_base), ts->row, l2_policy_evict_normal());
            } else if (row0 < p.M && col0 < p.N) {
                if (p.splits > 1)  // partial tile -> workspace slice `split`, read once by the reduction
                    tma_store_3d_hint(tmC, stg, int32_t(col0), int32_t(row0), split, l2_policy_evict_normal());
                else if (p.l2_mode & 1u)  // C is never read again: do not keep it in L2
                    tma_store_2d_hint(tmC, stg, int32_t(col0), int32_t(row0), l2_policy_evict_first());
                else
                    tma_store_2d(tmC, stg, int32_t(col0), int32_t(row0));
            }
            bulk_commit_group();
        }
    } else {
        __syncwarp();  // every lane has read the buffer's previous contents
#pragma unroll
        for (int u = 0; u < 8; ++u)
            st_shared_v4(stg + swz128(lane, u), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        __syncwarp();
        // all 32 staging reads first, so that no read waits behind a store
#pragma unroll
        for (int r = 0; r < 32; ++r) v[r] = ld_shared_b32(stg + swz128(r, lane >> 2) + (lane & 3) * 4);
        const int64_t col = col0 + lane, rows = p.M - row0;
        if (col < p.N) {
            float *dst = p.C + row0 * p.scm + col;
#pragma unroll
            for (int r = 0; r < 32; ++r)
                if (r < rows && G16_CHECK(row0 + r >= 0 && row0 + r < p.M && col >= 0))
                    dst[r * p.scm] = __uint_as_float(v[r]);
        }
    }
}

template <bool kTmaStore, typename Drained>
__device__ __forceinline__ void epilogue_tile(uint32_t t_row, int64_t row0, int64_t col_base, int c0, int n,
                                              const Params &p, const CUtensorMap *tmC, uint32_t stg, int lane,
                                              Drained drained, int32_t split = 0,
                                              const TailStore *ts = nullptr) {
    if (n == 0) {
        drained();
        return;
    }
    uint32_t va[32], vb[32];
    tmem_ld_32x32b_x32(t_row + c0 * EPI_COLS, va);
#pragma unroll 1
    for (int c = c0; c < c0 + n; c += 2) {
        tmem_ld_wait();
        tmem_ld_32x32b_x32(t_row + (c + 1) * EPI_COLS, vb);
        store_chunk32<kTmaStore>(va, row0, col_base + c * EPI_COLS, p, tmC, stg, lane, split, ts);
        tmem_ld_wait();
        const bool more = c + 2 < c0 + n;
        if (more)
            tmem_ld_32x32b_x32(t_row + (c + 2) * EPI_COLS, va);
        else
            drained();
        store_chunk32<kTmaStore>(vb, row0, col_base + (c + 1) * EPI_COLS, p, tmC, stg, lane, split, ts);
    }
}

// ------------------------------------------------------------------ C stored per row class
// fp32 C whose rows do not all start on a 16-byte boundary (and whose base and
// row stride are multiples of 4 bytes): row i starts m_i floats (0..3) into a
// granule, and rows with the same i mod P (P = 1, 2 or 4, from the row stride)
// share m. Class q (rows q, q + P, ...) has a tensor map whose rows begin at the
// granule boundary below each row start, so map column x is C column x - m_q;
// its inner extent ends on a granule at or before column N, so no store reaches
// past a row. A warp's 32 rows hold 32 / P rows of each class; lane l's row goes
// to staging row (l % P) * (32 / P) + l / P, so that each class is one box.
// Per warp column range [col0, end):
//  * first chunk: the box at map column col0 + 4 (m > 0) holds C columns
//    [col0 + d, col0 + d + 32), d = 4 - m: this chunk from column d on and the
//    next chunk's first d values; columns [col0, col0 + d) go out as plain
//    stores (m = 0: the box at col0, nothing plain);
//  * chunk k > 0: the box at map column col0_k holds C columns [col0_k - m,
//    col0_k - m + 32): the last m values of chunk k - 1, carried in registers,
//    then the first 32 - m of chunk k. The one granule it shares with the first
//    chunk's box is written twice with the same values;
//  * columns [end - m, end), the carry after the last chunk: plain stores.
// Units that reach C's last column use the plain path throughout.

// This lane's row offset inside its 16-byte granule, in floats.
__device__ __forceinline__ uint32_t row_misalignment(const Params &p, int64_t row) {
    return (uint32_t(reinterpret_cast<uintptr_t>(p.C) >> 2) + uint32_t(uint64_t(row) * uint64_t(p.scm))) & 3u;
}

// o[t] = e(t + s) for t = 0..31, s = 0..3, e(i) a run of 35 values: two select
// steps on the bits of s (whole registers only; s is uniform per lane).
template <typename E>
__device__ __forceinline__ void shift_run(E e, uint32_t s, uint32_t (&o)[32]) {
    const bool b1 = (s & 1u) != 0, b2 = (s & 2u) != 0;
    uint32_t y[34];  // y[i] = e(i + (s & 1)), i = 0 .. 33
#pragma unroll
    for (int i = 0; i < 34; ++i) y[i] = b1 ? e(i + 1) : e(i);
#pragma unroll
    for (int t = 0; t < 32; ++t) o[t] = b2 ? y[t + 2] : y[t];
}

template <typename Drained>
__device__ __forceinline__ void epilogue_tile_class(uint32_t t_row, int64_t row0, int64_t col_base, int c0, int n,
                                                    const Params &p, const CUtensorMap *cmaps, uint32_t stg,
                                                    int lane, Drained drained) {
    if (n == 0) {
        drained();
        return;
    }
    const uint32_t P = p.c_classes;
    const uint32_t rpc = 32u / P;  // rows of each class in the warp's 32
    const uint32_t m = row_misalignment(p, row0 + lane);
    const uint32_t srow = (uint32_t(lane) % P) * rpc + uint32_t(lane) / P;
    const bool row_ok = row0 + lane < p.M;
    float *row_ptr = p.C + (row0 + lane) * p.scm;
    uint32_t carry[3] = {0u, 0u, 0u};
    auto scale = [&](uint32_t x) { return __float_as_uint(p.alpha * __uint_as_float(x)); };
    // stage o (this lane's row of the boxes), then one box store per class
    auto put = [&](const uint32_t (&o)[32], int32_t x) {
        if (lane < int(P)) bulk_wait_group_read<0>();  // the buffer's previous stores have read it
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u)
            st_shared_v4(stg + swz128(srow, u), o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane < int(P)) {  // lane q's row is of class q
            tma_store_2d_hint(&cmaps[lane], stg + uint32_t(lane) * rpc * 128u, x, int32_t(row0 / P),
                              l2_policy_evict_first());
            bulk_commit_group();
        }
    };
    auto emit = [&](uint32_t (&v)[32], int c, const uint32_t (*next)[32]) {
        const int64_t col0 = col_base + int64_t(c) * EPI_COLS;
        if (p.alpha != 1.0f) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = scale(v[i]);
        }
        uint32_t o[32];
        if (next != nullptr) {  // the range's first chunk
            const uint32_t d = (4u - m) & 3u;
            uint32_t nx[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) nx[i] = p.alpha != 1.0f ? scale((*next)[i]) : (*next)[i];
#pragma unroll
            for (int i = 0; i < 3; ++i)
                if (row_ok && uint32_t(i) < d && G16_CHECK(col0 + i < p.N)) row_ptr[col0 + i] = __uint_as_float(v[i]);
            shift_run([&](int i) -> uint32_t { return i < 32 ? v[i] : nx[i - 32]; }, d, o);
            put(o, int32_t(col0) + (m != 0 ? 4 : 0));
        } else {
            shift_run([&](int i) -> uint32_t { return i < 3 ? carry[i] : v[i - 3]; }, 3u - m, o);
            put(o, int32_t(col0));
        }
        carry[0] = v[29];
        carry[1] = v[30];
        carry[2] = v[31];
    };
    uint32_t va[32], vb[32];
    tmem_ld_32x32b_x32(t_row + c0 * EPI_COLS, va);
#pragma unroll 1
    for (int c = c0; c < c0 + n; c += 2) {
        tmem_ld_wait();
        tmem_ld_32x32b_x32(t_row + (c + 1) * EPI_COLS, vb);
        if (c == c0) {
            tmem_ld_wait();  // the first chunk's box takes the next chunk's first values
            emit(va, c, &vb);
        } else {
            emit(va, c, nullptr);
        }
        tmem_ld_wait();
        if (c + 2 < c0 + n)
            tmem_ld_32x32b_x32(t_row + (c + 2) * EPI_COLS, va);
        else
            drained();
        emit(vb, c + 1, nullptr);
    }
    // the carry of the last chunk: columns [end - m, end)
    const int64_t end = col_base + int64_t(c0 + n) * EPI_COLS;
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (row_ok && uint32_t(3 - i) <= m && G16_CHECK(end - 3 + i < p.N))
            row_ptr[end - 3 + i] = __uint_as_float(carry[i]);
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

__device__ __forceinline__ void pack_half_chunk(const uint32_t (&v)[32], uint32_t *w, float alpha,
                                                uint32_t dtype) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        w[i] = pack_16x2(alpha * __uint_as_float(v[2 * i]), alpha * __uint_as_float(v[2 * i + 1]), dtype);
}

// Stores one chunk of 32 rows x 64 16-bit values (one 128-byte staging row per
// lane; the TMA box is 64 x 32 elements).
template <bool kTmaStore>
__device__ __forceinline__ void store_chunk16(uint32_t (&w)[32], int64_t row0, int64_t col0, const Params &p,
                                              const CUtensorMap *tmC, uint32_t stg, int lane) {
    if (kTmaStore) {
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u)
            st_shared_v4(stg + swz128(lane, u), w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (row0 < p.M && col0 < p.N && G16_CHECK((col0 & 7) == 0))
                tma_store_2d_hint(tmC, stg, int32_t(col0), int32_t(row0), l2_policy_evict_first());
            bulk_commit_group();
        }
    } else {
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u)
            st_shared_v4(stg + swz128(lane, u), w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 32; ++r) w[r] = ld_shared_b32(stg + swz128(r, lane >> 2) + (lane & 3) * 4);
        const int64_t col = col0 + 2 * lane, rows = p.M - row0;  // this lane: columns col, col + 1
        if (col < p.N) {
            uint16_t *dst = reinterpret_cast<uint16_t *>(p.C) + row0 * p.scm + col;
            const bool both = col + 1 < p.N;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                if (r < rows && G16_CHECK(row0 + r >= 0 && row0 + r < p.M && col >= 0)) {
                    dst[r * p.scm] = uint16_t(w[r] & 0xffffu);
                    if (both) dst[r * p.scm + 1] = uint16_t(w[r] >> 16);
                }
            }
        }
    }
}

// 16-bit C: like epilogue_tile, with chunks of 64 columns (two 32-column TMEM
// loads), scaled by alpha and rounded.
template <bool kTmaStore, typename Drained>
__device__ __forceinline__ void epilogue_tile16(uint32_t t_row, int64_t row0, int64_t col_base, int c0, int n,
                                                const Params &p, const CUtensorMap *tmC, uint32_t stg,
                                                int lane, Drained drained) {
    if (n == 0) {
        drained();
        return;
    }
    const float alpha = p.alpha;
    uint32_t va[32], vb[32], w[32];
    tmem_ld_32x32b_x32(t_row + c0 * 64, va);
#pragma unroll 1
    for (int c = c0; c < c0 + n; ++c) {
        tmem_ld_wait();
        tmem_ld_32x32b_x32(t_row + c * 64 + 32, vb);
        pack_half_chunk(va, w, alpha, p.out_dtype);
        tmem_ld_wait();
        const bool more = c + 1 < c0 + n;
        if (more)
            tmem_ld_32x32b_x32(t_row + (c + 1) * 64, va);
        else
            drained();
        pack_half_chunk(vb, w + 16, alpha, p.out_dtype);
        store_chunk16<kTmaStore>(w, row0, col_base + c * 64, p, tmC, stg, lane);
    }
}

// A unit of the split tail (u >= tail_first): its tile, k-block range and
// scratch slot; other units keep what the caller decoded, with slot -1.
__device__ __forceinline__ void tail_unit(const Params &p, int32_t u, int32_t &tile, int32_t &kb0,
                                          int32_t &kb1, int32_t &slot) {
    slot = -1;
    if (u < p.tail_first) return;
    const int32_t v = u - p.tail_first;
    const int32_t j = v / p.tail_tiles;
    tile = p.tail_first + (v - j * p.tail_tiles);
    kb0 = j * p.tail_kps;
    kb1 = min(p.num_kb, kb0 + p.tail_kps);
    slot = v;
}

// ------------------------------------------------------------------ the kernel
template <bool kTmaLoad, bool kTmaStore>
__global__ void __launch_bounds__(cta_threads(kTmaLoad), 1)
    gemm_f16_persistent(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const Params p,
                        const __grid_constant__ typename ClassMapsFor<kTmaLoad>::type cm) {
    constexpr int LOAD_WARPS = load_warps(kTmaLoad);
    constexpr int MMA_WARP = LOAD_WARPS;
    constexpr int EPI_WARP0 = LOAD_WARPS + 1;
    using Lay = Layout<kTmaLoad>;
    constexpr int NST = Lay::stages;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);

    const uint32_t sA = base + Lay::off_a;
    const uint32_t sB = base + Lay::off_b;
    const uint32_t bar0 = base + Lay::off_bar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (NST + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * NST + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * NST + NUM_ACC + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * NST + 2 * NUM_ACC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay::off_tmem_slot);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(full_bar(s), kTmaLoad ? 1 : LOAD_WARPS * 32);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EPI_WARPS * 32);
        }
        mbar_init(drain_bar, 1);
        for (int q = 0; q < Lay::copy_slots; ++q) mbar_init(bar0 + 8u * (Lay::copy_bar0 + q), 1);
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
    if constexpr (!kTmaLoad) {
        if (warp == 0 && lane < 2 * MAX_CLASSES) {  // the maps of classes that hold rows
            const int op = lane / MAX_CLASSES, cls = lane % MAX_CLASSES;
            if ((p.cls_live[op] >> cls) & 1u) prefetch_tensormap(op == 0 ? &cm.a[cls] : &cm.b[cls]);
        }
    }
    if (kTmaStore && warp == EPI_WARP0 && lane == 0) prefetch_tensormap(&tmC);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The set-up above may overlap the end of the previous kernel on the
    // stream; nothing below touches global memory before that kernel is done.
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;

    const int32_t grid = gridDim.x;
    const int32_t num_kb = p.num_kb;

    if (warp < LOAD_WARPS) {
        // ============================================================ producer
        if constexpr (kTmaLoad) {
            // The whole warp walks the stages; lane 0 arms the barrier and each
            // of the stage's copies (A: 1 box or 2 chunks, B: 1 box or 4 chunks)
            // is issued by its own lane, as in the CTA-pair kernel.
            uint32_t stage = 0, phase = 0;
            uint32_t issued = 0;
            bool ok = true;
            int32_t it = 0;
            const int na = p.a_mn ? BM / MN_CHUNK : 1;
            const int nb = p.b_mn ? BN / MN_CHUNK : 1;
            for (int32_t tile = blockIdx.x; ok && tile < p.num_tiles; tile += grid, ++it) {
                int32_t tm, tn;
                tile_coords(tile, p.sched, tm, tn);
                if (!p.cross_tile && it > 0) {
                    const int32_t j = it - 1;  // wait until tile j's accumulator is drained
                    if (!__all_sync(0xffffffffu, mbar_wait(tempty_bar(j & 1), (j >> 1) & 1, p.wait))) {
                        ok = false;
                        break;
                    }
                }
                const int32_t m0 = tm * BM, n0 = tn * BN;
                for (int32_t kb = 0; kb < num_kb; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait(empty_bar(stage), phase ^ 1u, p.wait))) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(stage);
                    if (lane == 0) mbar_arrive_expect_tx(fb, A_STAGE_BYTES + B_STAGE_BYTES);
                    const int32_t k0 = kb * BK;
                    if (lane < na + nb) {  // lane: copy `lane` of A, or copy `lane - na` of B
                        const bool is_a = lane < na;
                        const int c = is_a ? lane : lane - na;
                        const CUtensorMap *map = is_a ? &tmA : &tmB;
                        const uint32_t dst =
                            (is_a ? sA + stage * A_STAGE_BYTES : sB + stage * B_STAGE_BYTES) + uint32_t(c) * MN_CHUNK_BYTES;
                        const bool mn_major = (is_a ? p.a_mn : p.b_mn) != 0;
                        const int32_t mn = (is_a ? m0 : n0) + c * MN_CHUNK;
                        tma_load_2d(dst, map, mn_major ? mn : k0, mn_major ? k0 : mn, fb);
                    }
                    ++issued;
                    if (++stage == NST) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok && lane == 0) {
                // Let the copies this warp started land before the CTA exits.
                const uint32_t n = issued < NST ? issued : NST;
                for (uint32_t q = issued - n; q < issued; ++q)
                    mbar_wait_slow(full_bar(q % NST), (q / NST) & 1u, cleanup_wait(p.wait), false);
            }
            __syncwarp();
        } else {
            // Per-warp pipeline over this warp's copy groups: lane 0 keeps up to
            // COPY_DEPTH groups of TMA copies in flight into the warp's staging
            // ring while the warp places the oldest one into the stage. With
            // cross-tile off, copies stop at each tile boundary until the
            // previous tile's accumulator has been drained.
            const uint32_t ring = base + Lay::off_copy + uint32_t(warp) * (COPY_DEPTH * GROUP_BYTES);
            auto copy_bar = [&](uint32_t q) { return bar0 + 8u * (Lay::copy_bar0 + warp * COPY_DEPTH + q); };
            LineCursor iss, fix;
            iss.start(blockIdx.x, p);
            fix = iss;
            uint32_t issued = 0, placed = 0;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            while (fix.valid(p)) {
                if (fix.g == 0 && fix.kb == 0 && !p.cross_tile && fix.it > 0) {
                    const int32_t j = fix.it - 1;
                    if (!mbar_wait(tempty_bar(j & 1), (j >> 1) & 1, p.wait)) { ok = false; break; }
                }
                while (issued - placed < COPY_DEPTH && iss.valid(p) && (p.cross_tile || iss.it == fix.it)) {
                    const uint32_t q = issued % COPY_DEPTH;
                    const int gamma = warp + PRED_LOAD_WARPS * iss.g;
                    const int op = gamma < A_GROUPS ? 0 : 1;
                    const GroupShape gs = group_shape(p, op, op == 0 ? gamma : gamma - A_GROUPS, op == 0 ? 7 : 8,
                                                      op == 0 ? iss.m0 : iss.n0);
                    issue_class_group(p, cm, gs, int64_t(iss.kb) * BK, ring + q * GROUP_BYTES, copy_bar(q), lane);
                    iss.next(p, grid);
                    ++issued;
                }
                if (fix.g == 0 && !mbar_wait(empty_bar(stage), phase ^ 1u, p.wait)) { ok = false; break; }
                const uint32_t q = placed % COPY_DEPTH;
                if (!mbar_wait(copy_bar(q), (placed / COPY_DEPTH) & 1u, p.wait)) { ok = false; break; }
                const int gamma = warp + PRED_LOAD_WARPS * fix.g;
                const int op = gamma < A_GROUPS ? 0 : 1;
                const GroupShape gs = group_shape(p, op, op == 0 ? gamma : gamma - A_GROUPS, op == 0 ? 7 : 8,
                                                  op == 0 ? fix.m0 : fix.n0);
                const uint32_t dst = gs.op == 0 ? sA + stage * A_STAGE_BYTES : sB + stage * B_STAGE_BYTES;
                place_class_group(p, gs, ring + q * GROUP_BYTES, dst, lane);
                __syncwarp();  // slot q is free for the next copies into it
                if (fix.g == WARP_GROUPS - 1) {
                    fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
                    mbar_arrive(full_bar(stage));
                    if (++stage == NST) { stage = 0; phase ^= 1u; }
                }
                fix.next(p, grid);
                ++placed;
            }
            if (!ok) {
                // Let the copies this warp started land before the CTA exits.
                for (uint32_t q = placed; q < issued; ++q)
                    mbar_wait_slow(copy_bar(q % COPY_DEPTH), (q / COPY_DEPTH) & 1u, cleanup_wait(p.wait),
                                   false);
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
                if (++stage == NST) { stage = 0; phase ^= 1u; }
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
        const int half = ew / 4;  // which of the two warps of its TMEM lane quarter
        const uint32_t stg = base + Lay::off_epi + uint32_t(ew) * (EPI_BUFS * EPI_BUF_BYTES);
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
            const int64_t col_base = int64_t(tn) * BN;
            const bool last = tile + grid >= p.num_tiles;
            int c0, n;
            if (p.out_dtype == 0) {
                epilogue_chunks(num_kb, last, half, EPI_CHUNKS32, c0, n);
                epilogue_tile<kTmaStore>(t_row, row0, col_base, c0, n, p, &tmC, stg, lane, release);
            } else {
                epilogue_chunks(num_kb, last, half, EPI_CHUNKS16, c0, n);
                epilogue_tile16<kTmaStore>(t_row, row0, col_base, c0, n, p, &tmC, stg, lane, release);
            }
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

#ifdef GEMM_DEBUG
// Debug-check self-test: one check that fails and guards no access, so that
// the reporting path is exercised without any faulty access.
__global__ void check_selftest_kernel() {
    if (threadIdx.x == 0) (void)G16_CHECK(false);
}
#endif

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
    griddep_wait();  // the partial slices are the previous kernel's output
    griddep_launch_dependents();
    const int64_t nq = (N + 3) / 4;
    const int64_t total = M * nq;
    const int64_t slice = M * ldw;
    float *C = static_cast<float *>(Cv);
    const bool vec_c = (scm % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0);
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = e / nq, j = (e - i * nq) * 4;
        if (!G16_CHECK(i < M && j < N && j + 4 <= ldw)) continue;
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

// Split tail: C over each tail tile = the sum, in slice order 0, 1, ..., S-1,
// of its S fp32 partial tiles in the scratch (slot j * tail_tiles + i holds
// slice j of tail tile i; TILE x TILE floats each, row-major), times alpha,
// rounded to C's type. Fixed order: the result does not depend on scheduling.
// Four consecutive columns per thread.
template <int TILE>
__global__ void tail_reduce_kernel(const float *__restrict__ W, void *__restrict__ Cv, int64_t M, int64_t N,
                                   int64_t scm, Sched sched, int32_t first, int32_t tiles, int32_t S,
                                   uint32_t out_dtype, float alpha) {
    griddep_wait();  // the partial tiles are the previous kernel's output
    griddep_launch_dependents();
    constexpr int QUADS = TILE * TILE / 4;
    const int64_t total = int64_t(tiles) * QUADS;
    float *C = static_cast<float *>(Cv);
    const bool vec_c = (scm % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0);
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int32_t i = int32_t(e / QUADS);
        const int32_t q = int32_t(e - int64_t(i) * QUADS);
        const int32_t r = q / (TILE / 4), c = (q - r * (TILE / 4)) * 4;
        int32_t tm, tn;
        tile_coords(first + i, sched, tm, tn);
        const int64_t row = int64_t(tm) * TILE + r, col = int64_t(tn) * TILE + c;
        if (row >= M || col >= N) continue;
        const float *w = W + (int64_t(i) * TILE + r) * TILE + c;
        const int64_t slot = int64_t(tiles) * TILE * TILE;
        float4 acc = *reinterpret_cast<const float4 *>(w);
        for (int32_t s = 1; s < S; ++s) {
            const float4 v = *reinterpret_cast<const float4 *>(w + s * slot);
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
        if (!G16_CHECK(row >= 0 && col >= 0)) continue;
        if (out_dtype != 0) {
            uint16_t *c16 = static_cast<uint16_t *>(Cv) + row * scm + col;
            const uint32_t w01 = pack_16x2(acc.x, acc.y, out_dtype);
            const uint32_t w23 = pack_16x2(acc.z, acc.w, out_dtype);
            c16[0] = uint16_t(w01 & 0xffffu);
            if (col + 1 < N) c16[1] = uint16_t(w01 >> 16);
            if (col + 2 < N) c16[2] = uint16_t(w23 & 0xffffu);
            if (col + 3 < N) c16[3] = uint16_t(w23 >> 16);
            continue;
        }
        float *cp = C + row * scm + col;
        if (vec_c && col + 3 < N) {
            *reinterpret_cast<float4 *>(cp) = acc;
        } else {
            cp[0] = acc.x;
            if (col + 1 < N) cp[1] = acc.y;
            if (col + 2 < N) cp[2] = acc.z;
            if (col + 3 < N) cp[3] = acc.w;
        }
    }
}

// ------------------------------------------------------------------ operand packing
// One operand as `rows` rows of `inner` contiguous fp16 elements: element
// (r, i) of the source at src[r * ld_src + i] (any 2-byte-aligned base, any
// ld_src >= inner), of the copy at dst[r * ld_dst + i] (dst 128-byte aligned,
// ld_dst a multiple of 64), so that every 64-element K-block row of the copy is
// one whole 128-byte line.
struct PackJob {
    const uint16_t *src;
    uint16_t *dst;
    int64_t rows, inner, ld_src, ld_dst;
    int64_t gpr;       // 16-byte granules of a copied row: cdiv(inner, 8)
    int64_t granules;  // rows * gpr; 0 when the operand is not copied
};

// Copies A's and then B's granules, one 16-byte granule of the copy per thread
// and step: the (one or two) aligned 16-byte source granules that hold its
// elements are loaded and shifted into place; elements past `inner` are written
// as zero. A source granule is read only when it holds an element of the row.
__global__ void pack_rows_kernel(PackJob a, PackJob b) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t total = a.granules + b.granules;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const bool second = e >= a.granules;
        const PackJob &J = second ? b : a;
        const int64_t f = second ? e - a.granules : e;
        const int64_t r = f / J.gpr, j = f - r * J.gpr;
        const int64_t i0 = 8 * j;
        if (!G16_CHECK(r < J.rows && i0 < J.inner)) continue;
        const int64_t left = J.inner - i0;
        const uint32_t cnt = left < 8 ? uint32_t(left) : 8u;  // elements of this granule in the row
        const uintptr_t s = reinterpret_cast<uintptr_t>(J.src + r * J.ld_src + i0);
        const uintptr_t g0 = s & ~uintptr_t(15);
        const uint32_t m = uint32_t(s - g0);  // even: fp16 elements
        uint32_t w[8];
        const uint4 lo = __ldg(reinterpret_cast<const uint4 *>(g0));
        w[0] = lo.x, w[1] = lo.y, w[2] = lo.z, w[3] = lo.w;
        if (m + 2 * cnt > 16) {  // the last elements lie in the next granule
            const uint4 hi = __ldg(reinterpret_cast<const uint4 *>(g0 + 16));
            w[4] = hi.x, w[5] = hi.y, w[6] = hi.z, w[7] = hi.w;
        } else {
            w[4] = w[5] = w[6] = w[7] = 0u;
        }
        uint32_t o[4];
        window16(w, m, o);
        if (cnt < 8) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (uint32_t(2 * t) >= cnt) o[t] = 0u;
                else if (uint32_t(2 * t + 1) >= cnt) o[t] &= 0xffffu;
            }
        }
        uint4 out;
        out.x = o[0], out.y = o[1], out.z = o[2], out.w = o[3];
        *reinterpret_cast<uint4 *>(J.dst + r * J.ld_dst + i0) = out;
    }
}

// K == 0: C := 0 (the accumulator starts at zero and no K step adds to it).
__global__ void zero_c_kernel(void *C, int64_t M, int64_t N, int64_t scm, int32_t esize) {
    const int64_t total = M * N;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e - i * N;
        if (!G16_CHECK(i < M && j < N)) continue;
        if (esize == 4)
            static_cast<float *>(C)[i * scm + j] = 0.0f;
        else
            static_cast<uint16_t *>(C)[i * scm + j] = 0;
    }
}

}  // namespace g16
