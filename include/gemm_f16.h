/*
 * gemm_f16 — persistent FP16 GEMM for GB300 (sm_103a), C ABI.
 *
 *   C[M,N] = A[M,K] @ B[K,N]   fp16 inputs, fp32 accumulation, fp32 output.
 *
 * The operation and its scheduling follow four pages:
 *  [persistent] "(1/n) Triton matmul 커널 탐험 - persistent kernel은 그 자체로
 *               빠르지 않다": sections "naive tiled matmul" (masked tile GEMM,
 *               FP32 accumulator from zero, C stored, never read),
 *               "naive persistent matmul" (grid = min(#SMs, #tiles); program
 *               pid visits tile_id = pid, pid + grid, ...).
 *  [swizzle]    "(2/n) Triton matmul 커널 탐험 - grouped ordering(CTA swizzle)도
 *               늘 빠르게 만들지는 않는다": section "구현" (grouped tile order).
 *  [flatten]    "(3/n) Triton matmul 커널 탐험 - cross tile pipelining 적용":
 *               one flattened (tile, k) loop so the next tile's loads overlap
 *               the current tile's store.
 *  [roofline]   "4주차 정리: Roofline과 Tiling": section 5 (FLOPs = 2MNK).
 *
 * Conventions shared by every entry point:
 *  - All pointers to matrices are DEVICE pointers owned by the caller. The
 *    library allocates no device memory per call; its only device state is a
 *    few status words in the library image (one copy per device).
 *  - Strides are in ELEMENTS, as in the pages' kernels
 *    (stride_am, stride_ak, stride_bk, stride_bn, stride_cm, stride_cn):
 *    A(i,k) = A[i*stride_am + k*stride_ak], B(k,j) = B[k*stride_bk + j*stride_bn],
 *    C(i,j) = C[i*stride_cm + j*stride_cn].
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and the
 *    call returns without waiting. Launch errors are returned; errors raised
 *    while the kernel runs (a bounded wait that ran out) are reported by
 *    gemm_f16_sync_status().
 *  - Each kernel of a call is launched with programmatic stream serialization
 *    allowed (programmatic dependent launch): its CTAs may be scheduled while
 *    the kernel before it on the stream is finishing, and set themselves up
 *    (barriers, tensor memory), but touch no global memory until that kernel
 *    has completed and its writes are visible. Each kernel also lets the next
 *    kernel on the stream be scheduled early; a kernel that is launched with
 *    the same attribute must itself wait (griddepcontrol.wait) before it
 *    reads this call's output, as one launched without it always does.
 *    Ordering on the stream is that of plain launches.
 *  - Every entry point validates its arguments before touching the GPU and
 *    returns GEMM_ERR_INVALID_ARG / GEMM_ERR_UNSUPPORTED without side effects.
 *  - Thread safety: calls from several host threads are allowed; calls that
 *    overlap on the GPU and write the same C race (the caller's problem).
 */
#ifndef GEMM_F16_H
#define GEMM_F16_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
struct CUstream_st;
typedef struct CUstream_st *gemm_stream_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad stride/flag/G */
    GEMM_ERR_UNSUPPORTED = 2, /* layout the kernels do not take (see gemm_f16) */
    GEMM_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed            */
    GEMM_ERR_TIMEOUT = 4,     /* a bounded device wait ran out (kernel gave up) */
    GEMM_ERR_CHECK = 5        /* debug build (GEMM_DEBUG) only: a device-side bounds or
                                 alignment check failed; the access was skipped and the
                                 source line is printed by gemm_f16_sync_status */
} gemm_status_t;

/* schedule_flags bits */
#define GEMM_SCHED_GROUPED 0x1u    /* grouped ("CTA swizzle") tile order; else row-major */
#define GEMM_SCHED_CROSS_TILE 0x2u /* overlap the next tile's loads/MMAs with the current
                                      tile's epilogue; else drain at every tile boundary */
#define GEMM_SCHED_SINGLE_CTA 0x4u /* one CTA per 128x256 tile instead of a CTA pair per
                                      256x256 tile (same results, lower throughput) */
#define GEMM_SCHED_NON_PERSISTENT 0x8u /* one program per tile (grid = #tiles, the hardware
                                          assigns programs to SMs) instead of a persistent
                                          grid of co-resident programs */
#define GEMM_SCHED_DYNAMIC 0x10u /* CTA-pair tiles with TMA-loadable A and B: launch one
                                     cluster per tile and let resident clusters take the
                                     tiles of clusters that have not started (cluster launch
                                     control), in ascending tile_id; ignored otherwise */
#define GEMM_SCHED_TAIL_SPLIT 0x20u /* CTA-pair tiles, TMA-loadable A and B, TMA-storable C,
                                       persistent static order: when the last round of
                                       tiles would leave at least three quarters of the
                                       programs idle, split those tiles along K across the
                                       idle programs (see gemm_f16) */
#define GEMM_SCHED_ALL_FLAGS 0x3Fu

/*
 * gemm_f16 — C = A @ B.
 *
 * Defined by [persistent] "naive tiled matmul" / "naive persistent matmul",
 * the tile order by [swizzle] "구현", the cross-tile overlap by [flatten].
 *
 * A: __half[M,K] (device), B: __half[K,N] (device), C: float[M,N] (device).
 * C is overwritten and never read; it must not overlap A or B (undefined).
 * Only the M x N elements are written: memory between rows (stride_cm > N)
 * keeps its contents.
 * group_size_m: GROUP_SIZE_M of the grouped order, >= 1 when
 *   GEMM_SCHED_GROUPED is set (ignored otherwise; G >= #m-tiles gives one
 *   group, G == 1 gives the row-major order).
 * schedule_flags: OR of GEMM_SCHED_* bits; any other bit -> INVALID_ARG.
 *
 * Layouts taken: A with stride_ak == 1 (K-major) or stride_am == 1 (M-major);
 * B with stride_bk == 1 (K-major) or stride_bn == 1 (N-major); C with
 * stride_cn == 1. Other layouts -> GEMM_ERR_UNSUPPORTED. All strides >= 1.
 * Operands whose base address is 16-byte aligned and whose non-unit stride is
 * a multiple of 8 elements (A, B) or 4 elements (C) go through TMA; others
 * (e.g. K = 257 row-major) through a predicated load/store path with the same
 * results. C also needs N to be a multiple of 4 for TMA stores (a clipped TMA
 * store writes whole 16-byte granules; the plain path writes exactly the M x N
 * elements). An fp32 C that fails these conditions (rows not all 16-byte
 * aligned, or N not a multiple of 4) is still stored mostly through TMA by the
 * CTA-pair kernel (static order, N >= 8, a row in every class): rows that share their offset
 * in a 16-byte granule form a class with a tensor map of its own whose rows
 * end on a granule at or before column N, each row's values are shifted in
 * registers so that every box starts on a granule, and the at most 3 leading
 * and 3 trailing values of each row segment outside those boxes, and tiles
 * that reach column N, are written with plain stores: only the M x N elements
 * are written. On the predicated path the rows of A and B are copied per alignment class
 * (rows whose start shares its offset in a 16-byte granule), from the granule
 * boundary below each row start: it may read, and discard, bytes that share
 * an aligned 16-byte granule with an element of A or B, never others. If the
 * driver rejects such a class description -> GEMM_ERR_UNSUPPORTED.
 * The work is split into 256x256 output tiles, each computed by a pair of
 * CTAs on the two SMs of a TPC (tcgen05 cta_group::2), or with
 * GEMM_SCHED_SINGLE_CTA into 128x256 tiles of one CTA each. The tile order
 * (row-major / grouped) applies to whichever tiles are used; a "program" of
 * the persistent order is a CTA pair or a CTA.
 * GEMM_SCHED_TAIL_SPLIT (the pages only name Stream-K, [persistent] "naive
 * persistent matmul"): the tiles of the last round, t of them with t <= P/4,
 * become S >= 2 units each (consecutive K slices of at least 8 k-blocks of 64;
 * S*t <= P), computed by the programs that round would leave idle: unit
 * T - t + v is slice v / t of tile
 * T - t + v % t. Their fp32 partial tiles go to a 24 MiB scratch array built
 * into the library (held by every GPU that loads it); a second kernel on the
 * same stream sums each tile's slices in slice order 0, 1, ..., scales by alpha
 * and rounds into C. Results are deterministic, but the tail tiles' sums are no
 * longer bit-identical to the unsplit order's; integer-valued inputs (every
 * partial sum exact) stay exact. Calls with this flag that overlap on the GPU
 * share the scratch and race: serialise them. The first call on a device that
 * splits a tail looks up the scratch's device address (kept once a lookup
 * succeeds); make it before any stream capture. Where the conditions above do
 * not hold the flag has no effect.
 * GEMM_SCHED_NON_PERSISTENT launches one program per tile ([persistent]
 * "naive tiled matmul" grid); program p then computes tile_id p only, and
 * GEMM_SCHED_CROSS_TILE has nothing to overlap. GEMM_SCHED_DYNAMIC (no
 * counterpart on the pages) keeps programs resident like the persistent order
 * but hands out tiles as programs become free instead of tile_id = pid + i*grid;
 * the tile map itself is unchanged.
 * A and B must be 2-byte aligned and C aligned to its element size, else
 * GEMM_ERR_INVALID_ARG.
 * Sizes: M, N, K >= 0, each < 2^31. M == 0 or N == 0: nothing is done.
 * K == 0: C is set to 0.
 * Returns GEMM_OK once the work is enqueued.
 */
gemm_status_t gemm_f16(const void *A, const void *B, float *C,
                       int64_t M, int64_t N, int64_t K,
                       int64_t stride_am, int64_t stride_ak,
                       int64_t stride_bk, int64_t stride_bn,
                       int64_t stride_cm, int64_t stride_cn,
                       int32_t group_size_m, uint32_t schedule_flags,
                       gemm_stream_t stream);

/* Element type of C for gemm_f16_out. */
#define GEMM_OUT_F32 0
#define GEMM_OUT_F16 1
#define GEMM_OUT_BF16 2

/*
 * gemm_f16_out — C = alpha * (A @ B) stored as fp32, fp16 or bf16.
 *
 * The pages keep the product in an FP32 accumulator and store it ([persistent]
 * "naive tiled matmul"); their C type is never stated. This entry point adds a
 * scale and 16-bit output: every element is the fp32 accumulator times alpha
 * (an fp32 multiply, skipped when alpha == 1), rounded to nearest-even into
 * c_dtype (GEMM_OUT_*; unknown values -> GEMM_ERR_INVALID_ARG). Halving the
 * output bytes matters when K is small and the store dominates the traffic.
 * C: device pointer to M x N elements of c_dtype, stride_cn == 1; TMA stores
 * need a 16-byte-aligned base, stride_cm and N multiples of 16 bytes, otherwise
 * the predicated store path is used. K == 0 writes +0. All other arguments,
 * layouts and errors as gemm_f16; gemm_f16 equals gemm_f16_out with
 * GEMM_OUT_F32 and alpha = 1.
 */
gemm_status_t gemm_f16_out(const void *A, const void *B, void *C, int32_t c_dtype, float alpha,
                           int64_t M, int64_t N, int64_t K,
                           int64_t stride_am, int64_t stride_ak,
                           int64_t stride_bk, int64_t stride_bn,
                           int64_t stride_cm, int64_t stride_cn,
                           int32_t group_size_m, uint32_t schedule_flags,
                           gemm_stream_t stream);

/*
 * gemm_f16_packed — gemm_f16 on copies of A and B whose rows start on
 * 128-byte boundaries, made in a caller workspace. No counterpart on the pages
 * (their operands are contiguous and aligned).
 *
 * The kernels read each operand as K-blocks of 64 elements: one 128-byte line
 * per row. When an operand's base address or its row stride in bytes is not a
 * multiple of 128, every such line straddles two lines of the L2 and costs two
 * requests (measured on GB300: 4000 x 5000 x 3000 with row strides of 3000
 * elements 106.6 us, with 3072 79.5 us); when it is not even a multiple of 16
 * bytes the operand takes the alignment-class loader, several times slower at
 * long K (8192^2 x 4100: 1042 us, 312 us on aligned copies). Each such operand
 * is first copied, in its own orientation (a K-major operand stays K-major),
 * into rows of round_up(inner, 64) elements at the start of the workspace (A)
 * or 256-byte aligned after A's copy (B), by one copy kernel on `stream`; then
 * gemm_f16 runs on the copies. An operand already on 128-byte lines is read in
 * place. C is bit-identical to gemm_f16's (the same products, summed in the
 * same order).
 *
 * Arguments, layouts and errors as gemm_f16, plus:
 * workspace: DEVICE buffer owned by the caller, 128-byte aligned, of at least
 *   gemm_f16_packed_workspace_size() bytes; NULL, misaligned or smaller ->
 *   GEMM_ERR_INVALID_ARG (nothing is launched). The copies are left there; a
 *   call that overlaps on the GPU must not use the same workspace.
 * The copy reads whole aligned 16-byte granules of the source: it may read,
 * and discard, bytes that share such a granule with an element of A or B,
 * never others.
 */
gemm_status_t gemm_f16_packed(const void *A, const void *B, float *C,
                              int64_t M, int64_t N, int64_t K,
                              int64_t stride_am, int64_t stride_ak,
                              int64_t stride_bk, int64_t stride_bn,
                              int64_t stride_cm, int64_t stride_cn,
                              int32_t group_size_m, uint32_t schedule_flags,
                              void *workspace, uint64_t workspace_bytes,
                              gemm_stream_t stream);

/*
 * gemm_f16_packed_workspace_size — workspace bytes gemm_f16_packed needs for
 * these sizes and operand strides (as gemm_f16's; they decide each operand's
 * orientation): room for copies of both operands, whether or not a call ends
 * up copying them. 0 when M, N or K is 0. Sizes or strides out of range ->
 * GEMM_ERR_INVALID_ARG. `bytes` may be NULL. Needs no device.
 */
gemm_status_t gemm_f16_packed_workspace_size(int64_t M, int64_t N, int64_t K,
                                             int64_t stride_am, int64_t stride_ak,
                                             int64_t stride_bk, int64_t stride_bn,
                                             uint64_t *bytes);

/*
 * gemm_f16_splitk — C = A @ B with the K dimension split across CTA pairs
 * (for problems with fewer output tiles than CTA pairs, e.g. small M x N with
 * long K). The pages name Stream-K as a later step without describing it
 * ([persistent] "naive persistent matmul"); this is its plain split-K form.
 *
 * Same arguments, layouts and semantics as gemm_f16, plus:
 * splits: requested K slices (>= 1), or 0 to choose: enough slices to give
 *   every co-resident CTA pair a unit, at most 32. The count used never gives
 *   a slice zero k-blocks (see gemm_f16_splitk_workspace_size).
 * workspace: DEVICE buffer owned by the caller, 16-byte aligned, of at least
 *   gemm_f16_splitk_workspace_size() bytes (may be NULL when that size is 0).
 * Work unit u computes tile u % T over slice u / T into workspace[slice]
 * (fp32, [slices][M][round_up(N, 4)]); a second kernel on the same stream then
 * sums the slices into C in slice order 0, 1, ... (deterministic). The
 * workspace must not be used by another call that overlaps on the GPU.
 * Needs TMA-loadable A and B (see gemm_f16); otherwise, or with
 * GEMM_SCHED_SINGLE_CTA, returns GEMM_ERR_UNSUPPORTED. A workspace smaller
 * than required, or misaligned -> GEMM_ERR_INVALID_ARG.
 */
gemm_status_t gemm_f16_splitk(const void *A, const void *B, float *C,
                              int64_t M, int64_t N, int64_t K,
                              int64_t stride_am, int64_t stride_ak,
                              int64_t stride_bk, int64_t stride_bn,
                              int64_t stride_cm, int64_t stride_cn,
                              int32_t splits, void *workspace, uint64_t workspace_bytes,
                              int32_t group_size_m, uint32_t schedule_flags,
                              gemm_stream_t stream);

/*
 * gemm_f16_splitk_workspace_size — workspace bytes and slice count that
 * gemm_f16_splitk will use for these sizes and `splits` (0 = automatic, which
 * needs a device). *bytes is 0 when one slice is used (no workspace needed).
 * Either output may be NULL.
 */
gemm_status_t gemm_f16_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int32_t splits,
                                             uint64_t *bytes, int32_t *splits_used);

/*
 * gemm_f16_splitk_noalloc — gemm_f16_splitk with no device allocation at all.
 * The pages have no counterpart to this entry point.
 *
 * For callers that must not allocate device memory where they multiply: their
 * memory belongs to another allocator or a fixed arena, or they cannot take
 * the device-wide synchronisation and out-of-memory failures that cudaMalloc
 * brings on that path. Instead of a caller workspace it uses a 32 MiB array
 * built into the library (every GPU that loads the library holds it until the
 * process exits). Arguments as gemm_f16_splitk, without the workspace.
 * - Problems whose split-K workspace (gemm_f16_splitk_workspace_size) exceeds
 *   32 MiB are rejected with GEMM_ERR_UNSUPPORTED; nothing is launched.
 * - The first call on a device that needs the scratch looks up the array's
 *   device address (cudaGetSymbolAddress) with that device current; make that
 *   first call before any stream capture. Only a lookup that succeeds is kept:
 *   if it fails, the call returns GEMM_ERR_CUDA and the next call tries again.
 * - All calls share the one array and it keeps the last call's contents;
 *   nothing in it needs to start at zero. Calls that overlap on the GPU (on
 *   different streams, or from different threads) race on it: serialise them.
 * - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
gemm_status_t gemm_f16_splitk_noalloc(const void *A, const void *B, float *C,
                                      int64_t M, int64_t N, int64_t K,
                                      int64_t stride_am, int64_t stride_ak,
                                      int64_t stride_bk, int64_t stride_bn,
                                      int64_t stride_cm, int64_t stride_cn,
                                      int32_t splits, int32_t group_size_m,
                                      uint32_t schedule_flags, gemm_stream_t stream);

/*
 * gemm_f16_tile_map — the kernel's own tile scheduler, run on the GPU.
 *
 * Defined by [persistent] "naive persistent matmul" (visiting order) and
 * [swizzle] "구현" (grouped map) / [persistent] "naive tiled matmul"
 * (row-major map). Uses the same device function as gemm_f16.
 * out_dev: int32[num_m_tiles*num_n_tiles][3] (device, caller-owned); row
 * tile_id receives {program id that processes it, tile_m, tile_n} where
 * program p visits tile_id = p, p + grid, p + 2*grid, ...
 * grid >= 1; num_m_tiles, num_n_tiles >= 1 and their product < 2^31;
 * flags: only GEMM_SCHED_GROUPED matters (others allowed). Under
 * GEMM_SCHED_DYNAMIC the map tile_id -> (tile_m, tile_n) is this one, but
 * which program computes a tile is decided at run time, so the program
 * column describes the static order only.
 */
gemm_status_t gemm_f16_tile_map(int32_t num_m_tiles, int32_t num_n_tiles,
                                int32_t group_size_m, uint32_t flags, int32_t grid,
                                int32_t *out_dev, gemm_stream_t stream);

/*
 * gemm_f16_get_config — tile shape and launch size gemm_f16 uses for an M x N
 * output with TMA-loadable operands and these schedule_flags, on the current
 * device. The grid rule is [persistent] "naive persistent matmul" (grid =
 * min(#SMs, #tiles), here min(co-resident programs, #tiles)); the tile and K
 * step stand in for the pages' BLOCK_SIZE_M/N/K and num_stages meta-parameters.
 * It takes M, N and the flags because the grid depends on them (the pages
 * compute the grid from the problem size in the launcher).
 * Any output pointer may be NULL; unknown flag bits -> INVALID_ARG.
 * bm, bn, bk: output tile (256x256 per CTA pair, or 128x256 per CTA with
 * GEMM_SCHED_SINGLE_CTA) and K step; stages: shared-memory ring depth; grid:
 * persistent programs (CTA pairs or CTAs) = min(co-resident programs,
 * cdiv(M,bm)*cdiv(N,bn)), or the tile count with GEMM_SCHED_NON_PERSISTENT
 * (needs a device; 0 when M or N is 0).
 */
gemm_status_t gemm_f16_get_config(int64_t M, int64_t N, uint32_t schedule_flags, int32_t *bm,
                                  int32_t *bn, int32_t *bk, int32_t *stages, int32_t *grid);

/*
 * gemm_f16_kernel_info — compiled resource use of a kernel variant
 * (cudaFuncGetAttributes). The pages print the same figures (registers, shared
 * memory) from Triton's kernel metadata ([persistent] "Block Limit 값 직접
 * 계산해보기"); as an entry point it has no counterpart there. One-CTA tiles: variant 0 = TMA loads + TMA store,
 * 1 = TMA loads + predicated store, 2 = predicated loads + TMA store,
 * 3 = predicated loads + predicated store. CTA-pair tiles, in the same
 * order: 4, 5, 6, 7; with GEMM_SCHED_DYNAMIC (TMA loads): 8 = TMA store,
 * 9 = predicated store; 10 = the CTA-pair kernel with a split tail
 * (GEMM_SCHED_TAIL_SPLIT); CTA pairs storing fp32 C per row class (C not
 * TMA-storable as one map, see gemm_f16): 11 = TMA loads, 12 = predicated
 * loads. Outputs may be NULL. Needs a device.
 */
gemm_status_t gemm_f16_kernel_info(int32_t variant, int32_t *regs_per_thread,
                                   int32_t *static_smem, int32_t *dynamic_smem,
                                   int32_t *threads_per_cta);

/*
 * gemm_f16_sync_status — no counterpart on the pages (they describe no
 * failure handling). Synchronize `stream`, then return and clear the
 * sticky device status of the current device: GEMM_ERR_TIMEOUT if any
 * kernel's bounded wait ran out since the last call (that call's C is
 * undefined), GEMM_ERR_CHECK if a debug-build device check failed (the source
 * line goes to stderr), GEMM_ERR_CUDA if the synchronize failed, else GEMM_OK.
 * Calls of the other entry points enqueue work only (no synchronisation, no
 * allocation after the first call on a device), so they can be captured in a
 * CUDA graph; a replayed launch reuses its captured abort epoch, which this
 * call clears together with the status.
 */
gemm_status_t gemm_f16_sync_status(gemm_stream_t stream);

/*
 * gemm_f16_set_wait_timeout — no counterpart on the pages. Upper bound, in
 * nanoseconds of GPU global time, on any single wait inside the kernels
 * (default 2e9 = 2 s). Applies
 * to launches enqueued after the call. ns must be >= 1000.
 */
gemm_status_t gemm_f16_set_wait_timeout(uint64_t ns);

/*
 * gemm_f16_selftest_wait_timeout — failure-detection self-test (the pages have
 * no counterpart: they describe no failure handling). Enqueues one thread that
 * waits, through the same bounded-wait routine as every wait inside gemm_f16,
 * on an mbarrier nothing arrives on. After timeout_ns (1e3 .. 1e10) the wait
 * gives up, the sticky status becomes GEMM_ERR_TIMEOUT (read and cleared by
 * gemm_f16_sync_status) and the kernel returns; the CUDA context stays usable.
 */
gemm_status_t gemm_f16_selftest_wait_timeout(uint64_t timeout_ns, gemm_stream_t stream);

/*
 * gemm_f16_selftest_pair_abort — failure-detection self-test of the CTA-pair
 * kernel (no counterpart on the pages). Enqueues gemm_f16 on row-major A
 * [M,K], B [K,N] and C [M,N] (device, 16-byte-aligned A and B, K and N
 * multiples of 8; otherwise GEMM_ERR_UNSUPPORTED), grouped order with
 * GEMM_SCHED_CROSS_TILE, except that both CTAs of every pair stop issuing
 * copies once they have issued `stop_after` (>= 1) pipeline stages, while
 * still waiting for stages to be freed as in a normal run. No stage is then
 * left half-counted, and the MMA warp's wait for the first missing stage runs
 * out after the current wait limit (gemm_f16_set_wait_timeout): the kernel
 * records GEMM_ERR_TIMEOUT, every CTA's other waits give up, each CTA waits
 * (bounded) for its own work in flight, frees its TMEM and returns. The
 * sticky status is read and cleared by gemm_f16_sync_status; C is undefined
 * and the context stays usable.
 */
gemm_status_t gemm_f16_selftest_pair_abort(const void *A, const void *B, float *C,
                                           int64_t M, int64_t N, int64_t K, int32_t stop_after,
                                           gemm_stream_t stream);

/*
 * gemm_f16_selftest_check — debug build (GEMM_DEBUG) only: launches one
 * device-side check that fails without guarding any access, so that
 * gemm_f16_sync_status then returns GEMM_ERR_CHECK (and clears it). The product
 * build has no device-side checks and returns GEMM_ERR_UNSUPPORTED.
 * No counterpart on the pages (it stands in for a sanitizer run).
 */
gemm_status_t gemm_f16_selftest_check(gemm_stream_t stream);

/* gemm_f16_status_str — static, human-readable name of a status code (no
 * counterpart on the pages). Unknown codes give "GEMM_ERR_UNKNOWN". */
const char *gemm_f16_status_str(gemm_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F16_H */
