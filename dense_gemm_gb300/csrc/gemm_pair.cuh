// CTA-pair variant of the persistent FP16 GEMM (sm_103a): one 256 x 256 output
// tile per pair of CTAs (a cluster of 2 on the two SMs of a TPC).
//
// Same method as gemm_f16_persistent (tile GEMM body, persistent visiting order,
// row-major / grouped tile maps, cross-tile overlap; see gemm_kernel.cuh for the
// pages each part follows); only the split of one tile across two SMs differs:
//   * CTA r (r = 0, 1) loads A rows [tile_m*256 + r*128, +128) and B columns
//     [tile_n*256 + r*128, +128) into its own ring; both CTAs' TMA copies count
//     on CTA 0's "full" barrier (cp.async.bulk.tensor .cta_group::2);
//   * CTA 0 issues tcgen05.mma.cta_group::2 (256 x 256 x 16): each SM's tensor
//     core computes its 128 rows from its own A half and both B halves, into its
//     own TMEM; commits are multicast to both CTAs' barriers;
//   * each CTA's epilogue drains its own 128 x 256 accumulator; CTA 0's MMA
//     reuses an accumulator only after both epilogues have released it.
// Per SM and 64-deep k-block this moves 32 KiB from L2 into shared memory
// (48 KiB for the single-CTA 128 x 256 tile) for the same tensor work.
#pragma once
#include "gemm_kernel.cuh"

namespace g16 {

namespace pair {
constexpr int TILE_M = 256;                 // rows per pair tile (128 per CTA)
constexpr int TILE_N = 256;                 // columns per pair tile (B: 128 per CTA)
constexpr int CTA_M = 128;
constexpr int CTA_N = 128;
constexpr int STAGES = 6;
constexpr int A_STAGE_BYTES = CTA_M * BK * 2;  // 16 KiB
constexpr int B_STAGE_BYTES = CTA_N * BK * 2;  // 16 KiB
constexpr uint32_t PAIR_TX_BYTES = 2u * (A_STAGE_BYTES + B_STAGE_BYTES);

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
constexpr int OFF_EPI = OFF_B + STAGES * B_STAGE_BYTES;
constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
// full[S], empty[S], tfull[2], tempty[2], tdone[2], drain
constexpr int NUM_BARS = 2 * STAGES + 3 * NUM_ACC + 1;
constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = OFF_TMEM_SLOT + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
constexpr int THREADS = (1 + 1 + EPI_WARPS) * 32;

static_assert(OFF_B % 1024 == 0 && OFF_EPI % 1024 == 0, "swizzled buffers need 1 KiB alignment");
static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KiB per-CTA shared memory limit");
}  // namespace pair

template <bool kTmaStore>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::THREADS, 1)
    gemm_f16_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmC, const Params p) {
    constexpr int MMA_WARP = 1;
    constexpr int EPI_WARP0 = 2;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // same offset in both CTAs
    uint8_t *smem = smem_raw + (base - raw);

    const uint32_t sA = base + pair::OFF_A;
    const uint32_t sB = base + pair::OFF_B;
    const uint32_t bar0 = base + pair::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (pair::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * pair::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * pair::STAGES + NUM_ACC + a); };
    auto tdone_bar = [&](int a) { return bar0 + 8u * (2 * pair::STAGES + 2 * NUM_ACC + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * pair::STAGES + 3 * NUM_ACC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + pair::OFF_TMEM_SLOT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
    const int32_t pair_id = int32_t(blockIdx.x >> 1);
    const int32_t num_pairs = int32_t(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < pair::STAGES; ++s) {
            mbar_init(full_bar(s), 1);   // CTA 0's arrive.expect_tx; both CTAs' bytes
            mbar_init(empty_bar(s), 1);  // CTA 0's MMA commit (multicast)
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            mbar_init(tfull_bar(a), 1);              // CTA 0's MMA commit (multicast)
            mbar_init(tempty_bar(a), 2 * EPI_WARPS);  // every epilogue warp of both CTAs
            mbar_init(tdone_bar(a), EPI_WARPS);       // this CTA's epilogue warps
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {  // one warp in each CTA of the pair, collectively
        tmem_alloc_pair(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (kTmaStore && warp == EPI_WARP0 && lane == 0) prefetch_tensormap(&tmC);
    tc_fence_before();
    cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int32_t num_kb = p.num_kb;

    if (warp == 0) {
        // ============================================================ producer (both CTAs)
        if (lane == 0) {
            const uint64_t pol_ld = l2_policy_evict_last();
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            int32_t it = 0;
            for (int32_t u = pair_id; ok && u < p.num_units; u += num_pairs, ++it) {
                const int32_t tile = u % p.num_tiles, split = u / p.num_tiles;
                const int32_t kb0 = split * p.kb_per_split;
                const int32_t kb1 = min(num_kb, kb0 + p.kb_per_split);
                int32_t tm, tn;
                tile_coords(tile, p.sched, tm, tn);
                if (!p.cross_tile && it > 0) {
                    const int32_t j = it - 1;  // this CTA's epilogue has drained unit j
                    if (!mbar_wait(tdone_bar(j & 1), (j >> 1) & 1, p.wait)) { ok = false; break; }
                }
                const int32_t m0 = tm * pair::TILE_M + int32_t(rank) * pair::CTA_M;
                const int32_t n0 = tn * pair::TILE_N + int32_t(rank) * pair::CTA_N;
                for (int32_t kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.wait)) { ok = false; break; }
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), pair::PAIR_TX_BYTES);
                    const uint32_t fb = mapa_shared(full_bar(stage), 0);
                    const int32_t k0 = kb * BK;
                    const uint32_t a_dst = sA + stage * pair::A_STAGE_BYTES;
                    const uint32_t b_dst = sB + stage * pair::B_STAGE_BYTES;
                    if (p.l2_mode & 2u) {  // operand tiles are re-read by other pairs: keep in L2
                        if (!p.a_mn) {
                            tma_load_2d_pair_hint(a_dst, &tmA, k0, m0, fb, pol_ld);
                        } else {
#pragma unroll
                            for (int c = 0; c < pair::CTA_M / MN_CHUNK; ++c)
                                tma_load_2d_pair_hint(a_dst + c * MN_CHUNK_BYTES, &tmA, m0 + c * MN_CHUNK,
                                                      k0, fb, pol_ld);
                        }
                        if (!p.b_mn) {
                            tma_load_2d_pair_hint(b_dst, &tmB, k0, n0, fb, pol_ld);
                        } else {
#pragma unroll
                            for (int c = 0; c < pair::CTA_N / MN_CHUNK; ++c)
                                tma_load_2d_pair_hint(b_dst + c * MN_CHUNK_BYTES, &tmB, n0 + c * MN_CHUNK,
                                                      k0, fb, pol_ld);
                        }
                    } else {
                        if (!p.a_mn) {
                            tma_load_2d_pair(a_dst, &tmA, k0, m0, fb);
                        } else {
#pragma unroll
                            for (int c = 0; c < pair::CTA_M / MN_CHUNK; ++c)
                                tma_load_2d_pair(a_dst + c * MN_CHUNK_BYTES, &tmA, m0 + c * MN_CHUNK, k0, fb);
                        }
                        if (!p.b_mn) {
                            tma_load_2d_pair(b_dst, &tmB, k0, n0, fb);
                        } else {
#pragma unroll
                            for (int c = 0; c < pair::CTA_N / MN_CHUNK; ++c)
                                tma_load_2d_pair(b_dst + c * MN_CHUNK_BYTES, &tmB, n0 + c * MN_CHUNK, k0, fb);
                        }
                    }
                    ++issued;
                    if (++stage == pair::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                if (rank == 0) {
                    // Let the copies counted on this CTA's barriers land before exiting.
                    const uint32_t n = issued < pair::STAGES ? issued : pair::STAGES;
                    for (uint32_t q = issued - n; q < issued; ++q)
                        mbar_wait_slow(full_bar(q % pair::STAGES), (q / pair::STAGES) & 1u,
                                       cleanup_wait(p.wait), false);
                } else {
                    // The peer's copies count on CTA 0's barriers, which it cannot
                    // wait on; give copies already issued time to land (each is a
                    // 16 KiB L2/HBM read, microseconds at most).
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 200000ull) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ============================================================ MMA issuer (CTA 0)
        // Whole warp, warp-uniform values; one elected lane issues (see the
        // single-CTA kernel).
        if (rank == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            int32_t it = 0;
            const DescStep da = make_desc_step(sA, p.a_mn, pair::A_STAGE_BYTES);
            const DescStep db = make_desc_step(sB, p.b_mn, pair::B_STAGE_BYTES);
            const uint32_t idesc = p.idesc;
            for (int32_t u = pair_id; ok && u < p.num_units; u += num_pairs, ++it) {
                const int32_t kb0 = (u / p.num_tiles) * p.kb_per_split;
                const int32_t kb1 = min(num_kb, kb0 + p.kb_per_split);
                const uint32_t acc = it & 1, use = it >> 1;
                // both CTAs' epilogues have released this accumulator (remote arrivals)
                if (!__all_sync(0xffffffffu,
                                mbar_wait_cluster(tempty_bar(acc), (use & 1u) ^ 1u, p.wait))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * pair::TILE_N;
                for (int32_t kb = kb0; kb < kb1; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait(full_bar(stage), phase, p.wait))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a0 = da.base + stage * da.stage;
                    const uint64_t b0 = db.base + stage * db.stage;
#pragma unroll
                    for (int k16 = 0; k16 < BK / UMMA_K; ++k16)
                        mma_f16_pair_elect(d_tmem, a0 + k16 * da.k16, b0 + k16 * db.k16, idesc,
                                           ((kb - kb0) | k16) != 0 ? 1u : 0u);
                    mma_commit_pair_mc_elect(empty_bar(stage), 0x3);  // both CTAs' slots reusable
                    if (++stage == pair::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair_mc_elect(tfull_bar(acc), 0x3);  // both halves of the tile complete
            }
            mma_commit_pair_elect(drain_bar);
            __all_sync(0xffffffffu, mbar_wait_slow(drain_bar, 0, cleanup_wait(p.wait), false));
        }
    } else {
        // ============================================================ epilogue (both CTAs)
        const int q = warp & 3;
        const int ew = warp - EPI_WARP0;
        const int half = ew / 4;
        const uint32_t stg = base + pair::OFF_EPI + uint32_t(ew) * (EPI_BUFS * EPI_BUF_BYTES);
        int32_t it = 0;
        for (int32_t u = pair_id; u < p.num_units; u += num_pairs, ++it) {
            const int32_t tile = u % p.num_tiles, split = u / p.num_tiles;
            const int32_t kb0 = split * p.kb_per_split;
            const int32_t unit_kb = min(num_kb, kb0 + p.kb_per_split) - kb0;
            int32_t tm, tn;
            tile_coords(tile, p.sched, tm, tn);
            const uint32_t acc = it & 1, use = it >> 1;
            const bool ready = __all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), use & 1u, p.wait));
            if (!ready) break;
            tc_fence_after();
            const int64_t row0 = int64_t(tm) * pair::TILE_M + int64_t(rank) * pair::CTA_M + q * 32;
            const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + acc * pair::TILE_N;
            auto release = [&] {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(tdone_bar(acc));
                    mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
                }
            };
            const int64_t col_base = int64_t(tn) * pair::TILE_N;
            int c0, n;
            if (p.out_dtype == 0 || p.splits > 1) {  // split-K partials are fp32
                epilogue_chunks(unit_kb, half, EPI_CHUNKS32, c0, n);
                epilogue_tile<kTmaStore>(t_row, row0, col_base, c0, n, p, &tmC, stg, lane, release, split,
                                         epilogue_pace_ns(unit_kb, p.cross_tile, n));
            } else {
                epilogue_chunks(unit_kb, half, EPI_CHUNKS16, c0, n);
                epilogue_tile16<kTmaStore>(t_row, row0, col_base, c0, n, p, &tmC, stg, lane, release,
                                           epilogue_pace_ns(unit_kb, p.cross_tile, n));
            }
        }
        if (kTmaStore && lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    cluster_sync();  // no CTA leaves while its peer may still use its smem or barriers
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace g16
