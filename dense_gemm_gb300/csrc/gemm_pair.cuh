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
// kDyn (TMA loads only) replaces the static pid + i*P stream by cluster launch
// control: one cluster per unit in the grid, resident clusters cancel those that
// have not started and take their units, in ascending order.
// Predicated-load variant (kTmaLoad = false, operands not describable by one
// tensor map): per CTA one warp issues the TMA copies of the alignment-class
// boxes (see gemm_kernel.cuh) into four staging rings, and four warps each
// shift one 64-line copy group per K-block into the stage (a TMA issue stalls
// its warp ~110-175 cycles, so issuing apart from the shifting overlaps the
// two). In CTA 0 the shifting warps arrive on the "full" barrier directly; in
// CTA 1 on a local
// "placed" barrier, from which CTA 1's otherwise idle MMA warp relays one
// cluster-scope arrival to CTA 0 (a release at cluster scope costs a loader
// warp 1000-3500 cycles; measured with clock64 timestamps).
#pragma once
#include <type_traits>

#include "gemm_kernel.cuh"

namespace g16 {

namespace pair {
constexpr int TILE_M = 256;                 // rows per pair tile (128 per CTA)
constexpr int TILE_N = 256;                 // columns per pair tile (B: 128 per CTA)
constexpr int CTA_M = 128;
constexpr int CTA_N = 128;
constexpr int STAGES = 6;                   // TMA-load variant
constexpr int A_STAGE_BYTES = CTA_M * BK * 2;  // 16 KiB
constexpr int B_STAGE_BYTES = CTA_N * BK * 2;  // 16 KiB
constexpr uint32_t PAIR_TX_BYTES = 2u * (A_STAGE_BYTES + B_STAGE_BYTES);
constexpr int PLACE_WARPS = 4;              // predicated loads: one copy group (64 lines) each per K-block
static_assert(PLACE_WARPS * GROUP_LINES == CTA_M + CTA_N, "loader shares");
// Dynamic units (cluster launch control): CTA 0's producer requests the
// cancellations, both CTAs' producers read the answers and publish the unit
// sequence into their own CTA's ring of QDEPTH ids. Every reader trails the
// producer by at most STAGES units (the producer waits for the MMA to free a
// stage) plus NUM_ACC (the MMA waits for the epilogue to free an accumulator),
// so slots are reused only after every reader has read them.
constexpr int QDEPTH = 16;
static_assert(QDEPTH > STAGES + NUM_ACC + 3, "unit ring shorter than the readers' lag");
// Cancellation answers arrive in both CTAs (multicast); CTA 1's producer may
// trail CTA 0's by up to STAGES units, so answers rotate over more slots.
constexpr int NCLC = 8;
static_assert(NCLC > STAGES + 1, "answer slots reused before CTA 1 read them");

// Shared-memory map. The predicated-load variant keeps two operand stages and
// holds the loader warps' staging rings (one mbarrier per slot) instead.
template <bool kTmaLoad>
struct Layout {
    static constexpr int stages = kTmaLoad ? STAGES : 2;
    // TMA loads: one producer warp. Predicated loads: PLACE_WARPS warps that
    // shift staged lines into the stages, then one warp that issues their copies.
    static constexpr int load_warps = kTmaLoad ? 1 : PLACE_WARPS + 1;
    static constexpr int threads = (load_warps + 1 + EPI_WARPS) * 32;
    static constexpr int off_a = 0;
    static constexpr int off_b = off_a + stages * A_STAGE_BYTES;
    static constexpr int off_epi = off_b + stages * B_STAGE_BYTES;
    static constexpr int off_copy = off_epi + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
    static constexpr int copy_slots = kTmaLoad ? 0 : PLACE_WARPS * COPY_DEPTH;
    static constexpr int off_bar = off_copy + copy_slots * GROUP_BYTES;
    // full[S], empty[S], tfull[2], tempty[2], tdone[2], drain, then for predicated
    // loads placed[S] (CTA 1's loaders -> its relay), the copy-slot barriers
    // (copies landed) and slot_free[COPY_DEPTH] (slot read by every placing warp)
    static constexpr int placed_bar0 = 2 * stages + 3 * NUM_ACC + 1;
    static constexpr int copy_bar0 = placed_bar0 + (kTmaLoad ? 0 : stages);
    static constexpr int free_bar0 = copy_bar0 + copy_slots;
    // cluster launch control: two response slots and their barriers, the unit ring
    static constexpr int clc_bar0 = free_bar0 + (kTmaLoad ? 0 : COPY_DEPTH);
    static constexpr int qfull_bar0 = clc_bar0 + NCLC;
    static constexpr int num_bars = qfull_bar0 + QDEPTH;
    static constexpr int off_tmem_slot = off_bar + num_bars * 8;
    static constexpr int off_clc_resp = (off_tmem_slot + 16 + 15) / 16 * 16;
    static constexpr int off_qids = off_clc_resp + NCLC * 16;
    static constexpr int smem_bytes = off_qids + QDEPTH * 4 + 1024;
    static_assert(off_b % 1024 == 0 && off_epi % 1024 == 0, "swizzled buffers need 1 KiB alignment");
    static_assert(off_copy % 128 == 0, "TMA box destinations need 128-byte alignment");
    static_assert(smem_bytes <= 232448, "exceeds the 227 KiB per-CTA shared memory limit");
};
constexpr int SMEM_BYTES = Layout<true>::smem_bytes;
constexpr int THREADS = Layout<true>::threads;
}  // namespace pair

// C's class maps of a kernel's map parameter (nullptr where it holds none).
template <typename Maps>
__device__ __forceinline__ const CUtensorMap *cm_c(const Maps &m) {
    if constexpr (std::is_same_v<Maps, CClassMaps> || std::is_same_v<Maps, ClassMapsAndC>)
        return m.c;
    else
        return nullptr;
}

// kDyn: units handed out by cluster launch control (TMA loads only); a
// separate instantiation, so the static schedule carries none of its code.
// kTail (TMA loads and stores, static schedule): the tiles of a last, partial
// round are split along K across the programs that round would leave idle;
// their fp32 partial tiles go to the scratch described by tmW, and a second
// kernel sums them into C.
// kClassStore (static schedule, fp32 C whose rows are not all 16-byte aligned):
// C goes out per row class through the maps in cm.c (epilogue_tile_class).
template <bool kTmaLoad, bool kTmaStore, bool kDyn = false, bool kTail = false, bool kClassStore = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::Layout<kTmaLoad>::threads, 1)
    gemm_f16_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmW,
                  const Params p, const __grid_constant__ typename PairMapsFor<kTmaLoad, kClassStore>::type cm) {
    static_assert(!kTail || (kTmaLoad && kTmaStore && !kDyn), "split tail: TMA loads and stores, static stream");
    static_assert(!kClassStore || (!kTmaStore && !kDyn && !kTail), "class stores: plain-store C, static stream");
    using Lay = pair::Layout<kTmaLoad>;
    constexpr int NST = Lay::stages;
    constexpr int LOAD_WARPS = Lay::load_warps;
    constexpr int MMA_WARP = LOAD_WARPS;
    constexpr int EPI_WARP0 = LOAD_WARPS + 1;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // same offset in both CTAs
    uint8_t *smem = smem_raw + (base - raw);

    const uint32_t sA = base + Lay::off_a;
    const uint32_t sB = base + Lay::off_b;
    const uint32_t bar0 = base + Lay::off_bar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (NST + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * NST + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * NST + NUM_ACC + a); };
    auto tdone_bar = [&](int a) { return bar0 + 8u * (2 * NST + 2 * NUM_ACC + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * NST + 3 * NUM_ACC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay::off_tmem_slot);
    // per accumulator: CTA 1's epilogue warps that have drained it (predicated loads)
    const uint32_t drained_ctr = base + Lay::off_tmem_slot + 8u;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
    const int32_t pair_id = int32_t(blockIdx.x >> 1);
    const int32_t num_pairs = int32_t(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            // TMA loads: CTA 0's arrive.expect_tx, both CTAs' bytes; predicated
            // loads: CTA 0's shifting warps plus CTA 1's relay
            mbar_init(full_bar(s), kTmaLoad ? 1 : pair::PLACE_WARPS + 1);
            mbar_init(empty_bar(s), 1);  // CTA 0's MMA commit (multicast)
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            mbar_init(tfull_bar(a), 1);              // CTA 0's MMA commit (multicast)
            // CTA 0's epilogue warps, and CTA 1's through one arrive (or each of them)
            mbar_init(tempty_bar(a), p.relay ? EPI_WARPS + 1 : 2 * EPI_WARPS);
            st_shared_s32(drained_ctr + 4u * a, 0);
            mbar_init(tdone_bar(a), EPI_WARPS);       // this CTA's epilogue warps
        }
        mbar_init(drain_bar, 1);
        if (!kTmaLoad) {
            for (int q = 0; q < NST; ++q) mbar_init(bar0 + 8u * (Lay::placed_bar0 + q), pair::PLACE_WARPS);
            for (int q = 0; q < COPY_DEPTH; ++q) mbar_init(bar0 + 8u * (Lay::free_bar0 + q), pair::PLACE_WARPS);
        }
        for (int q = 0; q < Lay::copy_slots; ++q) mbar_init(bar0 + 8u * (Lay::copy_bar0 + q), 1);
        for (int q = 0; q < pair::NCLC + pair::QDEPTH; ++q) mbar_init(bar0 + 8u * (Lay::clc_bar0 + q), 1);
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {  // one warp in each CTA of the pair, collectively
        tmem_alloc_pair(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    if constexpr (kTmaLoad) {
        if (warp == 0 && lane == 0) {
            prefetch_tensormap(&tmA);
            prefetch_tensormap(&tmB);
        }
    } else {
        if (warp == 0 && lane < 2 * MAX_CLASSES) {  // the maps of classes that hold rows
            const int op = lane / MAX_CLASSES, cls = lane % MAX_CLASSES;
            if ((p.cls_live[op] >> cls) & 1u) prefetch_tensormap(op == 0 ? &cm.a[cls] : &cm.b[cls]);
        }
    }
    if (kTmaStore && warp == EPI_WARP0 && lane == 0) prefetch_tensormap(&tmC);
    if constexpr (kClassStore) {
        if (warp == EPI_WARP0 && lane < int(p.c_classes)) prefetch_tensormap(&cm_c(cm)[lane]);
    }
    tc_fence_before();
    cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
    tc_fence_after();
    // The set-up above may overlap the end of the previous kernel on the
    // stream; nothing below touches global memory before that kernel is done.
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    const int32_t num_kb = p.num_kb;

    // ---- unit sequence of this pair: pair_id, then pair_id + num_pairs, ... (static), or
    // with dynamic units pair_id (= this cluster's own unit) followed by the units of the
    // clusters CTA 0's producer cancels, published into the ring.
    static_assert(!kDyn || kTmaLoad, "dynamic units need TMA loads");
    constexpr bool dyn = kDyn;
    const uint32_t qids = base + Lay::off_qids;
    auto qfull_bar = [&](uint32_t q) { return bar0 + 8u * (Lay::qfull_bar0 + q); };
    // unit number k >= 1 of the sequence is published in ring entry k - 1 (unit 0 is the
    // cluster's own and never published)
    auto read_unit = [&](uint32_t k, int32_t &u) -> bool {
        const uint32_t q = (k - 1) % pair::QDEPTH;
        if (!mbar_wait_cluster(qfull_bar(q), ((k - 1) / pair::QDEPTH) & 1u, p.wait)) return false;
        u = ld_shared_s32(qids + 4u * q);
        return true;
    };
    auto next_unit = [&](uint32_t it, int32_t &u) -> bool {  // readers: advance past unit number it
        if (!dyn) {
            u += num_pairs;
            return true;
        }
        return read_unit(it + 1, u);
    };
    // true if unit number k is known to be the end of the sequence (readers, no waiting)
    auto known_end = [&](uint32_t k, int32_t u) -> bool {
        if (!dyn) return u + num_pairs >= p.num_units;
        const uint32_t q = (k - 1) % pair::QDEPTH;
        return mbar_test_wait_cluster(qfull_bar(q), ((k - 1) / pair::QDEPTH) & 1u) &&
               ld_shared_s32(qids + 4u * q) < 0;
    };

    if (!kTmaLoad && warp < LOAD_WARPS) {
        // ============================================================ predicated loads (both CTAs)
        // Warp w < PLACE_WARPS shifts copy group w & 1 of operand w >> 1 (this
        // CTA's 128 rows of A, or 128 columns of B) for every K-block out of its
        // COPY_DEPTH-slot staging ring; warp PLACE_WARPS issues the copies, up to
        // COPY_DEPTH K-blocks ahead. With cross-tile off the copies of a unit
        // start only after this CTA's epilogue has drained the previous unit.
        if constexpr (!kTmaLoad) {
            constexpr int PW = pair::PLACE_WARPS;
            auto ring = [&](int w) { return base + Lay::off_copy + uint32_t(w) * (COPY_DEPTH * GROUP_BYTES); };
            auto copy_bar = [&](int w, uint32_t q) { return bar0 + 8u * (Lay::copy_bar0 + w * COPY_DEPTH + q); };
            auto free_bar = [&](uint32_t q) { return bar0 + 8u * (Lay::free_bar0 + q); };
            struct Cursor {
                int32_t u, it, kb, kb0, kb1;
                int64_t m0, n0;  // this CTA's first row of A and column of B
            };
            auto setup = [&](Cursor &c) {
                if (c.u >= p.num_units) return;
                const int32_t tile = c.u % p.num_tiles, split = c.u / p.num_tiles;
                c.kb0 = split * p.kb_per_split;
                c.kb1 = min(num_kb, c.kb0 + p.kb_per_split);
                c.kb = c.kb0;
                int32_t tm, tn;
                tile_coords(tile, p.sched, tm, tn);
                c.m0 = int64_t(tm) * pair::TILE_M + int64_t(rank) * pair::CTA_M;
                c.n0 = int64_t(tn) * pair::TILE_N + int64_t(rank) * pair::CTA_N;
            };
            auto advance = [&](Cursor &c) {
                if (++c.kb < c.kb1) return;
                c.u += num_pairs;
                ++c.it;
                setup(c);
            };
            Cursor c{pair_id, 0, 0, 0, 0, 0, 0};
            setup(c);
            uint32_t n = 0;  // K-blocks handled so far
            bool ok = true;
            if (warp == PW) {
                // ---- copy issuer: lane 8w + i issues box i of shifting warp w's group
                const int w = lane >> 3, bi = lane & 7;
                for (; c.u < p.num_units; advance(c), ++n) {
                    if (c.kb == c.kb0 && !p.cross_tile && c.it > 0) {
                        const int32_t j = c.it - 1;  // this CTA's epilogue has drained unit j
                        if (!__all_sync(0xffffffffu, mbar_wait(tdone_bar(j & 1), (j >> 1) & 1, p.wait))) {
                            ok = false;
                            break;
                        }
                    }
                    const uint32_t q = n % COPY_DEPTH;
                    // every shifting warp has read the slot's previous contents
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(free_bar(q), ((n / COPY_DEPTH) & 1u) ^ 1u, p.wait))) {
                        ok = false;
                        break;
                    }
                    const int op = w >> 1;
                    const GroupShape gs = group_shape(p, op, w & 1, 7, op == 0 ? c.m0 : c.n0);
                    issue_class_group_lanes(p, cm, gs, int64_t(c.kb) * BK, ring(w) + q * GROUP_BYTES,
                                            copy_bar(w, q), bi);
                }
                if (!ok) {
                    // Let the copies this warp started land before the CTA exits.
                    const uint32_t first = n > COPY_DEPTH ? n - COPY_DEPTH : 0;
                    for (uint32_t m = first; m < n; ++m)
                        for (int w2 = 0; w2 < PW; ++w2)
                            mbar_wait_slow(copy_bar(w2, m % COPY_DEPTH), (m / COPY_DEPTH) & 1u,
                                           cleanup_wait(p.wait), false);
                }
            } else {
                // ---- shifting warp
                const int op = warp >> 1, grp = warp & 1;
                uint32_t stage = 0, phase = 0;
                // CTA 0 signals its own full barrier, CTA 1 its placed barrier (relayed)
                const uint32_t done0 = rank == 0 ? full_bar(0) : bar0 + 8u * Lay::placed_bar0;
                for (; c.u < p.num_units; advance(c), ++n) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.wait)) break;
                    const uint32_t q = n % COPY_DEPTH;
                    if (!mbar_wait(copy_bar(warp, q), (n / COPY_DEPTH) & 1u, p.wait)) break;
                    const GroupShape gs = group_shape(p, op, grp, 7, op == 0 ? c.m0 : c.n0);
                    place_class_group(p, gs, ring(warp) + q * GROUP_BYTES,
                                      op == 0 ? sA + stage * pair::A_STAGE_BYTES : sB + stage * pair::B_STAGE_BYTES,
                                      lane);
                    // generic-proxy writes -> visible to the tensor core; this
                    // warp's staging reads ordered before the slot's next copies
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(done0 + 8u * stage);
                        mbar_arrive(free_bar(q));
                    }
                    if (++stage == NST) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 0) {
        // ============================================================ producer (both CTAs)
        // The whole warp walks the stage sequence with warp-uniform values. Lane 0
        // arms the barriers and makes the cluster-launch-control requests; the
        // copies of a stage (A: one box, or two 64-wide chunks when M-major; B
        // likewise) are issued by separate lanes in one instruction. One thread
        // issuing them in series took a measurable share of each k-block
        // (device-timed on GB300: 16384^2 x 4096 1.266 -> 1.237 ms, 8192^2 x 4096
        // 328.5 -> 321.8 us).
        {
            const uint64_t pol_ld = l2_policy_evict_last();
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            int32_t it = 0;
            const int na = p.a_mn ? pair::CTA_M / MN_CHUNK : 1;  // copies of A per stage
            const int nb = p.b_mn ? pair::CTA_N / MN_CHUNK : 1;  // copies of B per stage
            // dynamic units: CTA 0 asks for the next cluster's cancellation one unit
            // ahead; the answer lands in both CTAs, whose producers each arm their own
            // barrier for it, read it and publish the unit into their CTA's ring
            uint32_t requested = 0, answered = 0;
            bool ended = false;
            auto clc_resp = [&](uint32_t i) { return base + Lay::off_clc_resp + 16u * (i % pair::NCLC); };
            auto clc_bar = [&](uint32_t i) { return bar0 + 8u * (Lay::clc_bar0 + i % pair::NCLC); };
            auto request = [&] {  // CTA 0
                if (lane == 0) {
                    mbar_arrive_expect_tx(clc_bar(requested), 16);
                    clc_try_cancel_all(clc_resp(requested), clc_bar(requested));
                }
                ++requested;
            };
            auto publish = [&](uint32_t k, int32_t id) {  // unit number k >= 1 -> ring entry k - 1
                if (lane == 0) {
                    const uint32_t q = (k - 1) % pair::QDEPTH;
                    st_shared_s32(qids + 4u * q, id);
                    mbar_arrive(qfull_bar(q));
                }
            };
            if (dyn && rank == 0) request();
            for (int32_t u = pair_id; ok && (!kDyn || u >= 0) && u < p.num_units; ++it) {
                int32_t tile = u % p.num_tiles, split = u / p.num_tiles;
                int32_t kb0 = split * p.kb_per_split;
                int32_t kb1 = min(num_kb, kb0 + p.kb_per_split);
                if constexpr (kTail) {
                    int32_t slot;
                    tail_unit(p, u, tile, kb0, kb1, slot);
                }
                int32_t tm, tn;
                tile_coords(tile, p.sched, tm, tn);
                if (!p.cross_tile && it > 0) {
                    const int32_t j = it - 1;  // this CTA's epilogue has drained unit j
                    if (!__all_sync(0xffffffffu, mbar_wait(tdone_bar(j & 1), (j >> 1) & 1, p.wait))) {
                        ok = false;
                        break;
                    }
                }
                const int32_t m0 = tm * pair::TILE_M + int32_t(rank) * pair::CTA_M;
                const int32_t n0 = tn * pair::TILE_N + int32_t(rank) * pair::CTA_N;
                for (int32_t kb = kb0; kb < kb1; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait(empty_bar(stage), phase ^ 1u, p.wait))) {
                        ok = false;
                        break;
                    }
                    if (p.stop_after > 0 && issued >= uint32_t(p.stop_after)) {  // self-test: nothing more
                        if (++stage == NST) { stage = 0; phase ^= 1u; }
                        continue;
                    }
                    if (lane == 0 && rank == 0) mbar_arrive_expect_tx(full_bar(stage), pair::PAIR_TX_BYTES);
                    const uint32_t fb = mapa_shared(full_bar(stage), 0);
                    const int32_t k0 = kb * BK;
                    if (lane < na + nb) {  // lane: copy `lane` of A, or copy `lane - na` of B
                        const bool is_a = lane < na;
                        const int c = is_a ? lane : lane - na;
                        const CUtensorMap *map = is_a ? &tmA : &tmB;
                        const uint32_t dst = (is_a ? sA + stage * pair::A_STAGE_BYTES : sB + stage * pair::B_STAGE_BYTES) +
                                             uint32_t(c) * MN_CHUNK_BYTES;
                        const bool mn_major = (is_a ? p.a_mn : p.b_mn) != 0;
                        const int32_t mn = (is_a ? m0 : n0) + c * MN_CHUNK;
                        const int32_t x = mn_major ? mn : k0, y = mn_major ? k0 : mn;
                        if (p.l2_mode & 2u)  // operand tiles are re-read by other pairs: keep in L2
                            tma_load_2d_pair_hint(dst, map, x, y, fb, pol_ld);
                        else
                            tma_load_2d_pair(dst, map, x, y, fb);
                    }
                    ++issued;
                    if (++stage == NST) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                // ---- the next unit
                if (!dyn) {
                    u += num_pairs;
                } else {
                    int32_t nx = -1;
                    if (!ended) {
                        if (rank != 0 && lane == 0) mbar_arrive_expect_tx(clc_bar(answered), 16);  // this CTA's copy
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait(clc_bar(answered), (answered / pair::NCLC) & 1u, p.wait))) {
                            ok = false;
                            break;
                        }
                        const int32_t x = clc_cancelled_ctaid_x(clc_resp(answered));
                        ++answered;
                        nx = x < 0 ? -1 : (x >> 1);  // a failed request ends the sequence: ask no more
                        ended = nx < 0;
                        if (rank == 0 && nx >= 0) request();
                    }
                    publish(uint32_t(it) + 1, nx);
                    u = nx;
                }
            }
            if (lane == 0) {
                // no cancellation answer may still be on its way into shared memory
                for (uint32_t i = answered; i < requested; ++i)
                    mbar_wait_slow(clc_bar(i), (i / pair::NCLC) & 1u, cleanup_wait(p.wait), false);
                if (!ok) {
                    if (rank == 0) {
                        // Let the copies counted on this CTA's barriers land before exiting.
                        const uint32_t n = issued < NST ? issued : NST;
                        for (uint32_t q = issued - n; q < issued; ++q)
                            mbar_wait_slow(full_bar(q % NST), (q / NST) & 1u,
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
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        if (kTmaLoad && rank == 1 && p.relay) {
            // ======================================================== relay (CTA 1, TMA loads)
            // Once all of this CTA's epilogue warps have drained a unit's
            // accumulator (local arrivals), one release at cluster scope tells CTA
            // 0's MMA warp, instead of one such arrival per epilogue warp (each
            // costs its warp a cluster-scope fence on the drain's critical path).
            int32_t it = 0;
            for (int32_t u = pair_id; (!kDyn || u >= 0) && u < p.num_units; ++it) {
                const uint32_t acc = it & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(tdone_bar(acc), (uint32_t(it) >> 1) & 1u, p.wait))) break;
                if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
                __syncwarp();
                if constexpr (kDyn) {
                    if (!__all_sync(0xffffffffu, next_unit(uint32_t(it), u))) break;
                } else {
                    u += num_pairs;
                }
            }
        }
        if (!kTmaLoad && rank == 1) {
            // ======================================================== relay (CTA 1, predicated loads)
            // Once this CTA's loader warps have filled a stage, one release at
            // cluster scope hands it to CTA 0's full barrier.
            uint32_t stage = 0, phase = 0;
            const uint32_t full0 = mapa_shared(full_bar(0), 0);
            for (int32_t u = pair_id; u < p.num_units; u += num_pairs) {
                const int32_t kb0 = (u / p.num_tiles) * p.kb_per_split;
                const int32_t kb1 = min(num_kb, kb0 + p.kb_per_split);
                bool ok = true;
                for (int32_t kb = kb0; kb < kb1; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(bar0 + 8u * (Lay::placed_bar0 + stage), phase, p.wait))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_cluster(full0 + 8u * stage);
                    __syncwarp();
                    if (++stage == NST) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
        }
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
            for (int32_t u = pair_id; ok && (!kDyn || u >= 0) && u < p.num_units; ++it) {
                int32_t kb0 = (u / p.num_tiles) * p.kb_per_split;
                int32_t kb1 = min(num_kb, kb0 + p.kb_per_split);
                if constexpr (kTail) {
                    int32_t tile = 0, slot;
                    tail_unit(p, u, tile, kb0, kb1, slot);
                }
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
                    // predicated loads: arrivals from the peer CTA's loader warps,
                    // acquired at cluster scope
                    const bool full = kTmaLoad ? mbar_wait(full_bar(stage), phase, p.wait)
                                               : mbar_wait_cluster(full_bar(stage), phase, p.wait);
                    if (!__all_sync(0xffffffffu, full)) {
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
                    if (++stage == NST) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair_mc_elect(tfull_bar(acc), 0x3);  // both halves of the tile complete
                if constexpr (kDyn) {
                    if (!__all_sync(0xffffffffu, next_unit(uint32_t(it), u))) {
                        ok = false;
                        break;
                    }
                } else {
                    u += num_pairs;
                }
            }
            mma_commit_pair_elect(drain_bar);
            __all_sync(0xffffffffu, mbar_wait_slow(drain_bar, 0, cleanup_wait(p.wait), false));
        }
    } else {
        // ============================================================ epilogue (both CTAs)
        const int q = warp & 3;
        const int ew = warp - EPI_WARP0;
        const int half = ew / 4;
        const uint32_t stg = base + Lay::off_epi + uint32_t(ew) * (EPI_BUFS * EPI_BUF_BYTES);
        int32_t it = 0;
        for (int32_t u = pair_id; (!kDyn || u >= 0) && u < p.num_units; ++it) {
            int32_t tile = u % p.num_tiles, split = u / p.num_tiles;
            int32_t kb0 = split * p.kb_per_split;
            int32_t kb1 = min(num_kb, kb0 + p.kb_per_split);
            int32_t slot = -1;
            if constexpr (kTail) tail_unit(p, u, tile, kb0, kb1, slot);
            const int32_t unit_kb = kb1 - kb0;
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
                    if (rank == 0) {
                        mbar_arrive(tempty_bar(acc));  // the MMA warp is in this CTA
                    } else if (!p.relay) {
                        mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
                    } else if constexpr (!kTmaLoad) {
                        // predicated loads (CTA 1's MMA warp relays the loaders' stages):
                        // the last of this CTA's epilogue warps to drain the unit makes
                        // the one cluster-scope arrive, having acquired the others' releases
                        if ((atom_add_acq_rel_cta(drained_ctr + 4u * acc, 1u) + 1u) % uint32_t(EPI_WARPS) == 0)
                            mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
                    }
                }
            };
            const int64_t col_base = int64_t(tn) * pair::TILE_N;
            // no unit follows (dynamic units: if already published)
            bool last;
            if constexpr (kDyn)
                last = __shfl_sync(0xffffffffu, known_end(uint32_t(it) + 1, u) ? 1 : 0, 0) != 0;
            else
                last = u + num_pairs >= p.num_units;
            int c0, n;
            if (kTail && slot >= 0) {  // partial tile of the split tail -> scratch slot, fp32
                const TailStore ts{&tmW, int32_t(slot * pair::TILE_M + int32_t(rank) * pair::CTA_M + q * 32),
                                   col_base};
                epilogue_chunks(unit_kb, last, half, EPI_CHUNKS32, c0, n);
                epilogue_tile<kTmaStore>(t_row, row0, col_base, c0, n, p, &tmC, stg, lane, release, 0, &ts);
            } else if (p.out_dtype == 0 || p.splits > 1) {  // split-K partials are fp32
                epilogue_chunks(unit_kb, last, half, EPI_CHUNKS32, c0, n);
                if (kClassStore && col_base + pair::TILE_N <= p.N) {
                    epilogue_tile_class(t_row, row0, col_base, c0, n, p, cm_c(cm), stg, lane, release);
                } else {
                    if (kClassStore) {  // the plain path reuses the buffer the class stores may still read
                        if (lane < int(p.c_classes)) bulk_wait_group_read<0>();
                        __syncwarp();
                    }
                    epilogue_tile<kTmaStore>(t_row, row0, col_base, c0, n, p, &tmC, stg, lane, release, split);
                }
            } else {
                epilogue_chunks(unit_kb, last, half, EPI_CHUNKS16, c0, n);
                epilogue_tile16<kTmaStore>(t_row, row0, col_base, c0, n, p, &tmC, stg, lane, release);
            }
            if constexpr (kDyn) {
                if (!__all_sync(0xffffffffu, next_unit(uint32_t(it), u))) break;
            } else {
                u += num_pairs;
            }
        }
        if ((kTmaStore && lane == 0) || (kClassStore && lane < int(p.c_classes))) bulk_wait_group<0>();
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
