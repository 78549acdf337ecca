// Host side of the gemm_f16 C ABI (declared in include/gemm_f16.h): argument
// validation, layout/path selection, TMA tensor-map encoding and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <numeric>
#include <utility>

#include "gemm_f16.h"
#include "gemm_kernel.cuh"
#include "gemm_pair.cuh"

namespace {

using namespace g16;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<uint32_t> g_epoch{0};

// Per-device set-up, done by the first call on a device that succeeds; a call
// whose set-up fails returns the error and the next call tries again.
struct DeviceState {
    std::mutex mu;
    std::atomic<bool> ready{false};
    int num_sms = 0;
    int max_pairs = 0;       // co-resident 2-CTA clusters of the pair kernel (TMA loads)
    int max_pairs_pred = 0;  // the same for its predicated-load variant
};
DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

bool log_enabled() {
    static const bool on = [] {
        const char *e = std::getenv("GEMM_LOG");
        return e != nullptr && e[0] != '\0' && e[0] != '0';
    }();
    return on;
}

template <bool L, bool S>
cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(gemm_f16_persistent<L, S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Layout<L>::smem_bytes);
}

template <bool L, bool S, bool D = false, bool T = false, bool K = false>
cudaError_t set_pair_smem_attr() {
    return cudaFuncSetAttribute(gemm_f16_pair<L, S, D, T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                pair::Layout<L>::smem_bytes);
}

// How many 2-CTA clusters of the pair kernel (TMA-load variant L = true, or
// predicated-load variant) fit on the device at once.
template <bool L>
int query_max_pairs(int num_sms) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(pair::Layout<L>::threads, 1, 1);
    cfg.dynamicSmemBytes = pair::Layout<L>::smem_bytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_f16_pair<L, true>, &cfg) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = num_sms / 2;
    }
    return n;
}

cudaError_t device_init(int dev, DeviceState **out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    DeviceState &d = g_dev[dev];
    *out = &d;
    if (d.ready.load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(d.mu);
    if (d.ready.load(std::memory_order_relaxed)) return cudaSuccess;
    int num_sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = set_smem_attr<true, true>();
    if (e == cudaSuccess) e = set_smem_attr<true, false>();
    if (e == cudaSuccess) e = set_smem_attr<false, true>();
    if (e == cudaSuccess) e = set_smem_attr<false, false>();
    if (e == cudaSuccess) e = set_pair_smem_attr<true, true>();
    if (e == cudaSuccess) e = set_pair_smem_attr<true, false>();
    if (e == cudaSuccess) e = set_pair_smem_attr<false, true>();
    if (e == cudaSuccess) e = set_pair_smem_attr<false, false>();
    if (e == cudaSuccess) e = set_pair_smem_attr<true, true, true>();
    if (e == cudaSuccess) e = set_pair_smem_attr<true, false, true>();
    if (e == cudaSuccess) e = set_pair_smem_attr<true, true, false, true>();
    if (e == cudaSuccess) e = set_pair_smem_attr<true, false, false, false, true>();
    if (e == cudaSuccess) e = set_pair_smem_attr<false, false, false, false, true>();
    if (e != cudaSuccess) {
        (void)cudaGetLastError();  // not sticky: leave no error behind for the caller's next call
        return e;
    }
    d.num_sms = num_sms;
    d.max_pairs = query_max_pairs<true>(num_sms);
    d.max_pairs_pred = query_max_pairs<false>(num_sms);
    d.ready.store(true, std::memory_order_release);
    return cudaSuccess;
}

EncodeTiledFn encode_fn() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

// 2-D tiled tensor map, inner dimension first, 128-byte swizzle, OOB -> zero.
bool encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner,
               uint64_t outer, uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {outer_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Alignment classes of one operand for the predicated-load kernel: `rows` rows
// of `cols` contiguous fp16 elements, row rho starting at X + 2*S*rho bytes.
// Rows with rho mod P == c share their offset m_c inside a 16-byte granule and
// are 2*S*P bytes apart (a multiple of 16), so class c is one tensor map whose
// rows start m_c bytes early, at the granule boundary, and whose width grows by
// m_c/2 elements. Every byte TMA reads through these maps therefore shares its
// granule with an element of the operand. Returns false if a map is rejected.
bool encode_classes(CUtensorMap *maps, const void *X, int64_t S, int64_t rows, int64_t cols, bool mn_major,
                    uint32_t *lp_out, uint32_t *lh_out, uint32_t *mis, uint32_t *live) {
    const uint64_t r = (2u * uint64_t(S)) % 16u;
    const uint64_t P = r == 0 ? 1u : 16u / std::gcd(r, uint64_t(16));
    const int lp = __builtin_ctzll(P);
    const int lh = class_box_lh(mn_major, lp);
    *lp_out = uint32_t(lp);
    *lh_out = uint32_t(lh);
    *mis = 0;
    *live = 0;
    for (uint64_t c = 0; c < P; ++c) {
        if (uint64_t(rows) <= c) continue;  // no row in this class: its lines are placed as zeros
        const uint64_t nrows = (uint64_t(rows) - c + P - 1) / P;
        const uintptr_t a = reinterpret_cast<uintptr_t>(X) + 2u * uint64_t(S) * c;
        const uint32_t m = uint32_t(a & 15u);
        if (!encode_2d(&maps[c], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, reinterpret_cast<const void *>(a - m),
                       uint64_t(cols) + m / 2u, nrows, 2u * uint64_t(S) * P, BOX_W, 1u << lh,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
        *mis |= m << (4u * c);
        *live |= 1u << c;
    }
    return true;
}

// 3-D tiled tensor map (inner first) with a box of depth 1 in the outermost
// dimension: the split-K workspace [S][M][ldw], so that TMA clips each slice on
// its own M and N edges.
bool encode_3d_f32(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// TMA can describe an operand whose contiguous extent is `inner` and whose other
// stride is `outer_stride` elements of `esize` bytes.
bool tma_ok(const void *p, int64_t inner, int64_t outer_stride, int esize) {
    return aligned16(p) && (outer_stride * esize) % 16 == 0 && outer_stride >= inner &&
           outer_stride * esize < (int64_t(1) << 40);
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Launches a kernel of a GEMM call with programmatic stream serialization
// allowed: its CTAs may be scheduled while the kernel before it on the stream
// is finishing (once that kernel's CTAs have all called
// griddepcontrol.launch_dependents, or ended), run their set-up, and wait in
// griddepcontrol.wait, before their first global-memory access, until that
// kernel has completed and its writes are visible. Memory ordering on the
// stream is the same as for a plain launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), int grid, int threads, int smem, cudaStream_t stream,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(unsigned(threads), 1, 1);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e;
}

template <bool L, bool S>
cudaError_t launch(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c, const Params &p,
                   const ClassMaps &cm, int grid, cudaStream_t stream) {
    if constexpr (L)
        return launch_overlapped(gemm_f16_persistent<L, S>, grid, cta_threads(L), Layout<L>::smem_bytes, stream, a, b,
                                 c, p, NoClassMaps{});
    else
        return launch_overlapped(gemm_f16_persistent<L, S>, grid, cta_threads(L), Layout<L>::smem_bytes, stream, a, b,
                                 c, p, cm);
}

template <bool L, bool S, bool D = false, bool T = false>
cudaError_t launch_pair(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c, const CUtensorMap &w,
                        const Params &p, const ClassMaps &cm, int grid, cudaStream_t stream) {
    constexpr int threads = pair::Layout<L>::threads, smem = pair::Layout<L>::smem_bytes;
    if constexpr (L)
        return launch_overlapped(gemm_f16_pair<L, S, D, T>, grid, threads, smem, stream, a, b, c, w, p,
                                 NoClassMaps{});
    else
        return launch_overlapped(gemm_f16_pair<L, S>, grid, threads, smem, stream, a, b, c, w, p, cm);
}

// The CTA-pair kernel with C stored per row class (plain-store C, static order).
template <bool L>
cudaError_t launch_pair_class(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &w, const Params &p,
                              const ClassMaps &cm, const CClassMaps &cc, int grid, cudaStream_t stream) {
    constexpr int threads = pair::Layout<L>::threads, smem = pair::Layout<L>::smem_bytes;
    if constexpr (L) {
        return launch_overlapped(gemm_f16_pair<L, false, false, false, true>, grid, threads, smem, stream, a, b, w, w,
                                 p, cc);
    } else {
        ClassMapsAndC all;
        std::memcpy(all.a, cm.a, sizeof(all.a));
        std::memcpy(all.b, cm.b, sizeof(all.b));
        std::memcpy(all.c, cc.c, sizeof(all.c));
        return launch_overlapped(gemm_f16_pair<L, false, false, false, true>, grid, threads, smem, stream, a, b, w, w,
                                 p, all);
    }
}

// Row classes of an fp32 C that TMA cannot store as one map (see
// epilogue_tile_class): P classes by the row stride, one map each whose rows
// begin at the 16-byte boundary below the row starts and whose inner extent
// ends on a granule at or before column N. Returns P, or 0 if C does not take
// class stores (too small, or a map is rejected).
uint32_t encode_c_classes(CClassMaps *cc, void *C, int64_t M, int64_t N, int64_t ldc) {
    const int64_t d = ldc % 4;
    const uint32_t P = d == 0 ? 1u : d == 2 ? 2u : 4u;
    if (M < int64_t(P) || N < 8 || (reinterpret_cast<uintptr_t>(C) & 3u)) return 0;
    if (uint64_t(P) * uint64_t(ldc) * 4u >= (uint64_t(1) << 40)) return 0;
    std::memset(cc, 0, sizeof(*cc));
    for (uint32_t q = 0; q < P; ++q) {
        const uintptr_t row = reinterpret_cast<uintptr_t>(C) + uint64_t(q) * uint64_t(ldc) * 4u;
        const uint32_t m = uint32_t((row >> 2) & 3u);
        const uint64_t inner = (uint64_t(N) + m) / 4u * 4u;
        const uint64_t rows = (uint64_t(M) - q + P - 1) / P;
        if (!encode_2d(&cc->c[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, reinterpret_cast<const void *>(row - 4u * m),
                       inner, rows, uint64_t(P) * uint64_t(ldc) * 4u, EPI_COLS, 32u / P))
            return 0;
    }
    return P;
}

void tile_shape(uint32_t flags, int *bm, int *bn) {
    const bool single = (flags & GEMM_SCHED_SINGLE_CTA) != 0;
    *bm = single ? BM : pair::TILE_M;
    *bn = single ? BN : pair::TILE_N;
}

// Split-K plan: kb_per_split k-blocks per slice and the number of non-empty
// slices. `requested` == 0 picks enough slices to give every co-resident CTA
// pair a unit (at most 32, at least one k-block per slice).
struct SplitPlan {
    int32_t splits;
    int32_t kb_per_split;
    int64_t ldw;  // workspace row stride (elements), N rounded up to 4
};

SplitPlan plan_splits(int64_t M, int64_t N, int64_t K, int32_t requested, int max_pairs) {
    SplitPlan sp;
    const int64_t num_kb = cdiv(K, BK);
    const int64_t tiles = cdiv(M, pair::TILE_M) * cdiv(N, pair::TILE_N);
    int64_t want = requested;
    if (want <= 0) want = tiles >= max_pairs ? 1 : cdiv(max_pairs, tiles);
    if (want > 32) want = 32;
    if (want > num_kb) want = num_kb;
    if (want < 1) want = 1;
    sp.kb_per_split = int32_t(cdiv(num_kb, want));
    sp.splits = int32_t(cdiv(num_kb, sp.kb_per_split));
    sp.ldw = (N + 3) / 4 * 4;
    return sp;
}

// Device address of a file-scope __device__ array on the current device. In
// host code the array's name is only a stand-in, so the address is looked up
// with the device current, and kept only once a lookup succeeds (a failed one,
// say during a stream capture, returns nullptr and the next call retries).
struct SymbolAddress {
    std::mutex mu;
    std::atomic<void *> ptr{nullptr};
};

template <typename T>
void *symbol_address(SymbolAddress &s, const T &symbol) {
    void *p = s.ptr.load(std::memory_order_acquire);
    if (p != nullptr) return p;
    std::lock_guard<std::mutex> lock(s.mu);
    p = s.ptr.load(std::memory_order_relaxed);
    if (p != nullptr) return p;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return nullptr;
    }
    s.ptr.store(p, std::memory_order_release);
    return p;
}

// Split tail (GEMM_SCHED_TAIL_SPLIT): scratch for the fp32 partial tiles of a
// split last round, built into the library (every GPU that loads it holds it).
constexpr uint64_t kTailScratchBytes = 24ull << 20;
constexpr uint64_t kTailTileBytes = uint64_t(pair::TILE_M) * pair::TILE_N * 4;  // 256 KiB
constexpr int64_t kTailSlots = int64_t(kTailScratchBytes / kTailTileBytes);     // 96 partial tiles
static __device__ __align__(256) unsigned char g_tail_scratch[kTailScratchBytes];
SymbolAddress g_tail_addr[kMaxDevices];

struct TailPlan {
    int32_t first = 0, tiles = 0, splits = 1, kps = 0;
};

// The last round of the static tile stream tile_id = pid + i * P, when it
// would leave at least three quarters of the P programs idle: its tiles are
// split along K into as many slices (at least two) as the idle programs and
// the scratch allow, each of at least kTailMinKb k-blocks, so that the round
// takes a fraction of a tile's time. Measured on GB300 (device-timed loops):
// 4000 x 5000 x 3000 (16 tiles of 76 in the last round) 108.8 -> 105.6 us;
// with a fuller last round (8192^2 x 4096: 36 of 76) the second pass cost more
// than it saved (320 -> 326 us), since the SMs that sit out a partial round let
// the busy ones clock higher under the power limit; for short problems (512^3)
// the second launch dominates.
constexpr int64_t kTailMinKb = 8;

TailPlan plan_tail(int64_t num_tiles, int64_t num_kb, int64_t programs) {
    TailPlan t;
    const int64_t rest = num_tiles % programs;
    if (rest == 0 || 4 * rest > programs) return t;
    int64_t S = programs / rest;
    if (S > kTailSlots / rest) S = kTailSlots / rest;
    if (S > num_kb / kTailMinKb) S = num_kb / kTailMinKb;
    if (S < 2) return t;
    const int64_t kps = cdiv(num_kb, S);
    S = cdiv(num_kb, kps);  // no empty slice
    if (S < 2) return t;
    t.first = int32_t(num_tiles - rest);
    t.tiles = int32_t(rest);
    t.splits = int32_t(S);
    t.kps = int32_t(kps);
    return t;
}

uint32_t next_epoch() {
    uint32_t e = g_epoch.fetch_add(1) + 1;
    if (e == 0) e = g_epoch.fetch_add(1) + 1;  // 0 means "no abort"
    return e;
}

}  // namespace

extern "C" {

const char *gemm_f16_status_str(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
        case GEMM_ERR_CHECK: return "GEMM_ERR_CHECK";
    }
    return "GEMM_ERR_UNKNOWN";
}

gemm_status_t gemm_f16_set_wait_timeout(uint64_t ns) {
    if (ns < 1000) return GEMM_ERR_INVALID_ARG;
    g_timeout_ns.store(ns);
    return GEMM_OK;
}

}  // extern "C"

namespace {

// Split-K request of one call: requested slices (0 = automatic) and the
// caller's fp32 workspace.
struct SplitReq {
    bool enabled = false;
    int32_t splits = 1;
    void *workspace = nullptr;
    uint64_t workspace_bytes = 0;
    int32_t stop_after = 0;  // failure-detection self-test (gemm_f16_selftest_pair_abort)
};

// Operand copies of one gemm_f16_packed call: the caller's workspace.
struct PackReq {
    bool enabled = false;
    void *workspace = nullptr;
    uint64_t workspace_bytes = 0;
};

// One operand's row layout: `rows` rows of `inner` contiguous elements, `ld`
// elements apart (from the strides as gemm_impl classifies them).
struct OperandRows {
    int64_t rows, inner, ld;
};

OperandRows rows_of_a(int64_t M, int64_t K, int64_t stride_am, int64_t stride_ak) {
    if (stride_ak == 1) return {M, K, stride_am};  // K-major
    return {K, M, stride_ak};                      // M-major
}

OperandRows rows_of_b(int64_t N, int64_t K, int64_t stride_bk, int64_t stride_bn) {
    if (stride_bn == 1) return {K, N, stride_bk};  // N-major
    return {N, K, stride_bn};                      // K-major
}

// Elements per row of an operand's copy: whole 128-byte lines.
int64_t packed_ld(int64_t inner) { return (inner + 63) / 64 * 64; }

uint64_t packed_bytes(const OperandRows &o) { return uint64_t(o.rows) * uint64_t(packed_ld(o.inner)) * 2u; }

uint64_t round256(uint64_t x) { return (x + 255u) / 256u * 256u; }

// TMA reads every 64-element row of a K-block as one whole 128-byte line only
// when the base and the row stride are multiples of 128 bytes.
bool rows_on_lines(const void *p, const OperandRows &o) {
    return (reinterpret_cast<uintptr_t>(p) & 127u) == 0 && (o.ld * 2) % 128 == 0 && o.ld >= o.inner;
}

gemm_status_t gemm_impl(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                        int64_t stride_am, int64_t stride_ak, int64_t stride_bk, int64_t stride_bn,
                        int64_t stride_cm, int64_t stride_cn, int32_t group_size_m,
                        uint32_t schedule_flags, gemm_stream_t stream_, const SplitReq &sk,
                        uint32_t out_dtype = GEMM_OUT_F32, float alpha = 1.0f, const PackReq &pk = PackReq()) {
    if (out_dtype > GEMM_OUT_BF16) return GEMM_ERR_INVALID_ARG;
    const int esize = out_dtype == GEMM_OUT_F32 ? 4 : 2;
    // ---- validation (no GPU work before this point)
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return GEMM_ERR_INVALID_ARG;
    if (stride_am < 1 || stride_ak < 1 || stride_bk < 1 || stride_bn < 1 || stride_cm < 1 ||
        stride_cn < 1)
        return GEMM_ERR_INVALID_ARG;
    if (schedule_flags & ~GEMM_SCHED_ALL_FLAGS) return GEMM_ERR_INVALID_ARG;
    const bool grouped = (schedule_flags & GEMM_SCHED_GROUPED) != 0;
    if (grouped && group_size_m < 1) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))) return GEMM_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 1u) ||
        (reinterpret_cast<uintptr_t>(C) & uintptr_t(esize - 1)))
        return GEMM_ERR_INVALID_ARG;  // not aligned to the element size
    if (stride_cn != 1) return GEMM_ERR_UNSUPPORTED;
    if (M > 1 && stride_cm < N) return GEMM_ERR_INVALID_ARG;  // C rows would overlap

    const bool a_k = stride_ak == 1, a_m = !a_k && stride_am == 1;
    const bool b_n = stride_bn == 1, b_k = !b_n && stride_bk == 1;
    if (K > 0 && (!(a_k || a_m) || !(b_n || b_k))) return GEMM_ERR_UNSUPPORTED;

    // gemm_f16_packed: the workspace holds both copies (checked before any GPU work)
    const OperandRows pk_a = rows_of_a(M, K, stride_am, stride_ak);
    const OperandRows pk_b = rows_of_b(N, K, stride_bk, stride_bn);
    const uint64_t pk_off_b = round256(packed_bytes(pk_a));
    if (pk.enabled && K > 0 &&
        (pk.workspace == nullptr || (reinterpret_cast<uintptr_t>(pk.workspace) & 127u) ||
         pk.workspace_bytes < pk_off_b + packed_bytes(pk_b)))
        return GEMM_ERR_INVALID_ARG;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    DeviceState *ds = nullptr;
    if (device_init(dev, &ds) != cudaSuccess) return GEMM_ERR_CUDA;

    if (K == 0) {
        const int64_t total = M * N;
        const int threads = 256;
        const int64_t blocks64 = cdiv(total, threads);
        const int blocks = int(blocks64 < 8 * int64_t(ds->num_sms) ? blocks64 : 8 * int64_t(ds->num_sms));
        zero_c_kernel<<<blocks, threads, 0, stream>>>(C, M, N, stride_cm, esize);
        return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }

    // ---- operand copies into whole 128-byte lines (gemm_f16_packed)
    if (pk.enabled) {
        const OperandRows &ra = pk_a, &rb = pk_b;
        uint16_t *wa = static_cast<uint16_t *>(pk.workspace);
        uint16_t *wb = reinterpret_cast<uint16_t *>(static_cast<unsigned char *>(pk.workspace) + pk_off_b);
        auto job = [](const void *src, const OperandRows &o, uint16_t *dst, bool copy) {
            PackJob j;
            j.src = static_cast<const uint16_t *>(src);
            j.dst = dst;
            j.rows = o.rows;
            j.inner = o.inner;
            j.ld_src = o.ld;
            j.ld_dst = packed_ld(o.inner);
            j.gpr = (o.inner + 7) / 8;
            j.granules = copy ? o.rows * j.gpr : 0;
            return j;
        };
        const bool copy_a = !rows_on_lines(A, ra), copy_b = !rows_on_lines(B, rb);
        const PackJob ja = job(A, ra, wa, copy_a), jb = job(B, rb, wb, copy_b);
        const int64_t total = ja.granules + jb.granules;
        if (total > 0) {
            const int threads = 256;
            const int64_t want = cdiv(total, threads);
            const int blocks = int(want < 8 * int64_t(ds->num_sms) ? want : 8 * int64_t(ds->num_sms));
            if (launch_overlapped(pack_rows_kernel, blocks, threads, 0, stream, ja, jb) != cudaSuccess)
                return GEMM_ERR_CUDA;
        }
        if (copy_a) {
            A = wa;
            if (a_k) stride_am = packed_ld(ra.inner);
            else stride_ak = packed_ld(ra.inner);
        }
        if (copy_b) {
            B = wb;
            if (b_n) stride_bk = packed_ld(rb.inner);
            else stride_bn = packed_ld(rb.inner);
        }
    }

    // ---- path selection per tensor
    const bool a_tma = a_k ? tma_ok(A, K, stride_am, 2) : tma_ok(A, M, stride_ak, 2);
    const bool b_tma = b_n ? tma_ok(B, N, stride_bk, 2) : tma_ok(B, K, stride_bn, 2);
    const bool load_tma = a_tma && b_tma;
    // A TMA store clipped inside a 16-byte granule writes the whole granule
    // (measured: an fp32 C with N = 513 inside rows of 520 had columns 513..515
    // overwritten), so C goes through TMA only when its rows end on a granule;
    // a view with N mod 4 (fp32) or N mod 8 (16-bit) != 0 takes plain stores.
    const bool store_tma = tma_ok(C, N, stride_cm, esize) && (N * esize) % 16 == 0;
    // CTA pairs need TMA loads (both CTAs' copies count on one barrier)
    const bool use_pair = !(schedule_flags & GEMM_SCHED_SINGLE_CTA);
    if (sk.enabled && !(use_pair && load_tma)) return GEMM_ERR_UNSUPPORTED;  // split-K: CTA pairs, TMA loads
    const int tile_m = use_pair ? pair::TILE_M : BM;
    const int tile_n = use_pair ? pair::TILE_N : BN;
    const int cta_m = use_pair ? pair::CTA_M : BM;    // A rows one CTA loads
    const int cta_n = use_pair ? pair::CTA_N : BN;    // B columns one CTA loads
    const int64_t nm = cdiv(M, tile_m), nn = cdiv(N, tile_n);
    if (nm * nn > kMaxDim) return GEMM_ERR_UNSUPPORTED;

    CUtensorMap tmA, tmB, tmC, tmW;
    std::memset(&tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    std::memset(&tmC, 0, sizeof(tmC));
    std::memset(&tmW, 0, sizeof(tmW));
    if (load_tma) {
        const bool okA = a_k ? encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, K, M, stride_am * 2, BK,
                                         cta_m)
                             : encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, M, K, stride_ak * 2,
                                         MN_CHUNK, BK);
        const bool okB = b_k ? encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, K, N, stride_bn * 2, BK,
                                         cta_n)
                             : encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, N, K, stride_bk * 2,
                                         MN_CHUNK, BK);
        if (!okA || !okB) return GEMM_ERR_CUDA;
    }
    static_assert(sizeof(ClassMaps) == 2 * MAX_CLASSES * sizeof(CUtensorMap), "");
    ClassMaps cm;
    std::memset(&cm, 0, sizeof(cm));
    uint32_t cls_lp[2] = {0, 0}, cls_lh[2] = {4, 4}, cls_mis[2] = {0, 0}, cls_live[2] = {0, 0};
    if (!load_tma) {
        const bool okA = a_k ? encode_classes(cm.a, A, stride_am, M, K, false, &cls_lp[0], &cls_lh[0], &cls_mis[0],
                                              &cls_live[0])
                             : encode_classes(cm.a, A, stride_ak, K, M, true, &cls_lp[0], &cls_lh[0], &cls_mis[0],
                                              &cls_live[0]);
        const bool okB = b_n ? encode_classes(cm.b, B, stride_bk, K, N, true, &cls_lp[1], &cls_lh[1], &cls_mis[1],
                                              &cls_live[1])
                             : encode_classes(cm.b, B, stride_bn, N, K, false, &cls_lp[1], &cls_lh[1], &cls_mis[1],
                                              &cls_live[1]);
        if (!okA || !okB) return GEMM_ERR_UNSUPPORTED;
    }
    SplitPlan sp{1, int32_t(cdiv(K, BK)), N};
    if (sk.enabled) {
        sp = plan_splits(M, N, K, sk.splits, ds->max_pairs);
        if (sp.splits > 1) {
            const uint64_t need = uint64_t(sp.splits) * uint64_t(M) * uint64_t(sp.ldw) * 4u;
            if (sk.workspace == nullptr || sk.workspace_bytes < need || !aligned16(sk.workspace))
                return GEMM_ERR_INVALID_ARG;
            if (!encode_3d_f32(&tmC, sk.workspace, uint64_t(N), uint64_t(M), uint64_t(sp.splits),
                               uint64_t(sp.ldw) * 4u, uint64_t(M) * uint64_t(sp.ldw) * 4u, EPI_COLS, 32))
                return GEMM_ERR_CUDA;
        }
    }
    const bool split = sp.splits > 1;
    if (!split && store_tma) {
        const CUtensorMapDataType dt = out_dtype == GEMM_OUT_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : out_dtype == GEMM_OUT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        // one 128-byte row of the box: 32 fp32 or 64 16-bit elements, 32 rows
        if (!encode_2d(&tmC, dt, C, N, M, stride_cm * esize, 128 / esize, 32)) return GEMM_ERR_CUDA;
    }

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.A = static_cast<const uint16_t *>(A);
    p.B = static_cast<const uint16_t *>(B);
    p.C = static_cast<float *>(C);
    // split-K: the GEMM writes fp32 partials; the reduction scales and rounds
    p.out_dtype = split ? uint32_t(GEMM_OUT_F32) : out_dtype;
    p.alpha = split ? 1.0f : alpha;
    p.M = M;
    p.N = N;
    p.K = K;
    p.sam = stride_am;
    p.sak = stride_ak;
    p.sbk = stride_bk;
    p.sbn = stride_bn;
    p.scm = stride_cm;
    p.sched.nm = int32_t(nm);
    p.sched.nn = int32_t(nn);
    p.sched.group_m = grouped ? group_size_m : 1;
    p.sched.grouped = grouped ? 1 : 0;
    p.num_tiles = int32_t(nm * nn);
    p.num_kb = int32_t(cdiv(K, BK));
    p.splits = sp.splits;
    p.kb_per_split = split ? sp.kb_per_split : p.num_kb;
    if (int64_t(p.num_tiles) * sp.splits > kMaxDim) return GEMM_ERR_UNSUPPORTED;
    p.num_units = p.num_tiles * sp.splits;
    p.a_mn = a_k ? 0u : 1u;
    p.b_mn = b_n ? 1u : 0u;
    p.idesc = make_idesc(p.a_mn, p.b_mn, use_pair ? 2 * pair::CTA_M : BM, tile_n);
    p.cross_tile = (schedule_flags & GEMM_SCHED_CROSS_TILE) ? 1u : 0u;
    for (int op = 0; op < 2; ++op) {
        p.cls_lp[op] = cls_lp[op];
        p.cls_lh[op] = cls_lh[op];
        p.cls_mis[op] = cls_mis[op];
        p.cls_live[op] = cls_live[op];
    }
    if (!use_pair) {  // the one-CTA kernel walks whole tiles
        p.splits = 1;
        p.kb_per_split = p.num_kb;
        p.num_units = p.num_tiles;
    }
    // C is written once and never read again: its stores carry an evict-first
    // L2 policy. Operand loads keep the default policy (an evict-last hint on
    // them measured slower: tensor-pipe activity 86.3 % -> 83.7 % at 16384^2).
    p.l2_mode = 1u;
    p.wait.timeout_ns = g_timeout_ns.load();
    p.wait.epoch = next_epoch();
    p.stop_after = sk.stop_after;

    // dynamic units: one cluster per unit in the grid; the resident clusters take
    // the others' units through cluster launch control (CTA pairs with TMA loads)
    const bool dynamic = (schedule_flags & GEMM_SCHED_DYNAMIC) && use_pair && load_tma;
    p.dynamic = dynamic ? 1u : 0u;
    // CTA 1's epilogue warps report a drained accumulator to CTA 0 with one
    // cluster-scope arrive per unit: from CTA 1's MMA warp, idle with TMA loads,
    // or (predicated loads) from the last of the warps to finish. The per-warp
    // arrivals this replaces cost 16384^2 x 512 253 -> 228 us and x 128 183 ->
    // 167 us with TMA loads, 8191^2 x 257 134 -> 133 us with predicated loads
    // (device-timed on GB300, bit-identical C).
    p.relay = use_pair ? 1u : 0u;
    const bool persistent = !(schedule_flags & GEMM_SCHED_NON_PERSISTENT) && !dynamic;
    const int programs = !persistent ? p.num_units
                         : use_pair  ? (load_tma ? ds->max_pairs : ds->max_pairs_pred)
                                     : ds->num_sms;
    p.tail_first = p.num_units;  // no split tail
    p.tail_tiles = 1;
    p.tail_kps = p.num_kb;
    TailPlan tp;
    if ((schedule_flags & GEMM_SCHED_TAIL_SPLIT) && use_pair && load_tma && store_tma && !sk.enabled &&
        persistent)
        tp = plan_tail(p.num_tiles, p.num_kb, programs);
    void *tail_ws = nullptr;
    if (tp.splits > 1) {
        tail_ws = symbol_address(g_tail_addr[dev], g_tail_scratch);
        if (tail_ws == nullptr) return GEMM_ERR_CUDA;
        // slot v: rows [256 v, 256 v + 256) of a 256-column fp32 matrix
        if (!encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, tail_ws, pair::TILE_N,
                       uint64_t(tp.splits) * tp.tiles * pair::TILE_M, pair::TILE_N * 4u, EPI_COLS, 32))
            return GEMM_ERR_CUDA;
        p.tail_first = tp.first;
        p.tail_tiles = tp.tiles;
        p.tail_kps = tp.kps;
        p.num_units = tp.first + tp.splits * tp.tiles;
    }
    // fp32 C that TMA cannot store as one map: per row class (CTA pairs, static order)
    CClassMaps cc;
    std::memset(&cc, 0, sizeof(cc));
    if (use_pair && !store_tma && !split && tp.splits <= 1 && !dynamic && out_dtype == GEMM_OUT_F32)
        p.c_classes = encode_c_classes(&cc, C, M, N, stride_cm);
    const int grid_programs = int(p.num_units < programs ? p.num_units : programs);
    if (use_pair && int64_t(grid_programs) * 2 > kMaxDim) return GEMM_ERR_UNSUPPORTED;
    const int grid = use_pair ? 2 * grid_programs : grid_programs;
    if (log_enabled())
        std::fprintf(stderr,
                     "[gemm_f16] M=%lld N=%lld K=%lld kernel=%s tiles=%d grid=%d load=%s store=%s A=%s "
                     "B=%s order=%s G=%d cross_tile=%u persistent=%d dynamic=%u splits=%d tail=%dx%d\n",
                     (long long)M, (long long)N, (long long)K, use_pair ? "cta-pair 256x256" : "one-cta 128x256",
                     p.num_tiles, grid,
                     load_tma ? "tma" : "predicated", store_tma ? "tma" : "predicated",
                     p.a_mn ? "m-major" : "k-major", p.b_mn ? "n-major" : "k-major",
                     grouped ? "grouped" : "row-major", p.sched.group_m, p.cross_tile, int(persistent),
                     p.dynamic, sp.splits, tp.tiles, tp.splits);

    cudaError_t e;
    if (split) {
        e = dynamic ? launch_pair<true, true, true>(tmA, tmB, tmC, tmW, p, cm, grid, stream)
                    : launch_pair<true, true>(tmA, tmB, tmC, tmW, p, cm, grid, stream);
        if (e == cudaSuccess) {
            const int64_t quads = M * ((N + 3) / 4);
            const int threads = 256;
            const int64_t want = cdiv(quads, threads);
            const int blocks = int(want < 8 * int64_t(ds->num_sms) ? want : 8 * int64_t(ds->num_sms));
            e = launch_overlapped(splitk_reduce_kernel, blocks, threads, 0, stream,
                                  static_cast<const float *>(sk.workspace), C, M, N, sp.ldw, stride_cm, sp.splits,
                                  out_dtype, alpha);
        }
    } else if (tp.splits > 1) {
        e = launch_pair<true, true, false, true>(tmA, tmB, tmC, tmW, p, cm, grid, stream);
        if (e == cudaSuccess) {
            const int64_t quads = int64_t(tp.tiles) * (pair::TILE_M * pair::TILE_N / 4);
            const int threads = 256;
            const int64_t want = cdiv(quads, threads);
            const int blocks = int(want < 8 * int64_t(ds->num_sms) ? want : 8 * int64_t(ds->num_sms));
            e = launch_overlapped(tail_reduce_kernel<pair::TILE_M>, blocks, threads, 0, stream,
                                  static_cast<const float *>(tail_ws), C, M, N, stride_cm, p.sched, tp.first,
                                  tp.tiles, tp.splits, out_dtype, alpha);
        }
    } else if (dynamic) {
        e = store_tma ? launch_pair<true, true, true>(tmA, tmB, tmC, tmW, p, cm, grid, stream)
                      : launch_pair<true, false, true>(tmA, tmB, tmC, tmW, p, cm, grid, stream);
    } else if (use_pair && p.c_classes > 0) {
        e = load_tma ? launch_pair_class<true>(tmA, tmB, tmW, p, cm, cc, grid, stream)
                     : launch_pair_class<false>(tmA, tmB, tmW, p, cm, cc, grid, stream);
    } else if (use_pair) {
        if (load_tma)
            e = store_tma ? launch_pair<true, true>(tmA, tmB, tmC, tmW, p, cm, grid, stream)
                          : launch_pair<true, false>(tmA, tmB, tmC, tmW, p, cm, grid, stream);
        else
            e = store_tma ? launch_pair<false, true>(tmA, tmB, tmC, tmW, p, cm, grid, stream)
                          : launch_pair<false, false>(tmA, tmB, tmC, tmW, p, cm, grid, stream);
    }
    else if (load_tma && store_tma) e = launch<true, true>(tmA, tmB, tmC, p, cm, grid, stream);
    else if (load_tma) e = launch<true, false>(tmA, tmB, tmC, p, cm, grid, stream);
    else if (store_tma) e = launch<false, true>(tmA, tmB, tmC, p, cm, grid, stream);
    else e = launch<false, false>(tmA, tmB, tmC, p, cm, grid, stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

extern "C" {

gemm_status_t gemm_f16(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                       int64_t stride_am, int64_t stride_ak, int64_t stride_bk, int64_t stride_bn,
                       int64_t stride_cm, int64_t stride_cn, int32_t group_size_m,
                       uint32_t schedule_flags, gemm_stream_t stream) {
    return gemm_impl(A, B, C, M, N, K, stride_am, stride_ak, stride_bk, stride_bn, stride_cm, stride_cn,
                     group_size_m, schedule_flags, stream, SplitReq());
}

gemm_status_t gemm_f16_out(const void *A, const void *B, void *C, int32_t c_dtype, float alpha, int64_t M,
                           int64_t N, int64_t K, int64_t stride_am, int64_t stride_ak, int64_t stride_bk,
                           int64_t stride_bn, int64_t stride_cm, int64_t stride_cn, int32_t group_size_m,
                           uint32_t schedule_flags, gemm_stream_t stream) {
    if (c_dtype < GEMM_OUT_F32 || c_dtype > GEMM_OUT_BF16) return GEMM_ERR_INVALID_ARG;
    return gemm_impl(A, B, C, M, N, K, stride_am, stride_ak, stride_bk, stride_bn, stride_cm, stride_cn,
                     group_size_m, schedule_flags, stream, SplitReq(), uint32_t(c_dtype), alpha);
}

gemm_status_t gemm_f16_packed_workspace_size(int64_t M, int64_t N, int64_t K, int64_t stride_am,
                                             int64_t stride_ak, int64_t stride_bk, int64_t stride_bn,
                                             uint64_t *bytes) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_ARG;
    if (stride_am < 1 || stride_ak < 1 || stride_bk < 1 || stride_bn < 1) return GEMM_ERR_INVALID_ARG;
    if (bytes) {
        *bytes = 0;
        if (M > 0 && N > 0 && K > 0)
            *bytes = round256(packed_bytes(rows_of_a(M, K, stride_am, stride_ak))) +
                     packed_bytes(rows_of_b(N, K, stride_bk, stride_bn));
    }
    return GEMM_OK;
}

gemm_status_t gemm_f16_packed(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                              int64_t stride_am, int64_t stride_ak, int64_t stride_bk, int64_t stride_bn,
                              int64_t stride_cm, int64_t stride_cn, int32_t group_size_m,
                              uint32_t schedule_flags, void *workspace, uint64_t workspace_bytes,
                              gemm_stream_t stream) {
    PackReq pk;
    pk.enabled = true;
    pk.workspace = workspace;
    pk.workspace_bytes = workspace_bytes;
    return gemm_impl(A, B, C, M, N, K, stride_am, stride_ak, stride_bk, stride_bn, stride_cm, stride_cn,
                     group_size_m, schedule_flags, stream, SplitReq(), GEMM_OUT_F32, 1.0f, pk);
}

gemm_status_t gemm_f16_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int32_t splits,
                                             uint64_t *bytes, int32_t *splits_used) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || splits < 0)
        return GEMM_ERR_INVALID_ARG;
    int max_pairs = 1;
    if (splits == 0 && M > 0 && N > 0 && K > 0) {
        int dev = 0;
        DeviceState *ds = nullptr;
        if (cudaGetDevice(&dev) != cudaSuccess || device_init(dev, &ds) != cudaSuccess) return GEMM_ERR_CUDA;
        max_pairs = ds->max_pairs;
    }
    SplitPlan sp{1, 1, (N + 3) / 4 * 4};
    if (M > 0 && N > 0 && K > 0) sp = plan_splits(M, N, K, splits, max_pairs);
    if (bytes) *bytes = sp.splits > 1 ? uint64_t(sp.splits) * uint64_t(M) * uint64_t(sp.ldw) * 4u : 0u;
    if (splits_used) *splits_used = sp.splits;
    return GEMM_OK;
}

gemm_status_t gemm_f16_splitk(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                              int64_t stride_am, int64_t stride_ak, int64_t stride_bk, int64_t stride_bn,
                              int64_t stride_cm, int64_t stride_cn, int32_t splits, void *workspace,
                              uint64_t workspace_bytes, int32_t group_size_m, uint32_t schedule_flags,
                              gemm_stream_t stream) {
    if (splits < 0) return GEMM_ERR_INVALID_ARG;
    SplitReq sk;
    sk.enabled = true;
    sk.splits = splits;
    sk.workspace = workspace;
    sk.workspace_bytes = workspace_bytes;
    return gemm_impl(A, B, C, M, N, K, stride_am, stride_ak, stride_bk, stride_bn, stride_cm, stride_cn,
                     group_size_m, schedule_flags, stream, sk);
}

gemm_status_t gemm_f16_tile_map(int32_t num_m_tiles, int32_t num_n_tiles, int32_t group_size_m,
                                uint32_t flags, int32_t grid, int32_t *out_dev,
                                gemm_stream_t stream_) {
    if (num_m_tiles < 1 || num_n_tiles < 1 || grid < 1 || out_dev == nullptr)
        return GEMM_ERR_INVALID_ARG;
    if (int64_t(num_m_tiles) * num_n_tiles > kMaxDim) return GEMM_ERR_INVALID_ARG;
    const bool grouped = (flags & GEMM_SCHED_GROUPED) != 0;
    if (grouped && group_size_m < 1) return GEMM_ERR_INVALID_ARG;
    Sched s;
    s.nm = num_m_tiles;
    s.nn = num_n_tiles;
    s.group_m = grouped ? group_size_m : 1;
    s.grouped = grouped ? 1 : 0;
    tile_map_kernel<<<grid, 32, 0, reinterpret_cast<cudaStream_t>(stream_)>>>(
        s, num_m_tiles * num_n_tiles, out_dev);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

gemm_status_t gemm_f16_get_config(int64_t M, int64_t N, uint32_t flags, int32_t *bm, int32_t *bn,
                                  int32_t *bk, int32_t *stages, int32_t *grid) {
    if (M < 0 || N < 0 || M > kMaxDim || N > kMaxDim) return GEMM_ERR_INVALID_ARG;
    if (flags & ~GEMM_SCHED_ALL_FLAGS) return GEMM_ERR_INVALID_ARG;
    const bool single = (flags & GEMM_SCHED_SINGLE_CTA) != 0;
    int tm, tn;
    tile_shape(flags, &tm, &tn);
    if (bm) *bm = tm;
    if (bn) *bn = tn;
    if (bk) *bk = BK;
    if (stages) *stages = single ? STAGES : pair::STAGES;
    if (grid) {
        *grid = 0;
        if (M > 0 && N > 0) {
            int dev = 0;
            DeviceState *ds = nullptr;
            if (cudaGetDevice(&dev) != cudaSuccess || device_init(dev, &ds) != cudaSuccess)
                return GEMM_ERR_CUDA;
            const int64_t tiles = cdiv(M, tm) * cdiv(N, tn);
            const int64_t programs = (flags & (GEMM_SCHED_NON_PERSISTENT | GEMM_SCHED_DYNAMIC)) ? tiles
                                     : single ? ds->num_sms : ds->max_pairs;
            *grid = int32_t(tiles < programs ? tiles : programs);
        }
    }
    return GEMM_OK;
}

gemm_status_t gemm_f16_kernel_info(int32_t variant, int32_t *regs, int32_t *static_smem,
                                   int32_t *dynamic_smem, int32_t *threads) {
    if (variant < 0 || variant > 12) return GEMM_ERR_INVALID_ARG;
    cudaFuncAttributes a;
    cudaError_t e;
    int thr, dyn;
    switch (variant) {
        case 0: e = cudaFuncGetAttributes(&a, gemm_f16_persistent<true, true>); thr = cta_threads(true); dyn = Layout<true>::smem_bytes; break;
        case 1: e = cudaFuncGetAttributes(&a, gemm_f16_persistent<true, false>); thr = cta_threads(true); dyn = Layout<true>::smem_bytes; break;
        case 2: e = cudaFuncGetAttributes(&a, gemm_f16_persistent<false, true>); thr = cta_threads(false); dyn = Layout<false>::smem_bytes; break;
        case 3: e = cudaFuncGetAttributes(&a, gemm_f16_persistent<false, false>); thr = cta_threads(false); dyn = Layout<false>::smem_bytes; break;
        case 4: e = cudaFuncGetAttributes(&a, gemm_f16_pair<true, true>); thr = pair::Layout<true>::threads; dyn = pair::Layout<true>::smem_bytes; break;
        case 5: e = cudaFuncGetAttributes(&a, gemm_f16_pair<true, false>); thr = pair::Layout<true>::threads; dyn = pair::Layout<true>::smem_bytes; break;
        case 6: e = cudaFuncGetAttributes(&a, gemm_f16_pair<false, true>); thr = pair::Layout<false>::threads; dyn = pair::Layout<false>::smem_bytes; break;
        case 7: e = cudaFuncGetAttributes(&a, gemm_f16_pair<false, false>); thr = pair::Layout<false>::threads; dyn = pair::Layout<false>::smem_bytes; break;
        case 8: e = cudaFuncGetAttributes(&a, gemm_f16_pair<true, true, true>); thr = pair::Layout<true>::threads; dyn = pair::Layout<true>::smem_bytes; break;
        case 9: e = cudaFuncGetAttributes(&a, gemm_f16_pair<true, false, true>); thr = pair::Layout<true>::threads; dyn = pair::Layout<true>::smem_bytes; break;
        case 10: e = cudaFuncGetAttributes(&a, gemm_f16_pair<true, true, false, true>); thr = pair::Layout<true>::threads; dyn = pair::Layout<true>::smem_bytes; break;
        case 11: e = cudaFuncGetAttributes(&a, gemm_f16_pair<true, false, false, false, true>); thr = pair::Layout<true>::threads; dyn = pair::Layout<true>::smem_bytes; break;
        default: e = cudaFuncGetAttributes(&a, gemm_f16_pair<false, false, false, false, true>); thr = pair::Layout<false>::threads; dyn = pair::Layout<false>::smem_bytes; break;
    }
    if (e != cudaSuccess) return GEMM_ERR_CUDA;
    if (regs) *regs = a.numRegs;
    if (static_smem) *static_smem = int32_t(a.sharedSizeBytes);
    if (dynamic_smem) *dynamic_smem = dyn;
    if (threads) *threads = thr;
    return GEMM_OK;
}

gemm_status_t gemm_f16_selftest_wait_timeout(uint64_t timeout_ns, gemm_stream_t stream_) {
    if (timeout_ns < 1000 || timeout_ns > 10000000000ull) return GEMM_ERR_INVALID_ARG;
    WaitCtl w;
    w.timeout_ns = timeout_ns;
    w.epoch = next_epoch();
    wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream_)>>>(w);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

gemm_status_t gemm_f16_selftest_pair_abort(const void *A, const void *B, float *C, int64_t M, int64_t N,
                                           int64_t K, int32_t stop_after, gemm_stream_t stream) {
    if (stop_after < 1 || K < 1) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15u) return GEMM_ERR_UNSUPPORTED;
    if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_UNSUPPORTED;  // TMA loads: 16-byte row strides
    SplitReq sk;
    sk.stop_after = stop_after;
    return gemm_impl(A, B, C, M, N, K, K, 1, N, 1, N, 1, 8, GEMM_SCHED_GROUPED | GEMM_SCHED_CROSS_TILE, stream,
                     sk);
}

gemm_status_t gemm_f16_selftest_check(gemm_stream_t stream_) {
#ifdef GEMM_DEBUG
    check_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream_)>>>();
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
#else
    (void)stream_;
    return GEMM_ERR_UNSUPPORTED;  // the product build has no device-side checks
#endif
}

gemm_status_t gemm_f16_sync_status(gemm_stream_t stream_) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    unsigned int st = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&st, g_status, sizeof(st)) != cudaSuccess) return GEMM_ERR_CUDA;
#ifdef GEMM_DEBUG
    if (st == kStatusCheck) {
        unsigned int line = 0;
        if (cudaMemcpyFromSymbol(&line, g_check_line, sizeof(line)) == cudaSuccess)
            std::fprintf(stderr, "[gemm_f16] device check failed at source line %u\n", line);
    }
#endif
    if (st != 0) {
        // clear the status, and the aborted launch's epoch: a CUDA graph replays a
        // launch with the epoch it was captured with
        if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess ||
            cudaMemcpyToSymbol(g_abort_epoch, &zero, sizeof(zero)) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    return st == 0 ? GEMM_OK : static_cast<gemm_status_t>(st);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Split-K without any device allocation: the workspace is a fixed array in the
// library image instead of caller memory. Meant for callers that cannot call
// cudaMalloc at the point where they multiply: their device memory is owned by
// another allocator or a fixed arena, or they cannot afford the device-wide
// synchronisation and the failure modes of an allocation on that path.
// ---------------------------------------------------------------------------
namespace {

constexpr uint64_t kNoAllocScratchBytes = 32ull << 20;  // 32 MiB, held by every device that loads the library

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The scratch array's device address on each device (kept once a lookup
// succeeds; a failed one returns GEMM_ERR_CUDA and the next call retries).
SymbolAddress g_scratch[kMaxDevices];

}  // namespace

extern "C" gemm_status_t gemm_f16_splitk_noalloc(const void *A, const void *B, float *C, int64_t M,
                                                 int64_t N, int64_t K, int64_t stride_am,
                                                 int64_t stride_ak, int64_t stride_bk,
                                                 int64_t stride_bn, int64_t stride_cm,
                                                 int64_t stride_cn, int32_t splits,
                                                 int32_t group_size_m, uint32_t schedule_flags,
                                                 gemm_stream_t stream) {
    uint64_t need = 0;
    int32_t used = 1;
    const gemm_status_t st = gemm_f16_splitk_workspace_size(M, N, K, splits, &need, &used);
    if (st != GEMM_OK) return st;
    if (need > kNoAllocScratchBytes) return GEMM_ERR_UNSUPPORTED;  // larger than the built-in scratch
    void *ws = nullptr;
    if (need > 0) {
        // In host code the array's name is only a stand-in: its device address is
        // looked up with the device current, and kept once a lookup succeeds.
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
        ws = symbol_address(g_scratch[dev], g_noalloc_scratch);
        if (ws == nullptr) return GEMM_ERR_CUDA;
    }
    return gemm_f16_splitk(A, B, C, M, N, K, stride_am, stride_ak, stride_bk, stride_bn, stride_cm,
                           stride_cn, splits, ws, kNoAllocScratchBytes, group_size_m, schedule_flags,
                           stream);
}
