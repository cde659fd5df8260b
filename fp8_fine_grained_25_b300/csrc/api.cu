// The C ABI of libfp8q.so (declared in include/fp8q.h): argument checks,
// device checks, TMA descriptor encoding and kernel launches. No device
// memory is allocated here; every pointer belongs to the caller.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "fp8q.h"
#include "gemm.cuh"
#include "quant.cuh"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceInfo {
    bool init = false;
    bool supported = false;
    int sms = 0;
    // co-resident 2-CTA clusters of the pair kernel, per tile width
    // ([0]: 128, [1]: 256, [2]: 224, [3]: 160) and B-scale layout ([0]:
    // 128x128 blocks, [1]: one per row); -1: not queried yet
    int pair_clusters[4][2] = {{-1, -1}, {-1, -1}, {-1, -1}, {-1, -1}};
    int bs_pair_clusters[2] = {-1, -1};  // the same for the UE8M0 (hardware-scaled) GEMM
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;
uint64_t g_timeout_ns = 1000000000ull;
int g_force_bn = 0;
int g_force_splits = 0;  // 0: the split-K choice below; else this many K ranges
constexpr int kMaxSplits = 8;
std::atomic<uint32_t> g_epoch{0};
int g_pair_mode = 1;  // 1: use 2-CTA pairs for the dense GEMM where they fit
uint32_t g_inject = 0;  // FP8Q_INJECT_* bits for failure-path tests
constexpr int64_t kI32Max = 2147483647;

int current_device(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FP8Q_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FP8Q_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.sms = sms;
        d.init = true;
    }
    if (!d.supported) return FP8Q_ERR_DEVICE;
    *out = &d;
    return FP8Q_OK;
}

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A row-major [outer, inner] tensor, boxes of [box_outer, box_inner]
// elements, swizzled shared-memory layout, zero fill outside the tensor.
bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, uint64_t elem_bytes,
                 const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * elem_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t elem_strides[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Output-tile width by a wave model: rounds of work units over the units
// that run at once, times the cost of one unit at that width.
// Pair tiles of the block-scaled GEMM (256 rows on a 2-CTA cluster, 74
// clusters): a unit's cost relative to 256 columns, measured back to back
// at 2032 MHz on 4096 x {576, 1536}, 2048 x 7168 and 8192 x {2048, 7168}
// (K = 7168): 0.74 for 128, 0.85 for 160, 0.97 for 224. The K loop costs
// ~600-740 cycles per K block at every width, so narrow tiles pay only
// where they save a round: 160 at 4096 x 576 (one round of 64 units instead
// of two of 80 at 128; 24.8 against 26.9 us at 224), 224 at 4096 x 1536
// and 2048 x 7168, 256 for the large layers.
// One-CTA tiles and the row-scaled GEMM: tiles over the SMs, a tile costing
// its width plus a fixed share for the per-K-block handshake; the shares
// reproduce measured per-column costs relative to 256 of 1.2 for 128 and
// ~1.08 for 224 (in long power-capped runs).
// Ties keep the earlier candidate.
int choose_bn(int64_t M, int64_t N, int sms, bool block_scaled, bool pair) {
    int best = 256;
    int64_t best_cost = -1;
    for (int bn : {256, 128, 224, 160}) {
        if ((bn == 224 || bn == 160) && !block_scaled) continue;
        if (bn == 160 && !pair) continue;
        int64_t cost;
        if (pair && block_scaled) {
            const int64_t units = cdiv(cdiv(M, 128), 2) * cdiv(N, bn);
            const int unit_cost = bn == 128 ? 237 : bn == 160 ? 272 : bn == 224 ? 310 : 320;
            cost = cdiv(units, std::max(1, sms / 2)) * unit_cost;
        } else {
            const int64_t tiles = cdiv(M, 128) * cdiv(N, bn);
            cost = cdiv(tiles, sms) * (bn + (bn == 224 ? 80 : 64));
        }
        if (best_cost < 0 || cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

// Split K for the dense GEMM: the number of K ranges S (1: none). Each
// split unit ends with a partial-tile store, a GPU-scope fence, an arrival
// count and (last unit) a read of the other partials, a few microseconds
// during which the tile's MMA pipeline waits; so split K only pays where
// few tiles run over a long K range. Measured on the B300 (K = 7168, 9
// shapes from 256 x 576 to 2048 x 7168): the best S keeps about half the
// co-resident units busy, S = round(slots / (2 units)), capped at 4; shapes
// with more than ~slots / 3 tile units are fastest unsplit.
int choose_splits(int64_t units, int64_t slots, int64_t KB) {
    const int64_t kb4 = cdiv(KB, 4);
    if (units <= 0 || kb4 < 2) return 1;
    int64_t s = (slots + units) / (2 * units);  // round(slots / (2 units))
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({s, 4, kb4})));
}

// Workspace of a split-K call: S FP32 partial tiles of 128 rows x bn
// columns for every output tile (m-tiles rounded up to pairs), then one
// 32-bit arrival word per tile.
size_t splitk_bytes(int64_t M, int64_t N, int splits, int bn) {
    if (splits <= 1) return 0;
    const int64_t tiles = 2 * cdiv(cdiv(M, 128), 2) * cdiv(N, bn);
    const size_t part = static_cast<size_t>(splits) * tiles * bn * 128 * 4;
    const size_t ctr = static_cast<size_t>(tiles) * 4;
    return (part + 255) / 256 * 256 + (ctr + 255) / 256 * 256;
}

}  // namespace

extern "C" {

const char* fp8q_status_string(int status) {
    switch (status) {
        case FP8Q_OK: return "ok";
        case FP8Q_ERR_NULL: return "a required pointer is NULL";
        case FP8Q_ERR_SHAPE: return "invalid size (negative, zero, or too large)";
        case FP8Q_ERR_ALIGN: return "K must be a multiple of 16, N of 8, and pointers 16-byte aligned";
        case FP8Q_ERR_DEVICE: return "the current device is not sm_103 (B300)";
        case FP8Q_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case FP8Q_ERR_TIMEOUT: return "a pipeline wait inside a kernel exceeded its time limit";
        case FP8Q_ERR_UNSUPPORTED: return "unsupported request";
        case FP8Q_ERR_OFFSETS: return "expert offsets are malformed";
        default: return "unknown status";
    }
}

void fp8q_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns = ns ? ns : 1000000000ull; }

int fp8q_set_gemm_tile_n(int bn) {
    if (bn != 0 && bn != 128 && bn != 160 && bn != 224 && bn != 256) return FP8Q_ERR_UNSUPPORTED;
    g_force_bn = bn;
    return FP8Q_OK;
}

int fp8q_set_gemm_splits(int splits) {
    if (splits < 0 || splits > kMaxSplits) return FP8Q_ERR_UNSUPPORTED;
    g_force_splits = splits;
    return FP8Q_OK;
}

int fp8q_set_fault_injection(uint32_t flags) {
    g_inject = flags & FP8Q_INJECT_STALLED_STAGE;
    return FP8Q_OK;
}

int fp8q_set_gemm_pairs(int enable) {
    g_pair_mode = enable ? 1 : 0;
    return FP8Q_OK;
}

int fp8q_get_device_status(cudaStream_t stream, uint32_t* status_out, int clear) {
    if (!status_out) return FP8Q_ERR_NULL;
    uint32_t gemm_status = 0, quant_status = 0, bs_status = 0;
    if (fp8q::read_device_status(stream, &gemm_status, clear != 0) != cudaSuccess ||
        fp8q::read_quant_status(&quant_status, clear != 0) != cudaSuccess ||
        fp8q::read_bs_status(&bs_status, clear != 0) != cudaSuccess)
        return FP8Q_ERR_CUDA;
    *status_out = gemm_status | quant_status | bs_status;
    return FP8Q_OK;
}

}  // extern "C"

namespace {

int quant_act_impl(const void* x_bf16, int64_t M, int64_t K, void* q_e4m3, void* scales, bool pow2,
                   cudaStream_t stream) {
    if (M < 0 || K <= 0 || M > kI32Max || K > kI32Max) return FP8Q_ERR_SHAPE;
    if (M == 0) return FP8Q_OK;
    if (!x_bf16 || !q_e4m3 || !scales) return FP8Q_ERR_NULL;
    if (K % 16 != 0 || !aligned(x_bf16, 16) || !aligned(q_e4m3, 16) || !aligned(scales, pow2 ? 1 : 4))
        return FP8Q_ERR_ALIGN;
    if (M * cdiv(K, 128) > kI32Max) return FP8Q_ERR_SHAPE;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;
    return fp8q::launch_quant_act(x_bf16, M, K, q_e4m3, scales, pow2, stream, dev->sms, g_timeout_ns) ==
                   cudaSuccess
               ? FP8Q_OK
               : FP8Q_ERR_CUDA;
}

int quant_weight_impl(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3, void* scales, bool pow2,
                      cudaStream_t stream) {
    if (N < 0 || K <= 0 || N > kI32Max || K > kI32Max) return FP8Q_ERR_SHAPE;
    if (N == 0) return FP8Q_OK;
    if (!w_bf16 || !q_e4m3 || !scales) return FP8Q_ERR_NULL;
    if (K % 16 != 0 || !aligned(w_bf16, 16) || !aligned(q_e4m3, 16) || !aligned(scales, pow2 ? 1 : 4))
        return FP8Q_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;
    CUtensorMap tmW;
    if (!make_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_bf16, K, N, 128, 128,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
        return FP8Q_ERR_CUDA;
    return fp8q::launch_quant_weight(&tmW, q_e4m3, scales, pow2, N, K, stream, dev->sms, g_timeout_ns) ==
                   cudaSuccess
               ? FP8Q_OK
               : FP8Q_ERR_CUDA;
}

}  // namespace

extern "C" {

int fp8q_quant_act(const void* x_bf16, int64_t M, int64_t K, void* q_e4m3, float* scales,
                   cudaStream_t stream) {
    return quant_act_impl(x_bf16, M, K, q_e4m3, scales, false, stream);
}

int fp8q_quant_weight(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3, float* scales,
                      cudaStream_t stream) {
    return quant_weight_impl(w_bf16, N, K, q_e4m3, scales, false, stream);
}

int fp8q_quant_act_ue8m0(const void* x_bf16, int64_t M, int64_t K, void* q_e4m3, uint8_t* scales,
                         cudaStream_t stream) {
    return quant_act_impl(x_bf16, M, K, q_e4m3, scales, true, stream);
}

int fp8q_quant_weight_ue8m0(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3, uint8_t* scales,
                            cudaStream_t stream) {
    return quant_weight_impl(w_bf16, N, K, q_e4m3, scales, true, stream);
}

}  // extern "C"

namespace {

int quant_act_t_impl(const void* x_bf16, int64_t M, int64_t K, void* qt_e4m3, void* st, bool pow2,
                     cudaStream_t stream) {
    if (M < 0 || K <= 0 || M > kI32Max || K > kI32Max) return FP8Q_ERR_SHAPE;
    if (M == 0) return FP8Q_OK;
    if (!x_bf16 || !qt_e4m3 || !st) return FP8Q_ERR_NULL;
    if (K % 16 != 0 || M % 16 != 0 || !aligned(x_bf16, 16) || !aligned(qt_e4m3, 16) ||
        !aligned(st, pow2 ? 1 : 4))
        return FP8Q_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;
    if (cdiv(M, 128) * cdiv(K, 128) > kI32Max) return FP8Q_ERR_SHAPE;
    return fp8q::launch_quant_act_t(x_bf16, qt_e4m3, st, pow2, M, K, stream, dev->sms) == cudaSuccess
               ? FP8Q_OK
               : FP8Q_ERR_CUDA;
}

int quant_weight_t_impl(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3, void* scales,
                        void* qt_e4m3, void* st, bool pow2, cudaStream_t stream) {
    if (N < 0 || K <= 0 || N > kI32Max || K > kI32Max) return FP8Q_ERR_SHAPE;
    if (N == 0) return FP8Q_OK;
    if (!w_bf16 || !qt_e4m3 || !st || (q_e4m3 == nullptr) != (scales == nullptr))
        return FP8Q_ERR_NULL;
    const uintptr_t sal = pow2 ? 1 : 4;
    if (K % 16 != 0 || N % 16 != 0 || !aligned(w_bf16, 16) || !aligned(qt_e4m3, 16) ||
        !aligned(st, sal) || (q_e4m3 && !aligned(q_e4m3, 16)) || (scales && !aligned(scales, sal)))
        return FP8Q_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;
    if (cdiv(N, 128) * cdiv(K, 128) > kI32Max) return FP8Q_ERR_SHAPE;
    return fp8q::launch_quant_weight_t(w_bf16, q_e4m3, scales, qt_e4m3, st, pow2, N, K, stream, dev->sms) ==
                   cudaSuccess
               ? FP8Q_OK
               : FP8Q_ERR_CUDA;
}

}  // namespace

extern "C" {

int fp8q_quant_act_t(const void* x_bf16, int64_t M, int64_t K, void* qt_e4m3, float* st,
                     cudaStream_t stream) {
    return quant_act_t_impl(x_bf16, M, K, qt_e4m3, st, false, stream);
}

int fp8q_quant_weight_t(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3, float* scales,
                        void* qt_e4m3, float* st, cudaStream_t stream) {
    return quant_weight_t_impl(w_bf16, N, K, q_e4m3, scales, qt_e4m3, st, false, stream);
}

int fp8q_quant_act_t_ue8m0(const void* x_bf16, int64_t M, int64_t K, void* qt_e4m3, uint8_t* st,
                           cudaStream_t stream) {
    return quant_act_t_impl(x_bf16, M, K, qt_e4m3, st, true, stream);
}

int fp8q_quant_weight_t_ue8m0(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3, uint8_t* scales,
                              void* qt_e4m3, uint8_t* st, cudaStream_t stream) {
    return quant_weight_t_impl(w_bf16, N, K, q_e4m3, scales, qt_e4m3, st, true, stream);
}

int fp8q_gather_rows(const void* q_src, const float* s_src, int64_t T, int64_t K,
                     const int32_t* index, int64_t R, void* q_dst, float* s_dst,
                     cudaStream_t stream) {
    if (T < 0 || R < 0 || K <= 0 || T > kI32Max || R > kI32Max || K > kI32Max)
        return FP8Q_ERR_SHAPE;
    if (R == 0) return FP8Q_OK;
    if (!q_src || !s_src || !index || !q_dst || !s_dst) return FP8Q_ERR_NULL;
    if (K % 16 != 0 || !aligned(q_src, 16) || !aligned(q_dst, 16) || !aligned(s_src, 4) ||
        !aligned(s_dst, 4) || !aligned(index, 4))
        return FP8Q_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;
    return fp8q::launch_gather_rows(q_src, s_src, T, K, index, R, q_dst, s_dst, stream, dev->sms) ==
                   cudaSuccess
               ? FP8Q_OK
               : FP8Q_ERR_CUDA;
}

}  // extern "C"

namespace {

// The dense GEMM C = A * B^T; row_scaled_b selects sb [N][KB] (one scale per
// row of B) instead of sb [ceil(N/128)][KB].
// The tile width, pair mode and co-resident clusters of a dense GEMM call.
struct DensePlan {
    int bn;
    bool pair;
    int clusters;  // pair mode: co-resident 2-CTA clusters
    int64_t units; // tile units (pairs of m-tiles in pair mode) x n-tiles
    int64_t slots; // units that run at once
};

// Co-resident clusters of the pair kernel of tile width bn (queried once).
int pair_clusters(DeviceInfo* dev, int bn, bool row_scaled_b) {
    int* pc = &dev->pair_clusters[bn == 256 ? 1 : bn == 224 ? 2 : bn == 160 ? 3 : 0][row_scaled_b ? 1 : 0];
    std::lock_guard<std::mutex> lock(g_mutex);
    if (*pc < 0) *pc = fp8q::gemm_pair_max_clusters(bn, row_scaled_b);
    return *pc;
}

int plan_dense(DeviceInfo* dev, int64_t M, int64_t N, bool row_scaled_b, DensePlan* p) {
    // 2-CTA pairs (256-row tiles over two SMs) when there are at least two
    // m-tiles to pair.
    const bool want_pair = g_pair_mode && M > 128;
    // the 160- and 224-wide tiles exist for block-scaled B only; forced,
    // they run the row-scaled GEMM 256 wide
    int bn = g_force_bn ? g_force_bn : choose_bn(M, N, dev->sms, !row_scaled_b, want_pair);
    if ((bn == 224 || bn == 160) && row_scaled_b) bn = 256;
    int clusters = want_pair ? pair_clusters(dev, bn, row_scaled_b) : 0;
    bool pair = clusters > 0;
    if (bn == 160 && !pair) {
        // 160-wide tiles are pair tiles only: the best one-CTA width
        bn = choose_bn(M, N, dev->sms, !row_scaled_b, false);
        clusters = 0;
    }
    p->bn = bn;
    p->pair = pair;
    p->clusters = clusters;
    const int64_t mt = cdiv(M, 128);
    p->units = (pair ? cdiv(mt, 2) : mt) * cdiv(N, bn);
    p->slots = pair ? clusters : dev->sms;
    return FP8Q_OK;
}

// K ranges of a split-K call with this plan before the workspace limit: the
// forced or chosen count, at most one range per 4 K blocks; 1 for 160-wide
// tiles, which have no split-K form.
int plan_splits(const DensePlan& plan, int64_t K) {
    if (plan.bn == 160) return 1;
    const int splits = g_force_splits ? g_force_splits : choose_splits(plan.units, plan.slots, cdiv(K, 128));
    return static_cast<int>(std::min<int64_t>(splits, cdiv(cdiv(K, 128), 4)));
}

int dense_gemm(const void* A, const float* sa, const void* B, const float* sb, void* C_bf16,
               int64_t M, int64_t N, int64_t K, bool row_scaled_b, void* workspace, size_t workspace_bytes,
               cudaStream_t stream) {
    if (M < 0 || N <= 0 || K <= 0 || M > kI32Max || N > kI32Max || K > kI32Max)
        return FP8Q_ERR_SHAPE;
    if (M == 0) return FP8Q_OK;
    if (!A || !sa || !B || !sb || !C_bf16) return FP8Q_ERR_NULL;
    if (K % 16 != 0 || N % 8 != 0 || !aligned(A, 16) || !aligned(B, 16) || !aligned(C_bf16, 16) ||
        !aligned(sa, 4) || !aligned(sb, 4))
        return FP8Q_ERR_ALIGN;
    if (workspace && !aligned(workspace, 256)) return FP8Q_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;
    DensePlan plan;
    plan_dense(dev, M, N, row_scaled_b, &plan);
    const int bn = plan.bn;
    const bool pair = plan.pair;
    // split K only with a workspace (block-scaled B): the requested or chosen
    // count, reduced until the workspace holds it
    int splits = 1;
    if (workspace && !row_scaled_b) {
        splits = plan_splits(plan, K);
        while (splits > 1 && splitk_bytes(M, N, splits, bn) > workspace_bytes) --splits;
    }
    CUtensorMap tmA, tmB, tmC;
    if (!make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K, M, 128, 128) ||
        !make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K, N, 128, pair ? bn / 2 : bn))
        return FP8Q_ERR_CUDA;
    const int cbox = fp8q::gemm_c_box_cols(bn, pair);  // 64, 32 or 16 columns (128/64/32-byte swizzle)
    if (!make_map_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C_bf16, N, M, cbox, 32,
                     cbox == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                     : cbox == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : CU_TENSOR_MAP_SWIZZLE_32B))
        return FP8Q_ERR_CUDA;

    fp8q::GemmLaunch g{};
    g.tmA = &tmA;
    g.tmB = &tmB;
    g.tmC = &tmC;
    g.bn = bn;
    g.grouped = false;
    g.pair = pair;
    g.row_scaled_b = row_scaled_b;
    g.stream = stream;
    fp8q::GemmArgs& a = g.args;
    a.sa = sa;
    a.sb = sb;
    a.C = static_cast<__nv_bfloat16*>(C_bf16);
    a.offsets = nullptr;
    a.M = static_cast<int32_t>(M);
    a.N = static_cast<int32_t>(N);
    a.K = static_cast<int32_t>(K);
    a.KB = static_cast<int32_t>(cdiv(K, 128));
    a.NB = static_cast<int32_t>(cdiv(N, 128));
    a.E = 1;
    a.mt_count = static_cast<int32_t>(cdiv(M, 128));
    a.nt_count = static_cast<int32_t>(cdiv(N, bn));
    a.mp_count = static_cast<int32_t>(cdiv(a.mt_count, 2));
    // work units: tiles, or pairs of m-tiles in pair mode, times K ranges
    const int64_t units = static_cast<int64_t>(pair ? a.mp_count : a.mt_count) * a.nt_count * splits;
    if (units > kI32Max) return FP8Q_ERR_SHAPE;
    a.num_tiles = static_cast<int32_t>(units);
    a.splits = splits;
    a.tile_units = static_cast<int32_t>(units / splits);
    if (splits > 1) {
        a.ws = static_cast<float*>(workspace);
        const int64_t tiles = 2 * cdiv(cdiv(M, 128), 2) * cdiv(N, bn);
        const size_t part = static_cast<size_t>(splits) * tiles * bn * 128 * 4;
        a.counters = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + (part + 255) / 256 * 256);
        a.epoch = g_epoch.fetch_add(1) % 0xFFFFFFu + 1u;
    }
    a.timeout_ns = g_timeout_ns;
    a.debug = g_inject;
    if (pair) {
        const int64_t clusters = units < plan.clusters ? units : plan.clusters;
        g.grid = static_cast<unsigned>(2 * clusters);
    } else {
        g.grid = static_cast<unsigned>(units < dev->sms ? units : dev->sms);
    }
    return fp8q::launch_gemm(g) == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

}  // namespace

extern "C" {

int fp8_block_gemm(const void* A, const float* sa, const void* B, const float* sb, void* C_bf16,
                   int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return dense_gemm(A, sa, B, sb, C_bf16, M, N, K, false, nullptr, 0, stream);
}

int fp8_block_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (!bytes) return FP8Q_ERR_NULL;
    *bytes = 0;
    if (M < 0 || N <= 0 || K <= 0 || M > kI32Max || N > kI32Max || K > kI32Max) return FP8Q_ERR_SHAPE;
    if (M == 0) return FP8Q_OK;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;
    DensePlan plan;
    plan_dense(dev, M, N, false, &plan);
    *bytes = splitk_bytes(M, N, plan_splits(plan, K), plan.bn);
    return FP8Q_OK;
}

int fp8_block_gemm_ws(const void* A, const float* sa, const void* B, const float* sb, void* C_bf16,
                      int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
    return dense_gemm(A, sa, B, sb, C_bf16, M, N, K, false, workspace, workspace_bytes, stream);
}

int fp8_wgrad_gemm(const void* A, const float* sa, const void* B, const float* sb, void* C_bf16,
                   int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return dense_gemm(A, sa, B, sb, C_bf16, M, N, K, true, nullptr, 0, stream);
}

}  // extern "C"

namespace {

int gemm_ue8m0_impl(const void* A, const uint8_t* sa, const void* B, const uint8_t* sb, void* C_bf16,
                    int64_t M, int64_t N, int64_t K, bool row_scaled_b, cudaStream_t stream) {
    if (M < 0 || N <= 0 || K <= 0 || M > kI32Max || N > kI32Max || K > kI32Max)
        return FP8Q_ERR_SHAPE;
    if (M == 0) return FP8Q_OK;
    if (!A || !sa || !B || !sb || !C_bf16) return FP8Q_ERR_NULL;
    if (K % 16 != 0 || N % 8 != 0 || !aligned(A, 16) || !aligned(B, 16) || !aligned(C_bf16, 16))
        return FP8Q_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;
    bool pair = g_pair_mode && M > 128;
    int* pc = &dev->bs_pair_clusters[row_scaled_b ? 1 : 0];
    if (pair) {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (*pc < 0) *pc = fp8q::gemm_bs_pair_max_clusters(row_scaled_b);
        pair = *pc > 0;
    }
    const uint32_t bn = static_cast<uint32_t>(fp8q::gemm_bs_tile_n());
    CUtensorMap tmA, tmB, tmC;
    if (!make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K, M, 128, 128) ||
        !make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K, N, 128, pair ? bn / 2 : bn) ||
        !make_map_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C_bf16, N, M, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_64B))
        return FP8Q_ERR_CUDA;
    return fp8q::launch_gemm_bs(&tmA, &tmB, &tmC, sa, sb, static_cast<int32_t>(M), static_cast<int32_t>(N),
                                static_cast<int32_t>(K), row_scaled_b, pair, *pc, g_timeout_ns, g_inject,
                                dev->sms, stream) == cudaSuccess
               ? FP8Q_OK
               : FP8Q_ERR_CUDA;
}

}  // namespace

extern "C" {

int fp8_block_gemm_ue8m0(const void* A, const uint8_t* sa, const void* B, const uint8_t* sb,
                         void* C_bf16, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return gemm_ue8m0_impl(A, sa, B, sb, C_bf16, M, N, K, false, stream);
}

int fp8_wgrad_gemm_ue8m0(const void* A, const uint8_t* sa, const void* B, const uint8_t* sb,
                         void* C_bf16, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return gemm_ue8m0_impl(A, sa, B, sb, C_bf16, M, N, K, true, stream);
}

int fp8_grouped_gemm(const void* A, const float* sa, const void* B, const float* sb,
                     void* C_bf16, const int32_t* expert_offsets, int32_t E, int64_t total_M,
                     int64_t N, int64_t K, cudaStream_t stream) {
    if (E < 1 || E > fp8q::kMaxExperts || total_M < 0 || N <= 0 || K <= 0 ||
        total_M > kI32Max || N > kI32Max || K > kI32Max ||
        static_cast<int64_t>(E) * N > kI32Max)
        return FP8Q_ERR_SHAPE;
    if (total_M == 0) return FP8Q_OK;
    if (!A || !sa || !B || !sb || !C_bf16 || !expert_offsets) return FP8Q_ERR_NULL;
    if (K % 16 != 0 || N % 8 != 0 || !aligned(A, 16) || !aligned(B, 16) || !aligned(C_bf16, 16) ||
        !aligned(sa, 4) || !aligned(sb, 4) || !aligned(expert_offsets, 4))
        return FP8Q_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;

    const int bn = 256;
    CUtensorMap tmA, tmB;
    if (!make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K, total_M, 128, 128) ||
        !make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K, static_cast<uint64_t>(E) * N,
                     128, bn))
        return FP8Q_ERR_CUDA;

    fp8q::GemmLaunch g{};
    g.tmA = &tmA;
    g.tmB = &tmB;
    g.tmC = &tmA;  // unused: the grouped epilogue stores directly
    g.bn = bn;
    g.grouped = true;
    g.pair = false;
    g.row_scaled_b = false;
    g.stream = stream;
    fp8q::GemmArgs& a = g.args;
    a.sa = sa;
    a.sb = sb;
    a.C = static_cast<__nv_bfloat16*>(C_bf16);
    a.offsets = expert_offsets;
    a.M = static_cast<int32_t>(total_M);
    a.N = static_cast<int32_t>(N);
    a.K = static_cast<int32_t>(K);
    a.KB = static_cast<int32_t>(cdiv(K, 128));
    a.NB = static_cast<int32_t>(cdiv(N, 128));
    a.E = E;
    a.mt_count = 0;
    a.mp_count = 0;
    a.nt_count = static_cast<int32_t>(cdiv(N, bn));
    // Upper bound of the tile count (sum over experts of ceil(rows/128) *
    // n-tiles) must fit the kernel's int32 tile ids.
    if ((cdiv(total_M, 128) + E) * a.nt_count > kI32Max) return FP8Q_ERR_SHAPE;
    a.num_tiles = 0;
    a.timeout_ns = g_timeout_ns;
    a.debug = g_inject;
    g.grid = static_cast<unsigned>(dev->sms);
    return fp8q::launch_gemm(g) == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Split-K GEMM for callers that cannot allocate device memory.
//
// fp8_block_gemm_ws needs a workspace from its caller. Some callers have no
// way to provide one: code that may not call cudaMalloc (which can
// synchronise the device and is not allowed everywhere a GEMM is issued), or
// a framework that hands a custom operation only its input and output
// buffers. fp8_block_gemm_static runs the same split-K kernel with its
// scratch in a fixed array that lives in this library's device image: every
// GPU that loads the library holds FP8Q_STATIC_SCRATCH_BYTES for it until
// the process exits, and no call allocates anything.
static __device__ __align__(256) unsigned char g_static_scratch[FP8Q_STATIC_SCRATCH_BYTES];

namespace {

// Device address of g_static_scratch on each device; the host-side name is
// only a stand-in and must never reach a kernel. Resolved on the first call
// per device, under g_mutex.
void* g_static_scratch_addr[kMaxDevices];

}  // namespace

extern "C" {

int fp8_block_gemm_static(const void* A, const float* sa, const void* B, const float* sb, void* C_bf16,
                          int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    if (M < 0 || N <= 0 || K <= 0 || M > kI32Max || N > kI32Max || K > kI32Max) return FP8Q_ERR_SHAPE;
    if (M == 0) return FP8Q_OK;
    if (!A || !sa || !B || !sb || !C_bf16) return FP8Q_ERR_NULL;
    if (K % 16 != 0 || N % 8 != 0 || !aligned(A, 16) || !aligned(B, 16) || !aligned(C_bf16, 16) ||
        !aligned(sa, 4) || !aligned(sb, 4))
        return FP8Q_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    if (int rc = current_device(&dev)) return rc;
    // the split count this call runs with, and the scratch it needs
    DensePlan plan;
    plan_dense(dev, M, N, false, &plan);
    const size_t need = splitk_bytes(M, N, plan_splits(plan, K), plan.bn);
    if (need > FP8Q_STATIC_SCRATCH_BYTES) return FP8Q_ERR_SHAPE;
    if (need == 0) return dense_gemm(A, sa, B, sb, C_bf16, M, N, K, false, nullptr, 0, stream);
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return FP8Q_ERR_CUDA;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!g_static_scratch_addr[d]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return FP8Q_ERR_CUDA;
            g_static_scratch_addr[d] = p;
        }
        scratch = g_static_scratch_addr[d];
    }
    return dense_gemm(A, sa, B, sb, C_bf16, M, N, K, false, scratch, FP8Q_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"
