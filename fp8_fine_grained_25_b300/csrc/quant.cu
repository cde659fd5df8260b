// Fine-grained FP8 quantizers: activations per 1x128 tile, weights per
// 128x128 block (news.qq.com/rain/a/20241229A05OQF00, "FP8 低精度训练",
// item "细粒度量化", Fig. 7a; developer.aliyun.com/article/1776647 §4.1).
//
// Both are HBM-bound streams: 2 bytes read and 1 byte written per element
// plus one fp32 scale per tile/block. A producer warp streams the input into
// a ring of shared-memory stages with bulk copies (TMA), so the bytes in
// flight do not depend on registers; consumer warps read a stage, reduce the
// amax, encode, and store codes (8-byte vectors) and scales to global memory.
//
// Arithmetic per tile (bit-exact with the definition):
//   amax  = max |x|                 (bf16 -> fp32 is exact, max is exact)
//   s     = fl32(amax / 448)        (IEEE round-to-nearest divide)
//   q_i   = E4M3_rn_satfinite(fl32(x_i / s)),  all-zero tile: s = 0, q = 0
// The per-element quotient uses the tile's reciprocal and one FMA
// correction instead of a full divide (see div_by_scale).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8q.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace fp8q {

__device__ uint32_t g_quant_status;

namespace {

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// max |x| of eight bf16 values as bf16 bits: for finite values with the
// sign cleared, the bit patterns order like the values.
__device__ __forceinline__ uint32_t absmax_bits8(const uint4& v) {
    const uint32_t a = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
    const uint32_t b = __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
    const uint32_t c = __vmaxu2(a, b);
    return max(c & 0xFFFFu, c >> 16);
}

// Two fp32 values -> two E4M3 codes (round to nearest even, saturating to
// +-448); `lo` lands in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// x / s rounded to nearest, from r = RN(1/s) and one exact-residual
// correction (Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
//   q0 = RN(x * r);  e = RN(q0 * s - x) (exact);  q = RN(q0 - e * r).
// Writing the residual negated keeps the sign of a zero quotient (-0 / s
// gives -0). For every bf16 x with |x| <= amax and every bf16 amax >= 2^-90
// this equals the IEEE quotient whenever |x / s| >= 2^-12; smaller
// quotients may differ in the last bits but keep their sign, and all of
// them encode to a signed E4M3 zero either way.
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
    const float q0 = __fmul_rn(x, r);
    const float e = __fmaf_rn(q0, s, -x);
    return __fmaf_rn(-e, r, q0);
}

constexpr float kFastDivMinAmax = 0x1p-90f;

// s = amax / 448 rounded to nearest, by the same reciprocal-and-correction
// steps with the constant RN(1/448); equal to the IEEE quotient for every
// finite non-negative bf16 amax (checked exhaustively by the test suite).
__device__ __forceinline__ float tile_scale(float amax) {
    const float r448 = 1.0f / 448.0f;  // RN(1/448), folded at compile time
    const float q0 = __fmul_rn(amax, r448);
    const float e = __fmaf_rn(q0, 448.0f, -amax);
    return __fmaf_rn(-e, r448, q0);
}

// Eight values of a tile whose scale s and reciprocal r = RN(1/s) (or 0 for
// the IEEE-divide range, amax < 2^-90) are known, encoded low byte first.
__device__ __forceinline__ uint2 encode8_r(const uint4& v, float s, float r, bool fast) {
    if (s == 0.0f) return make_uint2(0u, 0u);
    float f[8], y[8];
    unpack_bf16x8(v, f);
    if (fast) {
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = div_by_scale(f[i], s, r);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(f[i], s);
    }
    uint2 out;
    out.x = e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
    out.y = e4m3x2(y[4], y[5]) | (e4m3x2(y[6], y[7]) << 16);
    return out;
}

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// A bounded wait taken by a whole warp (see the GEMM kernel).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, limit));
}

// ------------------------------------------------------------ activations
// Tile t = (m, kb) = (t / KB, t % KB) covers row m, columns
// [128 kb, min(K, 128 kb + 128)). Consecutive tiles are adjacent in memory
// (the last tile of a row ends where the next row starts), so a run of whole
// tiles is one contiguous byte range: a chunk of kActChunkTiles tiles is one
// bulk copy. Four lanes encode one tile (8 tiles per warp): lane `sub` of
// the group owns the 16-byte chunks (4j + sub + 8 * (group & 1)) mod 16,
// j = 0..3, of the tile's 256 bytes; the rotation by 8 chunks for odd groups
// keeps every 8-lane shared-memory phase on distinct banks.
constexpr int kActConsumerWarps = 16;
constexpr int kActChunkTiles = 8 * kActConsumerWarps;  // 128 tiles, 32 KB of bf16 at most
constexpr int kActStages = 4;
constexpr int kActStageBytes = kActChunkTiles * 256;
constexpr int kActThreads = 32 * (1 + kActConsumerWarps);
constexpr int kActSmem = kActStages * kActStageBytes + 8 * (2 * kActStages) + 16 + 1024;

struct ActArgs {
    const uint8_t* x;  // bf16 [M, K]
    uint8_t* q;        // [M, K]
    float* s;          // [M, KB]
    int64_t K;
    uint32_t T, KB;
    uint32_t nchunks;
    uint64_t timeout_ns;
};

__device__ __forceinline__ int64_t tile_start(int64_t t, uint32_t KB, int64_t K) {
    const int64_t m = t / KB;
    return m * K + (t - m * KB) * 128;
}

template <bool FLAT>  // FLAT: K % 128 == 0, tile t starts at element 128 t
__global__ void __launch_bounds__(kActThreads, 1) quant_act_kernel(const ActArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t bar_base = sbase + kActStages * kActStageBytes;
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (kActStages + s); };
    volatile int* abort_flag =
        reinterpret_cast<volatile int*>(smem_raw + (bar_base - raw) + 8 * 2 * kActStages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kActStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kActConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    if (warp == 0) {
        // producer: one bulk copy per chunk of whole tiles
        int stage = 0;
        uint32_t phase = 0, issued = 0;
        for (uint32_t c = blockIdx.x; c < a.nchunks; c += gridDim.x) {
            if (!warp_wait(empty(stage), phase ^ 1u, abort_flag, a.timeout_ns)) break;
            const uint64_t t0 = static_cast<uint64_t>(c) * kActChunkTiles;
            const uint64_t t1 = t0 + kActChunkTiles < a.T ? t0 + kActChunkTiles : a.T;
            int64_t b0, b1;
            if constexpr (FLAT) {
                b0 = static_cast<int64_t>(t0) * 128;
                b1 = static_cast<int64_t>(t1) * 128;
            } else {
                b0 = tile_start(t0, a.KB, a.K);
                const int64_t last = t1 - 1, m = last / a.KB;
                b1 = min(m * a.K + (last - m * a.KB) * 128 + 128, (m + 1) * a.K);
            }
            if (elect_one()) {
                const uint32_t bytes = static_cast<uint32_t>(2 * (b1 - b0));
                mbar_arrive_expect_tx(full(stage), bytes);
                bulk_load_1d(sbase + stage * kActStageBytes, a.x + 2 * b0, bytes, full(stage));
            }
            __syncwarp();
            ++issued;
            if (++stage == kActStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        for (int s = 0; s < kActStages; ++s) {  // copies in flight land before exit
            if (static_cast<uint32_t>(s) >= issued) break;
            const uint32_t last = s + kActStages * ((issued - 1 - s) / kActStages);
            volatile int local_flag = 0;
            mbar_wait(full(s), (last / kActStages) & 1u, &local_flag, a.timeout_ns);
        }
    } else {
        const int cw = warp - 1;
        const uint32_t grp = lane >> 2, sub = lane & 3u;
        const uint32_t rot = (grp & 1u) * 8u;
        int stage = 0;
        uint32_t phase = 0;
        for (uint32_t c = blockIdx.x; c < a.nchunks; c += gridDim.x) {
            if (!warp_wait(full(stage), phase, abort_flag, a.timeout_ns)) break;
            const uint64_t t0 = static_cast<uint64_t>(c) * kActChunkTiles;
            const int64_t b0 = FLAT ? static_cast<int64_t>(t0) * 128 : tile_start(t0, a.KB, a.K);
            const uint64_t t = t0 + 8 * cw + grp;  // this group's tile
            const bool live = t < a.T;
            int64_t base;   // element offset of the tile in x / q
            int64_t len;    // elements in the tile (128, less for a K tail)
            if constexpr (FLAT) {
                base = static_cast<int64_t>(t) * 128;
                len = 128;
            } else {
                const int64_t m = static_cast<int64_t>(t / a.KB);
                const int64_t col = (static_cast<int64_t>(t) - m * a.KB) * 128;
                base = m * a.K + col;
                len = a.K - col < 128 ? a.K - col : 128;
            }
            const uint32_t st = sbase + stage * kActStageBytes + static_cast<uint32_t>(2 * (base - b0));
            uint4 v[4];
            uint32_t chunk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                chunk[j] = (4u * j + sub + rot) & 15u;
                v[j] = (live && 8 * chunk[j] < len) ? lds16(st + 16u * chunk[j]) : make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(stage));  // the stage is in registers now
            uint32_t bits = max(max(absmax_bits8(v[0]), absmax_bits8(v[1])),
                                max(absmax_bits8(v[2]), absmax_bits8(v[3])));
            bits = max(bits, __shfl_xor_sync(0xFFFFFFFFu, bits, 1));
            bits = max(bits, __shfl_xor_sync(0xFFFFFFFFu, bits, 2));
            const float amax = __uint_as_float(bits << 16);
            const float sc = tile_scale(amax);
            const bool fast = amax >= kFastDivMinAmax;
            const float r = fast ? __frcp_rn(sc) : 0.0f;
            if (live) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (8 * chunk[j] < len)
                        *reinterpret_cast<uint2*>(a.q + base + 8 * chunk[j]) = encode8_r(v[j], sc, r, fast);
                if (sub == 0) a.s[t] = sc;
            }
            if (++stage == kActStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_quant_status, FP8Q_DEVSTATUS_TIMEOUT);
}

// ---------------------------------------------------------------- weights
// One 128x128 block per stage, loaded as one 2-D TMA box (zero fill past the
// N and K edges). The consumer warps form two groups that take alternate
// blocks (the CTA's i-th block goes to stage i mod 4 and group i mod 2), so
// two blocks are encoded at once. Thread i of a group owns the 16-byte
// chunks c = i + 256 j (j = 0..7): block row c / 16, columns [8 (c % 16), +8).
constexpr int kWConsumerWarps = 16;
constexpr int kWGroups = 2;  // warp groups working on alternate blocks
constexpr int kWGroupWarps = kWConsumerWarps / kWGroups;
constexpr int kWChunksPerThread = 2048 / (32 * kWGroupWarps);
constexpr int kWStages = 4;
constexpr int kWStageBytes = 128 * 128 * 2;
constexpr int kWThreads = 32 * (1 + kWConsumerWarps);
// barriers: full[S], empty[S], red[groups] (the per-block amax exchange)
constexpr int kWBars = 2 * kWStages + kWGroups;
constexpr int kWSmem = kWStages * kWStageBytes + 8 * kWBars + 16 + 2 * 4 * kWConsumerWarps + 1024;
static_assert(kWStages % kWGroups == 0, "each group must cycle through its own stages");

struct WeightArgs {
    uint8_t* q;  // [N, K]
    float* s;    // [NB, KB]
    int64_t N, K;
    uint32_t NB, KB;
    uint64_t timeout_ns;
};

__global__ void __launch_bounds__(kWThreads, 1)
    quant_weight_kernel(const __grid_constant__ CUtensorMap tmW, const WeightArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sbase = raw + pad;
    const uint32_t bar_base = sbase + kWStages * kWStageBytes;
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (kWStages + s); };
    auto red_bar = [&](int g) { return bar_base + 8u * (2 * kWStages + g); };
    uint8_t* misc = smem_raw + pad + kWStages * kWStageBytes + 8 * kWBars;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc);
    float* red = reinterpret_cast<float*>(misc + 16);  // [2][kWConsumerWarps]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nblocks = static_cast<uint64_t>(a.NB) * a.KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kWGroupWarps);
        }
        for (int g = 0; g < kWGroups; ++g) mbar_init(red_bar(g), kWGroupWarps);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) prefetch_tmap(&tmW);
    __syncthreads();

    if (warp == 0) {
        int stage = 0;
        uint32_t phase = 0, issued = 0;
        for (uint64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
            if (!warp_wait(empty(stage), phase ^ 1u, abort_flag, a.timeout_ns)) break;
            const uint32_t nb = static_cast<uint32_t>(b / a.KB);
            const uint32_t kb = static_cast<uint32_t>(b - static_cast<uint64_t>(nb) * a.KB);
            if (elect_one()) {
                mbar_arrive_expect_tx(full(stage), kWStageBytes);
                tma_load_2d(sbase + stage * kWStageBytes, &tmW, full(stage), kb * 128, nb * 128);
            }
            __syncwarp();
            ++issued;
            if (++stage == kWStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        for (int s = 0; s < kWStages; ++s) {
            if (static_cast<uint32_t>(s) >= issued) break;
            const uint32_t last = s + kWStages * ((issued - 1 - s) / kWStages);
            volatile int local_flag = 0;
            mbar_wait(full(s), (last / kWStages) & 1u, &local_flag, a.timeout_ns);
        }
    } else {
        const int cw = warp - 1;
        const int grp = cw / kWGroupWarps, gw = cw % kWGroupWarps;
        const uint32_t tid = static_cast<uint32_t>(gw * 32 + lane);  // thread within the group
        float* red_g = red + grp * 2 * kWGroupWarps;                  // [2][kWGroupWarps]
        int stage = grp;
        uint32_t phase = 0, iter = 0;
        for (uint64_t b = blockIdx.x + static_cast<uint64_t>(grp) * gridDim.x; b < nblocks;
             b += static_cast<uint64_t>(kWGroups) * gridDim.x, ++iter) {
            if (!warp_wait(full(stage), phase, abort_flag, a.timeout_ns)) break;
            const uint32_t nb = static_cast<uint32_t>(b / a.KB);
            const uint32_t kb = static_cast<uint32_t>(b - static_cast<uint64_t>(nb) * a.KB);
            const uint32_t st = sbase + stage * kWStageBytes;
            constexpr uint32_t kStride = 32 * kWGroupWarps;
            uint4 v[kWChunksPerThread];
#pragma unroll
            for (int j = 0; j < kWChunksPerThread; ++j) v[j] = lds16(st + 16u * (tid + kStride * j));
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(stage));
            uint32_t bits = 0;
#pragma unroll
            for (int j = 0; j < kWChunksPerThread; ++j) bits = max(bits, absmax_bits8(v[j]));
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) bits = max(bits, __shfl_xor_sync(0xFFFFFFFFu, bits, d));
            // Block amax across the group's warps: each publishes its partial
            // in one half of its group's red[] (alternating per block, so a warp
            // that is a block ahead never overwrites values still being read)
            // and arrives on the group's barrier, whose phase for the group's
            // block `iter` has parity iter & 1.
            float* rb = red_g + (iter & 1u) * kWGroupWarps;
            if (lane == 0) {
                rb[gw] = __uint_as_float(bits << 16);
                mbar_arrive(red_bar(grp));
            }
            if (!warp_wait(red_bar(grp), iter & 1u, abort_flag, a.timeout_ns)) break;
            float amax = rb[0];
#pragma unroll
            for (int i = 1; i < kWGroupWarps; ++i) amax = fmaxf(amax, rb[i]);
            const float sc = tile_scale(amax);
            const bool fast = amax >= kFastDivMinAmax;
            const float r = fast ? __frcp_rn(sc) : 0.0f;
            const int64_t k = static_cast<int64_t>(kb) * 128 + 8 * (tid & 15u);
            const int64_t n0 = static_cast<int64_t>(nb) * 128 + (tid >> 4);
#pragma unroll
            for (int j = 0; j < kWChunksPerThread; ++j) {
                const int64_t n = n0 + (kStride / 16) * j;
                if (n < a.N && k < a.K)
                    *reinterpret_cast<uint2*>(a.q + n * a.K + k) = encode8_r(v[j], sc, r, fast);
            }
            if (tid == 0) a.s[b] = sc;
            stage += kWGroups;
            if (stage >= kWStages) {
                stage -= kWStages;
                phase ^= 1u;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_quant_status, FP8Q_DEVSTATUS_TIMEOUT);
}

// ------------------------------------------------------------------ gather
// One warp per output row: the row's K code bytes move as 16-byte vectors
// (four in flight per lane), its ceil(K/128) scales as 4-byte words.
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(
    const uint8_t* __restrict__ q_src, const float* __restrict__ s_src, int64_t T, int64_t K,
    uint32_t KB, const int32_t* __restrict__ index, int64_t R, uint8_t* __restrict__ q_dst,
    float* __restrict__ s_dst) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t vecs = K / 16;
    for (int64_t r = warp; r < R; r += nwarps) {
        const int64_t src = __ldg(index + r);
        const bool ok = src >= 0 && src < T;
        if (!ok && lane == 0) atomicOr(&g_quant_status, FP8Q_DEVSTATUS_BAD_INDEX);
        const uint4* in = reinterpret_cast<const uint4*>(q_src + (ok ? src : 0) * K);
        uint4* out = reinterpret_cast<uint4*>(q_dst + r * K);
        for (int64_t v0 = 0; v0 < vecs; v0 += 4 * 32) {
            uint4 buf[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t v = v0 + u * 32 + lane;
                buf[u] = (ok && v < vecs) ? __ldg(in + v) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t v = v0 + u * 32 + lane;
                if (v < vecs) out[v] = buf[u];
            }
        }
        for (uint32_t j = lane; j < KB; j += 32)
            s_dst[r * KB + j] = ok ? __ldg(s_src + src * KB + j) : 0.0f;
    }
}

}  // namespace

cudaError_t launch_gather_rows(const void* q_src, const float* s_src, int64_t T, int64_t K,
                               const int32_t* index, int64_t R, void* q_dst, float* s_dst,
                               cudaStream_t stream, int num_sms) {
    const int64_t warps_wanted = R;
    const int64_t blocks_wanted = (warps_wanted + kGatherThreads / 32 - 1) / (kGatherThreads / 32);
    const int64_t cap = static_cast<int64_t>(num_sms) * (2048 / kGatherThreads);
    const unsigned grid = static_cast<unsigned>(blocks_wanted < cap ? blocks_wanted : cap);
    gather_rows_kernel<<<grid, kGatherThreads, 0, stream>>>(
        static_cast<const uint8_t*>(q_src), s_src, T, K, static_cast<uint32_t>((K + 127) / 128),
        index, R, static_cast<uint8_t*>(q_dst), s_dst);
    return cudaGetLastError();
}

cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, void* q, float* s,
                             cudaStream_t stream, int num_sms, uint64_t timeout_ns) {
    ActArgs a;
    a.x = static_cast<const uint8_t*>(x);
    a.q = static_cast<uint8_t*>(q);
    a.s = s;
    a.K = K;
    a.KB = static_cast<uint32_t>((K + 127) / 128);
    a.T = static_cast<uint32_t>(M * a.KB);
    a.nchunks = (a.T + kActChunkTiles - 1) / kActChunkTiles;
    a.timeout_ns = timeout_ns;
    const unsigned grid = a.nchunks < static_cast<uint32_t>(num_sms) ? a.nchunks : num_sms;
    if (K % 128 == 0) {
        cudaError_t err = cudaFuncSetAttribute(quant_act_kernel<true>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kActSmem);
        if (err != cudaSuccess) return err;
        quant_act_kernel<true><<<grid, kActThreads, kActSmem, stream>>>(a);
    } else {
        cudaError_t err = cudaFuncSetAttribute(quant_act_kernel<false>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kActSmem);
        if (err != cudaSuccess) return err;
        quant_act_kernel<false><<<grid, kActThreads, kActSmem, stream>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_weight(const CUtensorMap* tmW, void* q, float* s, int64_t N, int64_t K,
                                cudaStream_t stream, int num_sms, uint64_t timeout_ns) {
    WeightArgs a;
    a.q = static_cast<uint8_t*>(q);
    a.s = s;
    a.N = N;
    a.K = K;
    a.NB = static_cast<uint32_t>((N + 127) / 128);
    a.KB = static_cast<uint32_t>((K + 127) / 128);
    a.timeout_ns = timeout_ns;
    const uint64_t nblocks = static_cast<uint64_t>(a.NB) * a.KB;
    const unsigned grid = static_cast<unsigned>(nblocks < static_cast<uint64_t>(num_sms) ? nblocks : num_sms);
    cudaError_t err =
        cudaFuncSetAttribute(quant_weight_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
    if (err != cudaSuccess) return err;
    quant_weight_kernel<<<grid, kWThreads, kWSmem, stream>>>(*tmW, a);
    return cudaGetLastError();
}

cudaError_t read_quant_status(uint32_t* out, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(out, g_quant_status, sizeof(uint32_t));
    if (err != cudaSuccess || !clear) return err;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_quant_status, &zero, sizeof(uint32_t));
}

}  // namespace fp8q
