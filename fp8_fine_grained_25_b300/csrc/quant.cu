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
//
// With the transposed output (TRANS), each group also writes its block's
// codes into a shared-memory tile [128 n][128 k] (two per group, used on
// alternate blocks), then reads it back by columns: warp w of the group
// takes rows [16 w, 16 w + 16), lane l the 4-byte column word l, and four
// 4x4 byte transposes turn the 16 words into 4 rows of qt, 16 bytes each.
constexpr int kWConsumerWarps = 16;
constexpr int kWGroups = 2;  // warp groups working on alternate blocks
constexpr int kWGroupWarps = kWConsumerWarps / kWGroups;
constexpr int kWChunksPerThread = 2048 / (32 * kWGroupWarps);
constexpr int kWStages = 4;
constexpr int kWStageBytes = 128 * 128 * 2;
constexpr int kWThreads = 32 * (1 + kWConsumerWarps);
constexpr int kWCodeTile = 128 * 128;  // bytes of one block's codes
// barriers: full[S], empty[S], red[groups] (the per-block amax exchange),
// codes[groups] (TRANS: the group's code tile is complete)
constexpr int kWBars = 2 * kWStages + 2 * kWGroups;
constexpr int kWMiscBytes = 8 * kWBars + 16 + 2 * 4 * kWConsumerWarps;
constexpr int kWSmem = kWStages * kWStageBytes + kWMiscBytes + 1024;
constexpr int kWCodeOff = kWStages * kWStageBytes + (kWMiscBytes + 127) / 128 * 128;
constexpr int kWSmemT = kWCodeOff + 2 * kWGroups * kWCodeTile + 1024;
static_assert(kWStages % kWGroups == 0, "each group must cycle through its own stages");

struct WeightArgs {
    uint8_t* q;   // [N, K], or null (TRANS only)
    float* s;     // [NB, KB], or null with q
    uint8_t* qt;  // TRANS: [K, N]
    float* st;    // TRANS: [KB, NB]
    int64_t N, K;
    uint32_t NB, KB;
    uint64_t timeout_ns;
};

// Four 4-byte words (rows r0..r3 of a byte matrix, column bytes 0..3) ->
// four words holding its columns: out[i] byte j = in[j] byte i.
__device__ __forceinline__ void transpose4x4(const uint32_t (&in)[4], uint32_t (&out)[4]) {
    const uint32_t t0 = __byte_perm(in[0], in[1], 0x5140);  // r0b0 r1b0 r0b1 r1b1
    const uint32_t t1 = __byte_perm(in[0], in[1], 0x7362);  // r0b2 r1b2 r0b3 r1b3
    const uint32_t t2 = __byte_perm(in[2], in[3], 0x5140);
    const uint32_t t3 = __byte_perm(in[2], in[3], 0x7362);
    out[0] = __byte_perm(t0, t2, 0x5410);
    out[1] = __byte_perm(t0, t2, 0x7632);
    out[2] = __byte_perm(t1, t3, 0x5410);
    out[3] = __byte_perm(t1, t3, 0x7632);
}

// The producer warp of the block quantizers: block b = (b / KB, b % KB) of a
// 2-D bf16 map (128-row, 128-column units) as one 128x128 TMA box into the
// stage ring, blocks blockIdx.x, + gridDim.x, ...; full[s] and empty[s] are
// the barriers at bar_base + 8 s and bar_base + 8 (kWStages + s).
__device__ __forceinline__ void block_producer(const CUtensorMap* tm, uint64_t nblocks, uint32_t KB,
                                               uint32_t sbase, uint32_t bar_base,
                                               volatile int* abort_flag, uint64_t timeout_ns) {
    auto full = [&](int s) { return bar_base + 8u * s; };
    auto empty = [&](int s) { return bar_base + 8u * (kWStages + s); };
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    for (uint64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        if (!warp_wait(empty(stage), phase ^ 1u, abort_flag, timeout_ns)) break;
        const uint32_t rb = static_cast<uint32_t>(b / KB);
        const uint32_t cb = static_cast<uint32_t>(b - static_cast<uint64_t>(rb) * KB);
        if (elect_one()) {
            mbar_arrive_expect_tx(full(stage), kWStageBytes);
            tma_load_2d(sbase + stage * kWStageBytes, tm, full(stage), cb * 128, rb * 128);
        }
        __syncwarp();
        ++issued;
        if (++stage == kWStages) {
            stage = 0;
            phase ^= 1u;
        }
    }
    // copies in flight land before the CTA may exit
    for (int s = 0; s < kWStages; ++s) {
        if (static_cast<uint32_t>(s) >= issued) break;
        const uint32_t last = s + kWStages * ((issued - 1 - s) / kWStages);
        volatile int local_flag = 0;
        mbar_wait(full(s), (last / kWStages) & 1u, &local_flag, timeout_ns);
    }
}

template <bool TRANS>
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
    auto codes_bar = [&](int g) { return bar_base + 8u * (2 * kWStages + kWGroups + g); };
    uint8_t* misc = smem_raw + pad + kWStages * kWStageBytes + 8 * kWBars;
    // TRANS: code tiles [group][2][128 x 128], after the barriers and misc
    const uint32_t code_base = sbase + kWCodeOff;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc);
    float* red = reinterpret_cast<float*>(misc + 16);  // [2][kWConsumerWarps]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nblocks = static_cast<uint64_t>(a.NB) * a.KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kWGroupWarps);
        }
        for (int g = 0; g < kWGroups; ++g) {
            mbar_init(red_bar(g), kWGroupWarps);
            mbar_init(codes_bar(g), kWGroupWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) prefetch_tmap(&tmW);
    __syncthreads();

    if (warp == 0) {
        block_producer(&tmW, nblocks, a.KB, sbase, bar_base, abort_flag, a.timeout_ns);
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
            // this group's code tile for this block (TRANS)
            const uint32_t ct = code_base + (2 * grp + (iter & 1u)) * kWCodeTile;
#pragma unroll
            for (int j = 0; j < kWChunksPerThread; ++j) {
                const int64_t n = n0 + (kStride / 16) * j;
                const uint2 code = encode8_r(v[j], sc, r, fast);
                if (a.q != nullptr && n < a.N && k < a.K)
                    *reinterpret_cast<uint2*>(a.q + n * a.K + k) = code;
                if constexpr (TRANS) {
                    // tile row (tid >> 4) + 16 j, bytes 8 (tid & 15) .. + 7
                    const uint32_t off = 128u * ((tid >> 4) + (kStride / 16) * j) + 8u * (tid & 15u);
                    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(ct + off), "r"(code.x),
                                 "r"(code.y)
                                 : "memory");
                }
            }
            if (tid == 0) {
                if (a.s != nullptr) a.s[b] = sc;
                if constexpr (TRANS) a.st[static_cast<uint64_t>(kb) * a.NB + nb] = sc;
            }
            if constexpr (TRANS) {
                // All of the group's codes are in the tile once every warp has
                // arrived; the tile used two blocks ago is free, because every
                // warp passed this block's amax exchange after its last read.
                __syncwarp();
                if (lane == 0) mbar_arrive(codes_bar(grp));
                if (!warp_wait(codes_bar(grp), iter & 1u, abort_flag, a.timeout_ns)) break;
                const int64_t nrow = static_cast<int64_t>(nb) * 128 + 16 * gw;  // first n of the warp
                uint32_t cols[4][4];  // [row quad][k byte i] -> 4 codes of n = nrow + 4 quad ..
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    uint32_t w[4];
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) {
                        const uint32_t addr = ct + 128u * (16 * gw + 4 * qd + rr) + 4u * lane;
                        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[rr]) : "r"(addr));
                    }
                    transpose4x4(w, cols[qd]);
                }
                if (nrow < a.N) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int64_t kk = static_cast<int64_t>(kb) * 128 + 4 * lane + i;
                        if (kk < a.K)
                            *reinterpret_cast<uint4*>(a.qt + kk * a.N + nrow) =
                                make_uint4(cols[0][i], cols[1][i], cols[2][i], cols[3][i]);
                    }
                }
            }
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

// ------------------------------------------------- activations, transposed
// 128x1 tiles (one column, 128 consecutive rows): block (mb, kb) of x [M, K]
// is one 128x128 TMA box holding 128 tiles, one per column. In a group, lane
// l of warp w takes the column pair p = l + 32 (w & 1) (columns 2p, 2p + 1)
// over the rows [32 (w >> 1), +32): one 4-byte word per row, so each
// warp-wide load reads 32 consecutive words of one row. The four row
// segments' column maxima meet in shared memory; each thread then encodes
// its 2 x 32 values and writes 32 bytes into each of two rows of qt.
struct ActTArgs {
    uint8_t* qt;  // [K, M]
    float* st;    // [K, MB]
    int64_t M, K;
    uint32_t MB, KB;
    uint64_t timeout_ns;
};

constexpr int kTRedWords = 2 * 4 * 64;  // per group: [parity][row segment][column pair]
constexpr int kTMiscBytes = 8 * kWBars + 16 + kWGroups * kTRedWords * 4;
constexpr int kTSmem = kWStages * kWStageBytes + kTMiscBytes + 1024;

// 32 values of one tile column (bf16 in the low or high half of w[r]) with
// scale s and reciprocal r (0: the IEEE-divide range) -> 32 codes, row order.
template <bool HI>
__device__ __forceinline__ float col_value(uint32_t v) {
    return __uint_as_float(HI ? (v & 0xFFFF0000u) : (v << 16));
}

template <bool HI>
__device__ __forceinline__ void encode_col32(const uint32_t (&w)[32], float s, float r, bool fast,
                                             uint32_t (&out)[8]) {
    if (s == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = 0u;
    } else if (fast) {  // one branch per column, not per element
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float y0 = div_by_scale(col_value<HI>(w[4 * i]), s, r);
            const float y1 = div_by_scale(col_value<HI>(w[4 * i + 1]), s, r);
            const float y2 = div_by_scale(col_value<HI>(w[4 * i + 2]), s, r);
            const float y3 = div_by_scale(col_value<HI>(w[4 * i + 3]), s, r);
            out[i] = e4m3x2(y0, y1) | (e4m3x2(y2, y3) << 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float y0 = __fdiv_rn(col_value<HI>(w[4 * i]), s);
            const float y1 = __fdiv_rn(col_value<HI>(w[4 * i + 1]), s);
            const float y2 = __fdiv_rn(col_value<HI>(w[4 * i + 2]), s);
            const float y3 = __fdiv_rn(col_value<HI>(w[4 * i + 3]), s);
            out[i] = e4m3x2(y0, y1) | (e4m3x2(y2, y3) << 16);
        }
    }
}

__global__ void __launch_bounds__(kWThreads, 1)
    quant_act_t_kernel(const __grid_constant__ CUtensorMap tmX, const ActTArgs a) {
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
    uint32_t* red = reinterpret_cast<uint32_t*>(misc + 16);  // [groups][kTRedWords]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nblocks = static_cast<uint64_t>(a.MB) * a.KB;

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
    if (warp == 0 && lane == 0) prefetch_tmap(&tmX);
    __syncthreads();

    if (warp == 0) {
        block_producer(&tmX, nblocks, a.KB, sbase, bar_base, abort_flag, a.timeout_ns);
    } else {
        const int cw = warp - 1;
        const int grp = cw / kWGroupWarps, gw = cw % kWGroupWarps;
        const uint32_t pr = static_cast<uint32_t>(lane) + 32u * (gw & 1);  // column pair
        const uint32_t seg = static_cast<uint32_t>(gw >> 1);               // row segment
        uint32_t* red_g = red + grp * kTRedWords;
        int stage = grp;
        uint32_t phase = 0, iter = 0;
        for (uint64_t b = blockIdx.x + static_cast<uint64_t>(grp) * gridDim.x; b < nblocks;
             b += static_cast<uint64_t>(kWGroups) * gridDim.x, ++iter) {
            if (!warp_wait(full(stage), phase, abort_flag, a.timeout_ns)) break;
            const uint32_t mb = static_cast<uint32_t>(b / a.KB);
            const uint32_t kb = static_cast<uint32_t>(b - static_cast<uint64_t>(mb) * a.KB);
            const uint32_t st = sbase + stage * kWStageBytes + 256u * 32u * seg + 4u * pr;
            uint32_t w[32];
#pragma unroll
            for (int r = 0; r < 32; ++r)
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[r]) : "r"(st + 256u * r));
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(stage));
            uint32_t mx = 0;
#pragma unroll
            for (int r = 0; r < 32; ++r) mx = __vmaxu2(mx, w[r] & 0x7FFF7FFFu);
            // column maxima across the four row segments (halves of red_g
            // alternate per block, as in the weight kernel's exchange)
            uint32_t* rb = red_g + (iter & 1u) * (kTRedWords / 2);
            rb[64 * seg + pr] = mx;
            __syncwarp();
            if (lane == 0) mbar_arrive(red_bar(grp));
            if (!warp_wait(red_bar(grp), iter & 1u, abort_flag, a.timeout_ns)) break;
            const uint32_t m2 = __vmaxu2(__vmaxu2(rb[pr], rb[64 + pr]), __vmaxu2(rb[128 + pr], rb[192 + pr]));
            const float amax0 = __uint_as_float(m2 << 16), amax1 = __uint_as_float(m2 & 0xFFFF0000u);
            const float s0 = tile_scale(amax0), s1 = tile_scale(amax1);
            const bool fast0 = amax0 >= kFastDivMinAmax, fast1 = amax1 >= kFastDivMinAmax;
            const float r0 = fast0 ? __frcp_rn(s0) : 0.0f, r1 = fast1 ? __frcp_rn(s1) : 0.0f;
            uint32_t c0[8], c1[8];
            encode_col32<false>(w, s0, r0, fast0, c0);
            encode_col32<true>(w, s1, r1, fast1, c1);
            const int64_t k = static_cast<int64_t>(kb) * 128 + 2 * pr;
            const int64_t m0 = static_cast<int64_t>(mb) * 128 + 32 * seg;
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // 16 rows each (M % 16 == 0)
                if (m0 + 16 * h < a.M) {
                    if (k < a.K)
                        *reinterpret_cast<uint4*>(a.qt + k * a.M + m0 + 16 * h) =
                            make_uint4(c0[4 * h], c0[4 * h + 1], c0[4 * h + 2], c0[4 * h + 3]);
                    if (k + 1 < a.K)
                        *reinterpret_cast<uint4*>(a.qt + (k + 1) * a.M + m0 + 16 * h) =
                            make_uint4(c1[4 * h], c1[4 * h + 1], c1[4 * h + 2], c1[4 * h + 3]);
                }
            }
            if (seg == 0) {
                if (k < a.K) a.st[k * a.MB + mb] = s0;
                if (k + 1 < a.K) a.st[(k + 1) * a.MB + mb] = s1;
            }
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

cudaError_t launch_quant_weight(const CUtensorMap* tmW, void* q, float* s, void* qt, float* st,
                                int64_t N, int64_t K, cudaStream_t stream, int num_sms,
                                uint64_t timeout_ns) {
    WeightArgs a;
    a.q = static_cast<uint8_t*>(q);
    a.s = s;
    a.qt = static_cast<uint8_t*>(qt);
    a.st = st;
    a.N = N;
    a.K = K;
    a.NB = static_cast<uint32_t>((N + 127) / 128);
    a.KB = static_cast<uint32_t>((K + 127) / 128);
    a.timeout_ns = timeout_ns;
    const uint64_t nblocks = static_cast<uint64_t>(a.NB) * a.KB;
    const unsigned grid = static_cast<unsigned>(nblocks < static_cast<uint64_t>(num_sms) ? nblocks : num_sms);
    if (qt != nullptr) {
        cudaError_t err = cudaFuncSetAttribute(quant_weight_kernel<true>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmemT);
        if (err != cudaSuccess) return err;
        quant_weight_kernel<true><<<grid, kWThreads, kWSmemT, stream>>>(*tmW, a);
    } else {
        cudaError_t err = cudaFuncSetAttribute(quant_weight_kernel<false>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
        if (err != cudaSuccess) return err;
        quant_weight_kernel<false><<<grid, kWThreads, kWSmem, stream>>>(*tmW, a);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_act_t(const CUtensorMap* tmX, void* qt, float* st, int64_t M, int64_t K,
                               cudaStream_t stream, int num_sms, uint64_t timeout_ns) {
    ActTArgs a;
    a.qt = static_cast<uint8_t*>(qt);
    a.st = st;
    a.M = M;
    a.K = K;
    a.MB = static_cast<uint32_t>((M + 127) / 128);
    a.KB = static_cast<uint32_t>((K + 127) / 128);
    a.timeout_ns = timeout_ns;
    const uint64_t nblocks = static_cast<uint64_t>(a.MB) * a.KB;
    const unsigned grid = static_cast<unsigned>(nblocks < static_cast<uint64_t>(num_sms) ? nblocks : num_sms);
    cudaError_t err =
        cudaFuncSetAttribute(quant_act_t_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmem);
    if (err != cudaSuccess) return err;
    quant_act_t_kernel<<<grid, kWThreads, kTSmem, stream>>>(*tmX, a);
    return cudaGetLastError();
}

cudaError_t read_quant_status(uint32_t* out, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(out, g_quant_status, sizeof(uint32_t));
    if (err != cudaSuccess || !clear) return err;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_quant_status, &zero, sizeof(uint32_t));
}

}  // namespace fp8q
