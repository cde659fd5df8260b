// Fine-grained FP8 quantizers: activations per 1x128 tile, weights per
// 128x128 block (news.qq.com/rain/a/20241229A05OQF00, "FP8 低精度训练",
// item "细粒度量化", Fig. 7a; developer.aliyun.com/article/1776647 §4.1), and
// the transposed layouts the backward GEMMs read.
//
// All are HBM-bound streams: 2 bytes read and 1 byte written per element
// (2 for both layouts) plus one fp32 scale per tile/block.
//  - Row-major outputs (quant_act, quant_weight): a producer warp streams the
//    input into a ring of shared-memory stages with bulk copies (TMA), so the
//    bytes in flight do not depend on registers; consumer warps read a stage,
//    reduce the amax, encode, and store codes and scales.
//  - Transposed outputs (quant_act_t, quant_weight_t): persistent CTAs read
//    128x128 blocks straight into registers (the next block's loads in flight
//    while the current one is encoded) and write 16-byte runs of the
//    transposed codes; the block order keeps those runs adjacent.
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

// Two quotients at once on packed pairs: (y0, y1) = (x0 / s0, x1 / s1) by
// the steps of div_by_scale (q0 = RN(x r), e = RN(q0 s - x) exact,
// q = RN(q0 - e r)), written with nx = -x and nr = -r so that every step is
// a plain packed multiply or FMA; bit-identical to div_by_scale per lane.
__device__ __forceinline__ void div2_by_scale(float x0, float x1, float nx0, float nx1, float s0,
                                              float s1, float r0, float r1, float nr0, float nr1,
                                              float& y0, float& y1) {
    asm("{\n\t.reg .b64 x, nx, s, r, nr, q, e;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 nx, {%4, %5};\n\t"
        "mov.b64 s, {%6, %7};\n\t"
        "mov.b64 r, {%8, %9};\n\t"
        "mov.b64 nr, {%10, %11};\n\t"
        "mul.rn.f32x2 q, x, r;\n\t"
        "fma.rn.f32x2 e, q, s, nx;\n\t"
        "fma.rn.f32x2 q, e, nr, q;\n\t"
        "mov.b64 {%0, %1}, q;\n\t}"
        : "=f"(y0), "=f"(y1)
        : "f"(x0), "f"(x1), "f"(nx0), "f"(nx1), "f"(s0), "f"(s1), "f"(r0), "f"(r1), "f"(nr0),
          "f"(nr1));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// the same, negated (the sign bit flipped)
__device__ __forceinline__ float bf16_lo_neg(uint32_t w) { return __uint_as_float(w * 65536u + 0x80000000u); }
__device__ __forceinline__ float bf16_hi_neg(uint32_t w) { return __uint_as_float((w & 0xFFFF0000u) ^ 0x80000000u); }

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

// Power-of-two (UE8M0) scales: the byte e + 127 of the smallest power of two
// 2^e with amax / 2^e <= 448, clamped below at 0. With amax's fp32 exponent
// field E8 and mantissa field m, amax / 448 = (1.m / 1.75) * 2^(E8 - 135), so
// e = E8 - 135 when 1.m <= 1.75 and E8 - 134 otherwise; subnormal and zero
// amax clamp to byte 0.
__device__ __forceinline__ uint32_t ue8m0_byte(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int v = static_cast<int>((b >> 23) & 0xFFu) - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return v < 0 ? 0u : static_cast<uint32_t>(v);
}
// 2^(byte - 127) (2^-127 is an fp32 subnormal) and 2^(127 - byte), byte <= 253
__device__ __forceinline__ float pow2_of_byte(uint32_t byte) {
    return byte == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(byte << 23);
}
__device__ __forceinline__ float inv_pow2_of_byte(uint32_t byte) { return __uint_as_float((254u - byte) << 23); }

// The tile's scale, reciprocal and fast-path flag for encode8_r. POW2: the
// UE8M0 scale, for which x * 2^-e is exact, so the correction step of
// div_by_scale is zero and the fast path always applies; all-zero tiles get
// s = 0 (codes 0) and byte 0.
template <bool POW2>
__device__ __forceinline__ void tile_scale_for(float amax, float& sc, float& r, bool& fast, uint32_t& byte) {
    if constexpr (POW2) {
        byte = ue8m0_byte(amax);
        sc = amax == 0.0f ? 0.0f : pow2_of_byte(byte);
        r = inv_pow2_of_byte(byte);
        fast = true;
    } else {
        sc = tile_scale(amax);
        fast = amax >= kFastDivMinAmax;
        r = fast ? __frcp_rn(sc) : 0.0f;
        byte = 0;
    }
}

// Eight values of a tile whose scale s and reciprocal r = RN(1/s) (or 0 for
// the IEEE-divide range, amax < 2^-90) are known, encoded low byte first.
// PACKED runs the quotients two lanes per instruction (same results); the
// weight kernel gains from it, while the activation kernel measured slower
// with it at 32768 rows (6.55 -> 5.88 TB/s) and keeps the scalar form.
template <bool PACKED>
__device__ __forceinline__ uint2 encode8_r(const uint4& v, float s, float r, bool fast) {
    if (s == 0.0f) return make_uint2(0u, 0u);
    float f[8], y[8];
    unpack_bf16x8(v, f);
    if (fast && PACKED) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            div2_by_scale(bf16_lo(w[i]), bf16_hi(w[i]), bf16_lo_neg(w[i]), bf16_hi_neg(w[i]), s, s, r, r,
                          -r, -r, y[2 * i], y[2 * i + 1]);
    } else if (fast) {
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
// j = 0..3, of the tile's 256 bytes. A 16-byte shared load is served 8
// lanes (two tiles 256 bytes apart) per pass, and with this rotation the two
// tiles' chunks share banks: ncu counts 2 wavefronts per pass where 1 would
// do. A rotation by 4 removes the conflicts but measured no faster (equal at
// 8192 x 7168, 3 % slower at 32768 x 7168): the kernel is bound by HBM, not
// by shared memory.
constexpr int kActConsumerWarps = 16;
constexpr int kActChunkTiles = 8 * kActConsumerWarps;  // 128 tiles, 32 KB of bf16 at most
constexpr int kActStages = 4;
constexpr int kActStageBytes = kActChunkTiles * 256;
constexpr int kActThreads = 32 * (1 + kActConsumerWarps);
constexpr int kActSmem = kActStages * kActStageBytes + 8 * (2 * kActStages) + 16 + 1024;

struct ActArgs {
    const uint8_t* x;  // bf16 [M, K]
    uint8_t* q;        // [M, K]
    float* s;          // [M, KB] fp32 scales
    uint8_t* s8;       // [M, KB] UE8M0 scale bytes (POW2)
    int64_t K;
    uint32_t T, KB;
    uint32_t nchunks;
    uint64_t timeout_ns;
};

__device__ __forceinline__ int64_t tile_start(int64_t t, uint32_t KB, int64_t K) {
    const int64_t m = t / KB;
    return m * K + (t - m * KB) * 128;
}

// FLAT: K % 128 == 0, tile t starts at element 128 t; POW2: UE8M0 scales
template <bool FLAT, bool POW2>
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
            float sc, r;
            bool fast;
            uint32_t byte;
            tile_scale_for<POW2>(amax, sc, r, fast, byte);
            if (live) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (8 * chunk[j] < len)
                        *reinterpret_cast<uint2*>(a.q + base + 8 * chunk[j]) = encode8_r<false>(v[j], sc, r, fast);
                if (sub == 0) {
                    if constexpr (POW2) a.s8[t] = static_cast<uint8_t>(byte);
                    else a.s[t] = sc;
                }
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
// N and K edges). The consumer warps form three groups of 8 that take the
// CTA's blocks in turn (the CTA's i-th block goes to stage i mod 6 and group
// i mod 3), so three blocks are encoded at once while three more load; each
// group double-buffers through its own two stages. Thread i of a group owns
// the 16-byte chunks c = i + 256 j (j = 0..7): block row c / 16, columns
// [8 (c % 16), +8). Measured on the B300 at 7168 x 7168, launched alone:
// 32.8 us with two groups and four stages, 29.0-29.6 us with three groups
// and six stages (four groups of four warps: 30.7 us; six of four warps
// spill registers at 800 threads).
constexpr int kWConsumerWarps = 24;
constexpr int kWGroups = 3;  // warp groups working on the CTA's blocks in turn
constexpr int kWGroupWarps = kWConsumerWarps / kWGroups;
constexpr int kWChunksPerThread = 2048 / (32 * kWGroupWarps);
constexpr int kWStages = 6;
constexpr int kWStageBytes = 128 * 128 * 2;
constexpr int kWThreads = 32 * (1 + kWConsumerWarps);
// barriers: full[S], empty[S], red[groups] (the per-block amax exchange)
constexpr int kWBars = 2 * kWStages + kWGroups;
constexpr int kWSmem = kWStages * kWStageBytes + 8 * kWBars + 16 + 2 * 4 * kWConsumerWarps + 1024;
static_assert(kWStages % kWGroups == 0, "each group must cycle through its own stages");

struct WeightArgs {
    uint8_t* q;  // [N, K]
    float* s;    // [NB, KB] fp32 scales
    uint8_t* s8; // [NB, KB] UE8M0 scale bytes (POW2)
    int64_t N, K;
    uint32_t NB, KB;
    uint64_t timeout_ns;
};

template <bool POW2>  // POW2: UE8M0 scales
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
            float sc, r;
            bool fast;
            uint32_t byte;
            tile_scale_for<POW2>(amax, sc, r, fast, byte);
            const int64_t k = static_cast<int64_t>(kb) * 128 + 8 * (tid & 15u);
            const int64_t n0 = static_cast<int64_t>(nb) * 128 + (tid >> 4);
#pragma unroll
            for (int j = 0; j < kWChunksPerThread; ++j) {
                const int64_t n = n0 + (kStride / 16) * j;
                if (n < a.N && k < a.K)
                    *reinterpret_cast<uint2*>(a.q + n * a.K + k) = encode8_r<true>(v[j], sc, r, fast);
            }
            if (tid == 0) {
                if constexpr (POW2) a.s8[b] = static_cast<uint8_t>(byte);
                else a.s[b] = sc;
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
// 128x1 tiles (one column, 128 consecutive rows), codes written transposed.
// A CTA of 256 threads handles 128x128 blocks b = blockIdx.x, + gridDim.x,
// ...; block b is (mb, kb) = (b % MB, b / MB), so the CTAs running at the
// same time cover consecutive 128-row blocks of the same columns and their
// writes to qt form long runs. In a block, warp w holds rows [16 w, 16 w +
// 16) and lane l columns [4 l, 4 l + 4), read with 8-byte loads (a warp reads
// 256 contiguous bytes of a row). The loads of the CTA's next block are
// issued before the current block is encoded, so two blocks per CTA are in
// flight. Column maxima meet in shared memory, one thread per column forms
// the column's scale and reciprocal, and each thread then encodes its 16 x 4
// values and writes one 16-byte run of qt per column.
constexpr int kTThreads = 256;

struct ActTArgs {
    const uint8_t* x;  // bf16 [M, K]
    uint8_t* qt;       // [K, M]
    float* st;         // [K, MB] fp32 scales
    uint8_t* st8;      // [K, MB] UE8M0 scale bytes (POW2)
    int64_t M, K;
    uint32_t MB, KB;
};

// Four columns x four rows: y[i][c] = x[row i][column c] / s_c, rows from
// the words v[i] (columns 0, 1 in .x, 2, 3 in .y), then the codes of each
// column's four rows packed low row first.
template <bool FAST>
__device__ __forceinline__ void encode_quad(const uint2 (&v)[4], const float4& s, const float4& r,
                                            const float4& nr, uint32_t (&code)[4]) {
    float y[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = v[i].x, b = v[i].y;
        if constexpr (FAST) {
            div2_by_scale(bf16_lo(a), bf16_hi(a), bf16_lo_neg(a), bf16_hi_neg(a), s.x, s.y, r.x, r.y,
                          nr.x, nr.y, y[i][0], y[i][1]);
            div2_by_scale(bf16_lo(b), bf16_hi(b), bf16_lo_neg(b), bf16_hi_neg(b), s.z, s.w, r.z, r.w,
                          nr.z, nr.w, y[i][2], y[i][3]);
        } else {
            y[i][0] = __fdiv_rn(bf16_lo(a), s.x);
            y[i][1] = __fdiv_rn(bf16_hi(a), s.y);
            y[i][2] = __fdiv_rn(bf16_lo(b), s.z);
            y[i][3] = __fdiv_rn(bf16_hi(b), s.w);
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) code[c] = e4m3x2(y[0][c], y[1][c]) | (e4m3x2(y[2][c], y[3][c]) << 16);
}

__device__ __forceinline__ void load_block_t(const ActTArgs& a, uint32_t b, int w, int l,
                                             uint2 (&v)[16]) {
    const uint32_t mb = b % a.MB, kb = b / a.MB;
    const int64_t k = static_cast<int64_t>(kb) * 128 + 4 * l;
    const int64_t m0 = static_cast<int64_t>(mb) * 128 + 16 * w;
    const bool live = k < a.K && m0 < a.M;  // K % 4 == 0 and M % 16 == 0: all or nothing
    const uint2* src = reinterpret_cast<const uint2*>(a.x + 2 * (live ? m0 * a.K + k : 0));
    const int64_t pitch = a.K / 4;  // uint2 per row
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = live ? __ldg(src + i * pitch) : make_uint2(0u, 0u);
}

template <bool POW2>  // POW2: UE8M0 scales
__global__ void __launch_bounds__(kTThreads, 2) quant_act_t_kernel(const ActTArgs a) {
    __shared__ uint32_t red[8][64];  // [warp][column pair]: packed |bf16| maxima
    __shared__ float4 s_sh[32], r_sh[32];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const uint32_t nblocks = a.MB * a.KB;
    uint2 v[16];
    if (blockIdx.x < nblocks) load_block_t(a, blockIdx.x, w, l, v);
    for (uint32_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        uint2 vn[16];
        if (b + gridDim.x < nblocks) load_block_t(a, b + gridDim.x, w, l, vn);
        const uint32_t mb = b % a.MB, kb = b / a.MB;
        const int64_t k = static_cast<int64_t>(kb) * 128 + 4 * l;
        const int64_t m0 = static_cast<int64_t>(mb) * 128 + 16 * w;
        const bool live = k < a.K && m0 < a.M;
        uint32_t mx0 = 0, mx1 = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            mx0 = __vmaxu2(mx0, v[i].x & 0x7FFF7FFFu);
            mx1 = __vmaxu2(mx1, v[i].y & 0x7FFF7FFFu);
        }
        red[w][2 * l] = mx0;
        red[w][2 * l + 1] = mx1;
        __syncthreads();
        if (threadIdx.x < 128) {
            const int c = threadIdx.x;  // column of the block
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = __vmaxu2(m, red[i][c >> 1]);
            const float amax = __uint_as_float((c & 1) ? (m & 0xFFFF0000u) : (m << 16));
            float sc, rc;
            bool fast;
            uint32_t byte;
            tile_scale_for<POW2>(amax, sc, rc, fast, byte);
            if (!fast) rc = 0.0f;  // the IEEE-divide range (fp32 scales only)
            reinterpret_cast<float*>(s_sh)[c] = sc;
            reinterpret_cast<float*>(r_sh)[c] = rc;
            const int64_t col = static_cast<int64_t>(kb) * 128 + c;
            if (col < a.K) {
                if constexpr (POW2) a.st8[col * a.MB + mb] = static_cast<uint8_t>(byte);
                else a.st[col * a.MB + mb] = sc;
            }
        }
        __syncthreads();
        if (live) {
            const float4 s = s_sh[l], r = r_sh[l];
            const float4 nr = make_float4(-r.x, -r.y, -r.z, -r.w);
            // every column either all-zero (s = 0, masked below) or in the fast range
            const bool fast = (s.x == 0.0f || r.x != 0.0f) && (s.y == 0.0f || r.y != 0.0f) &&
                              (s.z == 0.0f || r.z != 0.0f) && (s.w == 0.0f || r.w != 0.0f);
            uint32_t code[4][4];  // [column][row quad]
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint2 vq[4] = {v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]};
                uint32_t cq[4];
                if (fast) encode_quad<true>(vq, s, r, nr, cq);
                else encode_quad<false>(vq, s, r, nr, cq);
#pragma unroll
                for (int c = 0; c < 4; ++c) code[c][q] = cq[c];
            }
            const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 out = sv[c] == 0.0f
                                      ? make_uint4(0u, 0u, 0u, 0u)
                                      : make_uint4(code[c][0], code[c][1], code[c][2], code[c][3]);
                *reinterpret_cast<uint4*>(a.qt + (k + c) * a.M + m0) = out;
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = vn[i];
    }
}

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

// ------------------------------------------------- weights, plain blocks
// 128x128 blocks with one scale each, the same thread layout as the
// transposed activation kernel (warp w: rows [16 w, +16); lane l: columns
// [4 l, +4); the next block's loads in flight while the current one is
// encoded). WQ writes the codes row-major (q [N, K], 4 bytes per row per
// lane: a warp writes 128 contiguous bytes of each row), WT transposed
// (qt [K, N], one 16-byte run per column per lane). Blocks are taken with
// the 128-row blocks fastest when WT is set (runs along qt rows), else the
// 128-column blocks fastest (runs along q rows).
struct WeightPlainArgs {
    const uint8_t* w;  // bf16 [N, K]
    uint8_t* q;        // [N, K] (WQ)
    float* s;          // [NB, KB] (WQ)
    uint8_t* s8;       // [NB, KB] UE8M0 bytes (WQ, POW2)
    uint8_t* qt;       // [K, N] (WT)
    float* st;         // [KB, NB] (WT)
    uint8_t* st8;      // [KB, NB] UE8M0 bytes (WT, POW2)
    int64_t N, K;
    uint32_t NB, KB;
};

template <bool WT>
__device__ __forceinline__ void weight_block_coords(const WeightPlainArgs& a, uint32_t b, uint32_t& nb,
                                                    uint32_t& kb) {
    if constexpr (WT) {
        nb = b % a.NB;
        kb = b / a.NB;
    } else {
        kb = b % a.KB;
        nb = b / a.KB;
    }
}

template <bool WT>
__device__ __forceinline__ void load_weight_block(const WeightPlainArgs& a, uint32_t b, int w, int l,
                                                  uint2 (&v)[16]) {
    uint32_t nb, kb;
    weight_block_coords<WT>(a, b, nb, kb);
    const int64_t k = static_cast<int64_t>(kb) * 128 + 4 * l;
    const int64_t n0 = static_cast<int64_t>(nb) * 128 + 16 * w;
    const uint2* src = reinterpret_cast<const uint2*>(a.w + 2 * (k < a.K ? n0 * a.K + k : 0));
    const int64_t pitch = a.K / 4;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = (k < a.K && n0 + i < a.N) ? __ldg(src + i * pitch) : make_uint2(0u, 0u);
}

template <bool WQ, bool WT, bool POW2>  // POW2: UE8M0 scales
__global__ void __launch_bounds__(kTThreads, 2) quant_weight_plain_kernel(const WeightPlainArgs a) {
    // per-warp partial maxima, double-buffered by block parity: one barrier
    // per block, after which every thread forms the block scale itself.
    // Why one barrier suffices: a warp writes red[p] for block b + 2 only
    // after it has passed the barrier of block b + 1, and every warp reads
    // red[p] for block b before it arrives at that barrier, so no write to a
    // buffer can land while another warp still reads that buffer's previous
    // contents (a warp is at most one block ahead of the slowest one).
    __shared__ uint32_t red[2][8];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const uint32_t nblocks = a.NB * a.KB;
    uint32_t par = 0;
    uint2 v[16];
    if (blockIdx.x < nblocks) load_weight_block<WT>(a, blockIdx.x, w, l, v);
    for (uint32_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        uint2 vn[16];
        if (b + gridDim.x < nblocks) load_weight_block<WT>(a, b + gridDim.x, w, l, vn);
        uint32_t nb, kb;
        weight_block_coords<WT>(a, b, nb, kb);
        const int64_t k = static_cast<int64_t>(kb) * 128 + 4 * l;
        const int64_t n0 = static_cast<int64_t>(nb) * 128 + 16 * w;
        uint32_t mx = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) mx = __vmaxu2(mx, __vmaxu2(v[i].x & 0x7FFF7FFFu, v[i].y & 0x7FFF7FFFu));
        mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, d));
        if (l == 0) red[par][w] = mx;
        __syncthreads();
        uint32_t m = red[par][0];
#pragma unroll
        for (int i = 1; i < 8; ++i) m = max(m, red[par][i]);
        par ^= 1u;
        const float amax = __uint_as_float(m << 16);
        float sc, rc;
        bool fast;
        uint32_t byte;
        tile_scale_for<POW2>(amax, sc, rc, fast, byte);
        const float2 sr = make_float2(sc, fast ? rc : 0.0f);
        if (threadIdx.x == 0) {
            if constexpr (POW2) {
                if constexpr (WQ) a.s8[static_cast<uint64_t>(nb) * a.KB + kb] = static_cast<uint8_t>(byte);
                if constexpr (WT) a.st8[static_cast<uint64_t>(kb) * a.NB + nb] = static_cast<uint8_t>(byte);
            } else {
                if constexpr (WQ) a.s[static_cast<uint64_t>(nb) * a.KB + kb] = sc;
                if constexpr (WT) a.st[static_cast<uint64_t>(kb) * a.NB + nb] = sc;
            }
        }
        if (k < a.K && sr.x != 0.0f) {
            const float4 s4 = make_float4(sr.x, sr.x, sr.x, sr.x);
            const float4 r4 = make_float4(sr.y, sr.y, sr.y, sr.y);
            const float4 nr4 = make_float4(-sr.y, -sr.y, -sr.y, -sr.y);
            uint32_t colc[4][4];  // [column][row quad]
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint2 vq[4] = {v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]};
                uint32_t cq[4];
                if (sr.y != 0.0f) encode_quad<true>(vq, s4, r4, nr4, cq);
                else encode_quad<false>(vq, s4, r4, nr4, cq);
                if constexpr (WQ) {
                    uint32_t rows[4];  // row i: the codes of columns k .. k + 3
                    transpose4x4(cq, rows);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (n0 + 4 * q + i < a.N)
                            *reinterpret_cast<uint32_t*>(a.q + (n0 + 4 * q + i) * a.K + k) = rows[i];
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) colc[c][q] = cq[c];
            }
            if constexpr (WT) {
                if (n0 < a.N) {  // N % 16 == 0: the 16 rows are all present
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(a.qt + (k + c) * a.N + n0) =
                            make_uint4(colc[c][0], colc[c][1], colc[c][2], colc[c][3]);
                }
            }
        } else if (k < a.K) {  // all-zero block: codes 0
            if constexpr (WQ) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (n0 + i < a.N) *reinterpret_cast<uint32_t*>(a.q + (n0 + i) * a.K + k) = 0u;
            }
            if constexpr (WT) {
                if (n0 < a.N) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(a.qt + (k + c) * a.N + n0) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = vn[i];
    }
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

template <bool FLAT, bool POW2>
cudaError_t launch_act(const ActArgs& a, unsigned grid, cudaStream_t stream) {
    cudaError_t err = cudaFuncSetAttribute(quant_act_kernel<FLAT, POW2>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kActSmem);
    if (err != cudaSuccess) return err;
    quant_act_kernel<FLAT, POW2><<<grid, kActThreads, kActSmem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, void* q, void* s, bool pow2,
                             cudaStream_t stream, int num_sms, uint64_t timeout_ns) {
    ActArgs a;
    a.x = static_cast<const uint8_t*>(x);
    a.q = static_cast<uint8_t*>(q);
    a.s = pow2 ? nullptr : static_cast<float*>(s);
    a.s8 = pow2 ? static_cast<uint8_t*>(s) : nullptr;
    a.K = K;
    a.KB = static_cast<uint32_t>((K + 127) / 128);
    a.T = static_cast<uint32_t>(M * a.KB);
    a.nchunks = (a.T + kActChunkTiles - 1) / kActChunkTiles;
    a.timeout_ns = timeout_ns;
    const unsigned grid = a.nchunks < static_cast<uint32_t>(num_sms) ? a.nchunks : num_sms;
    if (K % 128 == 0) return pow2 ? launch_act<true, true>(a, grid, stream) : launch_act<true, false>(a, grid, stream);
    return pow2 ? launch_act<false, true>(a, grid, stream) : launch_act<false, false>(a, grid, stream);
}

cudaError_t launch_quant_weight(const CUtensorMap* tmW, void* q, void* s, bool pow2, int64_t N,
                                int64_t K, cudaStream_t stream, int num_sms, uint64_t timeout_ns) {
    WeightArgs a;
    a.q = static_cast<uint8_t*>(q);
    a.s = pow2 ? nullptr : static_cast<float*>(s);
    a.s8 = pow2 ? static_cast<uint8_t*>(s) : nullptr;
    a.N = N;
    a.K = K;
    a.NB = static_cast<uint32_t>((N + 127) / 128);
    a.KB = static_cast<uint32_t>((K + 127) / 128);
    a.timeout_ns = timeout_ns;
    const uint64_t nblocks = static_cast<uint64_t>(a.NB) * a.KB;
    const unsigned grid = static_cast<unsigned>(nblocks < static_cast<uint64_t>(num_sms) ? nblocks : num_sms);
    auto kern = pow2 ? quant_weight_kernel<true> : quant_weight_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmem);
    if (err != cudaSuccess) return err;
    kern<<<grid, kWThreads, kWSmem, stream>>>(*tmW, a);
    return cudaGetLastError();
}

template <bool WQ, bool WT, bool POW2>
cudaError_t launch_weight_plain(const WeightPlainArgs& a, cudaStream_t stream, int num_sms) {
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, quant_weight_plain_kernel<WQ, WT, POW2>, kTThreads, 0);
    if (err != cudaSuccess) return err;
    const uint64_t nblocks = static_cast<uint64_t>(a.NB) * a.KB;
    const uint64_t cap = static_cast<uint64_t>(num_sms) * (per_sm > 0 ? per_sm : 1);
    quant_weight_plain_kernel<WQ, WT, POW2>
        <<<static_cast<unsigned>(nblocks < cap ? nblocks : cap), kTThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight_t(const void* w, void* q, void* s, void* qt, void* st, bool pow2, int64_t N,
                                  int64_t K, cudaStream_t stream, int num_sms) {
    WeightPlainArgs p;
    p.w = static_cast<const uint8_t*>(w);
    p.q = static_cast<uint8_t*>(q);
    p.s = pow2 ? nullptr : static_cast<float*>(s);
    p.s8 = pow2 ? static_cast<uint8_t*>(s) : nullptr;
    p.qt = static_cast<uint8_t*>(qt);
    p.st = pow2 ? nullptr : static_cast<float*>(st);
    p.st8 = pow2 ? static_cast<uint8_t*>(st) : nullptr;
    p.N = N;
    p.K = K;
    p.NB = static_cast<uint32_t>((N + 127) / 128);
    p.KB = static_cast<uint32_t>((K + 127) / 128);
    if (pow2) {
        if (q == nullptr) return launch_weight_plain<false, true, true>(p, stream, num_sms);
        return launch_weight_plain<true, true, true>(p, stream, num_sms);
    }
    if (q == nullptr) return launch_weight_plain<false, true, false>(p, stream, num_sms);
    return launch_weight_plain<true, true, false>(p, stream, num_sms);
}

template <bool POW2>
cudaError_t launch_act_t(const ActTArgs& a, cudaStream_t stream, int num_sms) {
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_act_t_kernel<POW2>,
                                                                    kTThreads, 0);
    if (err != cudaSuccess) return err;
    const uint64_t nblocks = static_cast<uint64_t>(a.MB) * a.KB;
    const uint64_t cap = static_cast<uint64_t>(num_sms) * (per_sm > 0 ? per_sm : 1);
    quant_act_t_kernel<POW2>
        <<<static_cast<unsigned>(nblocks < cap ? nblocks : cap), kTThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_t(const void* x, void* qt, void* st, bool pow2, int64_t M, int64_t K,
                               cudaStream_t stream, int num_sms) {
    ActTArgs a;
    a.x = static_cast<const uint8_t*>(x);
    a.qt = static_cast<uint8_t*>(qt);
    a.st = pow2 ? nullptr : static_cast<float*>(st);
    a.st8 = pow2 ? static_cast<uint8_t*>(st) : nullptr;
    a.M = M;
    a.K = K;
    a.MB = static_cast<uint32_t>((M + 127) / 128);
    a.KB = static_cast<uint32_t>((K + 127) / 128);
    return pow2 ? launch_act_t<true>(a, stream, num_sms) : launch_act_t<false>(a, stream, num_sms);
}

cudaError_t read_quant_status(uint32_t* out, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(out, g_quant_status, sizeof(uint32_t));
    if (err != cudaSuccess || !clear) return err;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_quant_status, &zero, sizeof(uint32_t));
}

}  // namespace fp8q