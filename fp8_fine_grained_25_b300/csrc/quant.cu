// Fine-grained FP8 quantizers: activations per 1x128 tile, weights per
// 128x128 block (news.qq.com/rain/a/20241229A05OQF00, "FP8 低精度训练",
// item "细粒度量化", Fig. 7a; developer.aliyun.com/article/1776647 §4.1).
//
// Both are HBM-bound streams: 2 bytes read and 1 byte written per element
// plus one fp32 scale per tile/block. Loads and stores are 16-byte / 8-byte
// vectors, each half-warp owns one 128-element tile row, and the tile amax
// is a 4-step xor-shuffle max inside the half-warp.
//
// Arithmetic per tile (bit-exact with the definition):
//   amax  = max |x|                 (bf16 -> fp32 is exact, max is exact)
//   s     = fl32(amax / 448)        (IEEE round-to-nearest divide)
//   q_i   = E4M3_rn_satfinite(fl32(x_i / s)),  all-zero tile: s = 0, q = 0
// The per-element quotient uses the tile's reciprocal and one FMA
// correction instead of a full divide (see div_by_scale).
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "quant.cuh"

namespace fp8q {

namespace {

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ float absmax8(const float (&f)[8]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    return m;
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

// Eight values divided by the tile scale and encoded, low byte first.
// `amax` is the tile's absolute maximum (s = amax / 448).
__device__ __forceinline__ uint2 encode8(const float (&f)[8], float s, float amax) {
    if (s == 0.0f) return make_uint2(0u, 0u);
    float y[8];
    if (amax >= kFastDivMinAmax) {
        const float r = __frcp_rn(s);
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

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

constexpr int kActThreads = 256;
constexpr int kActUnroll = 4;  // tile pairs per warp per iteration

// One half-warp per 1x128 tile; lane `sub` of the half owns columns
// [8*sub, 8*sub+8) of the tile. A tile t = (m, kb) covers row m, columns
// [128*kb, min(K, 128*kb + 128)); its scale goes to s[m * KB + kb].
__global__ void __launch_bounds__(kActThreads) quant_act_kernel(const uint8_t* __restrict__ x,
                                                                uint8_t* __restrict__ q,
                                                                float* __restrict__ s,
                                                                uint32_t T, uint32_t KB,
                                                                int64_t K) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t half = lane >> 4, sub = lane & 15u;
    const uint64_t warp = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;
    for (uint64_t base = warp * (2 * kActUnroll); base < T; base += nwarps * (2 * kActUnroll)) {
        uint4 v[kActUnroll];
        int64_t off[kActUnroll];
        bool live[kActUnroll];
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            const uint64_t t = base + 2 * u + half;
            const uint32_t m = static_cast<uint32_t>(t / KB);
            const uint32_t kb = static_cast<uint32_t>(t - static_cast<uint64_t>(m) * KB);
            const int64_t col = static_cast<int64_t>(kb) * 128 + 8 * sub;
            off[u] = static_cast<int64_t>(m) * K + col;
            live[u] = (t < T) && (col < K);
            v[u] = live[u] ? ld_stream16(x + 2 * off[u]) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kActUnroll; ++u) {
            float f[8];
            unpack_bf16x8(v[u], f);
            float amax = absmax8(f);
#pragma unroll
            for (int d = 8; d >= 1; d >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
            const float sc = __fdiv_rn(amax, 448.0f);
            const uint64_t t = base + 2 * u + half;
            if (live[u]) {
                *reinterpret_cast<uint2*>(q + off[u]) = encode8(f, sc, amax);
                if (sub == 0) s[t] = sc;
            }
        }
    }
}

constexpr int kWThreads = 256;
constexpr int kWChunks = 8;  // 16-byte chunks per thread: 128 rows x 16 chunks / 256

// One CTA per 128x128 block (grid-stride). Chunk c = tid + 256 * i covers
// block row c / 16 and columns [8 * (c % 16), +8).
__global__ void __launch_bounds__(kWThreads) quant_weight_kernel(const uint8_t* __restrict__ w,
                                                                 uint8_t* __restrict__ q,
                                                                 float* __restrict__ s,
                                                                 int64_t N, int64_t K,
                                                                 uint32_t NB, uint32_t KB) {
    __shared__ float red[kWThreads / 32];
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint64_t nblocks = static_cast<uint64_t>(NB) * KB;
    for (uint64_t b = blockIdx.x; b < nblocks; b += gridDim.x) {
        const uint32_t nb = static_cast<uint32_t>(b / KB);
        const uint32_t kb = static_cast<uint32_t>(b - static_cast<uint64_t>(nb) * KB);
        uint4 v[kWChunks];
        int64_t off[kWChunks];
        bool live[kWChunks];
#pragma unroll
        for (int i = 0; i < kWChunks; ++i) {
            const uint32_t c = tid + kWThreads * i;
            const int64_t n = static_cast<int64_t>(nb) * 128 + (c >> 4);
            const int64_t k = static_cast<int64_t>(kb) * 128 + 8 * (c & 15u);
            live[i] = (n < N) && (k < K);
            off[i] = n * K + k;
            v[i] = live[i] ? ld_stream16(w + 2 * off[i]) : make_uint4(0, 0, 0, 0);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kWChunks; ++i) {
            float f[8];
            unpack_bf16x8(v[i], f);
            amax = fmaxf(amax, absmax8(f));
        }
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int i = 1; i < kWThreads / 32; ++i) amax = fmaxf(amax, red[i]);
        const float sc = __fdiv_rn(amax, 448.0f);
#pragma unroll
        for (int i = 0; i < kWChunks; ++i) {
            if (!live[i]) continue;
            float f[8];
            unpack_bf16x8(v[i], f);
            *reinterpret_cast<uint2*>(q + off[i]) = encode8(f, sc, amax);
        }
        if (tid == 0) s[b] = sc;
        __syncthreads();  // red[] is reused by the next block
    }
}

}  // namespace

cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, void* q, float* s,
                             cudaStream_t stream, int num_sms) {
    const int64_t KB = (K + 127) / 128;
    const uint64_t T = static_cast<uint64_t>(M) * KB;
    const uint64_t per_block = (kActThreads / 32) * 2 * kActUnroll;  // tiles per block-iteration
    uint64_t want = (T + per_block - 1) / per_block;
    const uint64_t cap = static_cast<uint64_t>(num_sms) * (2048 / kActThreads);
    const unsigned grid = static_cast<unsigned>(want < cap ? (want ? want : 1) : cap);
    quant_act_kernel<<<grid, kActThreads, 0, stream>>>(
        static_cast<const uint8_t*>(x), static_cast<uint8_t*>(q), s, static_cast<uint32_t>(T),
        static_cast<uint32_t>(KB), K);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight(const void* w, int64_t N, int64_t K, void* q, float* s,
                                cudaStream_t stream, int num_sms) {
    const int64_t KB = (K + 127) / 128, NB = (N + 127) / 128;
    const uint64_t nblocks = static_cast<uint64_t>(NB) * KB;
    const uint64_t cap = static_cast<uint64_t>(num_sms) * (2048 / kWThreads);
    const unsigned grid = static_cast<unsigned>(nblocks < cap ? nblocks : cap);
    quant_weight_kernel<<<grid, kWThreads, 0, stream>>>(
        static_cast<const uint8_t*>(w), static_cast<uint8_t*>(q), s, N, K,
        static_cast<uint32_t>(NB), static_cast<uint32_t>(KB));
    return cudaGetLastError();
}

}  // namespace fp8q
