// FP8 GEMM with power-of-two (UE8M0) block scales applied by the tensor
// core, C = A * B^T. The quantization granularity is the pages' (1x128 tiles
// of A, 128x128 blocks of B: news.qq.com/rain/a/20241229A05OQF00, "FP8
// 低精度训练", Fig. 7a); the power-of-two scales are a variant the pages do
// not describe. Because every scale is an exact power of two, the tensor
// core applies it per 32-wide K slice (tcgen05.mma kind::mxf8f6f4
// .block_scale) and accumulates the whole K range in its FP32 accumulator in
// tensor memory: there is no per-K-block promotion through registers.
//
// Per CTA (persistent, one 128 x 224 output tile at a time, 12 warps):
//   warp 0      TMA producer: per K block a 128x128 A box and a 224x128 B box
//               (E4M3, 128-byte swizzle) into a ring of shared-memory stages.
//   warp 1      MMA issuer (one elected lane): per K block 4 block-scaled MMAs
//               (K = 32 each) accumulating into the tile's TMEM accumulator;
//               commits free the stage and the scale slot, and after the
//               tile's last K block mark the accumulator full. Allocates and
//               frees tensor memory.
//   warps 4-7   scale writers: per K block one warp per 32-lane quarter of
//               tensor memory writes the tile's scale-factor bytes (A rows
//               32 j + r at column j, B columns 32 j + r at column 8 + j of
//               a 16-column slot, every quarter holding the same bytes) with
//               tcgen05.st into a ring of 4 slots.
//   warps 8-11  epilogue: tcgen05.ld the finished accumulator (32 lanes and
//               224 columns per warp), release it, convert to bf16 and
//               TMA-store 32x32 boxes.
// Tensor memory: two 224-column accumulators (the epilogue of one tile
// overlaps the MMAs of the next) and 4 scale slots of 16 columns: 512.
// Every wait is bounded; on expiry the CTA raises an abort flag, drains its
// copies and MMAs, frees tensor memory and returns, and the status word gets
// FP8Q_DEVSTATUS_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8q.h"
#include "gemm.cuh"
#include "ptx.cuh"

namespace fp8q {

__device__ uint32_t g_bs_status;

namespace {

constexpr int kBM = 128, kBK = 128, kBN = 224;
constexpr int kThreads = 384;
constexpr int kSfSlots = 4, kSfCols = 16, kSfbOff = 8;
constexpr int kAccCols = 2 * kBN;
constexpr int kTmemCols = 512;
constexpr int kGroupM = 16;
constexpr int kSmemLimit = 232448;
constexpr int A_BYTES = kBM * kBK;
constexpr int B_BYTES = kBN * kBK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 44 KB, a multiple of 1024
constexpr int EPI_BOX_BYTES = 32 * 32 * 2;
constexpr int EPI_WARP_BYTES = 2 * EPI_BOX_BYTES;
constexpr int EPI_BYTES = 4 * EPI_WARP_BYTES;
constexpr int RESERVE = 1024 + 512;
constexpr int STAGES = (kSmemLimit - RESERVE - EPI_BYTES) / STAGE_BYTES;
constexpr int EPI_OFF = STAGES * STAGE_BYTES;
constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
// barriers: full[S], empty[S], sf_full[slots], sf_empty[slots], tmem_full[2],
// tmem_empty[2], drain
constexpr int FULL = 0, EMPTY = STAGES, SFFULL = 2 * STAGES, SFEMPTY = SFFULL + kSfSlots,
              TFULL = SFEMPTY + kSfSlots, TEMPTY = TFULL + 2, DRAIN = TEMPTY + 2, NUM_BARS = DRAIN + 1;
constexpr int MISC_OFF = BAR_OFF + 8 * NUM_BARS;
constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
static_assert(kAccCols + kSfSlots * kSfCols <= kTmemCols, "tensor memory budget");
static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "128-byte-swizzle tiles need 1 KB alignment");
static_assert(STAGES >= 2, "not enough shared memory for two stages");
static_assert(8 * NUM_BARS + 16 <= 512, "barrier area overflow");

struct BsArgs {
    const uint8_t* sa;  // UE8M0 bytes [M, KB]
    const uint8_t* sb;  // UE8M0 bytes [NB, KB]
    int32_t M, N, KB, NB;
    int32_t mt_count, nt_count, num_tiles;
    uint64_t timeout_ns;
    uint32_t debug;  // FP8Q_INJECT_STALLED_STAGE
};

__device__ __forceinline__ void tile_of(const BsArgs& a, int t, int& m0, int& n0) {
    const int per_group = kGroupM * a.nt_count;
    const int g = t / per_group, in = t - g * per_group;
    const int first = g * kGroupM;
    const int gm = min(kGroupM, a.mt_count - first);
    m0 = (first + in % gm) * kBM;
    n0 = (in / gm) * kBN;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, limit));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t rep4(uint32_t byte) { return byte * 0x01010101u; }

__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const BsArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    auto bar = [&](int i) -> uint32_t { return sbase + BAR_OFF + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + MISC_OFF + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t limit = args.timeout_ns;
    const int KB = args.KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1);
        }
        for (int j = 0; j < kSfSlots; ++j) {
            mbar_init(bar(SFFULL + j), 4);  // one arrive per scale-writer warp
            mbar_init(bar(SFEMPTY + j), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(TFULL + b), 1);
            mbar_init(bar(TEMPTY + b), 4);  // one arrive per epilogue warp
        }
        mbar_init(bar(DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(sbase + MISC_OFF, kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0, issued = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < args.num_tiles; t += gridDim.x) {
            int m0, n0;
            tile_of(args, t, m0, n0);
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait(bar(EMPTY + stage), phase ^ 1u, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    uint32_t bytes = STAGE_BYTES;
                    if ((args.debug & FP8Q_INJECT_STALLED_STAGE) && issued == 0) bytes += 16;
                    const uint32_t sA = sbase + stage * STAGE_BYTES;
                    mbar_arrive_expect_tx(bar(FULL + stage), bytes);
                    tma_load_2d(sA, &tmA, bar(FULL + stage), kb * kBK, m0);
                    tma_load_2d(sA + A_BYTES, &tmB, bar(FULL + stage), kb * kBK, n0);
                }
                __syncwarp();
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        for (int s = 0; s < STAGES; ++s) {  // copies in flight land before the CTA may exit
            if (static_cast<uint32_t>(s) >= issued) break;
            const uint32_t last = s + STAGES * ((issued - 1 - s) / STAGES);
            volatile int local_flag = 0;
            mbar_wait(bar(FULL + s), (last / STAGES) & 1u, &local_flag, limit);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_e4m3_bs(kBM, kBN, 0, 0);
        int stage = 0, slot = 0;
        uint32_t phase = 0, sphase = 0, abuf = 0, aphase = 0;
        bool ok = true, issued_any = false;
        for (int t = blockIdx.x; ok && t < args.num_tiles; t += gridDim.x) {
            if (!warp_wait(bar(TEMPTY + abuf), aphase ^ 1u, abort_flag, limit)) break;
            tc_fence_after_sync();
            const uint32_t d = tmem_base + abuf * kBN;
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait(bar(FULL + stage), phase, abort_flag, limit) ||
                    !warp_wait(bar(SFFULL + slot), sphase, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sA = sbase + stage * STAGE_BYTES;
                const uint64_t ad = sdesc_k_sw128(sA);
                const uint64_t bd = sdesc_k_sw128(sA + A_BYTES);
                const uint32_t sfa = tmem_base + kAccCols + slot * kSfCols;
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k)
                        mma_e4m3_bs(d, ad + 2u * k, bd + 2u * k, idesc, sfa, sfa + kSfbOff,
                                    (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit(bar(EMPTY + stage));
                    mma_commit(bar(SFEMPTY + slot));
                    if (kb == KB - 1) mma_commit(bar(TFULL + abuf));
                }
                __syncwarp();
                issued_any = true;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++slot == kSfSlots) {
                    slot = 0;
                    sphase ^= 1u;
                }
            }
            abuf ^= 1u;
            if (abuf == 0) aphase ^= 1u;
        }
        if (issued_any) {  // every MMA issued above has completed once this arrives
            if (elect_one()) mma_commit(bar(DRAIN));
            __syncwarp();
            volatile int local_flag = 0;
            mbar_wait(bar(DRAIN), 0, &local_flag, limit);
        }
    } else if (warp >= 4 && warp < 8) {
        // ----------------------------------------------------- scale writers
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const uint32_t lane_addr = tmem_base + ((quarter * 32u) << 16);
        int slot = 0;
        uint32_t sphase = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < args.num_tiles; t += gridDim.x) {
            int m0, n0;
            tile_of(args, t, m0, n0);
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait(bar(SFEMPTY + slot), sphase ^ 1u, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                uint32_t v[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {  // A rows 32 j + lane
                    const int m = m0 + 32 * j + lane;
                    v[j] = rep4(m < args.M ? __ldg(args.sa + static_cast<int64_t>(m) * KB + kb) : 127u);
                }
#pragma unroll
                for (int j = 4; j < kSfbOff; ++j) v[j] = rep4(127u);
#pragma unroll
                for (int j = 0; j < kBN / 32; ++j) {  // B columns 32 j + lane
                    const int n = n0 + 32 * j + lane;
                    v[kSfbOff + j] =
                        rep4(n < args.N ? __ldg(args.sb + static_cast<int64_t>(n >> 7) * KB + kb) : 127u);
                }
#pragma unroll
                for (int j = kSfbOff + kBN / 32; j < 16; ++j) v[j] = rep4(127u);
                tmem_st16(lane_addr + kAccCols + slot * kSfCols, v);
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SFFULL + slot));
                if (++slot == kSfSlots) {
                    slot = 0;
                    sphase ^= 1u;
                }
            }
        }
    } else if (warp >= 8) {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - 8;
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const uint32_t lane_addr = tmem_base + ((quarter * 32u) << 16);
        uint8_t* ebuf0 = smem + EPI_OFF + ew * EPI_WARP_BYTES;
        const uint32_t ebuf0_s = sbase + EPI_OFF + ew * EPI_WARP_BYTES;
        uint32_t abuf = 0, aphase = 0;
        for (int t = blockIdx.x; t < args.num_tiles; t += gridDim.x) {
            int m0, n0;
            tile_of(args, t, m0, n0);
            if (!warp_wait(bar(TFULL + abuf), aphase, abort_flag, limit)) break;
            tc_fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(lane_addr + abuf * kBN + 32 * c, r);
                tmem_wait_ld32(r);
                if (c == kBN / 32 - 1) {  // the accumulator is in registers: release it
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(TEMPTY + abuf));
                }
                uint8_t* ebuf = ebuf0 + (c & 1) * EPI_BOX_BYTES;
                const uint32_t ebuf_s = ebuf0_s + (c & 1) * EPI_BOX_BYTES;
                // the store issued two boxes ago (same buffer) must have read it
                if (lane == 0) bulk_wait_group_read1();
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 pk;
                    pk.x = pack_bf16x2(__uint_as_float(r[8 * j]), __uint_as_float(r[8 * j + 1]));
                    pk.y = pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3]));
                    pk.z = pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5]));
                    pk.w = pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7]));
                    const int phys = j ^ ((lane >> 1) & 3);  // 64-byte swizzle
                    *reinterpret_cast<uint4*>(ebuf + lane * 64 + phys * 16) = pk;
                }
                fence_proxy_async_smem();
                __syncwarp();
                const int x = n0 + 32 * c, y = m0 + 32 * static_cast<int>(quarter);
                if (lane == 0 && x < args.N && y < args.M) {
                    tma_store_2d(&tmC, ebuf_s, x, y);
                    bulk_commit_group();
                }
            }
            abuf ^= 1u;
            if (abuf == 0) aphase ^= 1u;
        }
        if (lane == 0) bulk_wait_group0();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_bs_status, FP8Q_DEVSTATUS_TIMEOUT);
}

}  // namespace

int gemm_bs_tile_n() { return kBN; }

cudaError_t launch_gemm_bs(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC,
                           const uint8_t* sa, const uint8_t* sb, int32_t M, int32_t N, int32_t K,
                           uint64_t timeout_ns, uint32_t debug, int num_sms, cudaStream_t stream) {
    BsArgs a;
    a.sa = sa;
    a.sb = sb;
    a.M = M;
    a.N = N;
    a.KB = (K + kBK - 1) / kBK;
    a.NB = (N + 127) / 128;
    a.mt_count = (M + kBM - 1) / kBM;
    a.nt_count = (N + kBN - 1) / kBN;
    const int64_t tiles = static_cast<int64_t>(a.mt_count) * a.nt_count;
    if (tiles > 2147483647) return cudaErrorInvalidValue;
    a.num_tiles = static_cast<int32_t>(tiles);
    a.timeout_ns = timeout_ns;
    a.debug = debug;
    cudaError_t err =
        cudaFuncSetAttribute(fp8_gemm_bs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const unsigned grid = static_cast<unsigned>(tiles < num_sms ? tiles : num_sms);
    fp8_gemm_bs_kernel<<<grid, kThreads, SMEM_BYTES, stream>>>(*tmA, *tmB, *tmC, a);
    return cudaGetLastError();
}

cudaError_t read_bs_status(uint32_t* out, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(out, g_bs_status, sizeof(uint32_t));
    if (err != cudaSuccess || !clear) return err;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_bs_status, &zero, sizeof(uint32_t));
}

}  // namespace fp8q
