// FP8 GEMM with power-of-two (UE8M0) block scales applied by the tensor
// core, C = A * B^T. The quantization granularity is the pages' (1x128 tiles
// of A, 128x128 blocks of B: news.qq.com/rain/a/20241229A05OQF00, "FP8
// 低精度训练", Fig. 7a); the power-of-two scales are a variant the pages do
// not describe. Because every scale is an exact power of two, the tensor
// core applies it per 32-wide K slice (tcgen05.mma kind::mxf8f6f4
// .block_scale) and accumulates the whole K range in its FP32 accumulator in
// tensor memory: there is no per-K-block promotion through registers.
//
// Per CTA (persistent, one 128 x 224 output tile at a time, 12 warps; in
// pair mode two CTAs of a cluster compute a 256 x 224 tile with the 2-CTA
// MMA, each CTA holding its 128 rows of A and 112 of B's 224 rows, which
// cuts each SM's shared-memory traffic per K block from 88 to 60 KB):
//   warp 0      TMA producer: per K block a 128x128 A box and a 224x128 B box
//               (E4M3, 128-byte swizzle) into a ring of shared-memory stages.
//   warp 1      MMA issuer (one elected lane): per K block 4 block-scaled MMAs
//               (K = 32 each) accumulating into the tile's TMEM accumulator;
//               commits free the stage and the scale slot, and after the
//               tile's last K block mark the accumulator full. Allocates and
//               frees tensor memory.
//   warps 4-7   scale writers: per group of 4 K blocks one warp per 32-lane
//               quarter of tensor memory writes the tile's scale-factor bytes
//               into a 16-column slot of a 4-slot ring with tcgen05.st: A row
//               32 j + r at column j, B column 32 j + r at column 8 + j, lane
//               r of every quarter; byte i of each 32-bit cell holds K block
//               4 g + i, so one 32-bit load of the row-major byte scales
//               fills a cell and the MMA selects the byte with the
//               instruction's scale-factor ids. The next group's scales are
//               loaded while the current group is written.
//   warps 8-11  epilogue: tcgen05.ld the finished accumulator (32 lanes and
//               224 columns per warp), release it, convert to bf16 and
//               TMA-store 32x32 boxes.
// Tensor memory: two 224-column accumulators (the epilogue of one tile
// overlaps the MMAs of the next) and 4 scale slots of 16 columns: 512.
// Pair mode: the even CTA issues the MMAs; both CTAs' loads count on its
// "full" barriers, both CTAs' scale writers and epilogue warps arrive on its
// scale-slot and accumulator barriers, and its commits arrive on the
// barriers of both CTAs. Each CTA's tensor memory holds the scale factors of
// its own A rows and of all the tile's B columns.
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
static_assert(kAccCols + kSfSlots * kSfCols <= kTmemCols, "tensor memory budget");

template <bool PAIR>
struct BsLayout {
    static constexpr int A_BYTES = kBM * kBK;
    static constexpr int B_ROWS = PAIR ? kBN / 2 : kBN;
    static constexpr int B_BYTES = B_ROWS * kBK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_BOX_BYTES = 32 * 32 * 2;
    static constexpr int EPI_WARP_BYTES = 2 * EPI_BOX_BYTES;
    static constexpr int EPI_BYTES = 4 * EPI_WARP_BYTES;
    static constexpr int RESERVE = 1024 + 512;
    static constexpr int STAGES_FIT = (kSmemLimit - RESERVE - EPI_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
    // barriers: full[S], empty[S], sf_full[slots], sf_empty[slots],
    // tmem_full[2], tmem_empty[2], drain
    static constexpr int FULL = 0, EMPTY = STAGES, SFFULL = 2 * STAGES, SFEMPTY = SFFULL + kSfSlots,
                         TFULL = SFEMPTY + kSfSlots, TEMPTY = TFULL + 2, DRAIN = TEMPTY + 2,
                         NUM_BARS = DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + 8 * NUM_BARS;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
    static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "128-byte-swizzle tiles need 1 KB alignment");
    static_assert(STAGES >= 2, "not enough shared memory for two stages");
    static_assert(8 * NUM_BARS + 16 <= 512, "barrier area overflow");
};

struct BsArgs {
    const uint8_t* sa;  // UE8M0 bytes [M, KB]
    const uint8_t* sb;  // UE8M0 bytes [NB, KB]
    int32_t M, N, KB, NB;
    int32_t mt_count, nt_count;
    int32_t rows;       // row units: m-tiles, or pairs of m-tiles in pair mode
    int32_t num_units;  // rows * nt_count
    uint64_t timeout_ns;
    uint32_t debug;  // FP8Q_INJECT_STALLED_STAGE
};

// Work unit u -> this CTA's tile origin. Groups of kGroupM row units share
// n-tiles for L2 reuse; in pair mode CTA `rank` takes m-tile 2 r + rank of
// row unit r.
template <bool PAIR>
__device__ __forceinline__ void tile_of(const BsArgs& a, int u, uint32_t rank, int& m0, int& n0) {
    const int per_group = kGroupM * a.nt_count;
    const int g = u / per_group, in = u - g * per_group;
    const int first = g * kGroupM;
    const int gm = min(kGroupM, a.rows - first);
    const int ru = first + in % gm;
    m0 = (PAIR ? 2 * ru + static_cast<int>(rank) : ru) * kBM;
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

// ROWB: one scale per row of B (sb [N][KB], the weight-gradient layout)
// instead of one per 128-row block.
template <bool PAIR, bool ROWB>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const BsArgs args) {
    using L = BsLayout<PAIR>;
    constexpr int S = L::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    auto bar = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t limit = args.timeout_ns;
    const int KB = args.KB;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    // a barrier of the even CTA (the MMA side) as seen from this CTA
    auto lead_bar = [&](int i) -> uint32_t { return PAIR ? mapa_shared(bar(i), 0) : bar(i); };
    const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int unit_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(L::FULL + s), PAIR ? 2 : 1);  // pair: both CTAs' producers
            mbar_init(bar(L::EMPTY + s), 1);
        }
        for (int j = 0; j < kSfSlots; ++j) {
            mbar_init(bar(L::SFFULL + j), PAIR ? 8 : 4);  // one arrive per scale-writer warp
            mbar_init(bar(L::SFEMPTY + j), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::TFULL + b), 1);
            mbar_init(bar(L::TEMPTY + b), PAIR ? 8 : 4);  // one arrive per epilogue warp
        }
        mbar_init(bar(L::DRAIN), 1);
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
        tmem_alloc<PAIR>(sbase + L::MISC_OFF, kTmemCols);
        tmem_relinquish_alloc_permit<PAIR>();
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // peer barriers initialised before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0, issued = 0;
        bool ok = true;
        for (int u = unit0; ok && u < args.num_units; u += unit_step) {
            int m0, n0;
            tile_of<PAIR>(args, u, rank, m0, n0);
            const int brow = n0 + (PAIR ? static_cast<int>(rank) * L::B_ROWS : 0);
            for (int kb = 0; kb < KB; ++kb) {
                if (!warp_wait(bar(L::EMPTY + stage), phase ^ 1u, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    uint32_t bytes = L::STAGE_BYTES;
                    if ((args.debug & FP8Q_INJECT_STALLED_STAGE) && issued == 0) bytes += 16;
                    const uint32_t sA = sbase + stage * L::STAGE_BYTES;
                    if constexpr (PAIR) {
                        const uint32_t fb = lead_bar(L::FULL + stage);
                        mbar_arrive_expect_tx_cluster(fb, bytes);
                        tma_load_2d_pair(sA, &tmA, fb, kb * kBK, m0);
                        tma_load_2d_pair(sA + L::A_BYTES, &tmB, fb, kb * kBK, brow);
                    } else {
                        mbar_arrive_expect_tx(bar(L::FULL + stage), bytes);
                        tma_load_2d(sA, &tmA, bar(L::FULL + stage), kb * kBK, m0);
                        tma_load_2d(sA + L::A_BYTES, &tmB, bar(L::FULL + stage), kb * kBK, brow);
                    }
                }
                __syncwarp();
                ++issued;
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // copies in flight land before the CTA may exit (in pair mode the even
        // CTA's full barriers count both CTAs' bytes; the odd CTA leaves only
        // after the closing cluster barrier)
        for (int s = 0; s < S && leader; ++s) {
            if (static_cast<uint32_t>(s) >= issued) break;
            const uint32_t last = s + S * ((issued - 1 - s) / S);
            volatile int local_flag = 0;
            mbar_wait(bar(L::FULL + s), (last / S) & 1u, &local_flag, limit);
        }
    } else if (warp == 1 && leader) {
        // -------------------------------------------------------- MMA issuer
        int stage = 0, slot = 0;
        uint32_t phase = 0, sphase = 0, abuf = 0, aphase = 0;
        bool ok = true, issued_any = false;
        for (int u = unit0; ok && u < args.num_units; u += unit_step) {
            if (!warp_wait(bar(L::TEMPTY + abuf), aphase ^ 1u, abort_flag, limit)) break;
            tc_fence_after_sync();
            const uint32_t d = tmem_base + abuf * kBN;
            for (int kb = 0; kb < KB; ++kb) {
                const uint32_t i = static_cast<uint32_t>(kb & 3);  // byte of the scale cells
                if (!warp_wait(bar(L::FULL + stage), phase, abort_flag, limit) ||
                    (i == 0 && !warp_wait(bar(L::SFFULL + slot), sphase, abort_flag, limit))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sA = sbase + stage * L::STAGE_BYTES;
                const uint64_t ad = sdesc_k_sw128(sA);
                const uint64_t bd = sdesc_k_sw128(sA + L::A_BYTES);
                const uint32_t sfa = tmem_base + kAccCols + slot * kSfCols;
                const uint32_t idesc = idesc_e4m3_bs(PAIR ? 2 * kBM : kBM, kBN, i, i);
                const bool group_end = i == 3 || kb == KB - 1;
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k) {
                        const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
                        if constexpr (PAIR)
                            mma_e4m3_bs_pair(d, ad + 2u * k, bd + 2u * k, idesc, sfa, sfa + kSfbOff, acc);
                        else
                            mma_e4m3_bs(d, ad + 2u * k, bd + 2u * k, idesc, sfa, sfa + kSfbOff, acc);
                    }
                    if constexpr (PAIR) {
                        mma_commit_pair(bar(L::EMPTY + stage));
                        if (group_end) mma_commit_pair(bar(L::SFEMPTY + slot));
                        if (kb == KB - 1) mma_commit_pair(bar(L::TFULL + abuf));
                    } else {
                        mma_commit(bar(L::EMPTY + stage));
                        if (group_end) mma_commit(bar(L::SFEMPTY + slot));
                        if (kb == KB - 1) mma_commit(bar(L::TFULL + abuf));
                    }
                }
                __syncwarp();
                issued_any = true;
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (group_end && ++slot == kSfSlots) {
                    slot = 0;
                    sphase ^= 1u;
                }
            }
            abuf ^= 1u;
            if (abuf == 0) aphase ^= 1u;
        }
        if (issued_any) {  // every MMA issued above has completed once this arrives
            if (elect_one()) {
                if constexpr (PAIR) mma_commit_pair_local(bar(L::DRAIN));
                else mma_commit(bar(L::DRAIN));
            }
            __syncwarp();
            volatile int local_flag = 0;
            mbar_wait(bar(L::DRAIN), 0, &local_flag, limit);
        }
    } else if (warp >= 4 && warp < 8) {
        // ----------------------------------------------------- scale writers
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const uint32_t lane_addr = tmem_base + ((quarter * 32u) << 16);
        const int groups = (KB + 3) >> 2;
        // 32-bit loads of 4 consecutive K-block bytes when every row's group
        // starts on a 4-byte boundary; byte loads otherwise
        const bool wide = (KB & 3) == 0 && ((reinterpret_cast<uintptr_t>(args.sa) |
                                             reinterpret_cast<uintptr_t>(args.sb)) & 3u) == 0;
        auto cell = [&](const uint8_t* row, int kb0) -> uint32_t {
            if (wide) return __ldg(reinterpret_cast<const uint32_t*>(row + kb0));
            uint32_t w = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w |= static_cast<uint32_t>(kb0 + i < KB ? __ldg(row + kb0 + i) : 127u) << (8 * i);
            return w;
        };
        // the cells of group g of unit u: this CTA's A rows 32 j + lane, and
        // the tile's B columns 32 j + lane
        auto load_group = [&](int u, int g, uint32_t (&v)[16]) {
            int m0, n0;
            tile_of<PAIR>(args, u, rank, m0, n0);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int m = m0 + 32 * j + lane;
                v[j] = m < args.M ? cell(args.sa + static_cast<int64_t>(m) * KB, 4 * g) : 0x7F7F7F7Fu;
            }
#pragma unroll
            for (int j = 4; j < kSfbOff; ++j) v[j] = 0x7F7F7F7Fu;
#pragma unroll
            for (int j = 0; j < kBN / 32; ++j) {
                const int n = n0 + 32 * j + lane;
                const int64_t brow = ROWB ? n : (n >> 7);
                v[kSfbOff + j] = n < args.N ? cell(args.sb + brow * KB, 4 * g) : 0x7F7F7F7Fu;
            }
#pragma unroll
            for (int j = kSfbOff + kBN / 32; j < 16; ++j) v[j] = 0x7F7F7F7Fu;
        };
        const uint32_t sffull_base = lead_bar(L::SFFULL);
        int slot = 0;
        uint32_t sphase = 0;
        int u = unit0, g = 0;
        uint32_t cur[16];
        if (u < args.num_units) load_group(u, 0, cur);
        while (u < args.num_units) {
            // the next group's coordinates, its loads issued before this group is written
            int un = u, gn = g + 1;
            if (gn == groups) {
                gn = 0;
                un += unit_step;
            }
            uint32_t nxt[16];
            if (un < args.num_units) load_group(un, gn, nxt);
            if (!warp_wait(bar(L::SFEMPTY + slot), sphase ^ 1u, abort_flag, limit)) break;
            tmem_st16(lane_addr + kAccCols + slot * kSfCols, cur);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cluster(sffull_base + 8u * slot);
                else mbar_arrive(bar(L::SFFULL + slot));
            }
            if (++slot == kSfSlots) {
                slot = 0;
                sphase ^= 1u;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) cur[j] = nxt[j];
            u = un;
            g = gn;
        }
    } else if (warp >= 8) {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - 8;
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const uint32_t lane_addr = tmem_base + ((quarter * 32u) << 16);
        uint8_t* ebuf0 = smem + L::EPI_OFF + ew * L::EPI_WARP_BYTES;
        const uint32_t ebuf0_s = sbase + L::EPI_OFF + ew * L::EPI_WARP_BYTES;
        const uint32_t tempty_base = lead_bar(L::TEMPTY);
        uint32_t abuf = 0, aphase = 0;
        uint32_t ebox = 0;  // boxes staged so far: their buffer alternates, across tiles too
        for (int u = unit0; u < args.num_units; u += unit_step) {
            int m0, n0;
            tile_of<PAIR>(args, u, rank, m0, n0);
            if (!warp_wait(bar(L::TFULL + abuf), aphase, abort_flag, limit)) break;
            tc_fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(lane_addr + abuf * kBN + 32 * c, r);
                tmem_wait_ld32(r);
                if (c == kBN / 32 - 1) {  // the accumulator is in registers: release it
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR) mbar_arrive_cluster(tempty_base + 8u * abuf);
                        else mbar_arrive(bar(L::TEMPTY + abuf));
                    }
                }
                const uint32_t eb = ebox++ & 1u;
                uint8_t* ebuf = ebuf0 + eb * L::EPI_BOX_BYTES;
                const uint32_t ebuf_s = ebuf0_s + eb * L::EPI_BOX_BYTES;
                // the store issued two boxes ago (same buffer) must have read it:
                // every box commits one bulk group, so at most the previous box's
                // may still be reading
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
                if (lane == 0) {
                    if (x < args.N && y < args.M) tma_store_2d(&tmC, ebuf_s, x, y);
                    bulk_commit_group();  // empty when the box lies past C
                }
            }
            abuf ^= 1u;
            if (abuf == 0) aphase ^= 1u;
        }
        if (lane == 0) bulk_wait_group0();
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the even CTA's MMAs (drained) may write our TMEM
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<PAIR>(tmem_base, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_bs_status, FP8Q_DEVSTATUS_TIMEOUT);
}

template <bool PAIR, bool ROWB>
cudaError_t launch_bs(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC,
                      const BsArgs& a, unsigned grid, cudaStream_t stream) {
    using L = BsLayout<PAIR>;
    auto kern = fp8_gemm_bs_kernel<PAIR, ROWB>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    if constexpr (!PAIR) {
        kern<<<grid, kThreads, L::SMEM_BYTES, stream>>>(*tmA, *tmB, *tmC, a);
        return cudaGetLastError();
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = L::SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, *tmA, *tmB, *tmC, a);
    }
}

template <bool ROWB>
int bs_pair_max_clusters() {
    using L = BsLayout<true>;
    if (cudaFuncSetAttribute(fp8_gemm_bs_kernel<true, ROWB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::SMEM_BYTES) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_bs_kernel<true, ROWB>, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace

int gemm_bs_tile_n() { return kBN; }

int gemm_bs_pair_max_clusters(bool row_scaled_b) {
    return row_scaled_b ? bs_pair_max_clusters<true>() : bs_pair_max_clusters<false>();
}

cudaError_t launch_gemm_bs(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC,
                           const uint8_t* sa, const uint8_t* sb, int32_t M, int32_t N, int32_t K,
                           bool row_scaled_b, bool pair, int pair_clusters, uint64_t timeout_ns,
                           uint32_t debug, int num_sms, cudaStream_t stream) {
    BsArgs a;
    a.sa = sa;
    a.sb = sb;
    a.M = M;
    a.N = N;
    a.KB = (K + kBK - 1) / kBK;
    a.NB = (N + 127) / 128;
    a.mt_count = (M + kBM - 1) / kBM;
    a.nt_count = (N + kBN - 1) / kBN;
    a.rows = pair ? (a.mt_count + 1) / 2 : a.mt_count;
    const int64_t units = static_cast<int64_t>(a.rows) * a.nt_count;
    if (units > 2147483647) return cudaErrorInvalidValue;
    a.num_units = static_cast<int32_t>(units);
    a.timeout_ns = timeout_ns;
    a.debug = debug;
    if (pair) {
        const int64_t clusters = units < pair_clusters ? units : pair_clusters;
        const unsigned grid = static_cast<unsigned>(2 * clusters);
        return row_scaled_b ? launch_bs<true, true>(tmA, tmB, tmC, a, grid, stream)
                            : launch_bs<true, false>(tmA, tmB, tmC, a, grid, stream);
    }
    const unsigned grid = static_cast<unsigned>(units < num_sms ? units : num_sms);
    return row_scaled_b ? launch_bs<false, true>(tmA, tmB, tmC, a, grid, stream)
                        : launch_bs<false, false>(tmA, tmB, tmC, a, grid, stream);
}

cudaError_t read_bs_status(uint32_t* out, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(out, g_bs_status, sizeof(uint32_t));
    if (err != cudaSuccess || !clear) return err;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_bs_status, &zero, sizeof(uint32_t));
}

}  // namespace fp8q
