// Block-scaled FP8 GEMM on the sm_103a tensor cores, C = A * B^T, with the
// fine-grained scales applied when each 128-wide K block's partial result is
// promoted into FP32 registers (news.qq.com/rain/a/20241229A05OQF00,
// "FP8 低精度训练": "细粒度量化" Fig. 7a for the scale granularity,
// "提高累加精度" Fig. 7b for the promotion into FP32 registers).
//
// Per CTA (persistent, one 128 x BN output tile at a time, BN = 128, 160,
// 224 or 256, 12 warps):
//   warp 0      TMA producer: per K block, a 128x128 A box and a BNx128 B box
//               (E4M3, 128-byte swizzle) into a ring of shared-memory stages.
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::f8f6f4 (K = 32 each) write
//               P_kb = A_kb * B_kb^T into one of 512/BN TMEM buffers (fresh
//               accumulate per K block), then commit to the stage's "empty"
//               barrier and the buffer's "full" barrier. Allocates and frees
//               TMEM. The warp stays converged and one elected lane issues.
//   warp 2      scale loader: per group of 4 K blocks, cp.async copies of
//               sa[m0..m0+127][kb..kb+3] and the tile's sb[nb][kb..kb+3] into a
//               shared-memory scale ring, so the promotion never waits on a
//               global load and touches the ring once per 4 K blocks.
//   warp 3      pair tiles: issues the TMA stores of each output tile the
//               promotion warps have staged (below).
//   warps 4-11  promotion + epilogue: tcgen05.ld P_kb (each warp owns 32
//               TMEM lanes = 32 rows and half of the BN columns), then
//               acc += P_kb * (sa[m][kb] * sb[n/128][kb]) with packed FP32
//               FMAs into registers, release the TMEM buffer; after the last
//               K block convert to bf16 and store: TMA stores through
//               swizzled shared-memory staging for the dense GEMM (pair tiles
//               stage a warp's whole slice at once, one-CTA tiles two boxes
//               at a time), masked vector stores for the grouped one.
//               Pair tiles leave the stores of the staged tile to warp 3
//               (but for a CTA's last tile narrower than 256), so the
//               promotion warps start on the next tile at once.
// Several TMEM buffers let the MMA of later K blocks overlap the promotion
// of earlier ones. Every wait is bounded in time; on expiry the CTA raises
// an abort flag, drains its copies and MMAs, frees TMEM and returns.
//
// Tile width 224 (block-scaled dense GEMM only) fills whole waves of 7168-
// wide outputs and wastes fewer columns at N = 576. Such a tile starts on a
// multiple of 32 but not of 128: the scale ring carries up to three
// 128-column B-scale blocks, each promotion warp's 112 columns touch at most
// two (two scale products per K block), and the warp reads TMEM in 32-column
// chunks that start on multiples of 32 plus one 16-column chunk. Tile width
// 160 (pair tiles of the block-scaled dense GEMM only) works the same way
// with 80 columns per warp; three of its accumulators fit in TMEM, so the
// MMA can run two K blocks ahead of the promotion instead of one.
//
// Pair mode (dense GEMM): two CTAs of a cluster compute a 256 x BN tile with
// the 2-CTA MMA (tcgen05 cta_group::2). Each CTA holds its own 128 rows of A
// and half of the tile's B rows, so each SM's shared memory carries 32 KB
// of operands per K block instead of 48 KB (TMA writes plus MMA reads are
// the shared-memory bandwidth bound of the one-CTA tile). The even CTA
// issues the MMAs; both CTAs' loads count on its "full" barrier, both CTAs'
// promotion warps release its TMEM barrier, and its commits arrive on the
// "empty"/"full" barriers of both CTAs. Each CTA promotes and stores the
// 128 x BN accumulator in its own tensor memory.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8q.h"
#include "gemm.cuh"
#include "ptx.cuh"

namespace fp8q {
namespace {

// Status word of the kernels of this translation unit (each unit that
// instantiates the kernel has its own; the host reads and clears them all).
__device__ uint32_t g_device_status;

constexpr int BM = 128;
constexpr int BK = 128;
constexpr int kThreads = 384;
constexpr int kScaleWarp = 2;
constexpr int kFirstEpiWarp = 4;
constexpr int kEpiWarps = 8;
constexpr int kGroupM = 16;     // rasterisation: m-tiles per group for L2 reuse
constexpr int kSmemLimit = 232448;
constexpr int kCtrlRegs = 40, kEpiRegs = 232;  // setmaxnreg split: 128*40 + 256*232 = 384*168
constexpr int kScaleKb = 4;     // K blocks of scales per ring slot
constexpr int kScaleSlots = 4;  // ring slots (16 K blocks staged ahead)

// ROWB: B carries one scale per row (1x128 tiles, the weight-gradient GEMM)
// instead of one per 128x128 block. AEPI: the whole output tile is staged
// in shared memory and warp 3 issues its TMA stores (pair kernels).
template <int BN, bool GROUPED, bool PAIR, bool ROWB = false, bool AEPI = false>
struct Layout {
    static constexpr int A_BYTES = BM * BK;
    // 128-column scale blocks one tile can touch: n0 = BN * t is 128-aligned
    // for BN = 128 and 256; a 160- or 224-wide tile can start inside a block
    static constexpr int MAX_NB = BN % 128 == 0 ? BN / 128 : BN / 128 + 2;
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // rows of B this CTA loads
    static constexpr int B_BYTES = B_ROWS * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // 32-row staging boxes. Pair tiles stage all of a warp's 32 x BN/2
    // outputs at once, in boxes 64 bf16 wide (128-byte swizzle), or 16 wide
    // (32-byte swizzle) when BN/2 is not a multiple of 64, so that a tile
    // needs one proxy fence and few TMA stores per warp. One-CTA tiles use two
    // boxes per warp, 32 wide (64-byte swizzle) or 16 wide: one is filled while
    // the TMA store of the other is still reading.
    static constexpr bool FULL_STAGE = PAIR && !GROUPED;
    static constexpr int EPI_BOX_COLS = FULL_STAGE ? ((BN / 2) % 64 == 0 ? 64 : 16)
                                                   : ((BN / 2) % 32 == 0 ? 32 : 16);
    static constexpr int EPI_BOX_BYTES = 32 * EPI_BOX_COLS * 2;
    static constexpr int EPI_WARP_BYTES = FULL_STAGE ? 32 * (BN / 2) * 2 : 2 * EPI_BOX_BYTES;
    static constexpr int EPI_BYTES = GROUPED ? 0 : kEpiWarps * EPI_WARP_BYTES;
    // slot: sa as [128 rows][kScaleKb], then sb as [MAX_NB][kScaleKb]
    // (ROWB: sb as [kScaleKb][BN], the tile's columns contiguous per K block)
    static constexpr int SB_PER_KB = ROWB ? BN : MAX_NB;
    static constexpr int SCALE_SLOT_BYTES = 4 * kScaleKb * (BM + SB_PER_KB);
    static constexpr int SCALE_BYTES = kScaleSlots * SCALE_SLOT_BYTES;
    static constexpr int NBUF = (512 / BN) > 4 ? 4 : (512 / BN);  // TMEM buffers of BN columns
    static_assert(NBUF * BN <= 512 && (BN % 32) == 0, "TMEM buffers start on multiples of 32 columns");
    static constexpr int TMEM_COLS = NBUF * BN <= 128 ? 128 : NBUF * BN <= 256 ? 256 : 512;
    static constexpr int RESERVE = 1024 /*alignment slack*/ + 512 /*barriers, flags*/ +
                                   (GROUPED ? 4 * (kMaxExperts + 1) : 0);
    static constexpr int STAGES_FIT =
        (kSmemLimit - RESERVE - EPI_BYTES - SCALE_BYTES) / STAGE_BYTES;
    // 256-wide pair tiles measured faster with four stages than with six
    static constexpr int MAX_STAGES = PAIR && BN == 256 ? 4 : 6;
    static constexpr int STAGES = STAGES_FIT > MAX_STAGES ? MAX_STAGES : STAGES_FIT;
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
    static constexpr int SCALE_OFF = EPI_OFF + EPI_BYTES;
    static constexpr int BAR_OFF = SCALE_OFF + SCALE_BYTES;
    // barriers: full[S], empty[S], tmem_full[NBUF], tmem_empty[NBUF],
    // scale_full[slots], scale_empty[slots], drain, split-K partial and
    // decided, staged output tile (AEPI) and staging free (AEPI)
    static constexpr int FULL = 0, EMPTY = STAGES, TFULL = 2 * STAGES, TEMPTY = TFULL + NBUF,
                         SFULL = TEMPTY + NBUF, SEMPTY = SFULL + kScaleSlots,
                         DRAIN = SEMPTY + kScaleSlots, PARTIAL = DRAIN + 1, DECIDED = PARTIAL + 1,
                         EFULL = DECIDED + 1, EFREE = EFULL + 1, NUM_BARS = EFREE + 1;
    static constexpr int MISC_OFF = BAR_OFF + 8 * NUM_BARS;  // tmem slot, abort flag, last-split flag
    static constexpr int TABLE_OFF = MISC_OFF + 16;
    static constexpr int HALF = BN / 2;       // columns per promotion warp
    static constexpr int CHUNKS = HALF / 32;  // 32-column TMEM loads, issued in pairs
    static_assert(BN == 128 || BN == 160 || BN == 224 || BN == 256, "tile width must be 128, 160, 224 or 256");
    static_assert(BN != 160 || (PAIR && !GROUPED && !ROWB), "160-wide tiles are pair tiles of the block-scaled dense GEMM");
    static_assert(HALF % 32 == 0 || (!GROUPED && !ROWB), "160- and 224-wide tiles are for the block-scaled dense GEMM");
    static_assert(HALF % 32 == 16 || CHUNKS % 2 == 0, "32-column TMEM chunks are loaded in pairs");
    static_assert((B_ROWS * BK) % 1024 == 0 && STAGE_BYTES % 1024 == 0,
                  "stages and their B tiles must start on 1024-byte swizzle atoms");
    static_assert(!(PAIR && GROUPED), "pair mode is for the dense GEMM");
    static_assert(!(ROWB && GROUPED), "row-scaled B is for the dense GEMM");
    static_assert(!AEPI || (PAIR && !GROUPED), "the staged-tile epilogue is for pair tiles");
    static_assert(STAGES >= 2, "not enough shared memory for two stages");
    static_assert(8 * NUM_BARS + 16 <= 512, "barrier area overflow");
    static constexpr int smem_bytes(int E) {
        return TABLE_OFF + (GROUPED ? 4 * (E + 1) : 0) + 1024;
    }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// First column, within a promotion warp's HALF columns, of its staging box
// c2 (BC columns wide), which holds acc[BC c2, +BC). When HALF = 16 mod 32
// the promotion's chunk order puts those at warp columns 16 h + 16 c2, and
// the last box at HALF - 16 - (HALF - 16) h.
template <int HALF, int BC>
__device__ __forceinline__ int epi_box_col(int c2, int h) {
    return HALF % 32 == 0 ? BC * c2 : c2 < HALF / 16 - 1 ? 16 * h + 16 * c2 : (HALF - 16) * (1 - h);
}

// Row r of a BC-column staging box holds BC / 8 16-byte pieces; the TMA
// swizzle puts piece j at j ^ (r % 8) (128-byte swizzle, 64 columns),
// j ^ (r / 2 % 4) (64-byte, 32 columns) or j ^ (r / 4 % 2) (32-byte, 16).
template <int BC>
__device__ __forceinline__ uint32_t epi_swizzle(int r) {
    return BC == 64 ? r & 7 : BC == 32 ? (r >> 1) & 3 : (r >> 2) & 1;
}

struct Tile {
    int m0;       // first row of A / C
    int row_end;  // rows >= row_end are not this tile's (expert end or M)
    int n0;       // first column of C (= row of the expert's B)
    int brow;     // B row coordinate in the 2-D B tensor ([E*N, K] when grouped)
    int e;        // expert (0 when dense)
    int kbeg, kend;  // this unit's K blocks (the whole K range unless split)
    int ksplit;      // which K range (0 unless split)
};

// First K block of K range s of `splits` (ranges start on multiples of 4 K
// blocks, the granularity of the scale ring).
__device__ __forceinline__ int split_kbeg(int s, int splits, int KB) {
    const int kb4 = (KB + 3) / 4;
    return min(KB, 4 * ((s * kb4) / splits));
}

// Work unit t -> tile. Dense: groups of kGroupM row-units share n-tiles
// for L2 reuse. Pair mode: a unit is a pair of m-tiles (2u, 2u + 1), CTA
// `rank` of the pair takes m-tile 2u + rank and B rows n0 + rank * BN / 2.
template <int BN, bool GROUPED, bool PAIR, bool SPLITK = false>
__device__ __forceinline__ Tile decode_tile(const GemmArgs& a, const int* table, int t,
                                            uint32_t rank) {
    Tile r;
    r.kbeg = 0;
    r.kend = a.KB;
    r.ksplit = 0;
    if constexpr (!GROUPED) {
        if constexpr (SPLITK) {  // split index slowest: a wave holds one K range of many tiles
            r.ksplit = t / a.tile_units;
            t -= r.ksplit * a.tile_units;
            r.kbeg = split_kbeg(r.ksplit, a.splits, a.KB);
            r.kend = split_kbeg(r.ksplit + 1, a.splits, a.KB);
        }
        const int rows = PAIR ? a.mp_count : a.mt_count;
        const int per_group = kGroupM * a.nt_count;
        const int g = t / per_group, in = t - g * per_group;
        const int first = g * kGroupM;
        const int gm = min(kGroupM, rows - first);
        const int mu = first + in % gm, nt = in / gm;
        const int mt = PAIR ? 2 * mu + static_cast<int>(rank) : mu;
        r.m0 = mt * BM;
        r.row_end = a.M;
        r.n0 = nt * BN;
        r.brow = r.n0 + (PAIR ? static_cast<int>(rank) * (BN / 2) : 0);
        r.e = 0;
    } else {
        int lo = 0, hi = a.E - 1;  // largest e with table[e] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (table[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int beg = __ldg(a.offsets + lo), end = __ldg(a.offsets + lo + 1);
        const int mtiles = (end - beg + BM - 1) / BM;
        const int local = t - table[lo];
        const int nt = local / mtiles, mt = local - nt * mtiles;
        r.m0 = beg + mt * BM;
        r.row_end = end;
        r.n0 = nt * BN;
        r.brow = lo * a.N + r.n0;
        r.e = lo;
    }
    return r;
}

// Grouped schedule, built by one warp: table[e] = number of tiles of experts
// before e (m-tiles of ceil(rows/128) times n-tiles), table[E] = total.
// Malformed offsets give total = 0 and set the device status.
__device__ void build_group_table(const GemmArgs& a, int* table) {
    const int lane = threadIdx.x & 31;
    const int per = (a.E + 31) / 32;
    const int b0 = min(a.E, lane * per), b1 = min(a.E, b0 + per);
    bool bad = false;
    int local = 0;
    for (int e = b0; e < b1; ++e) {
        const int lo = __ldg(a.offsets + e), hi = __ldg(a.offsets + e + 1);
        if (hi < lo) bad = true;
        else local += (hi - lo + BM - 1) / BM * a.nt_count;
    }
    if (lane == 0 && __ldg(a.offsets) != 0) bad = true;
    if (lane == 31 && __ldg(a.offsets + a.E) != a.M) bad = true;
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += v;
    }
    int run = incl - local;
    for (int e = b0; e < b1; ++e) {
        table[e] = run;
        const int lo = __ldg(a.offsets + e), hi = __ldg(a.offsets + e + 1);
        if (hi >= lo) run += (hi - lo + BM - 1) / BM * a.nt_count;
    }
    const bool any_bad = __any_sync(0xFFFFFFFFu, bad);
    const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (lane == 0) {
        table[a.E] = any_bad ? 0 : total;
        if (any_bad && blockIdx.x == 0) atomicOr(&g_device_status, FP8Q_DEVSTATUS_BAD_OFFSETS);
    }
}

// A bounded wait taken by a whole warp: true only if every lane saw the
// phase complete (the lanes may disagree only at the time limit).
template <bool CLUSTER = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit) {
    return __all_sync(0xFFFFFFFFu, mbar_wait<CLUSTER>(bar, parity, abort_flag, limit));
}

// acc[O .. O + NCOL) += P * c, packed.
template <int O, int NCOL, int HALF>
__device__ __forceinline__ void fma_cols(float (&acc)[HALF], const uint32_t* r, float c) {
#pragma unroll
    for (int i = 0; i < NCOL; i += 2) ffma2(acc[O + i], acc[O + i + 1], r[i], r[i + 1], c);
}

// Promotion of one warp's HALF columns when HALF = 16 mod 32 (112 of a
// 224-wide tile, 80 of a 160-wide one), the same code for both warpgroups (h):
// 32-column chunks at warp columns b + 32 i (b = 16 h) into acc[32 i, +32),
// i < HALF / 32, and a 16-column chunk at column (HALF - 16) (1 - h) into
// acc[HALF - 16, HALF). Every 32-column chunk then starts on a multiple of 32
// (the tile starts on one; a warpgroup's HALF columns leave 16 over), so
// none crosses a 128-column scale block: a chunk at warp column o uses cs
// when o < split, else csn. 112 columns: two TMEM loads per wait; 80
// columns: all three loads, then one wait.
template <int HALF>
__device__ __forceinline__ void promote_odd(float (&acc)[HALF], uint32_t taddr, int h, float cs,
                                            float csn, int split) {
    static_assert(HALF == 112 || HALF == 80, "112 or 80 columns per warp");
    const int b = 16 * h, o16 = (HALF - 16) * (1 - h);
    uint32_t r0[32], r1[32];
    if constexpr (HALF == 112) {
        tmem_ld32(taddr + b, r0);
        tmem_ld32(taddr + b + 32, r1);
        tmem_wait_ld64(r0, r1);
        fma_cols<0, 32>(acc, r0, b < split ? cs : csn);
        fma_cols<32, 32>(acc, r1, b + 32 < split ? cs : csn);
        uint32_t r2[32], r3[16];
        tmem_ld32(taddr + b + 64, r2);
        tmem_ld16(taddr + o16, r3);
        tmem_wait_ld48(r2, r3);
        fma_cols<64, 32>(acc, r2, b + 64 < split ? cs : csn);
        fma_cols<HALF - 16, 16>(acc, r3, o16 < split ? cs : csn);
    } else {
        uint32_t r3[16];
        tmem_ld32(taddr + b, r0);
        tmem_ld32(taddr + b + 32, r1);
        tmem_ld16(taddr + o16, r3);
        tmem_wait_ld64(r0, r1);
        reg_order16(r3);  // the wait above covers r3's load too
        fma_cols<0, 32>(acc, r0, b < split ? cs : csn);
        fma_cols<32, 32>(acc, r1, b + 32 < split ? cs : csn);
        fma_cols<HALF - 16, 16>(acc, r3, o16 < split ? cs : csn);
    }
}

// Column of this warp's tile slice that acc[i] holds: i itself, except for
// 112- and 80-column warps (224- and 160-wide tiles), whose chunk order puts
// warp columns 16 h .. 16 h + HALF - 17 in acc[0, HALF - 16) and the
// remaining 16 columns in acc[HALF - 16, HALF).
template <int HALF>
__device__ __forceinline__ int acc_col(int i, int h) {
    if constexpr (HALF % 32 == 0) {
        return i;
    } else {
        return i < HALF - 16 ? 16 * h + i : (HALF - 16) * (1 - h) + (i - (HALF - 16));
    }
}

// One arrival on a tile's arrival word, tagged with this call's epoch: a word
// holding another call's tag counts as zero. Returns the number of arrivals
// of this call including this one (0 if the bounded retry loop gave up).
__device__ __forceinline__ uint32_t arrive_count(uint32_t* word, uint32_t epoch, volatile int* abort_flag) {
    uint32_t cur = *reinterpret_cast<volatile uint32_t*>(word);
    for (int it = 0; it < (1 << 16); ++it) {
        const uint32_t next = (cur >> 8) == epoch ? cur + 1u : ((epoch << 8) | 1u);
        const uint32_t prev = atomicCAS(word, cur, next);
        if (prev == cur) return next & 0xFFu;
        cur = prev;
    }
    *abort_flag = 1;
    return 0;
}

// Release / acquire fences at GPU scope (lighter than a sequentially
// consistent fence): the partial tile's stores before the arrival count,
// the arrival count before the other units' partials are read.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Split K: write this unit's FP32 partial tile to the workspace, count the
// unit's arrival on the tile's word, and if it is the last unit of the tile,
// replace acc by the sum of all partials taken in range order (its own from
// registers), so that C does not depend on which unit finishes last.
// Workspace layout per K range and tile: [BN / 4 column groups][128 rows]
// of float4, so a warp (32 consecutive rows) moves 512 contiguous bytes per
// column group; tiles = m-tiles (rounded up to pairs in pair mode) x n-tiles,
// and columns past N / rows past M hold unused values. The 8 promotion warps
// meet on two barriers with bounded waits. Returns false if a wait gave up.
template <int BN, bool PAIR, int HALF>
__device__ __forceinline__ bool split_reduce(const GemmArgs& a, const Tile& tile, float (&acc)[HALF],
                                             int row, int h, int ew, int lane, uint32_t bar_partial,
                                             uint32_t bar_decided, uint32_t phase, volatile uint32_t* last_flag,
                                             volatile int* abort_flag, uint64_t limit, bool& last) {
    const int64_t tiles = static_cast<int64_t>(PAIR ? 2 * a.mp_count : a.mt_count) * a.nt_count;
    const int64_t ctile = static_cast<int64_t>(tile.m0 / BM) * a.nt_count + tile.n0 / BN;
    const int64_t range_f4 = tiles * (BN / 4) * BM;  // float4s per K range
    // this row's float4 in column group 0 of this warp's slice, K range 0;
    // column group g is g * 128 float4s further
    const float4* base = reinterpret_cast<const float4*>(a.ws) + ctile * (BN / 4) * BM + (h * HALF / 4) * BM + row;
    float4* mine = const_cast<float4*>(base) + tile.ksplit * range_f4;
#pragma unroll
    for (int i = 0; i < HALF; i += 4)
        __stcg(mine + (acc_col<HALF>(i, h) / 4) * BM, make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]));
    fence_acq_rel_gpu();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_partial);
    if (ew == 0) {
        if (!warp_wait(bar_partial, phase, abort_flag, limit)) return false;
        if (lane == 0) {
            const uint32_t n = arrive_count(a.counters + ctile, a.epoch, abort_flag);
            fence_acq_rel_gpu();
            *last_flag = n == static_cast<uint32_t>(a.splits) ? 1u : 0u;
            mbar_arrive(bar_decided);
        }
        __syncwarp();
    }
    if (!warp_wait(bar_decided, phase, abort_flag, limit)) return false;
    last = *last_flag != 0u;
    if (!last) return true;
    fence_acq_rel_gpu();
    // 16 columns at a time, all loads of one K range issued together:
    // (p_0 + ... + p_(me-1)) + acc, then + p_(me+1) + ... (range order)
    const int me = tile.ksplit;
#pragma unroll
    for (int i0 = 0; i0 < HALF; i0 += 16) {
        const float4* b = base + (acc_col<HALF>(i0, h) / 4) * BM;
        float* c = acc + i0;
        if (me > 0) {
            float4 r0 = __ldcg(b), r1 = __ldcg(b + BM), r2 = __ldcg(b + 2 * BM), r3 = __ldcg(b + 3 * BM);
            for (int s = 1; s < me; ++s) {
                const float4* q = b + s * range_f4;
                const float4 p0 = __ldcg(q), p1 = __ldcg(q + BM), p2 = __ldcg(q + 2 * BM), p3 = __ldcg(q + 3 * BM);
                r0.x += p0.x; r0.y += p0.y; r0.z += p0.z; r0.w += p0.w;
                r1.x += p1.x; r1.y += p1.y; r1.z += p1.z; r1.w += p1.w;
                r2.x += p2.x; r2.y += p2.y; r2.z += p2.z; r2.w += p2.w;
                r3.x += p3.x; r3.y += p3.y; r3.z += p3.z; r3.w += p3.w;
            }
            c[0] = r0.x + c[0]; c[1] = r0.y + c[1]; c[2] = r0.z + c[2]; c[3] = r0.w + c[3];
            c[4] = r1.x + c[4]; c[5] = r1.y + c[5]; c[6] = r1.z + c[6]; c[7] = r1.w + c[7];
            c[8] = r2.x + c[8]; c[9] = r2.y + c[9]; c[10] = r2.z + c[10]; c[11] = r2.w + c[11];
            c[12] = r3.x + c[12]; c[13] = r3.y + c[13]; c[14] = r3.z + c[14]; c[15] = r3.w + c[15];
        }
        for (int s = me + 1; s < a.splits; ++s) {
            const float4* q = b + s * range_f4;
            const float4 p0 = __ldcg(q), p1 = __ldcg(q + BM), p2 = __ldcg(q + 2 * BM), p3 = __ldcg(q + 3 * BM);
            c[0] += p0.x; c[1] += p0.y; c[2] += p0.z; c[3] += p0.w;
            c[4] += p1.x; c[5] += p1.y; c[6] += p1.z; c[7] += p1.w;
            c[8] += p2.x; c[9] += p2.y; c[10] += p2.z; c[11] += p2.w;
            c[12] += p3.x; c[13] += p3.y; c[14] += p3.z; c[15] += p3.w;
        }
    }
    return true;
}

// SPLITK: work units are (tile, K range) pairs and the epilogue reduces the
// partial tiles through the workspace (dense block-scaled GEMM only).
template <int BN, bool GROUPED, bool PAIR, bool ROWB, bool SPLITK>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
    // pair tiles stage the whole output tile and leave its stores to warp 3
    // (split K keeps the promotion warps' own stores)
    constexpr bool AEPI = PAIR && !GROUPED && !SPLITK;
    // ... except a CTA's last tile, which has nothing to overlap its stores
    // with: the narrower pair tiles (one wave at the MLA shapes) store it
    // from the promotion warps; 256-wide tiles measured faster without the
    // extra branch
    constexpr bool LAST_DIRECT = AEPI && BN != 256;
    using L = Layout<BN, GROUPED, PAIR, ROWB, AEPI>;
    constexpr int S = L::STAGES;
    constexpr int NBUF = L::NBUF;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    auto bar = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
    int* table = reinterpret_cast<int*>(smem + L::TABLE_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t limit = args.timeout_ns;
    // Pair mode: rank in the pair; the even CTA owns the MMA-side barriers.
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    auto lead_bar = [&](int i) -> uint32_t { return PAIR ? mapa_shared(bar(i), 0) : bar(i); };
    const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int unit_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(L::FULL + s), PAIR ? 2 : 1);  // pair: both CTAs' producers
            mbar_init(bar(L::EMPTY + s), 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(bar(L::TFULL + b), 1);
            mbar_init(bar(L::TEMPTY + b), PAIR ? 2 * kEpiWarps : kEpiWarps);
        }
        for (int j = 0; j < kScaleSlots; ++j) {
            mbar_init(bar(L::SFULL + j), 32);  // one cp.async completion arrive per lane
            mbar_init(bar(L::SEMPTY + j), kEpiWarps);
        }
        mbar_init(bar(L::DRAIN), 1);
        mbar_init(bar(L::PARTIAL), kEpiWarps);
        mbar_init(bar(L::DECIDED), 1);
        mbar_init(bar(L::EFULL), kEpiWarps);
        mbar_init(bar(L::EFREE), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if constexpr (!GROUPED) prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        tmem_alloc<PAIR>(sbase + L::MISC_OFF, L::TMEM_COLS);
        tmem_relinquish_alloc_permit<PAIR>();
    }
    if constexpr (GROUPED) {
        if (warp == 3) build_group_table(args, table);
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // peer barriers initialised before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const int num_tiles = GROUPED ? table[args.E] : args.num_tiles;
    const int KB = args.KB;

    // Registers: 384 threads launch with 168 each (64512). The control
    // warpgroup (producer, MMA, scale loader, store warp) gives most of its
    // share to the two promotion warpgroups, which hold a 128 x BN/2 FP32
    // accumulator slice (BN/2 registers per thread) plus two 32-column TMEM
    // chunks: 128 * 40 + 256 * 232 = 64512.
    if (warp < kFirstEpiWarp) {
        setmaxnreg_dec<kCtrlRegs>();
        if (warp == 0) {
            // -------------------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0, issued = 0;
            bool ok = true;
            for (int t = unit0; ok && t < num_tiles; t += unit_step) {
                const Tile tile = decode_tile<BN, GROUPED, PAIR, SPLITK>(args, table, t, rank);
                for (int kb = tile.kbeg; kb < tile.kend; ++kb) {
                    if (!warp_wait(bar(L::EMPTY + stage), phase ^ 1u, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        uint32_t bytes = L::STAGE_BYTES;
                        if ((args.debug & 1u) && issued == 0) bytes += 16;  // never-completing phase
                        const uint32_t sA = sbase + stage * L::STAGE_BYTES;
                        if constexpr (PAIR) {
                            const uint32_t fb = lead_bar(L::FULL + stage);
                            mbar_arrive_expect_tx_cluster(fb, bytes);
                            tma_load_2d_pair(sA, &tmA, fb, kb * BK, tile.m0);
                            tma_load_2d_pair(sA + L::A_BYTES, &tmB, fb, kb * BK, tile.brow);
                        } else {
                            mbar_arrive_expect_tx(bar(L::FULL + stage), bytes);
                            tma_load_2d(sA, &tmA, bar(L::FULL + stage), kb * BK, tile.m0);
                            tma_load_2d(sA + L::A_BYTES, &tmB, bar(L::FULL + stage), kb * BK, tile.brow);
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
            // Wait for the copies still landing in shared memory (normally
            // all consumed already) before the CTA may exit. In pair mode the
            // even CTA's full barriers count both CTAs' bytes, and the odd CTA
            // leaves only after the closing cluster barrier.
            for (int s = 0; s < S && leader; ++s) {
                if (static_cast<uint32_t>(s) >= issued) break;
                const uint32_t last = s + S * ((issued - 1 - s) / S);
                volatile int local_flag = 0;
                mbar_wait(bar(L::FULL + s), (last / S) & 1u, &local_flag, limit);
            }
        } else if (warp == 1 && leader) {
            // --------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_e4m3_f32(PAIR ? 2 * BM : BM, BN);
            int stage = 0;
            uint32_t phase = 0, abuf = 0, aphase = 0;
            bool ok = true, issued_any = false;
            for (int t = unit0; ok && t < num_tiles; t += unit_step) {
                const Tile tile = decode_tile<BN, GROUPED, PAIR, SPLITK>(args, table, t, rank);
                for (int kb = tile.kbeg; kb < tile.kend; ++kb) {
                    // the operands usually land long before the accumulator
                    // buffer is released: wait for them first, so that only
                    // the release stands between the promotion and the MMA
                    if (!warp_wait<PAIR>(bar(L::FULL + stage), phase, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = sbase + stage * L::STAGE_BYTES;
                    const uint64_t ad = sdesc_k_sw128(sA);
                    const uint64_t bd = sdesc_k_sw128(sA + L::A_BYTES);
                    const uint32_t d = tmem_base + abuf * BN;
                    if (!warp_wait<PAIR>(bar(L::TEMPTY + abuf), aphase ^ 1u, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (elect_one()) {
                        if constexpr (PAIR) {
#pragma unroll
                            for (int k = 0; k < BK / 32; ++k)
                                mma_e4m3_pair(d, ad + 2u * k, bd + 2u * k, idesc, k > 0 ? 1u : 0u);
                            mma_commit_pair(bar(L::EMPTY + stage));
                            mma_commit_pair(bar(L::TFULL + abuf));
                        } else {
#pragma unroll
                            for (int k = 0; k < BK / 32; ++k)
                                mma_e4m3(d, ad + 2u * k, bd + 2u * k, idesc, k > 0 ? 1u : 0u);
                            mma_commit(bar(L::EMPTY + stage));
                            mma_commit(bar(L::TFULL + abuf));
                        }
                    }
                    __syncwarp();
                    issued_any = true;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++abuf == NBUF) {
                        abuf = 0;
                        aphase ^= 1u;
                    }
                }
            }
            // Every MMA issued above has completed once this arrives.
            if (issued_any) {
                if (elect_one()) {
                    if constexpr (PAIR) mma_commit_pair_local(bar(L::DRAIN));
                    else mma_commit(bar(L::DRAIN));
                }
                __syncwarp();
                volatile int local_flag = 0;
                mbar_wait(bar(L::DRAIN), 0, &local_flag, limit);
            }
        } else if (warp == kScaleWarp) {
            // ------------------------------------------------- scale loader
            // Slot j holds K blocks [kb0, kb0 + 4): sa of the tile's 128 rows
            // (row r at floats 4r .. 4r + 3) and sb of the 128-column blocks the
            // tile touches (block i at floats 512 + 4i ..). Rows outside the tile,
            // blocks past the last one and K blocks past the end are zero.
            // When KB % 4 == 0 (and sa, sb are 16-byte aligned) each row's four
            // values are one 16-byte copy.
            const bool wide = (KB % kScaleKb) == 0 &&
                              ((reinterpret_cast<uintptr_t>(args.sa) |
                                reinterpret_cast<uintptr_t>(args.sb)) & 15u) == 0;
            int slot = 0;
            uint32_t sphase = 0;
            bool ok = true;
            for (int t = unit0; ok && t < num_tiles; t += unit_step) {
                const Tile tile = decode_tile<BN, GROUPED, PAIR, SPLITK>(args, table, t, rank);
                const float* sb_e = args.sb + static_cast<int64_t>(tile.e) * args.NB * KB;
                const int nb = (tile.n0 >> 7) + (lane < L::MAX_NB ? lane : 0);
                const bool sb_ok = lane < L::MAX_NB && nb < args.NB && (nb << 7) < tile.n0 + BN;
                for (int kb0 = tile.kbeg; kb0 < tile.kend; kb0 += kScaleKb) {
                    if (!warp_wait(bar(L::SEMPTY + slot), sphase ^ 1u, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sl = sbase + L::SCALE_OFF + slot * L::SCALE_SLOT_BYTES;
#pragma unroll
                    for (int i = 0; i < BM / 32; ++i) {
                        const int r = lane + 32 * i;
                        const int m = tile.m0 + r;
                        const bool live = m < tile.row_end;
                        const float* src = args.sa + (live ? static_cast<int64_t>(m) * KB + kb0 : 0);
                        if (wide) {
                            cp_async_16(sl + 16u * r, src, live ? 16u : 0u);
                        } else {
#pragma unroll
                            for (int j = 0; j < kScaleKb; ++j) {
                                const bool in = live && kb0 + j < KB;
                                cp_async_4(sl + 16u * r + 4u * j, in ? src + j : args.sa, in ? 4u : 0u);
                            }
                        }
                    }
                    if constexpr (ROWB) {
                        // sb[n][kb0 + j] -> slot float BM * kScaleKb + j * BN + (n - n0)
                        const uint32_t sbl = sl + 4u * kScaleKb * BM;
#pragma unroll 1
                        for (int i = 0; i < BN / 32; ++i) {
                            const int c = lane + 32 * i;
                            const int n = tile.n0 + c;
                            const bool col_ok = n < args.N;
                            const float* src = args.sb + (col_ok ? static_cast<int64_t>(n) * KB + kb0 : 0);
#pragma unroll
                            for (int j = 0; j < kScaleKb; ++j) {
                                const bool in = col_ok && kb0 + j < KB;
                                cp_async_4(sbl + 4u * (j * BN + c), in ? src + j : args.sb, in ? 4u : 0u);
                            }
                        }
                    } else if (lane < L::MAX_NB) {
                        const float* src = sb_e + (sb_ok ? static_cast<int64_t>(nb) * KB + kb0 : 0);
                        const uint32_t dst = sl + 16u * (BM + lane);
                        if (wide) {
                            cp_async_16(dst, src, sb_ok ? 16u : 0u);
                        } else {
#pragma unroll
                            for (int j = 0; j < kScaleKb; ++j) {
                                const bool in = sb_ok && kb0 + j < KB;
                                cp_async_4(dst + 4u * j, in ? src + j : args.sb, in ? 4u : 0u);
                            }
                        }
                    }
                    cp_async_mbar_arrive(bar(L::SFULL + slot));
                    if (++slot == kScaleSlots) {
                        slot = 0;
                        sphase ^= 1u;
                    }
                }
            }
            // Let the last copies land before the CTA may exit.
            asm volatile("cp.async.wait_all;" ::: "memory");
        } else if (warp == 3) {
            if constexpr (AEPI) {
                // ------------------------------------------------- C stores
                // Per tile: wait until the eight promotion warps have staged
                // their 32 x BN/2 outputs, issue the tile's TMA stores (lane i
                // those of promotion warp i), and hand the staging back once
                // the stores have read it. The promotion warps go on to the
                // next tile meanwhile.
                uint32_t ephase = 0;
                bool ok = true;
                for (int t = unit0; ok && t < num_tiles; t += unit_step) {
                    if (LAST_DIRECT && t + unit_step >= num_tiles) break;
                    const Tile tile = decode_tile<BN, GROUPED, PAIR, SPLITK>(args, table, t, rank);
                    if (!warp_wait(bar(L::EFULL), ephase, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    if (lane < kEpiWarps) {
                        constexpr int BC = L::EPI_BOX_COLS;
                        const int h = lane >> 2;
                        const int x0 = tile.n0 + h * L::HALF, y = tile.m0 + (lane & 3) * 32;
                        const uint32_t wbuf = sbase + L::EPI_OFF + lane * L::EPI_WARP_BYTES;
#pragma unroll 1
                        for (int c2 = 0; c2 < L::HALF / BC; ++c2) {
                            const int x = x0 + epi_box_col<L::HALF, BC>(c2, h);
                            if (x < args.N && y < args.M)
                                tma_store_2d(&tmC, wbuf + c2 * L::EPI_BOX_BYTES, x, y);
                        }
                        bulk_commit_group();
                        bulk_wait_group_read0();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(L::EFREE));
                    ephase ^= 1u;
                }
                if (lane < kEpiWarps) bulk_wait_group0();  // writes done before the CTA exits
            }
        }
    } else {
        // --------------------------------------------- promotion + epilogue
        setmaxnreg_inc<kEpiRegs>();
        const int ew = warp - kFirstEpiWarp;  // 0..7
        const int quarter = warp & 3;         // TMEM lanes 32*quarter .. +31
        const int h = ew >> 2;                // column half
        const int row = quarter * 32 + lane;  // row inside the tile
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        const float* scale_ring = reinterpret_cast<const float*>(smem + L::SCALE_OFF);
        uint32_t abuf = 0, aphase = 0;
        int slot = 0;
        uint32_t sphase = 0;
        uint32_t ebox = 0;  // epilogue boxes staged so far: their buffer alternates
        uint32_t ephase = 0;  // AEPI: output tiles staged so far (barrier parity)
        uint32_t sred_phase = 0;  // split-K reductions done so far (barrier parity)
        bool ok = true;
        const uint32_t temptry_base = PAIR ? mapa_shared(bar(L::TEMPTY), 0) : bar(L::TEMPTY);
        for (int t = unit0; ok && t < num_tiles; t += unit_step) {
            const Tile tile = decode_tile<BN, GROUPED, PAIR, SPLITK>(args, table, t, rank);
            const int m = tile.m0 + row;
            const bool row_ok = m < tile.row_end;
            const int col0 = tile.n0 + h * L::HALF;  // first column of this warp
            float acc[L::HALF];
#pragma unroll
            for (int j = 0; j < L::HALF; ++j) acc[j] = 0.0f;

            // For BN = 128 and 256 this warp's columns lie in one 128-column
            // block (n0 % BN == 0), so each K block needs one scale product
            // sa[m][kb] * sb[nb][kb]. A 160- or 224-wide tile starts at a multiple
            // of 32 and a warp's 80 or 112 columns touch at most two blocks: the first
            // `split` columns use block rel_nb, the rest block rel_nb + 1.
            const int wcol = (tile.n0 & 127) + h * L::HALF;  // from the tile's first block
            const int rel_nb = wcol >> 7;
            const int split = 128 - (wcol & 127);
            float4 sa4 = make_float4(0.f, 0.f, 0.f, 0.f), sb4 = sa4, sb4n = sa4;
            const float* sb_cols = scale_ring;  // ROWB: this warp's sb columns in the slot
            for (int kb = tile.kbeg; kb < tile.kend; ++kb) {
                const int j = kb & (kScaleKb - 1);
                if (j == 0) {
                    // scales of K blocks kb .. kb + 3, from the ring (staged ahead)
                    if (!warp_wait(bar(L::SFULL + slot), sphase, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    const float* sl = scale_ring + slot * (L::SCALE_SLOT_BYTES / 4);
                    sa4 = *reinterpret_cast<const float4*>(sl + 4 * row);
                    if constexpr (ROWB) {
                        // read per K block below; the slot is released after
                        // its last K block
                        sb_cols = sl + kScaleKb * BM + h * L::HALF;
                    } else {
                        sb4 = *reinterpret_cast<const float4*>(sl + 4 * (BM + rel_nb));
                        if constexpr (L::HALF % 32 == 16)
                            sb4n = *reinterpret_cast<const float4*>(sl + 4 * (BM + rel_nb + 1));
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(L::SEMPTY + slot));
                        if (++slot == kScaleSlots) {
                            slot = 0;
                            sphase ^= 1u;
                        }
                    }
                }
                const float a_s = j == 0 ? sa4.x : j == 1 ? sa4.y : j == 2 ? sa4.z : sa4.w;
                const float b_s = j == 0 ? sb4.x : j == 1 ? sb4.y : j == 2 ? sb4.z : sb4.w;
                const float cs = a_s * b_s;
                const float b_sn = j == 0 ? sb4n.x : j == 1 ? sb4n.y : j == 2 ? sb4n.z : sb4n.w;
                const float csn = a_s * b_sn;  // 160/224-wide tiles: the warp's second block

                if (!warp_wait<PAIR>(bar(L::TFULL + abuf), aphase, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t taddr = lane_base + abuf * BN + h * L::HALF;
                if constexpr (ROWB) {
                    // column n's scale product is sa[m][kb] * sb[n][kb]; one
                    // 32-column chunk at a time, its 32 sb values loaded from
                    // shared memory while the chunk's TMEM load is in flight
                    const uint32_t sbk = smem_u32(sb_cols + j * BN);
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; ++c) {
                        float4 b[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) b[i] = lds_f4(sbk + 4u * (32 * c + 4 * i));
                        uint32_t r0[32];
                        tmem_ld32(taddr + 32 * c, r0);
                        tmem_wait_ld32(r0);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            float* a = acc + 32 * c + 4 * i;
                            ffma2_cols(a[0], a[1], r0[4 * i], r0[4 * i + 1], a_s, b[i].x, b[i].y);
                            ffma2_cols(a[2], a[3], r0[4 * i + 2], r0[4 * i + 3], a_s, b[i].z, b[i].w);
                        }
                    }
                } else if constexpr (L::HALF % 32 == 16) {
                    promote_odd<L::HALF>(acc, taddr, h, cs, csn, split);
                } else {
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; c += 2) {
                        uint32_t r0[32], r1[32];
                        tmem_ld32(taddr + 32 * c, r0);
                        tmem_ld32(taddr + 32 * (c + 1), r1);
                        tmem_wait_ld64(r0, r1);
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            ffma2(acc[32 * c + i], acc[32 * c + i + 1], r0[i], r0[i + 1], cs);
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            ffma2(acc[32 * (c + 1) + i], acc[32 * (c + 1) + i + 1], r1[i], r1[i + 1], cs);
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR) mbar_arrive_cluster(temptry_base + 8u * abuf);
                    else mbar_arrive(bar(L::TEMPTY + abuf));
                }
                if constexpr (ROWB) {
                    if (j == kScaleKb - 1 || kb == tile.kend - 1) {
                        if (lane == 0) mbar_arrive(bar(L::SEMPTY + slot));
                        if (++slot == kScaleSlots) {
                            slot = 0;
                            sphase ^= 1u;
                        }
                    }
                }
                if (++abuf == NBUF) {
                    abuf = 0;
                    aphase ^= 1u;
                }
            }
            if (!ok) break;

            if constexpr (SPLITK) {
                {
                    bool last = false;
                    if (!split_reduce<BN, PAIR, L::HALF>(args, tile, acc, row, h, ew, lane,
                                               bar(L::PARTIAL), bar(L::DECIDED), sred_phase,
                                               reinterpret_cast<volatile uint32_t*>(smem + L::MISC_OFF + 8),
                                               abort_flag, limit, last)) {
                        ok = false;
                        break;
                    }
                    sred_phase ^= 1u;
                    if (!last) continue;  // another unit of this tile stores C
                }
            }

            if constexpr (AEPI) {
                // bf16 -> the warp's swizzled staging boxes (layout below), all
                // of them at once, once warp 3 has released the staging (the
                // previous tile's stores have read it); warp 3 stores them
                if (!warp_wait(bar(L::EFREE), ephase ^ 1u, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                constexpr int BC = L::EPI_BOX_COLS;
                const uint32_t wrow = sbase + L::EPI_OFF + ew * L::EPI_WARP_BYTES + lane * (2 * BC);
                const uint32_t sw = epi_swizzle<BC>(lane);
#pragma unroll
                for (int c2 = 0; c2 < L::HALF / BC; ++c2) {
#pragma unroll
                    for (int j = 0; j < BC / 8; ++j) {
                        const float* v = acc + BC * c2 + 8 * j;
                        sts_u4(wrow + c2 * L::EPI_BOX_BYTES + ((j ^ sw) << 4), pack_bf16x2(v[0], v[1]),
                               pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (!LAST_DIRECT || t + unit_step < num_tiles) {
                    if (lane == 0) mbar_arrive(bar(L::EFULL));
                } else if (lane == 0) {
                    const uint32_t wbuf = sbase + L::EPI_OFF + ew * L::EPI_WARP_BYTES;
                    const int y = tile.m0 + quarter * 32;
#pragma unroll
                    for (int c2 = 0; c2 < L::HALF / BC; ++c2) {
                        const int x = col0 + epi_box_col<L::HALF, BC>(c2, h);
                        if (x < args.N && y < args.M) tma_store_2d(&tmC, wbuf + c2 * L::EPI_BOX_BYTES, x, y);
                    }
                    bulk_commit_group();
                }
                ephase ^= 1u;
            } else if constexpr (L::FULL_STAGE) {
                // bf16 -> all of the warp's swizzled staging boxes (box c2
                // holds acc[BC c2, +BC), see epi_box_col), one proxy fence, then
                // the boxes' TMA stores. The previous tile's stores finished
                // reading the staging long ago; wait for that all the same.
                constexpr int BC = L::EPI_BOX_COLS;
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
                const uint32_t wrow = sbase + L::EPI_OFF + ew * L::EPI_WARP_BYTES + lane * (2 * BC);
                const uint32_t sw = epi_swizzle<BC>(lane);
#pragma unroll
                for (int c2 = 0; c2 < L::HALF / BC; ++c2) {
#pragma unroll
                    for (int j = 0; j < BC / 8; ++j) {
                        const float* v = acc + BC * c2 + 8 * j;
                        sts_u4(wrow + c2 * L::EPI_BOX_BYTES + ((j ^ sw) << 4), pack_bf16x2(v[0], v[1]),
                               pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t wbuf = sbase + L::EPI_OFF + ew * L::EPI_WARP_BYTES;
                    const int y = tile.m0 + quarter * 32;
#pragma unroll
                    for (int c2 = 0; c2 < L::HALF / BC; ++c2) {
                        const int x = col0 + epi_box_col<L::HALF, BC>(c2, h);
                        if (x < args.N && y < args.M) tma_store_2d(&tmC, wbuf + c2 * L::EPI_BOX_BYTES, x, y);
                    }
                    bulk_commit_group();
                }
            } else if constexpr (!GROUPED) {
                // bf16 -> swizzled staging (32 rows x EPI_BOX_COLS per box, two
                // boxes per warp, pieces placed by epi_swizzle) -> TMA store, one
                // box at a time. Box c2 stores acc[BC c2, +BC) (see epi_box_col).
                constexpr int BC = L::EPI_BOX_COLS;
                uint8_t* ebuf0 = smem + L::EPI_OFF + ew * L::EPI_WARP_BYTES;
                const uint32_t ebuf0_s = sbase + L::EPI_OFF + ew * L::EPI_WARP_BYTES;
#pragma unroll
                for (int c2 = 0; c2 < L::HALF / BC; ++c2) {
                    const uint32_t eb = ebox++ & 1u;  // across tiles too (odd box counts)
                    uint8_t* ebuf = ebuf0 + eb * L::EPI_BOX_BYTES;
                    const uint32_t ebuf_s = ebuf0_s + eb * L::EPI_BOX_BYTES;
                    // the store issued two boxes ago (same buffer) must have read
                    // it: every box commits one bulk group, so at most the previous
                    // box's may still be reading
                    if (lane == 0) bulk_wait_group_read1();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < BC / 8; ++j) {
                        const float* v = acc + BC * c2 + 8 * j;
                        uint4 pk;
                        pk.x = pack_bf16x2(v[0], v[1]);
                        pk.y = pack_bf16x2(v[2], v[3]);
                        pk.z = pack_bf16x2(v[4], v[5]);
                        pk.w = pack_bf16x2(v[6], v[7]);
                        const int phys = j ^ static_cast<int>(epi_swizzle<BC>(lane));
                        *reinterpret_cast<uint4*>(ebuf + lane * (2 * BC) + phys * 16) = pk;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    const int x = col0 + epi_box_col<L::HALF, BC>(c2, h), y = tile.m0 + quarter * 32;
                    if (lane == 0) {
                        if (x < args.N && y < args.M) tma_store_2d(&tmC, ebuf_s, x, y);
                        bulk_commit_group();  // empty when the box lies past C
                    }
                }
            } else {
                // masked direct stores: rows past the expert's end belong to
                // another expert's tile
                if (row_ok) {
                    __nv_bfloat16* crow = args.C + static_cast<int64_t>(m) * args.N;
#pragma unroll
                    for (int j = 0; j < L::HALF / 8; ++j) {
                        const int col = col0 + 8 * j;
                        if (col < args.N) {
                            const float* v = acc + 8 * j;
                            uint4 pk;
                            pk.x = pack_bf16x2(v[0], v[1]);
                            pk.y = pack_bf16x2(v[2], v[3]);
                            pk.z = pack_bf16x2(v[4], v[5]);
                            pk.w = pack_bf16x2(v[6], v[7]);
                            *reinterpret_cast<uint4*>(crow + col) = pk;
                        }
                    }
                }
            }
        }
        if constexpr (!GROUPED) {
            if (lane == 0) bulk_wait_group0();
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the even CTA's MMAs (drained) may write our TMEM
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<PAIR>(tmem_base, L::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&g_device_status, FP8Q_DEVSTATUS_TIMEOUT);
}

template <int BN, bool GROUPED, bool PAIR, bool ROWB, bool SPLITK = false>
cudaError_t prepare(int smem) {
    auto kern = fp8_gemm_kernel<BN, GROUPED, PAIR, ROWB, SPLITK>;
    // setmaxnreg.inc waits until the registers it asks for are free in the
    // CTA's launch pool; a pool smaller than the split would never satisfy
    // it, so refuse to launch in that case.
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, kern);
    if (err != cudaSuccess) return err;
    if (fa.numRegs * kThreads < kCtrlRegs * 128 + kEpiRegs * 256 || fa.maxThreadsPerBlock < kThreads)
        return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int BN, bool GROUPED, bool PAIR, bool ROWB = false, bool SPLITK = false>
cudaError_t launch_one(const GemmLaunch& g) {
    using L = Layout<BN, GROUPED, PAIR, ROWB, PAIR && !GROUPED && !SPLITK>;
    auto kern = fp8_gemm_kernel<BN, GROUPED, PAIR, ROWB, SPLITK>;
    const int smem = L::smem_bytes(GROUPED ? g.args.E : 0);
    cudaError_t err = prepare<BN, GROUPED, PAIR, ROWB, SPLITK>(smem);
    if (err != cudaSuccess) return err;
    if constexpr (!PAIR) {
        kern<<<g.grid, kThreads, smem, g.stream>>>(*g.tmA, *g.tmB, *g.tmC, g.args);
        return cudaGetLastError();
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(g.grid, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = g.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, *g.tmA, *g.tmB, *g.tmC, g.args);
    }
}

template <int BN, bool ROWB>
int pair_max_clusters() {
    using L = Layout<BN, false, true, ROWB, true>;
    const int smem = L::smem_bytes(0);
    if (prepare<BN, false, true, ROWB>(smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_kernel<BN, false, true, ROWB, false>, &cfg) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace
}  // namespace fp8q
