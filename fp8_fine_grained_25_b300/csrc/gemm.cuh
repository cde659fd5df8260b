// Internal interface between the C-ABI layer and the GEMM kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8q {

constexpr int kMaxExperts = 1024;

struct GemmArgs {
    const float* sa;         // [M, KB]
    const float* sb;         // [NB, KB], or [E][NB][KB] when grouped, or [N, KB] (row_scaled_b)
    __nv_bfloat16* C;        // [M, N] (written directly by the grouped epilogue)
    const int32_t* offsets;  // [E + 1], grouped only (device memory)
    int32_t M, N, K;         // M = total rows of A and C
    int32_t KB, NB;          // ceil(K / 128), ceil(N / 128)
    int32_t E;               // experts (grouped), else 1
    int32_t mt_count, nt_count;
    int32_t mp_count;        // pair mode: ceil(mt_count / 2) row units
    int32_t num_tiles;       // dense only (tile units x splits); the grouped kernel counts its own
    // Split K (dense block-scaled GEMM only): each tile's K blocks are cut
    // into `splits` ranges (multiples of 4 K blocks) computed by different
    // work units; every unit writes its FP32 partial tile to ws, and the last
    // unit of a tile to arrive sums the partials in split order and stores C.
    int32_t splits;          // 1: no split
    int32_t tile_units;      // work units per split (num_tiles = tile_units * splits)
    float* ws;               // splits > 1: FP32 partial tiles [splits][M][N]
    uint32_t* counters;      // splits > 1: one arrival word per 128-row x BN tile
    uint32_t epoch;          // splits > 1: this call's tag in the arrival words (1 .. 2^24 - 1)
    uint64_t timeout_ns;
    uint32_t debug;          // FP8Q_INJECT_STALLED_STAGE: first pipeline stage never completes
};

struct GemmLaunch {
    const CUtensorMap* tmA;
    const CUtensorMap* tmB;
    const CUtensorMap* tmC;
    GemmArgs args;
    int bn;                  // 128, 160 (pair tiles), 224 (both: dense, block-scaled B) or 256
    bool grouped;
    bool pair;               // 2-CTA clusters with the 2-CTA MMA (dense only)
    bool row_scaled_b;       // sb holds one scale per row of B (dense only)
    unsigned grid;           // CTAs (a multiple of 2 in pair mode)
    cudaStream_t stream;
};

cudaError_t launch_gemm(const GemmLaunch& g);
// Columns of the TMA-store box of C the kernel writes through (the tensor
// map's box width: 64 with a 128-byte swizzle, 32 with a 64-byte swizzle, or
// 16 with a 32-byte swizzle), for one-CTA or pair tiles.
int gemm_c_box_cols(int bn, bool pair);
// Pair mode: how many 2-CTA clusters of the dense kernel fit on the device
// at once (0 if none or on error).
int gemm_pair_max_clusters(int bn, bool row_scaled_b);
cudaError_t read_device_status(cudaStream_t stream, uint32_t* out, bool clear);

// gemm_pair.cu: the pair tiles of the block-scaled dense GEMM (launch, the
// co-resident cluster count, and that unit's device status word, read after
// the caller's stream synchronisation).
cudaError_t launch_gemm_dense_pair(const GemmLaunch& g);
int gemm_dense_pair_max_clusters(int bn);
cudaError_t read_dense_pair_status(uint32_t* out, bool clear);

// The GEMM with UE8M0 block scales applied by the tensor core (gemm_bs.cu):
// output tiles of 128 x gemm_bs_tile_n() per CTA; tmB's box is that many
// rows, or half of them in pair mode (2-CTA clusters, 256-row tiles).
int gemm_bs_tile_n();
// row_scaled_b: sb holds one UE8M0 byte per row of B ([N][KB]) instead of
// one per 128-row block
int gemm_bs_pair_max_clusters(bool row_scaled_b);
cudaError_t launch_gemm_bs(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC,
                           const uint8_t* sa, const uint8_t* sb, int32_t M, int32_t N, int32_t K,
                           bool row_scaled_b, bool pair, int pair_clusters, uint64_t timeout_ns,
                           uint32_t debug, int num_sms, cudaStream_t stream);
cudaError_t read_bs_status(uint32_t* out, bool clear);

}  // namespace fp8q
