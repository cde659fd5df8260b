// Host side of the block-scaled FP8 GEMM (the kernel is in
// gemm_kernel.cuh): tile-shape queries, the launch of every form of the
// kernel except the pair tiles of the block-scaled dense GEMM (gemm_pair.cu,
// a translation unit of their own), and the device status word.
#include "gemm_kernel.cuh"

namespace fp8q {

int gemm_c_box_cols(int bn, bool pair) {
    switch (bn) {
        case 128: return pair ? Layout<128, false, true>::EPI_BOX_COLS : Layout<128, false, false>::EPI_BOX_COLS;
        case 160: return pair ? Layout<160, false, true>::EPI_BOX_COLS : 0;  // pair tiles only
        case 224: return pair ? Layout<224, false, true>::EPI_BOX_COLS : Layout<224, false, false>::EPI_BOX_COLS;
        case 256: return pair ? Layout<256, false, true>::EPI_BOX_COLS : Layout<256, false, false>::EPI_BOX_COLS;
        default: return 0;
    }
}

int gemm_pair_max_clusters(int bn, bool row_scaled_b) {
    if (!row_scaled_b) return gemm_dense_pair_max_clusters(bn);
    switch (bn) {
        case 128: return pair_max_clusters<128, true>();
        case 256: return pair_max_clusters<256, true>();
        default: return 0;
    }
}

cudaError_t launch_gemm(const GemmLaunch& g) {
    if (g.grouped) {
        if (g.row_scaled_b) return cudaErrorInvalidValue;
        switch (g.bn) {
            case 128: return launch_one<128, true, false>(g);
            case 256: return launch_one<256, true, false>(g);
        }
    } else if (g.row_scaled_b) {
        if (g.pair) {
            switch (g.bn) {
                case 128: return launch_one<128, false, true, true>(g);
                case 256: return launch_one<256, false, true, true>(g);
            }
            return cudaErrorInvalidValue;
        }
        switch (g.bn) {
            case 128: return launch_one<128, false, false, true>(g);
            case 256: return launch_one<256, false, false, true>(g);
        }
    } else if (g.args.splits > 1) {
        // split K: the same tile widths with the partial-tile epilogue
        if (g.pair) {
            switch (g.bn) {
                case 128: return launch_one<128, false, true, false, true>(g);
                case 224: return launch_one<224, false, true, false, true>(g);
                case 256: return launch_one<256, false, true, false, true>(g);
            }
        } else {
            switch (g.bn) {
                case 128: return launch_one<128, false, false, false, true>(g);
                case 224: return launch_one<224, false, false, false, true>(g);
                case 256: return launch_one<256, false, false, false, true>(g);
            }
        }
    } else if (g.pair) {
        return launch_gemm_dense_pair(g);
    } else {
        switch (g.bn) {
            case 128: return launch_one<128, false, false>(g);
            case 224: return launch_one<224, false, false>(g);
            case 256: return launch_one<256, false, false>(g);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t read_device_status(cudaStream_t stream, uint32_t* out, bool clear) {
    cudaError_t err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return err;
    uint32_t mine = 0, pair = 0;
    err = cudaMemcpyFromSymbol(&mine, g_device_status, sizeof(uint32_t));
    if (err != cudaSuccess) return err;
    err = read_dense_pair_status(&pair, clear);
    if (err != cudaSuccess) return err;
    *out = mine | pair;
    if (!clear) return cudaSuccess;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(uint32_t));
}

}  // namespace fp8q
