// The pair tiles of the block-scaled dense GEMM (2-CTA clusters, tile widths
// 128, 160, 224 and 256; no split K) in a translation unit of their own, so that
// they can be compiled apart from the other forms of the kernel: the build
// passes ptxas -O1 here, under which these kernels run ~3 % faster on the
// B300 (dense 8192 x 7168 x 7168: 307 against 318 us) while the
// weight-gradient form loses ~2 % and stays at the default level.
#include "gemm_kernel.cuh"

namespace fp8q {

cudaError_t launch_gemm_dense_pair(const GemmLaunch& g) {
    switch (g.bn) {
        case 128: return launch_one<128, false, true>(g);
        case 160: return launch_one<160, false, true>(g);
        case 224: return launch_one<224, false, true>(g);
        case 256: return launch_one<256, false, true>(g);
    }
    return cudaErrorInvalidValue;
}

int gemm_dense_pair_max_clusters(int bn) {
    switch (bn) {
        case 128: return pair_max_clusters<128, false>();
        case 160: return pair_max_clusters<160, false>();
        case 224: return pair_max_clusters<224, false>();
        case 256: return pair_max_clusters<256, false>();
        default: return 0;
    }
}

cudaError_t read_dense_pair_status(uint32_t* out, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(out, g_device_status, sizeof(uint32_t));
    if (err != cudaSuccess || !clear) return err;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(uint32_t));
}

}  // namespace fp8q
