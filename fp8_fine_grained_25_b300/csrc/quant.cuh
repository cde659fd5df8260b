// Internal interface between the C-ABI layer and the quantizer kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8q {

// s: fp32 scales, or UE8M0 scale bytes when pow2
cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, void* q, void* s, bool pow2,
                             cudaStream_t stream, int num_sms, uint64_t timeout_ns);
// tmW: bf16 [N, K] tensor map, box 128 x 128, no swizzle
cudaError_t launch_quant_weight(const CUtensorMap* tmW, void* q, void* s, bool pow2, int64_t N,
                                int64_t K, cudaStream_t stream, int num_sms, uint64_t timeout_ns);
// w: bf16 [N, K] (N % 16 == 0, K % 16 == 0); writes qt [K, N] and st
// [KB, NB], and q [N, K] and s [NB, KB] unless q is null; scales fp32, or
// UE8M0 bytes when pow2
cudaError_t launch_quant_weight_t(const void* w, void* q, void* s, void* qt, void* st, bool pow2, int64_t N,
                                  int64_t K, cudaStream_t stream, int num_sms);
// x: bf16 [M, K] (M % 16 == 0, K % 16 == 0); 128x1 tiles, codes written
// transposed [K, M], scales [K, ceil(M/128)]
cudaError_t launch_quant_act_t(const void* x, void* qt, void* st, bool pow2, int64_t M, int64_t K,
                               cudaStream_t stream, int num_sms);
cudaError_t launch_gather_rows(const void* q_src, const float* s_src, int64_t T, int64_t K,
                               const int32_t* index, int64_t R, void* q_dst, float* s_dst,
                               cudaStream_t stream, int num_sms);
cudaError_t read_quant_status(uint32_t* out, bool clear);

}  // namespace fp8q
