// Internal interface between the C-ABI layer and the quantizer kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8q {

cudaError_t launch_quant_act(const void* x, int64_t M, int64_t K, void* q, float* s,
                             cudaStream_t stream, int num_sms);
cudaError_t launch_quant_weight(const void* w, int64_t N, int64_t K, void* q, float* s,
                                cudaStream_t stream, int num_sms);

}  // namespace fp8q
