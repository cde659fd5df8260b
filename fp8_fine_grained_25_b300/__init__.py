"""Fine-grained FP8 quantization (1x128 activation tiles, 128x128 weight
blocks) and the block-scaled FP8 GEMM with FP32 promotion, dense and
grouped per expert, as hand-written sm_103a CUDA behind a C ABI.

    from fp8_fine_grained_25_b300 import fp8q      # the binding (needs libfp8q.so)
    from fp8_fine_grained_25_b300 import workloads # seeded synthetic inputs

The binding is imported on demand so that the input generators and the
build step work on machines without the library or a GPU.
"""

__all__ = ["fp8q", "workloads", "build"]
