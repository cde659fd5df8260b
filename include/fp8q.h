/*
 * fp8q: fine-grained FP8 quantization and block-scaled FP8 GEMM for B300
 * (sm_103a), behind a plain C ABI.
 *
 * What the method computes (extracted web pages on DeepSeek-V3 training):
 *  - news.qq.com/rain/a/20241229A05OQF00, section "FP8 低精度训练",
 *    item "细粒度量化" (Fig. 7a): activations get one scale per 1x128 tile
 *    (per token, per 128 channels), weights one scale per 128x128 block.
 *  - same section, item "提高累加精度" (Fig. 7b): the FP8 MMA partial results
 *    are promoted into FP32 registers, which is where the fine-grained
 *    scales are applied.
 *  - developer.aliyun.com/article/1776647 §4.1 and m.jxzklqfsx.com/aigc/3586
 *    §三(二): block-wise quantization plus high-precision accumulation.
 * The pages name neither the FP8 encoding nor the scale formula. This
 * library uses E4M3 (OCP E4M3FN, max 448), scale = fl32(amax / 448), codes
 * q = E4M3_round_nearest_even_saturating(fl32(x / scale)), and an all-zero
 * tile gets scale 0 and all-zero codes.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers on the current CUDA device, owned by the
 *    caller, and must be 16-byte aligned. The library allocates no device
 *    memory and keeps no reference to a pointer after the call returns.
 *  - Matrices are dense and row-major with unit inner stride. FP8 codes are
 *    one byte each (E4M3 bit patterns); bf16 values are raw 16-bit patterns.
 *  - K must be a multiple of 16 (the FP8 row pitch must be a multiple of 16
 *    bytes) and N a multiple of 8 (the bf16 output row pitch likewise);
 *    otherwise the call returns FP8Q_ERR_ALIGN. M = 0 (or total_M = 0) is a
 *    no-op that returns FP8Q_OK. Sizes above 2^31 - 1 rows or columns give
 *    FP8Q_ERR_SHAPE.
 *  - Work is enqueued on `stream` and runs asynchronously. Argument checks
 *    happen before anything is enqueued; a failed check enqueues nothing.
 *    A launch failure returns FP8Q_ERR_CUDA.
 *  - Inputs must be finite; NaN or Inf input gives undefined codes.
 *  - Only sm_103 devices are supported (FP8Q_ERR_DEVICE otherwise).
 *  - Kernel-side failures (a pipeline wait that exceeds its time limit, or
 *    malformed expert offsets) set a device status word that
 *    fp8q_get_device_status() reads; the kernel then returns early.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

#if !defined(__DRIVER_TYPES_H__)
typedef struct CUstream_st* cudaStream_t; /* the CUDA runtime's stream handle */
#endif

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_NULL = 1,        /* a required pointer is NULL */
    FP8Q_ERR_SHAPE = 2,       /* a size is negative, zero where not allowed, or too large */
    FP8Q_ERR_ALIGN = 3,       /* K % 16 != 0, N % 8 != 0, or a pointer not 16-byte aligned */
    FP8Q_ERR_DEVICE = 4,      /* the current device is not sm_103 */
    FP8Q_ERR_CUDA = 5,        /* a CUDA runtime/driver call or a launch failed */
    FP8Q_ERR_TIMEOUT = 6,     /* device status: a pipeline wait exceeded its limit */
    FP8Q_ERR_UNSUPPORTED = 7, /* a valid request this build does not handle */
    FP8Q_ERR_OFFSETS = 8      /* device status: expert offsets malformed */
} fp8q_status;

/* Device status word bits (see fp8q_get_device_status). */
#define FP8Q_DEVSTATUS_TIMEOUT 0x1u
#define FP8Q_DEVSTATUS_BAD_OFFSETS 0x2u
#define FP8Q_DEVSTATUS_BAD_INDEX 0x4u

/*
 * Activation quantization, one scale per 1x128 tile (Fig. 7a, "1x128
 * tile-wise").
 *   x_bf16  in : bf16 [M, K]
 *   q_e4m3  out: uint8 E4M3 codes [M, K]
 *   scales  out: fp32 [M, ceil(K/128)]; scales[m][kb] = amax(|x[m, 128kb ..
 *                128kb+127]|) / 448, over the present columns when K % 128 != 0.
 * Codes and scales are bit-exact with the definition above.
 */
FP8Q_API int fp8q_quant_act(const void* x_bf16, int64_t M, int64_t K, void* q_e4m3, float* scales,
                   cudaStream_t stream);

/*
 * Weight quantization, one scale per 128x128 block (Fig. 7a, "128x128
 * block-wise"; aliyun §4.1 "块级量化（128×128 块）").
 *   w_bf16  in : bf16 [N, K]
 *   q_e4m3  out: uint8 E4M3 codes [N, K]
 *   scales  out: fp32 [ceil(N/128), ceil(K/128)]; the amax runs over the block's
 *                present rows and columns at the N and K tails.
 * A stack of E expert weights [E][N][K] with N % 128 == 0 is quantized in one
 * call as an [E*N, K] matrix; its scales come out as [E][N/128][ceil(K/128)].
 */
FP8Q_API int fp8q_quant_weight(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3, float* scales,
                      cudaStream_t stream);

/*
 * Power-of-two (UE8M0) scales: the same 1x128 / 128x128 tiles with each
 * scale rounded up to a power of two, the form that a tensor core with
 * hardware block scaling applies (8-bit exponent scale factors). The pages
 * do not describe this variant.
 *   scale byte = e + 127 with e = ceil(log2(amax / 448)) (the smallest power
 *   of two with amax / 2^e <= 448), clamped below at 0; the scale is
 *   2^(byte - 127). Codes q = E4M3_rn_satfinite(x / 2^e) (an exact quotient).
 *   An all-zero tile gets byte 0 and all-zero codes.
 *   fp8q_quant_act_ue8m0:    x [M, K] -> q [M, K], scales uint8 [M, ceil(K/128)]
 *   fp8q_quant_weight_ue8m0: w [N, K] -> q [N, K], scales uint8 [ceil(N/128), ceil(K/128)]
 * Same alignment and error rules as fp8q_quant_act / fp8q_quant_weight,
 * except that the byte scales need no alignment.
 */
FP8Q_API int fp8q_quant_act_ue8m0(const void* x_bf16, int64_t M, int64_t K, void* q_e4m3,
                                  uint8_t* scales, cudaStream_t stream);
FP8Q_API int fp8q_quant_weight_ue8m0(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3,
                                     uint8_t* scales, cudaStream_t stream);

/*
 * Activation quantization for the weight gradient: 128x1 tiles (128
 * consecutive rows of one column, i.e. 1x128 tiles along the token axis of
 * x^T), written transposed so that the tokens become the contraction axis
 * of fp8_wgrad_gemm. The tiling follows Fig. 7a's activation granularity
 * with the roles of the axes swapped, the layout the backward pass needs.
 *   x_bf16  in : bf16 [M, K] (M tokens)
 *   qt_e4m3 out: uint8 E4M3 codes [K, M]; qt[k][m] encodes x[m][k]
 *   st      out: fp32 [K, ceil(M/128)]; st[k][mb] = amax(|x[128mb .. 128mb+127][k]|)
 *                / 448, over the present rows when M % 128 != 0.
 * Codes and scales are bit-exact with quantizing x^T by fp8q_quant_act.
 * M % 16 == 0 (the row pitch of qt) and K % 16 == 0, else FP8Q_ERR_ALIGN.
 */
FP8Q_API int fp8q_quant_act_t(const void* x_bf16, int64_t M, int64_t K, void* qt_e4m3, float* st,
                              cudaStream_t stream);

/*
 * Weight quantization in 128x128 blocks with the codes also written in the
 * transposed layout, for the input gradient of the backward pass: dX = dY W
 * is fp8_block_gemm(quant_act(dY), qt) because a 128x128 block's scale is
 * the same for the block transposed.
 *   w_bf16  in : bf16 [N, K]
 *   q_e4m3, scales out: as fp8q_quant_weight, or both NULL to skip them
 *   qt_e4m3 out: uint8 E4M3 codes [K, N]; qt[k][n] = q[n][k]
 *   st      out: fp32 [ceil(K/128), ceil(N/128)]; st[kb][nb] = scales[nb][kb]
 * One pass over w writes both layouts. N % 16 == 0 (the row pitch of qt) and
 * K % 16 == 0, else FP8Q_ERR_ALIGN; passing only one of q_e4m3 and scales
 * gives FP8Q_ERR_NULL.
 */
FP8Q_API int fp8q_quant_weight_t(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3,
                                 float* scales, void* qt_e4m3, float* st, cudaStream_t stream);

/*
 * Row gather of quantized activations: the MoE dispatch in FP8 (news.qq.com
 * page, "FP8 低精度训练", item "低精度存储和通信", Fig. 10: activations are
 * stored and communicated in FP8). Quantizing the T tokens once and then
 * moving codes and scales into expert order gives exactly the codes and
 * scales of quantizing the gathered bf16 rows, because the 1x128 tiles are
 * row-local.
 *   q_src  in : E4M3 codes [T, K]        s_src in : fp32 [T, ceil(K/128)]
 *   index  in : DEVICE int32 [R]; output row r is source row index[r]
 *               (repeats allowed)
 *   q_dst  out: E4M3 codes [R, K]        s_dst out: fp32 [R, ceil(K/128)]
 * K % 16 == 0; q pointers 16-byte aligned, s and index 4-byte aligned.
 * An index outside [0, T) gives a zero row and sets
 * FP8Q_DEVSTATUS_BAD_INDEX in the device status word. R = 0 is a no-op.
 */
FP8Q_API int fp8q_gather_rows(const void* q_src, const float* s_src, int64_t T, int64_t K,
                              const int32_t* index, int64_t R, void* q_dst, float* s_dst,
                              cudaStream_t stream);

/*
 * Block-scaled FP8 GEMM, C = A * B^T (Fig. 7b: FP8 MMA per 128-wide K block,
 * promoted to FP32 with the fine-grained scales).
 *   A  in : E4M3 codes [M, K]        sa in: fp32 [M, ceil(K/128)]
 *   B  in : E4M3 codes [N, K]        sb in: fp32 [ceil(N/128), ceil(K/128)]
 *   C  out: bf16 [M, N]
 *   C[m][n] = bf16_rn( sum_kb  P_kb[m][n] * (sa[m][kb] * sb[n/128][kb]) ),
 *   P_kb = sum over k in block kb of dec(A[m][k]) * dec(B[n][k]), taken on the
 *   tensor cores with FP32 accumulation; the sum over kb runs in FP32.
 * Accuracy: |C - exact-definition-in-FP32| <= 1 bf16 ulp + 1e-5 * sum_k|a_k b_k|.
 */
FP8Q_API int fp8_block_gemm(const void* A, const float* sa, const void* B, const float* sb, void* C_bf16,
                   int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * fp8_block_gemm with split K, for shapes whose output tiles fill few waves
 * of the 148 SMs (the MLA down-projections of the news.qq.com page's
 * "Multi-head Latent Attention" section: N = 1536 and 576 at M = 4096).
 * The K blocks of each output tile are cut into S ranges (multiples of 4
 * K blocks) computed by different work units; each unit writes its FP32
 * partial tile into the workspace, and the last unit of a tile to finish
 * adds the S partials in range order and stores C. The result does not
 * depend on which unit finishes last, and differs from fp8_block_gemm only
 * by the order of the FP32 additions (within the same accuracy bound).
 *   workspace      in/out: DEVICE memory owned by the caller, 256-byte
 *                  aligned, of workspace_bytes bytes; it needs no
 *                  initialisation and keeps no state a later call relies on
 *                  (arrival words are tagged with a per-call number).
 *   workspace_bytes: the library uses the S it would pick for the shape (or
 *                  the one set by fp8q_set_gemm_splits), reduced until
 *                  S x M x N x 4 bytes of partials plus one 4-byte word per
 *                  128 x tile-width output tile fit; S = 1 (no workspace
 *                  used) is plain fp8_block_gemm. workspace may be NULL
 *                  (then S = 1).
 * Calls that share a workspace must not run concurrently (e.g. on two
 * streams). Other arguments, alignment rules and errors as fp8_block_gemm;
 * FP8Q_ERR_ALIGN also for a workspace not 256-byte aligned.
 */
FP8Q_API int fp8_block_gemm_ws(const void* A, const float* sa, const void* B, const float* sb,
                               void* C_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/*
 * fp8_block_gemm_ws for callers that cannot allocate device memory. There is
 * no counterpart of this call on the pages; it exists for code that may not
 * call cudaMalloc where it issues the GEMM (cudaMalloc can synchronise the
 * device), or that receives only its input and output buffers from a host
 * framework. It runs the same split-K kernel, with its scratch in a fixed
 * array inside the library's device image instead of a caller workspace:
 *   - every GPU that loads the library holds FP8Q_STATIC_SCRATCH_BYTES
 *     (32 MiB) of device memory for that array until the process exits;
 *   - the call allocates nothing and frees nothing;
 *   - a call whose split count (chosen per shape, or set with
 *     fp8q_set_gemm_splits) needs more scratch than the array holds
 *     (S x 128-row x tile-width FP32 partial tiles plus one 4-byte word per
 *     tile; see fp8_block_gemm_workspace_size) returns FP8Q_ERR_SHAPE and
 *     launches nothing; a shape that does not split runs as fp8_block_gemm;
 *   - all calls in the process share the array, and it keeps whatever the
 *     last call left in it. Nothing in it needs to start at zero (the
 *     arrival words carry a per-call tag), but calls that overlap on the
 *     GPU (two streams, or two host threads) race on it: serialise them;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before capturing the stream into a CUDA graph.
 * Arguments, layouts, alignment, accuracy and other errors as fp8_block_gemm.
 */
#define FP8Q_STATIC_SCRATCH_BYTES (32u << 20)
FP8Q_API int fp8_block_gemm_static(const void* A, const float* sa, const void* B, const float* sb,
                                   void* C_bf16, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * Bytes of workspace fp8_block_gemm_ws would use for an M x N x K call on
 * the current device with the current settings (0: it would not split K).
 * Returns FP8Q_OK, FP8Q_ERR_NULL, FP8Q_ERR_SHAPE or a device error.
 */
FP8Q_API int fp8_block_gemm_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);

/*
 * The block-scaled FP8 GEMM with power-of-two (UE8M0) scales from
 * fp8q_quant_act_ue8m0 / fp8q_quant_weight_ue8m0 (a variant the pages do not
 * describe). The tensor core applies the scales itself (block-scaled MMA,
 * one scale per row of A / column of B per 32-wide K slice) and accumulates
 * the whole K range in FP32, so there is no promotion through registers.
 *   A  in : E4M3 codes [M, K]     sa in: UE8M0 bytes [M, ceil(K/128)]
 *   B  in : E4M3 codes [N, K]     sb in: UE8M0 bytes [ceil(N/128), ceil(K/128)]
 *   C  out: bf16 [M, N] = bf16_rn( sum_k dec(A[m][k]) 2^(sa - 127) dec(B[n][k]) 2^(sb - 127) )
 * Accuracy: within 1 bf16 ulp + 1e-5 * sum_k |a_k b_k| of the block-wise FP32
 * definition (fp8_block_gemm with the scales 2^(byte - 127)). Alignment and
 * errors as fp8_block_gemm; the byte scales need no alignment.
 */
FP8Q_API int fp8_block_gemm_ue8m0(const void* A, const uint8_t* sa, const void* B, const uint8_t* sb,
                                  void* C_bf16, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * The UE8M0 forms of the backward pass (see fp8q_quant_act_t,
 * fp8q_quant_weight_t and fp8_wgrad_gemm for the layouts), with
 * power-of-two scales stored as UE8M0 bytes:
 *   fp8q_quant_act_t_ue8m0:    x [M, K] -> qt [K, M], st uint8 [K, ceil(M/128)]
 *   fp8q_quant_weight_t_ue8m0: w [N, K] -> q, scales (optional, uint8
 *                              [ceil(N/128), ceil(K/128)]), qt [K, N],
 *                              st uint8 [ceil(K/128), ceil(N/128)]
 *   fp8_wgrad_gemm_ue8m0:      C [M, N] = A [M, K] * B [N, K]^T with one
 *                              UE8M0 byte per row of A and of B per 128-wide
 *                              K block (sa [M][KB], sb [N][KB]), applied by
 *                              the tensor core.
 * Same alignment, error and accuracy rules as the FP32-scale forms, except
 * that the byte scales need no alignment.
 */
FP8Q_API int fp8q_quant_act_t_ue8m0(const void* x_bf16, int64_t M, int64_t K, void* qt_e4m3,
                                    uint8_t* st, cudaStream_t stream);
FP8Q_API int fp8q_quant_weight_t_ue8m0(const void* w_bf16, int64_t N, int64_t K, void* q_e4m3,
                                       uint8_t* scales, void* qt_e4m3, uint8_t* st, cudaStream_t stream);
FP8Q_API int fp8_wgrad_gemm_ue8m0(const void* A, const uint8_t* sa, const void* B, const uint8_t* sb,
                                  void* C_bf16, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * Grouped (per-expert) block-scaled FP8 GEMM for the MoE FFN (news.qq.com
 * page, "DeepSeekMoE 架构": 256 routed experts, 8 per token). Rows of A are
 * grouped by expert: rows [off[e], off[e+1]) use expert e's weights.
 *   A   in : E4M3 codes [total_M, K]      sa in: fp32 [total_M, ceil(K/128)]
 *   B   in : E4M3 codes [E][N][K]         sb in: fp32 [E][ceil(N/128)][ceil(K/128)]
 *   C   out: bf16 [total_M, N]; row m = A[m] * B_e^T for its expert e
 *   expert_offsets in: DEVICE int32 [E+1], off[0] = 0, nondecreasing,
 *                      off[E] = total_M (empty experts allowed)
 *   E: 1 .. 1024; total_M: passed from the host (= off[E]).
 * The host never reads the offsets. Malformed offsets (decreasing, off[0] != 0
 * or off[E] != total_M) are detected on the device: nothing is written to C
 * and the device status word gets FP8Q_DEVSTATUS_BAD_OFFSETS.
 */
FP8Q_API int fp8_grouped_gemm(const void* A, const float* sa, const void* B, const float* sb,
                     void* C_bf16, const int32_t* expert_offsets, int32_t E, int64_t total_M,
                     int64_t N, int64_t K, cudaStream_t stream);

/*
 * The weight-gradient GEMM of the backward pass (news.qq.com page: the
 * pipeline figure's "backward for weights" chunks, and Fig. 7, where the
 * linear layers' GEMMs run in FP8). dW = dY^T X contracts over tokens, so
 * both operands are activations quantized in 1x128 tiles along the token
 * axis (fp8q_quant_act_t), and the call is C = A * B^T with one scale per
 * row of B as well as of A:
 *   A  in : E4M3 codes [M, K] (dY^T)     sa in: fp32 [M, ceil(K/128)]
 *   B  in : E4M3 codes [N, K] (X^T)      sb in: fp32 [N, ceil(K/128)]
 *   C  out: bf16 [M, N] (dW)
 *   C[m][n] = bf16_rn( sum_kb  P_kb[m][n] * (sa[m][kb] * sb[n][kb]) ),
 * with P_kb and the FP32 promotion as in fp8_block_gemm (K is the number of
 * tokens here). Same alignment rules, errors and accuracy as fp8_block_gemm.
 * The pages do not fix the weight gradient's output type; like the forward
 * GEMM it is written in bf16.
 */
FP8Q_API int fp8_wgrad_gemm(const void* A, const float* sa, const void* B, const float* sb,
                            void* C_bf16, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * Synchronizes `stream`, then reads the device status word (an OR of
 * FP8Q_DEVSTATUS_* bits set by kernels since the last clear) of the current
 * device into *status_out, and clears it when `clear` is nonzero.
 * Returns FP8Q_OK, FP8Q_ERR_NULL or FP8Q_ERR_CUDA.
 */
FP8Q_API int fp8q_get_device_status(cudaStream_t stream, uint32_t* status_out, int clear);

/*
 * The fp8q_set_* calls below change process-wide settings that later calls
 * read when they launch; they are meant for tests and tuning, are not
 * synchronised with calls made concurrently from other host threads, and do
 * not affect work already enqueued.
 *
 * Time limit for every pipeline wait inside the GEMM kernels, in
 * nanoseconds (default 1e9). A wait that exceeds it sets
 * FP8Q_DEVSTATUS_TIMEOUT, and the kernel drains its in-flight copies,
 * frees its tensor memory and returns. 0 restores the default.
 */
FP8Q_API void fp8q_set_wait_timeout_ns(uint64_t ns);

/*
 * Output-tile width of fp8_block_gemm and fp8_wgrad_gemm: 128, 160, 224 or
 * 256 columns, or 0 (the default) to let the library pick per shape. 160 and
 * 224 apply to fp8_block_gemm only (fp8_wgrad_gemm then runs 256 wide); 160
 * applies to 2-CTA pair tiles only (M > 128) and is never split over K (a
 * call that cannot use it runs at the width the library picks). Affects
 * speed only, never results. Returns FP8Q_ERR_UNSUPPORTED for other values.
 */
FP8Q_API int fp8q_set_gemm_tile_n(int bn);

/*
 * Number of K ranges fp8_block_gemm_ws splits each output tile into: 1 .. 8,
 * or 0 (the default) to let the library pick per shape (still capped by the
 * workspace and by one range per 4 K blocks). Affects speed and the order
 * of FP32 additions only. Returns FP8Q_ERR_UNSUPPORTED for other values.
 */
FP8Q_API int fp8q_set_gemm_splits(int splits);

/*
 * Whether fp8_block_gemm, fp8_wgrad_gemm and fp8_block_gemm_ue8m0 may run an output tile of
 * 256 rows on a pair of SMs (2-CTA clusters with the 2-CTA tensor-core MMA,
 * each SM holding half of the B tile). 1 (the default) uses pairs whenever
 * M > 128, for both tile widths; 0 keeps one SM per 128 x N tile. Affects
 * speed only, never results. Returns FP8Q_OK.
 */
FP8Q_API int fp8q_set_gemm_pairs(int enable);

/*
 * Failure injection for tests of the device-side failure path. With
 * FP8Q_INJECT_STALLED_STAGE set, every fp8_block_gemm / fp8_wgrad_gemm /
 * fp8_block_gemm_ue8m0 / fp8_grouped_gemm launch announces 16 more bytes for its first pipeline stage than the
 * stage receives, so that stage never completes: the kernel's bounded waits
 * expire (see fp8q_set_wait_timeout_ns), it drains its copies, frees its
 * tensor memory, writes nothing further, returns, and the device status word
 * gets FP8Q_DEVSTATUS_TIMEOUT. The CUDA context stays usable. 0 (the
 * default) turns injection off. Returns FP8Q_OK.
 */
#define FP8Q_INJECT_STALLED_STAGE 0x1u
FP8Q_API int fp8q_set_fault_injection(uint32_t flags);

/* A short English description of a status code. Never NULL. */
FP8Q_API const char* fp8q_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
