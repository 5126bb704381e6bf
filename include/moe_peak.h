/* Measurement support of the fused MoE expert FFN library: the dense tensor-core rate of each
 * tcgen05 instruction kind the GEMM stages issue, measured on the GPU the library runs on.
 *
 * The pages have no counterpart of this call. The roofline fractions of the GEMM stages divide
 * their algorithmic flops by a peak; this probe gives that peak for the exact instruction kind
 * and operand types a stage uses (kind::f16 with bf16 or f16 operands, kind::mxf8f6f4.block_scale
 * with e4m3 x e2m1 or e4m3 x e4m3 operands), which no library GEMM measures.
 */
#ifndef MOE_PEAK_H
#define MOE_PEAK_H

#include "moe_ffn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_PEAK_BF16 = 0,        /* tcgen05.mma kind::f16, bf16 x bf16, fp32 accumulation (A16W16 GEMMs) */
    MOE_PEAK_F16 = 1,         /* kind::f16, f16 x f16 (the integer modes' exact f16 GEMMs)            */
    MOE_PEAK_E4M3_E2M1 = 2,   /* kind::mxf8f6f4.block_scale, e4m3 x e2m1, UE8M0 per 32 (FP8 x FP4)     */
    MOE_PEAK_E4M3_E4M3 = 3    /* kind::mxf8f6f4.block_scale, e4m3 x e4m3, UE8M0 per 32 (A8W8-FP8)      */
} moe_peak_kind;

/* Launches `grid` CTAs (grid <= 0: one per SM), each issuing iters_per_cta x 4 dense MMAs of
 * M = 128, N = 256 (K = 16 for kind::f16, 32 for kind::mxf8f6f4) from one thread, back to back, on
 * operand tiles that stay in its shared memory (finite pseudo-random values, no global memory
 * traffic) into a tensor-memory accumulator. Time the call with events on `stream`; the dense rate
 * is *flops_out / time.
 *   kind       a moe_peak_kind (else MOE_ERR_INVALID_ARG).
 *   iters_per_cta  >= 1 (else MOE_ERR_INVALID_ARG); about 2.7 us of MMA work per 10 iterations on
 *              one SM at 1.9 GHz, so 10^4 gives a launch of a few milliseconds.
 *   flops_out  host pointer: 2 * M * N * K * MMAs, all CTAs (required).
 *   workspace  device memory of at least 256 bytes, 256-byte aligned (its error word records
 *              MOE_ERR_TIMEOUT if the one bounded wait, for the last MMAs, ran out; read it with
 *              moe_check_device_error). Bytes [128, 144) receive two int64: the SM clock cycles
 *              and the nanoseconds (%globaltimer) of CTA 0 from its first MMA issue to the
 *              completion of its last, i.e. the SM clock during the probe. Nothing else in it is
 *              touched.
 * Asynchronous on `stream`; allocates nothing. */
MOE_API moe_status moe_tensor_peak_probe(moe_peak_kind kind, int64_t iters_per_cta, int grid, double* flops_out,
                                         void* workspace, size_t workspace_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PEAK_H */
