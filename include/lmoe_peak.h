/*
 * lmoe_peak — tensor-pipe throughput of the current GPU, measured with the
 * tcgen05 MMA forms the lmoe layer's kernels issue (and the packed-FP4
 * forms), for the tensor-bound rooflines of its benchmark.  The pages
 * measure no tensor rate of their own; this is the denominator the layer's
 * FLOP/s are divided by.
 *
 * One CTA per SM issues M = 128, N = 256 MMAs back to back on operands held
 * in shared memory (finite random values, unit block scales), accumulating
 * in tensor memory; nothing is loaded inside the loop.
 */
#ifndef LMOE_PEAK_H
#define LMOE_PEAK_H

#include "lmoe.h"

#ifdef __cplusplus
extern "C" {
#endif

enum {
  LMOE_TC_BF16 = 0,        /* kind::f16, bf16 x bf16, K = 16 per MMA */
  LMOE_TC_E4M3_E4M3 = 1,   /* kind::mxf8f6f4 block-scaled (UE8M0 per 32), E4M3 x E4M3, K = 32 */
  LMOE_TC_E2M1_E4M3 = 2,   /* kind::mxf8f6f4 block-scaled, E2M1 weights x E4M3: the MXFP4 expert GEMMs' form */
  LMOE_TC_MXFP4 = 3,       /* kind::mxf4, packed E2M1 x E2M1, UE8M0 per 32 (scale_vec::2X), K = 64 */
  LMOE_TC_NVFP4 = 4        /* kind::mxf4nvf4, packed E2M1 x E2M1, UE4M3 per 16 (scale_vec::4X), K = 64 */
};

/* Run the loop of `kind` for `iters` iterations of four MMAs per SM on
 * `stream` and synchronise; *ms = its CUDA-event time, *flops = the FLOPs it
 * executed (2 M N K per MMA).  1 <= iters <= 2^20.  Allocates one int of
 * device memory for the bounded-wait flag.  Errors: INVALID_ARG (NULL
 * outputs, bad kind or iters), UNSUPPORTED (not an sm_103 GPU), OOM, CUDA,
 * TIMEOUT (the completion wait gave up). */
LMOE_API lmoe_status lmoe_tc_peak(int kind, int iters, float* ms, double* flops, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* LMOE_PEAK_H */
