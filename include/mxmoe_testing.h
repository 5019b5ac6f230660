/*
 * mxmoe_testing.h -- internal entry of libmxmoe.so for tests and A/B measurements only.
 * Nothing on the product path calls it, and the source pages have no counterpart: it
 * exposes choices that the public grouped-GEMM calls fix.
 *
 *  - ctas_per_mma: the tile shape.  2: CTA pairs on an SM pair computing 256 x 256 tiles with
 *    tcgen05.mma.cta_group::2; 1: one CTA per 128 x 256 tile (cta_group::1); 0: the public
 *    calls' choice (pairs, except for forward and dgrad calls whose experts average fewer than
 *    512 rows, which get single-CTA tiles).  Outputs are the same either way.
 *  - wait_limit_ns: the time limit of every pipeline wait inside the GEMM kernel (0: the
 *    default of 2 s).  A wait that runs out sets MX_DEVERR_TIMEOUT in *dev_err, every role
 *    of the kernel leaves, the tensor memory is freed, and the outputs are invalid.
 *  - withhold_operands: non-zero makes the producer issue no operand copies, so no stage of
 *    the pipeline ever fills and the consumer's bounded wait has to run out (a test of the
 *    failure detector that cannot hang the GPU: every wait is bounded by wait_limit_ns).
 *  - raster_group: the order of an expert's output tiles: groups of G M tiles, M fastest inside
 *    a group, the groups one after another.  0: the default of the public calls (one group of
 *    all the expert's M tiles); G in 1..64 (G = 1: N tiles fastest).  Outputs are the same for
 *    every order.
 *  - cluster_pairs: 2 = clusters sharing an operand by multicast: with CTA pairs, two pairs on
 *    the two N tiles of one M tile, each A half-tile read from L2 once for both pairs; with
 *    single-CTA tiles, two CTAs on two M tiles of one N tile, each half of the B tile read once
 *    for both.  1 or 0 = no such clusters (the public calls' choice).  Outputs are the same
 *    either way.
 *
 * mx_testing_grouped_gemm runs pass MX_TESTING_FWD / _DGRAD with the arguments of
 * grouped_gemm_mxfp8_fwd_ex / _dgrad_ex (ld_tok ignored) and MX_TESTING_WGRAD with those of
 * grouped_gemm_mxfp8_wgrad_ex (A = dYc, SFA = SFdYc, B = Xc, SFB = SFXc, N, K, ld_tok; R
 * ignored; out fp32).  opt may be NULL (the public call's behaviour).  Errors as the
 * public calls, plus MX_ERR_INVALID_ARG for an unknown pass or ctas_per_mma.
 */
#ifndef MXMOE_TESTING_H
#define MXMOE_TESTING_H

#include "mxmoe.h"

#ifdef __cplusplus
extern "C" {
#endif

enum { MX_TESTING_FWD = 0, MX_TESTING_DGRAD = 1, MX_TESTING_WGRAD = 2 };

typedef struct {
    int ctas_per_mma;
    uint64_t wait_limit_ns;
    int withhold_operands;
    int raster_group;
    int cluster_pairs;
} mx_testing_gemm_options;

MX_API int mx_testing_grouped_gemm(int pass, const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
                                   const uint8_t* SFB, const int32_t* off, const int32_t* poff, int E, int64_t R,
                                   int64_t N, int64_t K, int64_t ld_tok, void* out, int flags,
                                   const mx_testing_gemm_options* opt, int* dev_err, mx_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MXMOE_TESTING_H */
