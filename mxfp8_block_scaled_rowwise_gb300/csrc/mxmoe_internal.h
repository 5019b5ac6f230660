// mxmoe_internal.h -- launchers shared between the kernel files and the C-ABI
// layer (api.cu).  Arguments are validated by api.cu before these are called.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mxmoe.h"

namespace mx {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// dtype: MX_DTYPE_BF16 / MX_DTYPE_F32; rule: MX_SCALE_FLOOR / MX_SCALE_RCEIL.
// src_row (nullable): quantize the gathered tensor whose row r is x row src_row[r] (x has src_rows rows);
// row_scale (nullable, bf16 gather with the floor rule only): row r is bf16(row_scale[r] * x row src_row[r])
int launch_quantize(const void* x, int dtype, int rule, const int32_t* src_row, const float* row_scale,
                    int64_t src_rows, int64_t rows,
                    int64_t cols, int mode, const int32_t* seg_off, const int32_t* seg_poff, int nseg, int64_t ld_col,
                    int64_t pbound, uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col, int* dev_err,
                    cudaStream_t stream);

size_t permute_workspace_bytes(int64_t T, int k, int E);
int launch_permute(const int32_t* ids, int64_t T, int k, int E, int32_t* counts, int32_t* off, int32_t* poff,
                   int32_t* src_row, int32_t* dst_of, const uint8_t* q_in, const uint8_t* sf_in, int64_t K,
                   uint8_t* q_out, uint8_t* sf_out, void* ws, int* dev_err, cudaStream_t stream);
int launch_gather_rows(const void* src, int64_t row_bytes, const int32_t* src_row, int64_t R, void* dst,
                       cudaStream_t stream);

// SwiGLU (+ its backward when bwd) fused with MXFP8 quantization of the result
int launch_swiglu_quantize(bool bwd, const void* a, const void* dh, int64_t R, int64_t I, int mode,
                           const int32_t* seg_off, const int32_t* seg_poff, int nseg, int64_t ld_col, int64_t pbound,
                           uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col, int* dev_err,
                           cudaStream_t stream);

int launch_combine_fwd(const void* Y, const float* gate, const int32_t* dst_of, int64_t T, int k, int64_t H,
                       int64_t R, void* out, int* dev_err, cudaStream_t stream);
int launch_combine_bwd(const void* dOut, const void* Y, const float* gate, const int32_t* dst_of, int64_t T, int k,
                       int64_t H, int64_t R, void* dY, float* dgate, float* gate_rows, int* dev_err,
                       cudaStream_t stream);

// Grouped GEMM problem in the one "NT" form all three passes reduce to:
//   out[tile rows][tile cols] = sum_k deq(A)[row][k] * deq(B)[col][k]
enum GemmKind { kGemmRows = 0, kGemmWgrad = 1 };

struct GemmProblem {
    int kind;                 // kGemmRows: fwd/dgrad (A rows grouped by expert); kGemmWgrad
    const uint8_t* A;         // codes, K-major
    const uint8_t* SFA;       // scales, tensor-core layout
    const uint8_t* B;
    const uint8_t* SFB;
    int64_t a_rows, a_cols;   // A viewed as [a_rows x a_cols] (a_cols = contraction extent of the view)
    int64_t b_rows, b_cols;
    int64_t b_row_step;       // expert e's B starts at row e * b_row_step ...
    int64_t b_col_step;       // ... and contraction column e * b_col_step
    int64_t n_out;            // output columns per expert (fwd/dgrad: N; wgrad: K)
    int64_t m_out;            // wgrad: output rows per expert (N)
    int64_t k_len;            // fwd/dgrad: contraction length
    const int32_t* off;
    const int32_t* poff;
    int E;
    void* out;                // bf16 [R x n_out] or fp32 [E x m_out x n_out]
    int* dev_err;
    // forward only: SwiGLU epilogue when swiglu_i = I > 0 (n_out = 2I; out = [gate | up] bf16),
    // h = silu(gate) * up quantized rowwise [R x I] and columnwise [I x h_ldcol] (expert segments)
    int64_t swiglu_i = 0;
    uint8_t* h_qrow = nullptr;
    uint8_t* h_sfrow = nullptr;
    uint8_t* h_qcol = nullptr;
    uint8_t* h_sfcol = nullptr;
    int h_sfrow_copies = 1;   // 4: the scale array in the four-copy layout
    int h_sfcol_copies = 1;
    int64_t h_ldcol = 0;
    int b_scales_x1 = 0;          // SFB in the one-copy layout (else the four-copy layout)
    int b_blocked = 0;            // B codes in 128 x 128 blocks of 16 KiB (else row-major)
    int ctas_per_mma = 0;         // 0 or 2: CTA pairs (cta_group::2); 1: single-CTA tiles
    uint64_t wait_limit_ns = 0;   // 0: the default limit of every pipeline wait
    int withhold_operands = 0;    // test only: no operand copies are issued (every wait runs out)
    int raster_group = 0;         // tile order inside an expert: groups of G M tiles, M fastest (0: G = all)
    int cluster_pairs = 0;        // CTA pairs per cluster sharing A by multicast (0: the default, 1 or 2)
};

int launch_grouped_gemm(const GemmProblem& pr, cudaStream_t stream);

}  // namespace mx
