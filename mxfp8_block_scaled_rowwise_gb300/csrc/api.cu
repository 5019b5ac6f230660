// api.cu -- the extern "C" boundary (declared in include/mxmoe.h): argument
// validation, status codes, and the mapping of forward / dgrad / wgrad onto the
// one grouped-GEMM kernel.  No allocation, no synchronization, no host reads of
// device memory happen here.
#include <cuda_runtime.h>

#include "mxmoe_internal.h"
#include "../../include/mxmoe_testing.h"

using mx::ceil_div;
using mx::round_up;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ROWWISE and/or COLWISE; an _X4 bit only together with its form
bool valid_mode(int mode) {
    if ((mode & ~(MX_ROWWISE | MX_COLWISE | MX_ROWWISE_X4 | MX_COLWISE_X4)) != 0) return false;
    if ((mode & (MX_ROWWISE | MX_COLWISE)) == 0) return false;
    if ((mode & MX_ROWWISE_X4) && !(mode & MX_ROWWISE)) return false;
    if ((mode & MX_COLWISE_X4) && !(mode & MX_COLWISE)) return false;
    return true;
}

// mxfp8_quantize(_ex): valid_mode plus the blocked-code bits, each only with its form; the
// blocked rowwise form takes whole 128-row blocks of an unsegmented input, the blocked
// columnwise form whole 128-column blocks (its positions are 128-aligned already)
bool valid_quantize_mode(int mode, int64_t rows, int64_t cols, int nseg) {
    const int base = mode & ~(MX_ROWWISE_BLK | MX_COLWISE_BLK);
    if (!valid_mode(base)) return false;
    if ((mode & MX_ROWWISE_BLK) && (!(mode & MX_ROWWISE) || nseg != 0 || rows % 128 != 0 || cols % 128 != 0))
        return false;
    if ((mode & MX_COLWISE_BLK) && (!(mode & MX_COLWISE) || cols % 128 != 0)) return false;
    return true;
}

inline int check_device() {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

// Per-call choices of the grouped GEMMs beyond their operands: the public flags (layout of
// the B-operand scales) and the internal options of mxmoe_testing.h.
struct GemmChoice {
    int flags = 0;
    int ctas_per_mma = 0;
    uint64_t wait_limit_ns = 0;
    int withhold_operands = 0;
    int raster_group = 0;
    int cluster_pairs = 0;
};

inline bool valid_gemm_flags(int flags) { return (flags & ~(MX_GEMM_B_SCALES_X1 | MX_GEMM_B_BLOCKED)) == 0; }

void apply_choice(mx::GemmProblem& pr, const GemmChoice& c) {
    pr.b_scales_x1 = (c.flags & MX_GEMM_B_SCALES_X1) ? 1 : 0;
    pr.b_blocked = (c.flags & MX_GEMM_B_BLOCKED) ? 1 : 0;
    pr.ctas_per_mma = c.ctas_per_mma;
    pr.wait_limit_ns = c.wait_limit_ns;
    pr.withhold_operands = c.withhold_operands;
    pr.raster_group = c.raster_group;
    pr.cluster_pairs = c.cluster_pairs;
}

int gemm_rows_common(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB, const int32_t* off,
                     const int32_t* poff, int E, int64_t R, int64_t N, int64_t K, void* C, int* dev_err,
                     mx_stream_t stream, bool dgrad, const GemmChoice& choice) {
    if (!valid_gemm_flags(choice.flags)) return MX_ERR_INVALID_ARG;
    if (!A || !SFA || !B || !SFB || !off || !poff || !C || !dev_err) return MX_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || R < 0 || N <= 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (N % 128 != 0 || K % 128 != 0) return MX_ERR_UNSUPPORTED;
    if (R >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) || N * E >= (int64_t(1) << 31))
        return MX_ERR_UNSUPPORTED;
    if (!aligned16(A) || !aligned16(SFA) || !aligned16(B) || !aligned16(SFB) || !aligned16(C))
        return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    if (R == 0) return MX_OK;
    mx::GemmProblem pr{};
    pr.kind = mx::kGemmRows;
    pr.A = A;
    pr.SFA = SFA;
    pr.B = B;
    pr.SFB = SFB;
    pr.a_rows = R;
    pr.a_cols = K;
    if (!dgrad) {
        pr.b_rows = static_cast<int64_t>(E) * N;   // B [E*N x K]
        pr.b_cols = K;
        pr.b_row_step = N;
        pr.b_col_step = 0;
    } else {
        pr.b_rows = N;                             // Wt [N x E*K]
        pr.b_cols = static_cast<int64_t>(E) * K;
        pr.b_row_step = 0;
        pr.b_col_step = K;
    }
    pr.n_out = N;
    pr.m_out = 0;
    pr.k_len = K;
    pr.off = off;
    pr.poff = poff;
    pr.E = E;
    pr.out = C;
    pr.dev_err = dev_err;
    apply_choice(pr, choice);
    return mx::launch_grouped_gemm(pr, reinterpret_cast<cudaStream_t>(stream));
}

int gemm_wgrad_common(const uint8_t* dYc, const uint8_t* SFdYc, const uint8_t* Xc, const uint8_t* SFXc,
                      const int32_t* off, const int32_t* poff, int E, int64_t N, int64_t K, int64_t ld_tok, float* dW,
                      int* dev_err, mx_stream_t stream, const GemmChoice& choice) {
    if (!valid_gemm_flags(choice.flags)) return MX_ERR_INVALID_ARG;
    if (!dYc || !SFdYc || !Xc || !SFXc || !off || !poff || !dW || !dev_err) return MX_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || N <= 0 || K <= 0 || ld_tok <= 0) return MX_ERR_INVALID_ARG;
    if (N % 128 != 0 || K % 128 != 0 || ld_tok % 128 != 0) return MX_ERR_UNSUPPORTED;
    if (ld_tok >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(E) * (N / 128) * ceil_div(K, 256) >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    if (!aligned16(dYc) || !aligned16(SFdYc) || !aligned16(Xc) || !aligned16(SFXc) || !aligned16(dW))
        return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    mx::GemmProblem pr{};
    pr.kind = mx::kGemmWgrad;
    pr.A = dYc;
    pr.SFA = SFdYc;
    pr.B = Xc;
    pr.SFB = SFXc;
    pr.a_rows = N;
    pr.a_cols = ld_tok;
    pr.b_rows = K;
    pr.b_cols = ld_tok;
    pr.b_row_step = 0;
    pr.b_col_step = 0;
    pr.n_out = K;
    pr.m_out = N;
    pr.k_len = 0;
    pr.off = off;
    pr.poff = poff;
    pr.E = E;
    pr.out = dW;
    pr.dev_err = dev_err;
    apply_choice(pr, choice);
    return mx::launch_grouped_gemm(pr, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

size_t mx_sf_bytes(int64_t rows, int64_t kb) {
    if (rows < 0 || kb < 0) return 0;
    return static_cast<size_t>(round_up(rows, 128) * round_up(kb, 4));
}

size_t mx_sf_bytes_x4(int64_t rows, int64_t kb) { return 4 * mx_sf_bytes(rows, kb); }

int64_t mx_padded_rows_bound(int64_t R, int64_t E) {
    if (R < 0 || E < 0) return 0;
    return round_up(R + 127 * E, 128);
}

int mxfp8_quantize_ex(const void* x, int dtype, int scale_rule, int64_t rows, int64_t cols, int mode,
                      const int32_t* seg_off, const int32_t* seg_poff, int nseg, int64_t ld_col, uint8_t* q_row,
                      uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col, int* dev_err, mx_stream_t stream) {
    if (dtype != MX_DTYPE_BF16 && dtype != MX_DTYPE_F32) return MX_ERR_INVALID_ARG;
    if (scale_rule != MX_SCALE_FLOOR && scale_rule != MX_SCALE_RCEIL) return MX_ERR_INVALID_ARG;
    if (rows < 0 || cols <= 0 || cols % 32 != 0) return MX_ERR_INVALID_ARG;
    if (!valid_quantize_mode(mode, rows, cols, nseg)) return MX_ERR_INVALID_ARG;
    if (rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    if (nseg < 0 || nseg > (1 << 20)) return MX_ERR_INVALID_ARG;
    if (nseg > 0 && (!seg_off || !seg_poff)) return MX_ERR_INVALID_ARG;
    if (rows > 0 && !x) return MX_ERR_INVALID_ARG;
    const bool row = (mode & MX_ROWWISE) != 0, col = (mode & MX_COLWISE) != 0;
    if ((row && (!q_row || !sf_row)) || (col && (!q_col || !sf_col))) return MX_ERR_INVALID_ARG;
    const int64_t pbound = nseg > 0 ? mx_padded_rows_bound(rows, nseg) : round_up(rows, 128);
    if (col && (ld_col < round_up(rows, 128) || ld_col % 128 != 0)) return MX_ERR_INVALID_ARG;
    if (!aligned16(x) || (row && (!aligned16(q_row) || !aligned16(sf_row))) ||
        (col && (!aligned16(q_col) || !aligned16(sf_col))))
        return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    if (pbound == 0) return MX_OK;
    return mx::launch_quantize(x, dtype, scale_rule, nullptr, nullptr, 0, rows, cols, mode, nseg > 0 ? seg_off : nullptr,
                               nseg > 0 ? seg_poff : nullptr, nseg, col ? ld_col : 0, pbound, q_row, sf_row, q_col,
                               sf_col, dev_err, reinterpret_cast<cudaStream_t>(stream));
}

int mxfp8_quantize(const void* x, int64_t rows, int64_t cols, int mode, const int32_t* seg_off,
                   const int32_t* seg_poff, int nseg, int64_t ld_col, uint8_t* q_row, uint8_t* sf_row,
                   uint8_t* q_col, uint8_t* sf_col, int* dev_err, mx_stream_t stream) {
    return mxfp8_quantize_ex(x, MX_DTYPE_BF16, MX_SCALE_FLOOR, rows, cols, mode, seg_off, seg_poff, nseg, ld_col,
                             q_row, sf_row, q_col, sf_col, dev_err, stream);
}

int mxfp8_gather_quantize(const void* x, int64_t T, int64_t cols, int mode, const int32_t* src_row,
                          const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t ld_col, uint8_t* q_row,
                          uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col, int* dev_err, mx_stream_t stream) {
    return mxfp8_gather_quantize_ex(x, T, cols, mode, src_row, nullptr, off, poff, E, R, ld_col, q_row, sf_row, q_col,
                                    sf_col, dev_err, stream);
}

int mxfp8_gather_quantize_ex(const void* x, int64_t T, int64_t cols, int mode, const int32_t* src_row,
                             const float* row_scale, const int32_t* off, const int32_t* poff, int E, int64_t R,
                             int64_t ld_col, uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                             int* dev_err, mx_stream_t stream) {
    if (!valid_mode(mode)) return MX_ERR_INVALID_ARG;
    if (T < 0 || R < 0 || cols <= 0 || cols % 32 != 0 || E < 1 || E > (1 << 20)) return MX_ERR_INVALID_ARG;
    if (T >= (int64_t(1) << 31) || R >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    if (!off || !poff || !dev_err || (R > 0 && (!x || !src_row))) return MX_ERR_INVALID_ARG;
    const bool row = (mode & MX_ROWWISE) != 0, col = (mode & MX_COLWISE) != 0;
    if ((row && (!q_row || !sf_row)) || (col && (!q_col || !sf_col))) return MX_ERR_INVALID_ARG;
    const int64_t pbound = mx_padded_rows_bound(R, E);
    if (col && (ld_col < round_up(R, 128) || ld_col % 128 != 0)) return MX_ERR_INVALID_ARG;
    if (!aligned16(x) || (row && (!aligned16(q_row) || !aligned16(sf_row))) ||
        (col && (!aligned16(q_col) || !aligned16(sf_col))))
        return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    if (pbound == 0) return MX_OK;
    return mx::launch_quantize(x, MX_DTYPE_BF16, MX_SCALE_FLOOR, src_row, row_scale, T, R, cols, mode, off, poff, E,
                               col ? ld_col : 0, pbound, q_row, sf_row, q_col, sf_col, dev_err,
                               reinterpret_cast<cudaStream_t>(stream));
}

namespace {
int swiglu_common(bool bwd, const void* dh, const void* a, int64_t R, int64_t I, int mode, const int32_t* seg_off,
                  const int32_t* seg_poff, int nseg, int64_t ld_col, uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col,
                  uint8_t* sf_col, int* dev_err, mx_stream_t stream) {
    if (!valid_mode(mode)) return MX_ERR_INVALID_ARG;
    if (R < 0 || I <= 0 || I % 128 != 0) return MX_ERR_INVALID_ARG;
    if (R >= (int64_t(1) << 31) || I >= (int64_t(1) << 30)) return MX_ERR_UNSUPPORTED;
    if (nseg < 0 || nseg > (1 << 20) || (nseg > 0 && (!seg_off || !seg_poff))) return MX_ERR_INVALID_ARG;
    if (R > 0 && (!a || (bwd && !dh))) return MX_ERR_INVALID_ARG;
    const bool row = (mode & MX_ROWWISE) != 0, col = (mode & MX_COLWISE) != 0;
    if ((row && (!q_row || !sf_row)) || (col && (!q_col || !sf_col))) return MX_ERR_INVALID_ARG;
    const int64_t pbound = nseg > 0 ? mx_padded_rows_bound(R, nseg) : round_up(R, 128);
    if (col && (ld_col < round_up(R, 128) || ld_col % 128 != 0)) return MX_ERR_INVALID_ARG;
    if (!aligned16(a) || (bwd && !aligned16(dh)) || (row && (!aligned16(q_row) || !aligned16(sf_row))) ||
        (col && (!aligned16(q_col) || !aligned16(sf_col))))
        return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    if (pbound == 0) return MX_OK;
    return mx::launch_swiglu_quantize(bwd, a, dh, R, I, mode, nseg > 0 ? seg_off : nullptr,
                                      nseg > 0 ? seg_poff : nullptr, nseg, col ? ld_col : 0, pbound, q_row, sf_row,
                                      q_col, sf_col, dev_err, reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace

int mxfp8_swiglu_quantize(const void* a, int64_t R, int64_t I, int mode, const int32_t* seg_off,
                          const int32_t* seg_poff, int nseg, int64_t ld_col, uint8_t* q_row, uint8_t* sf_row,
                          uint8_t* q_col, uint8_t* sf_col, int* dev_err, mx_stream_t stream) {
    return swiglu_common(false, nullptr, a, R, I, mode, seg_off, seg_poff, nseg, ld_col, q_row, sf_row, q_col, sf_col,
                         dev_err, stream);
}

int mxfp8_swiglu_bwd_quantize(const void* dh, const void* a, int64_t R, int64_t I, int mode, const int32_t* seg_off,
                              const int32_t* seg_poff, int nseg, int64_t ld_col, uint8_t* q_row, uint8_t* sf_row,
                              uint8_t* q_col, uint8_t* sf_col, int* dev_err, mx_stream_t stream) {
    return swiglu_common(true, dh, a, R, I, mode, seg_off, seg_poff, nseg, ld_col, q_row, sf_row, q_col, sf_col,
                         dev_err, stream);
}

size_t moe_permute_workspace_bytes(int64_t T, int k, int E) {
    if (T < 0 || k < 1 || E < 1) return 0;
    return mx::permute_workspace_bytes(T, k, E);
}

int moe_permute(const int32_t* topk_ids, int64_t T, int k, int E, int32_t* counts, int32_t* off, int32_t* poff,
                int32_t* src_row, int32_t* dst_of, const uint8_t* q_in, const uint8_t* sf_in, int64_t K,
                uint8_t* q_out, uint8_t* sf_out, void* ws, size_t ws_bytes, int* dev_err, mx_stream_t stream) {
    if (T < 0 || k < 1 || k > 64 || E < 1 || E > 1024) return MX_ERR_INVALID_ARG;
    if (T * k >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    if (!counts || !off || !poff || !dev_err || !ws) return MX_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !src_row || !dst_of)) return MX_ERR_INVALID_ARG;
    if (ws_bytes < mx::permute_workspace_bytes(T, k, E)) return MX_ERR_INVALID_ARG;
    const bool gather = q_in != nullptr;
    if (gather) {
        if (!sf_in || !q_out || !sf_out) return MX_ERR_INVALID_ARG;
        if (K <= 0 || K % 32 != 0) return MX_ERR_INVALID_ARG;
        if (!aligned16(q_in) || !aligned16(q_out) || !aligned16(sf_in) || !aligned16(sf_out)) return MX_ERR_ALIGNMENT;
    }
    if (!aligned16(ws)) return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    return mx::launch_permute(topk_ids, T, k, E, counts, off, poff, src_row, dst_of, gather ? q_in : nullptr, sf_in, K,
                              q_out, sf_out, ws, dev_err, reinterpret_cast<cudaStream_t>(stream));
}

int moe_gather_rows(const void* src, int64_t row_bytes, const int32_t* src_row, int64_t R, void* dst,
                    mx_stream_t stream) {
    if (R < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return MX_ERR_INVALID_ARG;
    if (R > 0 && (!src || !src_row || !dst)) return MX_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    return mx::launch_gather_rows(src, row_bytes, src_row, R, dst, reinterpret_cast<cudaStream_t>(stream));
}

int moe_combine_fwd(const void* Y, const float* gate, const int32_t* dst_of, int64_t T, int k, int64_t H, int64_t R,
                    void* out, int* dev_err, mx_stream_t stream) {
    if (T < 0 || k < 1 || k > 64 || H <= 0 || H % 8 != 0 || R < 0) return MX_ERR_INVALID_ARG;
    if (T >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    if (T > 0 && (!Y || !dst_of || !out || !dev_err)) return MX_ERR_INVALID_ARG;
    if (!aligned16(Y) || !aligned16(out)) return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    return mx::launch_combine_fwd(Y, gate, dst_of, T, k, H, R, out, dev_err, reinterpret_cast<cudaStream_t>(stream));
}

int moe_combine_bwd(const void* dOut, const void* Y, const float* gate, const int32_t* dst_of, int64_t T, int k,
                    int64_t H, int64_t R, void* dY, float* dgate, int* dev_err, mx_stream_t stream) {
    if (T > 0 && !dY) return MX_ERR_INVALID_ARG;
    return moe_combine_bwd_ex(dOut, Y, gate, dst_of, T, k, H, R, dY, dgate, nullptr, dev_err, stream);
}

int moe_combine_bwd_ex(const void* dOut, const void* Y, const float* gate, const int32_t* dst_of, int64_t T, int k,
                       int64_t H, int64_t R, void* dY, float* dgate, float* gate_rows, int* dev_err,
                       mx_stream_t stream) {
    if (T < 0 || k < 1 || k > 64 || H <= 0 || H % 8 != 0 || R < 0) return MX_ERR_INVALID_ARG;
    if (T >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    if (T > 0 && (!dOut || !Y || !gate || !dst_of || !dgate || !dev_err)) return MX_ERR_INVALID_ARG;
    if (!aligned16(dOut) || !aligned16(Y) || !aligned16(dY)) return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    return mx::launch_combine_bwd(dOut, Y, gate, dst_of, T, k, H, R, dY, dgate, gate_rows, dev_err,
                                  reinterpret_cast<cudaStream_t>(stream));
}

int grouped_gemm_mxfp8_fwd(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                           const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t N, int64_t K, void* C,
                           int* dev_err, mx_stream_t stream) {
    return gemm_rows_common(A, SFA, B, SFB, off, poff, E, R, N, K, C, dev_err, stream, false, GemmChoice{});
}

int grouped_gemm_mxfp8_fwd_ex(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                              const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t N, int64_t K,
                              void* C, int flags, int* dev_err, mx_stream_t stream) {
    GemmChoice c;
    c.flags = flags;
    return gemm_rows_common(A, SFA, B, SFB, off, poff, E, R, N, K, C, dev_err, stream, false, c);
}

int grouped_gemm_mxfp8_fwd_swiglu(const uint8_t* A, const uint8_t* SFA, const uint8_t* W1, const uint8_t* SFW1,
                                  const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t I, int64_t K,
                                  void* out1, uint8_t* h_qrow, uint8_t* h_sfrow, uint8_t* h_qcol, uint8_t* h_sfcol,
                                  int64_t ld_col, int h_mode, int* dev_err, mx_stream_t stream) {
    return grouped_gemm_mxfp8_fwd_swiglu_ex(A, SFA, W1, SFW1, off, poff, E, R, I, K, out1, h_qrow, h_sfrow, h_qcol,
                                            h_sfcol, ld_col, h_mode, 0, dev_err, stream);
}

int grouped_gemm_mxfp8_fwd_swiglu_ex(const uint8_t* A, const uint8_t* SFA, const uint8_t* W1, const uint8_t* SFW1,
                                     const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t I, int64_t K,
                                     void* out1, uint8_t* h_qrow, uint8_t* h_sfrow, uint8_t* h_qcol, uint8_t* h_sfcol,
                                     int64_t ld_col, int h_mode, int flags, int* dev_err, mx_stream_t stream) {
    if (!valid_gemm_flags(flags)) return MX_ERR_INVALID_ARG;
    if (!valid_mode(h_mode) || (h_mode & (MX_ROWWISE | MX_COLWISE)) != (MX_ROWWISE | MX_COLWISE))
        return MX_ERR_INVALID_ARG;
    if (!A || !SFA || !W1 || !SFW1 || !off || !poff || !out1 || !h_qrow || !h_sfrow || !h_qcol || !h_sfcol || !dev_err)
        return MX_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || R < 0 || I <= 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (I % 128 != 0 || K % 128 != 0) return MX_ERR_UNSUPPORTED;
    if (R >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) || 2 * I * E >= (int64_t(1) << 31)) return MX_ERR_UNSUPPORTED;
    if (ld_col % 128 != 0 || ld_col < mx_padded_rows_bound(R, E) || ld_col * I >= (int64_t(1) << 40))
        return MX_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(SFA) || !aligned16(W1) || !aligned16(SFW1) || !aligned16(out1) ||
        !aligned16(h_qrow) || !aligned16(h_sfrow) || !aligned16(h_qcol) || !aligned16(h_sfcol))
        return MX_ERR_ALIGNMENT;
    int st = check_device();
    if (st != MX_OK) return st;
    if (R == 0) return MX_OK;
    mx::GemmProblem pr{};
    pr.kind = mx::kGemmRows;
    pr.A = A;
    pr.SFA = SFA;
    pr.B = W1;
    pr.SFB = SFW1;
    pr.a_rows = R;
    pr.a_cols = K;
    pr.b_rows = static_cast<int64_t>(E) * 2 * I;
    pr.b_cols = K;
    pr.b_row_step = 2 * I;
    pr.b_col_step = 0;
    pr.n_out = 2 * I;
    pr.m_out = 0;
    pr.k_len = K;
    pr.off = off;
    pr.poff = poff;
    pr.E = E;
    pr.out = out1;
    pr.dev_err = dev_err;
    pr.swiglu_i = I;
    pr.h_qrow = h_qrow;
    pr.h_sfrow = h_sfrow;
    pr.h_qcol = h_qcol;
    pr.h_sfcol = h_sfcol;
    pr.h_ldcol = ld_col;
    pr.h_sfrow_copies = (h_mode & MX_ROWWISE_X4) ? 4 : 1;
    pr.h_sfcol_copies = (h_mode & MX_COLWISE_X4) ? 4 : 1;
    pr.b_scales_x1 = (flags & MX_GEMM_B_SCALES_X1) ? 1 : 0;
    pr.b_blocked = (flags & MX_GEMM_B_BLOCKED) ? 1 : 0;
    return mx::launch_grouped_gemm(pr, reinterpret_cast<cudaStream_t>(stream));
}

int grouped_gemm_mxfp8_dgrad(const uint8_t* dY, const uint8_t* SFdY, const uint8_t* Wt, const uint8_t* SFWt,
                             const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t N, int64_t K, void* dX,
                             int* dev_err, mx_stream_t stream) {
    return gemm_rows_common(dY, SFdY, Wt, SFWt, off, poff, E, R, N, K, dX, dev_err, stream, true, GemmChoice{});
}

int grouped_gemm_mxfp8_dgrad_ex(const uint8_t* dY, const uint8_t* SFdY, const uint8_t* Wt, const uint8_t* SFWt,
                                const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t N, int64_t K,
                                void* dX, int flags, int* dev_err, mx_stream_t stream) {
    GemmChoice c;
    c.flags = flags;
    return gemm_rows_common(dY, SFdY, Wt, SFWt, off, poff, E, R, N, K, dX, dev_err, stream, true, c);
}

int grouped_gemm_mxfp8_wgrad(const uint8_t* dYc, const uint8_t* SFdYc, const uint8_t* Xc, const uint8_t* SFXc,
                             const int32_t* off, const int32_t* poff, int E, int64_t N, int64_t K, int64_t ld_tok,
                             float* dW, int* dev_err, mx_stream_t stream) {
    return gemm_wgrad_common(dYc, SFdYc, Xc, SFXc, off, poff, E, N, K, ld_tok, dW, dev_err, stream, GemmChoice{});
}

int grouped_gemm_mxfp8_wgrad_ex(const uint8_t* dYc, const uint8_t* SFdYc, const uint8_t* Xc, const uint8_t* SFXc,
                                const int32_t* off, const int32_t* poff, int E, int64_t N, int64_t K, int64_t ld_tok,
                                float* dW, int flags, int* dev_err, mx_stream_t stream) {
    GemmChoice c;
    c.flags = flags;
    return gemm_wgrad_common(dYc, SFdYc, Xc, SFXc, off, poff, E, N, K, ld_tok, dW, dev_err, stream, c);
}

int mx_testing_grouped_gemm(int pass, const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                            const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t N, int64_t K,
                            int64_t ld_tok, void* out, int flags, const mx_testing_gemm_options* opt, int* dev_err,
                            mx_stream_t stream) {
    GemmChoice c;
    c.flags = flags;
    if (opt != nullptr) {
        if (opt->ctas_per_mma < 0 || opt->ctas_per_mma > 2) return MX_ERR_INVALID_ARG;
        c.ctas_per_mma = opt->ctas_per_mma;
        c.wait_limit_ns = opt->wait_limit_ns;
        c.withhold_operands = opt->withhold_operands != 0;
        if (opt->raster_group < 0 || opt->raster_group > 64) return MX_ERR_INVALID_ARG;
        c.raster_group = opt->raster_group;
        if (opt->cluster_pairs < 0 || opt->cluster_pairs > 2) return MX_ERR_INVALID_ARG;
        c.cluster_pairs = opt->cluster_pairs;
    }
    switch (pass) {
        case MX_TESTING_FWD:
            return gemm_rows_common(A, SFA, B, SFB, off, poff, E, R, N, K, out, dev_err, stream, false, c);
        case MX_TESTING_DGRAD:
            return gemm_rows_common(A, SFA, B, SFB, off, poff, E, R, N, K, out, dev_err, stream, true, c);
        case MX_TESTING_WGRAD:
            return gemm_wgrad_common(A, SFA, B, SFB, off, poff, E, N, K, ld_tok, static_cast<float*>(out), dev_err,
                                     stream, c);
        default:
            return MX_ERR_INVALID_ARG;
    }
}

const char* mx_status_str(int status) {
    switch (status) {
        case MX_OK: return "MX_OK";
        case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG";
        case MX_ERR_ALIGNMENT: return "MX_ERR_ALIGNMENT";
        case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED";
        case MX_ERR_CUDA: return "MX_ERR_CUDA";
        case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT";
        case MX_ERR_TOO_LARGE: return "MX_ERR_TOO_LARGE";
        default: return "MX_UNKNOWN_STATUS";
    }
}

}  // extern "C"
