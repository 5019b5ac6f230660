// swiglu.cu -- SwiGLU between the two expert GEMMs, fused with MXFP8 quantization of its
// result (kucoin.com, "Cursor's MoK демонстрирует повышение производительности на 2,37x на
// NVIDIA GB300 NVL72", section "02": MXFP8 quantization folded into the dispatch, grouped
// GEMM and SwiGLU data path, so no separate quantization kernel and no bf16 round trip of
// the intermediate).
//
//   forward   a = [gate | up] (bf16 [R x 2I], the GEMM1 output) ->
//             h = silu(gate) * up, quantized rowwise (the GEMM2 operand) and columnwise
//             over expert segments (the wgrad2 operand), never stored in bf16;
//   backward  dh (bf16 [R x I], the dgrad2 output) and a ->
//             dH = [dh * up * s (1 + gate (1 - s)) | dh * silu(gate)], s = sigmoid(gate),
//             quantized rowwise (the dgrad1 operand) and columnwise (the wgrad1 operand).
// The elementwise values are computed in fp32 and quantized from fp32 with the scale rule
// of the quantizer.  A CTA reads 64 gate and 64 up columns (whole 128-byte lines of every
// row): forward 128 padded rows, h[:, c0..c0+64); backward 64 padded rows, the 64 gate-part
// columns c0..c0+64 and the 64 up-part columns I+c0..I+c0+64, so that one read of gate, up
// and dh (and one sigmoid) serves both outputs of a column.  All of a thread's loads are
// issued before any arithmetic; the rowwise codes and scales are produced from registers;
// the columnwise ones through a 32 KiB fp32 tile in shared memory (forward 64 columns x 128
// rows, backward 128 x 64), whose 32-row blocks fill all (forward) or half (backward) of a
// column's 4-byte group of the column scale layout.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "mxmoe_internal.h"
#include "quant_common.cuh"

namespace mx {
namespace {

constexpr int kThreads = 256;

// Per-direction geometry: rows per tile, gate/up columns read per row (whole 128-byte lines),
// lanes per row (one 16-byte load of 8 bf16 each), rows covered by one pass of the CTA,
// passes per tile, loads per row, output column groups and output columns per tile.
template <bool BWD>
struct Geo {
    static constexpr int kRows = BWD ? 64 : 128;
    static constexpr int kInCols = 64;
    static constexpr int kLanesPerRow = kInCols / 8;
    static constexpr int kRowsPerPass = kThreads / kLanesPerRow;
    static constexpr int kPasses = kRows / kRowsPerPass;
    static constexpr int kLoads = BWD ? 3 : 2;
    static constexpr int kHalves = BWD ? 2 : 1;
    static constexpr int kOutCols = kInCols * kHalves;
};

struct SwigluParams {
    const uint16_t* a;    // [R x 2I]
    const uint16_t* dh;   // [R x I] (backward)
    int64_t rows, I, ncols;   // ncols = I (forward) or 2I (backward)
    uint8_t* q_row;
    uint8_t* sf_row;
    uint8_t* q_col;
    uint8_t* sf_col;
    int64_t ld_col;
    const int32_t* seg_off;
    const int32_t* seg_poff;
    int nseg;
    int64_t pbound;
    int64_t n_col_tiles;   // tiles across the gate/up columns
    int64_t n_atom_cols;   // 128-column scale atoms across the output (ncols / 128)
    int* dev_err;
};

// Eight E4M3 codes of o (scale byte b; b = 0xFF marks a NaN/Inf block: NaN scale, NaN codes).
__device__ __forceinline__ uint2 quant8_f32(const float (&o)[8], uint32_t b) {
    const float sc = inv_scale_or_nan(b);
    return make_uint2(quant_quad_f32(o[0], o[1], o[2], o[3], sc), quant_quad_f32(o[4], o[5], o[6], o[7], sc));
}

// The SwiGLU values of 8 columns of one row from the bf16 words of gate, up (and dh): forward
// h = g sigmoid(g) u; backward d/d gate = dh u (s (1 + g (1 - s))) and d/d up = dh (g s),
// s = sigmoid(g), in the operation order of the scalar forms, two columns per packed
// instruction.
template <bool BWD, bool FTZ>
__device__ __forceinline__ void swiglu8(const uint4& gv, const uint4& uv, const uint4& dv, float (&o0)[8],
                                        float (&o1)[8]) {
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
    const uint64_t one = pk2(1.0f, 1.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float g0 = bf16_lo(gw[k]), g1 = bf16_hi(gw[k]);
        const uint64_t G = pk2(g0, g1), U = pk2(bf16_lo(uw[k]), bf16_hi(uw[k]));
        const uint64_t S = sigmoid2<FTZ>(g0, g1);
        if (!BWD) {
            const uint64_t H = mul2(mul2(G, S), U);
            o0[2 * k] = lo2(H);
            o0[2 * k + 1] = hi2(H);
        } else {
            const uint64_t D = pk2(bf16_lo(dw[k]), bf16_hi(dw[k]));
            const uint64_t dG = mul2(mul2(D, U), mul2(S, fma2(G, sub2(one, S), one)));
            const uint64_t dU = mul2(D, mul2(G, S));
            o0[2 * k] = lo2(dG);
            o0[2 * k + 1] = hi2(dG);
            o1[2 * k] = lo2(dU);
            o1[2 * k + 1] = hi2(dU);
        }
    }
}

// Position of 4-float chunk c of tile row r in shared memory.  The row pass stores two chunks
// per thread (8 lanes per row, chunks 2 l and 2 l + 1) and the column pass reads one column
// of 8 (forward) or 4 (backward) rows 16 apart per instruction; with these swizzles both meet
// every bank group once.
template <bool BWD>
__device__ __forceinline__ int tile_chunk(int r, int c) {
    return BWD ? (c ^ (c >> 3) ^ (2 * ((r >> 4) & 3))) : (c ^ (c >> 3) ^ ((r >> 4) & 7));
}

// SFC: scale arrays in the four-copy layout (bit 0 rowwise, bit 1 columnwise), a compile-time
// choice so that the one-copy kernels compile exactly as without the option.  The backward
// kernel runs 4 CTAs per SM at up to 64 registers (at 5 CTAs and 48 registers it is slower).
template <bool BWD, bool ROW, bool COL, int SFC>
__global__ void __launch_bounds__(kThreads, BWD ? 4 : 5) swiglu_quant_kernel(const SwigluParams p) {
    constexpr int kRowCopies = (SFC & 1) ? 4 : 1, kColCopies = (SFC & 2) ? 4 : 1;
    using G = Geo<BWD>;
    constexpr int kRowBlocks = G::kInCols / 32;                 // 32-column blocks per row and half
    constexpr int kColBlocks = G::kRows / 32;                   // 32-row blocks per column
    __shared__ __align__(16) uint8_t sf_col_stage[G::kOutCols * kColBlocks];   // columnwise scale bytes, per column
    __shared__ __align__(16) uint8_t sf_row_stage[G::kHalves * G::kRows * kRowBlocks];   // rowwise scale bytes
    extern __shared__ __align__(16) float htile[];   // [kHalves][kRows][kInCols] fp32, columnwise only

    const int64_t bid = blockIdx.x;
    const int64_t ct = bid % p.n_col_tiles;
    const int64_t rt = bid / p.n_col_tiles;
    const int64_t p0 = rt * G::kRows;
    const int64_t c0 = ct * G::kInCols;
    int64_t row0, valid;
    if (p.nseg == 0) {
        row0 = p0;
        valid = p.rows - p0;
    } else {
        const int32_t ptotal = __ldg(p.seg_poff + p.nseg);
        if (p0 >= ptotal) return;
        const int lo = find_segment(p.seg_poff, p.nseg, p0);   // last g with poff[g] <= p0
        const int64_t pg = __ldg(p.seg_poff + lo);
        const int64_t og = __ldg(p.seg_off + lo);
        const int64_t te = __ldg(p.seg_off + lo + 1) - og;
        row0 = og + (p0 - pg);
        valid = te - (p0 - pg);
        if (te < 0 || (pg & 127) != 0 || og + te > p.rows || og < 0) {
            if (threadIdx.x == 0 && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
            return;
        }
    }
    if ((ROW && p0 + G::kRows > p.pbound) || (COL && p0 + G::kRows > p.ld_col)) {
        if (threadIdx.x == 0 && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
        return;
    }
    valid = valid < 0 ? 0 : (valid > G::kRows ? G::kRows : valid);
    const int lane_in_row = threadIdx.x % G::kLanesPerRow;
    const int row_in_pass = threadIdx.x / G::kLanesPerRow;
    const int64_t c = c0 + lane_in_row * 8;   // first gate/up column of this thread
    // pointers of the thread's first row; each pass moves kRowsPerPass rows on
    const int64_t r0 = row0 + row_in_pass;
    const uint16_t* ap = p.a + r0 * 2 * p.I + c;
    const uint16_t* dp = BWD ? p.dh + r0 * p.I + c : nullptr;
    uint8_t* qp = p.q_row + r0 * p.ncols + c;
    const int64_t a_pass = G::kRowsPerPass * 2 * p.I, d_pass = G::kRowsPerPass * p.I, q_pass = G::kRowsPerPass * p.ncols;

    // ---- every load of the thread in flight at once
    uint4 ld[G::kPasses][G::kLoads];
#pragma unroll
    for (int it = 0; it < G::kPasses; ++it) {
        const int r = it * G::kRowsPerPass + row_in_pass;
#pragma unroll
        for (int l = 0; l < G::kLoads; ++l) ld[it][l] = make_uint4(0u, 0u, 0u, 0u);
        if (r < valid) {
            ld[it][0] = ld_stream_16(ap + it * a_pass);
            ld[it][1] = ld_stream_16(ap + it * a_pass + p.I);
            if (BWD) ld[it][G::kLoads - 1] = ld_stream_16(dp + it * d_pass);
        }
    }

#pragma unroll
    for (int it = 0; it < G::kPasses; ++it) {
        const int r = it * G::kRowsPerPass + row_in_pass;
        // a warp whose gate values of this pass all have |g| < 64 takes the sigmoid with flushed
        // subnormals (identical results there, fewer instructions)
        const uint32_t gmax = amax_bf16x2(amax_bf16x2(ld[it][0].x, ld[it][0].y), amax_bf16x2(ld[it][0].z, ld[it][0].w));
        const bool big = (gmax & 0x7FFFu) >= 0x4280u || ((gmax >> 16) & 0x7FFFu) >= 0x4280u;
        float o[G::kHalves][8];
        if (!__any_sync(0xffffffffu, big))
            swiglu8<BWD, true>(ld[it][0], ld[it][1], ld[it][G::kLoads - 1], o[0], o[G::kHalves - 1]);
        else
            swiglu8<BWD, false>(ld[it][0], ld[it][1], ld[it][G::kLoads - 1], o[0], o[G::kHalves - 1]);
#pragma unroll
        for (int hf = 0; hf < G::kHalves; ++hf) {
            if (COL) {
                float* trow = htile + (hf * G::kRows + r) * G::kInCols;
                *reinterpret_cast<float4*>(trow + 4 * tile_chunk<BWD>(r, 2 * lane_in_row)) =
                    make_float4(o[hf][0], o[hf][1], o[hf][2], o[hf][3]);
                *reinterpret_cast<float4*>(trow + 4 * tile_chunk<BWD>(r, 2 * lane_in_row + 1)) =
                    make_float4(o[hf][4], o[hf][5], o[hf][6], o[hf][7]);
            }
            if (ROW) {
                float m = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) m = amax_step(m, o[hf][i]);
                // the 4 lanes of a 32-column block
                m = amax_step(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = amax_step(m, __shfl_xor_sync(0xffffffffu, m, 2));
                const uint32_t b = scale_byte_f32<0>(__float_as_uint(m));
                const uint2 q = quant8_f32(o[hf], b);
                if (r < valid) *reinterpret_cast<uint2*>(qp + it * q_pass + hf * p.I) = q;
                if ((lane_in_row & 3) == 0) sf_row_stage[(hf * G::kRows + r) * kRowBlocks + (lane_in_row >> 2)] = static_cast<uint8_t>(b);
            }
        }
    }

    __syncthreads();   // the staged row scales and (columnwise) the fp32 tile are complete
    if (ROW) {
        // the tile's rowwise scale bytes into their 512-byte atoms: per row and half, the
        // kRowBlocks adjacent bytes of its blocks
        const int t = threadIdx.x;
        if (t < G::kHalves * G::kRows) {
            const int hf = t / G::kRows;
            const int64_t pr = p0 + t % G::kRows;   // padded row
            const int64_t oc = hf * p.I + c0;   // first output column of the half
            const int ar = static_cast<int>(pr & 127);   // row within its 128-row scale atom
            uint8_t* sdst = p.sf_row + ((pr >> 7) * p.n_atom_cols + (oc >> 7)) * 512 * kRowCopies + (ar & 31) * 16 +
                            (ar >> 5) * 4 + ((oc >> 5) & 3);
            const uint8_t* src = sf_row_stage + t * kRowBlocks;
#pragma unroll
            for (int k = 0; k < kRowCopies; ++k) {
                if (kRowBlocks == 2) *reinterpret_cast<uint16_t*>(sdst + 512 * k) = static_cast<uint16_t>(src[0] | (src[1] << 8));
                else sdst[512 * k] = src[0];
            }
        }
    }

    if (COL) {
        // column pass: lane = (row group g of 16 rows, one of 32 / kG adjacent columns); a thread
        // holds 16 rows of one output column, the other 16 rows of its 32-row block in lane ^ 1,
        // and the kG lanes of a column write its kRows rows with one store each
        constexpr int kG = G::kRows / 16;                        // row groups (lanes per column)
        constexpr int kColsPerPass = kThreads / kG;              // columns per pass of the CTA
        const int t = threadIdx.x;
        const int lane = t & 31, warp = t >> 5;
        const int g = lane % kG;
#pragma unroll
        for (int u = 0; u < G::kOutCols / kColsPerPass; ++u) {
            const int cl = kColsPerPass * u + (32 / kG) * warp + lane / kG;   // output column of the tile
            const int hf = cl / G::kInCols;
            const int cc = cl % G::kInCols;                      // column within its half
            const float* src = htile + (hf * G::kRows + 16 * g) * G::kInCols + 4 * tile_chunk<BWD>(16 * g, cc >> 2) +
                               (cc & 3);
            float w[16];
            float m4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                w[j] = src[j * G::kInCols];
                m4[j & 3] = amax_step(m4[j & 3], w[j]);
            }
            float m = amax_step(amax_step(m4[0], m4[1]), amax_step(m4[2], m4[3]));
            m = amax_step(m, __shfl_xor_sync(0xffffffffu, m, 1));
            const uint32_t b = scale_byte_f32<0>(__float_as_uint(m));
            const float sc = inv_scale_or_nan(b);
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                o[j] = quant_quad_f32(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3], sc);
            const int64_t oc = hf * p.I + c0 + cc;
            *reinterpret_cast<uint4*>(p.q_col + oc * p.ld_col + p0 + 16 * g) = make_uint4(o[0], o[1], o[2], o[3]);
            if ((g & 1) == 0) sf_col_stage[cl * kColBlocks + (g >> 1)] = static_cast<uint8_t>(b);
        }
        __syncthreads();
        if (t < G::kOutCols) {
            // the column's kColBlocks scale bytes into its 4-byte group of the 128-row atom
            const int64_t oc2 = (t / G::kInCols) * p.I + c0 + (t % G::kInCols);
            uint8_t* sdst = p.sf_col + ((oc2 >> 7) * (p.ld_col / 128) + (p0 >> 7)) * 512 * kColCopies + (oc2 & 31) * 16 +
                            ((oc2 >> 5) & 3) * 4 + ((p0 & 127) >> 5);
            const uint8_t* cs = sf_col_stage + t * kColBlocks;
#pragma unroll
            for (int k = 0; k < kColCopies; ++k) {
                if (kColBlocks == 4) *reinterpret_cast<uint32_t*>(sdst + 512 * k) = *reinterpret_cast<const uint32_t*>(cs);
                else *reinterpret_cast<uint16_t*>(sdst + 512 * k) = *reinterpret_cast<const uint16_t*>(cs);
            }
        }
    }
}

template <bool BWD, bool ROW, bool COL, int SFC>
cudaError_t launch_one(unsigned blocks, const SwigluParams& p, cudaStream_t stream) {
    const int smem = COL ? Geo<BWD>::kRows * Geo<BWD>::kOutCols * 4 : 0;   // 32 KiB: no opt-in attribute needed
    swiglu_quant_kernel<BWD, ROW, COL, SFC><<<blocks, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <bool BWD>
cudaError_t launch_mode(int mode, unsigned blocks, const SwigluParams& p, cudaStream_t stream) {
    switch (mode & (MX_ROWWISE | MX_COLWISE)) {
        case MX_ROWWISE:
            return (mode & MX_ROWWISE_X4) ? launch_one<BWD, true, false, 1>(blocks, p, stream)
                                          : launch_one<BWD, true, false, 0>(blocks, p, stream);
        case MX_COLWISE:
            return (mode & MX_COLWISE_X4) ? launch_one<BWD, false, true, 2>(blocks, p, stream)
                                          : launch_one<BWD, false, true, 0>(blocks, p, stream);
        default:
            switch (((mode & MX_ROWWISE_X4) ? 1 : 0) | ((mode & MX_COLWISE_X4) ? 2 : 0)) {
                case 1: return launch_one<BWD, true, true, 1>(blocks, p, stream);
                case 2: return launch_one<BWD, true, true, 2>(blocks, p, stream);
                case 3: return launch_one<BWD, true, true, 3>(blocks, p, stream);
                default: return launch_one<BWD, true, true, 0>(blocks, p, stream);
            }
    }
}

}  // namespace

int launch_swiglu_quantize(bool bwd, const void* a, const void* dh, int64_t R, int64_t I, int mode,
                           const int32_t* seg_off, const int32_t* seg_poff, int nseg, int64_t ld_col, int64_t pbound,
                           uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col, int* dev_err,
                           cudaStream_t stream) {
    SwigluParams p;
    p.a = static_cast<const uint16_t*>(a);
    p.dh = static_cast<const uint16_t*>(dh);
    p.rows = R;
    p.I = I;
    p.ncols = bwd ? 2 * I : I;
    p.q_row = q_row;
    p.sf_row = sf_row;
    p.q_col = q_col;
    p.sf_col = sf_col;
    p.ld_col = ld_col;
    p.seg_off = seg_off;
    p.seg_poff = seg_poff;
    p.nseg = nseg;
    p.pbound = pbound;
    p.n_col_tiles = I / Geo<false>::kInCols;   // (the same in both directions)
    p.n_atom_cols = p.ncols / 128;
    p.dev_err = dev_err;
    const int64_t blocks = (pbound / (bwd ? Geo<true>::kRows : Geo<false>::kRows)) * p.n_col_tiles;
    if (blocks <= 0) return MX_OK;
    if (blocks > 0x7FFFFFFFLL) return MX_ERR_UNSUPPORTED;
    const cudaError_t e = bwd ? launch_mode<true>(mode, static_cast<unsigned>(blocks), p, stream)
                              : launch_mode<false>(mode, static_cast<unsigned>(blocks), p, stream);
    return e == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

}  // namespace mx
