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
// of the quantizer.  A CTA owns 128 padded rows x 64 output columns: forward h[:, c0..c0+64);
// backward the 32 gate-part columns c0..c0+32 and the 32 up-part columns I+c0..I+c0+32, so
// that one read of gate, up and dh (and one sigmoid) serves both outputs of a column.
// All of a thread's loads are issued before any arithmetic; the rowwise codes and scales
// are produced from registers; the columnwise ones through a 32 KiB fp32 tile in shared
// memory (64 output columns x 128 rows), whose four 32-row blocks fill complete 4-byte
// groups of the column scale layout.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "mxmoe_internal.h"
#include "quant_common.cuh"

namespace mx {
namespace {

constexpr int kTile = 128;       // padded rows per tile
constexpr int kThreads = 256;
constexpr int kOutCols = 64;     // output columns per tile

// Per-direction geometry: gate/up columns read per row, lanes per row (one 16-byte load
// of 8 bf16 each), rows covered by one pass of the CTA, passes per tile, loads per row.
template <bool BWD>
struct Geo {
    static constexpr int kInCols = BWD ? 32 : 64;
    static constexpr int kLanesPerRow = kInCols / 8;
    static constexpr int kRowsPerPass = kThreads / kLanesPerRow;
    static constexpr int kPasses = kTile / kRowsPerPass;
    static constexpr int kLoads = BWD ? 3 : 2;
    static constexpr int kHalves = BWD ? 2 : 1;   // output column groups per tile
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
// per thread (8 lanes per row forward, 4 backward) and the column pass reads one column of 8
// rows 16 apart per instruction; with this swizzle both meet every bank group once.
template <bool BWD>
__device__ __forceinline__ int tile_chunk(int r, int c) {
    return BWD ? (c ^ ((r >> 4) & 7) ^ (r & 1)) : (c ^ (c >> 3) ^ ((r >> 4) & 7));
}

// SFC: scale arrays in the four-copy layout (bit 0 rowwise, bit 1 columnwise), a compile-time
// choice so that the one-copy kernels compile exactly as without the option.  The backward
// kernel runs 4 CTAs per SM at up to 64 registers (at 48 its packed arithmetic spills).
template <bool BWD, bool ROW, bool COL, int SFC>
__global__ void __launch_bounds__(kThreads, BWD ? 4 : 5) swiglu_quant_kernel(const SwigluParams p) {
    constexpr int kRowCopies = (SFC & 1) ? 4 : 1, kColCopies = (SFC & 2) ? 4 : 1;
    using G = Geo<BWD>;
    constexpr int kRowBlocks = kOutCols / G::kHalves / 32;      // 32-column blocks per row and half
    __shared__ __align__(16) uint32_t sf_col_words[kOutCols];   // the 4 column-block scales of each output column
    __shared__ __align__(16) uint8_t sf_row_stage[G::kHalves * kTile * kRowBlocks];   // rowwise scale bytes
    extern __shared__ __align__(16) float htile[];   // [kHalves][128][64 / kHalves] fp32, columnwise only

    const int64_t bid = blockIdx.x;
    const int64_t ct = bid % p.n_col_tiles;
    const int64_t rt = bid / p.n_col_tiles;
    const int64_t p0 = rt * kTile;
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
    if ((ROW && p0 + kTile > p.pbound) || (COL && p0 + kTile > p.ld_col)) {
        if (threadIdx.x == 0 && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
        return;
    }
    valid = valid < 0 ? 0 : (valid > kTile ? kTile : valid);
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
                float* trow = htile + (hf * kTile + r) * G::kInCols;
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
                if ((lane_in_row & 3) == 0) sf_row_stage[(hf * kTile + r) * kRowBlocks + (lane_in_row >> 2)] = static_cast<uint8_t>(b);
            }
        }
    }

    __syncthreads();   // the staged row scales and (columnwise) the fp32 tile are complete
    if (ROW) {
        // the tile's rowwise scale bytes into their 512-byte atoms: per row and half, the
        // kRowBlocks adjacent bytes of its blocks
        const int t = threadIdx.x;
        if (t < G::kHalves * kTile) {
            const int hf = t / kTile, r = t % kTile;
            const int64_t oc = hf * p.I + c0;   // first output column of the half
            uint8_t* sdst = p.sf_row + (rt * p.n_atom_cols + (oc >> 7)) * 512 * kRowCopies + (r & 31) * 16 + (r >> 5) * 4 +
                            ((oc >> 5) & 3);
            const uint8_t* src = sf_row_stage + t * kRowBlocks;
#pragma unroll
            for (int k = 0; k < kRowCopies; ++k) {
                if (kRowBlocks == 2) *reinterpret_cast<uint16_t*>(sdst + 512 * k) = static_cast<uint16_t>(src[0] | (src[1] << 8));
                else sdst[512 * k] = src[0];
            }
        }
    }

    if (COL) {
        // column pass: lane = (row group g of 16 rows, one of 4 adjacent columns); a thread holds
        // 16 rows of one output column, the other 16 rows of its 32-row block in lane ^ 1, and
        // the 8 lanes of a column write its 128 rows (a whole line) with one store each
        constexpr int kColsPerHalf = kOutCols / G::kHalves;
        const int t = threadIdx.x;
        const int lane = t & 31, warp = t >> 5;
        const int g = lane & 7;
        uint8_t* sf_col_bytes = reinterpret_cast<uint8_t*>(sf_col_words);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int cl = 32 * u + 4 * warp + (lane >> 3);   // output column of the tile
            const int hf = BWD ? (cl >> 5) : 0;
            const int cc = BWD ? (cl & 31) : cl;                // column within its half
            const float* src = htile + (hf * kTile + 16 * g) * G::kInCols + (cc & 3);
            const int pc0 = tile_chunk<BWD>(16 * g, cc >> 2), pc1 = tile_chunk<BWD>(16 * g + 1, cc >> 2);
            float w[16];
            float m4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                w[j] = src[j * G::kInCols + 4 * ((j & 1) ? pc1 : pc0)];
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
            if ((g & 1) == 0) sf_col_bytes[(hf * kColsPerHalf + cc) * 4 + (g >> 1)] = static_cast<uint8_t>(b);
        }
        __syncthreads();
        if (t < kOutCols) {
            const int64_t oc2 = (t / kColsPerHalf) * p.I + c0 + (t % kColsPerHalf);
            uint8_t* sdst = p.sf_col + ((oc2 >> 7) * (p.ld_col / 128) + rt) * 512 * kColCopies + (oc2 & 31) * 16 +
                            ((oc2 >> 5) & 3) * 4;
#pragma unroll
            for (int k = 0; k < kColCopies; ++k) *reinterpret_cast<uint32_t*>(sdst + 512 * k) = sf_col_words[t];
        }
    }
}

template <bool BWD, bool ROW, bool COL, int SFC>
cudaError_t launch_one(unsigned blocks, const SwigluParams& p, cudaStream_t stream) {
    const int smem = COL ? kTile * kOutCols * 4 : 0;   // 32 KiB: no opt-in attribute needed
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
    p.n_col_tiles = I / (bwd ? Geo<true>::kInCols : Geo<false>::kInCols);
    p.n_atom_cols = p.ncols / 128;
    p.dev_err = dev_err;
    const int64_t blocks = (pbound / kTile) * p.n_col_tiles;
    if (blocks <= 0) return MX_OK;
    if (blocks > 0x7FFFFFFFLL) return MX_ERR_UNSUPPORTED;
    const cudaError_t e = bwd ? launch_mode<true>(mode, static_cast<unsigned>(blocks), p, stream)
                              : launch_mode<false>(mode, static_cast<unsigned>(blocks), p, stream);
    return e == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

}  // namespace mx
