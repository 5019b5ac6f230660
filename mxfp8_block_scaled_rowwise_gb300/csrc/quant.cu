// quant.cu -- bf16 -> MXFP8 quantizer for sm_103a.
//
// One CTA of 256 threads owns a tile of 128 padded rows x 128 columns (32 KiB of
// bf16).  The tile is read once with coalesced 16-byte loads; from the same
// registers it produces
//   * the rowwise form: 32-element blocks along the row, amax by a two-step
//     warp shuffle among the 4 lanes that hold a block, E4M3 codes stored with
//     8-byte stores, and the tile's 128 x 4 scale bytes assembled in shared
//     memory as one complete 512-byte atom of the tensor-core scale layout and
//     written with one coalesced 512-byte store;
//   * the columnwise (transposed) form: the tile goes through shared memory; each
//     thread reads 4 adjacent columns x 16 rows with 8-byte loads, the other 16 rows
//     of the 32-row block being in the lane 16 apart (one shuffle completes the
//     column amax), writes 4 x 16 contiguous codes of the transposed output, and the
//     128 x 4 column scales again form one complete 512-byte atom.
// The scale rule (OCP MX, which the pages' recipe -- E4M3, blocks of 32 --
// leaves to the standard): scale byte b = max(E(amax) - 8, 0) where E(amax) is the
// biased binary exponent field of the largest |x| (an all-zero block gives 0),
// elements E4M3(x * 2^(127 - b)) with round-to-nearest-even and saturation.
// Multiplying a bf16 value by that power of two is exact in fp32 whenever the
// result is normal, so every element sees exactly one rounding.
//
// Sources: aigc.bar "Blackwell性能陷阱？Cursor揭秘：重写内核让AI大模型MoE提速3.5倍的底层逻辑",
// section "“秘密武器”：自研量化内核与最佳精度配方" (E4M3, block 32, output layout that the
// MMA reads with no reshape); lpnh.cn, section "1. 为什么 MoE 内核在 Blackwell 上反而变慢了"
// (divide by the block scale then convert; backward transpose-quantize).
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "mxmoe_internal.h"
#include "quant_common.cuh"

namespace mx {
namespace {

constexpr int kTileRows = 128;
constexpr int kTileCols = 128;
constexpr int kThreads = 256;

struct QuantParams {
    const uint16_t* x;
    const int32_t* src_row;   // optional: row r of the quantized tensor is x row src_row[r]
    const float* row_scale;   // optional (SCALED kernels): row r is bf16(row_scale[r] * x row src_row[r])
    int64_t src_rows;         // rows of x when src_row is given (indices outside [0, src_rows) read as zero)
    int64_t rows, cols;
    uint8_t* q_row;
    uint8_t* sf_row;
    uint8_t* q_col;
    uint8_t* sf_col;
    int64_t ld_col;
    const int32_t* seg_off;
    const int32_t* seg_poff;
    int nseg;
    int64_t pbound;      // rows of the padded scale-row space the rowwise scale buffer holds
    int64_t n_col_tiles;
    int* dev_err;
    int lean;            // x 32-byte aligned: full tiles take the 256-bit-load path
    int64_t n_row_tiles;
    int col_major;       // tiles in column-slice order (all row tiles of a 128-column slice in turn)
    // Where a tile's codes go.  Row r of tile (rt, ct) starts at q_row + row0 * cols +
    // ct * qr_cstep + r * qr_ld, column c of it at q_col + col0 * ld_col + rt * qc_pstep +
    // c * qc_ld.  Row-major: qr_cstep = 128, qr_ld = cols, qc_pstep = 128, qc_ld = ld_col.
    // Blocked layout (128 x 128 blocks of 16 KiB, row-block major; a blocked rowwise form has
    // no segments, so row0 = 128 rt): qr_cstep = qc_pstep = 16384, qr_ld = qc_ld = 128 --
    // block (rt, ct) of [rows x cols] starts at (rt * cols / 128 + ct) * 16384 = 128 rt * cols
    // + 16384 ct, block (ct, rt) of [cols x ld_col] at 128 ct * ld_col + 16384 rt.
    int64_t qr_cstep, qr_ld, qc_pstep, qc_ld;
};

// Quantize 8 bf16 values (one 16-byte chunk) to 8 E4M3 codes packed little-endian.
__device__ __forceinline__ uint2 quant8(uint4 v, uint32_t b) {
    if (b == 0xFFu) return make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
    const float s = inv_scale(b);
    return make_uint2(quant_quad(v.x, v.y, s), quant_quad(v.z, v.w, s));
}

// 8 bf16 values times s, each product rounded to bf16 (round to nearest even).
__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float lo = bf16_lo(w[i]), hi = bf16_hi(w[i]);
        mul_f32x2(lo, hi, s);
        o[i] = pack_bf16x2(lo, hi);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// SFC: scale arrays in the four-copy layout (bit 0 rowwise, bit 1 columnwise): each 512-byte
// atom is stored four times in a row (a compile-time choice, so the one-copy kernels compile
// exactly as without the option).  SCALED: every input row first multiplied by its row scale
// and rounded to bf16 (the combine backward's dY = bf16(gate * dOut), formed on the fly).  All
// forms run 5 CTAs per SM at 48 registers; the row-scaled row + col form spills 72 bytes there
// and is still 2 % faster than at 4 CTAs and 64 registers.
template <bool ROW, bool COL, int RULE, int SFC, bool SCALED = false>
__global__ void __launch_bounds__(kThreads, 5) quantize_tile_kernel(const QuantParams p) {
    __shared__ __align__(16) uint32_t sf_atom_row[128];
    __shared__ __align__(16) uint8_t sf_atom_col[512];
    extern __shared__ __align__(16) uint8_t tile[];  // [128][256 bytes], columnwise only

    // Tile order.  A gather reads each x row once per routed slot, the slots of a token in
    // different experts' tiles: in column-slice order a 128-column slice of x (rows x 256
    // bytes) stays in L2 while every row tile reads it, so x comes from DRAM about once.
    const int64_t bid = blockIdx.x;
    const int64_t ct = p.col_major ? bid / p.n_row_tiles : bid % p.n_col_tiles;
    const int64_t rt = p.col_major ? bid % p.n_row_tiles : bid / p.n_col_tiles;
    const int64_t p0 = rt * kTileRows;   // first padded position of the tile
    const int64_t col0 = ct * kTileCols;

    // ---- which input rows feed this tile
    int64_t row0;    // input row of padded position p0
    int64_t valid;   // rows of the tile that hold data
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
        const bool bad = te < 0 || (pg & 127) != 0 || og + te > p.rows || og < 0;
        if (bad) {
            if (threadIdx.x == 0 && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
            return;
        }
    }
    // the output buffers must hold this 128-position range
    if ((ROW && p0 + kTileRows > p.pbound) || (COL && p0 + kTileRows > p.ld_col)) {
        if (threadIdx.x == 0 && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
        return;
    }
    valid = valid < 0 ? 0 : (valid > kTileRows ? kTileRows : valid);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (p.lean && valid == kTileRows && col0 + kTileCols <= p.cols) {
        // ---- full tile.  The L1 serves a warp's global access one 128-byte line per wavefront
        // and only merges neighbouring lanes, so consecutive lanes cover consecutive bytes
        // everywhere below; shared-memory accesses are free of bank conflicts.  Row pass: lane
        // l holds 16 columns (one 256-bit load; chunk c32 = l & 7) of row l >> 3 of each of 4
        // row groups; a 32-column block spans lanes l and l ^ 1.
        const int c32 = lane & 7;
        uint32_t x[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = u * 32 + warp * 4 + (lane >> 3);
            int64_t src = row0 + r;
            bool in_range = true;
            if (p.src_row != nullptr) {
                src = __ldg(p.src_row + row0 + r);
                in_range = src >= 0 && src < p.src_rows;
                if (!in_range && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
            }
            if (in_range) {
                ld_stream_32(p.x + src * p.cols + col0 + 16 * c32, x[u]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) x[u][i] = 0u;
            }
        }
        if (SCALED) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float rs = __ldg(p.row_scale + row0 + u * 32 + warp * 4 + (lane >> 3));
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const uint4 t = scale_bf16x8(make_uint4(x[u][4 * g], x[u][4 * g + 1], x[u][4 * g + 2], x[u][4 * g + 3]), rs);
                    x[u][4 * g] = t.x; x[u][4 * g + 1] = t.y; x[u][4 * g + 2] = t.z; x[u][4 * g + 3] = t.w;
                }
            }
        }
        if (COL) {
            // the tile in shared memory: 16-byte chunk c of row r at chunk c ^ (c >> 3) ^ ((r >> 4) & 7),
            // so that each 8-lane store phase (one row) and each 16-lane read phase below (8 rows,
            // one chunk) meets 8 different bank groups
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = u * 32 + warp * 4 + (lane >> 3);
                const int sw = (r >> 4) & 7;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int c = 2 * c32 + i;
                    *reinterpret_cast<uint4*>(tile + r * 256 + (c ^ (c >> 3) ^ sw) * 16) =
                        make_uint4(x[u][4 * i], x[u][4 * i + 1], x[u][4 * i + 2], x[u][4 * i + 3]);
                }
            }
        }
        if (ROW) {
            uint8_t* sf_bytes = reinterpret_cast<uint8_t*>(sf_atom_row);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = u * 32 + warp * 4 + (lane >> 3);
                uint32_t m = amax_bf16x2(amax_bf16x2(amax_bf16x2(x[u][0], x[u][1]), amax_bf16x2(x[u][2], x[u][3])),
                                         amax_bf16x2(amax_bf16x2(x[u][4], x[u][5]), amax_bf16x2(x[u][6], x[u][7])));
                m = amax_bf16x2(m, __byte_perm(m, 0u, 0x1032));
                m = amax_bf16x2(m, __shfl_xor_sync(0xffffffffu, m, 1));
                const uint32_t b = scale_byte_bf16<RULE>(m & 0x7FFFu);
                const float sc = inv_scale_or_nan(b);
                uint32_t c[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    c[k] = quant_quad(x[u][2 * k], x[u][2 * k + 1], sc);
                *reinterpret_cast<uint4*>(p.q_row + row0 * p.cols + ct * p.qr_cstep + r * p.qr_ld + 16 * c32) = make_uint4(c[0], c[1], c[2], c[3]);
                if ((c32 & 1) == 0) sf_bytes[(r & 31) * 16 + (r >> 5) * 4 + (c32 >> 1)] = static_cast<uint8_t>(b);
            }
        }
        if (COL) {
            __syncthreads();
            // column pass: lane = (quad qi, row group g of 16 rows); a thread holds 4 adjacent
            // columns (quad q) x 16 rows, the other 16 rows of its 32-row block in lane ^ 1; the
            // 8 lanes of a quad write one column's 128 rows (a whole line) per store
            const int g = lane & 7;
            const int qi = lane >> 3;
            const int q = 4 * warp + qi;
            const int lc = q >> 1;
            const uint8_t* tb = tile + g * 16 * 256 + ((lc ^ (lc >> 3) ^ g) * 16) + (q & 1) * 8;
            uint2 w[16];
            uint32_t ma[2] = {0u, 0u}, mb[2] = {0u, 0u};
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                w[j] = *reinterpret_cast<const uint2*>(tb + j * 256);
                ma[j & 1] = amax_bf16x2(ma[j & 1], w[j].x);
                mb[j & 1] = amax_bf16x2(mb[j & 1], w[j].y);
            }
            uint32_t m01 = amax_bf16x2(ma[0], ma[1]), m23 = amax_bf16x2(mb[0], mb[1]);
            m01 = amax_bf16x2(m01, __shfl_xor_sync(0xffffffffu, m01, 1));
            m23 = amax_bf16x2(m23, __shfl_xor_sync(0xffffffffu, m23, 1));
            uint8_t* qc = (p.q_col + col0 * p.ld_col + rt * p.qc_pstep) + 4 * q * p.qc_ld + g * 16;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t bc = scale_byte_bf16<RULE>(((c < 2 ? m01 : m23) >> (16 * (c & 1))) & 0x7FFFu);
                const float sc = inv_scale_or_nan(bc);
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t word = (c < 2) ? w[4 * j + i].x : w[4 * j + i].y;
                        v[i] = (c & 1) ? bf16_hi(word) : bf16_lo(word);
                    }
                    o[j] = cvt_e4m3x4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
                }
                *reinterpret_cast<uint4*>(qc + c * p.qc_ld) = make_uint4(o[0], o[1], o[2], o[3]);
                if ((g & 1) == 0) {
                    const int cc = 4 * q + c;
                    sf_atom_col[(cc & 31) * 16 + (cc >> 5) * 4 + (g >> 1)] = static_cast<uint8_t>(bc);
                }
            }
        }
    } else {
        const int chunk = lane & 15;                 // 16-byte chunk (8 columns) within the tile row
        const int64_t gcol = col0 + chunk * 8;
        const bool col_ok = gcol < p.cols;

        // ---- load: 8 rows per thread, two rows per warp per step, fully coalesced
        uint4 v[8];
    #pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = i * 16 + warp * 2 + (lane >> 4);
            v[i] = make_uint4(0u, 0u, 0u, 0u);
            if (r < valid && col_ok) {
                int64_t src = row0 + r;
                bool in_range = true;
                if (p.src_row != nullptr) {
                    src = __ldg(p.src_row + row0 + r);
                    in_range = src >= 0 && src < p.src_rows;
                    if (!in_range && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
                }
                if (in_range) v[i] = ld_stream_16(p.x + src * p.cols + gcol);
            }
        }
        if (SCALED) {
    #pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = i * 16 + warp * 2 + (lane >> 4);
                if (r < valid) v[i] = scale_bf16x8(v[i], __ldg(p.row_scale + row0 + r));
            }
        }

        if (COL) {
    #pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = i * 16 + warp * 2 + (lane >> 4);
                *reinterpret_cast<uint4*>(tile + r * 256 + chunk * 16) = v[i];
            }
        }

        if (ROW) {
            uint8_t* sf_bytes = reinterpret_cast<uint8_t*>(sf_atom_row);
    #pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = i * 16 + warp * 2 + (lane >> 4);
                const uint32_t m2 = amax_bf16x2(amax_bf16x2(v[i].x, v[i].y), amax_bf16x2(v[i].z, v[i].w));
                uint32_t m = amax_bf16x2(m2, __byte_perm(m2, 0u, 0x1032));   // both halves: max over the 8 values
                m = amax_bf16x2(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = amax_bf16x2(m, __shfl_xor_sync(0xffffffffu, m, 2));
                const uint32_t b = scale_byte_bf16<RULE>(m & 0x7FFFu);
                const uint2 q = quant8(v[i], b);
                if (r < valid && col_ok)
                    *reinterpret_cast<uint2*>(p.q_row + row0 * p.cols + ct * p.qr_cstep + r * p.qr_ld + chunk * 8) = q;
                // one lane per 32-element block writes its scale byte into the atom
                if ((chunk & 3) == 0) sf_bytes[(r & 31) * 16 + (r >> 5) * 4 + (chunk >> 2)] = static_cast<uint8_t>(b);
            }
        }

        if (COL) {
            __syncthreads();
            // one thread: 4 adjacent columns (quad q) x 16 rows (half h) of a 32-row block rb; the
            // other 16 rows of the block sit in lane ^ 16 of the same warp.  8-byte shared loads;
            // each half-warp reads 16 quads of one row: all 32 banks once.
            const int lane_c = threadIdx.x & 31;
            const int wq = threadIdx.x >> 5;
            const int q = (lane_c & 15) + 16 * (wq & 1);   // column quad: columns 4q .. 4q + 3
            const int h = lane_c >> 4;                     // rows 16h .. 16h + 15 of the block
            const int rb = wq >> 1;                        // 32-row block
            uint2 w[16];
            uint32_t ma[2] = {0u, 0u}, mb[2] = {0u, 0u};   // two independent chains per column pair
    #pragma unroll
            for (int j = 0; j < 16; ++j) {
                w[j] = *reinterpret_cast<const uint2*>(tile + (rb * 32 + h * 16 + j) * 256 + q * 8);
                ma[j & 1] = amax_bf16x2(ma[j & 1], w[j].x);
                mb[j & 1] = amax_bf16x2(mb[j & 1], w[j].y);
            }
            uint32_t m01 = amax_bf16x2(ma[0], ma[1]), m23 = amax_bf16x2(mb[0], mb[1]);
            m01 = amax_bf16x2(m01, __shfl_xor_sync(0xffffffffu, m01, 16));
            m23 = amax_bf16x2(m23, __shfl_xor_sync(0xffffffffu, m23, 16));
            const uint32_t bcol[4] = {scale_byte_bf16<RULE>(m01 & 0x7FFFu), scale_byte_bf16<RULE>((m01 >> 16) & 0x7FFFu),
                                      scale_byte_bf16<RULE>(m23 & 0x7FFFu), scale_byte_bf16<RULE>((m23 >> 16) & 0x7FFFu)};
            const int64_t c0 = col0 + 4 * q;
    #pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float s = inv_scale(bcol[c]);
                uint32_t o[4];
    #pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v[4];
    #pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t word = (c < 2) ? w[4 * j + i].x : w[4 * j + i].y;
                        v[i] = (c & 1) ? bf16_hi(word) : bf16_lo(word);
                    }
                    // scalar products here: the packed mul.f32x2 needs its operands in register
                    // pairs, which in this pass cost moves and spills (scalar: 2 % faster, no spills)
                    const uint32_t a01 = cvt_e4m3x4(v[0] * s, v[1] * s, v[2] * s, v[3] * s);
                    o[j] = bcol[c] == 0xFFu ? 0x7F7F7F7Fu : a01;
                }
                if (c0 + c < p.cols)
                    *reinterpret_cast<uint4*>((p.q_col + col0 * p.ld_col + rt * p.qc_pstep) + (4 * q + c) * p.qc_ld + rb * 32 + h * 16) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                if (h == 0) {
                    const int cc = 4 * q + c;
                    sf_atom_col[(cc & 31) * 16 + (cc >> 5) * 4 + rb] = static_cast<uint8_t>(bcol[c]);
                }
            }
        }
    }

    __syncthreads();
    constexpr int kRowCopies = (SFC & 1) ? 4 : 1, kColCopies = (SFC & 2) ? 4 : 1;
    if (threadIdx.x < 32) {
        if (ROW) {
            uint8_t* dst = p.sf_row + (rt * p.n_col_tiles + ct) * 512 * kRowCopies;
#pragma unroll
            for (int c = 0; c < kRowCopies; ++c)
                reinterpret_cast<uint4*>(dst + 512 * c)[threadIdx.x] = reinterpret_cast<const uint4*>(sf_atom_row)[threadIdx.x];
        }
    } else if (threadIdx.x < 64) {
        if (COL) {
            const int t = threadIdx.x - 32;
            uint8_t* dst = p.sf_col + (ct * (p.ld_col / 128) + rt) * 512 * kColCopies;
#pragma unroll
            for (int c = 0; c < kColCopies; ++c)
                reinterpret_cast<uint4*>(dst + 512 * c)[t] = reinterpret_cast<const uint4*>(sf_atom_col)[t];
        }
    }
}


// ---------------------------------------------------------------------------------
// fp32-input variant (the quantizer benchmark pseudo-code of the lpnh.cn page, section
// "4. 验证请求与成功结果…", reads float input).  Same tiles, outputs and scale layout; a
// warp covers one 128-column row (512 bytes) per load, 8 lanes per 32-element block.  The
// tile is taken in two halves of 64 rows (two 32-row column blocks each) through a 32 KiB
// shared-memory buffer, so that 4 CTAs fit on an SM.
// Position of 16-byte chunk c (0..31, four columns) of row lr of the fp32 half tile.  The row
// group term 2 ((lr >> 4) & 3) lets the column pass read 4 row groups x 2 chunks in one bank
// sweep; folding bit 3 of c into bit 0 gives the 8 lanes of one 16-byte store phase of the full
// path (chunks 2 c8 or 2 c8 + 1, c8 = 0..7) 8 different bank groups.
__device__ __forceinline__ int f32_chunk(int c, int lr) { return c ^ ((c >> 3) & 1) ^ (2 * ((lr >> 4) & 3)); }

template <bool ROW, bool COL, int RULE, int SFC>
__global__ void __launch_bounds__(kThreads, 4) quantize_tile_f32_kernel(const QuantParams p) {
    __shared__ __align__(16) uint8_t sf_atom_row[512];
    __shared__ __align__(16) uint8_t sf_atom_col[512];
    extern __shared__ __align__(16) uint8_t tile[];   // [64][512 bytes], columnwise only
    const float* x = reinterpret_cast<const float*>(p.x);
    const int64_t bid = blockIdx.x;
    const int64_t ct = p.col_major ? bid / p.n_row_tiles : bid % p.n_col_tiles;
    const int64_t rt = p.col_major ? bid % p.n_row_tiles : bid / p.n_col_tiles;
    const int64_t p0 = rt * kTileRows;
    const int64_t col0 = ct * kTileCols;
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
    if ((ROW && p0 + kTileRows > p.pbound) || (COL && p0 + kTileRows > p.ld_col)) {
        if (threadIdx.x == 0 && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
        return;
    }
    valid = valid < 0 ? 0 : (valid > kTileRows ? kTileRows : valid);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t gcol = col0 + lane * 4;
    const bool col_ok = gcol < p.cols;
    const bool full = valid == kTileRows && col0 + kTileCols <= p.cols;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        if (full && p.lean) {
            // full tile, x 32-byte aligned: lane l holds 8 columns (one 256-bit load; chunk
            // c8 = l & 15) of row l >> 4 of each of 4 row pairs, so a warp reads two whole rows
            // per instruction and a 32-column block spans 4 lanes (two shuffles)
            const int c8 = lane & 15;
            uint32_t xv[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = half * 64 + u * 16 + warp * 2 + (lane >> 4);
                int64_t src = row0 + r;
                bool in_range = true;
                if (p.src_row != nullptr) {
                    src = __ldg(p.src_row + row0 + r);
                    in_range = src >= 0 && src < p.src_rows;
                    if (!in_range && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
                }
                if (in_range) {
                    ld_stream_32(x + src * p.cols + col0 + 8 * c8, xv[u]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) xv[u][i] = 0u;
                }
            }
            if (COL && half == 1) __syncthreads();   // the first half's column pass has read the buffer
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int lr = u * 16 + warp * 2 + (lane >> 4);   // row within the half
                const int r = half * 64 + lr;
                if (COL) {
                    *reinterpret_cast<uint4*>(tile + lr * 512 + f32_chunk(2 * c8, lr) * 16) =
                        make_uint4(xv[u][0], xv[u][1], xv[u][2], xv[u][3]);
                    *reinterpret_cast<uint4*>(tile + lr * 512 + f32_chunk(2 * c8 + 1, lr) * 16) =
                        make_uint4(xv[u][4], xv[u][5], xv[u][6], xv[u][7]);
                }
                if (ROW) {
                    uint32_t m = 0u;
#pragma unroll
                    for (int i = 0; i < 8; ++i) m = max(m, xv[u][i] & 0x7FFFFFFFu);
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    const uint32_t b = scale_byte_f32<RULE>(m);
                    const float sc = inv_scale_or_nan(b);   // a NaN/Inf block: NaN scale, codes 0x7F
                    const uint32_t q0 = quant_quad_f32(__uint_as_float(xv[u][0]), __uint_as_float(xv[u][1]),
                                                       __uint_as_float(xv[u][2]), __uint_as_float(xv[u][3]), sc);
                    const uint32_t q1 = quant_quad_f32(__uint_as_float(xv[u][4]), __uint_as_float(xv[u][5]),
                                                       __uint_as_float(xv[u][6]), __uint_as_float(xv[u][7]), sc);
                    *reinterpret_cast<uint2*>(p.q_row + row0 * p.cols + ct * p.qr_cstep + r * p.qr_ld + 8 * c8) =
                        make_uint2(q0, q1);
                    if ((c8 & 3) == 0) sf_atom_row[(r & 31) * 16 + (r >> 5) * 4 + (c8 >> 2)] = static_cast<uint8_t>(b);
                }
            }
        } else {
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = (half * 8 + i) * 8 + warp;
            v[i] = make_uint4(0u, 0u, 0u, 0u);
            if (r < valid && col_ok) {
                int64_t src = row0 + r;
                bool in_range = true;
                if (p.src_row != nullptr) {
                    src = __ldg(p.src_row + row0 + r);
                    in_range = src >= 0 && src < p.src_rows;
                    if (!in_range && p.dev_err) atomicOr(p.dev_err, MX_DEVERR_BAD_SEGMENTS);
                }
                if (in_range) v[i] = ld_stream_16(x + src * p.cols + gcol);
            }
        }
        if (COL && half == 1) __syncthreads();   // the first half's column pass has read the buffer
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = (half * 8 + i) * 8 + warp;
            const int lr = i * 8 + warp;   // row within the half
            if (COL) *reinterpret_cast<uint4*>(tile + lr * 512 + f32_chunk(lane, lr) * 16) = v[i];
            if (ROW) {
                uint32_t m = max(max(v[i].x & 0x7FFFFFFFu, v[i].y & 0x7FFFFFFFu), max(v[i].z & 0x7FFFFFFFu, v[i].w & 0x7FFFFFFFu));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
                const uint32_t b = scale_byte_f32<RULE>(m);
                const float sc = inv_scale_or_nan(b);   // a NaN/Inf block: NaN scale, codes 0x7F
                const uint32_t q = quant_quad_f32(__uint_as_float(v[i].x), __uint_as_float(v[i].y),
                                                  __uint_as_float(v[i].z), __uint_as_float(v[i].w), sc);
                if (r < valid && col_ok) *reinterpret_cast<uint32_t*>(p.q_row + row0 * p.cols + ct * p.qr_cstep + r * p.qr_ld + lane * 4) = q;
                if ((lane & 7) == 0) sf_atom_row[(r & 31) * 16 + (r >> 5) * 4 + (lane >> 3)] = static_cast<uint8_t>(b);
            }
        }
        }
        if (!COL) continue;
        __syncthreads();
        if (full) {
            // lane = (column pair qi, row group g of 16 rows of the half): a thread takes 2
            // adjacent columns x 16 rows (8-byte reads; with the swizzle each 16-lane phase meets
            // every bank once), the 32-row block's other 16 rows in lane ^ 1; the 4 lanes of a
            // pair write one column's 64 positions of the half contiguously
            const int g = lane & 3;
            const int pi = 8 * warp + (lane >> 2);   // columns 2 pi, 2 pi + 1
            const uint8_t* tb = tile + g * 16 * 512 + f32_chunk(pi >> 1, 16 * g) * 16 + (pi & 1) * 8;
            float v0[16], v1[16];
            uint32_t m0 = 0u, m1 = 0u;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint2 w = *reinterpret_cast<const uint2*>(tb + j * 512);
                v0[j] = __uint_as_float(w.x);
                v1[j] = __uint_as_float(w.y);
                m0 = max(m0, w.x & 0x7FFFFFFFu);
                m1 = max(m1, w.y & 0x7FFFFFFFu);
            }
            m0 = max(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
            m1 = max(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
            uint8_t* qc = (p.q_col + col0 * p.ld_col + rt * p.qc_pstep) + half * 64 + 16 * g;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t b = scale_byte_f32<RULE>(c ? m1 : m0);
                const float sc = inv_scale_or_nan(b);
                const float* vv = c ? v1 : v0;
                uint32_t o[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    o[k] = quant_quad_f32(vv[4 * k], vv[4 * k + 1], vv[4 * k + 2], vv[4 * k + 3], sc);
                const int cc = 2 * pi + c;
                *reinterpret_cast<uint4*>(qc + cc * p.qc_ld) = make_uint4(o[0], o[1], o[2], o[3]);
                if ((g & 1) == 0)
                    sf_atom_col[(cc & 31) * 16 + (cc >> 5) * 4 + half * 2 + (g >> 1)] = static_cast<uint8_t>(b);
            }
        } else {
            // ragged tile: one column's 32-row block per task, the half's two blocks
#pragma unroll 1
            for (int task = threadIdx.x; task < 256; task += kThreads) {
                const int c = task & 127;
                const int hb = task >> 7;   // block within the half
                uint32_t w[32];
                uint32_t m = 0;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int lr = hb * 32 + j;
                    w[j] = *reinterpret_cast<const uint32_t*>(tile + lr * 512 + f32_chunk(c >> 2, lr) * 16 + (c & 3) * 4);
                    m = max(m, w[j] & 0x7FFFFFFFu);
                }
                const uint32_t b = scale_byte_f32<RULE>(m);
                const int rb = half * 2 + hb;
                const int64_t gc = col0 + c;
                if (gc < p.cols) {
                    uint32_t o[8];
                    const float sc = inv_scale_or_nan(b);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        o[j] = quant_quad_f32(__uint_as_float(w[4 * j]), __uint_as_float(w[4 * j + 1]),
                                              __uint_as_float(w[4 * j + 2]), __uint_as_float(w[4 * j + 3]), sc);
                    uint8_t* dst = (p.q_col + col0 * p.ld_col + rt * p.qc_pstep) + c * p.qc_ld + rb * 32;
                    reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
                    reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
                }
                sf_atom_col[(c & 31) * 16 + (c >> 5) * 4 + rb] = static_cast<uint8_t>(b);
            }
        }
    }
    __syncthreads();
    constexpr int kRowCopies = (SFC & 1) ? 4 : 1, kColCopies = (SFC & 2) ? 4 : 1;
    if (threadIdx.x < 32) {
        if (ROW) {
            uint8_t* dst = p.sf_row + (rt * p.n_col_tiles + ct) * 512 * kRowCopies;
#pragma unroll
            for (int c = 0; c < kRowCopies; ++c)
                reinterpret_cast<uint4*>(dst + 512 * c)[threadIdx.x] = reinterpret_cast<const uint4*>(sf_atom_row)[threadIdx.x];
        }
    } else if (threadIdx.x < 64) {
        if (COL) {
            const int t = threadIdx.x - 32;
            uint8_t* dst = p.sf_col + (ct * (p.ld_col / 128) + rt) * 512 * kColCopies;
#pragma unroll
            for (int c = 0; c < kColCopies; ++c)
                reinterpret_cast<uint4*>(dst + 512 * c)[t] = reinterpret_cast<const uint4*>(sf_atom_col)[t];
        }
    }
}

template <bool ROW, bool COL, int RULE, int SFC>
cudaError_t launch_bf16_one(unsigned blocks, size_t smem, const QuantParams& p, cudaStream_t stream) {
    if (p.row_scale != nullptr) {
        if constexpr (RULE == 0) {
            quantize_tile_kernel<ROW, COL, RULE, SFC, true><<<blocks, kThreads, smem, stream>>>(p);
            return cudaSuccess;
        }
        return cudaErrorInvalidValue;   // the API allows row scales with the floor rule only
    }
    quantize_tile_kernel<ROW, COL, RULE, SFC><<<blocks, kThreads, smem, stream>>>(p);
    return cudaSuccess;
}

template <bool ROW, bool COL, int RULE, int SFC>
cudaError_t launch_f32_one(unsigned blocks, size_t /*smem*/, const QuantParams& p, cudaStream_t stream) {
    const size_t smem = COL ? (kTileRows / 2) * 512 : 0;   // one 64-row half of the fp32 tile
    static bool attr_done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (COL && !attr_done[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(quantize_tile_f32_kernel<ROW, COL, RULE, SFC>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    quantize_tile_f32_kernel<ROW, COL, RULE, SFC><<<blocks, kThreads, smem, stream>>>(p);
    return cudaSuccess;
}

// mode (forms plus four-copy bits, validated by the caller) -> the kernel instantiation
template <bool F32, int RULE>
cudaError_t launch_mode(int mode, unsigned blocks, size_t smem, const QuantParams& p, cudaStream_t stream) {
#define MX_QL(R, C, S)                                                         \
    do {                                                                       \
        if constexpr (F32) return launch_f32_one<R, C, RULE, S>(blocks, smem, p, stream); \
        else return launch_bf16_one<R, C, RULE, S>(blocks, smem, p, stream);   \
    } while (0)
    const int sfc = ((mode & MX_ROWWISE_X4) ? 1 : 0) | ((mode & MX_COLWISE_X4) ? 2 : 0);
    switch (mode & (MX_ROWWISE | MX_COLWISE)) {
        case MX_ROWWISE:
            if (sfc & 1) MX_QL(true, false, 1);
            MX_QL(true, false, 0);
        case MX_COLWISE:
            if (sfc & 2) MX_QL(false, true, 2);
            MX_QL(false, true, 0);
        default:
            switch (sfc) {
                case 1: MX_QL(true, true, 1);
                case 2: MX_QL(true, true, 2);
                case 3: MX_QL(true, true, 3);
                default: MX_QL(true, true, 0);
            }
    }
#undef MX_QL
}

}  // namespace

int launch_quantize(const void* x, int dtype, int rule, const int32_t* src_row, const float* row_scale,
                    int64_t src_rows, int64_t rows, int64_t cols, int mode, const int32_t* seg_off,
                    const int32_t* seg_poff, int nseg, int64_t ld_col, int64_t pbound, uint8_t* q_row,
                    uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col, int* dev_err, cudaStream_t stream) {
    QuantParams p;
    p.x = static_cast<const uint16_t*>(x);
    p.src_row = src_row;
    p.row_scale = row_scale;
    p.src_rows = src_rows;
    p.rows = rows;
    p.cols = cols;
    p.q_row = q_row;
    p.sf_row = sf_row;
    p.q_col = q_col;
    p.sf_col = sf_col;
    p.ld_col = ld_col;
    p.seg_off = seg_off;
    p.seg_poff = seg_poff;
    p.nseg = nseg;
    p.pbound = pbound;
    p.n_col_tiles = (cols + kTileCols - 1) / kTileCols;
    p.dev_err = dev_err;
    p.lean = (reinterpret_cast<uintptr_t>(x) & 31) == 0;
    const int64_t n_row_tiles = pbound / kTileRows;
    p.n_row_tiles = n_row_tiles;
    p.col_major = src_row != nullptr ? 1 : 0;
    const bool blk_row = (mode & MX_ROWWISE_BLK) != 0, blk_col = (mode & MX_COLWISE_BLK) != 0;
    p.qr_cstep = blk_row ? 16384 : kTileCols;
    p.qr_ld = blk_row ? 128 : cols;
    p.qc_pstep = blk_col ? 16384 : kTileRows;
    p.qc_ld = blk_col ? 128 : ld_col;
    const int64_t blocks = n_row_tiles * p.n_col_tiles;
    if (blocks <= 0) return MX_OK;
    if (blocks > 0x7FFFFFFFLL) return MX_ERR_UNSUPPORTED;
    const unsigned nb = static_cast<unsigned>(blocks);
    const size_t smem = (mode & MX_COLWISE) ? kTileRows * 256 : 0;   // bf16 tile (the f32 kernel sizes its own)
    const bool f32 = dtype == MX_DTYPE_F32;
    const cudaError_t e = rule == MX_SCALE_RCEIL
                              ? (f32 ? launch_mode<true, 1>(mode, nb, smem, p, stream) : launch_mode<false, 1>(mode, nb, smem, p, stream))
                              : (f32 ? launch_mode<true, 0>(mode, nb, smem, p, stream) : launch_mode<false, 0>(mode, nb, smem, p, stream));
    if (e != cudaSuccess) return MX_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

}  // namespace mx
