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
// The elementwise values are computed in fp32 (expf, IEEE division) and quantized from
// fp32 with the same scale rule and 128 x 128 tiles as the quantizer: rowwise codes with
// one complete 512-byte scale atom per tile, columnwise through a shared-memory fp32 tile.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "mxmoe_internal.h"
#include "quant_common.cuh"

namespace mx {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;

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
    int64_t n_col_tiles;
    int* dev_err;
};

__device__ __forceinline__ float sigmoidf_(float g) { return 1.0f / (1.0f + expf(-g)); }

// Eight fp32 results for output columns [oc, oc + 8) of row r (input row `src`).
template <bool BWD>
__device__ __forceinline__ void swiglu8(const SwigluParams& p, int64_t src, int64_t oc, float (&o)[8]) {
    const bool up_part = BWD && oc >= p.I;
    const int64_t c = up_part ? oc - p.I : oc;                    // column within [0, I)
    const uint4 gv = ld_stream_16(p.a + src * 2 * p.I + c);
    const uint4 uv = ld_stream_16(p.a + src * 2 * p.I + p.I + c);
    float g[8], u[8];
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        g[2 * i] = bf16_lo(gw[i]);
        g[2 * i + 1] = bf16_hi(gw[i]);
        u[2 * i] = bf16_lo(uw[i]);
        u[2 * i + 1] = bf16_hi(uw[i]);
    }
    if (!BWD) {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = g[i] * sigmoidf_(g[i]) * u[i];
    } else {
        const uint4 dv = ld_stream_16(p.dh + src * p.I + c);
        const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
        float d[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            d[2 * i] = bf16_lo(dw[i]);
            d[2 * i + 1] = bf16_hi(dw[i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float s = sigmoidf_(g[i]);
            o[i] = up_part ? d[i] * (g[i] * s) : d[i] * u[i] * (s * (1.0f + g[i] * (1.0f - s)));
        }
    }
}

template <bool BWD, bool ROW, bool COL>
__global__ void __launch_bounds__(kThreads) swiglu_quant_kernel(const SwigluParams p) {
    __shared__ __align__(16) uint8_t sf_atom_row[512];
    __shared__ __align__(16) uint8_t sf_atom_col[512];
    extern __shared__ __align__(16) uint8_t tile[];   // [128][512 bytes] fp32, columnwise only

    const int64_t bid = blockIdx.x;
    const int64_t ct = bid % p.n_col_tiles;
    const int64_t rt = bid / p.n_col_tiles;
    const int64_t p0 = rt * kTile;
    const int64_t col0 = ct * kTile;
    int64_t row0, valid;
    if (p.nseg == 0) {
        row0 = p0;
        valid = p.rows - p0;
    } else {
        const int32_t ptotal = __ldg(p.seg_poff + p.nseg);
        if (p0 >= ptotal) return;
        int lo = 0, hi = p.nseg - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.seg_poff + mid) <= p0) lo = mid; else hi = mid - 1;
        }
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
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunk = lane & 15;           // 8 output columns
    const int64_t oc = col0 + chunk * 8;

#pragma unroll 2
    for (int i = 0; i < 8; ++i) {
        const int r = i * 16 + warp * 2 + (lane >> 4);
        float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (r < valid) swiglu8<BWD>(p, row0 + r, oc, o);
        if (COL) {
            float4* t4 = reinterpret_cast<float4*>(tile + r * 512 + chunk * 32);
            t4[0] = make_float4(o[0], o[1], o[2], o[3]);
            t4[1] = make_float4(o[4], o[5], o[6], o[7]);
        }
        if (ROW) {
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) m = max(m, __float_as_uint(o[j]) & 0x7FFFFFFFu);
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const uint32_t b = scale_byte_f32<0>(m);
            uint2 q = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
            if (b != 0xFFu) {
                const float sc = inv_scale(b);
                const uint32_t c0 = quant_pair2(o[0], o[1], sc), c1 = quant_pair2(o[2], o[3], sc);
                const uint32_t c2 = quant_pair2(o[4], o[5], sc), c3 = quant_pair2(o[6], o[7], sc);
                q = make_uint2(__byte_perm(c0, c1, 0x5410), __byte_perm(c2, c3, 0x5410));
            }
            if (r < valid) *reinterpret_cast<uint2*>(p.q_row + (row0 + r) * p.ncols + oc) = q;
            if ((chunk & 3) == 0) sf_atom_row[(r & 31) * 16 + (r >> 5) * 4 + (chunk >> 2)] = static_cast<uint8_t>(b);
        }
    }
    if (COL) {
        __syncthreads();
#pragma unroll 1
        for (int task = threadIdx.x; task < 512; task += kThreads) {
            const int c = task & 127;
            const int rb = task >> 7;
            float w[32];
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                w[j] = *reinterpret_cast<const float*>(tile + (rb * 32 + j) * 512 + c * 4);
                m = max(m, __float_as_uint(w[j]) & 0x7FFFFFFFu);
            }
            const uint32_t b = scale_byte_f32<0>(m);
            uint32_t o[8];
            const float sc = inv_scale(b);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t a0 = quant_pair2(w[4 * j], w[4 * j + 1], sc);
                const uint32_t a1 = quant_pair2(w[4 * j + 2], w[4 * j + 3], sc);
                o[j] = b == 0xFFu ? 0x7F7F7F7Fu : __byte_perm(a0, a1, 0x5410);
            }
            uint8_t* dst = p.q_col + (col0 + c) * p.ld_col + p0 + rb * 32;
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
            sf_atom_col[(c & 31) * 16 + (c >> 5) * 4 + rb] = static_cast<uint8_t>(b);
        }
    }
    __syncthreads();
    if (ROW && threadIdx.x < 32) {
        uint8_t* dst = p.sf_row + (rt * p.n_col_tiles + ct) * 512;
        reinterpret_cast<uint4*>(dst)[threadIdx.x] = reinterpret_cast<const uint4*>(sf_atom_row)[threadIdx.x];
    }
    if (COL && threadIdx.x >= 32 && threadIdx.x < 64) {
        const int q = threadIdx.x - 32;
        uint8_t* dst = p.sf_col + (ct * (p.ld_col / 128) + rt) * 512;
        reinterpret_cast<uint4*>(dst)[q] = reinterpret_cast<const uint4*>(sf_atom_col)[q];
    }
}

template <bool BWD, bool ROW, bool COL>
cudaError_t launch_one(unsigned blocks, const SwigluParams& p, cudaStream_t stream) {
    const int smem = COL ? kTile * 512 : 0;
    static bool attr_done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (COL && !attr_done[dev]) {
        const cudaError_t e =
            cudaFuncSetAttribute(swiglu_quant_kernel<BWD, ROW, COL>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    swiglu_quant_kernel<BWD, ROW, COL><<<blocks, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <bool BWD>
cudaError_t launch_mode(int mode, unsigned blocks, const SwigluParams& p, cudaStream_t stream) {
    switch (mode) {
        case MX_ROWWISE: return launch_one<BWD, true, false>(blocks, p, stream);
        case MX_COLWISE: return launch_one<BWD, false, true>(blocks, p, stream);
        default: return launch_one<BWD, true, true>(blocks, p, stream);
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
    p.n_col_tiles = p.ncols / kTile;
    p.dev_err = dev_err;
    const int64_t blocks = (pbound / kTile) * p.n_col_tiles;
    if (blocks <= 0) return MX_OK;
    if (blocks > 0x7FFFFFFFLL) return MX_ERR_UNSUPPORTED;
    const cudaError_t e = bwd ? launch_mode<true>(mode, static_cast<unsigned>(blocks), p, stream)
                              : launch_mode<false>(mode, static_cast<unsigned>(blocks), p, stream);
    return e == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

}  // namespace mx
