// combine.cu -- unpermute / combine: the weighted merge of the expert outputs back to
// token order, and its backward (kucoin.com, "Cursor's MoK демонстрирует повышение
// производительности на 2,37x на NVIDIA GB300 NVL72", section "03": the measured MoE layer
// ends with combine and the final weighted merge).
//
//   forward   out[t] = bf16( sum_j gate[t][j] * Y[dst_of[t][j]] )          fp32 accumulation
//   backward  dY[dst_of[t][j]] = bf16( gate[t][j] * dOut[t] )             (optional)
//             dgate[t][j]      = sum_h dOut[t][h] * Y[dst_of[t][j]][h]     fp32, fixed-order tree
//             gate_rows[dst_of[t][j]] = gate[t][j]                          (optional: the routing
//             weight of every routed row, for a quantize-on-gather that forms dY itself)
//
// One CTA per token; 16-byte vector loads of bf16 rows.  Both passes are bound by HBM
// (per token: k routed rows read, one row written; backward: k rows read and k written, dOut
// read once).
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "mxmoe_internal.h"

namespace mx {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxK = 64;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    f[4] = __uint_as_float(v.z << 16);
    f[5] = __uint_as_float(v.z & 0xFFFF0000u);
    f[6] = __uint_as_float(v.w << 16);
    f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// Destination rows and gates of token t into shared memory; rows outside [0, R) are
// dropped (and flagged).
__device__ __forceinline__ void load_routes(const float* gate, const int32_t* dst_of, int64_t t, int k, int64_t R,
                                            int* dev_err, int32_t* sd, float* sg) {
    if (threadIdx.x < k) {
        int32_t d = __ldg(dst_of + t * k + threadIdx.x);
        if (d >= R) {
            if (dev_err) atomicOr(dev_err, MX_DEVERR_BAD_SEGMENTS);
            d = -1;
        }
        sd[threadIdx.x] = d < 0 ? -1 : d;
        sg[threadIdx.x] = gate != nullptr ? __ldg(gate + t * k + threadIdx.x) : 1.0f;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads) combine_fwd_kernel(const uint4* __restrict__ Y,
                                                               const float* __restrict__ gate,
                                                               const int32_t* __restrict__ dst_of, int k,
                                                               int64_t Hc, int64_t R, uint4* __restrict__ out,
                                                               int* dev_err) {
    __shared__ int32_t sd[kMaxK];
    __shared__ float sg[kMaxK];
    const int64_t t = blockIdx.x;
    load_routes(gate, dst_of, t, k, R, dev_err, sd, sg);
    for (int64_t c = threadIdx.x; c < Hc; c += kThreads) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int j = 0; j < k; ++j) {
            const int32_t d = sd[j];
            if (d < 0) continue;
            float y[8];
            bf16x8_to_f32(__ldg(Y + d * Hc + c), y);
            const float g = sg[j];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, y[i], acc[i]);
        }
        out[t * Hc + c] = f32x8_to_bf16(acc);
    }
}

__global__ void __launch_bounds__(kThreads) combine_bwd_kernel(const uint4* __restrict__ dOut,
                                                               const uint4* __restrict__ Y,
                                                               const float* __restrict__ gate,
                                                               const int32_t* __restrict__ dst_of, int k,
                                                               int64_t Hc, int64_t R, uint4* __restrict__ dY,
                                                               float* __restrict__ dgate,
                                                               float* __restrict__ gate_rows, int* dev_err) {
    // One pass over the token's dOut row per group of 8 routes: each 16-byte piece of dOut is
    // read once and serves the dot products (and dY pieces) of all routes of the group, whose
    // Y pieces are in flight together.  Per route the summation order is that of a loop over
    // the route alone: a thread's pieces in order, then the warp tree, then the warps in order.
    constexpr int kGroup = 8;
    __shared__ int32_t sd[kMaxK];
    __shared__ float sg[kMaxK];
    __shared__ float red[kThreads / 32][kGroup];
    const int64_t t = blockIdx.x;
    load_routes(gate, dst_of, t, k, R, dev_err, sd, sg);
    if (gate_rows != nullptr && threadIdx.x < k && sd[threadIdx.x] >= 0) gate_rows[sd[threadIdx.x]] = sg[threadIdx.x];
    for (int j0 = 0; j0 < k; j0 += kGroup) {
        float dot[kGroup];
#pragma unroll
        for (int jj = 0; jj < kGroup; ++jj) dot[jj] = 0.f;
        for (int64_t c = threadIdx.x; c < Hc; c += kThreads) {
            float o[8];
            bf16x8_to_f32(__ldg(dOut + t * Hc + c), o);
            uint4 yv[kGroup];
#pragma unroll
            for (int jj = 0; jj < kGroup; ++jj) {
                const int j = j0 + jj;
                const int32_t d = j < k ? sd[j] : -1;
                yv[jj] = d >= 0 ? __ldg(Y + d * Hc + c) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int jj = 0; jj < kGroup; ++jj) {
                const int j = j0 + jj;
                const int32_t d = j < k ? sd[j] : -1;
                if (d < 0) continue;
                float y[8];
                bf16x8_to_f32(yv[jj], y);
#pragma unroll
                for (int i = 0; i < 8; ++i) dot[jj] = fmaf(o[i], y[i], dot[jj]);
                if (dY != nullptr) {
                    const float g = sg[j];
                    float sv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) sv[i] = g * o[i];
                    dY[d * Hc + c] = f32x8_to_bf16(sv);
                }
            }
        }
#pragma unroll
        for (int jj = 0; jj < kGroup; ++jj) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot[jj] += __shfl_xor_sync(0xffffffffu, dot[jj], off);
        }
        if ((threadIdx.x & 31) == 0) {
#pragma unroll
            for (int jj = 0; jj < kGroup; ++jj) red[threadIdx.x >> 5][jj] = dot[jj];
        }
        __syncthreads();
        if (threadIdx.x < kGroup && j0 + threadIdx.x < k) {
            const int j = j0 + threadIdx.x;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) sum += red[w][threadIdx.x];
            dgate[t * k + j] = sd[j] < 0 ? 0.f : sum;
        }
        __syncthreads();
    }
}

}  // namespace

int launch_combine_fwd(const void* Y, const float* gate, const int32_t* dst_of, int64_t T, int k, int64_t H,
                       int64_t R, void* out, int* dev_err, cudaStream_t stream) {
    if (T == 0) return MX_OK;
    combine_fwd_kernel<<<static_cast<unsigned>(T), kThreads, 0, stream>>>(
        static_cast<const uint4*>(Y), gate, dst_of, k, H / 8, R, static_cast<uint4*>(out), dev_err);
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

int launch_combine_bwd(const void* dOut, const void* Y, const float* gate, const int32_t* dst_of, int64_t T, int k,
                       int64_t H, int64_t R, void* dY, float* dgate, float* gate_rows, int* dev_err,
                       cudaStream_t stream) {
    if (T == 0) return MX_OK;
    combine_bwd_kernel<<<static_cast<unsigned>(T), kThreads, 0, stream>>>(
        static_cast<const uint4*>(dOut), static_cast<const uint4*>(Y), gate, dst_of, k, H / 8, R,
        static_cast<uint4*>(dY), dgate, gate_rows, dev_err);
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

}  // namespace mx
