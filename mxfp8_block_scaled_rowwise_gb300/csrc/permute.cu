// permute.cu -- token permutation by expert for sm_103a.
//
// kucoin.com, "Cursor's MoK демонстрирует повышение производительности на 2,37x на NVIDIA
// GB300 NVL72", section "01": before expert compute, count the tokens each expert
// receives, decide where each one goes, and keep one expert's tokens contiguous.
//
// Four small kernels, all deterministic (integer counts only, no ordering races):
//   1. histogram  -- each CTA counts the routed slots of its 2048-slot chunk per
//                    expert (shared-memory integer atomics) -> ws.blk_counts[b][e];
//   2. scan       -- one CTA: per expert, exclusive scan of the chunk counts over
//                    chunks (-> ws.blk_base), then exclusive scans over experts of
//                    the counts (off) and of the 128-padded counts (poff);
//   3. rank       -- each CTA re-reads its chunk; a warp owns 256 consecutive slots,
//                    per-warp per-expert counts (warp match + popcount) are scanned
//                    across the CTA's warps, then every slot gets
//                    off[e] + blk_base + warp base + rank among earlier equal lanes.
//                    The resulting order inside an expert is ascending slot index
//                    t*k + j, i.e. by token then slot: a stable counting sort;
//   4. gather     -- optional: one warp per padded destination row copies the E4M3
//                    row and moves its scale words from the source row's position in
//                    the tensor-core scale layout to the destination's padded row;
//                    padding rows get zero scales.
// A problem of one chunk (T*k <= 2048 slots) runs steps 1-3 in a single CTA and launch.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "mxmoe_internal.h"

namespace mx {
namespace {

constexpr int kChunk = 2048;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 1024;

__global__ void __launch_bounds__(kThreads) hist_kernel(const int32_t* __restrict__ ids, int64_t n, int E,
                                                        int32_t* __restrict__ blk_counts, int* dev_err) {
    __shared__ int32_t cnt[kMaxE];
    for (int e = threadIdx.x; e < E; e += kThreads) cnt[e] = 0;
    __syncthreads();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kChunk;
    bool bad = false;
    for (int j = threadIdx.x; j < kChunk; j += kThreads) {
        const int64_t i = base + j;
        if (i < n) {
            const int32_t e = __ldg(ids + i);
            if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
            else bad = true;
        }
    }
    if (bad) atomicOr(dev_err, MX_DEVERR_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads)
        blk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = cnt[e];
}

__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ blk_counts,
                                                    int32_t* __restrict__ blk_base, int64_t nblk, int E,
                                                    int64_t n, int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ off, int32_t* __restrict__ poff,
                                                    int32_t* __restrict__ src_row) {
    __shared__ int32_t s_warp[2][32];
    const int e = threadIdx.x;
    int32_t total = 0;
    if (e < E) {
        for (int64_t b = 0; b < nblk; ++b) {
            const int32_t v = blk_counts[b * E + e];
            blk_base[b * E + e] = total;
            total += v;
        }
        counts[e] = total;
    }
    // block-wide exclusive scans of total and ceil128(total) over experts
    int32_t a = (e < E) ? total : 0;
    int32_t p = (e < E) ? ((total + 127) / 128) * 128 : 0;
    const int lane = e & 31, warp = e >> 5;
    int32_t ia = a, ip = p;   // inclusive within warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t ta = __shfl_up_sync(0xffffffffu, ia, d);
        const int32_t tp = __shfl_up_sync(0xffffffffu, ip, d);
        if (lane >= d) { ia += ta; ip += tp; }
    }
    if (lane == 31) { s_warp[0][warp] = ia; s_warp[1][warp] = ip; }
    __syncthreads();
    if (warp == 0) {
        int32_t wa = s_warp[0][lane], wp = s_warp[1][lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t ta = __shfl_up_sync(0xffffffffu, wa, d);
            const int32_t tp = __shfl_up_sync(0xffffffffu, wp, d);
            if (lane >= d) { wa += ta; wp += tp; }
        }
        s_warp[0][lane] = wa;   // inclusive over warps
        s_warp[1][lane] = wp;
    }
    __syncthreads();
    const int32_t wa0 = warp > 0 ? s_warp[0][warp - 1] : 0;
    const int32_t wp0 = warp > 0 ? s_warp[1][warp - 1] : 0;
    if (e < E) {
        off[e] = wa0 + ia - a;
        poff[e] = wp0 + ip - p;
    }
    if (e == E - 1) {
        off[E] = wa0 + ia;
        poff[E] = wp0 + ip;
    }
    // rows past the last valid one (only when some ids were invalid) are marked -1
    __syncthreads();
    const int32_t valid_total = s_warp[0][31];
    for (int64_t r = valid_total + threadIdx.x; r < n; r += blockDim.x) src_row[r] = -1;
}

__global__ void __launch_bounds__(kThreads) rank_kernel(const int32_t* __restrict__ ids, int64_t n, int k, int E,
                                                        const int32_t* __restrict__ blk_base,
                                                        const int32_t* __restrict__ off,
                                                        int32_t* __restrict__ src_row,
                                                        int32_t* __restrict__ dst_of) {
    __shared__ int32_t wcnt[kWarps][kMaxE];
    for (int idx = threadIdx.x; idx < kWarps * E; idx += kThreads) wcnt[idx / E][idx % E] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t wbase = static_cast<int64_t>(blockIdx.x) * kChunk + warp * (kChunk / kWarps);
    const uint32_t lt_mask = (1u << lane) - 1u;
    // the warp's ids, all loaded before the first use (one load latency, not one per step; phase
    // C reuses them)
    constexpr int kIters = kChunk / kWarps / 32;
    int32_t ev[kIters];
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int64_t i = wbase + it * 32 + lane;
        ev[it] = (i < n) ? __ldg(ids + i) : -1;
    }

    // phase A: per-warp per-expert counts
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int32_t e = ev[it];
        const bool ok = e >= 0 && e < E;
        const uint32_t peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        if (ok && (peers & lt_mask) == 0) wcnt[warp][e] += __popc(peers);
    }
    __syncthreads();
    // phase B: scan across warps, seeded with the chunk's base inside each expert
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int32_t base = __ldg(off + e) + blk_base[static_cast<int64_t>(blockIdx.x) * E + e];
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int32_t t = wcnt[w][e];
            wcnt[w][e] = base;
            base += t;
        }
    }
    __syncthreads();
    // phase C: final ranks in slot order
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int64_t i = wbase + it * 32 + lane;
        const int32_t e = ev[it];
        const bool ok = e >= 0 && e < E;
        const uint32_t peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        int32_t r = -1;
        if (ok) r = wcnt[warp][e] + __popc(peers & lt_mask);
        __syncwarp();
        if (ok && (peers & lt_mask) == 0) wcnt[warp][e] += __popc(peers);
        __syncwarp();
        if (i < n) {
            dst_of[i] = r;
            if (ok) src_row[r] = static_cast<int32_t>(i / k);
        }
    }
}

// The whole permutation of a problem of at most one chunk (T*k <= 2048 slots) in one CTA: the
// histogram, the scans and the ranks of the three kernels above with the chunk base 0, in one
// launch instead of three (small batches are bound by launch latency).  Same results.
__global__ void __launch_bounds__(kThreads) permute_small_kernel(const int32_t* __restrict__ ids, int64_t n, int k,
                                                                 int E, int32_t* __restrict__ counts,
                                                                 int32_t* __restrict__ off,
                                                                 int32_t* __restrict__ poff,
                                                                 int32_t* __restrict__ src_row,
                                                                 int32_t* __restrict__ dst_of, int* dev_err) {
    __shared__ int32_t wcnt[kWarps][kMaxE];
    __shared__ int32_t s_warp[2][kWarps];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int idx = threadIdx.x; idx < kWarps * E; idx += kThreads) wcnt[idx / E][idx % E] = 0;
    constexpr int kIters = kChunk / kWarps / 32;
    const int64_t wbase = warp * (kChunk / kWarps);
    int32_t ev[kIters];
    bool bad = false;
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int64_t i = wbase + it * 32 + lane;
        ev[it] = (i < n) ? __ldg(ids + i) : -1;
        bad |= i < n && (ev[it] < 0 || ev[it] >= E);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(dev_err, MX_DEVERR_BAD_EXPERT_ID);
    __syncthreads();
    // per-warp per-expert counts
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int32_t e = ev[it];
        const bool ok = e >= 0 && e < E;
        const uint32_t peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        if (ok && (peers & lt_mask) == 0) wcnt[warp][e] += __popc(peers);
    }
    __syncthreads();
    // per expert: the total over warps (counts), then exclusive scans over experts of the totals
    // (off) and of their 128-padded sizes (poff); thread t owns experts [t * per, (t + 1) * per)
    const int per = (E + kThreads - 1) / kThreads;
    const int e0 = threadIdx.x * per;
    int32_t a = 0, pd = 0;
    for (int e = e0; e < e0 + per && e < E; ++e) {
        int32_t tot = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tot += wcnt[w][e];
        counts[e] = tot;
        a += tot;
        pd += (tot + 127) / 128 * 128;
    }
    int32_t ia = a, ip = pd;   // inclusive scans: within the warp, then across warps
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t ta = __shfl_up_sync(0xffffffffu, ia, d);
        const int32_t tp = __shfl_up_sync(0xffffffffu, ip, d);
        if (lane >= d) { ia += ta; ip += tp; }
    }
    if (lane == 31) { s_warp[0][warp] = ia; s_warp[1][warp] = ip; }
    __syncthreads();
    int32_t ra = ia - a, rp = ip - pd;   // exclusive: experts before e0
    for (int w = 0; w < warp; ++w) { ra += s_warp[0][w]; rp += s_warp[1][w]; }
    int32_t total_all = 0, ptotal = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) { total_all += s_warp[0][w]; ptotal += s_warp[1][w]; }
    // the warps' bases inside each expert: off[e] + the counts of the earlier warps
    for (int e = e0; e < e0 + per && e < E; ++e) {
        off[e] = ra;
        poff[e] = rp;
        int32_t base = ra, tot = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int32_t t = wcnt[w][e];
            wcnt[w][e] = base;
            base += t;
            tot += t;
        }
        ra += tot;
        rp += (tot + 127) / 128 * 128;
    }
    if (threadIdx.x == 0) {
        off[E] = total_all;
        poff[E] = ptotal;
    }
    __syncthreads();
    // ranks in slot order
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int64_t i = wbase + it * 32 + lane;
        const int32_t e = ev[it];
        const bool ok = e >= 0 && e < E;
        const uint32_t peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        int32_t r = -1;
        if (ok) r = wcnt[warp][e] + __popc(peers & lt_mask);
        __syncwarp();
        if (ok && (peers & lt_mask) == 0) wcnt[warp][e] += __popc(peers);
        __syncwarp();
        if (i < n) {
            dst_of[i] = r;
            if (ok) src_row[r] = static_cast<int32_t>(i / k);
        }
    }
    // rows past the last valid one (only when some ids were invalid) are marked -1
    for (int64_t r = total_all + threadIdx.x; r < n; r += kThreads) src_row[r] = -1;
}

__device__ __forceinline__ int64_t sf_word_offset(int64_t row, int64_t g, int64_t groups) {
    // byte offset of the 4 scale bytes (k-blocks 4g..4g+3) of `row` in the tensor-core layout
    return ((row >> 7) * groups + g) * 512 + (row & 31) * 16 + ((row & 127) >> 5) * 4;
}

__global__ void __launch_bounds__(kThreads) gather_kernel(const uint8_t* __restrict__ q_in,
                                                          const uint8_t* __restrict__ sf_in, int64_t K,
                                                          const int32_t* __restrict__ off,
                                                          const int32_t* __restrict__ poff,
                                                          const int32_t* __restrict__ src_row, int E,
                                                          int64_t pbound, uint8_t* __restrict__ q_out,
                                                          uint8_t* __restrict__ sf_out) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t p = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    if (p >= pbound) return;
    const int32_t ptotal = __ldg(poff + E);
    if (p >= ptotal) return;
    int lo = 0, hi = E - 1;   // last e with poff[e] <= p
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(poff + mid) <= p) lo = mid; else hi = mid - 1;
    }
    const int64_t local = p - __ldg(poff + lo);
    const int64_t cnt = __ldg(off + lo + 1) - __ldg(off + lo);
    const int64_t groups = (K + 127) / 128;
    if (local < cnt) {
        const int64_t r = __ldg(off + lo) + local;
        const int64_t t = __ldg(src_row + r);
        const uint4* src = reinterpret_cast<const uint4*>(q_in + t * K);
        uint4* dst = reinterpret_cast<uint4*>(q_out + r * K);
        for (int64_t v = lane; v < K / 16; v += 32) dst[v] = __ldg(src + v);
        for (int64_t g = lane; g < groups; g += 32) {
            const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(sf_in + sf_word_offset(t, g, groups)));
            *reinterpret_cast<uint32_t*>(sf_out + sf_word_offset(p, g, groups)) = w;
        }
    } else {
        for (int64_t g = lane; g < groups; g += 32)
            *reinterpret_cast<uint32_t*>(sf_out + sf_word_offset(p, g, groups)) = 0u;
    }
}

__global__ void __launch_bounds__(kThreads) gather_rows_kernel(const uint8_t* __restrict__ src, int64_t row_bytes,
                                                               const int32_t* __restrict__ src_row, int64_t R,
                                                               uint8_t* __restrict__ dst) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    if (r >= R) return;
    const int64_t t = __ldg(src_row + r);
    if (t < 0) return;
    const uint4* s = reinterpret_cast<const uint4*>(src + t * row_bytes);
    uint4* d = reinterpret_cast<uint4*>(dst + r * row_bytes);
    for (int64_t v = lane; v < row_bytes / 16; v += 32) d[v] = __ldg(s + v);
}

}  // namespace

size_t permute_workspace_bytes(int64_t T, int k, int E) {
    const int64_t n = T * k;
    const int64_t nblk = ceil_div(n, kChunk);
    return static_cast<size_t>(2 * nblk * E) * sizeof(int32_t) + 16;
}

int launch_permute(const int32_t* ids, int64_t T, int k, int E, int32_t* counts, int32_t* off, int32_t* poff,
                   int32_t* src_row, int32_t* dst_of, const uint8_t* q_in, const uint8_t* sf_in, int64_t K,
                   uint8_t* q_out, uint8_t* sf_out, void* ws, int* dev_err, cudaStream_t stream) {
    const int64_t n = T * k;
    const int64_t nblk = ceil_div(n, kChunk);
    int32_t* blk_counts = static_cast<int32_t*>(ws);
    int32_t* blk_base = blk_counts + nblk * E;
    if (nblk == 1) {   // one chunk: the three steps in one launch
        permute_small_kernel<<<1, kThreads, 0, stream>>>(ids, n, k, E, counts, off, poff, src_row, dst_of, dev_err);
    } else {
        if (nblk > 0)
            hist_kernel<<<static_cast<unsigned>(nblk), kThreads, 0, stream>>>(ids, n, E, blk_counts, dev_err);
        scan_kernel<<<1, 1024, 0, stream>>>(blk_counts, blk_base, nblk, E, n, counts, off, poff, src_row);
        if (nblk > 0)
            rank_kernel<<<static_cast<unsigned>(nblk), kThreads, 0, stream>>>(ids, n, k, E, blk_base, off, src_row,
                                                                             dst_of);
    }
    if (q_in != nullptr) {
        const int64_t pbound = round_up(n + 127 * static_cast<int64_t>(E), 128);
        const int64_t blocks = ceil_div(pbound, kWarps);
        gather_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(q_in, sf_in, K, off, poff, src_row, E,
                                                                             pbound, q_out, sf_out);
    }
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

int launch_gather_rows(const void* src, int64_t row_bytes, const int32_t* src_row, int64_t R, void* dst,
                       cudaStream_t stream) {
    if (R <= 0) return MX_OK;
    const int64_t blocks = ceil_div(R, kWarps);
    gather_rows_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        static_cast<const uint8_t*>(src), row_bytes, src_row, R, static_cast<uint8_t*>(dst));
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

}  // namespace mx
