// gemm.cu -- expert grouped GEMM on MXFP8 operands for sm_103a.
//
// Design (aigc.bar, "Blackwell性能陷阱？Cursor揭秘：重写内核让AI大模型MoE提速3.5倍的底层逻辑",
// section "破局之道：从零构建，释放硬件真正潜能", and section "1. Blackwell的TMEM架构瓶颈"):
// the block scales are applied by the tensor core itself (tcgen05.mma
// kind::mxf8f6f4.block_scale), the fp32 accumulator lives in tensor memory, and
// loading operands, loading scales, issuing the MMA and draining the accumulator
// are done by separate warps.
//
//   warp 0      TMA producer: per 128-deep K step, one 2-D tensor copy for the A
//               tile (128 rows x 128 bytes, 128-byte swizzle), one for the B tile
//               (256 rows), and 512-byte bulk copies of the matching scale atoms
//               (the quantizer writes every 128 x 4 scale block as one contiguous
//               512-byte atom, so no reshaping happens anywhere);
//   warp 1      allocates tensor memory, then one lane issues, per K step, three
//               tcgen05.cp (smem scale atoms -> TMEM) and four 128x256x32 block-scaled
//               MMAs, and commits to the stage's "empty" barrier;
//   warps 4-11  epilogue: tcgen05.ld of the 128 x 256 fp32 accumulator (each warp
//               one 32-lane quarter x 128 columns), conversion, release of the
//               accumulator, then predicated stores (rows past an expert's tokens
//               are never written).
// A persistent grid of one CTA per SM walks a static tile list.  Tiles of one
// expert are contiguous in the list, N-tile fastest, so the CTAs in flight share
// one expert's A rows and weight matrix in L2 (expert-wise grouping).  Every
// pipeline wait is bounded; a timeout sets MX_DEVERR_TIMEOUT and all roles leave.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "mxmoe_internal.h"

namespace mx {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int kStages = 4;
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kNumEpiWarps = 8;
constexpr int kMaxE = 1024;

constexpr uint32_t kABytes = BM * BK;      // 16 KiB
constexpr uint32_t kBBytes = BN * BK;      // 32 KiB
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffSFA = kOffB + kStages * kBBytes;
constexpr uint32_t kOffSFB = kOffSFA + kStages * 512;
constexpr uint32_t kOffBar = kOffSFB + kStages * 1024;
constexpr uint32_t kNumBars = 2 * kStages + 3;    // full[], empty[], tmem_full, tmem_empty, drain
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;   // tmem base (4 B), abort flag (4 B)
constexpr uint32_t kOffTable = (kOffMisc + 8 + 15) / 16 * 16;
constexpr uint32_t kSmemBytes = kOffTable + (kMaxE + 1) * 4 + 1024;   // + alignment slack

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSFA = 256;   // + 4 * stage
constexpr uint32_t kTmemSFB = 272;   // + 8 * stage

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait

struct GemmArgs {
    int kind;
    const uint8_t* SFA;
    const uint8_t* SFB;
    int64_t a_groups;    // 128-wide K groups per scale row of A (= ceil(a_cols / 128))
    int64_t b_groups;
    int64_t b_row_step, b_col_step;
    int64_t n_out, m_out, k_len;
    const int32_t* off;
    const int32_t* poff;
    int E;
    int64_t row_limit;   // fwd/dgrad: off[E] may not exceed the rows of A and C
    int64_t p_limit;     // poff[E] may not exceed the padded rows (positions) the scale / columnwise buffers hold
    void* out;
    int* dev_err;
};

struct Tile {
    int64_t a_row, a_sf_blk, a_col0;   // A tile origin (data row, 128-row scale block, first K column)
    int64_t b_row, b_col0;
    int64_t out_row0, out_col0;
    int num_kt;
    int valid_rows;
    bool b_half1;                      // B rows 128..255 of the tile exist
    int e;
};

__device__ __forceinline__ int64_t expert_rows(const GemmArgs& g, int e) {
    return static_cast<int64_t>(__ldg(g.off + e + 1)) - __ldg(g.off + e);
}

__device__ __forceinline__ Tile get_tile(const GemmArgs& g, const int32_t* table, int64_t L) {
    Tile t;
    const int64_t nt = (g.n_out + BN - 1) / BN;
    int e;
    int64_t local;
    if (g.kind == kGemmRows) {
        int lo = 0, hi = g.E - 1;   // last e with table[e] <= L
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (table[mid] <= L) lo = mid; else hi = mid - 1;
        }
        e = lo;
        local = L - table[e];
    } else {
        const int64_t per_e = (g.m_out / BM) * nt;
        e = static_cast<int>(L / per_e);
        local = L - static_cast<int64_t>(e) * per_e;
    }
    const int64_t mt = local / nt;
    const int64_t ntile = local - mt * nt;
    t.e = e;
    t.out_col0 = ntile * BN;
    t.b_half1 = t.out_col0 + 128 < g.n_out;
    if (g.kind == kGemmRows) {
        const int64_t te = expert_rows(g, e);
        t.a_row = __ldg(g.off + e) + mt * BM;
        t.a_sf_blk = __ldg(g.poff + e) / 128 + mt;
        t.a_col0 = 0;
        t.b_row = static_cast<int64_t>(e) * g.b_row_step + ntile * BN;
        t.b_col0 = static_cast<int64_t>(e) * g.b_col_step;
        t.num_kt = static_cast<int>((g.k_len + BK - 1) / BK);
        t.out_row0 = t.a_row;
        const int64_t vr = te - mt * BM;
        t.valid_rows = static_cast<int>(vr < BM ? vr : BM);
    } else {
        const int64_t p0 = __ldg(g.poff + e);
        const int64_t plen = static_cast<int64_t>(__ldg(g.poff + e + 1)) - p0;
        t.a_row = mt * BM;
        t.a_sf_blk = mt;
        t.a_col0 = p0;
        t.b_row = ntile * BN;
        t.b_col0 = p0;
        t.num_kt = static_cast<int>(plen / BK);
        t.out_row0 = static_cast<int64_t>(e) * g.m_out + mt * BM;
        t.valid_rows = BM;
    }
    return t;
}

template <bool kOutBf16>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + kOffBar;                  // + 8 * stage
    const uint32_t bar_empty = sbase + kOffBar + 8 * kStages;   // + 8 * stage
    const uint32_t bar_tmem_full = sbase + kOffBar + 16 * kStages;
    const uint32_t bar_tmem_empty = bar_tmem_full + 8;
    const uint32_t bar_drain = bar_tmem_full + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    int32_t* table = reinterpret_cast<int32_t*>(smem + kOffTable);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_tmem_full, 1);
        mbar_init(bar_tmem_empty, kNumEpiWarps);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 2) {
        // Validate the group offsets (every later address depends on them) and build
        // the tile list: table[e] = first tile of expert e, table[E] = tile count.
        const int64_t nt = (g.n_out + BN - 1) / BN;
        const int per = (g.E + 31) / 32;
        const int e0 = lane * per;
        int32_t sum = 0;
        bool bad = false;
        for (int e = e0; e < e0 + per && e < g.E; ++e) {
            const int64_t te = expert_rows(g, e);
            const int64_t pe = static_cast<int64_t>(__ldg(g.poff + e + 1)) - __ldg(g.poff + e);
            bad |= te < 0 || pe != (te + 127) / 128 * 128 || (__ldg(g.poff + e) & 127) != 0;
            if (g.kind == kGemmRows) sum += static_cast<int32_t>(((te + BM - 1) / BM) * nt);
        }
        if (lane == 31) {
            bad |= __ldg(g.off) != 0 || __ldg(g.poff) != 0 || __ldg(g.poff + g.E) > g.p_limit;
            if (g.kind == kGemmRows) bad |= __ldg(g.off + g.E) > g.row_limit;
        }
        bad = __any_sync(0xffffffffu, bad);
        int32_t incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (g.kind == kGemmRows) {
            int32_t run = incl - sum;
            for (int e = e0; e < e0 + per && e < g.E; ++e) {
                table[e] = run;
                run += static_cast<int32_t>(((expert_rows(g, e) + BM - 1) / BM) * nt);
            }
        }
        if (lane == 31) {
            if (bad) {
                table[g.E] = 0;
                atomicOr(g.dev_err, MX_DEVERR_BAD_SEGMENTS);
            } else if (g.kind == kGemmRows) {
                table[g.E] = incl;
            } else {
                table[g.E] = static_cast<int32_t>(static_cast<int64_t>(g.E) * (g.m_out / BM) * nt);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t total_tiles = table[g.E];

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t L = blockIdx.x; L < total_tiles && ok; L += gridDim.x) {
                const Tile t = get_tile(g, table, L);
                for (int kt = 0; kt < t.num_kt; ++kt) {
                    if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = bar_full + 8 * stage;
                    const uint32_t bytes = kABytes + kBBytes + 512 + (t.b_half1 ? 1024 : 512);
                    mbar_arrive_expect_tx(full, bytes);
                    const int32_t ax = static_cast<int32_t>(t.a_col0 + kt * BK);
                    const int32_t bx = static_cast<int32_t>(t.b_col0 + kt * BK);
                    tma_load_2d(sbase + kOffA + stage * kABytes, &tmA, full, ax, static_cast<int32_t>(t.a_row));
                    tma_load_2d(sbase + kOffB + stage * kBBytes, &tmB, full, bx, static_cast<int32_t>(t.b_row));
                    const int64_t agrp = t.a_col0 / 128 + kt;
                    const int64_t bgrp = t.b_col0 / 128 + kt;
                    bulk_load(sbase + kOffSFA + stage * 512, g.SFA + (t.a_sf_blk * g.a_groups + agrp) * 512, 512,
                              full);
                    const int64_t bblk = t.b_row / 128;
                    bulk_load(sbase + kOffSFB + stage * 1024, g.SFB + (bblk * g.b_groups + bgrp) * 512, 512, full);
                    if (t.b_half1)
                        bulk_load(sbase + kOffSFB + stage * 1024 + 512,
                                  g.SFB + ((bblk + 1) * g.b_groups + bgrp) * 512, 512, full);
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(g.dev_err, MX_DEVERR_TIMEOUT);
            }
            // let the copies still in flight land before the CTA can exit
            const int64_t outstanding = issued < kStages ? issued : kStages;
            for (int64_t i = 1; i <= outstanding; ++i) {
                const int64_t idx = issued - i;
                const int s = static_cast<int>(idx % kStages);
                const uint32_t ph = static_cast<uint32_t>((idx / kStages) & 1);
                mbar_wait_timeout(bar_full + 8 * s, ph, kWaitLimitNs / 4);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_iter = 0;
            bool ok = true;
            const uint32_t idesc0 = idesc_mxf8(BM, BN, 0, 0);
            for (int64_t L = blockIdx.x; L < total_tiles && ok; L += gridDim.x) {
                const Tile t = get_tile(g, table, L);
                if (t.num_kt == 0) continue;
                if (!mbar_wait_bounded(bar_tmem_empty, (acc_iter & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < t.num_kt; ++kt) {
                    if (!mbar_wait_bounded(bar_full + 8 * stage, phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem_base + kTmemSFA + 4 * stage;
                    const uint32_t sfb_t = tmem_base + kTmemSFB + 8 * stage;
                    tc_cp_32x128b_warpx4(sfa_t, smem_desc(sbase + kOffSFA + stage * 512, 0, 128, 0));
                    tc_cp_32x128b_warpx4(sfb_t, smem_desc(sbase + kOffSFB + stage * 1024, 0, 128, 0));
                    tc_cp_32x128b_warpx4(sfb_t + 4, smem_desc(sbase + kOffSFB + stage * 1024 + 512, 0, 128, 0));
                    const uint64_t adesc = smem_desc(sbase + kOffA + stage * kABytes, 16, 1024, 2);
                    const uint64_t bdesc = smem_desc(sbase + kOffB + stage * kBBytes, 16, 1024, 2);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k) {
                        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(k) << 29) | (static_cast<uint32_t>(k) << 4);
                        mma_mxf8(tmem_base, adesc + static_cast<uint64_t>((k * 32) >> 4),
                                 bdesc + static_cast<uint64_t>((k * 32) >> 4), idesc, sfa_t, sfb_t,
                                 (kt > 0 || k > 0) ? 1u : 0u);
                    }
                    tc_commit(bar_empty + 8 * stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(bar_tmem_full);
                ++acc_iter;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(g.dev_err, MX_DEVERR_TIMEOUT);
            }
            // every tcgen05 operation this thread issued has finished once this arrives
            tc_commit(bar_drain);
            mbar_wait_timeout(bar_drain, 0, kWaitLimitNs / 4);
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                       // TMEM lane quarter this warp may access
        const int half = (warp - kEpiWarp0) >> 2;     // column half of the 256-wide tile
        const int row = q * 32 + lane;                // accumulator row owned by this thread
        uint32_t acc_iter = 0;
        for (int64_t L = blockIdx.x; L < total_tiles; L += gridDim.x) {
            const Tile t = get_tile(g, table, L);
            const bool row_ok = row < t.valid_rows;
            if (t.num_kt == 0) {
                if (!kOutBf16 && row_ok) {   // expert without tokens: its weight gradient is zero
                    float* dst = static_cast<float*>(g.out) + (t.out_row0 + row) * g.n_out;
                    for (int c = 0; c < 4; ++c) {
                        const int64_t col = t.out_col0 + half * 128 + c * 32;
                        if (col >= g.n_out) break;
                        float4* d4 = reinterpret_cast<float4*>(dst + col);
#pragma unroll
                        for (int j = 0; j < 8; ++j) d4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                continue;
            }
            uint32_t okw = 1;
            if (lane == 0) okw = mbar_wait_bounded(bar_tmem_full, acc_iter & 1u, abort_flag, kWaitLimitNs) ? 1u : 0u;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            if (!okw) {
                if (lane == 0) {
                    *abort_flag = 1;
                    atomicOr(g.dev_err, MX_DEVERR_TIMEOUT);
                }
                break;
            }
            __syncwarp();
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + half * 128;
            if (kOutBf16) {
                uint32_t packed[4][16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        packed[c][j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_tmem_empty);
                if (row_ok) {
                    uint16_t* dst = static_cast<uint16_t*>(g.out) + (t.out_row0 + row) * g.n_out;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int64_t col = t.out_col0 + half * 128 + c * 32;
                        if (col < g.n_out) {
                            uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                d4[j] = make_uint4(packed[c][4 * j], packed[c][4 * j + 1], packed[c][4 * j + 2],
                                                   packed[c][4 * j + 3]);
                        }
                    }
                }
            } else {
                float* dst = static_cast<float*>(g.out) + (t.out_row0 + row) * g.n_out;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, r);
                    tmem_ld_wait();
                    const int64_t col = t.out_col0 + half * 128 + c * 32;
                    if (row_ok && col < g.n_out) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
                        for (int j = 0; j < 8; ++j) d4[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_tmem_empty);
            }
            ++acc_iter;
        }
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

int launch_grouped_gemm(const GemmProblem& pr, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MX_ERR_CUDA;
    static int num_sms[64] = {0};
    static bool attr_set[64][2] = {{false}};
    if (dev < 0 || dev >= 64) return MX_ERR_CUDA;
    if (num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return MX_ERR_CUDA;
        num_sms[dev] = n;
    }
    CUtensorMap tmA, tmB;
    if (!make_map(&tmA, pr.A, pr.a_rows, pr.a_cols, BM)) return MX_ERR_CUDA;
    if (!make_map(&tmB, pr.B, pr.b_rows, pr.b_cols, BN)) return MX_ERR_CUDA;
    GemmArgs g;
    g.kind = pr.kind;
    g.SFA = pr.SFA;
    g.SFB = pr.SFB;
    g.a_groups = ceil_div(pr.a_cols, 128);
    g.b_groups = ceil_div(pr.b_cols, 128);
    g.b_row_step = pr.b_row_step;
    g.b_col_step = pr.b_col_step;
    g.n_out = pr.n_out;
    g.m_out = pr.m_out;
    g.k_len = pr.k_len;
    g.off = pr.off;
    g.poff = pr.poff;
    g.E = pr.E;
    g.row_limit = pr.kind == kGemmRows ? pr.a_rows : 0;
    g.p_limit = pr.kind == kGemmRows ? round_up(pr.a_rows + 127 * static_cast<int64_t>(pr.E), 128) : pr.a_cols;
    g.out = pr.out;
    g.dev_err = pr.dev_err;
    const bool bf16 = pr.kind == kGemmRows;
    if (!attr_set[dev][bf16 ? 1 : 0]) {
        cudaError_t e = bf16 ? cudaFuncSetAttribute(grouped_gemm_kernel<true>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)
                             : cudaFuncSetAttribute(grouped_gemm_kernel<false>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return MX_ERR_CUDA;
        attr_set[dev][bf16 ? 1 : 0] = true;
    }
    const unsigned grid = static_cast<unsigned>(num_sms[dev]);
    if (bf16)
        grouped_gemm_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, g);
    else
        grouped_gemm_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(tmA, tmB, g);
    return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

}  // namespace mx
