// gemm.cu -- expert grouped GEMM on MXFP8 operands for sm_103a.
//
// Design (aigc.bar, "Blackwell性能陷阱？Cursor揭秘：重写内核让AI大模型MoE提速3.5倍的底层逻辑",
// section "破局之道：从零构建，释放硬件真正潜能", and section "1. Blackwell的TMEM架构瓶颈"):
// the block scales are applied by the tensor core itself (tcgen05.mma
// kind::mxf8f6f4.block_scale), the fp32 accumulator lives in tensor memory, loading
// operands, loading scales, issuing the MMA and draining the accumulator are done
// by separate warps, and two SMs cooperate on one MMA, sharing the B operand.
//
// Template NC = CTAs per MMA:
//   NC = 2 (default): a cluster of two CTAs on an SM pair computes 256 x 256 tiles
//          with tcgen05.mma.cta_group::2; each CTA stages its own 128 rows of A and
//          one 128-row half of B (so B is read from L2 once per pair); 3 pipeline
//          stages of two 128-deep K steps each (6 operand buffers);
//   NC = 1: one CTA computes 128 x 256 tiles (cta_group::1), 4 stages of one K step.
//
//   warp 0      TMA producer: per 128-deep K step, a 2-D tensor copy of the A tile
//               (128 rows x 128 bytes, 128-byte swizzle), one of the B tile (256/NC
//               rows), and 4-D tensor copies of the scale atoms (the quantizer writes
//               each 128 x 4 scale block as one contiguous 512-byte atom, so no
//               reshaping happens; the 4-D view makes every scale read bounds-checked).
//               With NC = 2 every copy of both CTAs completes on the leader CTA's
//               "full" barrier.
//   warp 1      allocates tensor memory; in the leader CTA one lane issues, per K
//               step, tcgen05.cp of the scale atoms into TMEM and four block-scaled
//               MMAs (K = 32 each), and per stage commits to its "empty" barrier in
//               every CTA of the pair.
//   warps 4-11  epilogue: tcgen05.ld of this CTA's 128 x 256 fp32 accumulator (each
//               warp one 32-lane quarter x 128 columns), conversion, release of the
//               accumulator, then predicated stores (rows past an expert's tokens are
//               never written).
// B-operand scales come in one of two layouts (template SFB1): the four-copy layout
// (each 512-byte atom stored four times), moved into tensor memory by one 128x256b copy per
// K step, or the plain one-copy atom layout, moved by two replicating 32x128b.warpx4 copies
// per K step (same tensor-memory contents, one more copy on the tensor pipe).
// A persistent grid (one CTA per SM) walks a static tile list built in shared memory
// from the device offsets.  Tiles of one expert are contiguous, M-tile fastest (one N tile
// at a time down the expert's rows), so the units in flight share one B tile and the
// expert's A strip stays in L2 across its N tiles (the pages' expert-wise grouping, realised
// as the raster order; the weight-gradient GEMM then reads its operands from DRAM once).
// Every pipeline wait is bounded; a timeout sets MX_DEVERR_TIMEOUT and all roles leave.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "mxmoe_internal.h"
#include "quant_common.cuh"

namespace mx {
namespace {

constexpr int BM = 128;    // accumulator rows per CTA
constexpr int BN = 256;    // tile columns
constexpr int BK = 128;    // K bytes per stage
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kNumEpiWarps = 8;
constexpr int kMaxE = 1024;
constexpr uint32_t kTmemCols = 512;
// epilogue modes: bf16 rows (forward, dgrad), fp32 (wgrad), SwiGLU + MXFP8 (GEMM1 forward)
constexpr int kEpiBf16 = 0;
constexpr int kEpiF32 = 1;
constexpr int kEpiSwiglu = 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait

template <int NC, int kEpi = kEpiBf16, bool SFB1 = false>
struct Cfg {
    // A CTA pair takes two 128-deep K steps per pipeline stage: one barrier wait and one
    // commit per 8 MMAs.  The single issuing thread spends ~190 cycles per mbarrier wait
    // and ~60 per commit, next to ~290 for four MMAs and ~180 for three scale copies;
    // per 128-step that overhead otherwise exceeds the 512 tensor cycles of the step.
    static constexpr int kSub = NC == 1 ? 1 : 2;                   // 128-deep K steps per pipeline stage
    static constexpr int kStages = NC == 1 ? 4 : 3;
    static constexpr int kSlots = kStages * kSub;                  // operand buffers
    static constexpr int kTileM = BM * NC;
    static constexpr int kBRows = BN / NC;                       // B rows staged per CTA
    static constexpr uint32_t kABytes = BM * BK;                 // 16 KiB
    static constexpr uint32_t kBBytes = kBRows * BK;             // 32 or 16 KiB
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffB = kOffA + kSlots * kABytes;
    static constexpr uint32_t kOffSFA = kOffB + kSlots * kBBytes;
    static constexpr uint32_t kOffSFB = kOffSFA + kSlots * 512;
    // B scales per K step: both 128-row atoms of the 256-row B tile, each in its four copies
    // (4 KiB, one 128x256b tensor-memory copy); with one-copy B scales, and in the SwiGLU
    // variant (gate and up atoms), the two atoms once (1 KiB, two replicating 32x128b.warpx4
    // copies)
    static constexpr uint32_t kSfbSlot = (kEpi == kEpiSwiglu || SFB1) ? 1024 : 4096;
    static constexpr uint32_t kOffBar = kOffSFB + kSlots * kSfbSlot;
    static constexpr uint32_t kNumBars = 2 * kStages + 4;        // full[], empty[], tmem_full, tmem_empty, drain, epi
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
    static constexpr uint32_t kOffTable = (kOffMisc + 8 + 15) / 16 * 16;
    static constexpr uint32_t kSmemBytes = kOffTable + (kMaxE + 1) * 4 + 1024;
    // SwiGLU epilogue: per epilogue warp a [32][17] fp32 staging tile, then two pairs of
    // 512-byte scale atoms (rowwise, columnwise; double-buffered across tiles)
    static constexpr uint32_t kOffEpi = (kOffTable + (kMaxE + 1) * 4 + 15) / 16 * 16;
    static constexpr uint32_t kEpiStage = 32 * 17;                // floats per warp
    static constexpr uint32_t kOffEpiAtoms = kOffEpi + kNumEpiWarps * kEpiStage * 4;
    static constexpr uint32_t kSmemBytesSwiglu = kOffEpiAtoms + 4 * 512 + 1024;
    static constexpr uint32_t kSlotTx = NC * (kABytes + kBBytes + 512 + kSfbSlot);   // bytes landing per K step
    static constexpr uint32_t kTmemSFA = 256;                     // + 4 * slot
    static constexpr uint32_t kTmemSFB = 256 + 4 * kSlots;        // + 8 * slot
    static_assert(kTmemSFB + 8 * kSlots <= kTmemCols, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kEpi != kEpiSwiglu || NC == 1 || kSmemBytesSwiglu <= 232448, "shared memory budget (SwiGLU epilogue)");
};

struct GemmArgs {
    int kind;
    int64_t b_row_step, b_col_step;
    int64_t n_out, m_out, k_len;
    const int32_t* off;
    const int32_t* poff;
    int E;
    int64_t row_limit;   // fwd/dgrad: off[E] may not exceed the rows of A and C
    int64_t p_limit;     // poff[E] may not exceed the padded rows the scale / columnwise buffers hold
    void* out;
    int* dev_err;
    // SwiGLU epilogue (swiglu_i = I > 0): out = [gate | up] bf16 [R x 2I]; h = silu(gate) * up
    // quantized rowwise (h_qrow [R x I], h_sfrow) and columnwise (h_qcol [I x h_ldcol], h_sfcol)
    int64_t swiglu_i;
    uint8_t* h_qrow;
    uint8_t* h_sfrow;
    uint8_t* h_qcol;
    uint8_t* h_sfcol;
    int64_t h_ldcol;
    int h_sfrow_copies, h_sfcol_copies;   // 1 or 4 copies of each scale atom
    int wide_store;                      // out is 32-byte aligned: whole-sector (32-byte) stores
    uint64_t wait_limit_ns;              // limit of every pipeline wait (kWaitLimitNs unless a test sets it)
    int withhold_operands;               // test only: issue no operand copies, so no stage ever fills
    int raster_group;                    // tile order inside an expert (see get_tile)
    int b_blocked;                       // B codes in 128 x 128 blocks of 16 KiB (a 4-D tensor map)
};

struct Tile {
    int64_t a_row, a_sf_blk, a_col0;   // this CTA's A tile origin (data row, 128-row scale block, first K column)
    int64_t b_row, b_sf_blk, b_col0;   // this CTA's B rows; first 128-row scale block of the whole B tile
    int64_t b_sf_blk2;                 // SwiGLU tiles: scale block of the up rows
    int64_t out_row0, out_col0;
    int num_kt;
    int valid_rows;
};

__device__ __forceinline__ int64_t expert_rows(const GemmArgs& g, int e) {
    return static_cast<int64_t>(__ldg(g.off + e + 1)) - __ldg(g.off + e);
}

// Tile L of the unit's list.  MP = 2 with CTA pairs: the unit is a cluster of two pairs that take
// the two N tiles 2 j and 2 j + 1 of one M tile (pair index pp), so the list runs over those
// N-tile pairs.  MP = 2 with single CTAs: the unit is a cluster of two CTAs that take the two M
// tiles 2 i and 2 i + 1 of one N tile (CTA index pp), so the list runs over M-tile pairs.
template <int NC, int MP>
__device__ __forceinline__ constexpr bool pairs_m_tiles() { return NC == 1 && MP == 2; }

template <int NC, int MP = 1>
__device__ __forceinline__ Tile get_tile(const GemmArgs& g, const int32_t* table, int64_t L, uint32_t rank,
                                         uint32_t pp = 0) {
    Tile t;
    constexpr bool kPM = pairs_m_tiles<NC, MP>();
    constexpr int kMG = kPM ? 2 : 1;   // M tiles per list entry
    const int64_t nt = ((g.n_out + BN - 1) / BN + (kPM ? 1 : MP) - 1) / (kPM ? 1 : MP);   // N tiles (or N-tile pairs)
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
        const int64_t per_e = (((g.m_out + Cfg<NC>::kTileM - 1) / Cfg<NC>::kTileM + kMG - 1) / kMG) * nt;
        e = static_cast<int>(L / per_e);
        local = L - static_cast<int64_t>(e) * per_e;
    }
    // Order of the expert's tiles: groups of G M tiles, M fastest inside a group, one N tile
    // at a time down the group's rows.  The units in flight then share one B tile, and the
    // group's A strip (G x 256 rows x K bytes) stays in L2 across the N tiles.  By default G
    // covers as many M tiles as keep that strip within 32 MiB (all of an expert's tiles at the
    // MoE FFN sizes); G = 1 is the N-fastest order.
    const int64_t rows = g.kind == kGemmRows ? expert_rows(g, e) : g.m_out;
    const int64_t mts = ((rows + Cfg<NC>::kTileM - 1) / Cfg<NC>::kTileM + kMG - 1) / kMG;   // (M-tile pairs)
    const int64_t kbytes = g.kind == kGemmRows ? g.k_len
                                               : static_cast<int64_t>(__ldg(g.poff + e + 1)) - __ldg(g.poff + e);
    int64_t G = g.raster_group;
    if (G <= 0) {
        G = (int64_t(32) << 20) / (Cfg<NC>::kTileM * kMG * (kbytes > 0 ? kbytes : 1));
        G = G < 1 ? 1 : (G > mts ? mts : G);
    }
    const int64_t grp = local / (G * nt);
    const int64_t in = local - grp * G * nt;
    const int64_t gs = mts - grp * G < G ? mts - grp * G : G;   // (>= 1: local < mts * nt)
    const int64_t ntile = kPM ? in / gs : (in / gs) * MP + pp;
    const int64_t mt = (grp * G + (in - (in / gs) * gs)) * kMG + (kPM ? pp : 0);
    const int64_t m_in = mt * Cfg<NC>::kTileM + static_cast<int64_t>(rank) * BM;   // this CTA's first row
    t.out_col0 = ntile * BN;
    int64_t vr;
    if (g.kind == kGemmRows) {
        t.a_row = __ldg(g.off + e) + m_in;
        t.a_sf_blk = __ldg(g.poff + e) / 128 + mt * NC + rank;
        t.a_col0 = 0;
        const int64_t b0 = static_cast<int64_t>(e) * g.b_row_step + ntile * BN;
        t.b_row = b0 + static_cast<int64_t>(rank) * Cfg<NC>::kBRows;
        t.b_sf_blk = b0 / 128;
        t.b_sf_blk2 = 0;
        if (g.swiglu_i > 0) {
            // 128 h columns per tile: the pair's first CTA stages the 128 gate rows of W1,
            // the second the matching up rows, so accumulator columns 0..127 are gate and
            // 128..255 up for the same h columns
            const int64_t g0 = static_cast<int64_t>(e) * g.b_row_step + ntile * 128;
            t.b_row = g0 + static_cast<int64_t>(rank) * g.swiglu_i;
            t.b_sf_blk = g0 / 128;
            t.b_sf_blk2 = (g0 + g.swiglu_i) / 128;
            t.out_col0 = ntile * 128;
        }
        t.b_col0 = static_cast<int64_t>(e) * g.b_col_step;
        t.num_kt = static_cast<int>((g.k_len + BK - 1) / BK);
        t.out_row0 = t.a_row;
        vr = expert_rows(g, e) - m_in;
    } else {
        const int64_t p0 = __ldg(g.poff + e);
        const int64_t plen = static_cast<int64_t>(__ldg(g.poff + e + 1)) - p0;
        t.a_row = m_in;
        t.a_sf_blk = m_in / 128;
        t.a_col0 = p0;
        t.b_row = ntile * BN + static_cast<int64_t>(rank) * Cfg<NC>::kBRows;
        t.b_sf_blk = ntile * BN / 128;
        t.b_col0 = p0;
        t.num_kt = static_cast<int>(plen / BK);
        t.out_row0 = static_cast<int64_t>(e) * g.m_out + m_in;
        vr = g.m_out - m_in;
    }
    t.valid_rows = static_cast<int>(vr < 0 ? 0 : (vr < BM ? vr : BM));
    return t;
}

// SwiGLU epilogue of the GEMM1 forward (aigc.bar and kucoin.com pages: MXFP8 quantization
// folded into the grouped-GEMM / SwiGLU data path).  This CTA's accumulator holds, for its
// 128 rows, gate in columns 0..127 and up in 128..255 for the tile's 128 h columns; epilogue
// warp (q, half) takes lane quarter q and h columns 64 half .. 64 half + 63.  gate and up are
// rounded to bf16 (the values stored in `out`), h = silu(gate) * up is formed from those in
// fp32 and quantized rowwise (a 32-column block is thread-local) and columnwise (16 columns at
// a time through the warp's staging tile; a warp's 32 rows are exactly one 32-row block, since
// tiles start on 128-row boundaries of the expert's padded positions).  The CTA's 128 x 4 scale
// bytes of each form make one 512-byte atom: assembled in shared memory, stored once.
// Returns false when a wait timed out.
template <int NC>
__device__ __forceinline__ bool epilogue_swiglu(const GemmArgs& g, const Tile& t, uint32_t taddr_q, int q, int half,
                                                int ew, int lane, int row, uint32_t lead_tmem_empty,
                                                uint32_t bar_epi, uint32_t acc_iter, float* st, uint8_t* atoms,
                                                const volatile int* abort_flag) {
    const int64_t I = g.swiglu_i;
    const bool row_ok = row < t.valid_rows;
    const bool any = t.valid_rows > 0;
    uint32_t gw[2][16], uw[2][16];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t rg[32], ru[32];
        tmem_ld_32x32b_x32(taddr_q + 64 * half + 32 * c, rg);
        tmem_ld_32x32b_x32(taddr_q + 128 + 64 * half + 32 * c, ru);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            gw[c][j] = pack_bf16x2(__uint_as_float(rg[2 * j]), __uint_as_float(rg[2 * j + 1]));
            uw[c][j] = pack_bf16x2(__uint_as_float(ru[2 * j]), __uint_as_float(ru[2 * j + 1]));
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster_relaxed(lead_tmem_empty);   // accumulator released: the next tile may start

    const int64_t p0 = t.a_sf_blk * 128;                   // padded position of accumulator row 0
    const int64_t hc0 = t.out_col0 + 64 * half;            // first h column of this warp
    const int64_t orow = t.out_row0 + row;
    uint8_t* arow = atoms + (acc_iter & 1u) * 1024;        // this tile's rowwise atom, then its columnwise atom
    uint8_t* acol = arow + 512;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        if (row_ok) {
            uint16_t* o = static_cast<uint16_t*>(g.out) + orow * 2 * I + hc0 + 32 * c;
            uint4* dg = reinterpret_cast<uint4*>(o);
            uint4* du = reinterpret_cast<uint4*>(o + I);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                dg[j] = make_uint4(gw[c][4 * j], gw[c][4 * j + 1], gw[c][4 * j + 2], gw[c][4 * j + 3]);
                du[j] = make_uint4(uw[c][4 * j], uw[c][4 * j + 1], uw[c][4 * j + 2], uw[c][4 * j + 3]);
            }
        }
        float h[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float g0 = bf16_lo(gw[c][j]), g1 = bf16_hi(gw[c][j]);
            const float u0 = bf16_lo(uw[c][j]), u1 = bf16_hi(uw[c][j]);
            h[2 * j] = row_ok ? g0 * sigmoid_f32(g0) * u0 : 0.0f;
            h[2 * j + 1] = row_ok ? g1 * sigmoid_f32(g1) * u1 : 0.0f;
        }
        // rowwise: these 32 values are one block
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) m = amax_step(m, h[j]);
        const uint32_t b = scale_byte_f32<0>(__float_as_uint(m));
        if (row_ok) {
            const float sc = inv_scale(b);
            uint32_t o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                o[j] = b == 0xFFu ? 0x7F7F7F7Fu
                                  : __byte_perm(quant_pair2(h[4 * j], h[4 * j + 1], sc),
                                                quant_pair2(h[4 * j + 2], h[4 * j + 3], sc), 0x5410);
            uint4* dq = reinterpret_cast<uint4*>(g.h_qrow + orow * I + hc0 + 32 * c);
            dq[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dq[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        arow[(row & 31) * 16 + (row >> 5) * 4 + 2 * half + c] = static_cast<uint8_t>(b);
        // columnwise: 16 columns at a time; lane (j, hh) takes column j, rows 16 hh .. 16 hh + 15
#pragma unroll
        for (int s = 0; s < 2; ++s) {
#pragma unroll
            for (int j = 0; j < 16; ++j) st[lane * 17 + j] = h[16 * s + j];
            __syncwarp();
            const int j = lane & 15, hh = lane >> 4;
            float v[16];
            float mc = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                v[k] = st[(16 * hh + k) * 17 + j];
                mc = amax_step(mc, v[k]);
            }
            mc = amax_step(mc, __shfl_xor_sync(0xffffffffu, mc, 16));
            const uint32_t bc = scale_byte_f32<0>(__float_as_uint(mc));
            const int cc = 64 * half + 32 * c + 16 * s + j;   // h column within the tile
            if (any) {
                const float sc = inv_scale(bc);
                uint32_t o[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    o[k] = bc == 0xFFu ? 0x7F7F7F7Fu
                                       : __byte_perm(quant_pair2(v[4 * k], v[4 * k + 1], sc),
                                                     quant_pair2(v[4 * k + 2], v[4 * k + 3], sc), 0x5410);
                *reinterpret_cast<uint4*>(g.h_qcol + (t.out_col0 + cc) * g.h_ldcol + p0 + q * 32 + 16 * hh) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            }
            if (hh == 0) acol[(cc & 31) * 16 + (cc >> 5) * 4 + q] = static_cast<uint8_t>(bc);
            __syncwarp();
        }
    }
    // every epilogue warp has written its bytes of both atoms (bounded wait, not bar.sync)
    if (lane == 0) mbar_arrive(bar_epi);
    uint32_t okw = 1;
    if (lane == 0) okw = mbar_wait_bounded(bar_epi, acc_iter & 1u, abort_flag, g.wait_limit_ns) ? 1u : 0u;
    okw = __shfl_sync(0xffffffffu, okw, 0);
    if (!okw) return false;
    if (any && ew < 2) {
        const int64_t ntile = t.out_col0 / 128;
        const int copies = ew == 0 ? g.h_sfrow_copies : g.h_sfcol_copies;
        uint8_t* dst = ew == 0 ? g.h_sfrow + ((p0 / 128) * (I / 128) + ntile) * 512 * copies
                               : g.h_sfcol + (ntile * (g.h_ldcol / 128) + p0 / 128) * 512 * copies;
        const uint4 v = reinterpret_cast<const uint4*>(ew == 0 ? arow : acol)[lane];
        for (int c = 0; c < copies; ++c) reinterpret_cast<uint4*>(dst + 512 * c)[lane] = v;
    }
    return true;
}

// MP = 2 (with NC = 2): clusters of two CTA pairs on the two N tiles of one M tile.  Each A
// half-tile is read from L2 once per cluster: CTA r copies 64 of its 128 rows and multicasts
// them to itself and to CTA r ^ 2 (the CTA of the other pair holding the same A rows), so A
// costs half the L2 reads; a stage is refilled only after both pairs' MMAs have consumed it.
template <int kEpi, int NC, bool SFB1, int MP = 1>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                        const GemmArgs g) {
    using C = Cfg<NC, kEpi, SFB1>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + C::kOffBar;                     // + 8 * stage (used in the leader)
    const uint32_t bar_empty = sbase + C::kOffBar + 8 * C::kStages;   // + 8 * stage
    const uint32_t bar_tmem_full = sbase + C::kOffBar + 16 * C::kStages;
    const uint32_t bar_tmem_empty = bar_tmem_full + 8;                // used in the leader
    const uint32_t bar_drain = bar_tmem_full + 16;
    const uint32_t bar_epi = bar_tmem_full + 24;                      // SwiGLU epilogue: 8 warps' scale atoms
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    int32_t* table = reinterpret_cast<int32_t*>(smem + C::kOffTable);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool kPM = pairs_m_tiles<NC, MP>();   // single CTAs in clusters of two, B multicast
    const uint32_t crank = NC * MP > 1 ? cluster_ctarank() : 0u;   // rank in the cluster
    const uint32_t rank = NC == 2 ? (crank & 1u) : 0u;             // rank in the CTA pair
    const uint32_t pp = NC == 2 ? crank >> 1 : crank;              // pair (or CTA) in the cluster
    const bool leader = rank == 0;
    const int64_t unit = blockIdx.x / (NC * MP);
    const int64_t num_units = gridDim.x / (NC * MP);
    // the pair leader's barriers as seen from this CTA (identity for NC == 1 and for a leader)
    const uint32_t lead_full = NC == 2 ? mapa_shared(bar_full, crank & ~1u) : bar_full;
    const uint32_t lead_tmem_empty = NC == 2 ? mapa_shared(bar_tmem_empty, crank & ~1u) : bar_tmem_empty;
    const uint16_t pair_ctas = static_cast<uint16_t>(NC == 2 ? (0x3u << (2 * pp)) : (0x1u << crank));   // this CTA's pair

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, MP);   // one commit per pair reading the stage
        }
        mbar_init(bar_tmem_full, 1);
        mbar_init(bar_tmem_empty, kNumEpiWarps * NC);
        mbar_init(bar_drain, 1);
        mbar_init(bar_epi, kNumEpiWarps);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSFA);
        tma_prefetch_desc(&tmSFB);
    }
    if (warp == 1) {
        tmem_alloc_g<NC>(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish_g<NC>();
    }
    if (warp == 2) {
        // Validate the group offsets (every later address depends on them) and build
        // the tile list: table[e] = first tile of expert e, table[E] = tile count (MP = 2:
        // tiles of a unit are N-tile pairs).
        const int64_t nt = ((g.n_out + BN - 1) / BN + (kPM ? 1 : MP) - 1) / (kPM ? 1 : MP);
        constexpr int kMG = kPM ? 2 : 1;   // M tiles per list entry
        const int per = (g.E + 31) / 32;
        const int e0 = lane * per;
        int32_t sum = 0;
        bool bad = false;
        for (int e = e0; e < e0 + per && e < g.E; ++e) {
            const int64_t te = expert_rows(g, e);
            const int64_t pe = static_cast<int64_t>(__ldg(g.poff + e + 1)) - __ldg(g.poff + e);
            bad |= te < 0 || pe != (te + 127) / 128 * 128 || (__ldg(g.poff + e) & 127) != 0;
            if (g.kind == kGemmRows) sum += static_cast<int32_t>((((te + C::kTileM - 1) / C::kTileM + kMG - 1) / kMG) * nt);
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
                run += static_cast<int32_t>((((expert_rows(g, e) + C::kTileM - 1) / C::kTileM + kMG - 1) / kMG) * nt);
            }
        }
        if (lane == 31) {
            if (bad) {
                table[g.E] = 0;
                if (leader) atomicOr(g.dev_err, MX_DEVERR_BAD_SEGMENTS);
            } else if (g.kind == kGemmRows) {
                table[g.E] = incl;
            } else {
                const int64_t mts = ((g.m_out + C::kTileM - 1) / C::kTileM + kMG - 1) / kMG;
                table[g.E] = static_cast<int32_t>(static_cast<int64_t>(g.E) * mts * nt);
            }
        }
    }
    tc_fence_before();
    if (NC * MP > 1) cluster_sync(); else __syncthreads();
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
            for (int64_t L = unit; L < total_tiles && ok; L += num_units) {
                const Tile t = get_tile<NC, MP>(g, table, L, rank, pp);
                for (int kt = 0; kt < t.num_kt; kt += C::kSub) {
                    const int nsub = t.num_kt - kt < C::kSub ? t.num_kt - kt : C::kSub;
                    if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, g.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    // withheld operands (a test of the bounded waits): this stage's "full" barrier
                    // is never armed, so the MMA issuer's wait for it has to run out
                    if (!g.withhold_operands) {
                        const uint32_t full = lead_full + 8 * stage;
                        if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, C::kSlotTx * static_cast<uint32_t>(nsub));
                        for (int sub = 0; sub < nsub; ++sub) {
                            const int slot = stage * C::kSub + sub;
                            const int32_t ax = static_cast<int32_t>(t.a_col0 + (kt + sub) * BK);
                            const int32_t bx = static_cast<int32_t>(t.b_col0 + (kt + sub) * BK);
                            if constexpr (NC == 2 && MP == 2)   // 64 of the 128 A rows, to both pairs' CTAs
                                tma_load_2d_pair_mc(sbase + C::kOffA + slot * C::kABytes + pp * (C::kABytes / 2), &tmA,
                                                    full, ax, static_cast<int32_t>(t.a_row + pp * (BM / 2)),
                                                    static_cast<uint16_t>((1u << crank) | (1u << (crank ^ 2u))));
                            else
                                tma_load_2d_g<NC>(sbase + C::kOffA + slot * C::kABytes, &tmA, full, ax,
                                                  static_cast<int32_t>(t.a_row));
                            if (g.b_blocked)   // the same bytes in shared memory: kBRows / 128 whole blocks
                                tma_load_4d_g<NC>(sbase + C::kOffB + slot * C::kBBytes, &tmB, full, 0, 0, bx / BK,
                                                  static_cast<int32_t>(t.b_row / 128));
                            else if constexpr (kPM)   // half of the B tile's rows, to both CTAs
                                tma_load_2d_mc(sbase + C::kOffB + slot * C::kBBytes + pp * (C::kBBytes / 2), &tmB, full,
                                               bx, static_cast<int32_t>(t.b_row + pp * (C::kBRows / 2)),
                                               static_cast<uint16_t>(0x3));
                            else
                                tma_load_2d_g<NC>(sbase + C::kOffB + slot * C::kBBytes, &tmB, full, bx,
                                                  static_cast<int32_t>(t.b_row));
                            tma_load_4d_g<NC>(sbase + C::kOffSFA + slot * 512, &tmSFA, full, 0, 0,
                                              static_cast<int32_t>(ax / BK), static_cast<int32_t>(t.a_sf_blk));
                            if constexpr (kEpi == kEpiSwiglu) {   // (the first copy of) the gate and up scale atoms
                                tma_load_4d_g<NC>(sbase + C::kOffSFB + slot * C::kSfbSlot, &tmSFB, full, 0, 0,
                                                  static_cast<int32_t>(bx / BK), static_cast<int32_t>(t.b_sf_blk));
                                tma_load_4d_g<NC>(sbase + C::kOffSFB + slot * C::kSfbSlot + 512, &tmSFB, full, 0, 0,
                                                  static_cast<int32_t>(bx / BK), static_cast<int32_t>(t.b_sf_blk2));
                            } else {   // both atoms of the tile's 256 B rows (four copies each in the SF4 layout)
                                tma_load_4d_g<NC>(sbase + C::kOffSFB + slot * C::kSfbSlot, &tmSFB, full, 0, 0,
                                                  static_cast<int32_t>(bx / BK), static_cast<int32_t>(t.b_sf_blk));
                            }
                        }
                        ++issued;
                    }
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(g.dev_err, MX_DEVERR_TIMEOUT);
            }
            if (leader) {
                // let the copies still in flight (both CTAs' for a pair) land before exit
                const int64_t outstanding = issued < C::kStages ? issued : C::kStages;
                for (int64_t i = 1; i <= outstanding; ++i) {
                    const int64_t idx = issued - i;
                    const int s = static_cast<int>(idx % C::kStages);
                    const uint32_t ph = static_cast<uint32_t>((idx / C::kStages) & 1);
                    mbar_wait_timeout(bar_full + 8 * s, ph, kWaitLimitNs / 4);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA)
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_iter = 0;
            bool ok = true;
            // a stage's "empty" goes to every CTA whose copies fill it (MP = 2: both pairs')
            const uint16_t fill_ctas = (NC == 2 && MP == 2) ? static_cast<uint16_t>(0xF) : pair_ctas;
            const uint32_t idesc0 = idesc_mxf8(C::kTileM, BN, 0, 0);
            for (int64_t L = unit; L < total_tiles && ok; L += num_units) {
                const Tile t = get_tile<NC, MP>(g, table, L, rank, pp);
                if (t.num_kt == 0) continue;
                if (!mbar_wait_bounded(bar_tmem_empty, (acc_iter & 1u) ^ 1u, abort_flag, g.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < t.num_kt; kt += C::kSub) {
                    const int nsub = t.num_kt - kt < C::kSub ? t.num_kt - kt : C::kSub;
                    if (!mbar_wait_bounded(bar_full + 8 * stage, phase, abort_flag, g.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int sub = 0; sub < C::kSub; ++sub) {
                        if (sub < nsub) {
                            const int slot = stage * C::kSub + sub;
                            const uint32_t sfa_t = tmem_base + C::kTmemSFA + 4 * slot;
                            const uint32_t sfb_t = tmem_base + C::kTmemSFB + 8 * slot;
                            tc_cp_32x128b_warpx4_g<NC>(sfa_t, smem_desc(sbase + C::kOffSFA + slot * 512, 0, 128, 0));
                            const uint32_t sfb_s = sbase + C::kOffSFB + slot * C::kSfbSlot;
                            if constexpr (kEpi == kEpiSwiglu || SFB1) {
                                // one copy of each of the two atoms: columns 0-3 and 4-7, replicated
                                // into every lane quarter
                                tc_cp_32x128b_warpx4_g<NC>(sfb_t, smem_desc(sfb_s, 0, 128, 0));
                                tc_cp_32x128b_warpx4_g<NC>(sfb_t + 4, smem_desc(sfb_s + 512, 0, 128, 0));
                            } else {
                                // every lane quarter needs all 256 B scales: lane l of quarter q
                                // takes row l of atom 0 (columns 0-3) and of atom 1 (columns 4-7)
                                // from copy q of each atom (rows 16 B apart, atom 1 at +2 KiB)
                                tc_cp_128x256b_g<NC>(sfb_t, smem_desc(sfb_s, 2048, 128, 0));
                            }
                            const uint64_t adesc = smem_desc(sbase + C::kOffA + slot * C::kABytes, 16, 1024, 2);
                            const uint64_t bdesc = smem_desc(sbase + C::kOffB + slot * C::kBBytes, 16, 1024, 2);
#pragma unroll
                            for (int k = 0; k < BK / 32; ++k) {
                                const uint32_t idesc =
                                    idesc0 | (static_cast<uint32_t>(k) << 29) | (static_cast<uint32_t>(k) << 4);
                                mma_mxf8_g<NC>(tmem_base, adesc + static_cast<uint64_t>((k * 32) >> 4),
                                               bdesc + static_cast<uint64_t>((k * 32) >> 4), idesc, sfa_t, sfb_t,
                                               (kt + sub > 0 || k > 0) ? 1u : 0u);
                            }
                        }
                    }
                    if constexpr (kPM) tc_commit_mc1(bar_empty + 8 * stage, static_cast<uint16_t>(0x3));
                    else tc_commit_g<NC>(bar_empty + 8 * stage, fill_ctas);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_g<NC>(bar_tmem_full, pair_ctas);
                ++acc_iter;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(g.dev_err, MX_DEVERR_TIMEOUT);
            }
            // every tcgen05 operation this thread issued has finished once this arrives
            tc_commit_g<NC>(bar_drain, static_cast<uint16_t>(1u << crank));
            mbar_wait_timeout(bar_drain, 0, kWaitLimitNs / 4);
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                       // TMEM lane quarter this warp may access
        const int half = (warp - kEpiWarp0) >> 2;     // column half of the 256-wide tile
        const int row = q * 32 + lane;                // accumulator row owned by this thread
        uint32_t acc_iter = 0;
        for (int64_t L = unit; L < total_tiles; L += num_units) {
            const Tile t = get_tile<NC, MP>(g, table, L, rank, pp);
            const bool row_ok = row < t.valid_rows;
            if (t.num_kt == 0) {
                if (kEpi == kEpiF32 && row_ok) {   // expert without tokens: its weight gradient is zero
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
            if (lane == 0) okw = mbar_wait_bounded(bar_tmem_full, acc_iter & 1u, abort_flag, g.wait_limit_ns) ? 1u : 0u;
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
            if constexpr (kEpi == kEpiSwiglu) {
                if (!epilogue_swiglu<NC>(g, t, tmem_base + (static_cast<uint32_t>(q * 32) << 16), q, half,
                                         warp - kEpiWarp0, lane, row, lead_tmem_empty, bar_epi, acc_iter,
                                         reinterpret_cast<float*>(smem + C::kOffEpi) + (warp - kEpiWarp0) * C::kEpiStage,
                                         smem + C::kOffEpiAtoms, abort_flag)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        atomicOr(g.dev_err, MX_DEVERR_TIMEOUT);
                    }
                    break;
                }
            } else if (kEpi == kEpiBf16) {
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
                // The release only says "the accumulator has been read": every lane's TMEM loads
                // completed at tcgen05.wait::ld, and no memory written here is consumed by the MMA
                // issuer, so a relaxed arrive suffices.  A cluster-scope release arrive cost ~2000
                // cycles per tile boundary, all of it idle tensor-pipe time.
                if (lane == 0) mbar_arrive_cluster_relaxed(lead_tmem_empty);
                if (row_ok) {
                    // a thread writes 256 bytes of its row: as 32-byte stores each fills one L2
                    // sector (16-byte stores would write every sector in two halves); marked
                    // evict-first so the streamed output does not push operand tiles out of L2
                    uint16_t* dst = static_cast<uint16_t*>(g.out) + (t.out_row0 + row) * g.n_out;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int64_t col = t.out_col0 + half * 128 + c * 32;
                        if (col < g.n_out) {
                            if (g.wide_store) {
#pragma unroll
                                for (int j = 0; j < 2; ++j)
                                    st_global_v8(dst + col + 16 * j, packed[c][8 * j], packed[c][8 * j + 1],
                                                 packed[c][8 * j + 2], packed[c][8 * j + 3], packed[c][8 * j + 4],
                                                 packed[c][8 * j + 5], packed[c][8 * j + 6], packed[c][8 * j + 7],
                                                 l2_policy_evict_first());
                            } else {
                                uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    d4[j] = make_uint4(packed[c][4 * j], packed[c][4 * j + 1], packed[c][4 * j + 2],
                                                       packed[c][4 * j + 3]);
                            }
                        }
                    }
                }
            } else {
                // fp32 out: all 128 columns into registers, release the accumulator, then store
                uint32_t r[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + c * 32, r[c]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(lead_tmem_empty);   // as in the bf16 path
                if (row_ok) {
                    float* dst = static_cast<float*>(g.out) + (t.out_row0 + row) * g.n_out;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int64_t col = t.out_col0 + half * 128 + c * 32;
                        if (col < g.n_out) {
                            if (g.wide_store) {   // whole-sector stores, as in the bf16 path
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    st_global_v8(dst + col + 8 * j, r[c][8 * j], r[c][8 * j + 1], r[c][8 * j + 2],
                                                 r[c][8 * j + 3], r[c][8 * j + 4], r[c][8 * j + 5], r[c][8 * j + 6],
                                                 r[c][8 * j + 7], l2_policy_evict_first());
                            } else {
                                uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    d4[j] = make_uint4(r[c][4 * j], r[c][4 * j + 1], r[c][4 * j + 2], r[c][4 * j + 3]);
                            }
                        }
                    }
                }
            }
            ++acc_iter;
        }
    }

    // both CTAs of a pair finish (and the leader's copies drain) before TMEM is freed
    tc_fence_before();
    if (NC * MP > 1) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_g<NC>(tmem_base, kTmemCols);
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

// 2-D map of E4M3 codes [rows x cols], boxes of 128 bytes x box_rows, 128-byte swizzle.
bool make_operand_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map of E4M3 codes [rows x cols] in the blocked code layout (128 x 128 blocks of 16 KiB,
// row-block major): (128 bytes, 128 rows, cols / 128 blocks, rows / 128 blocks).  A box of
// {128, 128, 1, n} is n consecutive row blocks of one 128-column K step -- in shared memory the
// same 128 n rows x 128 bytes, with the same 128-byte swizzle, as the row-major map's box.
bool make_blocked_operand_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(BK), 128, static_cast<cuuint64_t>(cols / BK),
                          static_cast<cuuint64_t>(rows / 128)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(BK) * 128,
                             static_cast<cuuint64_t>(cols) * 128};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(BK), 128, 1, box_rows / 128};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map of a scale buffer in the tensor-core layout: (256 bytes, 2 halves of an
// atom, K groups, 128-row blocks).  A box of {256, 2, 1, n} is n whole 512-byte atoms
// of consecutive row blocks; reads past the buffer are zero-filled.
bool make_scale_map(CUtensorMap* m, const void* base, int64_t row_blocks, int64_t groups, uint32_t box_blocks) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[4] = {256, 2, static_cast<cuuint64_t>(groups), static_cast<cuuint64_t>(row_blocks)};
    cuuint64_t strides[3] = {256, 512, static_cast<cuuint64_t>(512 * groups)};
    cuuint32_t box[4] = {256, 2, 1, box_blocks};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map of a scale buffer in the four-copy layout (each 512-byte atom stored four times,
// 2 KiB per 128-row block and K group): (256 bytes, 8 quarter-KiB pieces, K groups, 128-row
// blocks).  A box of {256, 2, 1, 1} is the first copy of one atom; {256, 8, 1, n} all four
// copies of n consecutive row blocks.
bool make_scale_map_x4(CUtensorMap* m, const void* base, int64_t row_blocks, int64_t groups, uint32_t box_pieces,
                       uint32_t box_blocks) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[4] = {256, 8, static_cast<cuuint64_t>(groups), static_cast<cuuint64_t>(row_blocks)};
    cuuint64_t strides[3] = {256, 2048, static_cast<cuuint64_t>(2048 * groups)};
    cuuint32_t box[4] = {256, box_pieces, 1, box_blocks};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kEpi, int NC, bool SFB1, int MP = 1>
int launch_variant(const GemmProblem& pr, const GemmArgs& g, int dev, int num_sms, cudaStream_t stream) {
    using C = Cfg<NC, kEpi, SFB1>;
    constexpr int CL = NC * MP;   // CTAs per cluster
    static bool attr_set[64] = {false};
    static int units[64] = {0};   // co-resident units (clusters) of this variant, per device
    auto kern = grouped_gemm_kernel<kEpi, NC, SFB1, MP>;
    const uint32_t smem_bytes = kEpi == kEpiSwiglu ? C::kSmemBytesSwiglu : C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes)) !=
            cudaSuccess)
            return MX_ERR_CUDA;
        // one unit per cluster that can actually be resident at once, so no unit of the
        // persistent grid waits for another to finish before it starts
        cfg.gridDim = dim3(static_cast<unsigned>((num_sms / CL) * CL), 1, 1);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = num_sms / CL;
        units[dev] = n < num_sms / CL ? n : num_sms / CL;
        attr_set[dev] = true;
    }
    CUtensorMap tmA, tmB, tmSFA, tmSFB;
    const int64_t a_rb = pr.kind == kGemmRows ? round_up(pr.a_rows + 127 * static_cast<int64_t>(pr.E), 128) / 128
                                              : ceil_div(pr.a_rows, 128);
    // MP = 2: each CTA copies (and multicasts) half of its 128 A rows
    if (!make_operand_map(&tmA, pr.A, pr.a_rows, pr.a_cols, (NC == 2 && MP == 2) ? BM / 2 : BM)) return MX_ERR_CUDA;
    if (pr.b_blocked) {
        if (pr.b_rows % 128 != 0 || pr.b_cols % BK != 0) return MX_ERR_UNSUPPORTED;
        if (!make_blocked_operand_map(&tmB, pr.B, pr.b_rows, pr.b_cols, C::kBRows)) return MX_ERR_CUDA;
    } else if (!make_operand_map(&tmB, pr.B, pr.b_rows, pr.b_cols, (NC == 1 && MP == 2) ? C::kBRows / 2 : C::kBRows)) {
        return MX_ERR_CUDA;
    }
    if (!make_scale_map(&tmSFA, pr.SFA, a_rb, ceil_div(pr.a_cols, 128), 1)) return MX_ERR_CUDA;
    // B scales: the SwiGLU tiles read (the first copy of) their gate and up atoms, one TMA copy
    // each; the others the two consecutive atoms of their 256 B rows in one TMA copy -- all four
    // copies of each (4 KiB) in the four-copy layout, one of each (1 KiB) in the one-copy layout
    const int64_t b_rb = ceil_div(pr.b_rows, 128), b_groups = ceil_div(pr.b_cols, 128);
    const uint32_t b_box_blocks = kEpi == kEpiSwiglu ? 1 : 2;
    if (pr.b_scales_x1) {
        if (!make_scale_map(&tmSFB, pr.SFB, b_rb, b_groups, b_box_blocks)) return MX_ERR_CUDA;
    } else {
        if (!make_scale_map_x4(&tmSFB, pr.SFB, b_rb, b_groups, kEpi == kEpiSwiglu ? 2 : 8, b_box_blocks))
            return MX_ERR_CUDA;
    }
    // a small problem gets no more units than it can have tiles (an upper bound from the host's
    // sizes; the exact count lives on the device): idle units would still allocate tensor memory
    // and join the start-up barriers
    constexpr bool kPM = NC == 1 && MP == 2;   // list entries are M-tile pairs
    const int64_t nt_host = kPM ? (pr.n_out + BN - 1) / BN : ((pr.n_out + BN - 1) / BN + MP - 1) / MP;
    int64_t mt_host = pr.kind == kGemmRows
                          ? (pr.a_rows + static_cast<int64_t>(C::kTileM - 1) * pr.E) / C::kTileM
                          : static_cast<int64_t>(pr.E) * ((pr.m_out + C::kTileM - 1) / C::kTileM);
    if (kPM)   // sum over experts of ceil(m_e / 2) <= (sum m_e + E) / 2
        mt_host = pr.kind == kGemmRows
                      ? (mt_host + pr.E + 1) / 2
                      : static_cast<int64_t>(pr.E) * (((pr.m_out + C::kTileM - 1) / C::kTileM + 1) / 2);
    const int64_t tiles_bound = mt_host * nt_host;
    const int64_t grid_units = tiles_bound < units[dev] ? (tiles_bound > 0 ? tiles_bound : 1) : units[dev];
    cfg.gridDim = dim3(static_cast<unsigned>(grid_units * CL), 1, 1);
    if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSFA, tmSFB, g) != cudaSuccess) return MX_ERR_CUDA;
    return MX_OK;
}

}  // namespace

int launch_grouped_gemm(const GemmProblem& pr, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MX_ERR_CUDA;
    static int num_sms[64] = {0};
    if (dev < 0 || dev >= 64) return MX_ERR_CUDA;
    if (num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return MX_ERR_CUDA;
        num_sms[dev] = n;
    }
    GemmArgs g;
    g.kind = pr.kind;
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
    g.swiglu_i = pr.swiglu_i;
    g.h_qrow = pr.h_qrow;
    g.h_sfrow = pr.h_sfrow;
    g.h_qcol = pr.h_qcol;
    g.h_sfcol = pr.h_sfcol;
    g.h_ldcol = pr.h_ldcol;
    g.h_sfrow_copies = pr.h_sfrow_copies;
    g.wide_store = (reinterpret_cast<uintptr_t>(pr.out) & 31u) == 0 ? 1 : 0;
    g.h_sfcol_copies = pr.h_sfcol_copies;
    g.wait_limit_ns = pr.wait_limit_ns > 0 ? pr.wait_limit_ns : kWaitLimitNs;
    g.withhold_operands = pr.withhold_operands;
    g.raster_group = pr.raster_group;
    g.b_blocked = pr.b_blocked;
    const int n = num_sms[dev];
    if (pr.swiglu_i > 0)   // the SwiGLU tiles read one atom of each B scale block, in either layout
        return launch_variant<kEpiSwiglu, 2, false>(pr, g, dev, n, stream);
    // CTAs per MMA: 2 (SM pairs sharing B, 256-row tiles) unless requested otherwise, or unless
    // the experts average fewer than 512 rows: then an expert's last, partly filled tile is a
    // large share of its work, and 128-row single-CTA tiles waste less of the tensor pipe on
    // padding rows (measured on 128 experts of ~256 rows: 3-4 % faster)
    const bool one = pr.ctas_per_mma == 1 ||
                     (pr.ctas_per_mma == 0 && pr.kind == kGemmRows && pr.a_rows < 512 * static_cast<int64_t>(pr.E));
    const bool x1 = pr.b_scales_x1 != 0;
    // Clusters sharing an operand by multicast only on request.  CTA pairs, two per cluster,
    // sharing A: A's reads from L2 halve, but only 36 four-CTA clusters fit on the 152 SMs (the
    // GPCs' SM counts are not all multiples of four), so 8 SMs idle; at the MoE FFN shapes it is
    // no faster (forward within 1 %, wgrad1 3 % slower).  Single CTAs, two per cluster, sharing
    // B: 13-15 % slower on the skewed 128-expert shapes (the two CTAs wait for each other at
    // every stage, and an expert with an odd M-tile count computes one idle tile).
    const bool mp2 = pr.cluster_pairs == 2;
    if (pr.kind == kGemmRows) {
        if (one && mp2) return x1 ? launch_variant<kEpiBf16, 1, true, 2>(pr, g, dev, n, stream)
                                  : launch_variant<kEpiBf16, 1, false, 2>(pr, g, dev, n, stream);
        if (one) return x1 ? launch_variant<kEpiBf16, 1, true>(pr, g, dev, n, stream)
                           : launch_variant<kEpiBf16, 1, false>(pr, g, dev, n, stream);
        if (mp2) return x1 ? launch_variant<kEpiBf16, 2, true, 2>(pr, g, dev, n, stream)
                           : launch_variant<kEpiBf16, 2, false, 2>(pr, g, dev, n, stream);
        return x1 ? launch_variant<kEpiBf16, 2, true>(pr, g, dev, n, stream)
                  : launch_variant<kEpiBf16, 2, false>(pr, g, dev, n, stream);
    }
    if (one && mp2) return x1 ? launch_variant<kEpiF32, 1, true, 2>(pr, g, dev, n, stream)
                              : launch_variant<kEpiF32, 1, false, 2>(pr, g, dev, n, stream);
    if (one) return x1 ? launch_variant<kEpiF32, 1, true>(pr, g, dev, n, stream)
                       : launch_variant<kEpiF32, 1, false>(pr, g, dev, n, stream);
    if (mp2) return x1 ? launch_variant<kEpiF32, 2, true, 2>(pr, g, dev, n, stream)
                       : launch_variant<kEpiF32, 2, false, 2>(pr, g, dev, n, stream);
    return x1 ? launch_variant<kEpiF32, 2, true>(pr, g, dev, n, stream)
              : launch_variant<kEpiF32, 2, false>(pr, g, dev, n, stream);
}

}  // namespace mx
