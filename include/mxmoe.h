/*
 * mxmoe.h -- C ABI of the GB300 (sm_103a) MXFP8 MoE hot path:
 *   bf16 -> MXFP8 quantizer (rowwise / columnwise, scales written in the layout
 *   the tensor core's block-scaled MMA reads), token permutation by expert, and
 *   expert grouped GEMMs (forward, dgrad, wgrad) with block scaling applied inside
 *   tcgen05.mma.
 *
 * Sources (page title and section):
 *  [P1] aigc.bar, "Blackwell性能陷阱？Cursor揭秘：重写内核让AI大模型MoE提速3.5倍的底层逻辑":
 *       section "1. Blackwell的TMEM架构瓶颈" (microscaling, TMEM accumulators),
 *       section "2. 被忽视的“量化税”" (quantization cost forward and, doubled, backward),
 *       section "破局之道：从零构建，释放硬件真正潜能" (tcgen05.mma applies the MX scales in
 *       hardware; warp specialization; 2-CTA; expert-wise supergrouping for grouped GEMM),
 *       section "“秘密武器”：自研量化内核与最佳精度配方" (E4M3, block 32, a quantizer whose output
 *       layout matches the MMA instruction so that no reshape step is needed).
 *  [P3] kucoin.com, "Cursor's MoK демонстрирует повышение производительности на 2,37x на NVIDIA
 *       GB300 NVL72", section "01" (count tokens per expert, place them contiguously).
 *  [P4] lpnh.cn blog, section "1. 为什么 MoE 内核在 Blackwell 上反而变慢了" (divide by the block
 *       scale, then convert; backward needs a transpose-quantize).
 *  The pages give no API; these calls restate their problem statement.  Rules the
 *  pages leave open follow the OCP Microscaling v1.0 specification: scale byte =
 *  E8M0 of 2^(floor(log2 amax) - 8), elements E4M3 round-to-nearest-even with
 *  saturation to +-448, an all-zero block takes scale byte 0x00.
 *
 * Conventions shared by every call:
 *  - Every pointer argument is a DEVICE pointer owned by the caller.  The library
 *    never allocates or frees memory, never synchronizes, and never reads device
 *    memory from the host.  Each call enqueues kernels on `stream` and returns.
 *  - Synchronous errors (bad sizes, null or misaligned pointers, unsupported
 *    shapes, a launch failure) come back as a negative mx_status and nothing is
 *    enqueued.  Asynchronous errors found by the kernels are OR-ed into the int at
 *    `dev_err` (MX_DEVERR_* bits); the caller reads it after synchronizing.  The
 *    kernels never clear it.
 *  - Group offsets (off, poff) stay on the device; no call copies them to the host.
 *  - Results are deterministic: no floating-point atomics.
 *  - "Scale layout" (SF layout) below always means: the [rows x kb] matrix of E8M0
 *    bytes (kb = cols / 32 blocks per row) padded to rows % 128 == 0 and
 *    kb % 4 == 0, cut into 128 x 4 atoms of 512 bytes stored atom-row-major
 *    (atom (i, j) at byte (i * ceil4(kb) / 4 + j) * 512); inside an atom entry
 *    (r, c) sits at (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4).  Padding
 *    entries written by this library are 0.  Size: mx_sf_bytes(rows, kb).
 *  - "Four-copy scale layout" (SF4 layout): the SF layout with every 512-byte atom
 *    stored four times in a row, atom (i, j) in bytes [(i * ceil4(kb) / 4 + j) * 2048,
 *    + 2048).  Size: mx_sf_bytes_x4(rows, kb).  The grouped GEMMs take the scales of
 *    their B operand (SFB, SFW1, SFWt, SFXc) in this layout by default: each 32-lane
 *    quarter of the tensor memory needs the scales of all 256 B rows of a tile, and with
 *    four copies in shared memory one 128x256b tensor-memory copy per K step delivers
 *    them (instead of two replicating copies).  The *_ex GEMM calls with the flag
 *    MX_GEMM_B_SCALES_X1 take B-operand scales in the plain SF layout instead (the layout
 *    of every A operand, and of library block-scaled GEMMs), at the cost of one more
 *    tensor-memory copy per K step.  The quantizing calls write either layout per output
 *    form (mode bits MX_ROWWISE_X4, MX_COLWISE_X4).
 *  - "Blocked code layout": E4M3 codes of a [rows x cols] operand (rows % 128 == 0,
 *    cols % 128 == 0) stored as 128 x 128 blocks of 16 KiB, each row-major, block (i, j)
 *    (rows 128i.., columns 128j..) at bytes [(i * cols / 128 + j) * 16384, + 16384): code
 *    (r, c) at (r / 128 * cols / 128 + c / 128) * 16384 + (r % 128) * 128 + c % 128.  A
 *    weight tile that the grouped GEMMs stage per K step (128 B x 128 or 256 rows) is then
 *    one or two contiguous 16 KiB pieces instead of 128-byte pieces of rows cols bytes
 *    apart, which streams from HBM at a higher rate when the weights are read only once
 *    (experts with few rows).  Written by the quantizing calls with the mode bits
 *    MX_ROWWISE_BLK / MX_COLWISE_BLK; read by the *_ex GEMM calls with MX_GEMM_B_BLOCKED.
 */
#ifndef MXMOE_H
#define MXMOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MX_API __attribute__((visibility("default")))
#else
#define MX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime and driver stream handles are the same type).
 * NULL selects the legacy default stream. */
typedef struct CUstream_st* mx_stream_t;

typedef enum {
    MX_OK = 0,
    MX_ERR_INVALID_ARG = -1, /* a size, count or mode is out of range, or a required pointer is NULL */
    MX_ERR_ALIGNMENT = -2,   /* a pointer or leading dimension breaks the 16-byte rule stated per call */
    MX_ERR_UNSUPPORTED = -3, /* a shape this build does not handle (stated per call) */
    MX_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed (no device, launch error, ...) */
    MX_ERR_TIMEOUT = -5,     /* reserved for callers that map MX_DEVERR_TIMEOUT to a status */
    MX_ERR_TOO_LARGE = -6    /* moe_permute_noalloc: the problem needs more than its fixed scratch */
} mx_status;

/* Bits OR-ed into *dev_err by the kernels. */
enum {
    MX_DEVERR_BAD_EXPERT_ID = 1, /* moe_permute: a routing id outside [0, E); that slot is dropped */
    MX_DEVERR_TIMEOUT = 2,       /* a pipeline wait in the grouped GEMM exceeded its time limit; outputs invalid */
    MX_DEVERR_BAD_SEGMENTS = 4   /* segment offsets that are not monotone or exceed the stated bounds */
};

/* mode bitmask of the quantizing calls: MX_ROWWISE and/or MX_COLWISE (both from one read);
 * MX_ROWWISE_X4 / MX_COLWISE_X4 (each only with its form) write that form's scales in the
 * SF4 layout (B operands of the grouped GEMMs); MX_ROWWISE_BLK / MX_COLWISE_BLK (each only
 * with its form) write that form's codes in the blocked code layout */
enum { MX_ROWWISE = 1, MX_COLWISE = 2, MX_ROWWISE_X4 = 4, MX_COLWISE_X4 = 8, MX_ROWWISE_BLK = 16,
       MX_COLWISE_BLK = 32 };
enum { MX_DTYPE_BF16 = 0, MX_DTYPE_F32 = 1 };     /* input element type for mxfp8_quantize_ex */
/* flags of the grouped-GEMM *_ex calls: MX_GEMM_B_SCALES_X1, B-operand scales in the plain SF
 * layout (one copy of each atom) instead of the SF4 layout; MX_GEMM_B_BLOCKED, B-operand codes
 * (B, W1, Wt, Xc) in the blocked code layout instead of row-major */
enum { MX_GEMM_B_SCALES_X1 = 1, MX_GEMM_B_BLOCKED = 2 };
enum { MX_SCALE_FLOOR = 0, MX_SCALE_RCEIL = 1 };  /* scale rule for mxfp8_quantize_ex (see there) */

/* Bytes of a scale array in the SF layout for a [rows x kb] scale matrix:
 * ceil128(rows) * ceil4(kb).  Returns 0 for negative arguments. */
MX_API size_t mx_sf_bytes(int64_t rows, int64_t kb);

/* Bytes of a scale array in the SF4 layout: 4 * mx_sf_bytes(rows, kb). */
MX_API size_t mx_sf_bytes_x4(int64_t rows, int64_t kb);

/* Upper bound of the padded row count poff[E] = sum_e ceil128(T_e) for R routed
 * rows over E experts: ceil128(R + 127 * E).  Buffers indexed by padded
 * positions (scale rows of the permuted operand, columns of the columnwise
 * operand) are sized with it, because the exact value lives on the device. */
MX_API int64_t mx_padded_rows_bound(int64_t R, int64_t E);

/*
 * mxfp8_quantize -- bf16 -> MXFP8 (E4M3 elements, one E8M0 scale per 32
 * elements).  [P1] "“秘密武器”", [P4] section 1; rule as stated at the top.
 *
 * x       bf16 [rows x cols], row-major, cols % 32 == 0, 16-byte aligned (32-byte
 *         aligned, as device allocations are, lets full 128 x 128 tiles take 256-bit
 *         loads; the results are the same either way).
 * mode    MX_ROWWISE, MX_COLWISE or both (one read of x feeds both outputs), plus
 *         MX_ROWWISE_X4 / MX_COLWISE_X4 for scales in the SF4 layout (then size that
 *         scale buffer with mx_sf_bytes_x4 instead of mx_sf_bytes), plus
 *         MX_ROWWISE_BLK / MX_COLWISE_BLK for that form's codes in the blocked code
 *         layout (same buffer sizes): q_row as the blocked [rows x cols] matrix (needs
 *         nseg == 0, rows % 128 == 0, cols % 128 == 0), q_col as the blocked
 *         [cols x ld_col] matrix (needs cols % 128 == 0).  Other combinations return
 *         MX_ERR_INVALID_ARG.
 * Segments (optional; nseg == 0 means one segment of all rows, with
 *   off = {0, rows} and poff = {0, ceil128(rows)} implied):
 *   seg_off[nseg+1]   device int32, exclusive scan of the segment row counts;
 *                     segment g is rows [seg_off[g], seg_off[g+1]) of x.
 *   seg_poff[nseg+1]  device int32, exclusive scan of ceil128 of those counts:
 *                     the segment's first padded position.  These are the off and
 *                     poff arrays moe_permute produces (segments = experts).
 *   rows must equal seg_off[nseg]; seg_poff[nseg] must not exceed
 *   mx_padded_rows_bound(rows, nseg) (violations set MX_DEVERR_BAD_SEGMENTS).
 * Rowwise outputs (mode & MX_ROWWISE):
 *   q_row   uint8 [rows x cols] E4M3 codes, row-major, same row order as x.
 *   sf_row  scale bytes in the SF layout for a [P x cols/32] matrix where the
 *           scale row of x's row seg_off[g] + l is row seg_poff[g] + l; rows
 *           seg_poff[g] + l for l >= T_g (padding) are written as 0.
 *           P = seg_poff[nseg]; size the buffer with mx_sf_bytes(Pbound, cols/32),
 *           Pbound = ceil128(rows) without segments, else mx_padded_rows_bound(rows, nseg).
 * Columnwise outputs (mode & MX_COLWISE), the transposed operand of the backward
 * pass ([P4] section 1, "transpose-quantize"):
 *   q_col   uint8 [cols x ld_col] E4M3 codes: element (c, p) at q_col[c * ld_col + p],
 *           p a padded position; blocks are 32 consecutive positions of one
 *           column inside one segment; positions past a segment's rows are 0.
 *   sf_col  scale bytes in the SF layout for a [cols x ld_col/32] matrix.
 *   ld_col  a multiple of 128, >= ceil128(rows) and >= seg_poff[nseg] (a tile
 *           whose positions would pass ld_col sets MX_DEVERR_BAD_SEGMENTS and
 *           is skipped); Pbound (above) is always large enough.  Positions
 *           >= seg_poff[nseg] are not written.
 * dev_err  optional (may be NULL); receives MX_DEVERR_BAD_SEGMENTS.
 * Returns MX_OK, MX_ERR_INVALID_ARG (rows/cols out of range, cols % 32 != 0,
 * bad mode, a needed output NULL, ld_col below ceil128(rows) or not a multiple
 * of 128), MX_ERR_ALIGNMENT (x, q_row,
 * q_col not 16-byte aligned, sf_* not 16-byte aligned) or MX_ERR_CUDA.
 */
MX_API int mxfp8_quantize(const void* x, int64_t rows, int64_t cols, int mode,
                   const int32_t* seg_off, const int32_t* seg_poff, int nseg, int64_t ld_col,
                   uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                   int* dev_err, mx_stream_t stream);

/*
 * mxfp8_quantize_ex -- mxfp8_quantize with a choice of input type and scale rule.
 * dtype       MX_DTYPE_BF16 (as mxfp8_quantize) or MX_DTYPE_F32 (fp32 input; the
 *             quantizer benchmark pseudo-code of the lpnh.cn page, section "4. 验证请求与
 *             成功结果", reads float input); x is then fp32 [rows x cols].
 * scale_rule  MX_SCALE_FLOOR: the OCP MX rule stated at the top (the default of
 *             mxfp8_quantize).  MX_SCALE_RCEIL: the smallest power of two X with
 *             amax <= 448 X (the ceiling rule of NVIDIA TransformerEngine's MXFP8 recipe,
 *             the library the aigc.bar page names in section "破局之道"); no element saturates.
 * Everything else as mxfp8_quantize.  mxfp8_quantize == mxfp8_quantize_ex(BF16, FLOOR).
 */
MX_API int mxfp8_quantize_ex(const void* x, int dtype, int scale_rule, int64_t rows, int64_t cols, int mode,
                             const int32_t* seg_off, const int32_t* seg_poff, int nseg, int64_t ld_col,
                             uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                             int* dev_err, mx_stream_t stream);

/*
 * mxfp8_gather_quantize -- quantize-on-gather: the result of mxfp8_quantize on the
 * expert-ordered tensor X_perm [R x cols] with X_perm row r = x row src_row[r] and
 * the experts as segments (seg_off = off, seg_poff = poff), computed in one pass
 * that reads x through src_row, so X_perm is never written.  (kucoin.com MoK page,
 * section "02": MXFP8 quantization folded into the dispatch data path instead of a
 * separate quantization kernel.)
 * x        bf16 [T x cols] in token order; src_row/off/poff as produced by moe_permute
 *          (R = off[E] routed rows).  An index outside [0, T) reads as a zero row and
 *          sets MX_DEVERR_BAD_SEGMENTS in *dev_err (required here).
 * Outputs, ld_col and errors exactly as mxfp8_quantize with nseg = E and rows = R.
 * Tiles run in column-slice order (all row tiles of 128 columns, then the next 128), so a
 * slice of x stays in L2 while the k routed copies of each token row read it.
 */
MX_API int mxfp8_gather_quantize(const void* x, int64_t T, int64_t cols, int mode, const int32_t* src_row,
                                 const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t ld_col,
                                 uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                                 int* dev_err, mx_stream_t stream);

/*
 * mxfp8_gather_quantize_ex -- mxfp8_gather_quantize of a row-scaled gather: X_perm row r =
 * bf16(row_scale[r] * x row src_row[r]) (fp32 product, rounded to nearest even), quantized as
 * above.  With x the output gradient dOut [T x cols] in token order and row_scale[r] the
 * routing weight of routed row r (moe_combine_bwd_ex writes it), X_perm is the combine
 * backward's dY [R x cols] -- quantized straight from dOut, so dY is never written or read
 * in bf16 (kucoin.com MoK page, section "02": quantization folded into the data path).
 * row_scale: device fp32 [R] in expert order, or NULL (= mxfp8_gather_quantize).  The rows'
 * scale bytes and codes are exactly those of mxfp8_quantize on the materialized X_perm.
 */
MX_API int mxfp8_gather_quantize_ex(const void* x, int64_t T, int64_t cols, int mode, const int32_t* src_row,
                                    const float* row_scale, const int32_t* off, const int32_t* poff, int E,
                                    int64_t R, int64_t ld_col, uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col,
                                    uint8_t* sf_col, int* dev_err, mx_stream_t stream);

/*
 * mxfp8_swiglu_quantize -- SwiGLU fused with MXFP8 quantization of its result (kucoin.com
 * MoK page, section "02": quantization folded into the SwiGLU step of the data path).
 *   a   bf16 [R x 2I] = [gate | up] (the GEMM1 output, expert order);
 *   h   = silu(gate) * up, computed in fp32 and quantized directly (never stored in bf16):
 *       outputs exactly as mxfp8_quantize of an fp32 [R x I] tensor with the same
 *       mode / segments / ld_col arguments (rowwise = the GEMM2 operand, columnwise over the
 *       expert segments = the wgrad2 operand).  I % 128 == 0.
 */
MX_API int mxfp8_swiglu_quantize(const void* a, int64_t R, int64_t I, int mode,
                                 const int32_t* seg_off, const int32_t* seg_poff, int nseg, int64_t ld_col,
                                 uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                                 int* dev_err, mx_stream_t stream);

/*
 * mxfp8_swiglu_bwd_quantize -- the SwiGLU backward fused with MXFP8 quantization:
 *   dH = [dh * up * s * (1 + gate * (1 - s)) | dh * silu(gate)],  s = sigmoid(gate),
 * for dh bf16 [R x I] (the dgrad2 output) and a as above; dH [R x 2I] is computed in fp32
 * and quantized as mxfp8_quantize of an fp32 [R x 2I] tensor would be (rowwise = the
 * dgrad1 operand, columnwise = the wgrad1 operand).  I % 128 == 0.
 */
MX_API int mxfp8_swiglu_bwd_quantize(const void* dh, const void* a, int64_t R, int64_t I, int mode,
                                     const int32_t* seg_off, const int32_t* seg_poff, int nseg, int64_t ld_col,
                                     uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                                     int* dev_err, mx_stream_t stream);

/* Scratch bytes moe_permute needs for T tokens, top-k, E experts. */
MX_API size_t moe_permute_workspace_bytes(int64_t T, int k, int E);

/*
 * moe_permute -- group routed (token, slot) pairs by expert.  [P3] section "01".
 *
 * topk_ids  device int32 [T x k]: expert of slot j of token t.
 * counts    device int32 [E]     rows routed to each expert.
 * off       device int32 [E+1]   exclusive scan of counts.
 * poff      device int32 [E+1]   exclusive scan of ceil128(counts).
 * src_row   device int32 [T*k]   src_row[off[e] + r] = token of the r-th row of
 *                                expert e; rows are ordered by token, then slot (a
 *                                stable counting sort); entries >= off[E] are -1.
 * dst_of    device int32 [T*k]   destination row of (t, j), or -1 for an invalid id.
 * Optional gather of an already rowwise-quantized activation (all three of
 * q_in, sf_in, q_out non-NULL, plus sf_out; else index-only):
 *   q_in  uint8 [T x K] E4M3 codes, sf_in its scales in the SF layout for [T x K/32];
 *   q_out uint8 [T*k x K]: row off[e] + r = q_in row src_row[off[e] + r];
 *   sf_out scales in the SF layout for [Pbound x K/32], Pbound =
 *          mx_padded_rows_bound(T*k, E): the scale row of output row off[e] + r
 *          is row poff[e] + r; padding rows up to poff[e+1] are 0.
 *   K % 32 == 0; q_in/q_out 16-byte aligned, K % 16 == 0.
 * ws, ws_bytes  scratch of at least moe_permute_workspace_bytes(T, k, E) bytes,
 *               16-byte aligned; its contents are undefined afterwards.
 * dev_err  required; receives MX_DEVERR_BAD_EXPERT_ID for ids outside [0, E).
 * Limits: 1 <= E <= 1024, 1 <= k <= 64, T*k < 2^31.
 */
MX_API int moe_permute(const int32_t* topk_ids, int64_t T, int k, int E,
                int32_t* counts, int32_t* off, int32_t* poff, int32_t* src_row, int32_t* dst_of,
                const uint8_t* q_in, const uint8_t* sf_in, int64_t K,
                uint8_t* q_out, uint8_t* sf_out,
                void* ws, size_t ws_bytes, int* dev_err, mx_stream_t stream);

/*
 * moe_permute_noalloc -- moe_permute for callers that cannot allocate device memory
 * (no counterpart on the pages: it exists for callers that hold no allocator at the
 * point of routing, or may not trigger cudaMalloc's device-wide synchronization).
 * Same arguments, results and errors as moe_permute, without ws / ws_bytes: the
 * scratch is a fixed 1 MiB array in the library's device image, so the problem must
 * satisfy moe_permute_workspace_bytes(T, k, E) <= 1 MiB, i.e. roughly
 * ceil(T*k / 2048) * E <= 131070; larger problems return MX_ERR_TOO_LARGE and
 * enqueue nothing.  The call itself calls no allocation routine (no cudaMalloc, no
 * cudaFree, nothing of torch's).  The array is created by the CUDA module loader when the
 * library's device code is loaded on a device; with lazy module loading (the CUDA default)
 * that happens at the first use on that device, which may allocate and synchronize the
 * device.  So make the first call on each device during set-up: it also looks up the
 * array's device address (cudaGetSymbolAddress, with that device current) and caches it
 * per device, which must happen before any stream capture.  The cached address belongs to
 * the device's context: after cudaDeviceReset in the same process the call must not be
 * used again.  Every call on a device shares the one array: calls whose kernels may
 * overlap on the GPU (other streams, unordered host threads) race on it and must be
 * serialized by the caller.  No scratch word needs clearing between calls: every word the
 * kernels read is written earlier in the same call.
 */
MX_API int moe_permute_noalloc(const int32_t* topk_ids, int64_t T, int k, int E,
                               int32_t* counts, int32_t* off, int32_t* poff, int32_t* src_row, int32_t* dst_of,
                               const uint8_t* q_in, const uint8_t* sf_in, int64_t K,
                               uint8_t* q_out, uint8_t* sf_out, int* dev_err, mx_stream_t stream);

/*
 * moe_gather_rows -- dst row r = src row src_row[r] for r < R (rows with
 * src_row[r] < 0 are left untouched).  Used to bring bf16 activations into
 * expert order for the wgrad operand ([P3] section "01").  row_bytes % 16 == 0,
 * src/dst 16-byte aligned.
 */
MX_API int moe_gather_rows(const void* src, int64_t row_bytes, const int32_t* src_row, int64_t R,
                    void* dst, mx_stream_t stream);

/*
 * moe_combine_fwd -- unpermute / combine: the final weighted merge of the expert
 * outputs back to token order (kucoin.com MoK page, section "03").
 *   out[t][h] = bf16( sum_j gate[t][j] * Y[dst_of[t][j]][h] ), fp32 accumulation.
 * Y       bf16 [R x H] expert-ordered rows (e.g. the forward GEMM output).
 * gate    fp32 [T x k] routing weights, or NULL for unit weights (the un-permute sum,
 *         e.g. of the input gradient); dst_of int32 [T x k] from moe_permute.
 * out     bf16 [T x H].  Slots with dst_of = -1 contribute nothing; an entry >= R is
 *         treated the same way and sets MX_DEVERR_BAD_SEGMENTS.
 * H % 8 == 0, 1 <= k <= 64; Y/out 16-byte aligned; dev_err required.
 */
MX_API int moe_combine_fwd(const void* Y, const float* gate, const int32_t* dst_of, int64_t T, int k, int64_t H,
                           int64_t R, void* out, int* dev_err, mx_stream_t stream);

/*
 * moe_combine_bwd -- backward of moe_combine_fwd for output gradient dOut bf16 [T x H]:
 *   dY[dst_of[t][j]][h] = bf16( gate[t][j] * dOut[t][h] )        (rows no slot maps to are untouched)
 *   dgate[t][j]         = sum_h dOut[t][h] * Y[dst_of[t][j]][h]   (fp32, fixed reduction order; 0 if dropped)
 * Same shapes and rules as moe_combine_fwd; dY bf16 [R x H], dgate fp32 [T x k].
 */
MX_API int moe_combine_bwd(const void* dOut, const void* Y, const float* gate, const int32_t* dst_of, int64_t T,
                           int k, int64_t H, int64_t R, void* dY, float* dgate, int* dev_err, mx_stream_t stream);

/*
 * moe_combine_bwd_ex -- moe_combine_bwd with dY optional (NULL: not written) and one more
 * optional output, gate_rows fp32 [R]: gate_rows[dst_of[t][j]] = gate[t][j], the routing weight
 * of every routed row in expert order (the row_scale of mxfp8_gather_quantize_ex; rows no slot
 * maps to are untouched).  dgate as moe_combine_bwd.
 */
MX_API int moe_combine_bwd_ex(const void* dOut, const void* Y, const float* gate, const int32_t* dst_of, int64_t T,
                              int k, int64_t H, int64_t R, void* dY, float* dgate, float* gate_rows, int* dev_err,
                              mx_stream_t stream);

/*
 * grouped_gemm_mxfp8_fwd -- for every expert e:
 *   C[off[e] + m][n] = bf16( sum_k deq(A)[off[e] + m][k] * deq(B_e)[n][k] ),  m < T_e,
 * fp32 accumulation in tensor memory, block scales applied by tcgen05.mma
 * ([P1] "破局之道", "1. Blackwell的TMEM架构瓶颈").
 *   A    uint8 [R x K] E4M3 codes (rows in expert order, as moe_permute writes them).
 *   SFA  A's scales in the SF layout for [Pbound x K/32] with the scale row of
 *        A's row off[e] + m at row poff[e] + m (as moe_permute / mxfp8_quantize
 *        with segments write them).
 *   B    uint8 [E*N x K]: expert e's weight is rows [e*N, (e+1)*N).
 *   SFB  B's scales in the SF4 layout for [E*N x K/32] (mxfp8_quantize with MX_ROWWISE_X4).
 *   off, poff  device int32 [E+1] (from moe_permute); off[E] <= R.
 *   C    bf16 [R x N] row-major; rows >= off[E] are not written.
 * Shapes: N % 128 == 0, K % 128 == 0, 1 <= E <= 1024; pointers 16-byte aligned.
 * dev_err required (MX_DEVERR_TIMEOUT).
 */
MX_API int grouped_gemm_mxfp8_fwd(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                           const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t N, int64_t K,
                           void* C, int* dev_err, mx_stream_t stream);

/* grouped_gemm_mxfp8_fwd with flags: MX_GEMM_B_SCALES_X1 takes SFB in the plain SF layout for
 * [E*N x K/32] (mxfp8_quantize MX_ROWWISE without MX_ROWWISE_X4); MX_GEMM_B_BLOCKED takes B's
 * codes in the blocked code layout of [E*N x K] (mxfp8_quantize with MX_ROWWISE_BLK); 0 is
 * grouped_gemm_mxfp8_fwd.  Unknown flag bits return MX_ERR_INVALID_ARG.  The same two flags
 * apply to every *_ex GEMM call below, each to its own B operand (W1, Wt, Xc). */
MX_API int grouped_gemm_mxfp8_fwd_ex(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                                     const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t N, int64_t K,
                                     void* C, int flags, int* dev_err, mx_stream_t stream);

/*
 * grouped_gemm_mxfp8_fwd_swiglu -- the first expert GEMM with SwiGLU and MXFP8 quantization
 * of its result in the GEMM's epilogue (kucoin.com MoK page, section "02": quantization
 * folded into the grouped GEMM and SwiGLU data path; aigc.bar page, section "“秘密武器”":
 * output written in the layout the next MMA reads).  Same outputs as
 *   grouped_gemm_mxfp8_fwd(A, SFA, W1, SFW1, off, poff, E, R, 2I, K, out1)
 *   mxfp8_swiglu_quantize(out1, R, I, MX_ROWWISE | MX_COLWISE, off, poff, E, ld_col, ...)
 * in one pass: out1 = [gate | up] bf16 [R x 2I] (rows >= off[E] not written), and
 * h = silu(gate) * up formed in fp32 from the bf16 values of out1, quantized
 *   rowwise:    h_qrow uint8 [R x I], h_sfrow in the SF layout for [Pbound x I/32]
 *               (scale row of data row off[e] + m at poff[e] + m);
 *   columnwise: h_qcol uint8 [I x ld_col] (position poff[e] + m; padding positions 0),
 *               h_sfcol in the SF layout for [I x ld_col/32].
 * h_mode: MX_ROWWISE | MX_COLWISE, plus MX_ROWWISE_X4 / MX_COLWISE_X4 to write h_sfrow /
 * h_sfcol in the SF4 layout instead (the columnwise h is the B operand of the second
 * weight gradient).  SFW1 is in the SF4 layout like every B-operand scale array.
 * A, SFA, W1 [E*2I x K] (expert e: rows [e*2I, e*2I + I) gate, [e*2I + I, (e+1)*2I) up),
 * SFW1, off, poff as for grouped_gemm_mxfp8_fwd.  Pbound = mx_padded_rows_bound(R, E).
 * Shapes: I % 128 == 0, K % 128 == 0, ld_col % 128 == 0, ld_col >= Pbound; pointers
 * 16-byte aligned.  Runs on CTA pairs (the pair's CTAs stage the gate and the up rows of
 * one tile).  dev_err required.  The pages give no such call; it is the fused form of
 * the two calls above.
 */
MX_API int grouped_gemm_mxfp8_fwd_swiglu(const uint8_t* A, const uint8_t* SFA, const uint8_t* W1, const uint8_t* SFW1,
                                         const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t I, int64_t K,
                                         void* out1, uint8_t* h_qrow, uint8_t* h_sfrow, uint8_t* h_qcol,
                                         uint8_t* h_sfcol, int64_t ld_col, int h_mode, int* dev_err,
                                         mx_stream_t stream);

/* grouped_gemm_mxfp8_fwd_swiglu with flags (MX_GEMM_B_SCALES_X1: SFW1 in the plain SF layout). */
MX_API int grouped_gemm_mxfp8_fwd_swiglu_ex(const uint8_t* A, const uint8_t* SFA, const uint8_t* W1,
                                            const uint8_t* SFW1, const int32_t* off, const int32_t* poff, int E,
                                            int64_t R, int64_t I, int64_t K, void* out1, uint8_t* h_qrow,
                                            uint8_t* h_sfrow, uint8_t* h_qcol, uint8_t* h_sfcol, int64_t ld_col,
                                            int h_mode, int flags, int* dev_err, mx_stream_t stream);

/*
 * grouped_gemm_mxfp8_dgrad -- for every expert e:
 *   dX[off[e] + m][n] = bf16( sum_k deq(dY)[off[e] + m][k] * deq(Wt)[n][e*K + k] ),
 * the input gradient through expert e's weight W_e [K x N] (forward y = x W_e^T):
 * contraction over the forward output dimension K.
 *   dY   uint8 [R x K] rowwise codes of the output gradient (expert order), SFdY
 *        its scales as SFA of the forward call.
 *   Wt   uint8 [N x E*K]: the columnwise quantization of the stacked weights
 *        [E*K x N] (mxfp8_quantize MX_COLWISE with segment offsets e*K), so
 *        expert e occupies columns [e*K, (e+1)*K); SFWt its scales in the SF4
 *        layout for [N x E*K/32] (MX_COLWISE_X4).
 *   dX   bf16 [R x N].
 * Shapes: N % 128 == 0, K % 128 == 0.  Other rules as for the forward call.
 */
MX_API int grouped_gemm_mxfp8_dgrad(const uint8_t* dY, const uint8_t* SFdY, const uint8_t* Wt, const uint8_t* SFWt,
                             const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t N, int64_t K,
                             void* dX, int* dev_err, mx_stream_t stream);

/* grouped_gemm_mxfp8_dgrad with flags (MX_GEMM_B_SCALES_X1: SFWt in the plain SF layout for
 * [N x E*K/32], i.e. mxfp8_quantize MX_COLWISE without MX_COLWISE_X4). */
MX_API int grouped_gemm_mxfp8_dgrad_ex(const uint8_t* dY, const uint8_t* SFdY, const uint8_t* Wt, const uint8_t* SFWt,
                                       const int32_t* off, const int32_t* poff, int E, int64_t R, int64_t N, int64_t K,
                                       void* dX, int flags, int* dev_err, mx_stream_t stream);

/*
 * grouped_gemm_mxfp8_wgrad -- for every expert e (contraction over its tokens,
 * a length that differs per expert):
 *   dW[e][n][k] = sum_{t < T_e} deq(dYc)[n][poff[e] + t] * deq(Xc)[k][poff[e] + t]   (fp32)
 * and dW[e] = 0 for an expert without tokens.
 *   dYc  uint8 [N x ld_tok] columnwise codes of the output gradient (mxfp8_quantize
 *        MX_COLWISE with the experts as segments), SFdYc its scales in the SF
 *        layout for [N x ld_tok/32].
 *   Xc   uint8 [K x ld_tok] columnwise codes of the expert-ordered activations,
 *        SFXc its scales in the SF4 layout for [K x ld_tok/32] (MX_COLWISE_X4).
 *   poff device int32 [E+1]; off device int32 [E+1] (T_e = off[e+1] - off[e]).
 *   dW   fp32 [E x N x K].
 * Shapes: N % 128 == 0, K % 128 == 0, ld_tok % 128 == 0 and >= poff[E].
 */
MX_API int grouped_gemm_mxfp8_wgrad(const uint8_t* dYc, const uint8_t* SFdYc, const uint8_t* Xc, const uint8_t* SFXc,
                             const int32_t* off, const int32_t* poff, int E, int64_t N, int64_t K, int64_t ld_tok,
                             float* dW, int* dev_err, mx_stream_t stream);

/* grouped_gemm_mxfp8_wgrad with flags (MX_GEMM_B_SCALES_X1: SFXc in the plain SF layout for
 * [K x ld_tok/32]). */
MX_API int grouped_gemm_mxfp8_wgrad_ex(const uint8_t* dYc, const uint8_t* SFdYc, const uint8_t* Xc,
                                       const uint8_t* SFXc, const int32_t* off, const int32_t* poff, int E, int64_t N,
                                       int64_t K, int64_t ld_tok, float* dW, int flags, int* dev_err,
                                       mx_stream_t stream);

/* Human-readable name of an mx_status value (static string). */
MX_API const char* mx_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* MXMOE_H */
