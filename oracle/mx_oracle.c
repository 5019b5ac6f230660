/*
 * mx_oracle.c -- plain, slow, single-threaded CPU oracle for the MXFP8 MoE hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; it is written from the definitions below, in double
 * precision, without blocking, fusion or reordering.
 *
 * Sources (cited by page title and section):
 *  [P1] aigc.bar, "Blackwell性能陷阱？Cursor揭秘：重写内核让AI大模型MoE提速3.5倍的底层逻辑",
 *       section "1. Blackwell的TMEM架构瓶颈" (microscaling: one scale per data block) and
 *       section "“秘密武器”：自研量化内核与最佳精度配方" (FP8 E4M3 elements, block size 32).
 *  [P4] lpnh.cn blog on the same kernels, section "1. 为什么 MoE 内核在 Blackwell 上反而变慢了"
 *       (blocks of 32 elements, divide by the block scale, then convert to FP8).
 *  [P3] kucoin.com, "Cursor's MoK демонстрирует повышение производительности на 2,37x на NVIDIA
 *       GB300 NVL72", section "01" (count tokens per expert, decide placement, keep one expert's
 *       tokens contiguous).
 *  The pages do not print the scale rule, the E4M3 rounding or the scale-byte
 *  format.  Where they are silent this file takes the OCP Microscaling (MX) v1.0
 *  reading: shared exponent = floor(log2(amax)) - emax_elem with emax_elem = 8
 *  for E4M3, scale stored as an E8M0 byte (bias 127), elements converted with
 *  round-to-nearest-even and saturation to +-448.
 *
 * Parity pins (tests/test_oracle_*.py): exhaustive agreement of the definitional
 * E4M3 encoder with a brute-force nearest-code search, decode/encode round trips,
 * closed-form blocks, hand-computed fixtures under tests/golden/, the
 * transposition identity colwise(X) == rowwise(X^T), a brute-force stable sort
 * for the permutation, and exact rational arithmetic for small GEMMs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------
 * Element formats
 * ------------------------------------------------------------------------- */

/* A bf16 value is the upper 16 bits of an IEEE binary32 value. */
double orc_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 holds subnormals m * 2^-9.  S.1111.111 is NaN; there is no
 * infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* E8M0 scale byte: 2^(b - 127); 0xFF encodes NaN. */
double orc_e8m0_decode(uint8_t b)
{
    if (b == 0xFF)
        return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* E4M3 encode, written from the definition: round to nearest with ties to the
 * even mantissa, subnormal spacing 2^-9, magnitudes that round above 448
 * saturate to 448 ("satfinite").  The sign of the input is kept, also when the
 * magnitude rounds to zero.  NaN encodes 0x7F. */
uint8_t orc_e4m3_encode(double v)
{
    uint8_t sign;
    double a;
    int ex, e, mi;

    if (isnan(v))
        return 0x7F;
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs(v);
    if (isinf(a))
        return sign | 0x7E;
    if (a == 0.0)
        return sign;
    frexp(a, &ex);          /* a = f * 2^ex with f in [0.5, 1) */
    e = ex - 1;             /* so floor(log2 a) = e */
    if (e < -6) {
        /* subnormal range: a multiple of 2^-9, nearbyint rounds ties to even */
        double m = nearbyint(ldexp(a, 9));
        if (m >= 8.0)
            return sign | 0x08;     /* rounded up to the smallest normal, 2^-6 */
        return sign | (uint8_t)m;
    }
    /* normal range: a / 2^e in [1, 2); the mantissa has 3 fraction bits */
    mi = (int)nearbyint(ldexp(a, 3 - e));   /* in [8, 16] */
    if (mi == 16) {
        mi = 8;
        e += 1;
    }
    if (e > 8 || (e == 8 && mi - 8 > 6))
        return sign | 0x7E;                  /* saturate to 448 */
    return sign | (uint8_t)(((e + 7) << 3) | (mi - 8));
}

/* E4M3 encode by brute force: among the finite codes that carry the input's
 * sign, take the one whose value is nearest; on a tie take the code whose
 * mantissa LSB is 0.  Saturation falls out because 448 is the largest finite
 * code.  Independent of orc_e4m3_encode; the tests require both to agree. */
uint8_t orc_e4m3_encode_brute(double v)
{
    int c, base, best = -1;
    double bestd = 0.0;
    if (isnan(v))
        return 0x7F;
    base = signbit(v) ? 0x80 : 0x00;
    for (c = base; c < base + 0x80; c++) {
        double d;
        if ((c & 0x7F) == 0x7F)
            continue;               /* NaN code */
        d = fabs(orc_e4m3_decode((uint8_t)c) - v);
        if (best < 0 || d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)best;
}

/* Exhaustive cross-check helper: every finite bf16 value times 2^shift for
 * shift in [shift_lo, shift_hi] is encoded by both encoders; returns the number
 * of disagreements and the first offending (bits, shift) pair. */
int64_t orc_check_encoders(int shift_lo, int shift_hi, int32_t* first_bits, int32_t* first_shift)
{
    int64_t bad = 0;
    int s;
    uint32_t h;
    *first_bits = -1;
    *first_shift = 0;
    for (s = shift_lo; s <= shift_hi; s++) {
        for (h = 0; h < 0x10000u; h++) {
            double x = orc_bf16_to_double((uint16_t)h);
            double v;
            if (isnan(x) || isinf(x))
                continue;
            v = ldexp(x, s);
            if (orc_e4m3_encode(v) != orc_e4m3_encode_brute(v)) {
                if (bad == 0) {
                    *first_bits = (int32_t)h;
                    *first_shift = s;
                }
                bad++;
            }
        }
    }
    return bad;
}

void orc_e4m3_encode_array(const double* v, int64_t n, uint8_t* out)
{
    int64_t i;
    for (i = 0; i < n; i++)
        out[i] = orc_e4m3_encode(v[i]);
}

void orc_e4m3_decode_array(const uint8_t* c, int64_t n, double* out)
{
    int64_t i;
    for (i = 0; i < n; i++)
        out[i] = orc_e4m3_decode(c[i]);
}

/* ---------------------------------------------------------------------------
 * One MX block ([P1] TMEM section, [P4] section 1): amax over the block,
 * shared exponent s = floor(log2 amax) - 8 clamped to the E8M0 range,
 * elements E4M3(x_i / 2^s).  A block whose amax is 0 takes the smallest scale,
 * s = -127 (byte 0x00).  A block holding NaN or infinity gets the NaN scale
 * 0xFF and NaN elements (out of the workloads' contract; kept for definiteness).
 * x holds n <= 32 values; a short block counts the missing ones as zeros.
 * ------------------------------------------------------------------------- */
uint8_t orc_mx_block(const double* x, int n, uint8_t* q)
{
    double amax = 0.0;
    int i, ex, s;
    for (i = 0; i < n; i++) {
        if (isnan(x[i]) || isinf(x[i])) {
            for (i = 0; i < n; i++)
                q[i] = 0x7F;
            return 0xFF;
        }
        if (fabs(x[i]) > amax)
            amax = fabs(x[i]);
    }
    if (amax == 0.0) {
        s = -127;
    } else {
        frexp(amax, &ex);   /* floor(log2 amax) = ex - 1, exact */
        s = (ex - 1) - 8;
        if (s < -127)
            s = -127;
        if (s > 127)
            s = 127;
    }
    for (i = 0; i < n; i++)
        q[i] = orc_e4m3_encode(ldexp(x[i], -s));   /* x / 2^s is exact in double */
    return (uint8_t)(s + 127);
}

/* Rowwise quantization: blocks are 32 consecutive elements of a row.
 * x: bf16 [rows][cols], cols % 32 == 0.  q: [rows][cols].  sf: row-major
 * [rows][cols/32] scale bytes. */
void orc_quantize_rowwise(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf)
{
    int64_t r, b, kb = cols / 32;
    double blk[32];
    int i;
    for (r = 0; r < rows; r++) {
        for (b = 0; b < kb; b++) {
            for (i = 0; i < 32; i++)
                blk[i] = orc_bf16_to_double(x[r * cols + b * 32 + i]);
            sf[r * kb + b] = orc_mx_block(blk, 32, &q[r * cols + b * 32]);
        }
    }
}

/* Columnwise quantization over expert segments (the transposed operand the
 * backward pass contracts over tokens).  Rows [off[g], off[g+1]) of x form
 * segment g; in the output the segment starts at padded position poff[g] and
 * spans ceil128(off[g+1]-off[g]) positions.  Blocks are 32 consecutive
 * positions of one column inside one segment; positions past the segment's
 * rows hold zeros.  q: [cols][ld], element (c, p) at q[c*ld + p].
 * sf: row-major [cols][ld/32].  Positions at or past poff[nseg] are not written. */
void orc_quantize_colwise_seg(const uint16_t* x, int64_t rows, int64_t cols,
                              const int32_t* off, const int32_t* poff, int nseg, int64_t ld,
                              uint8_t* q, uint8_t* sf)
{
    int g, i;
    int64_t c, p0;
    double blk[32];
    uint8_t qb[32];
    (void)rows;
    for (g = 0; g < nseg; g++) {
        int64_t te = off[g + 1] - off[g];
        int64_t padded = (te + 127) / 128 * 128;
        for (c = 0; c < cols; c++) {
            for (p0 = 0; p0 < padded; p0 += 32) {
                for (i = 0; i < 32; i++) {
                    int64_t l = p0 + i;
                    blk[i] = (l < te) ? orc_bf16_to_double(x[(off[g] + l) * cols + c]) : 0.0;
                }
                sf[c * (ld / 32) + (poff[g] + p0) / 32] = orc_mx_block(blk, 32, qb);
                for (i = 0; i < 32; i++)
                    q[c * ld + poff[g] + p0 + i] = qb[i];
            }
        }
    }
}

/* Rowwise scale rows placed at padded positions: the scale row of data row
 * off[g] + l goes to row poff[g] + l; rows poff[g] + l for l in
 * [T_g, ceil128(T_g)) are padding and hold 0.  sf_dense: [rows][kb] as made by
 * orc_quantize_rowwise.  sf_pad: [poff[nseg]][kb]. */
void orc_place_sf_rows(const uint8_t* sf_dense, int64_t kb, const int32_t* off, const int32_t* poff,
                       int nseg, uint8_t* sf_pad)
{
    int g;
    int64_t l, b;
    for (g = 0; g < nseg; g++) {
        int64_t te = off[g + 1] - off[g];
        int64_t padded = (te + 127) / 128 * 128;
        for (l = 0; l < padded; l++)
            for (b = 0; b < kb; b++)
                sf_pad[(poff[g] + l) * kb + b] = (l < te) ? sf_dense[(off[g] + l) * kb + b] : 0;
    }
}

/* ---------------------------------------------------------------------------
 * Scale-byte layout read by the tensor core's block-scaled MMA.  The pages
 * only say that the quantizer writes scales in the layout the tcgen05 MMA
 * reads, with no reshape pass ([P1] "“秘密武器”" section).  The layout is the
 * one in NVIDIA's public PTX ISA / cuBLAS block-scaling documentation: the
 * [rows x kb] scale matrix, padded to rows % 128 == 0 and kb % 4 == 0, is cut
 * into 128 x 4 atoms of 512 bytes stored atom-row-major; inside an atom,
 * (r, c) sits at (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4).
 * Padding entries are 0.  out has ceil128(rows) * ceil4(kb) bytes.
 * ------------------------------------------------------------------------- */
static int64_t orc_sf_index(int64_t r, int64_t c, int64_t kb4)
{
    int64_t atom = (r / 128) * (kb4 / 4) + c / 4;
    return atom * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

void orc_sf_to_tcgen05(const uint8_t* sf_rm, int64_t rows, int64_t kb, uint8_t* out)
{
    int64_t rows128 = (rows + 127) / 128 * 128;
    int64_t kb4 = (kb + 3) / 4 * 4;
    int64_t r, c;
    for (r = 0; r < rows128; r++)
        for (c = 0; c < kb4; c++)
            out[orc_sf_index(r, c, kb4)] = (r < rows && c < kb) ? sf_rm[r * kb + c] : 0;
}

void orc_sf_from_tcgen05(const uint8_t* sf_sw, int64_t rows, int64_t kb, uint8_t* sf_rm)
{
    int64_t kb4 = (kb + 3) / 4 * 4;
    int64_t r, c;
    for (r = 0; r < rows; r++)
        for (c = 0; c < kb; c++)
            sf_rm[r * kb + c] = sf_sw[orc_sf_index(r, c, kb4)];
}

/* ---------------------------------------------------------------------------
 * Token permutation by expert ([P3] section "01": count the tokens of every
 * expert, decide where each goes, keep one expert's tokens contiguous).
 * ids: [T][k] expert of slot j of token t.  A stable counting sort by expert
 * over the flattened index i = t*k + j, which orders an expert's rows by token,
 * then by slot.  counts[E]; off[E+1] = exclusive scan of counts;
 * poff[E+1] = exclusive scan of ceil128(counts); src_row[off[e]+r] = token;
 * dst_of[i] = destination row, or -1 for an id outside [0, E).
 * Returns the number of ids outside [0, E).
 * ------------------------------------------------------------------------- */
int64_t orc_permute(const int32_t* ids, int64_t T, int k, int E,
                    int32_t* counts, int32_t* off, int32_t* poff, int32_t* src_row, int32_t* dst_of)
{
    int64_t i, n = T * (int64_t)k, bad = 0;
    int e;
    int32_t* fill = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
    for (e = 0; e < E; e++)
        counts[e] = 0;
    for (i = 0; i < n; i++) {
        if (ids[i] >= 0 && ids[i] < E)
            counts[ids[i]]++;
        else
            bad++;
    }
    off[0] = 0;
    poff[0] = 0;
    for (e = 0; e < E; e++) {
        off[e + 1] = off[e] + counts[e];
        poff[e + 1] = poff[e] + (counts[e] + 127) / 128 * 128;
    }
    for (i = 0; i < n; i++) {
        int32_t x = ids[i];
        if (x >= 0 && x < E) {
            int32_t r = off[x] + fill[x]++;
            src_row[r] = (int32_t)(i / k);
            dst_of[i] = r;
        } else {
            dst_of[i] = -1;
        }
    }
    free(fill);
    return bad;
}

/* Row gather: dst row r = src row src_row[r], row_bytes bytes each. */
void orc_gather_rows(const uint8_t* src, int64_t row_bytes, const int32_t* src_row, int64_t R, uint8_t* dst)
{
    int64_t r;
    for (r = 0; r < R; r++)
        memcpy(dst + r * row_bytes, src + (int64_t)src_row[r] * row_bytes, (size_t)row_bytes);
}

/* ---------------------------------------------------------------------------
 * Reference GEMM over dequantized operands, fp64 accumulation:
 *   C[m][n] = sum_k deq(A)[m][k] * deq(B)[n][k]
 * with deq(A)[m][k] = E4M3(qa[m*lda + k]) * 2^(sfa[m*ldsa + k/32] - 127), and
 * likewise for B.  Both operands hold the contraction axis contiguously (the
 * "NT" form that the grouped GEMM's forward, dgrad and wgrad all reduce to);
 * the scale arrays are row-major.  The pages state the computation only as a
 * block-scaled FP8 matrix product done inside the tensor core ([P1] "破局之道").
 * ------------------------------------------------------------------------- */
void orc_gemm_nt(int64_t M, int64_t N, int64_t K,
                 const uint8_t* qa, int64_t lda, const uint8_t* sfa, int64_t ldsa,
                 const uint8_t* qb, int64_t ldb, const uint8_t* sfb, int64_t ldsb,
                 double* c, int64_t ldc)
{
    int64_t m, n, kk;
    double* arow = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    double* bdeq = (double*)malloc(sizeof(double) * (size_t)((N * K) > 0 ? N * K : 1));
    for (n = 0; n < N; n++)
        for (kk = 0; kk < K; kk++)
            bdeq[n * K + kk] = orc_e4m3_decode(qb[n * ldb + kk]) * orc_e8m0_decode(sfb[n * ldsb + kk / 32]);
    for (m = 0; m < M; m++) {
        for (kk = 0; kk < K; kk++)
            arow[kk] = orc_e4m3_decode(qa[m * lda + kk]) * orc_e8m0_decode(sfa[m * ldsa + kk / 32]);
        for (n = 0; n < N; n++) {
            double acc = 0.0;
            for (kk = 0; kk < K; kk++)
                acc += arow[kk] * bdeq[n * K + kk];
            c[m * ldc + n] = acc;
        }
    }
    free(arow);
    free(bdeq);
}

/* Round a double to bf16 (round to nearest, ties to even), via binary32.  Used
 * only to express the final output rounding of the forward and dgrad GEMMs. */
uint16_t orc_double_to_bf16(double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------------------
 * Combine (unpermute) -- the final weighted merge of the expert outputs back to
 * token order (kucoin.com MoK page, section "03": the measured layer ends with
 * "combine" and the final weighted merge).  Y: bf16 [R][H] in expert order;
 * gate: fp32 [T][k]; dst_of: [T][k] destination row of (t, j), -1 = dropped.
 *   out[t][h] = bf16( sum_j gate[t][j] * Y[dst_of[t][j]][h] )      (sum in double)
 * Backward, with dOut bf16 [T][H]:
 *   dY[dst_of[t][j]][h] = bf16( float( gate[t][j] * dOut[t][h] ) )
 *   dgate[t][j]        = sum_h dOut[t][h] * Y[dst_of[t][j]][h]     (double)
 * The bf16 rounding goes through binary32 (round to nearest even twice), which
 * is exact for the single products here because a binary32 times bf16 product has
 * at most 32 significant bits.
 * ------------------------------------------------------------------------- */
static uint16_t orc_float_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

void orc_combine_fwd(const uint16_t* Y, const float* gate, const int32_t* dst_of, int64_t T, int k, int64_t H,
                     uint16_t* out)
{
    int64_t t, h;
    int j;
    for (t = 0; t < T; t++) {
        for (h = 0; h < H; h++) {
            double acc = 0.0;
            for (j = 0; j < k; j++) {
                int32_t d = dst_of[t * k + j];
                if (d >= 0)
                    acc += (double)gate[t * k + j] * orc_bf16_to_double(Y[(int64_t)d * H + h]);
            }
            out[t * H + h] = orc_float_to_bf16((float)acc);
        }
    }
}

void orc_combine_bwd(const uint16_t* dOut, const uint16_t* Y, const float* gate, const int32_t* dst_of, int64_t T,
                     int k, int64_t H, uint16_t* dY, double* dgate)
{
    int64_t t, h;
    int j;
    for (t = 0; t < T; t++) {
        for (j = 0; j < k; j++) {
            int32_t d = dst_of[t * k + j];
            double dot = 0.0;
            if (d < 0) {
                dgate[t * k + j] = 0.0;
                continue;
            }
            for (h = 0; h < H; h++) {
                double g = orc_bf16_to_double(dOut[t * H + h]);
                dY[(int64_t)d * H + h] = orc_float_to_bf16((float)((double)gate[t * k + j] * g));
                dot += g * orc_bf16_to_double(Y[(int64_t)d * H + h]);
            }
            dgate[t * k + j] = dot;
        }
    }
}

/* ---------------------------------------------------------------------------
 * Scale-rule and input-type variants.
 *  rule 0 (default, OCP MX): s = floor(log2 amax) - 8, as in orc_mx_block.
 *  rule 1 ("RCEIL", the ceiling rule of NVIDIA TransformerEngine's MXFP8 recipe, which
 *         the aigc.bar page names in section "破局之道"): the smallest s with
 *         amax <= 448 * 2^s, so no element saturates.
 *  dtype 0 = bf16 input, 1 = fp32 input (the quantizer benchmark pseudo-code of the
 *  lpnh.cn page, section "4. 验证请求与成功结果", reads float input).
 * ------------------------------------------------------------------------- */
uint8_t orc_mx_block_rule(const double* x, int n, uint8_t* q, int rule)
{
    double amax = 0.0;
    int i, ex, s;
    if (rule == 0)
        return orc_mx_block(x, n, q);
    for (i = 0; i < n; i++) {
        if (isnan(x[i]) || isinf(x[i])) {
            for (i = 0; i < n; i++)
                q[i] = 0x7F;
            return 0xFF;
        }
        if (fabs(x[i]) > amax)
            amax = fabs(x[i]);
    }
    if (amax == 0.0) {
        s = -127;
    } else {
        frexp(amax, &ex);
        s = (ex - 1) - 9;                      /* 448 * 2^s < amax here ... */
        while (ldexp(448.0, s) < amax)        /* ... so step up to the smallest s that covers amax */
            s++;
        if (s < -127)
            s = -127;
        if (s > 127)
            s = 127;
    }
    for (i = 0; i < n; i++)
        q[i] = orc_e4m3_encode(ldexp(x[i], -s));
    return (uint8_t)(s + 127);
}

static double orc_load(const void* x, int dtype, int64_t i)
{
    if (dtype == 1)
        return (double)((const float*)x)[i];
    return orc_bf16_to_double(((const uint16_t*)x)[i]);
}

void orc_quantize_rowwise_ex(const void* x, int dtype, int64_t rows, int64_t cols, int rule, uint8_t* q, uint8_t* sf)
{
    int64_t r, b, kb = cols / 32;
    double blk[32];
    int i;
    for (r = 0; r < rows; r++) {
        for (b = 0; b < kb; b++) {
            for (i = 0; i < 32; i++)
                blk[i] = orc_load(x, dtype, r * cols + b * 32 + i);
            sf[r * kb + b] = orc_mx_block_rule(blk, 32, &q[r * cols + b * 32], rule);
        }
    }
}

void orc_quantize_colwise_seg_ex(const void* x, int dtype, int64_t rows, int64_t cols, const int32_t* off,
                                 const int32_t* poff, int nseg, int64_t ld, int rule, uint8_t* q, uint8_t* sf)
{
    int g, i;
    int64_t c, p0;
    double blk[32];
    uint8_t qb[32];
    (void)rows;
    for (g = 0; g < nseg; g++) {
        int64_t te = off[g + 1] - off[g];
        int64_t padded = (te + 127) / 128 * 128;
        for (c = 0; c < cols; c++) {
            for (p0 = 0; p0 < padded; p0 += 32) {
                for (i = 0; i < 32; i++) {
                    int64_t l = p0 + i;
                    blk[i] = (l < te) ? orc_load(x, dtype, (off[g] + l) * cols + c) : 0.0;
                }
                sf[c * (ld / 32) + (poff[g] + p0) / 32] = orc_mx_block_rule(blk, 32, qb, rule);
                for (i = 0; i < 32; i++)
                    q[c * ld + poff[g] + p0 + i] = qb[i];
            }
        }
    }
}

/* ---------------------------------------------------------------------------
 * SwiGLU between the two expert GEMMs, whose output and input gradient the MXFP8
 * data path quantizes directly (kucoin.com MoK page, section "02": quantization
 * folded into the SwiGLU step).  a: bf16 [R][2I], gate = columns [0, I), up =
 * columns [I, 2I).  silu(g) = g / (1 + e^-g).
 *   forward   h[r][i]        = silu(g) * u                                   -> fp32
 *   backward  dgate[r][i]    = dh * u * s * (1 + g (1 - s)),  s = 1/(1+e^-g)  -> fp32
 *             dup[r][i]      = dh * silu(g)                                   -> fp32
 * computed in double and rounded once to fp32, the precision the fused kernels
 * quantize from.  dH is stored [R][2I] as [dgate | dup].
 * ------------------------------------------------------------------------- */
void orc_swiglu_fwd(const uint16_t* a, int64_t R, int64_t I, float* h)
{
    int64_t r, i;
    for (r = 0; r < R; r++)
        for (i = 0; i < I; i++) {
            double g = orc_bf16_to_double(a[r * 2 * I + i]);
            double u = orc_bf16_to_double(a[r * 2 * I + I + i]);
            h[r * I + i] = (float)(g / (1.0 + exp(-g)) * u);
        }
}

void orc_swiglu_bwd(const uint16_t* dh, const uint16_t* a, int64_t R, int64_t I, float* dH)
{
    int64_t r, i;
    for (r = 0; r < R; r++)
        for (i = 0; i < I; i++) {
            double g = orc_bf16_to_double(a[r * 2 * I + i]);
            double u = orc_bf16_to_double(a[r * 2 * I + I + i]);
            double d = orc_bf16_to_double(dh[r * I + i]);
            double s = 1.0 / (1.0 + exp(-g));
            dH[r * 2 * I + i] = (float)(d * u * s * (1.0 + g * (1.0 - s)));
            dH[r * 2 * I + I + i] = (float)(d * g * s);
        }
}
