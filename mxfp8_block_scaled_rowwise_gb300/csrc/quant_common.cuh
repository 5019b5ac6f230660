// quant_common.cuh -- device helpers shared by the MXFP8 quantizing kernels (the
// quantizer and the fused SwiGLU kernels): streaming loads, the scale-byte rules, the
// exact power-of-two rescale and the E4M3 conversion of value pairs.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace mx {

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 32 bytes of global memory in one 256-bit load (p 32-byte aligned), not kept in L1.
__device__ __forceinline__ void ld_stream_32(const void* p, uint32_t* w) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

// 32 bytes to global memory in one 256-bit store (p 32-byte aligned).
__device__ __forceinline__ void st_global_32(void* p, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Segment of padded position p0: the last g in [0, nseg) with poff[g] <= p0 (poff
// nondecreasing from poff[0] = 0).  The whole warp searches at once: each lane tests one
// offset per round of 32 and a ballot counts the offsets <= p0, so the lookup costs one round
// of independent loads instead of log2(nseg) dependent ones.  All 32 lanes must call it.
__device__ __forceinline__ int find_segment(const int32_t* poff, int nseg, int64_t p0) {
    const int lane = threadIdx.x & 31;
    int count = 0;
    for (int base = 0; base < nseg; base += 32) {
        const int i = base + lane;
        const bool le = i < nseg && __ldg(poff + i) <= p0;
        count += __popc(__ballot_sync(0xffffffffu, le));
    }
    return count > 0 ? count - 1 : 0;
}

// Two fp32 products in one packed instruction.
__device__ __forceinline__ void mul_f32x2(float& a, float& b, float s) {
    uint64_t x = static_cast<uint64_t>(__float_as_uint(a)) | (static_cast<uint64_t>(__float_as_uint(b)) << 32);
    const uint64_t y = static_cast<uint64_t>(__float_as_uint(s)) | (static_cast<uint64_t>(__float_as_uint(s)) << 32);
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(x) : "l"(y));
    a = __uint_as_float(static_cast<uint32_t>(x));
    b = __uint_as_float(static_cast<uint32_t>(x >> 32));
}

// max(|a|, |b|) of each bf16 half in one packed instruction, NaN-propagating.  Only the
// magnitude bits of the result are meaningful (the sign bit is the xor of the inputs'); a
// NaN half comes back as a NaN pattern, so its exponent field reads 0xFF.
__device__ __forceinline__ uint32_t amax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Scale byte of a block from the magnitude bits of its largest |bf16| value (a block holding
// NaN or Inf has exponent field 0xFF there and gets the NaN scale).
__device__ __forceinline__ uint32_t scale_byte(uint32_t amax_bits) {
    const uint32_t e = amax_bits >> 7;
    if (e == 0xFFu) return 0xFFu;
    return e > 8u ? e - 8u : 0u;
}

// The ceiling rule: the smallest power of two X with amax <= 448 X.  With amax = m 2^e,
// m in [1, 2): X = 2^(e - 8) when m <= 1.75, else 2^(e - 7).  frac_bits / frac_over
// give the width of the mantissa field and the pattern of 0.75 in it.
__device__ __forceinline__ uint32_t scale_byte_ceil(uint32_t amax_bits, int frac_bits, uint32_t frac_075) {
    const uint32_t e = amax_bits >> frac_bits;
    if (e == 0xFFu) return 0xFFu;
    const uint32_t up = (amax_bits & ((1u << frac_bits) - 1u)) > frac_075 ? 1u : 0u;
    return e + up > 8u ? e + up - 8u : 0u;
}

template <int RULE>
__device__ __forceinline__ uint32_t scale_byte_bf16(uint32_t amax_bits) {
    return RULE == 0 ? scale_byte(amax_bits) : scale_byte_ceil(amax_bits, 7, 0x60u);
}

template <int RULE>
__device__ __forceinline__ uint32_t scale_byte_f32(uint32_t amax_bits) {
    if (RULE == 0) {
        const uint32_t e = amax_bits >> 23;
        if (e == 0xFFu) return 0xFFu;
        return e > 8u ? e - 8u : 0u;
    }
    return scale_byte_ceil(amax_bits, 23, 0x600000u);
}

// 2^(127 - b) as an fp32 (b <= 246 for finite blocks, so the exponent field 254 - b >= 8).
__device__ __forceinline__ float inv_scale(uint32_t b) {
    return __uint_as_float((254u - b) << 23);
}

// The same, or a quiet NaN for the NaN scale byte 0xFF: every product with it is NaN, which
// converts to the E4M3 NaN code 0x7F, so a block holding NaN or Inf needs no separate path.
__device__ __forceinline__ float inv_scale_or_nan(uint32_t b) {
    return b == 0xFFu ? __uint_as_float(0x7FFFFFFFu) : inv_scale(b);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// E4M3 codes of the two bf16 values of a word, scaled by s (low value in the low byte).
__device__ __forceinline__ uint32_t quant_pair(uint32_t w, float s) {
    float lo = bf16_lo(w), hi = bf16_hi(w);
    mul_f32x2(lo, hi, s);
    return cvt_e4m3x2(lo, hi);
}

// E4M3 codes of two values taken from the low (or high) halves of two words.
__device__ __forceinline__ uint32_t quant_pair2(float a, float b, float s) {
    mul_f32x2(a, b, s);
    return cvt_e4m3x2(a, b);
}

// Four E4M3 codes (one register) of the four bf16 values of two words, scaled by s.
__device__ __forceinline__ uint32_t quant_quad(uint32_t w0, uint32_t w1, float s) {
    float a = bf16_lo(w0), b = bf16_hi(w0), c = bf16_lo(w1), d = bf16_hi(w1);
    mul_f32x2(a, b, s);
    mul_f32x2(c, d, s);
    return cvt_e4m3x4(a, b, c, d);
}

// Four E4M3 codes (one register) of four fp32 values scaled by s.
__device__ __forceinline__ uint32_t quant_quad_f32(float a, float b, float c, float d, float s) {
    mul_f32x2(a, b, s);
    mul_f32x2(c, d, s);
    return cvt_e4m3x4(a, b, c, d);
}


// ---- SwiGLU arithmetic shared by the fused SwiGLU kernels and the GEMM epilogue
constexpr float kLog2e = 1.4426950408889634f;

// sigmoid(g) from e = e^-|g| in (0, 1] (e^x = 2^(x log2 e) on the special-function unit,
// subnormal results kept) and r = 1 / (1 + e) in [1/2, 1): sigmoid(g) = r for g >= 0 and
// e r for g < 0.  Neither step can overflow, whatever the sign of g; NaN propagates.
__device__ __forceinline__ float sigmoid_f32(float g) {
    float e, r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(e) : "f"(-fabsf(g) * kLog2e));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return g >= 0.0f ? r : e * r;
}

// Packed fp32 pairs (low value in the low half) and their f32x2 arithmetic on the FMA pipe;
// every operation rounds to nearest like its scalar form.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float lo2(uint64_t v) {
    float lo;
    asm("mov.b64 {%0, _}, %1;" : "=f"(lo) : "l"(v));
    return lo;
}
__device__ __forceinline__ float hi2(uint64_t v) {
    float hi;
    asm("mov.b64 {_, %0}, %1;" : "=f"(hi) : "l"(v));
    return hi;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// 2^x on the special-function unit; FTZ: subnormal results flush to zero (one instruction),
// otherwise they are kept (extra instructions around it).
template <bool FTZ>
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    if (FTZ) asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    else asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float rcp_approx_ftz(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Sigmoid of the pair (g0, g1) in the arithmetic of sigmoid_f32: e = e^-|g|, r = 1 / (1 + e),
// sigmoid = r (g >= 0) or e r (g < 0).  With FTZ the e^-|g| step flushes subnormal results,
// which changes nothing while |g| < 87 (e normal there, and for g >= 0, 1 + e == 1 below it).
template <bool FTZ>
__device__ __forceinline__ uint64_t sigmoid2(float g0, float g1) {
    const float e0 = ex2_approx<FTZ>(-fabsf(g0) * kLog2e), e1 = ex2_approx<FTZ>(-fabsf(g1) * kLog2e);
    const uint64_t E = pk2(e0, e1);
    const uint64_t T = add2(pk2(1.0f, 1.0f), E);
    const float r0 = rcp_approx_ftz(lo2(T)), r1 = rcp_approx_ftz(hi2(T));
    const uint64_t ER = mul2(E, pk2(r0, r1));
    return pk2(g0 >= 0.0f ? r0 : lo2(ER), g1 >= 0.0f ? r1 : hi2(ER));
}

// max(|x|, m) with NaN propagating, so a NaN block gets the NaN scale.
__device__ __forceinline__ float amax_step(float m, float x) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(x)));
    return r;
}

}  // namespace mx
