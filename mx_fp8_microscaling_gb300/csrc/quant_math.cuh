// QuantizeMX element arithmetic shared by the standalone quantizer and the
// fused activation quantize inside the GEMM, so that both produce the same
// bits.  The steps are those of the page "MX Microscaling: Quantize,
// Block-Scaling and E8M0": the binary32 exponent byte of each element, the
// block maximum (sign dropped), E8M0 = max(1, max(0, maxExp - EMAX)), one
// binary32 multiply by 2^(127 - E8M0), and a round-to-nearest-even saturating
// narrow (NaN -> 0x7F|sign for FP8, a signed zero nibble for e2m1; Inf -> the
// format maximum).
#pragma once

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace qdev {

using namespace dev;

template <bool F16>
__device__ __forceinline__ float widen_lo(uint32_t w) {
    if constexpr (F16) return f16_bits_to_f32(w & 0xFFFFu);
    else return __uint_as_float(w << 16);
}
template <bool F16>
__device__ __forceinline__ float widen_hi(uint32_t w) {
    if constexpr (F16) return f16_bits_to_f32(w >> 16);
    else return __uint_as_float(w & 0xFFFF0000u);
}
template <bool F16>
__device__ __forceinline__ float widen1(uint32_t h) {
    if constexpr (F16) return f16_bits_to_f32(h);
    else return __uint_as_float(h << 16);
}

// Binary32 exponent byte of the widened value whose 16-bit magnitude is m16.
template <bool F16>
__device__ __forceinline__ uint32_t exp_byte_of_mag(uint32_t m16) {
    if constexpr (F16) return __float_as_uint(f16_bits_to_f32(m16)) >> 23;
    else return m16 >> 7;
}

// E8M0 from the block's max exponent byte: floor at 0, then at 1.
__device__ __forceinline__ uint32_t e8m0_of(uint32_t max_exp, int bias) {
    int v = static_cast<int>(max_exp) - bias;
    return static_cast<uint32_t>(v < 1 ? 1 : v);
}

// 2^(127 - E): the binary32 with exponent field 254 - E and zero fraction.
__device__ __forceinline__ float prescale_mul(uint32_t e8m0) {
    return __uint_as_float((254u - e8m0) << 23);
}

__device__ __forceinline__ uint32_t mag2(uint32_t w) { return w & 0x7FFF7FFFu; }
__device__ __forceinline__ uint32_t hmax(uint32_t m) {
    uint32_t lo = m & 0xFFFFu, hi = m >> 16;
    return lo > hi ? lo : hi;
}


template <int FMT>
__device__ __forceinline__ uint32_t cvt_pair(float hi, float lo) {
    if constexpr (FMT == kE4M3) return cvt_e4m3x2(hi, lo);
    else if constexpr (FMT == kE5M2) return cvt_e5m2x2(hi, lo);
    else return cvt_e2m1x2(hi, lo);
}

// One element, special values handled explicitly (used where a block holds
// Inf/NaN, and by the generic kernel).
template <int FMT>
__device__ __forceinline__ uint32_t encode1(float y) {
    const uint32_t sign = __float_as_uint(y) >> 31;
    if constexpr (FMT == kE2M1) {
        if (isnan(y)) return sign << 3;
        if (isinf(y)) return (sign << 3) | 7u;
        return cvt_e2m1x2(0.0f, y) & 0xFu;
    } else {
        constexpr uint32_t kMax = (FMT == kE4M3) ? 0x7Eu : 0x7Bu;
        if (isnan(y)) return (sign << 7) | 0x7Fu;
        if (isinf(y)) return (sign << 7) | kMax;
        return cvt_pair<FMT>(0.0f, y) & 0xFFu;
    }
}

// 8 prescaled values of one row -> packed output.
// FP8: two 32-bit words, byte j = element j.
// e2m1: one 32-bit word; pair p = elements (2p, 2p+1) forms one byte (the
// even element in the high nibble for parity 0), and the four pair-bytes are
// placed by the lane-remap permutation `perm`.
template <int FMT>
__device__ __forceinline__ void pack8(const float (&y)[8], bool special, int parity, uint32_t perm,
                                      uint32_t& w0, uint32_t& w1) {
    if constexpr (FMT == kE2M1) {
        uint32_t b[4];
        if (!special) {
#pragma unroll
            for (int p = 0; p < 4; ++p)
                b[p] = parity ? cvt_pair<FMT>(y[2 * p + 1], y[2 * p]) : cvt_pair<FMT>(y[2 * p], y[2 * p + 1]);
        } else {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t n0 = encode1<FMT>(y[2 * p]), n1 = encode1<FMT>(y[2 * p + 1]);
                b[p] = parity ? ((n1 << 4) | n0) : ((n0 << 4) | n1);
            }
        }
        uint32_t src = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
        w0 = __byte_perm(src, 0u, perm);
        w1 = 0;
    } else {
        if (!special) {
            w0 = cvt_pair<FMT>(y[1], y[0]) | (cvt_pair<FMT>(y[3], y[2]) << 16);
            w1 = cvt_pair<FMT>(y[5], y[4]) | (cvt_pair<FMT>(y[7], y[6]) << 16);
        } else {
            uint32_t c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = encode1<FMT>(y[j]);
            w0 = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
            w1 = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
        }
    }
}

// Widening for the elements of a block that holds Inf/NaN: as widen1, but a
// NaN keeps its sign (cvt.f32.f16 returns a canonical NaN whatever the
// input's sign; the narrow only needs NaN-ness and the sign).
template <bool F16>
__device__ __forceinline__ float widen_keep_nan(uint32_t h) {
    if constexpr (F16) {
        if ((h & 0x7FFFu) > 0x7C00u) return __uint_as_float(((h & 0x8000u) << 16) | 0x7FC00000u);
        return f16_bits_to_f32(h);
    } else {
        return __uint_as_float(h << 16);
    }
}

// y = x * 2^(127 - E8M0) for an element of a block that holds Inf/NaN: a
// NaN element is passed on unchanged, so the narrow sees its sign (the GPU's
// binary32 multiply returns a canonical NaN whatever the operand's sign).
__device__ __forceinline__ float prescale_keep_nan(float x, float s) { return isnan(x) ? x : mul_rn(x, s); }

// Prescale and pack 8 elements of one row: input words w[j] hold elements
// 2j (low half) and 2j+1 (high half); elements 0-3 take scale s0, 4-7 s1.
// `special` (the element's block holds Inf/NaN) selects the per-element
// path; the common path multiplies and converts two elements at a time.
template <bool F16, int FMT>
__device__ __forceinline__ void quantize8(const uint32_t (&w)[4], float s0, float s1, bool special, int parity,
                                          uint32_t perm, uint32_t& o0, uint32_t& o1) {
    float y[8];
    if (!special) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float sc = j < 2 ? s0 : s1;
            y[2 * j] = mul_rn(widen_lo<F16>(w[j]), sc);
            y[2 * j + 1] = mul_rn(widen_hi<F16>(w[j]), sc);
        }
        pack8<FMT>(y, false, parity, perm, o0, o1);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float sc = j < 2 ? s0 : s1;
            y[2 * j] = prescale_keep_nan(widen_keep_nan<F16>(w[j] & 0xFFFFu), sc);
            y[2 * j + 1] = prescale_keep_nan(widen_keep_nan<F16>(w[j] >> 16), sc);
        }
        pack8<FMT>(y, true, parity, perm, o0, o1);
    }
}

}  // namespace qdev
}  // namespace mx
