// Device-side helpers for the libmx kernels (sm_103a): PTX conversions and
// memory access wrappers.  Everything here is written against the public PTX
// ISA; no library math routine is reproduced.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace mx {
namespace dev {

// ---------------------------------------------------------------- memory

// 16-byte streaming load that does not allocate in L1 (inputs are read once).
// 32 bytes, read once: 256-bit load that skips L1.
__device__ __forceinline__ void ld_stream_v8(const void* p, uint32_t (&r)[8]) {
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "l"(p));
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_u16(const uint8_t* p) {
    return *reinterpret_cast<const uint16_t*>(p);
}

// --------------------------------------------------------------- integers

// Per-halfword unsigned max of two packed pairs (PTX max.u16x2, sm_90+).
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ------------------------------------------------------------ conversions

// Exact widening of one f16 (bit pattern in the low 16 bits) to binary32.
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
    float f;
    unsigned short s = static_cast<unsigned short>(h);
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(s));
    return f;
}

// Two binary32 -> two FP8 codes with round-to-nearest-even and saturation to
// the largest finite value; `hi` lands in bits 15..8, `lo` in bits 7..0.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t cvt_e5m2x2(float hi, float lo) {
    unsigned short r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// Two binary32 -> two e2m1 nibbles in one byte: `hi` in bits 7..4, `lo` in 3..0.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float hi, float lo) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Binary32 multiply, round to nearest even, no flush-to-zero, never fused.
__device__ __forceinline__ float mul_rn(float a, float b) { return __fmul_rn(a, b); }

}  // namespace dev
}  // namespace mx
