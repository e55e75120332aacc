// MX dequantize: element value = decode(code) * 2^(E8M0 - 127).
//
// The page "MX Microscaling: Quantize, Block-Scaling and E8M0" states that
// the matmul side reads the scale back as ldexpf(x, E8M0 - 127), the exact
// inverse of the quantizer's prescale ("quantizeDataApplyingMxScales"), and
// that e2m1 nibbles are read back through the same lane permutation that
// packed them ("FP4 x4-Pack and Intra-x4 Lane Order").
//
// FP8 and e2m1 codes convert exactly to f16 (cvt.rn.f16x2.{e4m3,e5m2,e2m1}x2),
// then to f32, and one binary32 multiply by 2^(E - 127) scales them; every
// product is exact in f32 (smallest 2^-9 * 2^-127 for e4m3fn, 2^-16 * 2^-127
// for e5m2, both above the f32 subnormal quantum), except overflow to Inf.
// E = 0xFF (the E8M0 NaN) gives NaN.  bf16 output rounds that exact value to
// nearest even.
//
// HBM-bound: 1 byte (FP8) or 0.5 byte (e2m1) + 1/32 byte of scale read, 4 or 2
// bytes written per element, and at 3 bytes an element (FP8 -> bf16) the
// instruction count per element decides as much as the bytes: a thread
// converts 16 consecutive elements of a row with one 16-byte (FP8) or 8-byte
// (e2m1) load and one 32-byte (bf16) or two (f32) 32-byte stores, and every
// pair of elements is scaled by one packed multiply.  Consecutive threads take
// consecutive chunks of a row.

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "pdl.cuh"

namespace mx {
namespace {

constexpr int kThreads = 256;
constexpr int kMinBlocksBf16 = 8;  // 32 registers a thread: 8 blocks resident per SM
constexpr int kMinBlocksF32 = 6;   // the f32 path needs up to 40 registers
constexpr int kGridPerSm = 32;   // blocks launched per SM (rows permitting)
constexpr int kChunk = 16;       // elements a thread converts per step

// Two codes (bits 15..8 and 7..0 of `pair`) -> f16x2 with the high byte in
// the upper half; e2m1: one byte, high nibble in the upper half.
template <int FMT>
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t pair) {
    uint32_t r;
    if constexpr (FMT == kE4M3) {
        unsigned short v = static_cast<unsigned short>(pair);
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    } else if constexpr (FMT == kE5M2) {
        unsigned short v = static_cast<unsigned short>(pair);
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(r) : "h"(v));
    } else {
        asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(pair));
    }
    return r;
}

// Two E8M0 scales (bits 15..8 and 7..0) -> bf16x2 2^(E - 127), high byte in
// the upper half.  E = 0 is the bf16 subnormal 2^-127, E = 255 is NaN.
__device__ __forceinline__ uint32_t e8m0x2_to_bf16x2(uint32_t pair) {
    uint32_t r;
    unsigned short v = static_cast<unsigned short>(pair);
    asm("cvt.rn.bf16x2.ue8m0x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

// f16x2 -> bf16x2.  Exact for decoded FP8 / FP4 codes: at most 4 significant
// bits, and bf16's exponent range covers f16's.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h2) {
    unsigned short lo = static_cast<unsigned short>(h2), hi = static_cast<unsigned short>(h2 >> 16), a, b;
    asm("cvt.rn.bf16.f16 %0, %1;" : "=h"(a) : "h"(lo));
    asm("cvt.rn.bf16.f16 %0, %1;" : "=h"(b) : "h"(hi));
    return static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
}

// x * s for both halves, one rounding to nearest even: the product of a code
// (<= 4 significant bits) and a power of two is exact unless it falls below
// the normal range, where one RNE step matches rounding the exact value.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t x, uint32_t s) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(s));
    return r;
}

__device__ __forceinline__ int64_t scale_slot(int64_t i, int mode) {
    return mode == 1 ? (i & 3) + 32 * (i >> 2) : i;
}

// Scale pairs (bf16x2) for the 8 element pairs of the chunk [c0, c0 + n) of
// one row.  BC is the block's extent along columns (4, 8, 32 or 1): the chunk
// spans 4, 2, 1 or 16 blocks.
template <int BC>
__device__ __forceinline__ void chunk_scales(const DequantArgs& q, const uint8_t* srow_ptr, int64_t srow,
                                             int64_t c0, int n, uint32_t (&sp)[8]) {
    if constexpr (BC == 1) {
        // one scale per element: the pair's two scale bytes are adjacent
        const uint8_t* src = srow_ptr + c0;
        uint32_t b[4];
        if (n == kChunk && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
            const uint4 v = *reinterpret_cast<const uint4*>(src);
            b[0] = v.x, b[1] = v.y, b[2] = v.z, b[3] = v.w;
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                b[k] = 0;
                for (int j = 0; j < 4; ++j)
                    if (4 * k + j < n) b[k] |= static_cast<uint32_t>(src[4 * k + j]) << (8 * j);
            }
        }
#pragma unroll
        for (int p = 0; p < 8; ++p) sp[p] = e8m0x2_to_bf16x2(b[p >> 1] >> (16 * (p & 1)));
    } else if constexpr (BC == 4 || BC == 8) {
        constexpr int kBlocks = kChunk / BC;  // 4 or 2 scales
        const uint8_t* src = srow_ptr + c0 / BC;
        const int live = (n + BC - 1) / BC;
        uint32_t e[kBlocks];
        if (live == kBlocks && (reinterpret_cast<uintptr_t>(src) & (kBlocks - 1)) == 0) {
            const uint32_t v = kBlocks == 4 ? *reinterpret_cast<const uint32_t*>(src)
                                            : static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(src));
#pragma unroll
            for (int k = 0; k < kBlocks; ++k) e[k] = (v >> (8 * k)) & 0xFFu;
        } else {
#pragma unroll
            for (int k = 0; k < kBlocks; ++k) e[k] = k < live ? src[k] : 0u;
        }
        uint32_t s[kBlocks];
#pragma unroll
        for (int k = 0; k < kBlocks; ++k) s[k] = e8m0x2_to_bf16x2(e[k] * 0x101u);
#pragma unroll
        for (int p = 0; p < 8; ++p) sp[p] = s[(2 * p) / BC];
    } else {
        const int64_t scol = c0 / BC;
        uint32_t v;
        if (q.scale_mode == 2) {
            const int64_t tile = (srow >> 7) * q.sf_ntk + (scol >> 2);
            v = q.scale[tile * 512 + (srow & 31) * 16 + ((srow >> 5) & 3) * 4 + (scol & 3)];
        } else {
            v = srow_ptr[scol];
        }
        const uint32_t s = e8m0x2_to_bf16x2(v * 0x101u);
#pragma unroll
        for (int p = 0; p < 8; ++p) sp[p] = s;
    }
}

// Raw codes of the chunk [c0, c0 + n), n in {4, 8, 12, 16}: FP8 16 bytes in
// w[0..3], e2m1 8 bytes in w[0..1].  Codes past n are 0.
template <int FMT>
__device__ __forceinline__ void load_chunk(const DequantArgs& q, int64_t r, int64_t c0, int n, uint32_t (&w)[4]) {
    if constexpr (FMT == kE2M1) {
        // linear nibble index r*cols + c0 is a multiple of 4: 2-byte aligned
        const uint8_t* src = q.data + (r * q.cols + c0) / 2;
        w[2] = w[3] = 0;
        if (n == kChunk && (reinterpret_cast<uintptr_t>(src) & 7u) == 0) {
            const uint2 v = *reinterpret_cast<const uint2*>(src);
            w[0] = v.x, w[1] = v.y;
        } else {
            const uint16_t* h = reinterpret_cast<const uint16_t*>(src);
            uint32_t t[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) t[k] = 4 * k < n ? h[k] : 0u;
            w[0] = t[0] | (t[1] << 16), w[1] = t[2] | (t[3] << 16);
        }
    } else {
        const uint8_t* src = q.data + r * q.cols + c0;  // 4-byte aligned
        if (n == kChunk && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
            const uint4 v = *reinterpret_cast<const uint4*>(src);
            w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
        } else {
            const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src);
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = 4 * k < n ? s32[k] : 0u;
        }
    }
}

// Decode the chunk's 8 element pairs to f16x2, element 2p in the low half.
template <int FMT>
__device__ __forceinline__ void decode_chunk(const DequantArgs& q, const uint32_t (&w)[4], uint32_t (&h)[8]) {
    if constexpr (FMT == kE2M1) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            // undo the lane permutation of each 8-element group: byte p holds
            // elements (2p, 2p+1)
            const uint32_t src32 = __byte_perm(w[g], 0u, q.fp4_inv_perm);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                // cvt puts the high nibble in the upper half; with parity 0
                // the high nibble is the even element
                const uint32_t h2 = codes_to_f16x2<FMT>((src32 >> (8 * p)) & 0xFFu);
                h[4 * g + p] = q.fp4_parity ? h2 : __byte_perm(h2, 0u, 0x1032);
            }
        }
    } else {
#pragma unroll
        for (int p = 0; p < 8; ++p) h[p] = codes_to_f16x2<FMT>((w[p >> 1] >> (16 * (p & 1))) & 0xFFFFu);
    }
}

__device__ __forceinline__ void store_v8(void* dst, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Scale and store one chunk of n elements.
template <bool BF16>
__device__ __forceinline__ void store_chunk(const DequantArgs& q, const uint32_t (&h)[8], const uint32_t (&sp)[8],
                                            int64_t r, int64_t c0, int n) {
    if constexpr (BF16) {
        uint32_t o[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) o[p] = mul_bf16x2(f16x2_to_bf16x2(h[p]), sp[p]);
        uint16_t* dst = reinterpret_cast<uint16_t*>(q.out) + r * q.ld_out + c0;
        if (n == kChunk && (reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
            store_v8(dst, o);
        } else if (n == kChunk && q.vec_ok) {
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
        } else {
            for (int j = 0; j < n; ++j) dst[j] = static_cast<uint16_t>(o[j >> 1] >> (16 * (j & 1)));
        }
    } else {
        // f32: the product of an exact f32 code and 2^(E - 127) (bf16 scale bits
        // widened to f32) is exact unless it overflows.  Two halves of 8
        // elements keep the live registers down.
        float* dst = reinterpret_cast<float*>(q.out) + r * q.ld_out + c0;
        const bool v8 = n == kChunk && (reinterpret_cast<uintptr_t>(dst) & 31u) == 0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int p = 4 * half + i;
                const float lo = dev::f16_bits_to_f32(h[p] & 0xFFFFu), hi = dev::f16_bits_to_f32(h[p] >> 16);
                o[2 * i] = __float_as_uint(__fmul_rn(lo, __uint_as_float(sp[p] << 16)));
                o[2 * i + 1] = __float_as_uint(__fmul_rn(hi, __uint_as_float(sp[p] & 0xFFFF0000u)));
            }
            float* d = dst + 8 * half;
            if (v8) {
                store_v8(d, o);
            } else if (n == kChunk && q.vec_ok) {
                reinterpret_cast<uint4*>(d)[0] = make_uint4(o[0], o[1], o[2], o[3]);
                reinterpret_cast<uint4*>(d)[1] = make_uint4(o[4], o[5], o[6], o[7]);
            } else {
                for (int j = 0; j < 8 && 8 * half + j < n; ++j) d[j] = __uint_as_float(o[j]);
            }
        }
    }
}

// Block b takes rows b, b + gridDim.x, ...; in a row, thread t takes chunks
// t, t + blockDim.x, ...  BR / BC: the block's extent along rows / columns.
template <int FMT, bool BF16, int BR, int BC>
__global__ void __launch_bounds__(kThreads, BF16 ? kMinBlocksBf16 : kMinBlocksF32) dequant_kernel(DequantArgs q) {
    dev::pdl_allow_next();
    dev::pdl_wait_prior();
    const int64_t nchunk = (q.cols + kChunk - 1) / kChunk;
    for (int64_t r = blockIdx.x; r < q.rows; r += gridDim.x) {
        const int64_t srow = r / BR;
        const uint8_t* srow_ptr = q.scale + scale_slot(srow, q.scale_mode) * q.scale_cols;  // unused for SF
        // two chunks a step (t and t + blockDim.x), both loads issued first
        for (int64_t ch = threadIdx.x; ch < nchunk; ch += 2 * blockDim.x) {
            const int64_t chb = ch + blockDim.x;
            const bool two = chb < nchunk;
            const int64_t c0 = ch * kChunk, c1 = chb * kChunk;
            const int n0 = q.cols - c0 >= kChunk ? kChunk : static_cast<int>(q.cols - c0);
            const int n1 = !two ? 0 : q.cols - c1 >= kChunk ? kChunk : static_cast<int>(q.cols - c1);
            uint32_t w0[4], w1[4], h[8], sp[8];
            load_chunk<FMT>(q, r, c0, n0, w0);
            if (two) load_chunk<FMT>(q, r, c1, n1, w1);
            chunk_scales<BC>(q, srow_ptr, srow, c0, n0, sp);
            decode_chunk<FMT>(q, w0, h);
            store_chunk<BF16>(q, h, sp, r, c0, n0);
            if (two) {
                chunk_scales<BC>(q, srow_ptr, srow, c1, n1, sp);
                decode_chunk<FMT>(q, w1, h);
                store_chunk<BF16>(q, h, sp, r, c1, n1);
            }
        }
    }
}

template <int FMT, bool BF16, int BR, int BC>
cudaError_t launch_shape(const DequantArgs& q, cudaStream_t stream) {
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * kGridPerSm;
    const int64_t blocks = q.rows < cap ? q.rows : cap;
    return launch_pdl(dequant_kernel<FMT, BF16, BR, BC>, static_cast<unsigned>(blocks), kThreads, 0, stream, q);
}

template <int FMT, bool BF16>
cudaError_t launch_typed(const DequantArgs& q, cudaStream_t stream) {
    if (q.block_rows == 8) return launch_shape<FMT, BF16, 8, 4>(q, stream);
    if (q.block_rows == 4) return launch_shape<FMT, BF16, 4, 8>(q, stream);
    if (q.block_rows == 1) return launch_shape<FMT, BF16, 1, 32>(q, stream);
    return launch_shape<FMT, BF16, 32, 1>(q, stream);
}

}  // namespace

cudaError_t launch_dequantize(const DequantArgs& q, int fmt, bool out_bf16, cudaStream_t stream) {
    if (q.rows == 0 || q.cols == 0) return cudaSuccess;
    if (out_bf16) {
        switch (fmt) {
        case kE4M3: return launch_typed<kE4M3, true>(q, stream);
        case kE5M2: return launch_typed<kE5M2, true>(q, stream);
        default: return launch_typed<kE2M1, true>(q, stream);
        }
    }
    switch (fmt) {
    case kE4M3: return launch_typed<kE4M3, false>(q, stream);
    case kE5M2: return launch_typed<kE5M2, false>(q, stream);
    default: return launch_typed<kE2M1, false>(q, stream);
    }
}

}  // namespace mx
