// Internal declarations shared by the libmx translation units (host side).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "mx.h"

namespace mx {

// Element formats as the kernels see them.
enum Fmt : int { kE4M3 = 0, kE5M2 = 1, kE2M1 = 2 };

// One QuantizeMX launch, already validated and normalised by the C-ABI layer.
struct QuantArgs {
    const uint8_t* in;      // bf16/f16 elements, byte pointer
    int64_t rows, cols;     // logical extents
    int64_t ld_in;          // input pitch in elements
    uint8_t* data;          // dense output
    int64_t ld_data;        // output pitch in bytes (cols or cols/2)
    uint8_t* scale;         // scale buffer
    int64_t scale_cols;     // columns of the scale tensor
    int32_t block_rows;     // block extent along rows (8, 4, 1, 32)
    int32_t block_cols;     // block extent along columns (4, 8, 32, 1)
    int32_t scale_mode;     // 0 plain, 1 interleave (row i -> (i & 3) + 32 * (i >> 2)),
                            // 2 tensor-core SF tiles (1x32 blocks along rows only)
    int64_t sf_ntk;         // SF mode: 128-column tiles per 128-row tile band
    int32_t emax_bias;      // EMAX (or EMAX-1)
    int32_t fp4_stride;     // lane_remap stride (0 = none)
    int32_t fp4_parity;     // nibble parity
    uint32_t fp4_perm;      // __byte_perm selector placing the 4 pair-bytes of an 8-element chunk
    int32_t vec_ok;         // 16-byte input rows and 8-byte output rows: vectorised kernels allowed
    int32_t vec32_ok;       // 32-byte input rows and 16-byte output rows (FP8; 8-byte e2m1)
};

cudaError_t launch_quantize(const QuantArgs& q, bool in_f16, int fmt, cudaStream_t stream);

// One MX dequantize launch (see mx_dequantize).
struct DequantArgs {
    const uint8_t* data;    // dense codes: rows*cols bytes (FP8) or rows*cols/2 (e2m1)
    const uint8_t* scale;   // scale buffer in the layout of `scale_mode`
    int64_t rows, cols;
    int32_t block_rows, block_cols;  // (8,4), (4,8), (1,32) or (32,1)
    int32_t scale_mode;     // 0 plain, 1 interleave, 2 tensor-core SF
    int64_t scale_cols;     // scale tensor columns (SF: rounded up to 4)
    int64_t sf_ntk;
    uint32_t fp4_inv_perm;  // __byte_perm selector undoing the lane permutation of an 8-element chunk
    int32_t fp4_parity;
    void* out;              // f32 or bf16
    int64_t ld_out;         // elements
    int32_t vec_ok;         // 16-byte aligned output rows
};

cudaError_t launch_dequantize(const DequantArgs& q, int fmt, bool out_bf16, cudaStream_t stream);

// Scale-factor repack: plain [mn, k/32] -> SF tiles (see mx_repack_scales).
cudaError_t launch_repack_scales(const uint8_t* plain, int64_t mn, int64_t k, int64_t ld_plain,
                                 uint8_t* sf, cudaStream_t stream);
// `batch` problems: plain scales every plain_batch_stride bytes, SF layouts
// back to back (sf_layout_bytes(mn, k) each).
cudaError_t launch_repack_scales_batched(const uint8_t* plain, int64_t mn, int64_t k, int64_t ld_plain,
                                         int64_t plain_batch_stride, int64_t batch, uint8_t* sf,
                                         cudaStream_t stream);
// The same from scales stored [k/32, mn] (mn innermost, rows ld_plain bytes).
cudaError_t launch_repack_scales_mn_inner(const uint8_t* plain, int64_t mn, int64_t k, int64_t ld_plain,
                                          int64_t plain_batch_stride, int64_t batch, uint8_t* sf,
                                          cudaStream_t stream);

// Byte-tensor permutation: dst (dense, `rank` axes of extents dst_dims,
// outermost first) takes dst[i_0, .., i_{r-1}] = src[sum_a i_a * src_stride[a]].
constexpr int kMaxPermuteRank = 8;
struct PermuteArgs {
    const uint8_t* src;
    uint8_t* dst;
    int rank;
    int64_t dst_dims[kMaxPermuteRank];
    int64_t src_stride[kMaxPermuteRank];  // elements
};
cudaError_t launch_permute_bytes(const PermuteArgs& a, cudaStream_t stream);
size_t sf_layout_bytes(int64_t mn, int64_t k);

// Block-scaled GEMM on SF-layout scales.
struct GemmArgs {
    const uint8_t* a;        // [M, K] FP8
    const uint8_t* bt;       // [N, K] FP8
    const uint8_t* sfa;      // SF layout for A
    const uint8_t* sfb;      // SF layout for Bt
    int64_t M, N, K;
    void* c;
    int64_t ldc;             // elements
    int32_t elem_fmt;        // kE4M3 | kE5M2
    int32_t out_bf16;        // 1: bf16 output, 0: f32
    int32_t vec_store;       // 1: c and ldc allow 16-byte row stores
    // `batch` independent problems: A, Bt and C advance by their batch strides
    // (bytes, bytes, elements); sfa / sfb hold the problems' SF layouts back
    // to back (sf_layout_bytes(M, K) / (N, K) each).
    int64_t batch;
    int64_t a_batch_stride, b_batch_stride, c_batch_stride;
    // Fused activation quantize (mx_fused_quantize_matmul): the launch
    // itself writes A (a: codes, sfa: SF-layout scales) from X [M, K]
    // bf16/f16, publishing one ready word per 128-row x 256-element item in
    // q_flags ([ceil(M/128), ceil(K/256)] 64-bit words).
    const uint8_t* x;
    int64_t ld_x_bytes;
    int32_t x_f16;
    uint64_t* q_flags;
    // FP8, not fused: A stored [batch, K, M] / Bt stored [batch, K, N] (M / N
    // innermost, rows M / N bytes, a multiple of 16; the batch strides still
    // count the whole problem); read as MN-major tiles by either kernel.
    int32_t a_mn_major, b_mn_major;
};
cudaError_t launch_scaled_matmul(const GemmArgs& g, cudaStream_t stream);
// Whether launch_scaled_matmul runs `g` on the pair kernel (else the 1-SM one).
bool scaled_matmul_takes_pair(const GemmArgs& g);
// Whether the fused call runs as one launch of the pair kernel (else
// QuantizeMX, then launch_scaled_matmul), and that launch.
bool fused_single_launch(const GemmArgs& g);
cudaError_t launch_fused_matmul(const GemmArgs& g, cudaStream_t stream);

// Which kernel the last ScaledMatmul launch on this host used (testing aid).
struct GemmLaunchInfo {
    int kernel;   // 1: 1-SM kernel, 2: 2-SM pair kernel, 3: pair kernel with the
                  // fused activation quantize, 0: none yet
    int split_k;  // CTAs per tile along K (1-SM kernel), else 1
    int a_mn_major, b_mn_major;  // operands read MN-major
};
GemmLaunchInfo last_gemm_launch();

// Per-device properties, cached.
int device_sm_count();
bool device_is_sm103();

// Device status word (first device-side error since the last read).
cudaError_t read_and_clear_device_status(int* status);

}  // namespace mx
