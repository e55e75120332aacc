// Byte-tensor permutation for the general block-scaled dot: brings an FP8
// operand (and its E8M0 scale tensor) into the [batch, rows, K] order the
// tensor-core kernels read, K innermost.
//
// After axes of extent 1 are dropped and axes that stay adjacent and in order
// are merged, one of two kernels runs:
//   rows       the innermost destination axis is contiguous in the source:
//              each block copies whole rows (16-byte accesses when aligned);
//              the source offset of a row is found once per row.
//   transpose  otherwise: each block moves 128 x 128-byte tiles between the
//              axis that is contiguous in the source (i) and the
//              destination's innermost axis (j) through shared memory, whole
//              128-byte lines on both sides; 4 x 4 byte blocks are
//              transposed in registers with byte permutes.  Tiles at the
//              edges, or unaligned ones, go byte by byte.

#include <cstdint>

#include "mx_internal.h"
#include "pdl.cuh"

namespace mx {
namespace {

constexpr int kThreads = 256;

struct Dims {
    int rank;
    int64_t dst_dims[kMaxPermuteRank];
    int64_t src_stride[kMaxPermuteRank];
    int64_t dst_stride[kMaxPermuteRank];
};

// Source offset of destination row `row` (all axes but the innermost).
__device__ __forceinline__ int64_t row_offset(const Dims& d, int64_t row) {
    int64_t off = 0;
    for (int a = d.rank - 2; a >= 0; --a) {
        const int64_t n = d.dst_dims[a];
        const int64_t q = row / n;
        off += (row - q * n) * d.src_stride[a];
        row = q;
    }
    return off;
}

__global__ void __launch_bounds__(kThreads) permute_rows(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                         Dims d, int64_t rows) {
    dev::pdl_allow_next();
    dev::pdl_wait_prior();
    const int64_t len = d.dst_dims[d.rank - 1];
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint8_t* s = src + row_offset(d, r);
        uint8_t* o = dst + r * len;
        if (((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(o)) & 15u) == 0) {
            const int64_t n16 = len / 16;
            for (int64_t i = threadIdx.x; i < n16; i += blockDim.x)
                reinterpret_cast<uint4*>(o)[i] = reinterpret_cast<const uint4*>(s)[i];
            for (int64_t i = n16 * 16 + threadIdx.x; i < len; i += blockDim.x) o[i] = s[i];
        } else {
            for (int64_t i = threadIdx.x; i < len; i += blockDim.x) o[i] = s[i];
        }
    }
}

// 4 x 4 byte transpose: out[m] byte k = in[k] byte m.
__device__ __forceinline__ void transpose4x4(const uint32_t (&in)[4], uint32_t (&out)[4]) {
    const uint32_t lo01 = __byte_perm(in[0], in[1], 0x5140), hi01 = __byte_perm(in[0], in[1], 0x7362);
    const uint32_t lo23 = __byte_perm(in[2], in[3], 0x5140), hi23 = __byte_perm(in[2], in[3], 0x7362);
    out[0] = __byte_perm(lo01, lo23, 0x5410);
    out[1] = __byte_perm(lo01, lo23, 0x7632);
    out[2] = __byte_perm(hi01, hi23, 0x5410);
    out[3] = __byte_perm(hi01, hi23, 0x7632);
}

constexpr int kTile = 128;     // bytes of both tile axes
constexpr int kPitchWords = 33;  // shared tile row: 128 bytes + one word against bank conflicts

// Block tiles of 128 x 128 bytes between destination axis `ai` (contiguous
// in the source) and the innermost destination axis j; every other axis
// indexes whole tiles.  A full, aligned tile moves in three steps:
//   1. 128 source rows (one per j) of 128 bytes (i): 16-byte global loads,
//      8 threads a row, stored as words into a shared tile [j][i];
//   2. thread (bi, jg) reads the 4 x 16 bytes at i = 4 bi .. 4 bi + 3,
//      j = 16 jg .. 16 jg + 15 as 16 words and transposes them (4 x 4 byte
//      blocks, byte permutes) into 4 destination rows of 16 bytes;
//   3. 16-byte global stores: the 8 threads of a destination row write its
//      128 bytes, a warp 4 whole rows an instruction.
// A tile cut by the tensor's edge takes this path too when both of its
// extents are multiples of 16 bytes (threads past them idle); other edge
// tiles, or tiles whose rows do not allow 16-byte accesses, go byte by byte.
// `aligned`: source and destination rows are 16-byte aligned.
__global__ void __launch_bounds__(kThreads) permute_transpose(const uint8_t* __restrict__ src,
                                                              uint8_t* __restrict__ dst, Dims d, int ai,
                                                              int64_t tiles_i, int64_t tiles_j, int64_t units,
                                                              int aligned) {
    __shared__ uint32_t tile[kTile * kPitchWords];
    dev::pdl_allow_next();
    dev::pdl_wait_prior();
    const int aj = d.rank - 1;
    const int64_t ni = d.dst_dims[ai], nj = d.dst_dims[aj];
    const int64_t sj = d.src_stride[aj], di = d.dst_stride[ai];
    const int t = threadIdx.x;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        int64_t rest = u;
        const int64_t tj = rest % tiles_j;
        rest /= tiles_j;
        const int64_t ti = rest % tiles_i;
        rest /= tiles_i;
        int64_t sbase = 0, dbase = 0;
        for (int a = d.rank - 2; a >= 0; --a) {
            if (a == ai) continue;
            const int64_t n = d.dst_dims[a];
            const int64_t q = rest / n;
            const int64_t idx = rest - q * n;
            sbase += idx * d.src_stride[a];
            dbase += idx * d.dst_stride[a];
            rest = q;
        }
        const int64_t i0 = ti * kTile, j0 = tj * kTile;
        const int ei = static_cast<int>(ni - i0 < kTile ? ni - i0 : kTile);  // the tile's extents
        const int ej = static_cast<int>(nj - j0 < kTile ? nj - j0 : kTile);
        if (aligned && ei % 16 == 0 && ej % 16 == 0) {
            const uint8_t* s = src + sbase + i0 + j0 * sj;
            // 1. rows j = t / 8 + 32 p, 16 bytes c = t % 8 of each
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int r = t / 8 + 32 * p, c = t % 8;
                if (r < ej && 16 * c < ei) {
                    const uint4 v = *reinterpret_cast<const uint4*>(s + r * sj + 16 * c);
                    uint32_t* w = &tile[r * kPitchWords + 4 * c];
                    w[0] = v.x;
                    w[1] = v.y;
                    w[2] = v.z;
                    w[3] = v.w;
                }
            }
            __syncthreads();
            // 2. thread (bi, jg): words bi of rows 16 jg .. 16 jg + 15
            const int bi = t / 8, jg = t % 8;
            if (4 * bi < ei && 16 * jg < ej) {
                uint32_t o[4][4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t in[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) in[r] = tile[(16 * jg + 4 * k + r) * kPitchWords + bi];
                    transpose4x4(in, o[k]);  // o[k][m]: row i = 4 bi + m, bytes j = 16 jg + 4 k .. + 3
                }
                // 3. destination rows i0 + 4 bi + m, bytes j0 + 16 jg .. + 15
                uint8_t* o_row = dst + dbase + (i0 + 4 * bi) * di + j0 + 16 * jg;
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    *reinterpret_cast<uint4*>(o_row + m * di) = make_uint4(o[0][m], o[1][m], o[2][m], o[3][m]);
            }
            __syncthreads();  // the tile is reused by the next unit
        } else {
            for (int64_t e = t; e < static_cast<int64_t>(ei) * ej; e += blockDim.x) {
                const int64_t ii = e / ej, jj = e - ii * ej;
                dst[dbase + (i0 + ii) * di + j0 + jj] = src[sbase + i0 + ii + (j0 + jj) * sj];
            }
        }
    }
}

}  // namespace

cudaError_t launch_permute_bytes(const PermuteArgs& a, cudaStream_t stream) {
    // drop extent-1 axes, merge neighbours that stay adjacent in the source
    Dims d{};
    int64_t total = 1;
    for (int i = 0; i < a.rank; ++i) {
        total *= a.dst_dims[i];
        if (a.dst_dims[i] == 1) continue;
        if (d.rank > 0 && d.src_stride[d.rank - 1] == a.src_stride[i] * a.dst_dims[i]) {
            d.dst_dims[d.rank - 1] *= a.dst_dims[i];
            d.src_stride[d.rank - 1] = a.src_stride[i];
            continue;
        }
        d.dst_dims[d.rank] = a.dst_dims[i];
        d.src_stride[d.rank] = a.src_stride[i];
        ++d.rank;
    }
    if (total == 0) return cudaSuccess;
    if (d.rank == 0) {  // a single element
        d.rank = 1;
        d.dst_dims[0] = 1;
        d.src_stride[0] = 1;
    }
    int64_t stride = 1;
    for (int i = d.rank - 1; i >= 0; --i) {
        d.dst_stride[i] = stride;
        stride *= d.dst_dims[i];
    }
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (d.src_stride[d.rank - 1] == 1) {
        const int64_t rows = total / d.dst_dims[d.rank - 1];
        const int64_t grid = rows < cap ? rows : cap;
        return launch_pdl(permute_rows, static_cast<unsigned>(grid), kThreads, 0, stream, a.src, a.dst, d, rows);
    }
    int ai = -1;
    for (int i = 0; i < d.rank - 1; ++i)
        if (d.src_stride[i] == 1) ai = i;
    if (ai < 0) return cudaErrorInvalidValue;  // not a permutation of a dense tensor
    const int64_t tiles_i = (d.dst_dims[ai] + kTile - 1) / kTile;
    const int64_t tiles_j = (d.dst_dims[d.rank - 1] + kTile - 1) / kTile;
    const int64_t units = total / (d.dst_dims[ai] * d.dst_dims[d.rank - 1]) * tiles_i * tiles_j;
    // 16-byte accesses along i in the source and along j in the destination
    bool aligned = (reinterpret_cast<uintptr_t>(a.src) & 15u) == 0 && (reinterpret_cast<uintptr_t>(a.dst) & 15u) == 0 &&
                   d.src_stride[d.rank - 1] % 16 == 0 && d.dst_stride[ai] % 16 == 0;
    for (int i = 0; i < d.rank - 1; ++i)
        if (i != ai) aligned = aligned && d.src_stride[i] % 16 == 0 && d.dst_stride[i] % 16 == 0;
    const int64_t grid = units < cap ? units : cap;
    return launch_pdl(permute_transpose, static_cast<unsigned>(grid), kThreads, 0, stream, a.src, a.dst, d, ai,
                      tiles_i, tiles_j, units, aligned ? 1 : 0);
}

}  // namespace mx
