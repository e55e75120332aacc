// Byte-tensor permutation for the general block-scaled dot: brings an FP8
// operand (and its E8M0 scale tensor) into the [batch, rows, K] order the
// tensor-core kernels read, K innermost.
//
// After axes of extent 1 are dropped and axes that stay adjacent and in order
// are merged, one of two kernels runs:
//   rows       the innermost destination axis is contiguous in the source:
//              each block copies whole rows (16-byte accesses when aligned);
//              the source offset of a row is found once per row.
//   transpose  otherwise: each warp moves a 64 x 32-byte tile between the
//              axis that is contiguous in the source (i) and the
//              destination's innermost axis (j).  A lane loads 16 words
//              (4 bytes of i from 16 rows of j), transposes them in registers
//              with byte permutes and stores 4 rows of 16 bytes: both sides
//              touch whole 32-byte sectors, and no shared memory is needed.
//              Tiles at the edges, or unaligned ones, go byte by byte.

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

constexpr int kTileI = 64;  // bytes of the source-contiguous axis per warp tile
constexpr int kTileJ = 32;  // bytes of the destination-contiguous axis per warp tile

// Warp tiles between destination axis `ai` (contiguous in the source) and
// the innermost destination axis; every other axis indexes whole tiles.
// `aligned`: source rows and destination rows allow 4- / 16-byte accesses.
__global__ void __launch_bounds__(kThreads) permute_transpose(const uint8_t* __restrict__ src,
                                                              uint8_t* __restrict__ dst, Dims d, int ai,
                                                              int64_t tiles_i, int64_t tiles_j, int64_t units,
                                                              int aligned) {
    dev::pdl_allow_next();
    dev::pdl_wait_prior();
    const int aj = d.rank - 1;
    const int64_t ni = d.dst_dims[ai], nj = d.dst_dims[aj];
    const int64_t sj = d.src_stride[aj], di = d.dst_stride[ai];
    const int lane = threadIdx.x & 31;
    const int bq = lane & 15, half = lane >> 4;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); u < units;
         u += warps) {
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
        const int64_t i = ti * kTileI + 4 * bq;    // this lane's 4 bytes of i
        const int64_t j = tj * kTileJ + 16 * half; // this lane's 16 rows of j
        const bool full = (ti + 1) * kTileI <= ni && (tj + 1) * kTileJ <= nj;
        if (aligned && full) {
            const uint8_t* s = src + sbase + i + j * sj;
            uint32_t w[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) w[r] = *reinterpret_cast<const uint32_t*>(s + r * sj);
            uint32_t o[4][4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t in[4] = {w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]};
                transpose4x4(in, o[k]);
            }
            uint8_t* o_row = dst + dbase + i * di + j;
#pragma unroll
            for (int m = 0; m < 4; ++m)
                *reinterpret_cast<uint4*>(o_row + m * di) = make_uint4(o[0][m], o[1][m], o[2][m], o[3][m]);
        } else {
            for (int m = 0; m < 4; ++m)
                for (int r = 0; r < 16; ++r)
                    if (i + m < ni && j + r < nj) dst[dbase + (i + m) * di + j + r] = src[sbase + (i + m) + (j + r) * sj];
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
    const int64_t tiles_i = (d.dst_dims[ai] + kTileI - 1) / kTileI;
    const int64_t tiles_j = (d.dst_dims[d.rank - 1] + kTileJ - 1) / kTileJ;
    const int64_t units = total / (d.dst_dims[ai] * d.dst_dims[d.rank - 1]) * tiles_i * tiles_j;
    // 4-byte source loads along i, 16-byte destination stores along j
    bool aligned = (reinterpret_cast<uintptr_t>(a.src) & 3u) == 0 && (reinterpret_cast<uintptr_t>(a.dst) & 15u) == 0 &&
                   d.src_stride[d.rank - 1] % 4 == 0 && d.dst_stride[ai] % 16 == 0;
    for (int i = 0; i < d.rank - 1; ++i)
        if (i != ai) aligned = aligned && d.src_stride[i] % 4 == 0 && d.dst_stride[i] % 16 == 0;
    const int64_t warps = (units + 7) / 8;
    const int64_t grid = warps < cap ? warps : cap;
    return launch_pdl(permute_transpose, static_cast<unsigned>(grid), kThreads, 0, stream, a.src, a.dst, d, ai,
                      tiles_i, tiles_j, units, aligned ? 1 : 0);
}

}  // namespace mx
