// Byte-tensor permutation for the general block-scaled dot: brings an FP8
// operand (and its E8M0 scale tensor) into the [batch, rows, K] order the
// tensor-core kernels read, K innermost.
//
// After axes of extent 1 are dropped and axes that stay adjacent and in order
// are merged, one of two kernels runs:
//   rows       the innermost destination axis is contiguous in the source:
//              each block copies whole rows (16-byte accesses when aligned);
//              the source offset of a row is found once per row.
//   transpose  otherwise: 64 x 64 tiles between the destination's innermost
//              axis and the axis that is contiguous in the source, staged
//              through shared memory so both the loads and the stores run
//              along contiguous bytes.

#include <cstdint>

#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;

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

// Tiles between destination axes `ai` (contiguous in the source) and the
// innermost destination axis; every other axis indexes whole tiles.
__global__ void __launch_bounds__(kThreads) permute_transpose(const uint8_t* __restrict__ src,
                                                              uint8_t* __restrict__ dst, Dims d, int ai,
                                                              int64_t tiles_i, int64_t tiles_j, int64_t units) {
    __shared__ uint8_t tile[kTile][kTile + 4];
    const int aj = d.rank - 1;
    const int64_t ni = d.dst_dims[ai], nj = d.dst_dims[aj];
    const int64_t sj = d.src_stride[aj], di = d.dst_stride[ai];
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
        const int col = threadIdx.x % kTile;
        __syncthreads();  // the previous unit's reads of `tile` are done
        for (int row = threadIdx.x / kTile; row < kTile; row += kThreads / kTile) {
            // row: j within the tile; col: i (contiguous in the source)
            if (i0 + col < ni && j0 + row < nj) tile[row][col] = src[sbase + (i0 + col) + (j0 + row) * sj];
        }
        __syncthreads();
        for (int row = threadIdx.x / kTile; row < kTile; row += kThreads / kTile) {
            // row: i within the tile; col: j (contiguous in the destination)
            if (i0 + row < ni && j0 + col < nj) dst[dbase + (i0 + row) * di + (j0 + col)] = tile[col][row];
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
        permute_rows<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a.src, a.dst, d, rows);
        return cudaGetLastError();
    }
    int ai = -1;
    for (int i = 0; i < d.rank - 1; ++i)
        if (d.src_stride[i] == 1) ai = i;
    if (ai < 0) return cudaErrorInvalidValue;  // not a permutation of a dense tensor
    const int64_t tiles_i = (d.dst_dims[ai] + kTile - 1) / kTile;
    const int64_t tiles_j = (d.dst_dims[d.rank - 1] + kTile - 1) / kTile;
    const int64_t units = total / (d.dst_dims[ai] * d.dst_dims[d.rank - 1]) * tiles_i * tiles_j;
    const int64_t grid = units < cap ? units : cap;
    permute_transpose<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a.src, a.dst, d, ai, tiles_i, tiles_j,
                                                                            units);
    return cudaGetLastError();
}

}  // namespace mx
