// Scale-factor repack: plain E8M0 [mn, k/32] -> the block-scaled tcgen05 MMA
// scale-factor layout.
//
// The tensor core reads the scale of row r from TMEM lane r % 32, column
// r / 32 of a 4-column group, byte = K-block within the group; one
// tcgen05.cp.32x128b.warpx4 moves a 512-byte tile (32 rows of 16 bytes) into
// that group.  So a tile covers 128 rows x 4 scale columns, and inside it
// scale (r, c) sits at byte (r % 32) * 16 + (r / 32) * 4 + c.  Tiles are
// ordered row-tile-major: tile (t_mn, t_k) at ((t_mn * ceil(k/128)) + t_k) * 512.
// Padding rows/columns are written as 0.
//
// One thread writes one 32-bit word (the four K-block scales of one row), so
// stores are fully coalesced; the reads gather four rows 32 apart.  A batch of
// problems is one launch: their SF layouts are written back to back.

#include <cstdint>

#include "mx_internal.h"

namespace mx {
namespace {

__global__ void __launch_bounds__(256) repack_sf_kernel(const uint8_t* __restrict__ plain, int64_t mn,
                                                       int64_t kb, int64_t ld, int64_t ntk, int64_t nwords,
                                                       int64_t plain_batch_stride, int64_t batch,
                                                       uint32_t* __restrict__ sf) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t total = nwords * batch;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t b = batch == 1 ? 0 : i / nwords;
        const int64_t w = i - b * nwords;
        const uint8_t* src = plain + b * plain_batch_stride;
        const int64_t tile = w >> 7;          // 128 words per 512-byte tile
        const int within = static_cast<int>(w & 127);
        const int64_t tm = tile / ntk, tk = tile - (tile / ntk) * ntk;
        const int64_t r = tm * 128 + (within >> 2) + 32 * (within & 3);
        const int64_t c0 = tk * 4;
        uint32_t word = 0;
        if (r < mn) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c0 + j < kb) word |= static_cast<uint32_t>(src[r * ld + c0 + j]) << (8 * j);
        }
        sf[i] = word;
    }
}

}  // namespace

size_t sf_layout_bytes(int64_t mn, int64_t k) {
    const int64_t kb = k / 32;
    return static_cast<size_t>((mn + 127) / 128) * static_cast<size_t>((kb + 3) / 4) * 512u;
}

cudaError_t launch_repack_scales_batched(const uint8_t* plain, int64_t mn, int64_t k, int64_t ld_plain,
                                         int64_t plain_batch_stride, int64_t batch, uint8_t* sf,
                                         cudaStream_t stream) {
    const int64_t kb = k / 32;
    const int64_t ntk = (kb + 3) / 4;
    const int64_t nwords = static_cast<int64_t>(sf_layout_bytes(mn, k) / 4);
    if (nwords == 0 || batch == 0) return cudaSuccess;
    int64_t blocks = (nwords * batch + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    repack_sf_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        plain, mn, kb, ld_plain, ntk, nwords, plain_batch_stride, batch, reinterpret_cast<uint32_t*>(sf));
    return cudaGetLastError();
}

cudaError_t launch_repack_scales(const uint8_t* plain, int64_t mn, int64_t k, int64_t ld_plain,
                                 uint8_t* sf, cudaStream_t stream) {
    return launch_repack_scales_batched(plain, mn, k, ld_plain, 0, 1, sf, stream);
}

}  // namespace mx
