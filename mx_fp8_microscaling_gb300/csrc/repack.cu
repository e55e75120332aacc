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
// A block takes 128 rows x up to 64 scale columns (16 tiles): it reads the
// rows' contiguous 64-byte segments (16-byte loads where aligned) into shared
// memory and writes the 16 tiles, which are contiguous in the output, with
// 16-byte stores.  A batch of problems is one launch: their SF layouts are
// written back to back.  Scales stored the other way round, [k/32, mn] with
// mn innermost (the scales of an operand stored [K, MN]), are read as 128-row
// segments per scale column and transposed through the same shared tile.

#include <cstdint>
#include <cstring>

#include "mx_internal.h"
#include "pdl.cuh"

namespace mx {
namespace {

constexpr int kRepackThreads = 256;
constexpr int kTilesPerBlock = 16;                 // 64 scale columns
constexpr int kCols = 4 * kTilesPerBlock;

__global__ void __launch_bounds__(kRepackThreads) repack_sf_kernel(const uint8_t* __restrict__ plain, int64_t mn,
                                                                  int64_t kb, int64_t ld, int64_t ntm, int64_t ntk,
                                                                  int64_t plain_batch_stride, int64_t batch,
                                                                  uint8_t* __restrict__ sf, int vec_ok,
                                                                  int mn_inner) {
    dev::pdl_allow_next();
    dev::pdl_wait_prior();
    __shared__ __align__(16) uint8_t rows[128][kCols + 16];
    const int64_t nchunk = (ntk + kTilesPerBlock - 1) / kTilesPerBlock;
    const int64_t units = batch * ntm * nchunk;
    const int64_t sf_batch_bytes = ntm * ntk * 512;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t chunk = u % nchunk;
        const int64_t tm = (u / nchunk) % ntm;
        const int64_t b = u / (nchunk * ntm);
        const uint8_t* src = plain + b * plain_batch_stride;
        const int64_t c0 = chunk * kCols;                  // first scale column
        const int tiles = static_cast<int>(ntk - chunk * kTilesPerBlock < kTilesPerBlock
                                               ? ntk - chunk * kTilesPerBlock
                                               : kTilesPerBlock);
        __syncthreads();  // the previous unit's reads of `rows` are done
        // rows tm*128 .. +127, columns c0 .. c0+63 (0 past the matrix)
        if (mn_inner) {
            // scale (r, c) at src[c * ld + r]: 16 rows of one column per step
            for (int i = threadIdx.x; i < kCols * 8; i += kRepackThreads) {
                const int cc = i >> 3, seg = i & 7;
                const int64_t c = c0 + cc, r = tm * 128 + 16 * seg;
                uint8_t v[16];
                if (c < kb && vec_ok && r + 16 <= mn) {
                    const uint4 w = *reinterpret_cast<const uint4*>(src + c * ld + r);
                    memcpy(v, &w, 16);
                } else {
                    for (int j = 0; j < 16; ++j) v[j] = (c < kb && r + j < mn) ? src[c * ld + r + j] : uint8_t(0);
                }
                for (int j = 0; j < 16; ++j) rows[16 * seg + j][cc] = v[j];
            }
        } else
        for (int i = threadIdx.x; i < 128 * (kCols / 16); i += kRepackThreads) {
            const int rr = i / (kCols / 16), seg = i % (kCols / 16);
            const int64_t r = tm * 128 + rr, c = c0 + 16 * seg;
            uint8_t* dst = &rows[rr][16 * seg];
            if (r < mn && c < kb && vec_ok && c + 16 <= kb) {
                *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src + r * ld + c);
            } else {
                for (int j = 0; j < 16; ++j) dst[j] = (r < mn && c + j < kb) ? src[r * ld + c + j] : uint8_t(0);
            }
        }
        __syncthreads();
        // tile t, 16-byte group q holds the 4-column words of rows q, q+32,
        // q+64, q+96
        uint4* out = reinterpret_cast<uint4*>(sf + b * sf_batch_bytes + (tm * ntk + chunk * kTilesPerBlock) * 512);
        for (int i = threadIdx.x; i < tiles * 32; i += kRepackThreads) {
            const int t = i >> 5, q = i & 31;
            uint4 v;
            v.x = *reinterpret_cast<const uint32_t*>(&rows[q][4 * t]);
            v.y = *reinterpret_cast<const uint32_t*>(&rows[q + 32][4 * t]);
            v.z = *reinterpret_cast<const uint32_t*>(&rows[q + 64][4 * t]);
            v.w = *reinterpret_cast<const uint32_t*>(&rows[q + 96][4 * t]);
            out[i] = v;
        }
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
    const int64_t ntm = (mn + 127) / 128;
    const int64_t ntk = (kb + 3) / 4;
    if (ntm == 0 || ntk == 0 || batch == 0) return cudaSuccess;
    const int64_t units = batch * ntm * ((ntk + kTilesPerBlock - 1) / kTilesPerBlock);
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    const int64_t blocks = units < cap ? units : cap;
    const int vec_ok = (reinterpret_cast<uintptr_t>(plain) & 15u) == 0 && ld_plain % 16 == 0 &&
                       plain_batch_stride % 16 == 0;
    return launch_pdl(repack_sf_kernel, static_cast<unsigned>(blocks), kRepackThreads, 0, stream, plain, mn, kb,
                      ld_plain, ntm, ntk, plain_batch_stride, batch, sf, vec_ok, 0);
}

cudaError_t launch_repack_scales_mn_inner(const uint8_t* plain, int64_t mn, int64_t k, int64_t ld_plain,
                                          int64_t plain_batch_stride, int64_t batch, uint8_t* sf,
                                          cudaStream_t stream) {
    const int64_t kb = k / 32;
    const int64_t ntm = (mn + 127) / 128;
    const int64_t ntk = (kb + 3) / 4;
    if (ntm == 0 || ntk == 0 || batch == 0) return cudaSuccess;
    const int64_t units = batch * ntm * ((ntk + kTilesPerBlock - 1) / kTilesPerBlock);
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    const int64_t blocks = units < cap ? units : cap;
    const int vec_ok = (reinterpret_cast<uintptr_t>(plain) & 15u) == 0 && ld_plain % 16 == 0 &&
                       plain_batch_stride % 16 == 0;
    return launch_pdl(repack_sf_kernel, static_cast<unsigned>(blocks), kRepackThreads, 0, stream, plain, mn, kb,
                      ld_plain, ntm, ntk, plain_batch_stride, batch, sf, vec_ok, 1);
}

cudaError_t launch_repack_scales(const uint8_t* plain, int64_t mn, int64_t k, int64_t ld_plain,
                                 uint8_t* sf, cudaStream_t stream) {
    return launch_repack_scales_batched(plain, mn, k, ld_plain, 0, 1, sf, stream);
}

}  // namespace mx
