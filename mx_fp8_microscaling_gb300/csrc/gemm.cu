// Block-scaled FP8 GEMM (ScaledMatmul) on the sm_103a tensor cores.
//
//   C[m,n] = sum_k dec(A[m,k]) 2^(sA[m,k/32]-127) * dec(Bt[n,k]) 2^(sB[n,k/32]-127)
//
// (ScaledMatmul of the page "MX-FP8 Microscaling Legalization", sections 3-4;
// the scale is applied as 2^(E8M0 - 127), the inverse of the quantizer's
// prescale, page "MX Microscaling", quantizeDataApplyingMxScales NOTE.)
//
// Two persistent, warp-specialised kernels share one structure (one CTA per
// SM, 352 threads):
//   warp 0      TMA producer: per 128-wide K block, 2-D TMA loads of the
//               operand tiles (128-byte swizzle) and of the scale-factor
//               tiles into a ring of shared-memory stages.
//   warp 10     scale copies (one thread): once a stage's operands land,
//               tcgen05.cp moves its scale tiles into tensor memory and a
//               tcgen05.commit tells the MMA thread.  A tcgen05.cp costs its
//               issuing thread about as much as the four MMAs of a K block,
//               so it is kept off the MMA thread.
//   warp 1      MMA issuer (one thread): four
//               tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each) per K
//               block accumulate into an f32 tile in tensor memory;
//               tcgen05.commit frees the stage / hands the tile over.
//   warps 2-9   epilogue: tcgen05.ld the accumulator (each warp its TMEM lane
//               quarter and one 128-column half, one x128 load), release
//               tensor memory, then
//               convert (f32, or bf16 round-to-nearest-even) and store rows to
//               global memory while the next tile's main loop runs.  Stores are
//               256-bit (a whole 32-byte sector each) where the rows allow:
//               4 % faster than 128-bit ones at 8192^3.  In the pair kernel
//               the CTA that issues the MMAs paces its stores by the MMA
//               thread's progress through the next tile (see the epilogue).
//
// Both kernels also run MXFP4 (packed e2m1 operands, kind::mxf4 with
// scale_vec::2X, K = 64 per MMA): a 128-byte stage row then holds 256 K
// elements and two scale tiles along K.
//
//   mx_gemm_kernel      1 SM per 128 x 256 tile (M = 128 MMA), 4 stages of
//                       A 16 KB + B 32 KB + scales 1.5 KB.  Used for M <= 128
//                       and for problems with too few tiles for the pair
//                       kernel (see prefer_pair).
//                       When the tiles are too few to fill the GPU it splits K:
//                       a cluster of S <= 8 CTAs per tile, CTA s accumulating
//                       the s-th slice of the K stages; each slice's f32 tile
//                       goes to its CTA's drained stage buffers, and the
//                       cluster sums the S partials chunk by chunk in slice
//                       order through distributed shared memory (the same
//                       bits on every run) and stores C.
//   mx_gemm_2sm_kernel  a cluster of 2 CTAs per 256 x 256 tile with the pair
//                       MMA (cta_group::2, M = 256): each CTA loads its own
//                       128 rows of A and 128 rows of B, so each SM takes in
//                       32 KB of operands per K block instead of 48 KB.
//                       6 stages.  Rank 0 issues the MMAs; both CTAs' loads
//                       complete on rank 0's barriers.
//
// Tensor memory (512 columns): accumulator in columns 0..255, scale factors
// of stage s at 256 + 16 s (A: 4 columns, B: 8 columns).  The scale-factor
// tile for 128 rows is 512 bytes (row r at byte (r%32)*16 + (r/32)*4 + kblock),
// the layout one tcgen05.cp.32x128b.warpx4 moves into a 4-column group.
//
// Every mbarrier wait is bounded (2 s of wall clock by default); a wait that
// gives up records MX_ERR_TIMEOUT in the device status word and all roles
// leave their loops, wait for their own asynchronous work, free tensor memory
// and return.

#include <atomic>
#include <chrono>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "pdl.cuh"
#include "quant_math.cuh"
#include "tcgen05.cuh"

namespace mx {

// First device-side error since the last read (an mx_status value).
__device__ int g_mx_status = 0;

namespace {

using namespace dev;

constexpr int BK = 128;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_SF = 256;
constexpr uint32_t kEpiBarrier = 1;  // named barrier of a CTA's epilogue warps (0 is __syncthreads)
// scale-factor columns per stage: FP8 A 4 + B 8; FP4 (two K groups) A 8 + B 16
__host__ __device__ constexpr uint32_t sf_cols(bool fp4) { return fp4 ? 32u : 16u; }

struct KParams {
    const uint8_t* sfa;
    const uint8_t* sfb;
    void* c;
    int64_t ldc;
    int M, N, K;
    int out_bf16;
    int vec_store;       // 16-byte row stores allowed (aligned c and pitch)
    int num_m_tiles, num_n_tiles, num_kb;  // num_kb: K stages (128 FP8 or 256 FP4 elements each)
    int sf_ntk;          // 512-byte scale tiles along K per 128 rows (one per 128 elements)
    int num_sf_n_tiles;  // 128-row scale tiles of B
    int batch;           // independent problems; tiles run batch-major
    int64_t c_batch_stride;   // elements between consecutive C matrices
    int64_t sfa_batch_tiles;  // 512-byte scale tiles per problem (A / B)
    int64_t sfb_batch_tiles;
    int group_m;
    int first_group_m;    // M-tiles of the first group (<= group_m; smaller in the fused kernel)
    uint32_t idesc;
    uint32_t idesc_half;  // the same MMA with N = 128 (split tail tiles of the pair kernel)
    int full_rounds;      // pair kernel: rounds of whole tiles before a split tail round
    int split_tail;       // 1: the last round's tiles run as two 256 x 128 halves each
    int split_k;          // 1-SM kernel: CTAs (one cluster) per tile, each a slice of K; 1 = none
    uint64_t timeout_ns;
    int skip_producer;   // fault injection: never issue loads (waits must time out)
    // Fused activation quantize (pair kernel instantiated with QFMT >= 0):
    // X [M, K] bf16/f16 is quantized along K into the A operand (q_xq) and
    // its SF-layout scales (q_sf, the buffer sfa points to), in items of 128
    // rows x kQChunk elements that the epilogue warps take between tiles.
    const uint8_t* q_x;
    int64_t q_ld_x;       // bytes between rows of X
    uint8_t* q_xq;        // codes [M, K] (FP8) or [M, K / 2] (e2m1)
    uint8_t* q_sf;
    uint64_t* q_flags;    // one ready word per item, [q_panels, q_nkc], then the launch's done word
    uint64_t q_tag;       // this launch's tag, 40 bits, nonzero (see wait_items_ready)
    int q_f16;            // X is f16 (else bf16)
    int q_panels;         // 128-row panels of X
    int q_nkc;            // items along K per panel
    int q_lookahead;      // tile groups past the CTA's current one whose items it may quantize
    int q_emax;           // EMAX of the element format
    int q_no_publish;     // fault injection: items are never published (the loads' waits time out)
    // FP8 only: A (B) is stored [batch, K, M] ([batch, K, N]), M (N)
    // innermost, and read as MN-major tiles.  The kernels take the layout
    // from their MN template bits; these record it for the launch's caller.
    int a_mn, b_mn;
};

// Tile order: problem by problem; inside one, groups of M-tiles (the first
// `first_group_m`, then `group_m` each), column-major inside a group, so the
// tiles running at once share A and B panels in L2.
__device__ __forceinline__ void tile_coords(int t, const KParams& p, int& b, int& mt, int& nt) {
    const int per_problem = p.num_m_tiles * p.num_n_tiles;
    b = t / per_problem;
    t -= b * per_problem;
    const int fm = min(p.first_group_m, p.num_m_tiles);
    int first_m, gm, idx;
    if (t < fm * p.num_n_tiles) {
        first_m = 0;
        gm = fm;
        idx = t;
    } else {
        t -= fm * p.num_n_tiles;
        const int group = p.group_m * p.num_n_tiles;
        const int g = t / group;
        first_m = fm + g * p.group_m;
        gm = min(p.num_m_tiles - first_m, p.group_m);
        idx = t - g * group;
    }
    mt = first_m + idx % gm;
    nt = idx / gm;
}

// Tile group of M-tile mt (0 for the first group).
__device__ __forceinline__ int m_tile_group(const KParams& p, int mt) {
    const int fm = min(p.first_group_m, p.num_m_tiles);
    return mt < fm ? 0 : 1 + (mt - fm) / p.group_m;
}

// Work units of the pair kernel's cluster `c` (of `nc`).  Whole 256 x 256
// tiles round-robin over the clusters; when the last round would leave most
// clusters idle (its tiles fit in half of them), each of its tiles runs as
// two 256 x 128 halves on two clusters instead, halving the tail.
__device__ __forceinline__ int pair_units(const KParams& p, int c, int nc) {
    if (p.split_tail) return p.full_rounds + (c < 2 * (p.batch * p.num_m_tiles * p.num_n_tiles - p.full_rounds * nc));
    const int tiles = p.batch * p.num_m_tiles * p.num_n_tiles;
    return c < tiles ? (tiles - c + nc - 1) / nc : 0;
}
// half: -1 for a whole tile, else which 128-column half
__device__ __forceinline__ void pair_unit_coords(int u, const KParams& p, int c, int nc, int& b, int& mt, int& nt,
                                                 int& half) {
    int t;
    if (!p.split_tail || u < p.full_rounds) {
        t = c + u * nc;
        half = -1;
    } else {
        t = p.full_rounds * nc + (c >> 1);
        half = c & 1;
    }
    tile_coords(t, p, b, mt, nt);
}

// Work of one 1-SM CTA.  Without split-K: tiles blockIdx.x, + gridDim.x, ...
// over all of K.  With split-K (p.split_k = S > 1, clusters of S CTAs, grid
// = tiles x S): the one tile blockIdx.x / S, K stages [s num_kb / S,
// (s + 1) num_kb / S) for cluster rank s.
struct Sm1Work {
    int first, step, kb0, kb1;
};
__device__ __forceinline__ Sm1Work sm1_work(const KParams& p, int num_tiles) {
    if (p.split_k > 1) {
        const int s = static_cast<int>(blockIdx.x) % p.split_k;
        return {static_cast<int>(blockIdx.x) / p.split_k, num_tiles, s * p.num_kb / p.split_k,
                (s + 1) * p.num_kb / p.split_k};
    }
    return {static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), 0, p.num_kb};
}

// Split-K partial tile in shared memory: 128 rows of 1024 bytes (256 f32);
// the 16-byte chunk j of row r sits in slot j ^ (r & 7), so 8 consecutive
// rows writing the same chunk, or one row's 8 consecutive chunks, hit 8
// different 16-byte bank groups.
__device__ __forceinline__ uint32_t partial_off(int r, int j) {
    return static_cast<uint32_t>(r) * 1024u + (static_cast<uint32_t>(j ^ (r & 7)) << 4);
}
constexpr int kMaxSplitK = 8;  // CTAs per split-K cluster (the portable cluster size)

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// One 256-bit store: every write is a whole 32-byte sector.  C is not read
// again by the kernel, so it goes to L2 marked evict-first and leaves the
// operand panels in place: 4-8 % faster at K = 512-1024 (where C is a large
// share of the traffic), no change at K >= 2048.
__device__ __forceinline__ void st_v8(void* dst, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                      uint32_t a5, uint32_t a6, uint32_t a7) {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(dst), "r"(a0),
                 "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7), "l"(pol)
                 : "memory");
}

// Store one accumulator row segment of problem b: row m, columns [n0, n0 + 128).
__device__ __forceinline__ void store_row128(const KParams& p, int b, int64_t m, int64_t n0,
                                             const uint32_t (&v)[4][32]) {
    if (m >= p.M || n0 >= p.N) return;
    const int64_t row = static_cast<int64_t>(b) * p.c_batch_stride + m * p.ldc + n0;
    if (p.out_bf16) {
        uint16_t* crow = reinterpret_cast<uint16_t*>(p.c) + row;
        if (p.vec_store && n0 + 128 <= p.N && (reinterpret_cast<uintptr_t>(crow) & 31u) == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint32_t* x = &v[j][16 * q];
                    st_v8(crow + 32 * j + 16 * q,
                          pack_bf16x2(__uint_as_float(x[0]), __uint_as_float(x[1])),
                          pack_bf16x2(__uint_as_float(x[2]), __uint_as_float(x[3])),
                          pack_bf16x2(__uint_as_float(x[4]), __uint_as_float(x[5])),
                          pack_bf16x2(__uint_as_float(x[6]), __uint_as_float(x[7])),
                          pack_bf16x2(__uint_as_float(x[8]), __uint_as_float(x[9])),
                          pack_bf16x2(__uint_as_float(x[10]), __uint_as_float(x[11])),
                          pack_bf16x2(__uint_as_float(x[12]), __uint_as_float(x[13])),
                          pack_bf16x2(__uint_as_float(x[14]), __uint_as_float(x[15])));
                }
        } else if (p.vec_store && n0 + 128 <= p.N) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(v[j][8 * q + 0]), __uint_as_float(v[j][8 * q + 1]));
                    w.y = pack_bf16x2(__uint_as_float(v[j][8 * q + 2]), __uint_as_float(v[j][8 * q + 3]));
                    w.z = pack_bf16x2(__uint_as_float(v[j][8 * q + 4]), __uint_as_float(v[j][8 * q + 5]));
                    w.w = pack_bf16x2(__uint_as_float(v[j][8 * q + 6]), __uint_as_float(v[j][8 * q + 7]));
                    *reinterpret_cast<uint4*>(crow + 32 * j + 8 * q) = w;
                }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (n0 + 32 * j + i < p.N)
                        crow[32 * j + i] =
                            static_cast<uint16_t>(pack_bf16x2(__uint_as_float(v[j][i]), 0.0f) & 0xFFFFu);
        }
    } else {
        float* crow = reinterpret_cast<float*>(p.c) + row;
        if (p.vec_store && n0 + 128 <= p.N && (reinterpret_cast<uintptr_t>(crow) & 31u) == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t* x = &v[j][8 * q];
                    st_v8(crow + 32 * j + 8 * q, x[0], x[1], x[2], x[3], x[4], x[5], x[6], x[7]);
                }
        } else if (p.vec_store && n0 + 128 <= p.N) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<uint4*>(crow + 32 * j + 4 * q) =
                        make_uint4(v[j][4 * q], v[j][4 * q + 1], v[j][4 * q + 2], v[j][4 * q + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (n0 + 32 * j + i < p.N) crow[32 * j + i] = __uint_as_float(v[j][i]);
        }
    }
}

// Columns [n, n + 8 x 32-bit words) of row m of problem b: 16 bf16 columns
// (w = packed pairs) or 8 f32 columns; columns past N are skipped.
__device__ __forceinline__ void store_row_chunk(const KParams& p, int b, int64_t m, int64_t n, const uint32_t (&w)[8]) {
    if (m >= p.M || n >= p.N) return;
    const int64_t row = static_cast<int64_t>(b) * p.c_batch_stride + m * p.ldc + n;
    const int cols = p.out_bf16 ? 16 : 8;
    void* dst = p.out_bf16 ? static_cast<void*>(reinterpret_cast<uint16_t*>(p.c) + row)
                           : static_cast<void*>(reinterpret_cast<float*>(p.c) + row);
    if (p.vec_store && n + cols <= p.N) {
        if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
            st_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
        } else {
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
    } else if (p.out_bf16) {
        uint16_t* c = static_cast<uint16_t*>(dst);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (n + i < p.N) c[i] = static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1)));
    } else {
        float* c = static_cast<float*>(dst);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (n + i < p.N) c[i] = __uint_as_float(w[i]);
    }
}

// Wait (lane 0, bounded) until the MMA thread has issued `target` K stages in
// all, counting from the kernel's start (a 32-bit count that may wrap).
__device__ __forceinline__ void wait_mma_progress(const volatile uint32_t* issued, uint32_t target,
                                                  volatile int* abort_flag, uint64_t limit_ns) {
    if (static_cast<int32_t>(*issued - target) >= 0) return;
    const uint64_t t0 = globaltimer_ns();
    while (static_cast<int32_t>(*issued - target) < 0) {
        if (*abort_flag || globaltimer_ns() - t0 > limit_ns) return;
        __nanosleep(128);
    }
}

// Store C[m, n .. n + 3] of problem b (columns past N skipped).
__device__ __forceinline__ void store_chunk4(const KParams& p, int b, int64_t m, int64_t n, float4 x) {
    const int64_t row = static_cast<int64_t>(b) * p.c_batch_stride + m * p.ldc + n;
    const float e[4] = {x.x, x.y, x.z, x.w};
    if (p.out_bf16) {
        uint16_t* c = reinterpret_cast<uint16_t*>(p.c) + row;
        if (p.vec_store && n + 4 <= p.N) {
            *reinterpret_cast<uint2*>(c) = make_uint2(pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]));
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (n + i < p.N) c[i] = static_cast<uint16_t>(pack_bf16x2(e[i], 0.0f) & 0xFFFFu);
        }
    } else {
        float* c = reinterpret_cast<float*>(p.c) + row;
        if (p.vec_store && n + 4 <= p.N) {
            *reinterpret_cast<float4*>(c) = x;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (n + i < p.N) c[i] = e[i];
        }
    }
}

// ============================================ fused activation quantize

// One quantize item: 128 rows (a 128-row panel of A, the rows of one
// scale-factor tile) x kQChunk elements of X along K, done by the 256 threads
// of the 8 epilogue warps.  Items are numbered in the order the tiles consume
// them: tile group by tile group (two panels per pair M-tile of the group),
// inside a group K chunk by K chunk, panel by panel; CTA c takes items c,
// c + gridDim.x, ...
constexpr int kQChunk = 256;  // K elements per item: 2 FP8 stages, 1 FP4 stage
// K stages of the current tile that must remain for the epilogue to start
// an item of a later tile group (an item takes about 8 us, a K stage about
// 0.33 us).
constexpr int kQOneStages = 24;

struct QItem {
    int group, panel, kc;
};
// Items of the first tile group.
__device__ __forceinline__ int first_group_items(const KParams& p) {
    return min(2 * min(p.first_group_m, p.num_m_tiles), p.q_panels) * p.q_nkc;
}

__device__ __forceinline__ QItem q_item(const KParams& p, int i) {
    QItem it;
    const int fp = min(2 * min(p.first_group_m, p.num_m_tiles), p.q_panels);  // panels of group 0
    if (i < fp * p.q_nkc) {
        it.group = 0;
        it.kc = i / fp;
        it.panel = i - it.kc * fp;
        return it;
    }
    i -= fp * p.q_nkc;
    const int per_group = 2 * p.group_m * p.q_nkc;
    const int g = i / per_group;
    const int j = i - g * per_group;
    const int first_panel = fp + g * 2 * p.group_m;
    const int gp = min(2 * p.group_m, p.q_panels - first_panel);
    it.group = g + 1;
    it.kc = j / gp;
    it.panel = first_panel + (j - it.kc * gp);
    return it;
}

// QuantizeMX of item i, 1x32 blocks along K, EMAX (the arithmetic of the
// standalone quantizer, qdev::).  Only the six epilogue warps that do not
// share a warp scheduler with the MMA-issuing thread (warp 1) do the work:
// warps 5 and 9 would take issue slots from it, and the MMA issue rate is
// what bounds the GEMM (with all eight warps quantizing, the fused launch
// measured 3 % slower).  Their 96 lane pairs take the item's 1024 row blocks
// (128 rows x 8 blocks of 32) in two batches, a lane pair per block (16
// elements a lane, one xor shuffle for the block maximum), consecutive pairs
// along a row so a warp reads 1 KB of two rows per load; all of a batch's
// loads are issued before any is used.  Codes go to q_xq, scales to their
// SF-layout bytes; scale columns past K inside the last scale tile are
// written as zero (E8M0 0, so the zero codes the tensor core reads there
// contribute exactly 0).  All eight warps then meet, and one thread
// publishes the item's ready word (release at GPU scope after the barrier,
// which orders every thread's stores before it).
constexpr int kQBlocks = 128 * (kQChunk / 32);      // row blocks of an item
constexpr int kQBatch = 6;                          // blocks a lane pair loads before using any
constexpr int kQEpiWarps = 6;                       // epilogue warps that quantize between tiles

__device__ __forceinline__ int q_warp_slot(int warp) {
    // epilogue warps 2..9; warps 5 and 9 (warp % 4 == 1, warp 1's scheduler) sit out
    return (warp & 3) == 1 ? -1 : (warp < 5 ? warp - 2 : warp - 3);
}

// The item's work for the lane pairs of NW warps (this warp's `slot` in
// 0 .. NW-1; -1 = none); the caller then synchronises its threads and
// publishes.
template <bool F16, int QFMT, int NW>
__device__ __forceinline__ void quant_item_body(const KParams& p, const QItem& it, int slot, int lane) {
    using namespace qdev;
    constexpr int kQPairs = NW * 16;
    constexpr int kQPerPair = (kQBlocks + kQPairs - 1) / kQPairs;
    if (slot >= 0) {
        const int pair = slot * 16 + (lane >> 1);
        const int half = lane & 1;
#pragma unroll
        for (int j0 = 0; j0 < kQPerPair; j0 += kQBatch) {
            uint32_t v[kQBatch][8];
            int64_t row[kQBatch], k0[kQBatch];
            bool live[kQBatch], kin[kQBatch];
#pragma unroll
            for (int jj = 0; jj < kQBatch; ++jj) {
                const int u = pair + kQPairs * (j0 + jj);
                live[jj] = j0 + jj < kQPerPair && u < kQBlocks;
                row[jj] = static_cast<int64_t>(it.panel) * 128 + (u >> 3);
                k0[jj] = static_cast<int64_t>(it.kc) * kQChunk + (u & 7) * 32 + half * 16;
                kin[jj] = k0[jj] < p.K;
                live[jj] = live[jj] && row[jj] < p.M;
                if (live[jj] && kin[jj]) {
                    ld_stream_v8(p.q_x + row[jj] * p.q_ld_x + k0[jj] * 2, v[jj]);
                } else {
#pragma unroll
                    for (int w = 0; w < 8; ++w) v[jj][w] = 0;
                }
            }
#pragma unroll
            for (int jj = 0; jj < kQBatch; ++jj) {
                // the block: maximum, E8M0, prescale, and whether it holds Inf/NaN
                uint32_t m = vmax_u16x2(vmax_u16x2(vmax_u16x2(mag2(v[jj][0]), mag2(v[jj][1])),
                                                   vmax_u16x2(mag2(v[jj][2]), mag2(v[jj][3]))),
                                        vmax_u16x2(vmax_u16x2(mag2(v[jj][4]), mag2(v[jj][5])),
                                                   vmax_u16x2(mag2(v[jj][6]), mag2(v[jj][7]))));
                m = hmax(m);
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
                const uint32_t x = exp_byte_of_mag<F16>(m);
                const bool special = x == 255u;
                const uint32_t e = e8m0_of(x, p.q_emax);
                const float sc = prescale_mul(e);
                if (!live[jj]) continue;
                if (kin[jj]) {
                    uint32_t w[4];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t hw[4] = {v[jj][4 * h], v[jj][4 * h + 1], v[jj][4 * h + 2], v[jj][4 * h + 3]};
                        // e2m1: the tensor cores' order, element 2i in the low nibble
                        quantize8<F16, QFMT>(hw, sc, sc, special, 1, 0x3210u, w[2 * h], w[2 * h + 1]);
                    }
                    if constexpr (QFMT == kE2M1) {
                        *reinterpret_cast<uint2*>(p.q_xq + row[jj] * (p.K / 2) + k0[jj] / 2) = make_uint2(w[0], w[2]);
                    } else {
                        *reinterpret_cast<uint4*>(p.q_xq + row[jj] * p.K + k0[jj]) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                const int64_t kb32 = k0[jj] >> 5;
                if (half == 0 && kb32 < 4 * static_cast<int64_t>(p.sf_ntk)) {
                    const int64_t r = row[jj];
                    const int64_t tile = (r >> 7) * p.sf_ntk + (kb32 >> 2);
                    p.q_sf[tile * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb32 & 3)] =
                        static_cast<uint8_t>(kin[jj] ? e : 0u);
                }
            }
        }
    }
}

// One thread publishes an item once every thread that wrote it has passed a
// barrier with it (release at GPU scope after the barrier, which orders
// every thread's stores before it).
__device__ __forceinline__ void publish_item(const KParams& p, const QItem& it) {
    if (p.q_no_publish) return;
    // the TMA loads that wait on this word read through the async proxy
    fence_proxy_async_global();
    st_release_gpu_u64(p.q_flags + static_cast<int64_t>(it.panel) * p.q_nkc + it.kc, p.q_tag);
}

// Item i by the epilogue warps (bf16 or f16 input): the six that do not
// share warp 1's scheduler work, all eight meet on the epilogue barrier.
template <int QFMT>
__device__ __forceinline__ void quant_item_any(const KParams& p, int i, int warp, int lane, int tid) {
    if constexpr (QFMT >= 0) {
        const QItem it = q_item(p, i);
        if (p.q_f16) quant_item_body<true, QFMT, kQEpiWarps>(p, it, q_warp_slot(warp), lane);
        else quant_item_body<false, QFMT, kQEpiWarps>(p, it, q_warp_slot(warp), lane);
        named_bar_sync(kEpiBarrier, NUM_EPI_WARPS * 32);
        if (tid == 0) publish_item(p, it);
    }
}

// Item i by all warps of the CTA, before the roles start (the kernel's
// prologue: nothing else runs yet, and the first tiles wait for these).
template <int QFMT, int NW>
__device__ __forceinline__ void quant_item_all(const KParams& p, int i, int warp, int lane) {
    if constexpr (QFMT >= 0) {
        const QItem it = q_item(p, i);
        if (p.q_f16) quant_item_body<true, QFMT, NW>(p, it, warp, lane);
        else quant_item_body<false, QFMT, NW>(p, it, warp, lane);
        __syncthreads();
        if (threadIdx.x == 0) publish_item(p, it);
    }
}

// Ready words.  An item's writer stores the launch's tag (40 bits, nonzero,
// different for every call); a word of an earlier launch never holds it, and
// a word of fresh memory only by a 2^-40 chance.  At its end every CTA counts
// itself on the done word that follows the ready words, and the last one sets
// all of them back to zero (end_of_launch), so a replay of the same launch
// (same tag) waits for its own items again.
//
// Bounded wait (one thread) for items kc0 .. kc1 - 1 (at most 4) of 128-row
// panel `panel`: the words are loaded together (one round trip), then any not
// yet written are polled.  Afterwards the thread's later TMA loads are
// ordered after the items' stores.  Gives up like mbar_wait_bounded
// (MX_ERR_TIMEOUT, abort flag).
constexpr int kMaxItemsPerWait = 4;
constexpr int kReadyBitsMax = 4096;  // 128-row panels the producer's shared-memory bitmap covers
__device__ __forceinline__ bool wait_items_ready(const KParams& p, int panel, int kc0, int kc1,
                                                 volatile int* abort_flag) {
    const uint64_t* w = p.q_flags + static_cast<int64_t>(panel) * p.q_nkc + kc0;
    const int n = kc1 - kc0;
    uint64_t v[kMaxItemsPerWait];
#pragma unroll
    for (int i = 0; i < kMaxItemsPerWait; ++i) v[i] = i < n ? ld_acquire_gpu_u64(w + i) : p.q_tag;
#pragma unroll
    for (int i = 0; i < kMaxItemsPerWait; ++i) {
        if (v[i] == p.q_tag) continue;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            __nanosleep(64);
            if (ld_acquire_gpu_u64(w + i) == p.q_tag) break;
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                atomicCAS(&g_mx_status, 0, 9);
                *abort_flag = 1;
                return false;
            }
        }
    }
    fence_proxy_async_global();
    return true;
}

// The ready-word warp (fused only): walk this CTA's work units in order
// and, for each unit's panel, poll all of its ready words together (a lane
// per word) until every item carries this launch's tag, then raise the
// panel's bit in `ready_bits` (release, CTA scope).  The TMA-issuing thread
// skips its own waits for a panel whose bit it reads as set (acquire), so in
// steady state no global ready word is read on the loads' critical path
// (polled by the issuing thread itself, the words cost 12 % of the fused
// call; polled by the producer warp's idle lanes, which share the issuing
// lane's warp, 25 %).  The warp only ever speeds the loads up: it stops
// (without an error) on the abort flag or after timeout_ns on one panel, and
// the issuing thread then waits itself.
__device__ __forceinline__ void ready_helper(const KParams& p, uint32_t bits_saddr, int num_units, int cluster,
                                             int num_clusters, uint32_t rank, int lane, volatile int* abort_flag) {
    const uint32_t mask = 0xFFFFFFFFu;
    for (int u = 0; u < num_units; ++u) {
        int b, mt, nt, hf;
        pair_unit_coords(u, p, cluster, num_clusters, b, mt, nt, hf);
        const int panel = 2 * mt + static_cast<int>(rank);
        if (panel >= p.q_panels || panel >= kReadyBitsMax) continue;
        const uint32_t word = bits_saddr + 4u * static_cast<uint32_t>(panel >> 5);
        if ((ld_acquire_cta_shared_u32(word) >> (panel & 31)) & 1u) continue;
        const uint64_t* w = p.q_flags + static_cast<int64_t>(panel) * p.q_nkc;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            // relaxed polls; the acquire fence below once all are seen
            bool mine = true;
            for (int kc = lane; kc < p.q_nkc; kc += 32) mine &= ld_relaxed_gpu_u64(w + kc) == p.q_tag;
            if (__all_sync(mask, mine)) break;
            // every lane leaves together (a lane left alone in __all_sync would wait forever)
            if (__any_sync(mask, *abort_flag != 0 || globaltimer_ns() - t0 > p.timeout_ns)) return;
            __nanosleep(1000);
        }
        fence_acq_rel_gpu();
        __syncwarp(mask);
        if (lane == 0) red_release_cta_shared_or(word, 1u << (panel & 31));
        __syncwarp(mask);
    }
}

// One thread per CTA, after every role of the CTA has finished: count this
// CTA on the done word ((tag << 24) | CTAs counted).  A plain add counts it
// when the word already carries this launch's tag (every CTA but the first
// to arrive); an add that finds another tag (a cleared word, or fresh
// memory) changed nothing that counts, and the CTA then installs the tag
// with a count of 1 by compare-and-swap, or adds again once another CTA has.
// Returns true for the last CTA of the launch, which then clears the ready
// words and the done word.
__device__ __forceinline__ bool end_of_launch_is_last(const KParams& p) {
    unsigned long long* d =
        reinterpret_cast<unsigned long long*>(p.q_flags + static_cast<int64_t>(p.q_panels) * p.q_nkc);
    __threadfence();
    unsigned long long now = atomicAdd(d, 1ull) + 1ull;
    while ((now >> 24) != p.q_tag) {
        const unsigned long long cur = atomicAdd(d, 0ull);
        if ((cur >> 24) == p.q_tag) {
            now = atomicAdd(d, 1ull) + 1ull;
        } else if (atomicCAS(d, cur, (p.q_tag << 24) | 1ull) == cur) {
            now = (p.q_tag << 24) | 1ull;
        }
    }
    __threadfence();
    return static_cast<unsigned>(now & 0xFFFFFFull) == gridDim.x;
}

// ====================================================== 1-SM, 128 x 256 tiles

namespace sm1 {
constexpr int BM = 128, BN = 256;
constexpr int STAGES = 4;
constexpr uint32_t A_STAGE = BM * BK;   // 16 KB
constexpr uint32_t B_STAGE = BN * BK;   // 32 KB
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE;
constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_STAGE;
// scale tiles per stage: one 512-byte tile per 128 rows per 128 K elements
// (FP8 stages span 128 K elements, FP4 stages 256)
__host__ __device__ constexpr uint32_t sfa_stage(bool fp4) { return fp4 ? 1024u : 512u; }
__host__ __device__ constexpr uint32_t sfb_stage(bool fp4) { return 2 * sfa_stage(fp4); }
__host__ __device__ constexpr uint32_t off_sfb(bool fp4) { return OFF_SFA + STAGES * sfa_stage(fp4); }
__host__ __device__ constexpr uint32_t off_bar(bool fp4) { return off_sfb(fp4) + STAGES * sfb_stage(fp4); }
constexpr int NUM_BARS = 3 * STAGES + 4;  // full, empty, sf_full [S]; tmem_full, tmem_empty, mma_done, sf_done
__host__ __device__ constexpr uint32_t off_misc(bool fp4) { return off_bar(fp4) + NUM_BARS * 8; }
__host__ __device__ constexpr uint32_t smem_alloc(bool fp4) { return off_misc(fp4) + 16 + 1024; }  // slack to align the base
constexpr int SF_WARP = 10;              // warp that copies scale factors to tensor memory
constexpr int THREADS = NUM_THREADS + 32;
}  // namespace sm1

// MN: operands read as MN-major tiles (bit 0: B, bit 1: A; FP8 only).  An
// MN-major B stage is two 128-row atom columns 16 KB apart (two TMA boxes);
// its B stages then come first in shared memory, so that every address its
// descriptors can name stays inside the CTA's allocation.
template <bool FP4, int MN = 0>
__global__ void __launch_bounds__(sm1::THREADS, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const KParams p) {
    using namespace sm1;
    constexpr bool a_mn = (MN & 2) != 0, b_mn = (MN & 1) != 0;
    constexpr uint32_t S_OFF_A = b_mn ? STAGES * B_STAGE : OFF_A;  // operand stages
    constexpr uint32_t S_OFF_B = b_mn ? 0u : OFF_B;
    constexpr uint32_t OFF_PARTIAL = 0;  // split-K partials reuse the drained operand stages
    constexpr uint32_t SFA_STAGE = sfa_stage(FP4), SFB_STAGE = sfb_stage(FP4);
    constexpr uint32_t OFF_SFB = off_sfb(FP4), OFF_BAR = off_bar(FP4), OFF_MISC = off_misc(FP4);
    constexpr uint32_t SF_COLS = sf_cols(FP4);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    auto full_bar = [&](int s) { return sb + OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + OFF_BAR + 8u * (STAGES + s); };
    auto sf_full_bar = [&](int s) { return sb + OFF_BAR + 8u * (2 * STAGES + s); };
    const uint32_t tmem_full = sb + OFF_BAR + 8u * (3 * STAGES);
    const uint32_t tmem_empty = tmem_full + 8;
    const uint32_t mma_done = tmem_full + 16;
    const uint32_t sf_done = tmem_full + 24;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

    pdl_allow_next();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(sf_full_bar(s), 1);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, NUM_EPI_WARPS);
        mbar_init(mma_done, 1);
        mbar_init(sf_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int num_tiles = p.batch * p.num_m_tiles * p.num_n_tiles;
    const Sm1Work work = sm1_work(p, num_tiles);
    pdl_wait_prior();  // set-up done; operands, scales and C belong to earlier kernels until here

    if (warp == 0) {
        if (lane == 0 && !p.skip_producer) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = work.first; t < num_tiles && ok; t += work.step) {
                int b, mt, nt;
                tile_coords(t, p, b, mt, nt);
                const int nsf0 = 2 * nt;
                const int nsf1 = (2 * nt + 1 < p.num_sf_n_tiles) ? 2 * nt + 1 : 2 * nt;
                const uint8_t* sfa = p.sfa + static_cast<size_t>(b) * p.sfa_batch_tiles * 512u;
                const uint8_t* sfb = p.sfb + static_cast<size_t>(b) * p.sfb_batch_tiles * 512u;
                for (int kb = work.kb0; kb < work.kb1; ++kb) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns, &g_mx_status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(stage);
                    // first scale tile of the stage along K; an FP4 stage takes
                    // two unless K ends inside it
                    const int t0 = FP4 ? 2 * kb : kb;
                    const uint32_t sf_bytes = (FP4 && t0 + 1 < p.sf_ntk) ? 1024u : 512u;
                    mbar_arrive_expect_tx(fb, A_STAGE + B_STAGE + 3u * sf_bytes);
                    // K-major tiles: (K bytes, rows); MN-major: (rows, K rows)
                    if constexpr (a_mn)
                        tma_load_3d(sb + S_OFF_A + stage * A_STAGE, &tmap_a, fb, mt * BM, kb * BK, b);
                    else
                        tma_load_3d(sb + S_OFF_A + stage * A_STAGE, &tmap_a, fb, kb * BK, mt * BM, b);
                    if constexpr (b_mn) {
                        tma_load_3d(sb + S_OFF_B + stage * B_STAGE, &tmap_b, fb, nt * BN, kb * BK, b);
                        tma_load_3d(sb + S_OFF_B + stage * B_STAGE + B_STAGE / 2, &tmap_b, fb, nt * BN + 128, kb * BK,
                                    b);
                    } else {
                        tma_load_3d(sb + S_OFF_B + stage * B_STAGE, &tmap_b, fb, kb * BK, nt * BN, b);
                    }
                    bulk_load(sb + OFF_SFA + stage * SFA_STAGE,
                              sfa + (static_cast<size_t>(mt) * p.sf_ntk + t0) * 512u, sf_bytes, fb);
                    bulk_load(sb + OFF_SFB + stage * SFB_STAGE,
                              sfb + (static_cast<size_t>(nsf0) * p.sf_ntk + t0) * 512u, sf_bytes, fb);
                    bulk_load(sb + OFF_SFB + stage * SFB_STAGE + SFB_STAGE / 2,
                              sfb + (static_cast<size_t>(nsf1) * p.sf_ntk + t0) * 512u, sf_bytes, fb);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Wait (bounded) until the loads of the last STAGES issued stages
            // have landed, so no copy is in flight when the CTA exits.  A stage
            // the MMA warp already consumed reads as complete at once.
            for (int i = 0; i < STAGES; ++i) {
                if (--stage < 0) {
                    stage = STAGES - 1;
                    phase ^= 1u;
                }
                volatile int no_abort = 0;
                (void)mbar_wait_bounded(full_bar(stage), phase, &no_abort, 100000000ull, &g_mx_status);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = work.first; t < num_tiles && ok; t += work.step) {
                if (!mbar_wait_bounded(tmem_empty, acc_phase ^ 1u, abort_flag, p.timeout_ns, &g_mx_status)) break;
                tc_fence_after();
                for (int kb = work.kb0; kb < work.kb1; ++kb) {
                    const bool first_kb = kb == work.kb0;
                    if (!mbar_wait_bounded(sf_full_bar(stage), phase, abort_flag, p.timeout_ns, &g_mx_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf_t = tmem_base + TMEM_SF + SF_COLS * stage;
                    const uint32_t sa = sb + S_OFF_A + stage * A_STAGE;
                    const uint32_t sbb = sb + S_OFF_B + stage * B_STAGE;
                    if constexpr (FP4) {
                        // 4 MMAs of K = 64; K group g = kk / 2 has its own scale
                        // columns, bytes {0,1} / {2,3} of them by scale data ID
                        const int kk_end = (kb * 256 + 128 < p.K) ? 4 : 2;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            if (kk >= kk_end) break;
                            const uint32_t id = 2u * static_cast<uint32_t>(kk & 1);
                            tc_mma_mxf4(tmem_base, sdesc_kmajor_sw128(sa + kk * 32),
                                        sdesc_kmajor_sw128(sbb + kk * 32), p.idesc | (id << 4) | (id << 29),
                                        sf_t + 4u * (kk >> 1), sf_t + 8u + 8u * (kk >> 1), !first_kb || kk != 0);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BK / 32; ++kk) {
                            const uint32_t idesc = p.idesc | (static_cast<uint32_t>(kk) << 4) |
                                                   (static_cast<uint32_t>(kk) << 29);
                            // 32 K elements: 32 bytes into a K-major row, 32
                            // rows of 128 bytes into an MN-major atom column
                            const uint64_t da = a_mn ? sdesc_mnmajor_sw128(sa + kk * 32 * 128)
                                                     : sdesc_kmajor_sw128(sa + kk * 32);
                            const uint64_t db = b_mn ? sdesc_mnmajor_sw128(sbb + kk * 32 * 128, B_STAGE / 2)
                                                     : sdesc_kmajor_sw128(sbb + kk * 32);
                            tc_mma_mxf8(tmem_base, da, db, idesc, sf_t, sf_t + 4u, !first_kb || kk != 0);
                        }
                    }
                    tc_commit(empty_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(tmem_full);
                acc_phase ^= 1u;
            }
            // Everything this thread issued must finish before tensor memory is freed.
            tc_commit(mma_done);
            volatile int no_abort = 0;
            (void)mbar_wait_bounded(mma_done, 0, &no_abort, 100000000ull, &g_mx_status);
        }
    } else if (warp == SF_WARP) {
        // scale-factor copies for each stage, off the MMA thread
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = work.first; t < num_tiles && ok; t += work.step) {
                for (int kb = work.kb0; kb < work.kb1; ++kb) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns, &g_mx_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf_t = tmem_base + TMEM_SF + SF_COLS * stage;
                    const uint32_t s_sfa = sb + OFF_SFA + stage * SFA_STAGE;
                    const uint32_t s_sfb = sb + OFF_SFB + stage * SFB_STAGE;
                    if constexpr (FP4) {
                        // A: K groups at +0, +4; B: K group g at +8 + 8g (rows
                        // 0-127, then 128-255 four columns on)
                        tc_cp_32x128b_warpx4(sf_t, sdesc_sf_tile(s_sfa));
                        tc_cp_32x128b_warpx4(sf_t + 4u, sdesc_sf_tile(s_sfa + 512u));
                        tc_cp_32x128b_warpx4(sf_t + 8u, sdesc_sf_tile(s_sfb));
                        tc_cp_32x128b_warpx4(sf_t + 12u, sdesc_sf_tile(s_sfb + 1024u));
                        tc_cp_32x128b_warpx4(sf_t + 16u, sdesc_sf_tile(s_sfb + 512u));
                        tc_cp_32x128b_warpx4(sf_t + 20u, sdesc_sf_tile(s_sfb + 1536u));
                    } else {
                        tc_cp_32x128b_warpx4(sf_t, sdesc_sf_tile(s_sfa));
                        tc_cp_32x128b_warpx4(sf_t + 4u, sdesc_sf_tile(s_sfb));
                        tc_cp_32x128b_warpx4(sf_t + 8u, sdesc_sf_tile(s_sfb + 512u));
                    }
                    tc_commit(sf_full_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            tc_commit(sf_done);
            volatile int no_abort = 0;
            (void)mbar_wait_bounded(sf_done, 0, &no_abort, 100000000ull, &g_mx_status);
        }
    } else {
        const int quarter = warp & 3;          // TMEM lanes this warp may access
        const int half = (warp - 2) >> 2;      // accumulator columns [128*half, +128)
        uint32_t acc_phase = 0;
        for (int t = work.first; t < num_tiles; t += work.step) {
            int b, mt, nt;
            tile_coords(t, p, b, mt, nt);
            // one lane waits; the warp follows its verdict so it never diverges
            bool ok = true;
            if (lane == 0) ok = mbar_wait_bounded(tmem_full, acc_phase, abort_flag, p.timeout_ns, &g_mx_status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int row = quarter * 32 + lane;
            const int64_t m = static_cast<int64_t>(mt) * BM + row;
            const int64_t n0 = static_cast<int64_t>(nt) * BN + half * 128;
            // a warp whose 32 rows or 128 columns all lie outside C stores nothing
            // (it still loads: skipping the load costs registers)
            const bool live = static_cast<int64_t>(mt) * BM + quarter * 32 < p.M && n0 < p.N;
            uint32_t v[4][32];
            {
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + half * 128;
                tmem_ld_32x32b_x128(taddr, v);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tmem_empty);
            acc_phase ^= 1u;
            if (!live) continue;
            if (p.split_k > 1) {
                // this slice's partial sums go into the drained operand stages
                // for the cluster to reduce
                fence_proxy_async_smem();
                if (m < p.M) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const uint32_t* x = &v[c >> 3][4 * (c & 7)];
                        st_shared_v4(sb + OFF_PARTIAL + partial_off(row, half * 32 + c), x[0], x[1], x[2], x[3]);
                    }
                }
            } else {
                store_row128(p, b, m, n0, v);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (p.split_k > 1) {
        // Split-K reduction: each CTA of the cluster takes a share of the
        // tile's 4-column chunks, sums the S partials in slice order (so the
        // result does not depend on timing) and stores C.
        cluster_sync_all();  // all partials written and visible cluster-wide
        const int S = p.split_k;
        const int s = static_cast<int>(cluster_ctarank());
        int b, mt, nt;
        tile_coords(work.first, p, b, mt, nt);
        const int rows = min(BM, p.M - mt * BM);
        const int chunks = (min(BN, p.N - nt * BN) + 3) / 4;  // per row
        const int total = rows * chunks;
        const int e_end = (s + 1) * total / S;
        for (int e = s * total / S + static_cast<int>(threadIdx.x); e < e_end; e += blockDim.x) {
            const int r = e / chunks, j = e - r * chunks;
            const float4* own = reinterpret_cast<const float4*>(generic_shared(sb + OFF_PARTIAL + partial_off(r, j)));
            float4 acc = *map_cluster(own, 0);
            // CTA q's partial, through the cluster window, 4 loads in flight
#pragma unroll
            for (int q0 = 1; q0 < kMaxSplitK; q0 += 4) {
                float4 x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (q0 + i < S) x[i] = *map_cluster(own, q0 + i);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (q0 + i < S) {
                        acc.x += x[i].x;
                        acc.y += x[i].y;
                        acc.z += x[i].z;
                        acc.w += x[i].w;
                    }
                }
            }
            store_chunk4(p, b, static_cast<int64_t>(mt) * BM + r, static_cast<int64_t>(nt) * BN + 4 * j, acc);
        }
        cluster_sync_all();  // no CTA leaves while another may still read its partial
    }
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ================================================ 2-SM pair, 256 x 256 tiles

namespace sm2 {
constexpr int BM = 256, BN = 256;        // pair tile; each CTA holds 128 rows of A and of B
constexpr int STAGES = 6;
constexpr uint32_t A_STAGE = 128 * BK;   // 16 KB
constexpr uint32_t B_STAGE = 128 * BK;   // 16 KB
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE;
constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_STAGE;
// Scale tiles travel in groups of sf_group() stages.  FP8: one TMA load per
// scale tensor per 8 stages, on a group barrier of its own, 2 groups in
// flight (per-stage loads of 512-byte tiles measured 2.6 % slower at 8192^3,
// and counting a group's bytes on its first stage's barrier 1.3 % slower).
// FP4: one stage per group, the scales riding with each stage's operands in
// the stage's own slot (grouping measured 6 % slower there).  A group holds
// this CTA's 128 rows of A and all 256 rows of B (both CTAs need them).
__host__ __device__ constexpr int sf_group(bool fp4) { return fp4 ? 1 : 8; }
__host__ __device__ constexpr int sf_slots(bool fp4) { return fp4 ? STAGES : 2; }
__host__ __device__ constexpr uint32_t sfa_stage(bool fp4) { return fp4 ? 1024u : 512u; }
__host__ __device__ constexpr uint32_t sfa_group(bool fp4) { return sf_group(fp4) * sfa_stage(fp4); }
__host__ __device__ constexpr uint32_t off_sfb(bool fp4) { return OFF_SFA + sf_slots(fp4) * sfa_group(fp4); }
__host__ __device__ constexpr uint32_t off_bar(bool fp4) { return off_sfb(fp4) + sf_slots(fp4) * 2 * sfa_group(fp4); }
// full, empty, sf_full [S]; tmem_full, tmem_empty, mma_done, sf_done; group full, empty [slots]
__host__ __device__ constexpr int num_bars(bool fp4) { return 3 * STAGES + 4 + 2 * sf_slots(fp4); }
__host__ __device__ constexpr uint32_t off_misc(bool fp4) { return off_bar(fp4) + num_bars(fp4) * 8; }
// misc: tensor-memory address, abort flag, MMA progress (16 bytes), then the
// fused producer's bitmap of panels seen ready (kReadyBitsMax bits)
__host__ __device__ constexpr uint32_t smem_alloc(bool fp4) { return off_misc(fp4) + 16 + kReadyBitsMax / 8 + 1024; }
constexpr uint32_t PAIR_TX = 2 * (A_STAGE + B_STAGE);  // both CTAs' operand tiles of a stage
__host__ __device__ constexpr uint32_t pair_sf_tx(bool fp4) { return 2 * 3 * sfa_group(fp4); }
constexpr int SF_WARP = 10;              // warp that copies scale factors to tensor memory
constexpr int READY_WARP = 11;           // fused only: polls the activation's ready words
constexpr int THREADS = NUM_THREADS + 32;
constexpr int THREADS_FUSED = THREADS + 32;
__host__ __device__ constexpr int threads(bool fused) { return fused ? THREADS_FUSED : THREADS; }
// Rank 0's C stores are paced over the first kPaceNum / kPaceDen of the next
// tile's K stages, when a tile has at least kPaceMinStages of them (A/B at
// 8192 x 8192, CUDA events: FP8 K = 8192 / 2048 +0.9 / +4.5 %, MXFP4 +2 %;
// spreading over the whole next tile was slower at K = 1024, where unpaced
// stores are kept).
constexpr int kPaceNum = 1, kPaceDen = 2, kPaceMinStages = 16;
}  // namespace sm2

// Scale-factor buffers are read by TMA as [2 * tiles, 256] bytes: a 512-byte
// tile t is rows 2t and 2t+1; one box is a scale group's consecutive tiles;
// tiles past the end read as zeros.  MN: which operands this instantiation
// reads as MN-major tiles (bit 0: B, bit 1: A; 0 = both K-major), fixed at
// compile time: the MMA-issuing thread is on the critical path, and a
// runtime test of the operands' layout per MMA cost 2 % at 8192^3.
template <bool FP4, int QFMT, int MN = 0>
__global__ void __launch_bounds__(sm2::threads(QFMT >= 0), 1)
    mx_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                       const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                       const KParams p) {
    using namespace sm2;
    constexpr uint32_t SFA_STAGE = sfa_stage(FP4), SFA_GROUP = sfa_group(FP4);
    constexpr uint32_t OFF_SFB = off_sfb(FP4), OFF_BAR = off_bar(FP4), OFF_MISC = off_misc(FP4);
    constexpr uint32_t SF_COLS = sf_cols(FP4);
    constexpr uint32_t PAIR_SF_TX = pair_sf_tx(FP4);
    constexpr int SF_TILES_PER_STAGE = FP4 ? 2 : 1;
    constexpr int SF_GROUP = sf_group(FP4), SF_SLOTS = sf_slots(FP4);
    constexpr bool FUSED = QFMT >= 0;  // quantize X into the A operand inside this launch
    constexpr bool a_mn = (MN & 2) != 0, b_mn = (MN & 1) != 0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;

    auto full_bar = [&](int s) { return sb + OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + OFF_BAR + 8u * (STAGES + s); };
    auto sf_full_bar = [&](int s) { return sb + OFF_BAR + 8u * (2 * STAGES + s); };
    const uint32_t tmem_full = sb + OFF_BAR + 8u * (3 * STAGES);
    const uint32_t tmem_empty = tmem_full + 8;
    const uint32_t mma_done = tmem_full + 16;
    const uint32_t sf_done = tmem_full + 24;
    auto sfg_full_bar = [&](int g) { return sb + OFF_BAR + 8u * (3 * STAGES + 4 + g); };
    auto sfg_empty_bar = [&](int g) { return sb + OFF_BAR + 8u * (3 * STAGES + 4 + SF_SLOTS + g); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    volatile uint32_t* mma_issued = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC + 8);  // K stages so far

    pdl_allow_next();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);     // rank 0's: its arrive + both CTAs' bytes
            mbar_init(empty_bar(s), 1);    // one multicast commit per use
            mbar_init(sf_full_bar(s), 1);  // rank 0's: the scale copies of the stage are done
        }
        for (int g = 0; g < SF_SLOTS; ++g) {
            mbar_init(sfg_full_bar(g), 1);   // rank 0's: its arrive + both CTAs' scale bytes
            mbar_init(sfg_empty_bar(g), 1);  // one multicast commit per use
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, NUM_EPI_WARPS + 1);  // rank 0's: its epilogue warps + one for rank 1's
        mbar_init(mma_done, 1);
        mbar_init(sf_done, 1);
        *abort_flag = 0;
        *mma_issued = 0;
        if constexpr (FUSED)
            for (int i = 0; i < kReadyBitsMax / 32; ++i) reinterpret_cast<uint32_t*>(smem + OFF_MISC + 16)[i] = 0;
        fence_mbar_init();
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        prefetch_tmap(&tmap_sfa);
        prefetch_tmap(&tmap_sfb);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int num_units = pair_units(p, cluster, num_clusters);
    pdl_wait_prior();  // set-up done; operands, scales and C belong to earlier kernels until here

    // fused: bitmap of panels whose items are all written (zeroed at set-up)
    const uint32_t ready_bits = sb + OFF_MISC + 16;
    // fused prologue: every warp quantizes this CTA's items of the first
    // tile group, which the first wave of tiles needs at once (with the
    // epilogue warps alone the first tiles ended 17 us later)
    int q_first = static_cast<int>(blockIdx.x);
    if constexpr (FUSED) {
        const int n0 = first_group_items(p);
        for (; q_first < n0; q_first += static_cast<int>(gridDim.x))
            quant_item_all<QFMT, THREADS_FUSED / 32>(p, q_first, warp, lane);
    }
    if (warp == 0) {
        if (lane == 0 && !p.skip_producer) {
            int stage = 0, gslot = 0;
            uint32_t phase = 0, gphase = 0;
            bool ok = true;
            for (int u = 0; u < num_units && ok; ++u) {
                int b, mt, nt, hf;
                pair_unit_coords(u, p, cluster, num_clusters, b, mt, nt, hf);
                const int a_row = mt * BM + static_cast<int>(rank) * 128;
                // a half tile's 128 B rows split 64 / 64 over the pair (the
                // 128-row box brings 64 rows more, which no MMA reads)
                const int b_row = hf < 0 ? nt * BN + static_cast<int>(rank) * 128
                                         : nt * BN + hf * 128 + static_cast<int>(rank) * 64;
                // scale tiles past this problem's last one belong to rows past
                // M / N (the next problem's tiles, or zeros past the buffer):
                // their products land in rows the epilogue never stores
                const int64_t sfa_tile = b * p.sfa_batch_tiles + (2 * mt + static_cast<int>(rank)) * p.sf_ntk;
                const int64_t sfb_tile0 = b * p.sfb_batch_tiles + (2 * nt + (hf < 0 ? 0 : hf)) * p.sf_ntk;
                const int64_t sfb_tile1 = hf < 0 ? sfb_tile0 + p.sf_ntk : sfb_tile0;
                // fused: this unit's panel of A must be quantized before its
                // loads.  Decided once per unit, before the unit's first
                // wait for a free stage: the panel's bit (raised by the
                // ready-word warp) says all its items are written; otherwise
                // each scale group waits for its own items (FP8: 8 stages =
                // 4 items; FP4: 1 stage = 1 item), also before that group's
                // wait for a free stage, off the path from a freed stage to
                // its next loads.
                const int panel = 2 * mt + static_cast<int>(rank);
                bool panel_ready = true;
                if constexpr (FUSED) {
                    panel_ready = panel >= p.q_panels;
                    if (!panel_ready && panel < kReadyBitsMax &&
                        ((ld_acquire_cta_shared_u32(ready_bits + 4u * (panel >> 5)) >> (panel & 31)) & 1u)) {
                        fence_proxy_async_global();
                        panel_ready = true;
                    }
                }
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    const bool group_start = kb % SF_GROUP == 0;
                    if (FUSED && !panel_ready && group_start) {
                        // the bit may have been raised since the unit began
                        if (panel < kReadyBitsMax &&
                            ((ld_acquire_cta_shared_u32(ready_bits + 4u * (panel >> 5)) >> (panel & 31)) & 1u)) {
                            fence_proxy_async_global();
                            panel_ready = true;
                        } else {
                            const int kc0 = FP4 ? kb : kb / 2;
                            const int kc1 = min(kc0 + (FP4 ? 1 : SF_GROUP / 2), p.q_nkc);
                            if (!wait_items_ready(p, panel, kc0, kc1, abort_flag)) {
                                ok = false;
                                break;
                            }
                        }
                    }
                    // a scale slot is free once its last group's copies into
                    // tensor memory have completed (for one-stage groups the
                    // stage's empty barrier already says so)
                    if (group_start && SF_GROUP > 1 &&
                        !mbar_wait_bounded(sfg_empty_bar(gslot), gphase ^ 1u, abort_flag, p.timeout_ns,
                                           &g_mx_status)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns, &g_mx_status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = mapa_shared(full_bar(stage), 0);
                    constexpr bool own_bar = SF_GROUP > 1;  // group bytes on a barrier of their own
                    if (rank == 0) {
                        mbar_arrive_expect_tx(full_bar(stage), PAIR_TX + (group_start && !own_bar ? PAIR_SF_TX : 0u));
                        if (group_start && own_bar) mbar_arrive_expect_tx(sfg_full_bar(gslot), PAIR_SF_TX);
                    }
                    if (group_start) {
                        // the scale tiles of stages kb .. kb + SF_GROUP - 1, one
                        // load per scale tensor; tiles past K (or past the
                        // buffer) feed no MMA
                        const uint32_t gb = own_bar ? mapa_shared(sfg_full_bar(gslot), 0) : fb;
                        const int64_t t0 = static_cast<int64_t>(SF_TILES_PER_STAGE) * kb;
                        const uint32_t sa_g = sb + OFF_SFA + gslot * SFA_GROUP;
                        const uint32_t sb_g = sb + OFF_SFB + gslot * 2 * SFA_GROUP;
                        tma_load_2d_pair(sa_g, &tmap_sfa, gb, 0, static_cast<int>(2 * (sfa_tile + t0)));
                        tma_load_2d_pair(sb_g, &tmap_sfb, gb, 0, static_cast<int>(2 * (sfb_tile0 + t0)));
                        tma_load_2d_pair(sb_g + SFA_GROUP, &tmap_sfb, gb, 0, static_cast<int>(2 * (sfb_tile1 + t0)));
                        if (++gslot == SF_SLOTS) {
                            gslot = 0;
                            gphase ^= 1u;
                        }
                    }
                    // K-major tiles: (K bytes, rows); MN-major: (rows, K rows)
                    if constexpr (a_mn)
                        tma_load_3d_pair(sb + OFF_A + stage * A_STAGE, &tmap_a, fb, a_row, kb * BK, b);
                    else
                        tma_load_3d_pair(sb + OFF_A + stage * A_STAGE, &tmap_a, fb, kb * BK, a_row, b);
                    if constexpr (b_mn)
                        tma_load_3d_pair(sb + OFF_B + stage * B_STAGE, &tmap_b, fb, b_row, kb * BK, b);
                    else
                        tma_load_3d_pair(sb + OFF_B + stage * B_STAGE, &tmap_b, fb, kb * BK, b_row, b);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (rank == 0) {
                // rank 0's full and group barriers count both CTAs' bytes: once
                // the last STAGES fills and SF_SLOTS groups have completed, no
                // copy of the pair is in flight
                for (int i = 0; i < STAGES; ++i) {
                    if (--stage < 0) {
                        stage = STAGES - 1;
                        phase ^= 1u;
                    }
                    volatile int no_abort = 0;
                    (void)mbar_wait_bounded(full_bar(stage), phase, &no_abort, 100000000ull, &g_mx_status);
                }
                for (int i = 0; SF_GROUP > 1 && i < SF_SLOTS; ++i) {
                    if (--gslot < 0) {
                        gslot = SF_SLOTS - 1;
                        gphase ^= 1u;
                    }
                    volatile int no_abort = 0;
                    (void)mbar_wait_bounded(sfg_full_bar(gslot), gphase, &no_abort, 100000000ull, &g_mx_status);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0, issued = 0;
            bool ok = true;
            for (int u = 0; u < num_units && ok; ++u) {
                const bool half_tile = p.split_tail && u >= p.full_rounds;
                const uint32_t unit_idesc = half_tile ? p.idesc_half : p.idesc;
                if (!mbar_wait_bounded(tmem_empty, acc_phase ^ 1u, abort_flag, p.timeout_ns, &g_mx_status)) break;
                tc_fence_after();
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    // the scale-copy warp has seen the stage's operands land
                    // and its copies into tensor memory have completed
                    if (!mbar_wait_bounded(sf_full_bar(stage), phase, abort_flag, p.timeout_ns, &g_mx_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf_t = tmem_base + TMEM_SF + SF_COLS * stage;
                    const uint32_t sa = sb + OFF_A + stage * A_STAGE;
                    const uint32_t sbb = sb + OFF_B + stage * B_STAGE;
                    if constexpr (FP4) {
                        const int kk_end = (kb * 256 + 128 < p.K) ? 4 : 2;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            if (kk >= kk_end) break;
                            const uint32_t id = 2u * static_cast<uint32_t>(kk & 1);
                            tc_mma_mxf4_pair(tmem_base, sdesc_kmajor_sw128(sa + kk * 32),
                                             sdesc_kmajor_sw128(sbb + kk * 32), unit_idesc | (id << 4) | (id << 29),
                                             sf_t + 4u * (kk >> 1), sf_t + 8u + 8u * (kk >> 1), (kb | kk) != 0);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BK / 32; ++kk) {
                            const uint32_t idesc = unit_idesc | (static_cast<uint32_t>(kk) << 4) |
                                                   (static_cast<uint32_t>(kk) << 29);
                            // 32 K elements: 32 bytes into a K-major row, 32
                            // rows of 128 bytes into an MN-major tile
                            const uint64_t da = a_mn ? sdesc_mnmajor_sw128(sa + kk * 32 * 128)
                                                     : sdesc_kmajor_sw128(sa + kk * 32);
                            const uint64_t db = b_mn ? sdesc_mnmajor_sw128(sbb + kk * 32 * 128)
                                                     : sdesc_kmajor_sw128(sbb + kk * 32);
                            tc_mma_mxf8_pair(tmem_base, da, db, idesc, sf_t, sf_t + 4u, (kb | kk) != 0);
                        }
                    }
                    tc_commit_pair_mc(empty_bar(stage), 3);
                    *mma_issued = ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_mc(tmem_full, 3);
                acc_phase ^= 1u;
            }
            tc_commit_pair_mc(mma_done, 3);
            volatile int no_abort = 0;
            (void)mbar_wait_bounded(mma_done, 0, &no_abort, 100000000ull, &g_mx_status);
        }
    } else if (warp == READY_WARP) {
        if constexpr (FUSED) {
            if (!p.skip_producer)
                ready_helper(p, ready_bits, num_units, cluster, num_clusters, rank, lane, abort_flag);
        }
    } else if (warp == SF_WARP) {
        // Scale-factor copies, one K block at a time, off the MMA thread: a
        // tcgen05.cp costs the issuing thread as much as the four MMAs of a
        // K block, so the MMA thread only waits for this warp's commit.  A
        // scale group is released (multicast commit) after its last stage.
        if (lane == 0 && rank == 0) {
            int stage = 0, gslot = 0;
            uint32_t phase = 0, gphase = 0;
            bool ok = true;
            for (int u = 0; u < num_units && ok; ++u) {
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    const int j = kb % SF_GROUP;
                    // a group's scales: on their own barrier, or (one-stage
                    // groups) with the stage's operands
                    if (SF_GROUP > 1 && j == 0 &&
                        !mbar_wait_bounded(sfg_full_bar(gslot), gphase, abort_flag, p.timeout_ns, &g_mx_status)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns, &g_mx_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf_t = tmem_base + TMEM_SF + SF_COLS * stage;
                    // stage j of the group: A at j * SFA_STAGE; B rows 0-127 and
                    // 128-255 in the group's two B row tiles
                    const uint32_t s_sfa = sb + OFF_SFA + gslot * SFA_GROUP + j * SFA_STAGE;
                    const uint32_t s_sfb0 = sb + OFF_SFB + gslot * 2 * SFA_GROUP + j * SFA_STAGE;
                    const uint32_t s_sfb1 = s_sfb0 + SFA_GROUP;
                    if constexpr (FP4) {
                        // K group g of the stage is scale tile g of each
                        tc_cp_pair_32x128b_warpx4(sf_t, sdesc_sf_tile(s_sfa));
                        tc_cp_pair_32x128b_warpx4(sf_t + 4u, sdesc_sf_tile(s_sfa + 512u));
                        tc_cp_pair_32x128b_warpx4(sf_t + 8u, sdesc_sf_tile(s_sfb0));
                        tc_cp_pair_32x128b_warpx4(sf_t + 12u, sdesc_sf_tile(s_sfb1));
                        tc_cp_pair_32x128b_warpx4(sf_t + 16u, sdesc_sf_tile(s_sfb0 + 512u));
                        tc_cp_pair_32x128b_warpx4(sf_t + 20u, sdesc_sf_tile(s_sfb1 + 512u));
                    } else {
                        tc_cp_pair_32x128b_warpx4(sf_t, sdesc_sf_tile(s_sfa));
                        tc_cp_pair_32x128b_warpx4(sf_t + 4u, sdesc_sf_tile(s_sfb0));
                        tc_cp_pair_32x128b_warpx4(sf_t + 8u, sdesc_sf_tile(s_sfb1));
                    }
                    tc_commit_pair_mc(sf_full_bar(stage), 1);
                    if (j == SF_GROUP - 1 || kb == p.num_kb - 1) {
                        if (SF_GROUP > 1) tc_commit_pair_mc(sfg_empty_bar(gslot), 3);  // both CTAs' producers
                        if (++gslot == SF_SLOTS) {
                            gslot = 0;
                            gphase ^= 1u;
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            tc_commit_pair_mc(sf_done, 1);
            volatile int no_abort = 0;
            (void)mbar_wait_bounded(sf_done, 0, &no_abort, 100000000ull, &g_mx_status);
        }
    } else {
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t tmem_empty_rank0 = mapa_shared(tmem_empty, 0);
        const int epi_tid = threadIdx.x - 64;  // 0 .. 255
        // the MMA thread's issued-stage count (rank 0's), read through the cluster window
        const uint32_t issued_rank0 = mapa_shared(smem_u32(const_cast<uint32_t*>(mma_issued)), 0);
        // fused: this CTA's next quantize item (after the prologue's) and the item count
        int q_next = q_first;
        const int q_total = FUSED ? p.q_panels * p.q_nkc : 0;
        uint32_t acc_phase = 0;
        for (int u = 0; u < num_units; ++u) {
            int b, mt, nt, hf;
            pair_unit_coords(u, p, cluster, num_clusters, b, mt, nt, hf);
            if constexpr (FUSED) {
                // Until the accumulator is ready, quantize items of X.  One
                // thread decides for all eight warps (they meet on named
                // barriers inside an item).  Items of this tile's group (or
                // an earlier one) go at once: tiles running now may wait for
                // them.  Items of later groups (up to q_lookahead ahead)
                // start only while at least kQOneStages of this tile's K
                // stages remain to be issued (the MMA thread's count), so
                // that they end before the accumulator does: an item still
                // running when the accumulator is ready holds up the next
                // tile.  Otherwise the warps wait for the accumulator.
                const int cur_group = m_tile_group(p, mt);
                const int G = static_cast<int>(gridDim.x);
                const uint32_t tile_end = static_cast<uint32_t>(u + 1) * static_cast<uint32_t>(p.num_kb);
                for (;;) {
                    bool go = false;
                    if (epi_tid == 0 && q_next < q_total && !*abort_flag && !mbar_test(tmem_full, acc_phase)) {
                        const int g = q_item(p, q_next).group;
                        go = g <= cur_group ||
                             (g <= cur_group + p.q_lookahead &&
                              static_cast<int>(tile_end - ld_shared_cluster_u32(issued_rank0)) >= kQOneStages);
                    }
                    if (!named_bar_or(kEpiBarrier, NUM_EPI_WARPS * 32, go)) break;
                    quant_item_any<QFMT>(p, q_next, warp, lane, epi_tid);
                    q_next += G;
                }
            }
            bool ok = true;
            if (lane == 0) ok = mbar_wait_bounded(tmem_full, acc_phase, abort_flag, p.timeout_ns, &g_mx_status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            // rank 1's warps (and, fused, every CTA's) meet on named
            // barriers: they leave the loop together or not at all
            if (rank == 1 || FUSED) ok = named_bar_and(kEpiBarrier, NUM_EPI_WARPS * 32, ok);
            if (!ok) break;
            tc_fence_after();
            // a half tile's accumulator is columns 0..127: the second half's
            // warps only release
            const bool live = hf < 0 || half == 0;
            uint32_t v[4][32];
            {
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + half * 128;
                tmem_ld_32x32b_x128(taddr, v);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            // Release the accumulator: rank 0's warps arrive locally; rank 1's
            // meet on a named barrier and one thread arrives across the
            // cluster, relaxed (eight remote release-arrives cost about 0.4 us
            // more per tile: 5 % at 8192^3, 15 % at K = 2048).
            if (rank == 0) {
                if (lane == 0) mbar_arrive(tmem_empty);
            } else {
                named_bar_sync(kEpiBarrier, NUM_EPI_WARPS * 32);
                if (warp == 2 && lane == 0) mbar_arrive_cluster_relaxed(tmem_empty_rank0);
            }
            acc_phase ^= 1u;
            if (!live) continue;
            // Rank 0 (the CTA that issues the MMAs and holds the pipeline's
            // barriers) stores its rows in 8 KB steps paced by the MMA
            // thread's progress through the next tile: C leaving that SM in
            // one 64 KB burst (from registers or through TMA stores alike)
            // held up the tensor core's completion signals the MMA thread
            // waits on (the next tile's first scale copies) by about 1.2 us
            // a tile, where the same bytes written to shared memory cost
            // nothing.  Rank 1's stores cost nothing measurable and go at once.
            const int64_t m = static_cast<int64_t>(mt) * BM + rank * 128 + quarter * 32 + lane;
            const int64_t n0 = static_cast<int64_t>(nt) * BN + (hf < 0 ? half : hf) * 128;
            // (fused: only once this CTA's items are all written, so the
            // wait never stands between a load and an item this CTA owes;
            // pacing as soon as the next tile's items were written measured
            // 0.8 % slower)
            const bool paced = rank == 0 && u + 1 < num_units && p.num_kb >= kPaceMinStages &&
                               (!FUSED || q_next >= q_total);
            const uint32_t next_tile = static_cast<uint32_t>(u + 1) * static_cast<uint32_t>(p.num_kb);
            auto pace = [&](int c, int chunks) {
                if (!paced) return;
                if (lane == 0)
                    wait_mma_progress(
                        mma_issued,
                        next_tile + static_cast<uint32_t>((c * p.num_kb * kPaceNum) / (chunks * kPaceDen)) + 1u,
                        abort_flag, p.timeout_ns);
                __syncwarp();
            };
            uint32_t w[8];
            if (p.out_bf16) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {  // 16 columns a step
                    const uint32_t* x = &v[c >> 1][16 * (c & 1)];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = pack_bf16x2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
                    pace(c, 8);
                    store_row_chunk(p, b, m, n0 + 16 * c, w);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 16; ++c) {  // 8 columns a step
                    const uint32_t* x = &v[c >> 2][8 * (c & 3)];
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[i] = x[i];
                    pace(c, 16);
                    store_row_chunk(p, b, m, n0 + 8 * c, w);
                }
            }
        }
        if constexpr (FUSED) {
            // items other CTAs' tiles still wait for (a CTA with no tiles
            // left, or none at all, still owes its share)
            const int G = static_cast<int>(gridDim.x);
            for (;;) {
                const bool stop = epi_tid == 0 && (q_next >= q_total || *abort_flag);
                if (named_bar_or(kEpiBarrier, NUM_EPI_WARPS * 32, stop)) break;
                quant_item_any<QFMT>(p, q_next, warp, lane, epi_tid);
                q_next += G;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA frees its memories while the pair may still use them
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    if constexpr (FUSED) {
        // the last CTA of the launch leaves the ready words zero
        volatile int* last = abort_flag + 2;  // the misc area's spare word
        if (threadIdx.x == 0) *last = end_of_launch_is_last(p) ? 1 : 0;
        __syncthreads();
        if (*last) {
            const int64_t n = static_cast<int64_t>(p.q_panels) * p.q_nkc + 1;
            for (int64_t i = threadIdx.x; i < n; i += blockDim.x) p.q_flags[i] = 0;
        }
    }
}

// ------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// K-major FP8 operands [batch, rows, k] (problem stride `batch_stride` bytes)
// as a 3-D tensor map with a (128 B x box_rows x 1) box, 128B swizzle.  Rows
// past `rows` read as zeros inside each problem.
bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k, uint32_t box_rows,
                      int64_t batch, int64_t batch_stride) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(batch_stride)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MN-major FP8 operands [batch, k, mn] (rows of `mn` bytes, one per K index;
// problem stride `batch_stride` bytes) with a (128 B x 128 K rows x 1) box,
// 128B swizzle: a K stage of 128 rows along MN.  `mn` must be a multiple of
// 16 (the row pitch of a tensor map).  Rows past K and columns past mn read
// as zeros inside each problem.
bool make_operand_map_mn(CUtensorMap* map, const void* base, int64_t mn, int64_t k, int64_t batch,
                         int64_t batch_stride) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(mn), static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(mn), static_cast<cuuint64_t>(batch_stride)};
    cuuint32_t box[3] = {128, static_cast<cuuint32_t>(BK), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A scale-factor buffer of `tiles` 512-byte tiles as [2 * tiles, 256] bytes.
// Tiles past the end read as zeros.  A box is `box_tiles` consecutive tiles
// (one scale group: SF_GROUP stages of 1 (FP8) or 2 (FP4) tiles).
bool make_sf_map(CUtensorMap* map, const void* base, int64_t tiles, uint32_t box_tiles) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {256, static_cast<cuuint64_t>(2 * tiles)};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {256, 2 * box_tiles};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

uint64_t g_timeout_ns = 2000000000ull;
int g_fault_skip_producer = 0;
// 0 automatic, 1 force the 1-SM kernel, 2 force the 2-SM kernel, 3 force the
// 1-SM kernel without split-K, 4 automatic but the fused call as two launches
int g_variant = 0;
GemmLaunchInfo g_last_launch{};

bool is_fp4(const GemmArgs& g) { return g.elem_fmt == kE2M1; }

// Bytes of one K-contiguous operand row.
int64_t row_bytes(const GemmArgs& g) { return is_fp4(g) ? g.K / 2 : g.K; }

KParams base_params(const GemmArgs& g, int bm, int bn) {
    const bool fp4 = is_fp4(g);
    const int64_t stage_k = fp4 ? 2 * BK : BK;  // elements per 128-byte stage row
    KParams p{};
    p.sfa = g.sfa;
    p.sfb = g.sfb;
    p.c = g.c;
    p.ldc = g.ldc;
    p.M = static_cast<int>(g.M);
    p.N = static_cast<int>(g.N);
    p.K = static_cast<int>(g.K);
    p.out_bf16 = g.out_bf16;
    p.vec_store = g.vec_store;
    p.num_m_tiles = static_cast<int>((g.M + bm - 1) / bm);
    p.num_n_tiles = static_cast<int>((g.N + bn - 1) / bn);
    p.num_kb = static_cast<int>((g.K + stage_k - 1) / stage_k);
    p.sf_ntk = static_cast<int>((g.K + 127) / 128);
    p.num_sf_n_tiles = static_cast<int>((g.N + 127) / 128);
    p.batch = static_cast<int>(g.batch);
    p.c_batch_stride = g.c_batch_stride;
    p.sfa_batch_tiles = ((g.M + 127) / 128) * static_cast<int64_t>(p.sf_ntk);
    p.sfb_batch_tiles = ((g.N + 127) / 128) * static_cast<int64_t>(p.sf_ntk);
    p.group_m = 16;
    p.first_group_m = 16;
    p.idesc = fp4 ? make_idesc_mxf4(bm, bn) : make_idesc_mxf8(g.elem_fmt, g.elem_fmt, bm, bn);
    p.timeout_ns = g_timeout_ns;
    p.skip_producer = g_fault_skip_producer & 1;
    return p;
}

constexpr int kMinStagesPerSlice = 4;  // K stages each split-K slice accumulates at least

// The kernels' dynamic shared memory exceeds the default limit: set the
// attribute before any launch or occupancy query, once per device (a
// function attribute belongs to the device it was set on).
template <typename Kernel>
cudaError_t ensure_smem_attr(Kernel kernel, uint32_t bytes, std::mutex& mu, bool (&done)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    return cudaSuccess;
}
template <bool FP4, int MN = 0>
cudaError_t ensure_1sm_attr() {
    static std::mutex mu;
    static bool done[64] = {};
    return ensure_smem_attr(mx_gemm_kernel<FP4, MN>, sm1::smem_alloc(FP4), mu, done);
}
template <bool FP4, int QFMT, int MN = 0>
cudaError_t ensure_2sm_attr() {
    static std::mutex mu;
    static bool done[64] = {};
    return ensure_smem_attr(mx_gemm_2sm_kernel<FP4, QFMT, MN>, sm2::smem_alloc(FP4), mu, done);
}

// attr: room for 2 (cluster shape, programmatic serialization)
void split_launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int tiles, int split, bool fp4,
                         cudaStream_t stream) {
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(static_cast<unsigned>(tiles * split), 1, 1);
    cfg->blockDim = dim3(sm1::THREADS, 1, 1);
    cfg->dynamicSmemBytes = sm1::smem_alloc(fp4);
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg->attrs = attr;
    cfg->numAttrs = 2;
}

// Co-resident clusters of `split` 1-SM GEMM CTAs on the current device (cached).
template <bool FP4>
int max_split_clusters(int split) {
    static std::mutex mu;
    static int cached[64][kMaxSplitK + 1] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (ensure_1sm_attr<FP4>() != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev][split] == 0) {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[2];
        split_launch_config(&cfg, attr, device_sm_count() / split, split, FP4, nullptr);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mx_gemm_kernel<FP4>, &cfg) != cudaSuccess) n = 0;
        cached[dev][split] = n > 0 ? n : -1;
    }
    return cached[dev][split] > 0 ? cached[dev][split] : 0;
}

// Split-K factor for `tiles` 128 x 256 tiles of `num_kb` K stages: the
// largest S <= 8 whose tiles x S CTAs run in one wave (all clusters resident
// at once) while every slice keeps at least kMinStagesPerSlice stages.
// Few-tile problems (small M) otherwise leave most SMs idle.
template <bool FP4>
int choose_split_k(int tiles, int num_kb) {
    const int sms = device_sm_count();
    for (int s = kMaxSplitK; s > 1; --s) {
        if (static_cast<int64_t>(tiles) * s > sms || num_kb < kMinStagesPerSlice * s) continue;
        if (max_split_clusters<FP4>(s) >= tiles) return s;
    }
    return 1;
}

template <bool FP4, int MN = 0>
cudaError_t launch_1sm(const GemmArgs& g, cudaStream_t stream, bool allow_split) {
    if ((g.a_mn_major ? 2 : 0) + (g.b_mn_major ? 1 : 0) != MN || (MN && FP4)) return cudaErrorInvalidValue;
    const cudaError_t attr_err = ensure_1sm_attr<FP4, MN>();
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap ma, mb;
    // MN-major maps load 128-row boxes: A's 128-row tile is one box, B's
    // 256-row tile two
    const bool map_a = g.a_mn_major ? make_operand_map_mn(&ma, g.a, g.M, g.K, g.batch, g.a_batch_stride)
                                    : make_operand_map(&ma, g.a, g.M, row_bytes(g), sm1::BM, g.batch, g.a_batch_stride);
    const bool map_b = g.b_mn_major ? make_operand_map_mn(&mb, g.bt, g.N, g.K, g.batch, g.b_batch_stride)
                                    : make_operand_map(&mb, g.bt, g.N, row_bytes(g), sm1::BN, g.batch, g.b_batch_stride);
    if (!map_a || !map_b) return cudaErrorInvalidValue;
    KParams p = base_params(g, sm1::BM, sm1::BN);
    p.a_mn = g.a_mn_major ? 1 : 0;
    p.b_mn = g.b_mn_major ? 1 : 0;
    p.idesc |= (p.a_mn ? kIdescAMnMajor : 0u) | (p.b_mn ? kIdescBMnMajor : 0u);
    const int tiles = p.batch * p.num_m_tiles * p.num_n_tiles;
    p.split_k = allow_split ? choose_split_k<FP4>(tiles, p.num_kb) : 1;
    g_last_launch = GemmLaunchInfo{1, p.split_k, p.a_mn, p.b_mn};
    if (p.split_k > 1) {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[2];
        split_launch_config(&cfg, attr, tiles, p.split_k, FP4, stream);
        return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<FP4, MN>, ma, mb, p);
    }
    const int sms = device_sm_count();
    const int grid = tiles < sms ? tiles : sms;
    return launch_pdl(mx_gemm_kernel<FP4, MN>, static_cast<unsigned>(grid), sm1::THREADS, sm1::smem_alloc(FP4),
                      stream, ma, mb, p);
}

// attr: room for 2 (cluster shape, programmatic serialization)
void pair_launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int clusters, bool fp4,
                        cudaStream_t stream, bool fused = false) {
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(2 * clusters, 1, 1);
    cfg->blockDim = dim3(sm2::threads(fused), 1, 1);
    cfg->dynamicSmemBytes = sm2::smem_alloc(fp4);
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg->attrs = attr;
    cfg->numAttrs = 2;
}

// Co-resident 2-CTA clusters of the pair kernel on the current device (cached).
template <bool FP4>
int max_pair_clusters() {
    static std::mutex mu;
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (ensure_2sm_attr<FP4, -1>() != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[2];
        pair_launch_config(&cfg, attr, device_sm_count() / 2, FP4, nullptr);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mx_gemm_2sm_kernel<FP4, -1>, &cfg) != cudaSuccess || n <= 0)
            n = device_sm_count() / 2;
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

// A launch tag (40 bits, nonzero): consecutive calls get different tags (a
// per-process counter), and memory never written by this library is
// unlikely to hold one (the counter starts at a mixed clock / address seed).
uint64_t next_tag() {
    static std::atomic<uint64_t> counter{[] {
        uint64_t z = static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count()) ^
                     (static_cast<uint64_t>(std::chrono::system_clock::now().time_since_epoch().count()) << 17) ^
                     reinterpret_cast<uintptr_t>(&g_timeout_ns);
        // splitmix64 finaliser
        z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
        z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
        return z ^ (z >> 31);
    }()};
    uint64_t e;
    do e = counter.fetch_add(1, std::memory_order_relaxed) & ((1ull << 40) - 1);
    while (e == 0);  // never the tag of zeroed memory
    return e;
}

int g_fused_lookahead = 1;

template <bool FP4, int QFMT, int MN = 0>
cudaError_t launch_2sm(const GemmArgs& g, cudaStream_t stream) {
    const cudaError_t attr_err = ensure_2sm_attr<FP4, QFMT, MN>();
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap ma, mb, msa, msb;
    const int64_t sfa_tiles = g.batch * ((g.M + 127) / 128) * ((g.K + 127) / 128);
    const int64_t sfb_tiles = g.batch * ((g.N + 127) / 128) * ((g.K + 127) / 128);
    if ((g.a_mn_major ? 2 : 0) + (g.b_mn_major ? 1 : 0) != MN || (MN && (FP4 || QFMT >= 0)))
        return cudaErrorInvalidValue;
    const bool map_a = g.a_mn_major ? make_operand_map_mn(&ma, g.a, g.M, g.K, g.batch, g.a_batch_stride)
                                    : make_operand_map(&ma, g.a, g.M, row_bytes(g), 128, g.batch, g.a_batch_stride);
    const bool map_b = g.b_mn_major ? make_operand_map_mn(&mb, g.bt, g.N, g.K, g.batch, g.b_batch_stride)
                                    : make_operand_map(&mb, g.bt, g.N, row_bytes(g), 128, g.batch, g.b_batch_stride);
    if (!map_a || !map_b || !make_sf_map(&msa, g.sfa, sfa_tiles, sm2::sf_group(FP4) * (FP4 ? 2 : 1)) ||
        !make_sf_map(&msb, g.sfb, sfb_tiles, sm2::sf_group(FP4) * (FP4 ? 2 : 1)))
        return cudaErrorInvalidValue;
    KParams p = base_params(g, sm2::BM, sm2::BN);
    const int tiles = p.batch * p.num_m_tiles * p.num_n_tiles;
    const int cap = max_pair_clusters<FP4>();
    // split the last round's tiles into 128-column halves when they fit in
    // half the clusters.  Measured against whole tiles: the same time at
    // 8192^3 (the launch's time follows its total work, not the last round's
    // length), 5 % less at 256 x 8192 x 8192; halves of K with the partials
    // added through a workspace measured the same as column halves.
    const int full_rounds = tiles / cap, tail = tiles - full_rounds * cap;
    p.split_tail = (tail > 0 && 2 * tail <= cap) ? 1 : 0;
    p.full_rounds = full_rounds;
    p.idesc_half = make_idesc_mxf8(g.elem_fmt, g.elem_fmt, sm2::BM, sm2::BN / 2);
    if (is_fp4(g)) p.idesc_half = make_idesc_mxf4(sm2::BM, sm2::BN / 2);
    p.a_mn = g.a_mn_major ? 1 : 0;
    p.b_mn = g.b_mn_major ? 1 : 0;
    const uint32_t major_bits = (p.a_mn ? kIdescAMnMajor : 0u) | (p.b_mn ? kIdescBMnMajor : 0u);
    p.idesc |= major_bits;
    p.idesc_half |= major_bits;
    const int clusters = p.split_tail ? (full_rounds > 0 ? cap : 2 * tail) : (tiles < cap ? tiles : cap);
    p.split_k = 1;
    if constexpr (QFMT >= 0) {
        p.q_x = g.x;
        p.q_ld_x = g.ld_x_bytes;
        p.q_xq = const_cast<uint8_t*>(g.a);
        p.q_sf = const_cast<uint8_t*>(g.sfa);
        p.q_flags = g.q_flags;
        p.q_tag = next_tag();
        p.q_f16 = g.x_f16;
        p.q_panels = static_cast<int>((g.M + 127) / 128);
        p.q_nkc = static_cast<int>((g.K + kQChunk - 1) / kQChunk);
        p.q_lookahead = g_fused_lookahead;
        // a small first tile group: the first wave of tiles then needs the
        // items of 8 panels of X, not 32, before it runs at full rate
        p.first_group_m = 4;
        p.q_emax = QFMT == kE4M3 ? 8 : QFMT == kE5M2 ? 15 : 2;
        p.q_no_publish = (g_fault_skip_producer & 2) ? 1 : 0;
        p.skip_producer = g_fault_skip_producer & 1;
    }
    g_last_launch = GemmLaunchInfo{QFMT >= 0 ? 3 : 2, 1, p.a_mn, p.b_mn};
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair_launch_config(&cfg, attr, clusters, FP4, stream, QFMT >= 0);
    return cudaLaunchKernelEx(&cfg, mx_gemm_2sm_kernel<FP4, QFMT, MN>, ma, mb, msa, msb, p);
}

}  // namespace

void set_gemm_fault_injection(int skip_producer, uint64_t timeout_ns) {
    g_fault_skip_producer = skip_producer;
    g_timeout_ns = timeout_ns ? timeout_ns : 2000000000ull;
}

void set_gemm_variant(int variant) { g_variant = variant; }

GemmLaunchInfo last_gemm_launch() { return g_last_launch; }

// Automatic kernel choice.  M <= 128: the 1-SM kernel.  Otherwise the pair
// kernel, unless its 256 x 256 tiles would fill at most a quarter of the
// clusters and the 1-SM kernel can split K over clusters of at least 2: such
// few-tile problems ran 1.3-2x faster on the 1-SM kernel with split-K than as
// the pair kernel's half tiles (e.g. 1024 x 1024 x 8192: 14.4 against 21.0
// us), while at about half the clusters the pair kernel was ahead again.
template <bool FP4>
bool prefer_pair(const GemmArgs& g) {
    if (g.M <= 128) return false;
    const int64_t pair_tiles = g.batch * ((g.M + 255) / 256) * ((g.N + 255) / 256);
    if (pair_tiles * 4 > max_pair_clusters<FP4>()) return true;
    const int64_t tiles_1sm = g.batch * ((g.M + sm1::BM - 1) / sm1::BM) * ((g.N + sm1::BN - 1) / sm1::BN);
    const int64_t stage_k = FP4 ? 2 * BK : BK;
    return choose_split_k<FP4>(static_cast<int>(tiles_1sm), static_cast<int>((g.K + stage_k - 1) / stage_k)) < 2;
}

bool scaled_matmul_takes_pair(const GemmArgs& g) {
    const bool fp4 = is_fp4(g);
    const bool automatic = g_variant == 0 || g_variant == 4;
    return g_variant == 2 || (automatic && (fp4 ? prefer_pair<true>(g) : prefer_pair<false>(g)));
}

cudaError_t launch_scaled_matmul(const GemmArgs& g, cudaStream_t stream) {
    const bool fp4 = is_fp4(g);
    const bool pair = scaled_matmul_takes_pair(g);
    const bool split = g_variant != 3;
    if (fp4) return pair ? launch_2sm<true, -1>(g, stream) : launch_1sm<true>(g, stream, split);
    // FP8 operands read MN-major (a dot operand stored [batch, K, rows]):
    // one instantiation of each kernel per combination
    switch ((g.a_mn_major ? 2 : 0) + (g.b_mn_major ? 1 : 0)) {
    case 1: return pair ? launch_2sm<false, -1, 1>(g, stream) : launch_1sm<false, 1>(g, stream, split);
    case 2: return pair ? launch_2sm<false, -1, 2>(g, stream) : launch_1sm<false, 2>(g, stream, split);
    case 3: return pair ? launch_2sm<false, -1, 3>(g, stream) : launch_1sm<false, 3>(g, stream, split);
    default: return pair ? launch_2sm<false, -1>(g, stream) : launch_1sm<false>(g, stream, split);
    }
}

// The fused call runs as one launch when the pair kernel takes the product
// and the launch is long: the single launch pays a fixed start-up (the first
// tiles wait for their panels of X, about 15-30 us) where two launches pay
// QuantizeMX at full bandwidth.  Measured (us, one launch / two launches):
// 4096 x 8192 x 8192 200 / 173, 8192^3 367 / 338, 8192 x 16384 x 8192
// 630 / 615; from about 32 pair tiles per cluster on the two are within the
// run-to-run spread.
constexpr int kFusedMinTilesPerCluster = 32;

bool fused_single_launch(const GemmArgs& g) {
    if (g_variant == 4 || g.batch != 1) return false;
    const bool x_ok = (reinterpret_cast<uintptr_t>(g.x) & 31u) == 0 && g.ld_x_bytes % 32 == 0 &&
                      (reinterpret_cast<uintptr_t>(g.a) & 15u) == 0 && (reinterpret_cast<uintptr_t>(g.q_flags) & 7u) == 0;
    if (!x_ok) return false;
    if (g_variant == 2) return true;
    if (g_variant == 1 || g_variant == 3) return false;
    const bool fp4 = is_fp4(g);
    if (!(fp4 ? prefer_pair<true>(g) : prefer_pair<false>(g))) return false;
    const int64_t pair_tiles = ((g.M + 255) / 256) * ((g.N + 255) / 256);
    const int clusters = fp4 ? max_pair_clusters<true>() : max_pair_clusters<false>();
    return pair_tiles >= static_cast<int64_t>(kFusedMinTilesPerCluster) * clusters;
}

cudaError_t launch_fused_matmul(const GemmArgs& g, cudaStream_t stream) {
    switch (g.elem_fmt) {
    case kE4M3: return launch_2sm<false, kE4M3>(g, stream);
    case kE5M2: return launch_2sm<false, kE5M2>(g, stream);
    default: return launch_2sm<true, kE2M1>(g, stream);
    }
}

cudaError_t read_and_clear_device_status(int* status) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_mx_status, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_mx_status, &zero, sizeof(int));
}

}  // namespace mx
