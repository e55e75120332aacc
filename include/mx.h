/*
 * mx.h -- libmx: OCP-MX microscaling on one GB300 GPU (sm_103a).
 *
 * Two operations, as the pages "MX-FP8 Microscaling Legalization" (sections 2-4,
 * the QuantizeMX and ScaledMatmul custom-call contracts) and "MX Microscaling:
 * Quantize, Block-Scaling and E8M0" (the numeric model) define them:
 *
 *   QuantizeMX    bf16/f16 tensor -> {FP8 e4m3fn/e5m2 or FP4 e2m1 data,
 *                 one E8M0 scale per 32-element block}, scale method EMAX.
 *   ScaledMatmul  block_scaled_dot(lhs, rhs, lhs_scale, rhs_scale) -> f32/bf16.
 *
 * Conventions for every call below:
 *   - Pointers named `in`, `out`, `a`, `bt`, `c`, `*_scale`, `workspace` are
 *     DEVICE pointers (memory of the current CUDA device).  The caller owns and
 *     allocates every buffer; the library allocates nothing.
 *   - 2-D tensors are row-major.  `ld_*` is the row pitch in elements of the
 *     tensor's own type.  Each call states its alignment needs; where a pointer
 *     only needs element alignment, 16-byte aligned rows select the faster
 *     vectorised kernels.
 *   - All calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Argument errors are returned synchronously and launch
 *     nothing.  Errors inside a kernel (a bounded wait that gave up) are
 *     recorded in a per-device status word, read by mx_get_device_status().
 *   - The current device must be compute capability 10.3 (sm_103a);
 *     otherwise calls return MX_ERR_DEVICE.
 *   - Calls are thread-safe with respect to each other; concurrent calls that
 *     write the same output buffer race, as any two kernels would.
 */
#ifndef MX_H_
#define MX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so C callers need no CUDA header. */
typedef struct CUstream_st* mx_stream;

typedef enum mx_status {
    MX_OK = 0,
    MX_ERR_INVALID_ARG = 1,       /* NULL pointer, negative size, unknown enum value, pitch < width */
    MX_ERR_UNSUPPORTED_DTYPE = 2, /* dtype combination outside the dispatch matrix */
    MX_ERR_BLOCK_SIZE = 3,        /* block_size other than 32 (0 selects 32) */
    MX_ERR_DIM = 4,               /* dim other than -1 / -2 (or 1 / 0 for a 2-D tensor); bad dot dimension numbers */
    MX_ERR_SHAPE = 5,             /* extents not divisible by the block / the x4 container */
    MX_ERR_ALIGNMENT = 6,         /* pointer or pitch not 16-byte aligned */
    MX_ERR_WORKSPACE = 7,         /* workspace missing or too small */
    MX_ERR_CUDA = 8,              /* a CUDA runtime call or launch failed */
    MX_ERR_TIMEOUT = 9,           /* a bounded device-side wait gave up (device status word) */
    MX_ERR_DEVICE = 10,           /* current device is not sm_103a */
    MX_ERR_SCALE_METHOD = 11      /* scale_method other than EMAX */
} mx_status;

typedef enum mx_dtype {
    MX_BF16 = 1,
    MX_F16 = 2,
    MX_F32 = 3,
    MX_E4M3FN = 4, /* OCP float8_e4m3fn: 1.4.3, bias 7, max 448, no Inf */
    MX_E5M2 = 5,   /* OCP float8_e5m2: 1.5.2, bias 15, max 57344 */
    MX_E2M1 = 6,   /* OCP float4_e2m1fn: 1.2.1, bias 1, max 6, finite only */
    MX_E8M0 = 7    /* OCP float8_e8m0fnu: 2^(E-127), 0xFF = NaN */
} mx_dtype;

/* Block geometry of QuantizeMX (32 elements per block either way). */
enum {
    MX_GEOM_8X4 = 0,  /* 8 along the `dim` axis x 4 along the other axis: the
                         page's 8-partition x 4-column block ("Block geometry",
                         scale [P//8, F//4]) */
    MX_GEOM_1X32 = 1  /* 32 consecutive elements along `dim` (HLO block_size
                         along dim, QuantizeMX backend_config) */
};

/* Scale tensor layout. */
enum {
    MX_SCALE_PLAIN = 0,        /* row-major [scale_rows, scale_cols] */
    MX_SCALE_INTERLEAVE32 = 1, /* scale row i stored at buffer row (i & 3) + 32 * (i >> 2)
                                  (page "MX Microscaling", section "E8M0 Scale-Tensor
                                  Layout"); buffer rows = 32 * ceil(scale_rows / 4);
                                  rows never addressed are not written */
    MX_SCALE_TC_SF = 2         /* the tensor-core scale-factor layout of mx_repack_scales,
                                  written directly (1x32 blocks along dim=-1 only); the
                                  buffer holds mx_sf_layout_bytes(rows, cols) bytes and its
                                  padding is written as 0.  No counterpart on the pages:
                                  it lets an activation feed mx_scaled_matmul with no
                                  repack */
};

enum { MX_SCALE_METHOD_EMAX = 0 };

/*
 * QuantizeMX configuration: the backend_config fields {dtype, dim,
 * block_size, scale_method} of the page "MX-FP8 Microscaling Legalization",
 * section 4.1, plus the layout choices of the numeric page.
 */
typedef struct mx_quant_cfg {
    int32_t geometry;          /* MX_GEOM_8X4 | MX_GEOM_1X32 */
    int32_t scale_layout;      /* MX_SCALE_PLAIN | MX_SCALE_INTERLEAVE32 | MX_SCALE_TC_SF */
    int32_t block_size;        /* must be 32; 0 selects the default 32 (section 2.2) */
    int32_t dim;               /* -1 (last) or -2 (second-to-last); 1 / 0 are folded to
                                  -1 / -2 for the 2-D view (section 2.3) */
    int32_t scale_method;      /* MX_SCALE_METHOD_EMAX only */
    int32_t fp4_lane_stride;   /* e2m1 packing: 0 (no lane permutation), 1, 2 or 4.
                                  The page's lane_remap reverses each window of
                                  2*stride nibbles.  Default 2. */
    int32_t fp4_nibble_parity; /* e2m1 packing: 0 puts even permuted indices in the
                                  high nibble (default), 1 the low nibble */
    int32_t emax_alt;          /* 0: E8M0 measured against EMAX (default);
                                  1: against EMAX-1 (the page's alternative mode) */
} mx_quant_cfg;

/* Fill `cfg` with the defaults: 8x4, plain scales, block 32, dim -2, EMAX,
 * FP4 stride 2 / parity 0, emax_alt 0.  Returns MX_ERR_INVALID_ARG on NULL. */
mx_status mx_quant_cfg_default(mx_quant_cfg* cfg);

/*
 * Sizes of QuantizeMX outputs for a [rows, cols] input.
 *   data_bytes   dense row-major data: rows*cols bytes (FP8, one byte per
 *                element; four consecutive bytes form the page's x4 U32
 *                container) or rows*cols/2 bytes (e2m1, two nibbles per byte).
 *   scale_rows   rows of the scale BUFFER (interleaved layout: 32*ceil(r/4);
 *                MX_SCALE_TC_SF: rows rounded up to 128).
 *   scale_cols   columns of the scale tensor (MX_SCALE_TC_SF: rounded up to 4).
 *   scale_bytes  scale_rows * scale_cols.
 * Scale tensor shape: the data shape with each axis divided by the block's
 * extent along it (8x4 dim=-2: [rows/8, cols/4]; 8x4 dim=-1: [rows/4, cols/8];
 * 1x32 dim=-1: [rows, cols/32]; 1x32 dim=-2: [rows/32, cols]).
 * Any output pointer may be NULL.  Same argument checks as mx_quantize.
 */
mx_status mx_quantize_sizes(mx_dtype in_dtype, mx_dtype out_dtype, int64_t rows, int64_t cols,
                            const mx_quant_cfg* cfg, size_t* data_bytes, int64_t* scale_rows,
                            int64_t* scale_cols, size_t* scale_bytes);

/*
 * QuantizeMX (page "MX Microscaling: Quantize, Block-Scaling and E8M0",
 * sections "Block-Scale Computation" and "Round-to-Grid"): for each 32-element
 * block, E8M0 = max(1, max(0, maxExp - EMAX)) where maxExp is the largest
 * binary32 exponent byte in the block (EMAX: e2m1 2, e4m3fn 8, e5m2 15); each
 * element is multiplied by 2^(127 - E8M0) in binary32 and rounded to nearest
 * (ties to even), saturating at the format maximum.  NaN inputs become
 * 0x7F|sign (FP8) or a signed zero nibble (e2m1); Inf saturates.
 *
 *   in         device, [rows, ld_in] bf16/f16, 2-byte aligned, ld_in >= cols
 *              (16-byte aligned rows with cols % 8 == 0 take the vectorised
 *              kernels; anything else a scalar kernel with the same results)
 *   in_dtype   MX_BF16 | MX_F16
 *   rows, cols logical extents (>= 0); cols % 4 == 0 (x4 container); rows and
 *              cols divisible by the block extents
 *   out_dtype  MX_E4M3FN | MX_E5M2 | MX_E2M1
 *   cfg        NULL selects the defaults of mx_quant_cfg_default
 *   out_data   device, data_bytes (see mx_quantize_sizes), dense, 2-byte aligned
 *   out_scale  device, scale_bytes; interleaved layout leaves unaddressed rows
 *              untouched
 * e2m1 with lane stride s > 1 also needs cols % (2*s) == 0.
 * Returns MX_OK after the launch (asynchronous) or an argument error.
 */
mx_status mx_quantize(const void* in, mx_dtype in_dtype, int64_t rows, int64_t cols, int64_t ld_in,
                      mx_dtype out_dtype, const mx_quant_cfg* cfg, void* out_data, void* out_scale,
                      mx_stream stream);

/*
 * QuantizeMX from HOST memory to HOST memory (no page counterpart: the
 * pipelined runtime around mx_quantize).  The rows are processed in chunks
 * through three device slots in `workspace`: chunk i+1 is copied in and
 * chunk i-1 copied out while chunk i is quantized on `stream` (the copies run
 * on two internal per-device streams; events order all three).  Results are
 * bit-identical to mx_quantize on the same data.
 *   in_host        host [rows, ld_in] bf16/f16; pinned (cudaHostAlloc /
 *                  cudaHostRegister) for the copies to overlap, pageable works
 *                  but serialises
 *   out_data_host, out_scale_host  host buffers of mx_quantize_sizes; in the
 *                  interleaved layout rows the layout never addresses are left
 *                  untouched
 *   chunk_rows     rows per chunk, a multiple of the block's row extent x 1
 *                  (plain scales), x 4 (interleaved) or x 128 (SF layout);
 *                  0 selects about 16 MiB of input per chunk
 *   workspace      device, 256-byte aligned, mx_quantize_host_workspace bytes
 * Other arguments and errors as mx_quantize; MX_ERR_SHAPE for a chunk_rows
 * that is not such a multiple.  Asynchronous: `stream` waits for the last copy
 * out; the host buffers must stay valid until then.
 */
mx_status mx_quantize_host_workspace(mx_dtype in_dtype, int64_t rows, int64_t cols, mx_dtype out_dtype,
                                     const mx_quant_cfg* cfg, int64_t chunk_rows, size_t* bytes);
mx_status mx_quantize_host(const void* in_host, mx_dtype in_dtype, int64_t rows, int64_t cols, int64_t ld_in,
                           mx_dtype out_dtype, const mx_quant_cfg* cfg, void* out_data_host, void* out_scale_host,
                           int64_t chunk_rows, void* workspace, size_t workspace_bytes, mx_stream stream);

/*
 * Several host-to-host QuantizeMX jobs in one pipeline: their chunks share the
 * slot ring, so one tensor's copies overlap the next one's (no drain between
 * tensors).  Each job is what mx_quantize_host takes (cfg by value).  All
 * jobs are checked before anything is enqueued; the workspace is
 * mx_quantize_host_batch_workspace bytes (the largest job's slots).
 * njobs <= 4096.  Results equal njobs separate mx_quantize_host calls.
 */
typedef struct mx_host_quant_job {
    const void* in_host;
    mx_dtype in_dtype;
    int64_t rows, cols, ld_in;
    mx_dtype out_dtype;
    mx_quant_cfg cfg;
    void* out_data_host;
    void* out_scale_host;
} mx_host_quant_job;

mx_status mx_quantize_host_batch_workspace(const mx_host_quant_job* jobs, int njobs, int64_t chunk_rows,
                                           size_t* bytes);
mx_status mx_quantize_host_batch(const mx_host_quant_job* jobs, int njobs, int64_t chunk_rows, void* workspace,
                                 size_t workspace_bytes, mx_stream stream);

/*
 * MX dequantize (page "MX Microscaling", quantizeDataApplyingMxScales NOTE:
 * the matmul side applies ldexpf(x, E8M0 - 127); "FP4 x4-Pack": the read-back
 * uses the same lane permutation): out[r,c] = decode(code) * 2^(E - 127).
 *   data       device codes as mx_quantize writes them (dense; 4-byte aligned)
 *   scale      device scale buffer in cfg's layout (plain / interleaved / SF)
 *   in_dtype   MX_E4M3FN | MX_E5M2 | MX_E2M1
 *   rows, cols, cfg   as for mx_quantize (geometry, dim, layout, FP4 stride
 *              and parity must match the ones that produced the data)
 *   out_dtype  MX_F32 (exact: every value is representable, E = 0xFF gives
 *              NaN, overflow gives Inf) | MX_BF16 (round to nearest even)
 *   out, ld_out  device [rows, ld_out], element aligned; caller owns every buffer
 * Errors (nothing launched): MX_ERR_SHAPE / MX_ERR_INVALID_ARG as for
 * mx_quantize, also ld_out < cols or a null pointer; MX_ERR_ALIGNMENT (data
 * not 4-byte aligned, out not element aligned); MX_ERR_UNSUPPORTED_DTYPE;
 * MX_ERR_DEVICE off sm_103.  Asynchronous on `stream`; allocates nothing.
 */
mx_status mx_dequantize(const void* data, const void* scale, mx_dtype in_dtype, int64_t rows, int64_t cols,
                        const mx_quant_cfg* cfg, mx_dtype out_dtype, void* out, int64_t ld_out,
                        mx_stream stream);

/*
 * Bytes of the tensor-core scale-factor ("SF") layout for an operand of `mn`
 * rows and K = `k` elements per row (k % 32 == 0): the E8M0 matrix
 * [mn, k/32] padded to 128-row x 4-column tiles of 512 bytes,
 * ceil(mn/128) * ceil(k/128) * 512.  The layout is that of the block-scaled
 * tcgen05 MMA (PTX ISA, tcgen05 "scale factor" matrices; also cuBLASLt's
 * 1-D block-scaling layout); the pages have no counterpart.
 */
mx_status mx_sf_layout_bytes(int64_t mn, int64_t k, size_t* bytes);

/*
 * Repack plain E8M0 scales [mn, k/32] (row pitch ld_plain bytes) into the SF
 * layout: tile (t_mn, t_k) = rows 128*t_mn.., scale columns 4*t_k.. is 512
 * contiguous bytes at ((t_mn * ceil(k/128)) + t_k) * 512, and inside a tile
 * scale (r, c) sits at byte (r % 32) * 16 + (r / 32) * 4 + c.  Padding bytes
 * are written as 0 (2^-127).  `plain` and `sf` are device pointers; `sf`
 * holds mx_sf_layout_bytes bytes.
 */
mx_status mx_repack_scales(const uint8_t* plain, int64_t mn, int64_t k, int64_t ld_plain,
                           uint8_t* sf, mx_stream stream);

/*
 * Workspace bytes mx_scaled_matmul needs: with plain scales, room for both
 * operands' SF-layout scales (16-byte aligned); with SF-layout scales, 0.
 */
mx_status mx_scaled_matmul_workspace(int64_t M, int64_t N, int64_t K, int scales_are_sf_layout,
                                     size_t* bytes);

/*
 * ScaledMatmul, block_scaled_dot(lhs, rhs, lhs_scale, rhs_scale) of the page
 * "MX-FP8 Microscaling Legalization" (sections 3 and 4.2; the scales are
 * bound by position), for the 2-D case with both operands contiguous along K:
 *
 *   C[m,n] = sum_k dec(A[m,k]) 2^(sA[m,k/32]-127) * dec(Bt[n,k]) 2^(sB[n,k/32]-127)
 *
 * accumulated in f32 on the tensor cores, written as f32 or bf16
 * (round to nearest even).
 *   a, bt        device codes, A [M, K] and Bt [N, K] (= rhs^T), dense,
 *                16-byte aligned; both of `elem_dtype`.  MX_E2M1 operands
 *                are packed two a byte, element 2i in the low nibble
 *                (mx_quantize with fp4_lane_stride 1, fp4_nibble_parity 1):
 *                rows of K/2 bytes
 *   a_scale,     device E8M0: plain [M, K/32] / [N, K/32] dense row-major
 *   b_scale      (scales_are_sf_layout = 0), or already in the SF layout of
 *                mx_repack_scales (scales_are_sf_layout = 1)
 *   elem_dtype   MX_E4M3FN | MX_E5M2 (ScaledMatmul_e4m3fn_e4m3fn_* /
 *                ScaledMatmul_e5m2_e5m2_*) | MX_E2M1 (MXFP4: an extension;
 *                the pages' ScaledMatmul takes FP8 only)
 *   M, N, K      M, N >= 1; K >= 32 and K % 32 == 0
 *   out_dtype    MX_F32 | MX_BF16
 *   c, ldc       device [M, ldc] output, ldc >= N, element aligned (16-byte
 *                aligned rows use vector stores)
 *   workspace    device scratch of mx_scaled_matmul_workspace bytes (may be
 *                NULL when that is 0); contents are overwritten
 */
mx_status mx_scaled_matmul(const void* a, const void* bt, const uint8_t* a_scale,
                           const uint8_t* b_scale, int scales_are_sf_layout, mx_dtype elem_dtype,
                           int64_t M, int64_t N, int64_t K, mx_dtype out_dtype, void* c,
                           int64_t ldc, void* workspace, size_t workspace_bytes, mx_stream stream);

/* Size of the fixed scratch array behind mx_scaled_matmul_noalloc (4 MiB). */
#define MX_NOALLOC_SCRATCH_BYTES (4 * 1024 * 1024)

/*
 * mx_scaled_matmul with plain scales, for callers that cannot allocate device
 * memory (no counterpart on the pages).  Some callers have no way to hand the
 * library a workspace: a plugin driven by a host runtime that owns all device
 * memory and gives the plugin no allocator, or a latency-critical path that
 * must not call cudaMalloc, which can synchronise the device.  This call keeps
 * the scratch for the two repacked scale tensors in a fixed device array
 * inside the library instead, and calls no allocating routine.
 *   Arguments as mx_scaled_matmul with scales_are_sf_layout = 0 and no
 *   workspace.
 *   Limit: the repacked scales, 16-byte rounded each, must fit in
 *   MX_NOALLOC_SCRATCH_BYTES (4 MiB), i.e.
 *   ceil(M/128)*ceil(K/128)*512 + ceil(N/128)*ceil(K/128)*512 <= 4 MiB
 *   (M = N = K = 8192 fits); larger problems get MX_ERR_WORKSPACE.
 *   The array takes 4 MiB on every device that loads the library, until
 *   process exit.  The first call on a device looks up the array's device
 *   address (make that first call before any stream capture on the device)
 *   and keeps it for the life of the process: do not use this call on a
 *   device after cudaDeviceReset there (the library's device arrays are
 *   loaded again, possibly at another address).
 *   Every call shares the array: calls whose kernels may overlap on the GPU
 *   (unordered streams) race on it; calls ordered on one stream are safe.
 */
mx_status mx_scaled_matmul_noalloc(const void* a, const void* bt, const uint8_t* a_scale,
                                   const uint8_t* b_scale, mx_dtype elem_dtype, int64_t M,
                                   int64_t N, int64_t K, mx_dtype out_dtype, void* c, int64_t ldc,
                                   mx_stream stream);

/*
 * Workspace bytes of mx_fused_quantize_matmul: the quantized activation
 * (M*K bytes, at offset 0), its SF-layout scales (at offset
 * round16(M*K)), then ceil(M/128) * ceil(K/256) + 1 64-bit ready words (at
 * offset round16(M*K) + round16(ceil(M/128) * ceil(K/128) * 512)), each
 * part 16-byte aligned; round16(x) rounds x up to a multiple of 16.
 */
mx_status mx_fused_quantize_matmul_workspace(int64_t M, int64_t N, int64_t K, size_t* bytes);

/*
 * Activation quantize fused with ScaledMatmul (page "MX-FP8 Microscaling
 * Legalization", section 4.3: QuantizeMX feeds ScaledMatmul by dataflow):
 * X [M, K] bf16/f16 is quantized along K (1x32 blocks, EMAX) to `elem_dtype`
 * and multiplied by a pre-quantized weight given K-contiguous as
 * Wt [N, K] with SF-layout scales.  The result equals QuantizeMX(X) followed
 * by mx_scaled_matmul bit for bit in the quantized operand.
 *   Where the pair GEMM kernel takes the product (M > 128 and enough 256 x 256
 *   tiles; see mx_debug_set_gemm_variant), the product is long (at least 32
 *   of its 256 x 256 tiles per pair of SMs: shorter ones run faster as two
 *   launches), and x is 32-byte aligned with a row pitch of a multiple of
 *   32 bytes, the call is ONE kernel launch: its
 *   epilogue warps quantize X in items of 128 rows x 256 elements, in the
 *   order the tiles consume them, while the tensor cores run, and publish
 *   each item through a ready word in the workspace that the operand loads
 *   wait on (bounded; a wait that runs out records MX_ERR_TIMEOUT).  Other
 *   shapes run QuantizeMX, then mx_scaled_matmul, on the stream.  Either way
 *   the workspace holds QuantizeMX(X) afterwards (codes and SF-layout scales
 *   at the offsets above; scale bytes of rows past M are unspecified).  The
 *   ready words need no clearing: a launch only accepts words it wrote itself
 *   (a per-call tag), and its last CTA sets them all back to zero, so
 *   reusing a workspace, and replaying a captured call, are both safe.
 *   Calls that share a workspace must not overlap on the GPU.
 *   x, x_dtype   device [M, ld_x] MX_BF16 | MX_F16
 *   wt, w_scale_sf  device codes [N, K] and SF-layout scales (mx_repack_scales);
 *                for MX_E2M1 X is packed in the tensor-core nibble order
 *                (element 2i low) and so must Wt be
 *   other arguments as mx_scaled_matmul; workspace per
 *   mx_fused_quantize_matmul_workspace.
 */
mx_status mx_fused_quantize_matmul(const void* x, mx_dtype x_dtype, int64_t ld_x, const void* wt,
                                   const uint8_t* w_scale_sf, mx_dtype elem_dtype, int64_t M,
                                   int64_t N, int64_t K, mx_dtype out_dtype, void* c, int64_t ldc,
                                   void* workspace, size_t workspace_bytes, mx_stream stream);

/* ------------------------------------------------ general block-scaled dot */

#define MX_MAX_RANK 8

/*
 * Dot dimension numbers of the ScaledMatmul contract (page "MX-FP8
 * Microscaling Legalization", section 4.2: lhs_batch_dimensions,
 * rhs_batch_dimensions, lhs_contracting_dimensions,
 * rhs_contracting_dimensions).  Indices are axes of the operand (negative
 * ones count from the end).  Exactly one contracting dimension per operand:
 * MX blocks run along one axis.
 */
typedef struct mx_dot_dims {
    int lhs_n_batch, rhs_n_batch;
    int64_t lhs_batch[MX_MAX_RANK], rhs_batch[MX_MAX_RANK];
    int lhs_n_contract, rhs_n_contract;
    int64_t lhs_contract[MX_MAX_RANK], rhs_contract[MX_MAX_RANK];
} mx_dot_dims;

/*
 * Result shape of mx_block_scaled_dot: the batch extents (in the listed
 * order), then the lhs free extents, then the rhs free extents, each in
 * operand axis order.  out_dims holds at least MX_MAX_RANK entries.
 * Errors as for mx_block_scaled_dot's dimension checks.
 */
mx_status mx_block_scaled_dot_shape(const int64_t* lhs_dims, int lhs_rank, const int64_t* rhs_dims, int rhs_rank,
                                    const mx_dot_dims* dims, int64_t* out_dims, int* out_rank);

/* Workspace bytes mx_block_scaled_dot needs for these shapes. */
mx_status mx_block_scaled_dot_workspace(const int64_t* lhs_dims, int lhs_rank, const int64_t* rhs_dims,
                                        int rhs_rank, const mx_dot_dims* dims, size_t* bytes);

/*
 * block_scaled_dot(lhs, rhs, lhs_scale, rhs_scale) with dot dimension
 * numbers (page "MX-FP8 Microscaling Legalization", sections 3.2 and 4.2):
 *   out[b.., i.., j..] = sum_k lhs(b.., i.., k) 2^(sl - 127) * rhs(b.., j.., k) 2^(sr - 127)
 * with the scale of each element the E8M0 of its 32-element block along the
 * contracting axis.
 *   lhs, rhs    device FP8 codes, dense row-major with extents lhs_dims /
 *               rhs_dims (rank 2..MX_MAX_RANK)
 *   lhs_scale, rhs_scale  device E8M0, dense, the operand's extents with the
 *               contracting one divided by 32 (what mx_quantize writes for
 *               1x32 blocks along that axis, plain layout)
 *   dims        dot dimension numbers
 *   elem_dtype  MX_E4M3FN | MX_E5M2 | MX_E2M1 (both operands; e2m1 packed
 *               as for mx_scaled_matmul, which needs the contracting axis
 *               innermost in both operands, else MX_ERR_UNSUPPORTED_DTYPE)
 *   out_dtype   MX_F32 | MX_BF16 (round to nearest even); `out` is dense in
 *               the order of mx_block_scaled_dot_shape, caller-owned
 *   workspace   device, 16-byte aligned, mx_block_scaled_dot_workspace bytes
 *               (room for canonical copies of operands that are not
 *               already [batch.., free.., K] in memory, and the scales in
 *               the tensor-core layout)
 * Operands already in [batch.., free.., K] order are read in place and must
 * be 16-byte aligned.  FP8 operands stored [batch.., K, free..] (the batch
 * axes in order, then the contracting axis) are read in place too, as
 * MN-major tiles, when their rows (the product of the free extents) are a
 * multiple of 16 bytes on a 16-byte aligned base; other layouts are copied
 * into [batch, rows, K] first.  Accumulation is f32 on the tensor cores.
 * Errors (nothing launched): MX_ERR_SHAPE (rank < 2 or > MX_MAX_RANK, batch
 * or contracting extents differ, K not a multiple of 32 or < 32, extents
 * over 2^30), MX_ERR_DIM (batch counts differ, an index out of bounds or
 * repeated, contracting overlapping batch, not exactly one contracting
 * dimension), MX_ERR_UNSUPPORTED_DTYPE, MX_ERR_INVALID_ARG, MX_ERR_ALIGNMENT,
 * MX_ERR_WORKSPACE, MX_ERR_DEVICE.  Asynchronous on `stream`.
 */
mx_status mx_block_scaled_dot(const void* lhs, const int64_t* lhs_dims, int lhs_rank, const void* lhs_scale,
                              const void* rhs, const int64_t* rhs_dims, int rhs_rank, const void* rhs_scale,
                              const mx_dot_dims* dims, mx_dtype elem_dtype, mx_dtype out_dtype, void* out,
                              void* workspace, size_t workspace_bytes, mx_stream stream);

/*
 * Read and clear the current device's status word (synchronises the device).
 * *status receives MX_OK or the first device-side error recorded since the
 * last read (MX_ERR_TIMEOUT when a bounded wait gave up).
 */
mx_status mx_get_device_status(int* status);

/* Static description of a status code; never NULL. */
const char* mx_status_string(mx_status status);

/* Library version, major*10000 + minor*100 + patch. */
int mx_version(void);

/*
 * Testing hook for the bounded-wait path (no counterpart on the pages).
 * skip_producer bit 0 makes later GEMM launches issue no loads; bit 1 makes
 * the single-launch mx_fused_quantize_matmul never publish its quantize
 * items (so its loads never start).  Either way the kernels' waits run out
 * after `timeout_ns` (0 = the default of 2 s) and record MX_ERR_TIMEOUT in
 * the device status word, with no fault and no hang.  skip_producer = 0
 * restores normal operation.  Not thread-safe; host only.
 */
mx_status mx_debug_gemm_fault_injection(int skip_producer, uint64_t timeout_ns);

/*
 * Testing hook (no counterpart on the pages): which ScaledMatmul kernel later
 * calls use.  0 = automatic (the 1-SM kernel when M <= 128, and when M > 128
 * but the pair kernel's 256 x 256 tiles would fill at most a quarter of its
 * clusters while the 1-SM kernel can split K at least two ways; otherwise
 * the 2-SM pair kernel), 1 = always the 1-SM kernel, 2 = always the pair kernel,
 * 3 = always the 1-SM kernel and never split K, 4 = automatic, but
 * mx_fused_quantize_matmul always as two launches (QuantizeMX, then
 * ScaledMatmul).  Under 2 the fused call runs as one launch whenever its
 * input allows it; under 1 and 3 it runs as two.  The 1-SM kernel splits K
 * over a cluster of up to 8 CTAs per tile when the problem has too few
 * tiles to fill the GPU (small M); the slices' f32 partial sums are added in
 * slice order, so a given shape always gives the same bits.  All variants
 * give results within the same tolerance.  Returns MX_ERR_INVALID_ARG for
 * other values.  Not thread-safe; host only.
 */
mx_status mx_debug_set_gemm_variant(int variant);

/*
 * Testing hook (no counterpart on the pages): the kernel of the last
 * ScaledMatmul launch made by this process (*kernel: 1 = 1-SM, 2 = pair,
 * 3 = pair with the fused activation quantize, 0 = none yet) and its split-K factor (*split_k: CTAs per tile along K, 1 =
 * no split).  MX_ERR_INVALID_ARG if a pointer is NULL.  Host only.
 */
mx_status mx_debug_last_gemm_launch(int* kernel, int* split_k);

/*
 * Testing hook (no counterpart on the pages): whether the last ScaledMatmul
 * launch read A (*a_mn_major) and B (*b_mn_major) in place as MN-major tiles
 * (1) or as K-major rows (0).  mx_block_scaled_dot reads an FP8 operand
 * stored [batch..., K, rows...] (batch axes in order, then the contracting
 * axis, then the free axes) in place when the operand's rows are a
 * multiple of 16 bytes on a 16-byte aligned base (either GEMM kernel);
 * otherwise it copies the operand into [batch, rows, K] first.
 * MX_ERR_INVALID_ARG if a pointer is NULL.  Host only.
 */
mx_status mx_debug_last_gemm_operands(int* a_mn_major, int* b_mn_major);

#ifdef __cplusplus
}
#endif

#endif /* MX_H_ */
