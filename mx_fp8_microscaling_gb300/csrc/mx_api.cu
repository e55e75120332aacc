// libmx C-ABI: argument validation, normalisation and dispatch.
//
// Every entry point validates its arguments on the host and returns an
// mx_status without launching anything when they are wrong; otherwise it
// launches on the caller's stream and returns at once.  The contract checks
// mirror the QuantizeMX / ScaledMatmul validators the page "MX-FP8
// Microscaling Legalization" lists (section 6 GOTCHA and section 7: block_size
// 32, the dtype sets, dim -1 / -2, divisibility by 4 for the x4 container, the
// operand and output types).

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "mx.h"
#include "mx_internal.h"

namespace mx {

void set_gemm_fault_injection(int skip_producer, uint64_t timeout_ns);
void set_gemm_variant(int variant);

namespace {

struct DeviceInfo {
    bool ready = false;
    bool sm103 = false;
    int sms = 0;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

const DeviceInfo& current_device() {
    static DeviceInfo none;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return none;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return none;
        d.sm103 = (major == 10 && minor == 3);
        d.sms = sms;
        d.ready = true;
    }
    return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Normalised QuantizeMX configuration.
struct QuantPlan {
    int fmt = 0;
    bool in_f16 = false;
    int br = 0, bc = 0;
    int scale_mode = 0;
    int emax_bias = 0;
    int stride = 0, parity = 0;
    int64_t scale_rows = 0, scale_cols = 0, scale_buf_rows = 0;
    size_t data_bytes = 0;
};

int emax_of(int fmt) { return fmt == kE2M1 ? 2 : (fmt == kE4M3 ? 8 : 15); }

mx_status plan_quantize(mx_dtype in_dtype, mx_dtype out_dtype, int64_t rows, int64_t cols,
                        const mx_quant_cfg* user_cfg, QuantPlan* plan) {
    mx_quant_cfg cfg;
    mx_quant_cfg_default(&cfg);
    if (user_cfg) cfg = *user_cfg;

    if (in_dtype != MX_BF16 && in_dtype != MX_F16) return MX_ERR_UNSUPPORTED_DTYPE;
    switch (out_dtype) {
    case MX_E4M3FN: plan->fmt = kE4M3; break;
    case MX_E5M2: plan->fmt = kE5M2; break;
    case MX_E2M1: plan->fmt = kE2M1; break;
    default: return MX_ERR_UNSUPPORTED_DTYPE;
    }
    plan->in_f16 = (in_dtype == MX_F16);
    if (cfg.block_size != 0 && cfg.block_size != 32) return MX_ERR_BLOCK_SIZE;
    if (cfg.scale_method != MX_SCALE_METHOD_EMAX) return MX_ERR_SCALE_METHOD;
    int dim = cfg.dim;
    if (dim == 1) dim = -1;
    if (dim == 0) dim = -2;
    if (dim != -1 && dim != -2) return MX_ERR_DIM;
    if (cfg.geometry == MX_GEOM_8X4) {
        plan->br = dim == -2 ? 8 : 4;
        plan->bc = dim == -2 ? 4 : 8;
    } else if (cfg.geometry == MX_GEOM_1X32) {
        plan->br = dim == -2 ? 32 : 1;
        plan->bc = dim == -2 ? 1 : 32;
    } else {
        return MX_ERR_INVALID_ARG;
    }
    if (cfg.scale_layout != MX_SCALE_PLAIN && cfg.scale_layout != MX_SCALE_INTERLEAVE32 &&
        cfg.scale_layout != MX_SCALE_TC_SF)
        return MX_ERR_INVALID_ARG;
    if (cfg.scale_layout == MX_SCALE_TC_SF && (cfg.geometry != MX_GEOM_1X32 || dim != -1))
        return MX_ERR_INVALID_ARG;
    plan->scale_mode = cfg.scale_layout;
    if (cfg.emax_alt != 0 && cfg.emax_alt != 1) return MX_ERR_INVALID_ARG;
    plan->emax_bias = emax_of(plan->fmt) - cfg.emax_alt;
    const int s = cfg.fp4_lane_stride;
    if (s != 0 && s != 1 && s != 2 && s != 4) return MX_ERR_INVALID_ARG;
    if (cfg.fp4_nibble_parity != 0 && cfg.fp4_nibble_parity != 1) return MX_ERR_INVALID_ARG;
    plan->stride = s;
    plan->parity = cfg.fp4_nibble_parity;

    if (rows < 0 || cols < 0) return MX_ERR_INVALID_ARG;
    if (cols % 4 != 0 || rows % plan->br != 0 || cols % plan->bc != 0) return MX_ERR_SHAPE;
    if (plan->fmt == kE2M1 && s > 1 && cols % (2 * s) != 0) return MX_ERR_SHAPE;

    plan->scale_rows = rows / plan->br;
    plan->scale_cols = cols / plan->bc;
    if (plan->scale_mode == MX_SCALE_INTERLEAVE32) {
        plan->scale_buf_rows = 32 * ((plan->scale_rows + 3) / 4);
    } else if (plan->scale_mode == MX_SCALE_TC_SF) {
        plan->scale_buf_rows = (plan->scale_rows + 127) / 128 * 128;
        plan->scale_cols = (plan->scale_cols + 3) / 4 * 4;
    } else {
        plan->scale_buf_rows = plan->scale_rows;
    }
    plan->data_bytes = static_cast<size_t>(plan->fmt == kE2M1 ? rows * cols / 2 : rows * cols);
    return MX_OK;
}

// __byte_perm selector that moves pair-byte p of an 8-element chunk to the
// byte the page's lane_remap gives element 2p: byte (remap(2p) >> 1).
uint32_t fp4_pair_perm(int stride) {
    int dest[4];
    for (int p = 0; p < 4; ++p) {
        int64_t n = 2 * p, r = n;
        if (stride) {
            const int64_t w = 2 * stride, q = n / w, rr = n % w;
            r = w * (q + 1) - rr;
            if ((n & 1) == 0) r -= 2;
        }
        dest[p] = static_cast<int>(r >> 1);
    }
    uint32_t sel = 0;
    for (int p = 0; p < 4; ++p) sel |= static_cast<uint32_t>(p) << (4 * dest[p]);
    return sel;
}

mx_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MX_OK : MX_ERR_CUDA; }

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// General block-scaled dot: each operand is brought to [batch, rows, K]
// (batch axes in the listed order, free axes in their own order, the
// contracting axis innermost); perm[c] is the operand axis at canonical
// position c.
struct DotPlan {
    int64_t batch = 1, M = 0, N = 0, K = 0;
    int lrank = 0, rrank = 0;
    int lperm[MX_MAX_RANK] = {}, rperm[MX_MAX_RANK] = {};
    int lc = 0, rc = 0;
    bool lcanon = true, rcanon = true;
    // stored [batch..., K, free...] (batch axes in order, then the
    // contracting one): an MN-major operand the GEMM kernels read in place
    bool lmn = false, rmn = false;
    size_t off_lq = 0, off_ls = 0, off_rq = 0, off_rs = 0, off_sfa = 0, off_sfb = 0, total = 0;
};

mx_status plan_dot(const int64_t* ldims, int lrank, const int64_t* rdims, int rrank, const mx_dot_dims* dn,
                   DotPlan* P) {
    if (!ldims || !rdims || !dn || !P) return MX_ERR_INVALID_ARG;
    // the contract's checks: rank >= 2, equal batch counts, indices in
    // bounds, batch extents equal, contracting sizes equal and disjoint from
    // the batch dimensions; one contracting dimension per operand
    if (lrank < 2 || rrank < 2 || lrank > MX_MAX_RANK || rrank > MX_MAX_RANK) return MX_ERR_SHAPE;
    for (int i = 0; i < lrank; ++i)
        if (ldims[i] < 0) return MX_ERR_INVALID_ARG;
    for (int i = 0; i < rrank; ++i)
        if (rdims[i] < 0) return MX_ERR_INVALID_ARG;
    if (dn->lhs_n_batch != dn->rhs_n_batch || dn->lhs_n_batch < 0 || dn->lhs_n_batch > MX_MAX_RANK) return MX_ERR_DIM;
    if (dn->lhs_n_contract != 1 || dn->rhs_n_contract != 1) return MX_ERR_DIM;
    auto norm = [](int64_t d, int r, int* out) {
        if (d < -r || d >= r) return false;
        *out = static_cast<int>(d < 0 ? d + r : d);
        return true;
    };
    const int nb = dn->lhs_n_batch;
    int lb[MX_MAX_RANK], rb[MX_MAX_RANK];
    bool lused[MX_MAX_RANK] = {}, rused[MX_MAX_RANK] = {};
    for (int i = 0; i < nb; ++i) {
        if (!norm(dn->lhs_batch[i], lrank, &lb[i]) || !norm(dn->rhs_batch[i], rrank, &rb[i])) return MX_ERR_DIM;
        if (lused[lb[i]] || rused[rb[i]]) return MX_ERR_DIM;
        lused[lb[i]] = rused[rb[i]] = true;
    }
    int lc, rc;
    if (!norm(dn->lhs_contract[0], lrank, &lc) || !norm(dn->rhs_contract[0], rrank, &rc)) return MX_ERR_DIM;
    if (lused[lc] || rused[rc]) return MX_ERR_DIM;
    lused[lc] = rused[rc] = true;
    int64_t batch = 1;
    for (int i = 0; i < nb; ++i) {
        if (ldims[lb[i]] != rdims[rb[i]]) return MX_ERR_SHAPE;
        batch *= ldims[lb[i]];
    }
    const int64_t K = ldims[lc];
    if (K != rdims[rc] || K < 32 || K % 32 != 0) return MX_ERR_SHAPE;
    DotPlan p;
    p.lrank = lrank;
    p.rrank = rrank;
    p.lc = lc;
    p.rc = rc;
    int n = 0;
    for (int i = 0; i < nb; ++i) p.lperm[n++] = lb[i];
    int64_t M = 1;
    for (int i = 0; i < lrank; ++i)
        if (!lused[i]) p.lperm[n++] = i, M *= ldims[i];
    p.lperm[n] = lc;
    n = 0;
    for (int i = 0; i < nb; ++i) p.rperm[n++] = rb[i];
    int64_t N = 1;
    for (int i = 0; i < rrank; ++i)
        if (!rused[i]) p.rperm[n++] = i, N *= rdims[i];
    p.rperm[n] = rc;
    for (int i = 0; i < lrank; ++i) p.lcanon = p.lcanon && p.lperm[i] == i;
    for (int i = 0; i < rrank; ++i) p.rcanon = p.rcanon && p.rperm[i] == i;
    auto mn_order = [nb](const int* perm, int rank) {
        if (perm[rank - 1] != nb) return false;
        for (int i = 0; i < nb; ++i)
            if (perm[i] != i) return false;
        for (int i = nb; i < rank - 1; ++i)
            if (perm[i] != i + 1) return false;
        return true;
    };
    p.lmn = !p.lcanon && mn_order(p.lperm, lrank);
    p.rmn = !p.rcanon && mn_order(p.rperm, rrank);
    if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || K > (int64_t(1) << 30)) return MX_ERR_SHAPE;
    // tiles of all problems are counted in 32-bit integers by the kernels
    if (batch * ((M + 127) / 128) * ((N + 127) / 128) > (int64_t(1) << 30)) return MX_ERR_SHAPE;
    p.batch = batch;
    p.M = M;
    p.N = N;
    p.K = K;
    size_t off = 0;
    if (!p.lcanon) {
        p.off_lq = off;
        off += align256(static_cast<size_t>(batch * M * K));
        p.off_ls = off;
        off += align256(static_cast<size_t>(batch * M * (K / 32)));
    }
    if (!p.rcanon) {
        p.off_rq = off;
        off += align256(static_cast<size_t>(batch * N * K));
        p.off_rs = off;
        off += align256(static_cast<size_t>(batch * N * (K / 32)));
    }
    p.off_sfa = off;
    off += align256(static_cast<size_t>(batch) * sf_layout_bytes(M, K));
    p.off_sfb = off;
    off += align256(static_cast<size_t>(batch) * sf_layout_bytes(N, K));
    p.total = off;
    *P = p;
    return MX_OK;
}

// Copy an operand (codes, or scales with the contracting axis divided by 32)
// into canonical order.
cudaError_t permute_operand(const void* src, const int64_t* dims, int rank, const int* perm, int contract,
                            int64_t contract_div, uint8_t* dst, cudaStream_t s) {
    int64_t ext[MX_MAX_RANK], stride[MX_MAX_RANK];
    for (int i = 0; i < rank; ++i) ext[i] = i == contract ? dims[i] / contract_div : dims[i];
    int64_t st = 1;
    for (int i = rank - 1; i >= 0; --i) {
        stride[i] = st;
        st *= ext[i];
    }
    PermuteArgs a{};
    a.src = static_cast<const uint8_t*>(src);
    a.dst = dst;
    a.rank = rank;
    for (int c = 0; c < rank; ++c) {
        a.dst_dims[c] = ext[perm[c]];
        a.src_stride[c] = stride[perm[c]];
    }
    return launch_permute_bytes(a, s);
}

}  // namespace

int device_sm_count() { return current_device().sms; }
bool device_is_sm103() { return current_device().sm103; }

}  // namespace mx

using namespace mx;

extern "C" {

mx_status mx_quant_cfg_default(mx_quant_cfg* cfg) {
    if (!cfg) return MX_ERR_INVALID_ARG;
    cfg->geometry = MX_GEOM_8X4;
    cfg->scale_layout = MX_SCALE_PLAIN;
    cfg->block_size = 32;
    cfg->dim = -2;
    cfg->scale_method = MX_SCALE_METHOD_EMAX;
    cfg->fp4_lane_stride = 2;
    cfg->fp4_nibble_parity = 0;
    cfg->emax_alt = 0;
    return MX_OK;
}

mx_status mx_quantize_sizes(mx_dtype in_dtype, mx_dtype out_dtype, int64_t rows, int64_t cols,
                            const mx_quant_cfg* cfg, size_t* data_bytes, int64_t* scale_rows,
                            int64_t* scale_cols, size_t* scale_bytes) {
    QuantPlan plan;
    mx_status st = plan_quantize(in_dtype, out_dtype, rows, cols, cfg, &plan);
    if (st != MX_OK) return st;
    if (data_bytes) *data_bytes = plan.data_bytes;
    if (scale_rows) *scale_rows = plan.scale_buf_rows;
    if (scale_cols) *scale_cols = plan.scale_cols;
    if (scale_bytes) *scale_bytes = static_cast<size_t>(plan.scale_buf_rows * plan.scale_cols);
    return MX_OK;
}

mx_status mx_quantize(const void* in, mx_dtype in_dtype, int64_t rows, int64_t cols, int64_t ld_in,
                      mx_dtype out_dtype, const mx_quant_cfg* cfg, void* out_data, void* out_scale,
                      mx_stream stream) {
    QuantPlan plan;
    mx_status st = plan_quantize(in_dtype, out_dtype, rows, cols, cfg, &plan);
    if (st != MX_OK) return st;
    if (ld_in < cols) return MX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MX_OK;
    if (!in || !out_data || !out_scale) return MX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(in) & 1u) || (reinterpret_cast<uintptr_t>(out_data) & 1u))
        return MX_ERR_ALIGNMENT;
    if (!device_is_sm103()) return MX_ERR_DEVICE;

    QuantArgs q{};
    q.in = static_cast<const uint8_t*>(in);
    q.rows = rows;
    q.cols = cols;
    q.ld_in = ld_in;
    q.data = static_cast<uint8_t*>(out_data);
    q.ld_data = plan.fmt == kE2M1 ? cols / 2 : cols;
    q.scale = static_cast<uint8_t*>(out_scale);
    q.scale_cols = plan.scale_cols;
    q.block_rows = plan.br;
    q.block_cols = plan.bc;
    q.scale_mode = plan.scale_mode;
    q.sf_ntk = plan.scale_cols / 4;
    q.emax_bias = plan.emax_bias;
    q.fp4_stride = plan.stride;
    q.fp4_parity = plan.parity;
    q.fp4_perm = fp4_pair_perm(plan.stride);
    q.vec_ok = aligned16(in) && (ld_in * 2) % 16 == 0 && (reinterpret_cast<uintptr_t>(out_data) & 7u) == 0 &&
               (reinterpret_cast<uintptr_t>(out_scale) & 1u) == 0;
    q.vec32_ok = q.vec_ok && (reinterpret_cast<uintptr_t>(in) & 31u) == 0 && (ld_in * 2) % 32 == 0 &&
                 (reinterpret_cast<uintptr_t>(out_data) & 15u) == 0 && cols % 32 == 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (plan.scale_mode == MX_SCALE_TC_SF && (rows % 128 != 0 || (cols / 32) % 4 != 0)) {
        // the kernel writes live scales only; padding of the SF tiles is 0
        if (cudaMemsetAsync(out_scale, 0, static_cast<size_t>(plan.scale_buf_rows * plan.scale_cols), s) !=
            cudaSuccess)
            return MX_ERR_CUDA;
    }
    return from_cuda(launch_quantize(q, plan.in_f16, plan.fmt, s));
}

mx_status mx_dequantize(const void* data, const void* scale, mx_dtype in_dtype, int64_t rows, int64_t cols,
                        const mx_quant_cfg* cfg, mx_dtype out_dtype, void* out, int64_t ld_out, mx_stream stream) {
    QuantPlan plan;
    // the codes' format and the block layout are checked as QuantizeMX checks them
    mx_status st = plan_quantize(MX_BF16, in_dtype, rows, cols, cfg, &plan);
    if (st != MX_OK) return st;
    if (out_dtype != MX_F32 && out_dtype != MX_BF16) return MX_ERR_UNSUPPORTED_DTYPE;
    if (ld_out < cols) return MX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MX_OK;
    if (!data || !scale || !out) return MX_ERR_INVALID_ARG;
    const uintptr_t esize = out_dtype == MX_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(data) & 3u) || (reinterpret_cast<uintptr_t>(out) & (esize - 1)))
        return MX_ERR_ALIGNMENT;
    if (!device_is_sm103()) return MX_ERR_DEVICE;
    DequantArgs q{};
    q.data = static_cast<const uint8_t*>(data);
    q.scale = static_cast<const uint8_t*>(scale);
    q.rows = rows;
    q.cols = cols;
    q.block_rows = plan.br;
    q.block_cols = plan.bc;
    q.scale_mode = plan.scale_mode;
    q.scale_cols = plan.scale_cols;
    q.sf_ntk = plan.scale_cols / 4;
    // inverse of the packing selector: source byte p sits at destination byte d(p)
    const uint32_t fwd = fp4_pair_perm(plan.stride);
    uint32_t inv = 0;
    for (int d = 0; d < 4; ++d) inv |= static_cast<uint32_t>(d) << (4 * ((fwd >> (4 * d)) & 0xFu));
    q.fp4_inv_perm = inv;
    q.fp4_parity = plan.parity;
    q.out = out;
    q.ld_out = ld_out;
    q.vec_ok = aligned16(out) && (ld_out * static_cast<int64_t>(esize)) % 16 == 0;
    return from_cuda(launch_dequantize(q, plan.fmt, out_dtype == MX_BF16, reinterpret_cast<cudaStream_t>(stream)));
}

mx_status mx_sf_layout_bytes(int64_t mn, int64_t k, size_t* bytes) {
    if (!bytes || mn < 0 || k < 0) return MX_ERR_INVALID_ARG;
    if (k % 32 != 0) return MX_ERR_SHAPE;
    *bytes = sf_layout_bytes(mn, k);
    return MX_OK;
}

mx_status mx_repack_scales(const uint8_t* plain, int64_t mn, int64_t k, int64_t ld_plain, uint8_t* sf,
                           mx_stream stream) {
    if (mn < 0 || k < 0) return MX_ERR_INVALID_ARG;
    if (k % 32 != 0) return MX_ERR_SHAPE;
    if (ld_plain < k / 32) return MX_ERR_INVALID_ARG;
    if (mn == 0 || k == 0) return MX_OK;
    if (!plain || !sf) return MX_ERR_INVALID_ARG;
    if (!aligned16(sf)) return MX_ERR_ALIGNMENT;
    if (!device_is_sm103()) return MX_ERR_DEVICE;
    return from_cuda(launch_repack_scales(plain, mn, k, ld_plain, sf, reinterpret_cast<cudaStream_t>(stream)));
}

mx_status mx_scaled_matmul_workspace(int64_t M, int64_t N, int64_t K, int scales_are_sf_layout, size_t* bytes) {
    if (!bytes || M < 0 || N < 0 || K < 0) return MX_ERR_INVALID_ARG;
    if (K % 32 != 0) return MX_ERR_SHAPE;
    *bytes = scales_are_sf_layout ? 0 : align16(sf_layout_bytes(M, K)) + align16(sf_layout_bytes(N, K));
    return MX_OK;
}

static int gemm_fmt(mx_dtype elem_dtype) {
    return elem_dtype == MX_E4M3FN ? kE4M3 : (elem_dtype == MX_E5M2 ? kE5M2 : kE2M1);
}

// Bytes of `k` elements of a K-contiguous operand row.
static int64_t elem_bytes(mx_dtype elem_dtype, int64_t k) { return elem_dtype == MX_E2M1 ? k / 2 : k; }

static mx_status check_matmul(const void* a, const void* bt, const uint8_t* a_scale, const uint8_t* b_scale,
                              mx_dtype elem_dtype, int64_t M, int64_t N, int64_t K, mx_dtype out_dtype, void* c,
                              int64_t ldc) {
    if (elem_dtype != MX_E4M3FN && elem_dtype != MX_E5M2 && elem_dtype != MX_E2M1) return MX_ERR_UNSUPPORTED_DTYPE;
    if (out_dtype != MX_F32 && out_dtype != MX_BF16) return MX_ERR_UNSUPPORTED_DTYPE;
    if (M < 0 || N < 0 || K < 0) return MX_ERR_INVALID_ARG;
    if (K < 32 || K % 32 != 0) return MX_ERR_SHAPE;
    if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || K > (int64_t(1) << 30)) return MX_ERR_SHAPE;
    if (ldc < N) return MX_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return MX_OK;
    if (!a || !bt || !a_scale || !b_scale || !c) return MX_ERR_INVALID_ARG;
    const uintptr_t esize = out_dtype == MX_F32 ? 4 : 2;
    if (!aligned16(a) || !aligned16(bt) || (reinterpret_cast<uintptr_t>(c) & (esize - 1))) return MX_ERR_ALIGNMENT;
    return MX_OK;
}

mx_status mx_scaled_matmul(const void* a, const void* bt, const uint8_t* a_scale, const uint8_t* b_scale,
                           int scales_are_sf_layout, mx_dtype elem_dtype, int64_t M, int64_t N, int64_t K,
                           mx_dtype out_dtype, void* c, int64_t ldc, void* workspace, size_t workspace_bytes,
                           mx_stream stream) {
    mx_status st = check_matmul(a, bt, a_scale, b_scale, elem_dtype, M, N, K, out_dtype, c, ldc);
    if (st != MX_OK || M == 0 || N == 0) return st;
    const uint8_t* sfa = a_scale;
    const uint8_t* sfb = b_scale;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (scales_are_sf_layout) {
        if (!aligned16(a_scale) || !aligned16(b_scale)) return MX_ERR_ALIGNMENT;
    } else {
        size_t need = 0;
        mx_scaled_matmul_workspace(M, N, K, 0, &need);
        if (!workspace || workspace_bytes < need) return MX_ERR_WORKSPACE;
        if (!aligned16(workspace)) return MX_ERR_ALIGNMENT;
    }
    if (!device_is_sm103()) return MX_ERR_DEVICE;
    if (!scales_are_sf_layout) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        uint8_t* wa = ws;
        uint8_t* wb = ws + align16(sf_layout_bytes(M, K));
        cudaError_t e = launch_repack_scales(a_scale, M, K, K / 32, wa, s);
        if (e == cudaSuccess) e = launch_repack_scales(b_scale, N, K, K / 32, wb, s);
        if (e != cudaSuccess) return MX_ERR_CUDA;
        sfa = wa;
        sfb = wb;
    }
    GemmArgs g{};
    g.a = static_cast<const uint8_t*>(a);
    g.bt = static_cast<const uint8_t*>(bt);
    g.sfa = sfa;
    g.sfb = sfb;
    g.M = M;
    g.N = N;
    g.K = K;
    g.c = c;
    g.ldc = ldc;
    g.elem_fmt = gemm_fmt(elem_dtype);
    g.out_bf16 = out_dtype == MX_BF16;
    g.vec_store = aligned16(c) && (ldc * (out_dtype == MX_F32 ? 4 : 2)) % 16 == 0;
    g.batch = 1;
    g.a_batch_stride = M * elem_bytes(elem_dtype, K);
    g.b_batch_stride = N * elem_bytes(elem_dtype, K);
    g.c_batch_stride = M * ldc;
    return from_cuda(launch_scaled_matmul(g, s));
}

// Fused workspace: the quantized activation (M*K bytes, enough for FP8 and
// e2m1), its SF-layout scales, then one 64-bit ready word per quantize item
// of the single-launch kernel (128 rows x 256 elements) and one done word.
static size_t fused_flags_offset(int64_t M, int64_t K) {
    return align16(static_cast<size_t>(M * K)) + align16(sf_layout_bytes(M, K));
}
static size_t fused_flag_bytes(int64_t M, int64_t K) {
    return (static_cast<size_t>((M + 127) / 128) * static_cast<size_t>((K + 255) / 256) + 1) * 8u;
}

mx_status mx_fused_quantize_matmul_workspace(int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (!bytes || M < 0 || N < 0 || K < 0) return MX_ERR_INVALID_ARG;
    if (K % 32 != 0) return MX_ERR_SHAPE;
    *bytes = fused_flags_offset(M, K) + align16(fused_flag_bytes(M, K));
    return MX_OK;
}

mx_status mx_fused_quantize_matmul(const void* x, mx_dtype x_dtype, int64_t ld_x, const void* wt,
                                   const uint8_t* w_scale_sf, mx_dtype elem_dtype, int64_t M, int64_t N, int64_t K,
                                   mx_dtype out_dtype, void* c, int64_t ldc, void* workspace,
                                   size_t workspace_bytes, mx_stream stream) {
    if (x_dtype != MX_BF16 && x_dtype != MX_F16) return MX_ERR_UNSUPPORTED_DTYPE;
    const void* dummy = workspace ? workspace : wt;
    mx_status st = check_matmul(dummy, wt, w_scale_sf, w_scale_sf, elem_dtype, M, N, K, out_dtype, c, ldc);
    if (st != MX_OK || M == 0 || N == 0) return st;
    if (ld_x < K) return MX_ERR_INVALID_ARG;
    if (!x) return MX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 1u) || !aligned16(w_scale_sf)) return MX_ERR_ALIGNMENT;
    size_t need = 0;
    mx_fused_quantize_matmul_workspace(M, N, K, &need);
    if (!workspace || workspace_bytes < need) return MX_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MX_ERR_ALIGNMENT;
    if (!device_is_sm103()) return MX_ERR_DEVICE;
    uint8_t* xq = static_cast<uint8_t*>(workspace);
    uint8_t* xs = xq + align16(static_cast<size_t>(M * K));
    {
        // one launch: the pair kernel quantizes X into the workspace itself
        GemmArgs g{};
        g.a = xq;
        g.bt = static_cast<const uint8_t*>(wt);
        g.sfa = xs;
        g.sfb = w_scale_sf;
        g.M = M;
        g.N = N;
        g.K = K;
        g.c = c;
        g.ldc = ldc;
        g.elem_fmt = gemm_fmt(elem_dtype);
        g.out_bf16 = out_dtype == MX_BF16;
        g.vec_store = aligned16(c) && (ldc * (out_dtype == MX_F32 ? 4 : 2)) % 16 == 0;
        g.batch = 1;
        g.a_batch_stride = M * elem_bytes(elem_dtype, K);
        g.b_batch_stride = N * elem_bytes(elem_dtype, K);
        g.c_batch_stride = M * ldc;
        g.x = static_cast<const uint8_t*>(x);
        g.ld_x_bytes = ld_x * 2;
        g.x_f16 = x_dtype == MX_F16;
        g.q_flags = reinterpret_cast<uint64_t*>(xq + fused_flags_offset(M, K));
        if (fused_single_launch(g)) return from_cuda(launch_fused_matmul(g, reinterpret_cast<cudaStream_t>(stream)));
    }
    mx_quant_cfg cfg;
    mx_quant_cfg_default(&cfg);
    cfg.geometry = MX_GEOM_1X32;
    cfg.dim = -1;
    cfg.scale_layout = MX_SCALE_TC_SF;
    if (elem_dtype == MX_E2M1) {  // the tensor cores' nibble order: element 2i in the low nibble
        cfg.fp4_lane_stride = 1;
        cfg.fp4_nibble_parity = 1;
    }
    st = mx_quantize(x, x_dtype, M, K, ld_x, elem_dtype, &cfg, xq, xs, stream);
    if (st != MX_OK) return st;
    return mx_scaled_matmul(xq, wt, xs, w_scale_sf, 1, elem_dtype, M, N, K, out_dtype, c, ldc, nullptr, 0, stream);
}

mx_status mx_block_scaled_dot_shape(const int64_t* lhs_dims, int lhs_rank, const int64_t* rhs_dims, int rhs_rank,
                                    const mx_dot_dims* dims, int64_t* out_dims, int* out_rank) {
    DotPlan P;
    mx_status st = plan_dot(lhs_dims, lhs_rank, rhs_dims, rhs_rank, dims, &P);
    if (st != MX_OK) return st;
    if (!out_dims || !out_rank) return MX_ERR_INVALID_ARG;
    int n = 0;
    for (int c = 0; c < lhs_rank - 1; ++c) out_dims[n++] = lhs_dims[P.lperm[c]];
    for (int c = dims->rhs_n_batch; c < rhs_rank - 1; ++c) out_dims[n++] = rhs_dims[P.rperm[c]];
    *out_rank = n;
    return MX_OK;
}

mx_status mx_block_scaled_dot_workspace(const int64_t* lhs_dims, int lhs_rank, const int64_t* rhs_dims,
                                        int rhs_rank, const mx_dot_dims* dims, size_t* bytes) {
    DotPlan P;
    mx_status st = plan_dot(lhs_dims, lhs_rank, rhs_dims, rhs_rank, dims, &P);
    if (st != MX_OK) return st;
    if (!bytes) return MX_ERR_INVALID_ARG;
    *bytes = P.total;
    return MX_OK;
}

mx_status mx_block_scaled_dot(const void* lhs, const int64_t* lhs_dims, int lhs_rank, const void* lhs_scale,
                              const void* rhs, const int64_t* rhs_dims, int rhs_rank, const void* rhs_scale,
                              const mx_dot_dims* dims, mx_dtype elem_dtype, mx_dtype out_dtype, void* out,
                              void* workspace, size_t workspace_bytes, mx_stream stream) {
    DotPlan P;
    mx_status st = plan_dot(lhs_dims, lhs_rank, rhs_dims, rhs_rank, dims, &P);
    if (st != MX_OK) return st;
    if (elem_dtype != MX_E4M3FN && elem_dtype != MX_E5M2 && elem_dtype != MX_E2M1) return MX_ERR_UNSUPPORTED_DTYPE;
    if (out_dtype != MX_F32 && out_dtype != MX_BF16) return MX_ERR_UNSUPPORTED_DTYPE;
    // packed e2m1 pairs run along the contracting axis: it must be innermost
    const bool fp4 = elem_dtype == MX_E2M1;
    if (fp4 && (P.lc != lhs_rank - 1 || P.rc != rhs_rank - 1)) return MX_ERR_UNSUPPORTED_DTYPE;
    if (P.batch == 0 || P.M == 0 || P.N == 0) return MX_OK;
    if (!lhs || !rhs || !lhs_scale || !rhs_scale || !out) return MX_ERR_INVALID_ARG;
    const uintptr_t esize = out_dtype == MX_F32 ? 4 : 2;
    if ((P.lcanon && !aligned16(lhs)) || (P.rcanon && !aligned16(rhs)) ||
        (reinterpret_cast<uintptr_t>(out) & (esize - 1)))
        return MX_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < P.total) return MX_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MX_ERR_ALIGNMENT;
    if (!device_is_sm103()) return MX_ERR_DEVICE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    GemmArgs g{};
    g.sfa = ws + P.off_sfa;
    g.sfb = ws + P.off_sfb;
    g.M = P.M;
    g.N = P.N;
    g.K = P.K;
    g.c = out;
    g.ldc = P.N;
    g.elem_fmt = gemm_fmt(elem_dtype);
    g.out_bf16 = out_dtype == MX_BF16;
    g.vec_store = aligned16(out) && (P.N * static_cast<int64_t>(esize)) % 16 == 0;
    g.batch = P.batch;
    g.a_batch_stride = P.M * elem_bytes(elem_dtype, P.K);
    g.b_batch_stride = P.N * elem_bytes(elem_dtype, P.K);
    g.c_batch_stride = P.M * P.N;
    // An FP8 operand stored [batch, K, rows] is read in place, MN-major, when
    // its rows are whole 16-byte multiples; otherwise it is copied into
    // [batch, rows, K] first.
    g.a_mn_major = !fp4 && P.lmn && P.M % 16 == 0 && aligned16(lhs);
    g.b_mn_major = !fp4 && P.rmn && P.N % 16 == 0 && aligned16(rhs);
    const uint8_t* a = static_cast<const uint8_t*>(lhs);
    const uint8_t* sa = static_cast<const uint8_t*>(lhs_scale);
    const uint8_t* bt = static_cast<const uint8_t*>(rhs);
    const uint8_t* sb = static_cast<const uint8_t*>(rhs_scale);
    cudaError_t e = cudaSuccess;
    const int64_t code_div = fp4 ? 2 : 1;  // elements per byte along the contracting axis
    if (!P.lcanon && !g.a_mn_major) {
        e = permute_operand(lhs, lhs_dims, lhs_rank, P.lperm, P.lc, code_div, ws + P.off_lq, s);
        if (e == cudaSuccess) e = permute_operand(lhs_scale, lhs_dims, lhs_rank, P.lperm, P.lc, 32, ws + P.off_ls, s);
        a = ws + P.off_lq;
        sa = ws + P.off_ls;
    }
    if (e == cudaSuccess && !P.rcanon && !g.b_mn_major) {
        e = permute_operand(rhs, rhs_dims, rhs_rank, P.rperm, P.rc, code_div, ws + P.off_rq, s);
        if (e == cudaSuccess) e = permute_operand(rhs_scale, rhs_dims, rhs_rank, P.rperm, P.rc, 32, ws + P.off_rs, s);
        bt = ws + P.off_rq;
        sb = ws + P.off_rs;
    }
    const int64_t kb = P.K / 32;
    if (e == cudaSuccess)
        e = g.a_mn_major ? launch_repack_scales_mn_inner(sa, P.M, P.K, P.M, P.M * kb, P.batch, ws + P.off_sfa, s)
                         : launch_repack_scales_batched(sa, P.M, P.K, kb, P.M * kb, P.batch, ws + P.off_sfa, s);
    if (e == cudaSuccess)
        e = g.b_mn_major ? launch_repack_scales_mn_inner(sb, P.N, P.K, P.N, P.N * kb, P.batch, ws + P.off_sfb, s)
                         : launch_repack_scales_batched(sb, P.N, P.K, kb, P.N * kb, P.batch, ws + P.off_sfb, s);
    if (e != cudaSuccess) return MX_ERR_CUDA;
    g.a = a;
    g.bt = bt;
    return from_cuda(launch_scaled_matmul(g, s));
}

mx_status mx_get_device_status(int* status) {
    if (!status) return MX_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return MX_ERR_CUDA;
    return from_cuda(read_and_clear_device_status(status));
}

const char* mx_status_string(mx_status status) {
    switch (status) {
    case MX_OK: return "MX_OK";
    case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG: invalid argument";
    case MX_ERR_UNSUPPORTED_DTYPE: return "MX_ERR_UNSUPPORTED_DTYPE: dtype combination not supported";
    case MX_ERR_BLOCK_SIZE: return "MX_ERR_BLOCK_SIZE: block_size must be 32";
    case MX_ERR_DIM: return "MX_ERR_DIM: only the last (-1) or second-to-last (-2) dim is supported";
    case MX_ERR_SHAPE: return "MX_ERR_SHAPE: extents not divisible by the block or the x4 container";
    case MX_ERR_ALIGNMENT: return "MX_ERR_ALIGNMENT: pointer or pitch not 16-byte aligned";
    case MX_ERR_WORKSPACE: return "MX_ERR_WORKSPACE: workspace missing or too small";
    case MX_ERR_CUDA: return "MX_ERR_CUDA: CUDA runtime error";
    case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT: a bounded device wait gave up";
    case MX_ERR_DEVICE: return "MX_ERR_DEVICE: current device is not sm_103a";
    case MX_ERR_SCALE_METHOD: return "MX_ERR_SCALE_METHOD: scale_method must be EMAX";
    }
    return "unknown mx_status";
}

int mx_version(void) { return 100; }

mx_status mx_debug_gemm_fault_injection(int skip_producer, uint64_t timeout_ns) {
    set_gemm_fault_injection(skip_producer, timeout_ns);
    return MX_OK;
}

mx_status mx_debug_set_gemm_variant(int variant) {
    if (variant < 0 || variant > 4) return MX_ERR_INVALID_ARG;
    set_gemm_variant(variant);
    return MX_OK;
}

mx_status mx_debug_last_gemm_launch(int* kernel, int* split_k) {
    if (!kernel || !split_k) return MX_ERR_INVALID_ARG;
    const GemmLaunchInfo info = last_gemm_launch();
    *kernel = info.kernel;
    *split_k = info.split_k;
    return MX_OK;
}

mx_status mx_debug_last_gemm_operands(int* a_mn_major, int* b_mn_major) {
    if (!a_mn_major || !b_mn_major) return MX_ERR_INVALID_ARG;
    const GemmLaunchInfo info = last_gemm_launch();
    *a_mn_major = info.a_mn_major;
    *b_mn_major = info.b_mn_major;
    return MX_OK;
}

}  // extern "C"
