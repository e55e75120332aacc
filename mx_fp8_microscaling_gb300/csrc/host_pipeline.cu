// QuantizeMX from host memory to host memory, pipelined.
//
// The rows are cut into chunks; chunk i goes through a ring of device slots:
// its input is copied in on a host-to-device copy stream, quantized on the
// caller's stream, and its codes and scales are copied out on a
// device-to-host copy stream.  Events order the three so that chunk i+1 is
// copied in and chunk i-1 copied out while chunk i is quantized, and a slot is
// refilled only after its previous output has left.  With pinned host memory
// both copy directions and the kernel run at the same time.
//
// The copy streams and events are per device and shared by all calls; a
// mutex serialises the enqueueing.  Nothing here allocates device memory: the
// slots live in the caller's workspace.

#include <cstdint>
#include <mutex>

#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kSlots = 3;

struct CopyEngines {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t entry = nullptr;
    cudaEvent_t in_done[kSlots] = {}, q_done[kSlots] = {}, out_done[kSlots] = {};
};

std::mutex g_pipe_mutex;
CopyEngines g_engines[64];

cudaError_t engines_for_current_device(CopyEngines** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    CopyEngines& c = g_engines[dev];
    if (!c.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&c.entry, ef)) != cudaSuccess) return e;
        for (int k = 0; k < kSlots; ++k) {
            if ((e = cudaEventCreateWithFlags(&c.in_done[k], ef)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&c.q_done[k], ef)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&c.out_done[k], ef)) != cudaSuccess) return e;
        }
        c.ready = true;
    }
    *out = &c;
    return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Geometry of one pipelined call.
struct HostPlan {
    int64_t chunk_rows = 0;      // rows per chunk (the last may be shorter)
    int64_t block_rows = 1;      // rows per scale row
    int64_t scale_cols = 0;      // bytes per scale-buffer row
    int64_t chunk_scale_rows = 0;  // scale-buffer rows a full chunk owns
    size_t in_bytes = 0, data_bytes = 0, scale_bytes = 0, slot_bytes = 0;
    bool fp4 = false, interleave = false;
};

mx_status plan_host(mx_dtype in_dtype, int64_t rows, int64_t cols, mx_dtype out_dtype, const mx_quant_cfg* cfg,
                    int64_t chunk_rows, HostPlan* P) {
    mx_quant_cfg c;
    if (cfg) c = *cfg;
    else mx_quant_cfg_default(&c);
    mx_status st = mx_quantize_sizes(in_dtype, out_dtype, rows, cols, &c, nullptr, nullptr, nullptr, nullptr);
    if (st != MX_OK) return st;
    if (chunk_rows < 0) return MX_ERR_INVALID_ARG;
    HostPlan p;
    // rows per scale row: the block's extent along rows
    const bool g1x32 = c.geometry == MX_GEOM_1X32;
    const int dim = c.dim >= 0 ? c.dim - 2 : c.dim;  // 1 / 0 of a 2-D view fold to -1 / -2
    p.block_rows = g1x32 ? (dim == -2 ? 32 : 1) : (dim == -2 ? 8 : 4);
    // chunks start on a whole scale row (plain), a whole 4-row interleave
    // group or a whole 128-row SF tile, so each chunk's piece of the scale
    // buffer is contiguous
    const int64_t group = c.scale_layout == MX_SCALE_TC_SF ? 128 : (c.scale_layout == MX_SCALE_INTERLEAVE32 ? 4 : 1);
    const int64_t granule = group * p.block_rows;
    if (chunk_rows == 0) {
        // about 16 MiB of input: measured faster than 8 MiB on a 128 MiB
        // input (fewer copies and events per call; the fill and drain of
        // each call stay short)
        const int64_t target = (int64_t(16) << 20) / (cols > 0 ? cols * 2 : 1);
        chunk_rows = target / granule * granule;
        if (chunk_rows < granule) chunk_rows = granule;
    } else if (chunk_rows % granule != 0) {
        return MX_ERR_SHAPE;
    }
    // a tensor shorter than a chunk needs slots of its own size only
    const int64_t whole = (rows + granule - 1) / granule * granule;
    if (whole > 0 && whole < chunk_rows) chunk_rows = whole;
    p.chunk_rows = chunk_rows;
    int64_t srows = 0, scols = 0;
    size_t dbytes = 0, sbytes = 0;
    st = mx_quantize_sizes(in_dtype, out_dtype, chunk_rows, cols, &c, &dbytes, &srows, &scols, &sbytes);
    if (st != MX_OK) return st;
    p.scale_cols = scols;
    p.chunk_scale_rows = srows;
    p.in_bytes = static_cast<size_t>(chunk_rows * cols * 2);
    p.data_bytes = dbytes;
    p.scale_bytes = sbytes;
    p.slot_bytes = align256(p.in_bytes) + align256(p.data_bytes) + align256(p.scale_bytes);
    p.fp4 = out_dtype == MX_E2M1;
    p.interleave = c.scale_layout == MX_SCALE_INTERLEAVE32;
    *P = p;
    return MX_OK;
}

// Chunks of several jobs stream through the same slot ring, so consecutive
// tensors overlap (no drain between them).
mx_status run_pipeline(const mx_host_quant_job* jobs, const HostPlan* plans, int njobs, void* workspace,
                       size_t slot_bytes, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    CopyEngines* E = nullptr;
    if (engines_for_current_device(&E) != cudaSuccess) return MX_ERR_CUDA;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // the workspace may still be in use by earlier work on the caller's stream
    if (!ok(cudaEventRecord(E->entry, s)) || !ok(cudaStreamWaitEvent(E->h2d, E->entry, 0))) return MX_ERR_CUDA;
    int64_t chunk_no = 0;
    int last_slot = -1;
    for (int jn = 0; jn < njobs; ++jn) {
        const mx_host_quant_job& J = jobs[jn];
        const HostPlan& P = plans[jn];
        if (J.rows == 0 || J.cols == 0) continue;
        const uint8_t* in = static_cast<const uint8_t*>(J.in_host);
        uint8_t* out_data = static_cast<uint8_t*>(J.out_data_host);
        uint8_t* out_scale = static_cast<uint8_t*>(J.out_scale_host);
        const int64_t nchunks = (J.rows + P.chunk_rows - 1) / P.chunk_rows;
        const int64_t data_row_bytes = P.fp4 ? J.cols / 2 : J.cols;
        for (int64_t i = 0; i < nchunks; ++i, ++chunk_no) {
            const int k = static_cast<int>(chunk_no % kSlots);
            uint8_t* d_in = static_cast<uint8_t*>(workspace) + k * slot_bytes;
            uint8_t* d_data = d_in + align256(P.in_bytes);
            uint8_t* d_scale = d_data + align256(P.data_bytes);
            const int64_t r0 = i * P.chunk_rows;
            const int64_t n = J.rows - r0 < P.chunk_rows ? J.rows - r0 : P.chunk_rows;

            // in: after the slot's previous output has been copied out
            if (!ok(cudaStreamWaitEvent(E->h2d, E->out_done[k], 0)) ||
                !ok(cudaMemcpy2DAsync(d_in, static_cast<size_t>(J.cols * 2), in + r0 * J.ld_in * 2,
                                      static_cast<size_t>(J.ld_in * 2), static_cast<size_t>(J.cols * 2),
                                      static_cast<size_t>(n), cudaMemcpyHostToDevice, E->h2d)) ||
                !ok(cudaEventRecord(E->in_done[k], E->h2d)))
                return MX_ERR_CUDA;
            // quantize on the caller's stream
            if (!ok(cudaStreamWaitEvent(s, E->in_done[k], 0))) return MX_ERR_CUDA;
            mx_status st = mx_quantize(d_in, J.in_dtype, n, J.cols, J.cols, J.out_dtype, &J.cfg, d_data, d_scale,
                                       reinterpret_cast<mx_stream>(s));
            if (st != MX_OK) return st;
            if (!ok(cudaEventRecord(E->q_done[k], s))) return MX_ERR_CUDA;
            // out: codes, then the chunk's piece of the scale buffer
            int64_t srows = 0;
            if (mx_quantize_sizes(J.in_dtype, J.out_dtype, n, J.cols, &J.cfg, nullptr, &srows, nullptr, nullptr) !=
                MX_OK)
                return MX_ERR_INVALID_ARG;
            uint8_t* h_scale = out_scale + i * P.chunk_scale_rows * P.scale_cols;
            if (!ok(cudaStreamWaitEvent(E->d2h, E->q_done[k], 0)) ||
                !ok(cudaMemcpyAsync(out_data + r0 * data_row_bytes, d_data, static_cast<size_t>(n * data_row_bytes),
                                    cudaMemcpyDeviceToHost, E->d2h)))
                return MX_ERR_CUDA;
            cudaError_t e;
            if (P.interleave) {
                // scale row j lives at buffer row (j & 3) + 32 (j >> 2): the first
                // 4 rows of every 32 (fewer in a last, partial group); the others
                // stay untouched in the caller's buffer
                const int64_t live = n / P.block_rows;
                const size_t pitch = static_cast<size_t>(32 * P.scale_cols);
                e = cudaSuccess;
                if (live / 4 > 0)
                    e = cudaMemcpy2DAsync(h_scale, pitch, d_scale, pitch, static_cast<size_t>(4 * P.scale_cols),
                                          static_cast<size_t>(live / 4), cudaMemcpyDeviceToHost, E->d2h);
                if (e == cudaSuccess && live % 4 != 0)
                    e = cudaMemcpyAsync(h_scale + (live / 4) * pitch, d_scale + (live / 4) * pitch,
                                        static_cast<size_t>((live % 4) * P.scale_cols), cudaMemcpyDeviceToHost,
                                        E->d2h);
            } else {
                e = cudaMemcpyAsync(h_scale, d_scale, static_cast<size_t>(srows * P.scale_cols),
                                    cudaMemcpyDeviceToHost, E->d2h);
            }
            if (!ok(e) || !ok(cudaEventRecord(E->out_done[k], E->d2h))) return MX_ERR_CUDA;
            last_slot = k;
        }
    }
    // the caller's stream continues once the last copy out has finished (the
    // copy stream runs in order)
    if (last_slot >= 0 && !ok(cudaStreamWaitEvent(s, E->out_done[last_slot], 0))) return MX_ERR_CUDA;
    return MX_OK;
}

// Plans every job; the slot size is the largest job's.
mx_status plan_jobs(const mx_host_quant_job* jobs, int njobs, int64_t chunk_rows, HostPlan* plans,
                    size_t* slot_bytes) {
    if (njobs < 0 || (njobs > 0 && !jobs) || !plans) return MX_ERR_INVALID_ARG;
    size_t slot = 0;
    for (int i = 0; i < njobs; ++i) {
        mx_status st = plan_host(jobs[i].in_dtype, jobs[i].rows, jobs[i].cols, jobs[i].out_dtype, &jobs[i].cfg,
                                 chunk_rows, &plans[i]);
        if (st != MX_OK) return st;
        if (plans[i].slot_bytes > slot) slot = plans[i].slot_bytes;
    }
    *slot_bytes = slot;
    return MX_OK;
}

mx_status check_jobs(const mx_host_quant_job* jobs, int njobs) {
    for (int i = 0; i < njobs; ++i) {
        const mx_host_quant_job& J = jobs[i];
        if (J.ld_in < J.cols) return MX_ERR_INVALID_ARG;
        if (J.rows == 0 || J.cols == 0) continue;
        if (!J.in_host || !J.out_data_host || !J.out_scale_host) return MX_ERR_INVALID_ARG;
    }
    return MX_OK;
}

}  // namespace
}  // namespace mx

using namespace mx;

extern "C" {

mx_status mx_quantize_host_batch_workspace(const mx_host_quant_job* jobs, int njobs, int64_t chunk_rows,
                                           size_t* bytes) {
    if (njobs > 4096) return MX_ERR_INVALID_ARG;
    HostPlan plans[1];
    HostPlan* P = njobs <= 1 ? plans : new HostPlan[njobs];
    size_t slot = 0;
    mx_status st = plan_jobs(jobs, njobs, chunk_rows, P, &slot);
    if (P != plans) delete[] P;
    if (st != MX_OK) return st;
    if (!bytes) return MX_ERR_INVALID_ARG;
    *bytes = kSlots * slot;
    return MX_OK;
}

mx_status mx_quantize_host_batch(const mx_host_quant_job* jobs, int njobs, int64_t chunk_rows, void* workspace,
                                 size_t workspace_bytes, mx_stream stream) {
    if (njobs > 4096) return MX_ERR_INVALID_ARG;
    HostPlan plans[1];
    HostPlan* P = njobs <= 1 ? plans : new HostPlan[njobs];
    size_t slot = 0;
    mx_status st = plan_jobs(jobs, njobs, chunk_rows, P, &slot);
    if (st == MX_OK) st = check_jobs(jobs, njobs);
    bool any = false;
    for (int i = 0; st == MX_OK && i < njobs; ++i) any = any || (jobs[i].rows > 0 && jobs[i].cols > 0);
    if (st == MX_OK && any) {
        if (!workspace || workspace_bytes < kSlots * slot) st = MX_ERR_WORKSPACE;
        else if (reinterpret_cast<uintptr_t>(workspace) & 255u) st = MX_ERR_ALIGNMENT;
        else if (!device_is_sm103()) st = MX_ERR_DEVICE;
        else st = run_pipeline(jobs, P, njobs, workspace, slot, reinterpret_cast<cudaStream_t>(stream));
    }
    if (P != plans) delete[] P;
    return st;
}

mx_status mx_quantize_host_workspace(mx_dtype in_dtype, int64_t rows, int64_t cols, mx_dtype out_dtype,
                                     const mx_quant_cfg* cfg, int64_t chunk_rows, size_t* bytes) {
    mx_host_quant_job j{};
    j.in_dtype = in_dtype;
    j.rows = rows;
    j.cols = cols;
    j.ld_in = cols;
    j.out_dtype = out_dtype;
    if (cfg) j.cfg = *cfg;
    else mx_quant_cfg_default(&j.cfg);
    return mx_quantize_host_batch_workspace(&j, 1, chunk_rows, bytes);
}

mx_status mx_quantize_host(const void* in_host, mx_dtype in_dtype, int64_t rows, int64_t cols, int64_t ld_in,
                           mx_dtype out_dtype, const mx_quant_cfg* cfg, void* out_data_host, void* out_scale_host,
                           int64_t chunk_rows, void* workspace, size_t workspace_bytes, mx_stream stream) {
    mx_host_quant_job j{};
    j.in_host = in_host;
    j.in_dtype = in_dtype;
    j.rows = rows;
    j.cols = cols;
    j.ld_in = ld_in;
    j.out_dtype = out_dtype;
    if (cfg) j.cfg = *cfg;
    else mx_quant_cfg_default(&j.cfg);
    j.out_data_host = out_data_host;
    j.out_scale_host = out_scale_host;
    return mx_quantize_host_batch(&j, 1, chunk_rows, workspace, workspace_bytes, stream);
}

}  // extern "C"
