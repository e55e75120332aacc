// mx_scaled_matmul_noalloc: ScaledMatmul with plain E8M0 scales for callers
// that cannot allocate device memory.
//
// mx_scaled_matmul with plain scales needs scratch space for the two scale
// tensors in the tensor-core layout, which the caller normally passes as a
// workspace.  Some callers have no way to obtain one: a plugin invoked by a
// host runtime that owns all device memory and offers it no allocator, or a
// latency-critical path that must not call cudaMalloc (which can synchronise
// the device).  For them this entry point keeps its scratch in a fixed
// file-scope device array instead, and calls no allocating routine.
//
// The array is MX_NOALLOC_SCRATCH_BYTES (4 MiB); every device that loads this
// library holds it until the process exits.  All calls share it, so calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on it; calls on one stream, or otherwise ordered, are safe.  Each
// call overwrites every scratch byte it reads (the repack writes padding too),
// so nothing needs clearing between calls.

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "mx.h"
#include "mx_internal.h"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MX_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current; the first call on a device does
// this look-up (make it before any stream capture).
mx_status scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return MX_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return MX_OK;
}

}  // namespace

extern "C" mx_status mx_scaled_matmul_noalloc(const void* a, const void* bt, const uint8_t* a_scale,
                                              const uint8_t* b_scale, mx_dtype elem_dtype, int64_t M, int64_t N,
                                              int64_t K, mx_dtype out_dtype, void* c, int64_t ldc,
                                              mx_stream stream) {
    if (M < 0 || N < 0 || K < 0) return MX_ERR_INVALID_ARG;
    if (K % 32 != 0) return MX_ERR_SHAPE;
    const size_t need = round16(mx::sf_layout_bytes(M, K)) + round16(mx::sf_layout_bytes(N, K));
    if (need > static_cast<size_t>(MX_NOALLOC_SCRATCH_BYTES)) return MX_ERR_WORKSPACE;
    if (M == 0 || N == 0) return MX_OK;
    if (!mx::device_is_sm103()) return MX_ERR_DEVICE;
    void* scratch = nullptr;
    mx_status st = scratch_on_current_device(&scratch);
    if (st != MX_OK) return st;
    return mx_scaled_matmul(a, bt, a_scale, b_scale, 0, elem_dtype, M, N, K, out_dtype, c, ldc, scratch,
                            MX_NOALLOC_SCRATCH_BYTES, stream);
}
