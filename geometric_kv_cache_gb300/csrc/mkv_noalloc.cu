// mkv_compress_noalloc: the whole compression path for callers that cannot
// allocate device memory.
//
// Who needs it: code that receives only input/output pointers and a stream
// and has no allocator it may call -- a custom operator behind a C plugin
// interface of an inference engine, a runtime whose memory planner reserves
// all device memory up front and forbids allocations while serving, or a
// latency-critical path where cudaMalloc's implicit device synchronisation
// is not acceptable. mkv_compress needs a caller-provided workspace; this
// entry point instead uses a fixed scratch array that lives in the library's
// own device image.
//
// The scratch is a file-scope __device__ array of MKV_NOALLOC_SCRATCH_BYTES
// (32 MiB). Every GPU that loads the library holds it until the process
// exits, whether or not this entry point is called. Problems whose workspace
// (mkv_workspace_size) exceeds it are refused with MKV_ERR_UNSUPPORTED.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mkv_internal.h"

namespace {

// Zero-initialised when the module loads. Its first word is the device
// status word of the path; every successful call leaves it at zero again.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
mkv_status scratch_on_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MKV_OK;
}

}  // namespace

extern "C" mkv_status mkv_compress_noalloc(const void *K, const void *V, mkv_shape shape, double ratio,
                                           const int32_t *n_keep, mkv_mode mode, int32_t window,
                                           int32_t keep_stride, void *K_out, void *V_out, int32_t *idx,
                                           int32_t *kept, uint32_t *status_out, mkv_stream_t stream)
{
    const size_t need = mkv_workspace_size(shape, window);
    if (need > (size_t)MKV_NOALLOC_SCRATCH_BYTES) return MKV_ERR_UNSUPPORTED;
    if (status_out && (reinterpret_cast<uintptr_t>(status_out) % 4) != 0) return MKV_ERR_INVALID_ARG;
    void *scratch = nullptr;
    mkv_status rc = scratch_on_current_device(&scratch);
    if (rc != MKV_OK) return rc;
    // mkv_compress checks every argument (a bad shape also makes `need` 0)
    // before it enqueues anything.
    rc = mkv_compress(K, V, shape, ratio, n_keep, mode, window, keep_stride, K_out, V_out, idx, kept, scratch,
                      (size_t)MKV_NOALLOC_SCRATCH_BYTES, stream);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (rc == MKV_ERR_CUDA) {
        // kernels may have run and set status bits: try to leave the shared
        // word at zero so that the next call does not report them
        (void)cudaMemsetAsync(scratch, 0, sizeof(uint32_t), st);
        return rc;
    }
    if (rc != MKV_OK) return rc;
    if (status_out && cudaMemcpyAsync(status_out, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return MKV_ERR_CUDA;
    // Leave the status word at zero for the next call.
    if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), st) != cudaSuccess) return MKV_ERR_CUDA;
    return MKV_OK;
}
