// fd_static_ws.cu -- fd_decode for callers that must not allocate device memory.
//
// Some callers run attention at a point where they cannot call cudaMalloc:
// the enqueue step of an inference-engine plugin, a runtime whose device
// memory is planned up front and handed out by someone else, or any code path
// that is not allowed to grow the process's memory.  For them this file keeps
// the scratch fd_decode needs (status word, merge tickets, split partials) in
// a fixed device array inside the library, so the caller passes only inputs
// and outputs.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fd.h"

namespace {

// The scratch of every fd_decode_static_workspace call.  Every GPU that loads
// the library holds these FD_STATIC_WORKSPACE_BYTES until the process exits.
__device__ __align__(256) unsigned char g_static_workspace[FD_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// In host code g_static_workspace names a host-side stand-in, not device
// memory: the device address is looked up once per device, with that device
// current, and cached.
int static_workspace(void **ptr)
{
    static std::mutex lock;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FD_ERR_CUDA;
    std::lock_guard<std::mutex> guard(lock);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p)
            return FD_ERR_CUDA;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return FD_OK;
}

}  // namespace

extern "C" int fd_decode_static_workspace(int batch, int num_qo_heads, int num_kv_heads,
                                          int head_dim, const int32_t *kv_indptr_host,
                                          const int32_t *kv_indptr_dev, const void *q,
                                          const void *k, const void *v, float scale, float *o,
                                          float *lse, void *stream)
{
    fd_plan_info info;
    int rc = fd_plan(batch, num_qo_heads, num_kv_heads, head_dim, kv_indptr_host, 0, 0, 0, &info);
    if (rc != FD_OK)
        return rc;
    if (info.workspace_bytes > FD_STATIC_WORKSPACE_BYTES)
        return FD_ERR_WORKSPACE;   // too large for the fixed array: use fd_decode
    void *ws = nullptr;
    if ((rc = static_workspace(&ws)) != FD_OK)
        return rc;
    // The array keeps the previous call's contents; the status word and the
    // merge tickets must start at zero.
    const size_t tickets = ((size_t)batch * num_kv_heads * 4 + 255) / 256 * 256;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, FD_WORKSPACE_HEADER_BYTES + tickets, s) != cudaSuccess)
        return FD_ERR_CUDA;
    return fd_decode(batch, num_qo_heads, num_kv_heads, head_dim, kv_indptr_host, kv_indptr_dev,
                     q, k, v, scale, o, lse, ws, FD_STATIC_WORKSPACE_BYTES, stream);
}
