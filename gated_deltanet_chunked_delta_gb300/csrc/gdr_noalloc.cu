// gdr_noalloc.cu -- a forward entry point for callers that cannot allocate
// device memory.
//
// gdr_fwd needs a caller-provided workspace.  Some callers have no way to
// provide one: a plugin running inside a host program that owns every byte of
// device memory and hands its plugins no allocator, or a latency-critical
// path where cudaMalloc (which may synchronise the device) is not allowed.
// gdr_fwd_noalloc serves them with a workspace that lives in this library's
// own device image: a fixed array that every GPU loading the library holds
// until the process exits.  The entry point itself calls no allocator.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "gdr.h"

namespace gdr {
int set_last_error(int code, const char *msg);
int fwd_check_and_size(const gdr_shape *shape, gdr_buf q, gdr_buf k, gdr_buf v, const float *g, const float *beta,
                       const float *h0, gdr_buf o, const float *final_state, const float *A, const float *h,
                       const gdr_opts *opts, size_t *need);
}

namespace {

// Fixed workspace of the allocation-free forward: 64 MiB per device.
constexpr size_t kNoallocBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoallocBytes];

constexpr int kMaxDevices = 64;
void *g_ws_addr[kMaxDevices];  // device address of g_noalloc_ws, per device
std::mutex g_ws_mu;

// Device address of the array on the current device, looked up once per
// device and kept for the life of the process.  A cudaDeviceReset() destroys
// the device's context and this library's device image with it; the address
// kept here is then stale, so the caller must not call gdr_fwd_noalloc on a
// device after resetting it.
int workspace_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return gdr::set_last_error(GDR_ERR_CUDA, "gdr_fwd_noalloc: no current CUDA device");
    }
    if (dev < 0 || dev >= kMaxDevices)
        return gdr::set_last_error(GDR_ERR_CUDA, "gdr_fwd_noalloc: device index out of range");
    std::lock_guard<std::mutex> lock(g_ws_mu);
    if (!g_ws_addr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_ws);
        if (e != cudaSuccess || !ptr) {
            cudaGetLastError();
            char msg[256];
            snprintf(msg, sizeof(msg), "gdr_fwd_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            return gdr::set_last_error(GDR_ERR_CUDA, msg);
        }
        g_ws_addr[dev] = ptr;
    }
    *out = g_ws_addr[dev];
    return GDR_OK;
}

}  // namespace

extern "C" GDR_API int gdr_fwd_noalloc(const gdr_shape *shape, gdr_buf q, gdr_buf k, gdr_buf v, const float *g,
                                       const float *beta, float scale, const float *h0, gdr_buf o,
                                       float *final_state, float *A, float *h, const gdr_opts *opts, void *stream) {
    // gdr_fwd's own checks, and the workspace of the plan this call takes (the
    // plan follows the input dtype: the tensor-core plan for bf16, the
    // CUDA-core plan with its fp32 tiles for fp32)
    size_t need = 0;
    const int bad = gdr::fwd_check_and_size(shape, q, k, v, g, beta, h0, o, final_state, A, h, opts, &need);
    if (bad) return bad;  // the message is already set
    if (need > kNoallocBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "gdr_fwd_noalloc: this problem needs %zu workspace bytes, more than the fixed %zu; use gdr_fwd",
                 need, kNoallocBytes);
        return gdr::set_last_error(GDR_ERR_WORKSPACE, msg);
    }
    void *ws = nullptr;
    const int rc = workspace_address(&ws);
    if (rc) return rc;
    // Every kernel writes each workspace byte it later reads within the same
    // call, so nothing left from an earlier call needs clearing.
    return gdr_fwd(shape, q, k, v, g, beta, scale, h0, o, final_state, A, h, ws, kNoallocBytes, opts, stream);
}
