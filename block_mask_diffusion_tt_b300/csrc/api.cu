// api.cu -- status codes, error messages and small shared host utilities of libtt.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"

namespace {
thread_local char g_last_error[512] = "";
}

namespace tt {

tt_status fail(tt_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

tt_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return TT_OK;
    return fail(TT_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

int sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();  // clear; the caller reports a size of 0
        return 0;
    }
    if (dev < 64) cache[dev] = n;
    return n;
}

}  // namespace tt

extern "C" {

const char *tt_status_string(tt_status s) {
    switch (s) {
        case TT_OK: return "TT_OK";
        case TT_ERR_INVALID_ARG: return "TT_ERR_INVALID_ARG";
        case TT_ERR_UNSUPPORTED: return "TT_ERR_UNSUPPORTED";
        case TT_ERR_WORKSPACE: return "TT_ERR_WORKSPACE";
        case TT_ERR_CUDA: return "TT_ERR_CUDA";
        case TT_ERR_TIMEOUT: return "TT_ERR_TIMEOUT";
        case TT_ERR_CALLBACK: return "TT_ERR_CALLBACK";
        case TT_ERR_INTERNAL: return "TT_ERR_INTERNAL";
    }
    return "TT_ERR_UNKNOWN";
}

const char *tt_last_error(void) { return g_last_error; }

int32_t tt_abi_version(void) { return 1000; }

tt_status tt_workspace_zero(void *workspace, size_t bytes, tt_stream_t stream) {
    if (bytes == 0) return TT_OK;
    if (!workspace) return tt::fail(TT_ERR_INVALID_ARG, "tt_workspace_zero: null workspace");
    return tt::cuda_status(cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream),
                           "tt_workspace_zero");
}

}  // extern "C"
