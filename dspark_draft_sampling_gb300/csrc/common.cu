// Error state, version string and device queries for libdspark.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "common.cuh"

namespace dspark {

static thread_local char g_last_error[512] = "";

dspark_status fail(dspark_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

dspark_status cuda_fail(cudaError_t e, const char *what) {
    return fail(DSPARK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

void clear_error() { g_last_error[0] = '\0'; }

int current_sm_count(int *sm_count) {
    static int cached[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(cuda_fail(e, "cudaGetDevice"));
    if (dev >= 0 && dev < 64 && cached[dev] > 0) {
        *sm_count = cached[dev];
        return DSPARK_OK;
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return static_cast<int>(cuda_fail(e, "cudaDeviceGetAttribute(SM count)"));
    if (dev >= 0 && dev < 64) cached[dev] = n;
    *sm_count = n;
    return DSPARK_OK;
}

}  // namespace dspark

extern "C" const char *dspark_last_error(void) { return dspark::g_last_error; }

extern "C" const char *dspark_version(void) { return "libdspark 0.1 sm_103a"; }
