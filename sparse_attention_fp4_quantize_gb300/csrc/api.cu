// Status strings, thread-local error detail and device-property caches.
#include <stdarg.h>
#include <string.h>

#include "common.cuh"
#include "tc.cuh"

namespace csa2 {

static thread_local char g_last_error[512] = "";

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
}

void clear_error() { g_last_error[0] = 0; }

static int cached_attr(cudaDeviceAttr attr, int *cache, int fallback) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fallback;
    if (cache[dev] <= 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess || v <= 0) return fallback;
        cache[dev] = v;
    }
    return cache[dev];
}

int num_sms() {
    static int cache[64];
    return cached_attr(cudaDevAttrMultiProcessorCount, cache, 148);
}

int max_smem_optin() {
    static int cache[64];
    return cached_attr(cudaDevAttrMaxSharedMemoryPerBlockOptin, cache, 227 * 1024);
}

}  // namespace csa2

namespace csa2 {
namespace {

// One CTA: an mbarrier expecting one arrival that never comes, waited on with
// the kernels' bounded wait; on giving up the CTA flags the timeout.
__global__ void bounded_wait_selftest_kernel(uint32_t max_polls, uint32_t *err_flag) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = tc::smem_u32(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);
        tc::mbar_init_fence();
    }
    __syncthreads();
    const bool ok = tc::mbar_wait(b, 0, max_polls);
    if (!ok && threadIdx.x == 0) flag_error(err_flag, CSA2_FLAG_TIMEOUT);
}

}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_selftest_bounded_wait(uint32_t max_polls, uint32_t *err_flag, csa2_stream_t stream) {
    csa2::clear_error();
    CSA2_REQUIRE(err_flag, "selftest_bounded_wait: err_flag required");
    CSA2_REQUIRE(max_polls >= 1 && max_polls <= (1u << 22), "selftest_bounded_wait: max_polls=%u not in [1, 2^22]",
                 max_polls);
    csa2::bounded_wait_selftest_kernel<<<1, 32, 0, csa2::stream_of(stream)>>>(max_polls, err_flag);
    CSA2_LAUNCH_CHECK("bounded_wait_selftest_kernel");
    return CSA2_OK;
}

extern "C" const char *csa2_status_string(csa2_status s) {
    switch (s) {
        case CSA2_OK: return "CSA2_OK";
        case CSA2_ERR_INVALID_ARG: return "CSA2_ERR_INVALID_ARG";
        case CSA2_ERR_UNSUPPORTED: return "CSA2_ERR_UNSUPPORTED";
        case CSA2_ERR_WORKSPACE: return "CSA2_ERR_WORKSPACE";
        case CSA2_ERR_CUDA: return "CSA2_ERR_CUDA";
        case CSA2_ERR_DEVICE_FLAG: return "CSA2_ERR_DEVICE_FLAG";
        case CSA2_ERR_TIMEOUT: return "CSA2_ERR_TIMEOUT";
    }
    return "CSA2_UNKNOWN_STATUS";
}

extern "C" const char *csa2_last_error(void) { return csa2::g_last_error; }

extern "C" int csa2_version(void) { return 100; }  // 0.1.0
