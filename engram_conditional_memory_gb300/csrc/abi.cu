// Library-wide parts of the Engram C ABI: status strings, per-thread error text,
// device facts, pointer checks and the library's device status word.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "engram_internal.cuh"

// OR-ed by kernels (ENGRAM_DEVERR_* bits); one copy per device that loads the library.
__device__ uint32_t g_engram_status_word;

namespace engram {

namespace {

thread_local char t_last_error[512] = "";
std::atomic<int32_t> g_validation{1};
std::atomic<int32_t> g_max_ctas{0};
std::atomic<int32_t> g_pdl{1};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
bool g_dev_ready[kMaxDevices];
DeviceInfo g_dev_info[kMaxDevices];

}  // namespace

bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }

engram_status fail(engram_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return st;
}

engram_status current_device(DeviceInfo *info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(ENGRAM_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DeviceInfo d{};
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
                cudaSuccess ||
            (e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status_word), g_engram_status_word)) !=
                cudaSuccess)
            return fail(ENGRAM_ERR_CUDA, "device %d query: %s", dev, cudaGetErrorString(e));
        g_dev_info[dev] = d;
        g_dev_ready[dev] = true;
    }
    *info = g_dev_info[dev];
    return ENGRAM_OK;
}

engram_status check_device_ptr(const void *p, int device, const char *name) {
    if (g_validation.load(std::memory_order_relaxed) == 0 || p == nullptr) return ENGRAM_OK;
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error state of the query
        return fail(ENGRAM_ERR_DEVICE, "%s: not a CUDA pointer (%s)", name, cudaGetErrorString(e));
    }
    if (a.type == cudaMemoryTypeManaged) return ENGRAM_OK;
    if (a.type != cudaMemoryTypeDevice || a.device != device)
        return fail(ENGRAM_ERR_DEVICE, "%s: not device memory of device %d (type %d, device %d)", name, device,
                    static_cast<int>(a.type), a.device);
    return ENGRAM_OK;
}

engram_status check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
    return ENGRAM_OK;
}

int64_t cap_grid(int64_t grid) {
    const int32_t cap = g_max_ctas.load(std::memory_order_relaxed);
    if (cap > 0 && grid > cap) grid = cap;
    return grid < 1 ? 1 : grid;
}

engram_status set_smem(const void *kernel, int bytes) {
    // The attribute is per kernel and per device; setting it again is harmless.
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "cudaFuncSetAttribute(%d B): %s", bytes, cudaGetErrorString(e));
    return ENGRAM_OK;
}

}  // namespace engram

namespace engram {

// The failure-detection self-check: one CTA waits, with the pipelines' own bounded wait, on an
// mbarrier that nothing ever completes (no copy, no arrival is pending on it), gives up after
// limit_ns and reports ENGRAM_DEVERR_TIMEOUT like a pipeline would.
__global__ void wait_timeout_check_kernel(uint64_t limit_ns, uint32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, limit_ns);
    if (__syncthreads_or(!ok) && threadIdx.x == 0) report(status, nullptr, ENGRAM_DEVERR_TIMEOUT);
}

}  // namespace engram

using namespace engram;

extern "C" {

engram_status engram_check_wait_timeout(uint32_t limit_us, engram_stream_t stream) {
    if (limit_us < 1 || limit_us > 2000000)
        return fail(ENGRAM_ERR_SHAPE, "engram_check_wait_timeout: limit_us = %u (1 .. 2000000)", limit_us);
    DeviceInfo dev;
    engram_status st = current_device(&dev);
    if (st != ENGRAM_OK) return st;
    wait_timeout_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint64_t>(limit_us) * 1000u, dev.status_word);
    return check_launch("engram_check_wait_timeout");
}

int32_t engram_abi_version(void) { return ENGRAM_ABI_VERSION; }

const char *engram_status_string(engram_status status) {
    switch (status) {
        case ENGRAM_OK: return "ok";
        case ENGRAM_ERR_NULL: return "a required pointer is NULL";
        case ENGRAM_ERR_SHAPE: return "invalid size";
        case ENGRAM_ERR_DTYPE: return "invalid dtype";
        case ENGRAM_ERR_ALIGN: return "tensor or row not 16-byte aligned";
        case ENGRAM_ERR_CUDA: return "CUDA runtime error";
        case ENGRAM_ERR_INDEX: return "device-side error bit set";
        case ENGRAM_ERR_DEVICE: return "pointer is not device memory of the current device";
    }
    return "unknown status";
}

const char *engram_last_error_string(void) { return t_last_error; }

int32_t engram_set_validation(int32_t level) { return g_validation.exchange(level != 0 ? 1 : 0); }

int32_t engram_set_max_ctas(int32_t max_ctas) { return g_max_ctas.exchange(max_ctas > 0 ? max_ctas : 0); }

int32_t engram_set_pdl(int32_t on) { return g_pdl.exchange(on != 0 ? 1 : 0); }

static engram_status read_error_word(const char *fn, const uint32_t *err_word, engram_stream_t stream,
                                     uint32_t *host_out) {
    if (!err_word || !host_out) return fail(ENGRAM_ERR_NULL, "%s: NULL argument", fn);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(host_out, err_word, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    return *host_out ? ENGRAM_ERR_INDEX : ENGRAM_OK;
}

engram_status engram_read_error_word(const uint32_t *err_word, engram_stream_t stream, uint32_t *host_out) {
    return read_error_word("engram_read_error_word", err_word, stream, host_out);
}

engram_status engram_get_error(const uint32_t *err_word, engram_stream_t stream, uint32_t *host_out) {
    return read_error_word("engram_get_error", err_word, stream, host_out);
}

engram_status engram_device_status(uint32_t *host_out, int32_t clear) {
    if (!host_out) return fail(ENGRAM_ERR_NULL, "engram_device_status: NULL argument");
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(host_out, g_engram_status_word, sizeof(uint32_t));
    if (e == cudaSuccess && clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_engram_status_word, &zero, sizeof(uint32_t));
    }
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_device_status: %s", cudaGetErrorString(e));
    return *host_out ? ENGRAM_ERR_INDEX : ENGRAM_OK;
}

}  // extern "C"
