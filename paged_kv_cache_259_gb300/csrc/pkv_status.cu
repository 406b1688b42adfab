// Status strings, the device error word and per-device caches.
#include <atomic>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "pkv_internal.cuh"

// Sticky error bits (pkv::kErr*) recorded by any kernel of this library on this device.
__device__ int g_pkv_error_word;

namespace pkv {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int*> g_err_ptr[kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];
}  // namespace

int* error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int* p = g_err_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_pkv_error_word);
    if (e != cudaSuccess) {
        cuda_fail("error word address", e);
        return nullptr;
    }
    g_err_ptr[dev].store(static_cast<int*>(addr), std::memory_order_release);
    return static_cast<int*>(addr);
}

namespace {
thread_local char g_last_error[256] = "";
}

int cuda_fail(const char* what, cudaError_t e) {
    (void)cudaGetLastError();   // leave no stale (non-sticky) error for the caller's next check
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
    return PKV_ERR_CUDA;
}

int kernel_setup(const void* kernel, int smem, int threads, int* occupancy) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> done;   // (device, kernel) -> occupancy
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("kernel set-up: current device", e);
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({dev, kernel});
    if (it != done.end()) {
        *occupancy = it->second;
        return PKV_OK;
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail("kernel set-up: max dynamic shared memory", e);
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem);
    if (e != cudaSuccess) return cuda_fail("kernel set-up: occupancy query", e);
    done[{dev, kernel}] = occ;
    *occupancy = occ;
    return PKV_OK;
}

namespace {
std::atomic<unsigned long long> g_launches{0};
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = g_sms[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev].store(n, std::memory_order_relaxed);
    return n;
}

// One thread waits, bounded, on a barrier that nothing arrives at: the wait
// gives up after kWaitLimitNs and records kErrTimeout, as a stuck wait in any
// kernel of the library would.
__global__ void wait_timeout_kernel(int* err) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t a = smem_addr(&bar);
    mbar_init(a, 1);
    if (!mbar_wait_bounded(a, 0, err)) flag_error(err, kErrTimeout);
}

}  // namespace pkv

extern "C" {

int pkv_check_wait_timeout(void* stream) {
    int* err = pkv::error_word();
    if (!err) return PKV_ERR_CUDA;
    pkv::wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(err);
    pkv::note_launch();
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail("pkv_check_wait_timeout: kernel launch", e);
}

const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        case PKV_ERR_OUT_OF_RANGE: return "index out of range";
        case PKV_ERR_POOL_EXHAUSTED: return "block pool exhausted";
        case PKV_ERR_TIMEOUT: return "device wait timed out";
        default: return "unknown status";
    }
}

const char* pkv_last_error_string(void) { return pkv::g_last_error; }

unsigned long long pkv_kernel_launches(void) {
    return pkv::g_launches.load(std::memory_order_relaxed);
}

int pkv_get_device_error(int* code, void* stream) {
    if (!code) return PKV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* p = pkv::error_word();
    if (!p) return PKV_ERR_CUDA;
    int host = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&host, p, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return pkv::cuda_fail("pkv_get_device_error", e);
    *code = (host & pkv::kErrTimeout) ? PKV_ERR_TIMEOUT
            : (host & pkv::kErrOutOfRange) ? PKV_ERR_OUT_OF_RANGE
            : (host & pkv::kErrBadPairs) ? PKV_ERR_INVALID_ARG : PKV_OK;
    return PKV_OK;
}

}  // extern "C"
