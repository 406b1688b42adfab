// Internal helpers shared by the libpagedkv translation units (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "../../include/pagedkv.h"

// ---------------------------------------------------------------- host side
namespace pkv {

// Device address of the current device's sticky error word (0 = no error;
// otherwise the first pkv_status a kernel recorded). Cached per device.
// Returns nullptr if the runtime cannot resolve it.
int* error_word();

// Streaming multiprocessor count of the current device (cached per device).
int num_sms();

// Record a failed CUDA runtime call (message for pkv_last_error_string) and
// return PKV_ERR_CUDA.
int cuda_fail(const char* what, cudaError_t e);

// One-time per-(device, kernel) set-up: raise the kernel's dynamic shared
// memory limit to `smem` bytes and return its resident CTAs per SM for `threads`
// threads in *occupancy. Cached; thread-safe. Returns PKV_OK or PKV_ERR_CUDA.
int kernel_setup(const void* kernel, int smem, int threads, int* occupancy);

// Count one kernel launch of this library (see pkv_kernel_launches).
void note_launch();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with programmatic stream serialisation: the kernel's CTAs may be
// scheduled once every CTA of the previous launch in the stream has allowed it
// (launch_dependents) or exited. Every kernel launched this way calls
// wait_prerequisites() before it touches global memory (the merge of a split
// decode excepted: it reads only what was written before the decode launch
// began until it waits), and allows its own dependents only after that wait,
// so each launch still sees all earlier work complete: the ordering of plain
// launches, without their launch gaps. Used for the decode step's launches
// (block copies, slot writes, decode, merge); the chunked-prefill attention
// measured ~1% slower this way and keeps a plain launch.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pkv

// ---------------------------------------------------------------- device side
namespace pkv {

// Upper bound on any spin-wait in these kernels. A wait that runs past it records
// kErrTimeout and gives up instead of hanging the GPU; once that bit is set every
// other wait of the library on the device gives up at once.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s

// Bits of the device error word (pkv_get_device_error maps them to a status).
constexpr int kErrOutOfRange = 1;
constexpr int kErrTimeout = 2;
constexpr int kErrBadPairs = 4;      // copy_blocks: a destination repeated or also a source

__device__ __forceinline__ void flag_error(int* err, int bit) {
    if (err) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch. launch_dependents: a launch queued behind
// this one with programmatic stream serialisation may start once every CTA of
// this launch has executed it (or exited). wait_prerequisites: block until the
// launches this one depends on have completed and their memory is visible (a
// no-op for a launch made without that attribute).
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// The first statement of every kernel launched with launch_pdl (see there).
__device__ __forceinline__ void pdl_enter() {
    wait_prerequisites();
    launch_dependents();
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One try: the thread is parked (not spinning) until the phase completes or
// `suspend_ns` pass, whichever is first.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier to complete, for at most kWaitLimitNs
// (or until another wait has timed out). Each try parks the thread for up to
// 20 us, so waiting warps leave the issue slots to working ones.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, const int* err) {
    constexpr uint32_t kSuspendNs = 20000;
    if (mbar_try_wait(bar, parity, kSuspendNs)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity, kSuspendNs)) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
        if (err && (*reinterpret_cast<const volatile int*>(err) & kErrTimeout)) return false;
    }
}

// The same arrive and bulk copy, executed by a whole converged warp: one lane
// (elect.sync) performs it, so the operands can stay warp-uniform values.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// L2 policy for data read exactly once (K/V tiles): evict first.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared (TMA engine, no tensor map), completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void bulk_g2s_elect(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar, uint64_t policy) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;\n\t}" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

}  // namespace pkv
