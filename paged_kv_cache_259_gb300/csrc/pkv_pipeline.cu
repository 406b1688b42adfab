// Stream and event plumbing of a pipelined step (host code only): the copy of
// one step's packed inputs to the device on an upload stream, ordered before
// the step's kernels on the compute stream, and the read-back of its output on
// a download stream once the kernels are done -- each as one call, so a host
// loop that feeds one step after another spends its time on the steps, not on
// the runtime calls between them.
#include <cuda_runtime.h>

#include "pkv_internal.cuh"

extern "C" {

int pkv_stage_upload(const void* host_src, void* dev_dst, size_t bytes, void* up_stream,
                     void* compute_stream, void* uploaded_event, void* reuse_computed_event,
                     void* reuse_downloaded_event) {
    using namespace pkv;
    if (!host_src || !dev_dst || !uploaded_event || bytes == 0) return PKV_ERR_INVALID_ARG;
    cudaStream_t up = static_cast<cudaStream_t>(up_stream);
    cudaStream_t comp = static_cast<cudaStream_t>(compute_stream);
    cudaError_t e = cudaSuccess;
    // the buffer set is reused: its previous step's kernels have read it
    if (reuse_computed_event)
        e = cudaStreamWaitEvent(up, static_cast<cudaEvent_t>(reuse_computed_event), 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dev_dst, host_src, bytes, cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess) e = cudaEventRecord(static_cast<cudaEvent_t>(uploaded_event), up);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(comp, static_cast<cudaEvent_t>(uploaded_event), 0);
    // ... and its previous output has been read back before it is overwritten
    if (e == cudaSuccess && reuse_downloaded_event)
        e = cudaStreamWaitEvent(comp, static_cast<cudaEvent_t>(reuse_downloaded_event), 0);
    return e == cudaSuccess ? PKV_OK : cuda_fail("pkv_stage_upload", e);
}

int pkv_stage_download(const void* dev_src, void* host_dst, size_t bytes, void* compute_stream,
                       void* down_stream, void* computed_event, void* downloaded_event) {
    using namespace pkv;
    if (!dev_src || !host_dst || !computed_event || !downloaded_event || bytes == 0)
        return PKV_ERR_INVALID_ARG;
    cudaStream_t comp = static_cast<cudaStream_t>(compute_stream);
    cudaStream_t down = static_cast<cudaStream_t>(down_stream);
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(computed_event), comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(down, static_cast<cudaEvent_t>(computed_event), 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(host_dst, dev_src, bytes, cudaMemcpyDeviceToHost, down);
    if (e == cudaSuccess) e = cudaEventRecord(static_cast<cudaEvent_t>(downloaded_event), down);
    return e == cudaSuccess ? PKV_OK : cuda_fail("pkv_stage_download", e);
}

}  // extern "C"
