// Stream and event plumbing of a pipelined step (host code only): the copy of
// one step's packed inputs to the device on an upload stream, ordered before
// the step's kernels on the compute stream, and the read-back of its output on
// a download stream once the kernels are done -- each as one call, so a host
// loop that feeds one step after another spends its time on the steps, not on
// the runtime calls between them.
#include <chrono>

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

int pkv_decode_pipeline_step(const pkv_decode_pipeline_step_args* a, int reuse, void* host_out,
                             int* counts, double* plan_us) {
    using namespace pkv;
    if (!a || !host_out) return PKV_ERR_INVALID_ARG;
    const bool grouped = a->max_members >= 1;
    int pairs = 0, groups = 0, ungrouped = 0, longest = 0;
    const auto t0 = std::chrono::steady_clock::now();
    int st = bm_plan_decode(a->bm, a->seq_ids, a->num_seqs, a->max_blocks, a->h_slots, a->h_pairs,
                            &pairs, a->h_tables, a->h_lens, grouped ? a->max_members : 0,
                            grouped ? a->h_group_members : nullptr,
                            grouped ? a->h_group_prefix : nullptr,
                            grouped ? a->h_seq_group : nullptr, grouped ? a->group_blocks : nullptr,
                            grouped ? a->h_ungrouped : nullptr, &groups, &ungrouped, &longest);
    if (plan_us)
        *plan_us = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0)
                       .count();
    if (counts) {
        counts[0] = pairs;
        counts[1] = groups;
        counts[2] = ungrouped;
        counts[3] = longest;
    }
    if (st != PKV_OK) return st;
    st = pkv_stage_upload(a->host_slab, a->dev_slab, a->slab_bytes, a->up_stream, a->compute_stream,
                          a->uploaded_event, reuse ? a->computed_event : nullptr,
                          reuse ? a->downloaded_event : nullptr);
    if (st != PKV_OK) return st;
    st = paged_decode_step(a->pairs, pairs, a->k_new, a->v_new, a->slots, a->out, a->q, a->k_pool,
                           a->v_pool, a->tables, a->lens, a->num_seqs, a->max_blocks, a->num_blocks,
                           a->num_heads, a->num_kv_heads, a->head_dim, a->block_size, a->scale,
                           a->q_dtype, a->kv_dtype, a->k_scale, a->v_scale,
                           grouped ? a->seq_group : nullptr, grouped ? a->group_members : nullptr,
                           grouped ? a->group_prefix : nullptr, grouped ? groups : 0,
                           grouped ? a->max_members : 0, grouped ? longest : 0,
                           grouped ? a->ungrouped : nullptr, grouped ? ungrouped : -1,
                           a->workspace, a->workspace_bytes, a->compute_stream);
    if (st != PKV_OK) return st;
    return pkv_stage_download(a->out, host_out, a->out_bytes, a->compute_stream, a->down_stream,
                              a->computed_event, a->downloaded_event);
}

}  // extern "C"
