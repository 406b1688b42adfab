// paged_attention_decode_noalloc: decode attention that allocates nothing and
// needs no workspace from the caller.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at the
// point where they decode -- for example a plug-in hosted by a runtime that owns
// all device memory and allows no allocation through another path, or a serving
// loop that fixes its memory plan at start-up so that nothing allocates (and
// possibly synchronises the device, or fails under fragmentation) while it
// serves. The regular paged_attention_decode takes its split-KV scratch from the
// caller; this variant uses a fixed scratch array that lives in the library
// itself, so the caller passes only inputs and outputs.
//
// The scratch is a file-scope __device__ array of PKV_NOALLOC_WORKSPACE_BYTES.
// Every GPU that loads the library holds it until the process exits. In host
// code its name is only a host-side stand-in, so its device address is looked up
// once per device (cudaGetSymbolAddress with that device current) by the first
// call made on that device; make that first call before any stream capture.
// The address is kept for the life of the process, so the library must not be
// used across a cudaDeviceReset of that device (its error word and per-kernel
// set-up are cached the same way). All
// calls on a device share the one array, so calls that overlap on the GPU (on
// different streams, or from different threads) race on it: serialise them. The
// array keeps the last call's contents; nothing in it needs to start at zero,
// because every partition slot the merge reads is first written by the same call.
#include <atomic>

#include "pkv_decode_impl.cuh"

static __device__ __align__(256) unsigned char g_noalloc_workspace[PKV_NOALLOC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<void*> g_noalloc_ptr[kMaxDevices];

// Device address of this device's scratch array (set-up on first use).
int noalloc_workspace(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pkv::cuda_fail("noalloc decode: current device", e);
    if (dev < 0 || dev >= kMaxDevices)
        return pkv::cuda_fail("noalloc decode: device index", cudaErrorInvalidDevice);
    void* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
        if (e != cudaSuccess) return pkv::cuda_fail("noalloc decode: scratch address", e);
        g_noalloc_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return PKV_OK;
}

}  // namespace

extern "C" int paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_pool, const void* v_pool,
    const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq,
    int num_blocks, int num_heads, int num_kv_heads, int head_dim, int block_size, float scale,
    int q_dtype, int kv_dtype, float k_scale, float v_scale, void* stream) {
    // A batch that can be split (some sequence may span more than one minimal
    // partition) needs the smallest split -- two partitions per sequence and
    // head -- to fit, or the call is refused: such a batch is beyond what the
    // fixed scratch serves. A batch that can never be split uses no scratch.
    if (num_seqs > 0 && num_heads > 0 && head_dim > 0 &&
        paged_attention_workspace_size(num_seqs, num_heads, head_dim, block_size,
                                       max_blocks_per_seq) > 0) {
        const size_t need =
            (size_t)num_seqs * num_heads * 2 * ((size_t)head_dim + 2) * sizeof(float);
        if (need > (size_t)PKV_NOALLOC_WORKSPACE_BYTES) return PKV_ERR_INVALID_ARG;
    }
    void* ws = nullptr;
    const int st = noalloc_workspace(&ws);
    if (st != PKV_OK) return st;
    return paged_attention_decode(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                                  max_blocks_per_seq, num_blocks, num_heads, num_kv_heads,
                                  head_dim, block_size, scale, q_dtype, kv_dtype, k_scale,
                                  v_scale, ws, (size_t)PKV_NOALLOC_WORKSPACE_BYTES, stream);
}
