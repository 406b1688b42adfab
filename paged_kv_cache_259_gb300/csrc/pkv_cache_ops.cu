// The two cache writes of a decode step.
//
// reshape_and_cache: slot-mapped write of each new token's K/V into the pools
//   ("PagedAttention" glossary, "Cách phân trang hoạt động": token pos lives in
//   block table[pos / block_size] at slot pos % block_size; the caller passes
//   the folded slot number). Optional FP8 E4M3 quantisation (related-techniques
//   section, FP8 cache item).
// copy_blocks: the block copy of copy-on-write ("KV cache paginado...",
//   "Como funciona"; glossary "Chia sẻ block giữa các chuỗi").
//
// Both are plain HBM traffic: 16-byte vector loads, one thread per 16-byte group
// of elements, grids sized over the SMs.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

// Destination-chunk type of the cache: 16 bytes = CV cache elements.
template <typename ST, typename CT>
struct ChunkConvert;

// Same type: the 16 bytes are copied unchanged.
template <typename T>
struct ChunkConvert<T, T> {
    static constexpr int CV = 16 / sizeof(T);
    __device__ __forceinline__ static uint4 run(const T* src, float) {
        return *reinterpret_cast<const uint4*>(src);
    }
};

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

// E4M3 cache: 16 source values -> 16 bytes, each x / scale (IEEE float32 divide)
// rounded to nearest even E4M3 with saturation to +-448.
template <typename ST>
struct ChunkConvert<ST, uint8_t> {
    static constexpr int CV = 16;
    __device__ __forceinline__ static uint4 run(const ST* src, float scale) {
        ST vals[16];
#pragma unroll
        for (int i = 0; i < 16 * (int)sizeof(ST) / 16; ++i)
            reinterpret_cast<uint4*>(vals)[i] = reinterpret_cast<const uint4*>(src)[i];
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float2 f;
                f.x = __fdiv_rn(to_float(vals[4 * i + 2 * j]), scale);
                f.y = __fdiv_rn(to_float(vals[4 * i + 2 * j + 1]), scale);
                const __nv_fp8x2_storage_t pr = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
                word |= static_cast<uint32_t>(pr) << (16 * j);
            }
            w[i] = word;
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Cache layout (per block and kv head), X = 16 bytes of cache elements: each
// tile is a sequence of 128-byte core matrices (8 rows of 16 bytes), K as
// [bs/8][D/X][8][X] (8 tokens x X dims each) and V as [bs/X][D/8][8][X] (8 dims x
// X tokens each). One thread converts one 16-byte group of X dims of one
// (token, head): for K it is one 16-byte store, for V X element stores, one into
// each of the X dims' rows at the token's column.
template <typename CT>
__device__ __forceinline__ void store_v_column(CT* tile, const uint4& v, int d0, int d, int off) {
    constexpr int CV = 16 / sizeof(CT);
    const CT* e = reinterpret_cast<const CT*>(&v);
    const long long col = (long long)(off / CV) * (d / 8) * 8 * CV + off % CV;
#pragma unroll
    for (int i = 0; i < CV; ++i) {
        const int dd = d0 + i;
        tile[col + (long long)(dd >> 3) * 8 * CV + (dd & 7) * CV] = e[i];
    }
}

template <typename ST, typename CT>
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const ST* __restrict__ k, const ST* __restrict__ v, CT* __restrict__ k_pool,
    CT* __restrict__ v_pool, const int64_t* __restrict__ slots, int num_tokens, int hkv, int d,
    int bs, int num_blocks, float k_scale, float v_scale, int* err) {
    pdl_enter();                                           // launched with launch_pdl
    using CC = ChunkConvert<ST, CT>;
    const int planes = d / CC::CV;                         // 16-byte groups per (token, head)
    const long long per_pool = (long long)num_tokens * hkv * planes;
    const long long total = 2 * per_pool;
    const long long slot_limit = (long long)num_blocks * bs;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const bool is_v = idx >= per_pool;
        long long r = is_v ? idx - per_pool : idx;
        const int j = (int)(r % planes);
        r /= planes;
        const int h = (int)(r % hkv);
        const int t = (int)(r / hkv);
        const long long slot = slots[t];
        if (slot < 0) continue;                            // padding token
        if (slot >= slot_limit) {
            flag_error(err, kErrOutOfRange);
            continue;
        }
        const long long blk = slot / bs, off = slot % bs;
        const ST* src = (is_v ? v : k) + ((long long)t * hkv + h) * d + (long long)j * CC::CV;
        const uint4 val = CC::run(src, is_v ? v_scale : k_scale);
        const long long tile = (blk * hkv + h) * (long long)d * bs;      // elements
        if (!is_v) {
            CT* dst = k_pool + tile + ((off >> 3) * planes + j) * 8 * CC::CV + (off & 7) * CC::CV;
            *reinterpret_cast<uint4*>(dst) = val;
        } else {
            store_v_column(v_pool + tile, val, j * CC::CV, d, (int)off);
        }
    }
}

// bf16 caches, written by aligned 8-slot windows. One warp per (group of 8
// consecutive tokens, kv head), walking its 8 tokens. Token i (slot s) looks at
// the window of slots s - s%8 .. s - s%8 + 7 (8 lanes check 8 slots at once): if
// tokens i - s%8 .. i - s%8 + 7 fill exactly that window (a prefill chunk away
// from its two ends), the window is one 8-token chunk of the block, whose K rows
// (plane j, token) and V rows (dim, 8 tokens) are each 2 KB of contiguous core
// matrices, and the window's first token writes both with coalesced 16-byte
// stores: K row j*8+t is token t's 16-byte chunk j, V row dim is that dim of the
// 8 tokens (gathered as 2-byte loads, lane by lane, already transposed); the
// window's other tokens are skipped (the walk jumps past them). So nearly every
// warp moves about one window.
// Every token not in such a window (decode steps, ragged chunk ends) is written
// on its own: lane j stores K chunk j and V dims 8j..8j+7 down their column.
// DT: the head dim when known at compile time (its row loops unroll), else 0.
template <int DT>
__global__ void __launch_bounds__(256) reshape_and_cache_bf16_windows(
    const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, const int64_t* __restrict__ slots, int num_tokens, int hkv,
    int d_rt, int bs, int num_blocks, int* err) {
    pdl_enter();                                           // launched with launch_pdl
    const int d = DT ? DT : d_rt;
    const int planes = d / 8;                              // 16-byte chunks per (token, head)
    const int lane = threadIdx.x & 31;
    const long long units = (long long)((num_tokens + 7) / 8) * hkv;
    const long long slot_limit = (long long)num_blocks * bs;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const unsigned short* vh = reinterpret_cast<const unsigned short*>(v);
    for (long long u = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5); u < units;
         u += warps) {
        const int grp = (int)(u / hkv), h = (int)(u - (long long)grp * hkv);
        // the slots of tokens grp*8-8 .. grp*8+15 (every window a token of this
        // group can be in), one per lane, read once; -1 outside the batch
        const int t_lo = grp * 8 - 8;
        const long long near =
            lane < 24 && t_lo + lane >= 0 && t_lo + lane < num_tokens ? slots[t_lo + lane] : -1LL;
        // after a token that is in a window, jump past the window's end
        for (int q = 0, step = 1; q < 8; q += step) {
            step = 1;
            const int t = grp * 8 + q;
            if (t >= num_tokens) break;
            const long long slot = __shfl_sync(0xffffffffu, near, 8 + q);
            if (slot < 0) continue;                        // padding token
            if (slot >= slot_limit) {
                if (lane == 0) flag_error(err, kErrOutOfRange);
                continue;
            }
            const int lead = t - (int)(slot & 7);          // first token of the window
            // lane i < 8 compares token lead + i's slot (lane lead - t_lo + i of `near`)
            const long long other = __shfl_sync(0xffffffffu, near, (lead - t_lo + (lane & 7)) & 31);
            const bool ok = lane >= 8 || (lead >= 0 && lead + 8 <= num_tokens &&
                                          (slot | 7) < slot_limit && other == (slot & ~7LL) + lane);
            const bool run = __all_sync(0xffffffffu, ok);
            if (run) step = lead + 8 - t;                  // the window's tokens are done here
            if (run && t != lead) continue;                // written by the window's first token
            const long long blk = slot / bs, off = slot - blk * bs;
            const long long tile = (blk * hkv + h) * (long long)(d * bs / 8);   // 16-byte units
            if (run) {
                const long long base = tile + (off >> 3) * planes * 8;   // the window's core matrices
                constexpr int kIters = DT ? DT / 32 : 1;
#pragma unroll
                for (int it = 0; it < kIters; ++it) {
                    for (int o = lane + it * 32; o < planes * 8; o += kIters * 32) {
                        // K row o: token o % 8, chunk o / 8
                        const uint4 kk =
                            k[((long long)(lead + (o & 7)) * hkv + h) * planes + (o >> 3)];
                        // V row o: dim o of the 8 tokens
                        uint32_t w[4];
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const uint32_t lo = vh[((long long)(lead + 2 * m) * hkv + h) * d + o];
                            const uint32_t hi = vh[((long long)(lead + 2 * m + 1) * hkv + h) * d + o];
                            w[m] = lo | (hi << 16);
                        }
                        k_pool[base + o] = kk;
                        v_pool[base + o] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                continue;
            }
            if (lane < planes) {                           // this token alone
                const long long src = ((long long)t * hkv + h) * planes + lane;
                k_pool[tile + ((off >> 3) * planes + lane) * 8 + (off & 7)] = k[src];
                store_v_column(reinterpret_cast<__nv_bfloat16*>(v_pool + tile), v[src], lane * 8,
                               d, (int)off);
            }
        }
    }
}

constexpr int kCopyThreads = 256;
constexpr int kCopyChunkBytes = kCopyThreads * 16 * 4;    // 16 KB per CTA
// Launches of at most this many pairs check copy_blocks' preconditions on the
// device (each pair's first CTA scans every pair once: P^2 pair reads in L2).
constexpr int kCopyCheckPairs = 4096;

// One CTA per (pair, pool, 16 KB chunk), 16-byte vector copies. The first CTA
// of each pair (K pool, first chunk) also checks the launch's preconditions for
// that pair while its loads are in flight: its destination is no other pair's
// destination and no pair's source (its own included). A violation sets
// kErrBadPairs; the copies still run (in bounds; which bytes land is then
// unspecified).
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    char* __restrict__ k_pool, char* __restrict__ v_pool, const int64_t* __restrict__ pairs,
    int num_pairs, int num_blocks, size_t block_bytes, int* err) {
    pdl_enter();                                           // launched with launch_pdl
    const int pair = blockIdx.x >> 1;
    char* pool = (blockIdx.x & 1) ? v_pool : k_pool;
    const int64_t src = pairs[2 * pair], dst = pairs[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && !(blockIdx.x & 1))
            flag_error(err, kErrOutOfRange);
        return;
    }
    const uint4* s = reinterpret_cast<const uint4*>(pool + (size_t)src * block_bytes);
    uint4* o = reinterpret_cast<uint4*>(pool + (size_t)dst * block_bytes);
    const size_t n16 = block_bytes / 16;
    const size_t beg = (size_t)blockIdx.y * (kCopyChunkBytes / 16);
    const size_t end = min(n16, beg + kCopyChunkBytes / 16);
    uint4 buf[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const size_t i = beg + threadIdx.x + (size_t)u * kCopyThreads;
        if (i < end) buf[u] = s[i];
    }
    if (blockIdx.y == 0 && !(blockIdx.x & 1) && num_pairs <= kCopyCheckPairs) {
        bool bad = false;
        for (int j = threadIdx.x; j < num_pairs; j += kCopyThreads) {
            const int64_t sj = pairs[2 * j], dj = pairs[2 * j + 1];
            bad |= sj == dst || (j != pair && dj == dst);
        }
        if (__syncthreads_or(bad) && threadIdx.x == 0) flag_error(err, kErrBadPairs);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const size_t i = beg + threadIdx.x + (size_t)u * kCopyThreads;
        if (i < end) o[i] = buf[u];
    }
}

template <typename ST, typename CT>
cudaError_t launch_reshape(const void* k, const void* v, void* kp, void* vp, const int64_t* slots,
                           int num_tokens, int hkv, int d, int bs, int num_blocks, float ks,
                           float vs, int* err, cudaStream_t stream) {
    const long long chunks = 2LL * num_tokens * hkv * (d / ChunkConvert<ST, CT>::CV);
    const int threads = 256;
    long long blocks = (chunks + threads - 1) / threads;
    const long long cap = 8LL * num_sms();                 // grid-stride beyond 8 CTAs/SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    note_launch();
    return launch_pdl(reshape_and_cache_kernel<ST, CT>, dim3((unsigned)blocks), dim3(threads), 0,
                      stream, static_cast<const ST*>(k), static_cast<const ST*>(v),
                      static_cast<CT*>(kp), static_cast<CT*>(vp), slots, num_tokens, hkv, d, bs,
                      num_blocks, ks, vs, err);
}

// Block copies between two pools (device or pinned host memory, both reached by
// the kernel through the device's own addresses: host memory over the CPU-GPU
// link). One CTA per (pair, pool, 16 KB chunk), 16-byte vector copies. A pair
// outside either pool is skipped and flagged.
__global__ void __launch_bounds__(kCopyThreads) swap_blocks_kernel(
    char* __restrict__ dst_k, char* __restrict__ dst_v, const char* __restrict__ src_k,
    const char* __restrict__ src_v, const int64_t* __restrict__ pairs, int src_blocks,
    int dst_blocks, size_t block_bytes, int* err) {
    const int pair = blockIdx.x >> 1;
    const bool is_v = blockIdx.x & 1;
    const int64_t src = pairs[2 * pair], dst = pairs[2 * pair + 1];
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && !is_v) flag_error(err, kErrOutOfRange);
        return;
    }
    const uint4* s = reinterpret_cast<const uint4*>((is_v ? src_v : src_k) + (size_t)src * block_bytes);
    uint4* o = reinterpret_cast<uint4*>((is_v ? dst_v : dst_k) + (size_t)dst * block_bytes);
    const size_t n16 = block_bytes / 16;
    const size_t beg = (size_t)blockIdx.y * (kCopyChunkBytes / 16);
    const size_t end = min(n16, beg + kCopyChunkBytes / 16);
    uint4 buf[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const size_t i = beg + threadIdx.x + (size_t)u * kCopyThreads;
        if (i < end) buf[u] = s[i];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const size_t i = beg + threadIdx.x + (size_t)u * kCopyThreads;
        if (i < end) o[i] = buf[u];
    }
}

// The address the device uses for a pool: itself for device memory, the mapped
// address for pinned host memory; nullptr for memory the device cannot reach.
void* device_address(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return const_cast<void*>(p);
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    return nullptr;
}

// Batches this large (a prefill chunk) go through the window kernel; smaller
// ones (a decode step: one token per sequence, no runs) skip its window checks.
constexpr int kGroupTokens = 512;

cudaError_t launch_reshape_groups(const void* k, const void* v, void* kp, void* vp,
                                  const int64_t* slots, int num_tokens, int hkv, int d, int bs,
                                  int num_blocks, int* err, cudaStream_t stream) {
    const long long items = (long long)((num_tokens + 7) / 8) * hkv;   // one warp each
    const int threads = 256;
    long long blocks = (items + threads / 32 - 1) / (threads / 32);
    const long long cap = 8LL * num_sms();
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    note_launch();
    auto kern = d == 128 ? reshape_and_cache_bf16_windows<128>
                         : d == 64 ? reshape_and_cache_bf16_windows<64>
                                   : reshape_and_cache_bf16_windows<0>;
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(threads), 0, stream,
                      static_cast<const uint4*>(k), static_cast<const uint4*>(v),
                      static_cast<uint4*>(kp), static_cast<uint4*>(vp), slots, num_tokens, hkv, d,
                      bs, num_blocks, err);
}

}  // namespace
}  // namespace pkv

extern "C" {

int reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                      const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, int src_dtype, int cache_dtype,
                      float k_scale, float v_scale, void* stream) {
    using namespace pkv;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (head_dim % 16 != 0 || block_size % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !k_pool || !v_pool || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID_ARG;
    const bool fp8 = cache_dtype == PKV_E4M3;
    if (fp8) {
        if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale))
            return PKV_ERR_INVALID_ARG;
    } else if (cache_dtype != src_dtype) {
        return PKV_ERR_UNSUPPORTED;
    }
    int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (src_dtype == PKV_F32 && cache_dtype == PKV_F32)
        e = launch_reshape<float, float>(k, v, k_pool, v_pool, slot_mapping, num_tokens,
                                         num_kv_heads, head_dim, block_size, num_blocks, 1.f, 1.f,
                                         err, s);
    else if (src_dtype == PKV_BF16 && cache_dtype == PKV_BF16 && num_tokens >= kGroupTokens)
        e = launch_reshape_groups(k, v, k_pool, v_pool, slot_mapping, num_tokens, num_kv_heads,
                                  head_dim, block_size, num_blocks, err, s);
    else if (src_dtype == PKV_BF16 && cache_dtype == PKV_BF16)
        e = launch_reshape<__nv_bfloat16, __nv_bfloat16>(k, v, k_pool, v_pool, slot_mapping,
                                                         num_tokens, num_kv_heads, head_dim,
                                                         block_size, num_blocks, 1.f, 1.f, err, s);
    else if (src_dtype == PKV_F32 && fp8)
        e = launch_reshape<float, uint8_t>(k, v, k_pool, v_pool, slot_mapping, num_tokens,
                                           num_kv_heads, head_dim, block_size, num_blocks, k_scale,
                                           v_scale, err, s);
    else if (src_dtype == PKV_BF16 && fp8)
        e = launch_reshape<__nv_bfloat16, uint8_t>(k, v, k_pool, v_pool, slot_mapping, num_tokens,
                                                   num_kv_heads, head_dim, block_size, num_blocks,
                                                   k_scale, v_scale, err, s);
    else
        return PKV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PKV_OK : cuda_fail("reshape_and_cache: kernel launch", e);
}

int copy_blocks(void* k_pool, void* v_pool, const int64_t* src_dst_pairs, int num_pairs,
                int num_blocks, size_t block_bytes, void* stream) {
    using namespace pkv;
    if (num_pairs < 0 || num_blocks <= 0 || block_bytes == 0 || block_bytes % 16 != 0)
        return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!k_pool || !v_pool || !src_dst_pairs || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID_ARG;
    if (num_pairs > (1 << 30) || block_bytes / kCopyChunkBytes >= 65535)
        return PKV_ERR_UNSUPPORTED;
    int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    const unsigned chunks = (unsigned)((block_bytes + kCopyChunkBytes - 1) / kCopyChunkBytes);
    dim3 grid(2u * (unsigned)num_pairs, chunks);
    note_launch();
    const cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(kCopyThreads), 0,
                                     static_cast<cudaStream_t>(stream), static_cast<char*>(k_pool),
                                     static_cast<char*>(v_pool), src_dst_pairs, num_pairs,
                                     num_blocks, block_bytes, err);
    return e == cudaSuccess ? PKV_OK : cuda_fail("copy_blocks: kernel launch", e);
}

int swap_blocks(void* dst_k_pool, void* dst_v_pool, const void* src_k_pool,
                const void* src_v_pool, const int64_t* src_dst_pairs, int num_pairs,
                int src_num_blocks, int dst_num_blocks, size_t block_bytes, void* stream) {
    using namespace pkv;
    if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || block_bytes == 0 ||
        block_bytes % 16 != 0)
        return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!dst_k_pool || !dst_v_pool || !src_k_pool || !src_v_pool || !src_dst_pairs)
        return PKV_ERR_INVALID_ARG;
    if (num_pairs > (1 << 30) || block_bytes / kCopyChunkBytes >= 65535)
        return PKV_ERR_UNSUPPORTED;
    void* dk = device_address(dst_k_pool);
    void* dv = device_address(dst_v_pool);
    const void* sk = device_address(src_k_pool);
    const void* sv = device_address(src_v_pool);
    const void* pp = device_address(src_dst_pairs);
    if (!dk || !dv || !sk || !sv || !pp) return PKV_ERR_INVALID_ARG;   // unreachable memory
    if (!aligned16(dk) || !aligned16(dv) || !aligned16(sk) || !aligned16(sv))
        return PKV_ERR_INVALID_ARG;
    int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    const unsigned chunks = (unsigned)((block_bytes + kCopyChunkBytes - 1) / kCopyChunkBytes);
    dim3 grid(2u * (unsigned)num_pairs, chunks);
    note_launch();
    swap_blocks_kernel<<<grid, kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<char*>(dk), static_cast<char*>(dv), static_cast<const char*>(sk),
        static_cast<const char*>(sv), static_cast<const int64_t*>(pp), src_num_blocks,
        dst_num_blocks, block_bytes, err);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_fail("swap_blocks: kernel launch", e);
}

}  // extern "C"
