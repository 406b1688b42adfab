// Decode-step attention over a paged KV cache (CUDA-core variant).
//
// "PagedAttention" (Ultralytics glossary), "Cách phân trang hoạt động": the
// attention kernel reads a request's keys and values back block by block
// through its block table, so the cache need not be contiguous. The related-
// techniques section's FlashAttention item: the score vector is never written to
// HBM; here it lives in registers/shared memory and softmax is computed online.
//
// Work decomposition
//   CTA  = (partition p, kv head hk, sequence b). A partition is PB consecutive
//          logical blocks of the sequence; with one partition per sequence the
//          CTA writes `out` directly, otherwise it writes a normalised partial
//          (o_p, m_p, l_p) to the workspace and a second kernel merges them.
//   warp = an independent streaming engine: warp w takes partition-local blocks
//          w, w+NW, w+2NW, ... Each has its own STAGES-deep ring of (K tile,
//          V tile) pairs in shared memory, filled by 1-D bulk copies (TMA engine,
//          no tensor map) issued by lane 0 and completed on one mbarrier per
//          stage. A (block, kv head) tile is block_size*head_dim contiguous
//          elements of the pool, so it is one copy.
//   lane = a 16-byte column chunk c of a token row and a row group rg; the warp
//          covers RPP = 32/LPR rows per pass (LPR lanes per row), i.e. one pass
//          reads 512 contiguous bytes of the tile from shared memory.
//
// Per tile: partial dot products of the lane's chunk with each of the G query
// heads (GQA: G query heads share the KV head, glossary item "Attention truy vấn
// theo nhóm"), a butterfly transpose-reduce across the LPR lanes of a row,
// scores masked beyond the sequence end, an online-softmax update (running
// max m, running sum l, rescale of the accumulator by 2^(m_old - m_new); logits
// pre-multiplied by log2 e so exp2 is used), then P.V accumulated per lane.
//
// Every spin-wait is bounded (pkv::mbar_wait_bounded); a block-table entry
// outside the pool is skipped and recorded in the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>

#include "pkv_internal.cuh"

namespace pkv {
namespace decode {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
    void* out;
    const void* q;
    const char* k_pool;
    const char* v_pool;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    float* ws_o;      // [B][Hq][max_parts][D]   normalised partial outputs
    float* ws_ml;     // [B][Hq][max_parts][2]   (m in log2 units, l)
    int* err;
    int num_seqs, max_blocks, num_blocks, num_heads, num_kv_heads;
    int part_blocks, max_parts;
    float qscale;     // scale * k_scale * log2(e)
    float v_scale;
};

template <typename T> struct Elt;
template <> struct Elt<float> { static constexpr int kSize = 4; };
template <> struct Elt<__nv_bfloat16> { static constexpr int kSize = 2; };
template <> struct Elt<uint8_t> { static constexpr int kSize = 1; };

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// 16 bytes of cache -> floats (4 x f32, 8 x bf16 or 16 x e4m3).
__device__ __forceinline__ void unpack(const uint4& r, float (&f)[4]) {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
}
__device__ __forceinline__ void unpack(const uint4& r, float (&f)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unpack(const uint4& r, float (&f)[16]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)((w[i] >> (16 * j)) & 0xffffu);
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
            const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            f[4 * i + 2 * j] = f2.x;
            f[4 * i + 2 * j + 1] = f2.y;
        }
    }
}

// Sum N per-lane values over aligned groups of W lanes (W a power of two).
// Afterwards v[0..R) with R = max(1, N/W) holds full sums of value indices
//   N >= W: j = (lane % W) * R + r
//   N <  W: j = (lane % W) / (W / N)    (one value, the same in W/N lanes)
// Each level halves the values a lane carries: the lane keeps one half and
// receives its partner's sums of that half.
template <int N, int W>
struct Butterfly {
    __device__ __forceinline__ static void run(float* v, int lane) {
        if constexpr (W > 1) {
            constexpr int M = W / 2;
            if constexpr (N > 1) {
                constexpr int H = N / 2;
                const bool upper = (lane & M) != 0;
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const float send = upper ? v[i] : v[i + H];
                    const float keep = upper ? v[i + H] : v[i];
                    v[i] = keep + __shfl_xor_sync(kFull, send, M);
                }
                Butterfly<H, M>::run(v, lane);
            } else {
                v[0] += __shfl_xor_sync(kFull, v[0], M);
                Butterfly<1, M>::run(v, lane);
            }
        }
    }
};

template <typename KV, int D, int BS, int G, int NW>
struct Shape {
    static constexpr int kElt = Elt<KV>::kSize;
    static constexpr int kVec = 16 / kElt;                  // elements per 16-byte chunk
    static constexpr int kLpr = D / kVec;                   // lanes per token row
    static constexpr int kRpp = 32 / kLpr;                  // rows per warp pass
    static constexpr int kTpl = BS / kRpp;                  // tokens per lane per tile
    static constexpr int kRowBytes = D * kElt;
    static constexpr int kTile = BS * kRowBytes;            // one (block, kv head) tile
    static constexpr int kNv = G * kTpl;                    // partial scores per lane
    static constexpr int kR = kNv >= kLpr ? kNv / kLpr : 1; // reduced scores per lane
    static constexpr int kGbs = G * BS;                     // scores per tile
    static constexpr int kSpl = kGbs >= 32 ? kGbs / 32 : 1; // scores per softmax lane
    static constexpr int kActive = kGbs >= 32 ? 32 : kGbs;  // softmax lanes
    static constexpr int kGs = BS / kSpl;                   // softmax lanes per head
    // about 96 KB of ring per CTA (two CTAs per SM); at least one stage per warp
    // (a 16 KB tile, float32 D128 with 32-token blocks, gets a single stage)
    static constexpr int kStages = (98304 / (NW * 2 * kTile)) < 1 ? 1
                                   : (98304 / (NW * 2 * kTile)) > 8 ? 8
                                   : (98304 / (NW * 2 * kTile));
    static constexpr int kRingBytes = NW * kStages * 2 * kTile;
    static constexpr int kSmem = kRingBytes + NW * kStages * 8   // mbarriers
                                 + NW * kStages * 4              // stage block ids
                                 + NW * kGbs * 4                 // scores / probabilities
                                 + NW * G * 4;                   // per-head rescale factors
    static_assert(32 % kLpr == 0 && kLpr >= 1, "row must map onto whole lanes");
    static_assert(BS % kRpp == 0, "block must hold whole warp passes");
    static_assert(NW * G * (D + 2) * 4 <= kRingBytes, "combine area must fit in the ring");
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static_assert(kGbs % kSpl == 0 && BS % kSpl == 0, "softmax lanes");
};

template <typename QT, typename KV, int D, int BS, int G, int NW>
__global__ void __launch_bounds__(NW * 32) paged_decode_kernel(const Params p) {
    using S = Shape<KV, D, BS, G, NW>;
    constexpr int VEC = S::kVec, LPR = S::kLpr, RPP = S::kRpp, TPL = S::kTpl;
    constexpr int TILE = S::kTile, ST = S::kStages, GBS = S::kGbs;
    constexpr int SPL = S::kSpl, ACTIVE = S::kActive, GS = S::kGs;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kRingBytes);
    int32_t* stage_id = reinterpret_cast<int32_t*>(bars + NW * ST);
    float* sc = reinterpret_cast<float*>(stage_id + NW * ST);
    float* alph = sc + NW * GBS;

    const int part = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    int L = p.seq_lens[b];
    if (L < 0 || L > p.max_blocks * BS) {                   // length the table cannot hold
        if (part == 0 && hk == 0 && threadIdx.x == 0) flag_error(p.err, kErrOutOfRange);
        L = L < 0 ? 0 : p.max_blocks * BS;
    }
    const int nblk = (L + BS - 1) / BS;
    const int PB = p.part_blocks;
    const int nparts = (nblk + PB - 1) / PB;
    if (part >= (nparts > 0 ? nparts : 1)) return;          // beyond this sequence
    const int blk0 = part * PB;
    const int nbp = max(0, min(PB, nblk - blk0));           // blocks in this partition

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int c = lane % LPR, rg = lane / LPR;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < ST; ++s) mbar_init(smem_addr(&bars[w * ST + s]), 1);
        fence_mbar_init();
    }
    __syncwarp();

    // query rows of the G heads that share kv head hk, pre-scaled
    float qf[G][VEC];
    {
        const QT* qb = static_cast<const QT*>(p.q) + ((size_t)b * p.num_heads + (size_t)hk * G) * D;
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int v = 0; v < VEC; ++v) qf[g][v] = to_f(qb[g * D + c * VEC + v]) * p.qscale;
    }

    float acc[G][VEC];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[g][v] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;

    const int nk = nbp > w ? (nbp - w + NW - 1) / NW : 0;  // this warp's blocks
    const int32_t* bt_row = p.block_tables + (size_t)b * p.max_blocks + blk0 + w;
    const uint64_t pol = l2_evict_first();

    // block ids, 32 per warp-wide load, double-buffered in registers; invalid -> -1
    auto load_chunk = [&](int chunk) -> int {
        const int kk = chunk * 32 + lane;
        int id = -1;
        if (kk < nk) {
            id = bt_row[(size_t)kk * NW];
            if (id < 0 || id >= p.num_blocks) {
                flag_error(p.err, kErrOutOfRange);
                id = -1;
            }
        }
        return id;
    };
    int id_cur = load_chunk(0), id_nxt = load_chunk(1), chunk_cur = 0;
    auto get_id = [&](int kk) -> int {                     // warp-uniform call
        while ((kk >> 5) > chunk_cur) {
            id_cur = id_nxt;
            ++chunk_cur;
            id_nxt = load_chunk(chunk_cur + 1);
        }
        return __shfl_sync(kFull, id_cur, kk & 31);
    };
    auto issue = [&](int kk, int id) {                      // lane 0 only
        const int s = kk % ST;
        const uint32_t bar = smem_addr(&bars[w * ST + s]);
        stage_id[w * ST + s] = id;
        if (id >= 0) {
            const uint32_t dst = smem_addr(ring + (size_t)((w * ST + s) * 2) * TILE);
            const size_t off = ((size_t)id * p.num_kv_heads + hk) * TILE;
            mbar_arrive_expect_tx(bar, 2 * TILE);
            bulk_g2s(dst, p.k_pool + off, TILE, bar, pol);
            bulk_g2s(dst + TILE, p.v_pool + off, TILE, bar, pol);
        } else {
            mbar_arrive(bar);
        }
    };

    const int pro = nk < ST ? nk : ST;
    for (int kk = 0; kk < pro; ++kk) {
        const int id = get_id(kk);
        if (lane == 0) issue(kk, id);
    }

    bool aborted = false;
    int k = 0;
    for (; k < nk; ++k) {
        const int s = k % ST;
        const bool ok = mbar_wait_bounded(smem_addr(&bars[w * ST + s]), (k / ST) & 1, p.err);
        if (__any_sync(kFull, !ok)) {
            aborted = true;
            break;
        }
        const int id = stage_id[w * ST + s];
        if (id >= 0) {
            const int ntok = min(BS, L - (blk0 + w + k * NW) * BS);
            const unsigned char* kt = ring + (size_t)((w * ST + s) * 2) * TILE;
            const unsigned char* vt = kt + TILE;

            // ---- scores: partial dots of this lane's chunk, then reduce over the row's lanes
            float part_s[S::kNv];
#pragma unroll
            for (int i = 0; i < TPL; ++i) {
                const int t = i * RPP + rg;
                float kf[VEC];
                unpack(*reinterpret_cast<const uint4*>(kt + t * S::kRowBytes + c * 16), kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a = 0.f;
#pragma unroll
                    for (int v = 0; v < VEC; ++v) a = fmaf(qf[g][v], kf[v], a);
                    part_s[g * TPL + i] = a;
                }
            }
            Butterfly<S::kNv, LPR>::run(part_s, lane);
            float* scw = sc + w * GBS;
#pragma unroll
            for (int r = 0; r < S::kR; ++r) {
                const int j = S::kNv >= LPR ? c * S::kR + r : c / (LPR / S::kNv);
                const bool leader = S::kNv >= LPR || (c % (LPR / S::kNv)) == 0;
                const int g = j / TPL, t = (j % TPL) * RPP + rg;
                if (leader) scw[g * BS + t] = t < ntok ? part_s[r] : -INFINITY;
            }
            __syncwarp();

            // ---- online softmax over the tile (lane owns SPL scores of one head)
            float sv[SPL];
            float tmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < SPL; ++i) {
                sv[i] = lane < ACTIVE ? scw[lane * SPL + i] : -INFINITY;
                tmax = fmaxf(tmax, sv[i]);
            }
#pragma unroll
            for (int msk = GS / 2; msk >= 1; msk >>= 1)
                tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, msk));
            if (lane < ACTIVE) {
                const float m_new = fmaxf(m_run, tmax);
                const float alpha = exp2f(m_run - m_new);
                float psum = 0.f;
#pragma unroll
                for (int i = 0; i < SPL; ++i) {
                    const float pv = exp2f(sv[i] - m_new);
                    psum += pv;
                    scw[lane * SPL + i] = pv;
                }
                l_run = l_run * alpha + psum;
                m_run = m_new;
                if (lane % GS == 0) alph[w * G + (lane * SPL) / BS] = alpha;
            }
            __syncwarp();

            // ---- P.V into this lane's chunk of each head's accumulator
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float a = alph[w * G + g];
#pragma unroll
                for (int v = 0; v < VEC; ++v) acc[g][v] *= a;
            }
#pragma unroll
            for (int i = 0; i < TPL; ++i) {
                const int t = i * RPP + rg;
                if (t < ntok) {
                    float vf[VEC];
                    unpack(*reinterpret_cast<const uint4*>(vt + t * S::kRowBytes + c * 16), vf);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float pg = scw[g * BS + t];
#pragma unroll
                        for (int v = 0; v < VEC; ++v) acc[g][v] = fmaf(pg, vf[v], acc[g][v]);
                    }
                }
            }
        }
        __syncwarp();
        if (k + ST < nk) {
            const int id = get_id(k + ST);
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(k + ST, id);
            }
        }
    }
    if (aborted) {
        // give up: record it, and let the copies already issued land before the
        // shared memory is reused or released
        if (lane == 0) flag_error(p.err, kErrTimeout);
        const int last = min(nk, k + ST);
        for (int kk = k; kk < last; ++kk)
            (void)mbar_wait_bounded(smem_addr(&bars[w * ST + (kk % ST)]), (kk / ST) & 1, p.err);
        m_run = -INFINITY;
        l_run = 0.f;
    }

    // ---- warp totals: l over the head's softmax lanes, acc over row groups
#pragma unroll
    for (int msk = GS / 2; msk >= 1; msk >>= 1) l_run += __shfl_xor_sync(kFull, l_run, msk);
#pragma unroll
    for (int msk = LPR; msk < 32; msk <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[g][v] += __shfl_xor_sync(kFull, acc[g][v], msk);

    __syncthreads();                                        // every warp is done with its ring
    float* cm = reinterpret_cast<float*>(ring);             // [NW][G]
    float* cl = cm + NW * G;                                // [NW][G]
    float* cacc = cl + NW * G;                              // [NW][G][D]
    if (lane < ACTIVE && lane % GS == 0) {
        const int g = (lane * SPL) / BS;
        cm[w * G + g] = aborted ? -INFINITY : m_run;
        cl[w * G + g] = aborted ? 0.f : l_run;
    }
    if (rg == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int v = 0; v < VEC; ++v)
                cacc[(w * G + g) * D + c * VEC + v] = aborted ? 0.f : acc[g][v];
    }
    __syncthreads();

    // ---- merge the warps (and write out, or the partition's partial)
    const bool single = nparts <= 1;
    for (int idx = tid; idx < G * D; idx += NW * 32) {
        const int g = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) M = fmaxf(M, cm[ww * G + g]);
        float Ssum = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int ww = 0; ww < NW; ++ww) {
                const float e = exp2f(cm[ww * G + g] - M);
                Ssum += e * cl[ww * G + g];
                O += e * cacc[(ww * G + g) * D + d];
            }
        }
        const int h = hk * G + g;
        const float o = Ssum > 0.f ? O / Ssum : 0.f;
        if (single) {
            store_out(static_cast<QT*>(p.out) + ((size_t)b * p.num_heads + h) * D + d, o * p.v_scale);
        } else {
            const size_t base = ((size_t)b * p.num_heads + h) * p.max_parts + part;
            p.ws_o[base * D + d] = o;
            if (d == 0) {
                p.ws_ml[2 * base] = M;
                p.ws_ml[2 * base + 1] = Ssum;
            }
        }
    }
}

// Merge the partitions of every (sequence, query head) that was split:
//   out = v_scale * sum_p 2^(m_p - M) l_p o_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p.
template <typename QT>
__global__ void __launch_bounds__(128) split_reduce_kernel(const Params p, int D, int BS) {
    const int h = blockIdx.x, b = blockIdx.y;
    const int L = min(max(p.seq_lens[b], 0), p.max_blocks * BS);   // as the decode kernel clamps
    const int nblk = (L + BS - 1) / BS;
    const int nparts = (nblk + p.part_blocks - 1) / p.part_blocks;
    if (nparts <= 1) return;                                // written by the decode kernel
    const size_t base = ((size_t)b * p.num_heads + h) * p.max_parts;
    float M = -INFINITY;
    for (int q = 0; q < nparts; ++q) M = fmaxf(M, p.ws_ml[2 * (base + q)]);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float Ssum = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int q = 0; q < nparts; ++q) {
                const float e = exp2f(p.ws_ml[2 * (base + q)] - M) * p.ws_ml[2 * (base + q) + 1];
                Ssum += e;
                O += e * p.ws_o[(base + q) * D + d];
            }
        }
        store_out(static_cast<QT*>(p.out) + ((size_t)b * p.num_heads + h) * D + d,
                  Ssum > 0.f ? O / Ssum * p.v_scale : 0.f);
    }
}

// ----------------------------------------------------------------- host launch
struct Args {
    void* out;
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    int num_seqs, max_blocks, num_blocks, num_heads, num_kv_heads, head_dim, block_size;
    float scale, k_scale, v_scale;
    void* workspace;
    size_t workspace_bytes;
    cudaStream_t stream;
    int* err;
};

constexpr int kNumWarps = 4;
constexpr int kMinPartBlocks = 2 * kNumWarps;   // finest split: 8 blocks per partition
constexpr int kMaxDevices = 64;

inline size_t workspace_need(int B, int Hq, int D, int parts) {
    return (size_t)B * Hq * parts * ((size_t)D + 2) * sizeof(float);
}

// Partition size: about 256 KB of K+V per CTA; smaller when that leaves fewer
// than ~2 waves of CTAs; never finer than kMinPartBlocks; one partition when the
// workspace cannot hold the split.
inline int choose_part_blocks(const Args& a, int tile_bytes, int ctas_per_sm, int* parts_out) {
    const int MB = a.max_blocks;
    int target = (256 * 1024) / (2 * tile_bytes);
    target = (target + kNumWarps - 1) / kNumWarps * kNumWarps;
    if (target < kMinPartBlocks) target = kMinPartBlocks;
    int PB = MB < target ? MB : target;
    const long long units = (long long)a.num_seqs * a.num_kv_heads;
    const long long wave = (long long)num_sms() * (ctas_per_sm > 0 ? ctas_per_sm : 1);
    while (PB > kMinPartBlocks && units * ((MB + PB - 1) / PB) < 2 * wave) {
        PB = PB / 2 < kMinPartBlocks ? kMinPartBlocks : PB / 2;
    }
    int parts = (MB + PB - 1) / PB;
    while (parts > 1 && (a.workspace == nullptr ||
                         workspace_need(a.num_seqs, a.num_heads, a.head_dim, parts) > a.workspace_bytes)) {
        PB *= 2;
        if (PB >= MB) PB = MB;
        parts = (MB + PB - 1) / PB;
    }
    if (PB < 1) PB = 1;
    *parts_out = parts;
    return PB;
}

template <typename QT, typename KV, int D, int BS, int G>
int launch_variant(const Args& a) {
    using S = Shape<KV, D, BS, G, kNumWarps>;
    auto kern = paged_decode_kernel<QT, KV, D, BS, G, kNumWarps>;
    static int attr_done[kMaxDevices];      // 0 = not yet, else occupancy + 1
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices)
        return cuda_fail("decode: current device", cudaErrorInvalidDevice);
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             S::kSmem);
        if (e != cudaSuccess) return cuda_fail("decode: set max dynamic shared memory", e);
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kNumWarps * 32, S::kSmem);
        if (e != cudaSuccess) return cuda_fail("decode: occupancy query", e);
        attr_done[dev] = occ + 1;
    }
    int parts = 1;
    const int PB = choose_part_blocks(a, S::kTile, attr_done[dev] - 1, &parts);

    Params p;
    p.out = a.out;
    p.q = a.q;
    p.k_pool = static_cast<const char*>(a.k_pool);
    p.v_pool = static_cast<const char*>(a.v_pool);
    p.block_tables = a.block_tables;
    p.seq_lens = a.seq_lens;
    p.ws_o = parts > 1 ? static_cast<float*>(a.workspace) : nullptr;
    p.ws_ml = parts > 1 ? p.ws_o + (size_t)a.num_seqs * a.num_heads * parts * D : nullptr;
    p.err = a.err;
    p.num_seqs = a.num_seqs;
    p.max_blocks = a.max_blocks;
    p.num_blocks = a.num_blocks;
    p.num_heads = a.num_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.part_blocks = PB;
    p.max_parts = parts;
    p.qscale = a.scale * a.k_scale * kLog2e;
    p.v_scale = a.v_scale;

    dim3 grid(parts, a.num_kv_heads, a.num_seqs);
    kern<<<grid, kNumWarps * 32, S::kSmem, a.stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail("decode: kernel launch", e);
    if (parts > 1) {
        split_reduce_kernel<QT><<<dim3(a.num_heads, a.num_seqs), 128, 0, a.stream>>>(p, D, BS);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail("decode: split merge launch", e);
    }
    return PKV_OK;
}

template <typename QT, typename KV, int D, int BS>
int dispatch_group(const Args& a) {
    switch (a.num_heads / a.num_kv_heads) {
        case 1: return launch_variant<QT, KV, D, BS, 1>(a);
        case 2: return launch_variant<QT, KV, D, BS, 2>(a);
        case 4: return launch_variant<QT, KV, D, BS, 4>(a);
        case 8: return launch_variant<QT, KV, D, BS, 8>(a);
        default: return PKV_ERR_UNSUPPORTED;
    }
}

template <typename QT, typename KV>
int dispatch(const Args& a) {
    if (a.head_dim == 64 && a.block_size == 16) return dispatch_group<QT, KV, 64, 16>(a);
    if (a.head_dim == 64 && a.block_size == 32) return dispatch_group<QT, KV, 64, 32>(a);
    if (a.head_dim == 128 && a.block_size == 16) return dispatch_group<QT, KV, 128, 16>(a);
    if (a.head_dim == 128 && a.block_size == 32) return dispatch_group<QT, KV, 128, 32>(a);
    return PKV_ERR_UNSUPPORTED;
}

}  // namespace decode
}  // namespace pkv
