// Decode-step attention over a paged KV cache.
//
// "PagedAttention" (Ultralytics glossary), "Cách phân trang hoạt động": the
// attention kernel reads a request's keys and values back block by block
// through its block table, so the cache need not be contiguous. The related-
// techniques section's FlashAttention item: the score vector is never written to
// HBM; here it lives in registers/shared memory and the softmax is computed
// online (running max m, running sum l, accumulator rescaled by 2^(m_old-m_new);
// logits pre-multiplied by log2 e so exp2 is used).
//
// Cache layout (per pool, per block, per kv head: one contiguous tile of
// block_size*head_dim elements, made of 128-byte core matrices of 8 rows x 16
// bytes; X = 16 bytes of elements):
//   K: [bs/8][D/X][8][X]  -- core matrix (g, c) = tokens 8g..8g+7 (rows) x
//                            dims cX..cX+X-1 (Layout::k_off);
//   V: [bs/X][D/8][8][X]  -- transposed: core matrix (c, g) = dims 8g..8g+7
//                            (rows) x tokens cX..cX+X-1 (Layout::v_off).
// Every ldmatrix / 16-byte operand read below is then one core-matrix row
// (bank-conflict-free), and a tile stays one 1-D bulk copy.
//
// Pipeline (shared by both tile-math variants)
//   CTA  = (partition p, kv head hk, sequence b). A partition is PB consecutive
//          logical blocks; with one partition per sequence the CTA writes `out`,
//          otherwise a normalised partial (o_p, m_p, l_p) to the workspace that
//          split_reduce_kernel merges.
//   warp = an independent streaming engine over partition-local blocks
//          w, w+NW, ...: its own STAGES-deep ring of (K tile, V tile) pairs in
//          shared memory, filled by 1-D bulk copies (TMA engine, no tensor map)
//          issued by lane 0 and completed on one mbarrier per stage; block ids
//          come 32 at a time in registers, double-buffered.
//
// Tile math
//   SimtMath (MHA, float32 caches): CUDA-core FMAs. Lanes = (token, chunk
//          plane) for Q.K; lanes own dims for P.V.
//   MmaMath (GQA G in {2,4,8}, bf16 or E4M3 cache; glossary item "Attention truy
//          vấn theo nhóm": G query heads share a KV head): the G heads are the
//          rows of warp-level tensor-core MMAs (m16n8k16, f32 accumulate);
//          S^T = Q K^T then O += P V per 16-token subtile, P kept in registers.
//          E4M3 is converted to f16 in registers (exact) and run as f16 MMA.
//
// Every spin-wait is bounded (pkv::mbar_wait_bounded); a block-table entry
// outside the pool is skipped and recorded in the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <climits>
#include <cmath>
#include <type_traits>

#include "pkv_internal.cuh"

namespace pkv {
namespace decode {

// Build-time tuning (defaults measured on GB300): shared-memory ring bytes per
// CTA, warps per CTA, and the K+V bytes a split-KV partition aims at.
#ifndef PKV_RING_BYTES
#define PKV_RING_BYTES 65536
#endif
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4
#endif
#ifndef PKV_PART_BYTES
#define PKV_PART_BYTES (512 * 1024)
#endif
// Group launches: K+V bytes a group-list partition aims at (coarser than a
// sequence's: a group CTA loads up to 8 query rows and its partials are merged
// per member row); whole lists while the group CTAs fill PKV_GROUP_WHOLE_WAVES
// waves; finer partitions while they fill fewer than PKV_GROUP_MIN_WAVES.
#ifndef PKV_GROUP_PART_BYTES
#define PKV_GROUP_PART_BYTES (768 * 1024)
#endif
#ifndef PKV_GROUP_WHOLE_WAVES
#define PKV_GROUP_WHOLE_WAVES 4
#endif
#ifndef PKV_GROUP_MIN_WAVES
#define PKV_GROUP_MIN_WAVES 2
#endif

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxMembers = 8;                 // members of a prefix group (<= query rows)

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
    // prefix-grouped decode (null / 0 otherwise)
    const int32_t* seq_group;      // [B] group of the sequence, -1 for none
    const int32_t* seq_list;       // regular launch over these batch indices (null: all)
    const int32_t* group_members;  // [num_groups][max_members] batch indices, -1 padded
    const int32_t* group_prefix;   // [num_groups] shared full blocks of the group
    int num_groups;
    int max_members;
    int group_part_blocks;         // partition size of the group launch
    int group_parts;               // partitions the group launch has (its grid x)
    int slots;                     // workspace slots per (sequence, head)
    // Launched right behind this call's own block copies and slot writes, which
    // change only the sequences' last blocks: wait for them only before the
    // copy of an entry holding a last block (see paged_decode_step).
    int defer;
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
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t h;
    const unsigned short in = (unsigned short)(two_bytes & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
    return h;
}
__device__ __forceinline__ void unpack(const uint4& r, float (&f)[16]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t h = e4m3x2_to_f16x2(w[i] >> (16 * j));
            const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&h));
            f[4 * i + 2 * j] = f2.x;
            f[4 * i + 2 * j + 1] = f2.y;
        }
    }
}

template <typename KV, int D, int BS>
struct Layout {
    static constexpr int kElt = Elt<KV>::kSize;
    static constexpr int kX = 16 / kElt;          // elements per 16-byte chunk
    static constexpr int kPlanes = D / kX;        // K chunks per token
    static constexpr int kTile = BS * D * kElt;   // bytes of one (block, kv head) tile
    static constexpr int kVRow = BS * kElt;       // bytes of one dim's tokens in V
    static_assert(D % kX == 0 && D % 8 == 0 && BS % 8 == 0 && BS % kX == 0,
                  "head_dim and block_size must be whole chunks");
    // Both tiles are stored as 128-byte core matrices (8 rows x 16 bytes):
    // K [BS/8][D/X][8][X] (8 tokens x X dims per core matrix), V [BS/X][D/8][8][X]
    // (8 dims x X tokens). Byte offset of K chunk `plane` of token `tok`:
    __host__ __device__ static constexpr int k_off(int plane, int tok) {
        return ((tok >> 3) * kPlanes + plane) * 128 + (tok & 7) * 16;
    }
    // Byte offset of the 16-byte V chunk holding tokens tc*X .. tc*X+X-1 of dim d:
    __host__ __device__ static constexpr int v_off(int d, int tc) {
        return (tc * (D / 8) + (d >> 3)) * 128 + (d & 7) * 16;
    }
};

// ============================================================ CUDA-core tile math
template <typename QT, typename KV, int D, int BS, int G>
struct SimtMath {
    using Lay = Layout<KV, D, BS>;
    using KVT = KV;
    static constexpr int X = Lay::kX, NPL = Lay::kPlanes;
    static constexpr int CPP = 32 / BS;              // chunk planes per warp pass
    static constexpr int PASSES = NPL / CPP;
    static constexpr int DPL = D / 32;               // dims per lane for P.V
    static constexpr int CR = Lay::kVRow / 16;       // 16-byte chunks per V row
    static constexpr int TPC = X;                    // tokens per V chunk
    static constexpr bool kQRegs = (G == 1) && (PASSES * X <= 64);
    static constexpr int kCtaSmemFloats = G * D;     // pre-scaled q rows
    static constexpr int kWarpSmemFloats = G * BS;   // probabilities of one tile
    static_assert(NPL % CPP == 0 && D % 32 == 0 && Lay::kVRow % 16 == 0, "shape");

    struct State {
        float acc[G][DPL];
        float m[G], l[G];
        float qr[kQRegs ? PASSES * X : 1];
    };

    static constexpr bool kPrescaledQ = true;                // q rows carry scale * log2 e
    static constexpr bool kPairStages = false;               // see paged_decode_kernel

    __device__ __forceinline__ static void init(State& st, const float* qs, int lane) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            st.m[g] = -INFINITY;
            st.l[g] = 0.f;
#pragma unroll
            for (int k = 0; k < DPL; ++k) st.acc[g][k] = 0.f;
        }
        if constexpr (kQRegs) {
            const int cp = lane / BS;
#pragma unroll
            for (int i = 0; i < PASSES; ++i)
#pragma unroll
                for (int x = 0; x < X; ++x) st.qr[i * X + x] = qs[(i * CPP + cp) * X + x];
        }
    }

    __device__ __forceinline__ static void tile(State& st, const unsigned char* kt,
                                                const unsigned char* vt, int ntok, int lane,
                                                const float* qs, float* pb) {
        const int t = lane % BS, cp = lane / BS;
        // ---- scores: lane (t, cp) covers chunk planes cp, cp+CPP, ...
        float s[G];
#pragma unroll
        for (int g = 0; g < G; ++g) s[g] = 0.f;
#pragma unroll
        for (int i = 0; i < PASSES; ++i) {
            const int j = i * CPP + cp;
            float kf[X];
            unpack(*reinterpret_cast<const uint4*>(kt + Lay::k_off(j, t)), kf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int x = 0; x < X; ++x) {
                    const float qv = kQRegs ? st.qr[i * X + x] : qs[g * D + j * X + x];
                    s[g] = fmaf(qv, kf[x], s[g]);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if constexpr (CPP == 2) s[g] += __shfl_xor_sync(kFull, s[g], 16);
            if (t >= ntok) s[g] = -INFINITY;
        }
        // ---- online softmax (every lane keeps every head's m, l)
        float alpha[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = s[g];
#pragma unroll
            for (int msk = BS / 2; msk >= 1; msk >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, msk));
            const float m_new = fmaxf(st.m[g], mx);        // finite: token 0 is valid
            alpha[g] = exp2f(st.m[g] - m_new);
            const float pv = exp2f(s[g] - m_new);
            st.m[g] = m_new;
            st.l[g] = st.l[g] * alpha[g] + (cp == 0 ? pv : 0.f);
            if (cp == 0) pb[g * BS + t] = pv;
        }
        __syncwarp();
        // ---- P.V: lane owns dims lane, lane+32, ...; V row = the dim's tokens
        bool moved = false;
#pragma unroll
        for (int g = 0; g < G; ++g) moved |= alpha[g] != 1.f;
        if (__any_sync(kFull, moved)) {                      // running max moved
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int k = 0; k < DPL; ++k) st.acc[g][k] *= alpha[g];
        }
#pragma unroll
        for (int ch = 0; ch < CR; ++ch) {
            if (ch * TPC >= ntok) break;
            const bool partial = (ch + 1) * TPC > ntok;
#pragma unroll
            for (int k = 0; k < DPL; ++k) {
                const int d = lane + 32 * k;
                float vf[TPC];
                unpack(*reinterpret_cast<const uint4*>(vt + Lay::v_off(d, ch)), vf);
                if (partial) {
#pragma unroll
                    for (int x = 0; x < TPC; ++x)
                        if (ch * TPC + x >= ntok) vf[x] = 0.f;      // unwritten slots
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int x4 = 0; x4 < TPC / 4; ++x4) {
                        const float4 pp = *reinterpret_cast<const float4*>(pb + g * BS + ch * TPC + 4 * x4);
                        st.acc[g][k] = fmaf(pp.x, vf[4 * x4 + 0], st.acc[g][k]);
                        st.acc[g][k] = fmaf(pp.y, vf[4 * x4 + 1], st.acc[g][k]);
                        st.acc[g][k] = fmaf(pp.z, vf[4 * x4 + 2], st.acc[g][k]);
                        st.acc[g][k] = fmaf(pp.w, vf[4 * x4 + 3], st.acc[g][k]);
                    }
                }
            }
        }
        __syncwarp();
    }

    __device__ __forceinline__ static void finish(State& st, float* cm, float* cl, float* cacc,
                                                  int w, int lane, bool dead) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float l = st.l[g];
#pragma unroll
            for (int msk = 16; msk >= 1; msk >>= 1) l += __shfl_xor_sync(kFull, l, msk);
            if (lane == 0) {
                cm[w * G + g] = dead ? -INFINITY : st.m[g];
                cl[w * G + g] = dead ? 0.f : l;
            }
#pragma unroll
            for (int k = 0; k < DPL; ++k) cacc[(w * G + g) * D + lane + 32 * k] = dead ? 0.f : st.acc[g][k];
        }
    }
};

// ============================================================ tensor-core tile math
__device__ __forceinline__ void mma16816(bool f16, float& d0, float& d1, uint32_t a0, uint32_t a2,
                                         uint32_t b0, uint32_t b1, float c0, float c1) {
    float j0, j1;
    if (f16)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%10,%11,%12,%13};"
            : "=f"(d0), "=f"(d1), "=f"(j0), "=f"(j1)
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(0.f),
              "f"(0.f));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%10,%11,%12,%13};"
            : "=f"(d0), "=f"(d1), "=f"(j0), "=f"(j1)
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(0.f),
              "f"(0.f));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Fragment roles (lane = 4r + c): rows of every MMA are query heads (row r < G
// real, the rest zero); S^T tile u (8 tokens) column 2c+e; O column 2c+e of
// n-tile nt is dim 8nt+2c+e.
//   bf16: token of S column (u, 2c+e) = 16h + 8u + 2c + e; K B-operand by
//         ldmatrix from the chunk planes, V B-operand by ldmatrix from V rows.
//   E4M3: Q.K dims are permuted inside each 16-dim k-step (lane c's four
//         k-values {2c,2c+1,2c+8,2c+9} are dims 4c..4c+3, one 32-bit load), and
//         so are tokens inside each 16-token subtile (S column (u, 2c+e) is token
//         16h + 4c + 2u + e) so that P's A-fragment needs V bytes 4c..4c+3 of a
//         V row: again one 32-bit load. Q uses the same dim permutation.
template <typename KV, int D, int BS, int G>
struct MmaMath {
    using Lay = Layout<KV, D, BS>;
    using KVT = KV;
    static constexpr bool F8 = std::is_same<KV, uint8_t>::value;
    static constexpr int KS = D / 16;                // k-steps of Q.K
    static constexpr int NT = D / 8;                 // n-tiles of P.V
    static constexpr int SUB = BS / 16;              // 16-token subtiles per block
    static constexpr int kCtaSmemFloats = G * D;     // raw q rows
    static constexpr int kWarpSmemFloats = 0;
    static_assert(G >= 2 && G <= 8 && BS % 16 == 0 && D % 16 == 0, "mma shape");

    struct State {
        uint32_t qa[KS][2];                          // A fragments of Q (a0, a2)
        float o[NT][2];
        float m, l;
    };

    static constexpr bool kPrescaledQ = false;               // scale applied to S in fp32
    // E4M3 cache in 16-token blocks: regular launches stage two blocks at a time
    // (one 32-token tile), halving the per-stage work (barrier, block ids, copy
    // issue) of its 2 KB tiles. Measured on the 16 x 32,768-token E4M3 batch:
    // 0.79 -> 0.81 of the copy bandwidth; the bf16 grouped-query batch lost
    // (0.89 -> 0.85: half as many stages in flight per warp), so bf16 keeps one
    // block per stage.
    static constexpr bool kPairStages = BS == 16 && F8;

    __device__ __forceinline__ static void init(State& st, const float* qs, int lane) {
        const int r = lane >> 2, c = lane & 3;
        const bool live = r < G;
#pragma unroll
        for (int s = 0; s < KS; ++s) {
            float q0 = 0.f, q1 = 0.f, q2 = 0.f, q3 = 0.f;
            const int d0 = F8 ? 16 * s + 4 * c : 16 * s + 2 * c;
            const int d2 = F8 ? 16 * s + 4 * c + 2 : 16 * s + 8 + 2 * c;
            if (live) {
                q0 = qs[r * D + d0];
                q1 = qs[r * D + d0 + 1];
                q2 = qs[r * D + d2];
                q3 = qs[r * D + d2 + 1];
            }
            st.qa[s][0] = F8 ? pack_f16(q0, q1) : pack_bf16(q0, q1);
            st.qa[s][1] = F8 ? pack_f16(q2, q3) : pack_bf16(q2, q3);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) st.o[nt][0] = st.o[nt][1] = 0.f;
        st.m = -INFINITY;
        st.l = 0.f;
    }

    // row_live: bit r set if query row r attends over this tile (all rows, except
    // in a group CTA's own tiles, which belong to one member's rows)
    // MASKED (group launches only): rows outside row_live see -inf scores.
    template <bool MASKED>
    __device__ __forceinline__ static void tile(State& st, const unsigned char* kt,
                                                const unsigned char* vt, int ntok, int lane,
                                                float qscale, const float*, float*, int row_live) {
        const int r = lane >> 2, c = lane & 3;
        const bool live = !MASKED || ((row_live >> r) & 1);
        const uint32_t kbase = smem_addr(kt), vbase = smem_addr(vt);
#pragma unroll
        for (int h = 0; h < SUB; ++h) {
            if (16 * h >= ntok) break;                       // warp-uniform
            // ---- S^T = Q K^T for 16 tokens (two n-tiles of 8); even and odd
            //      k-steps accumulate separately (shorter dependency chains)
            float s[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            float s2[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            uint32_t k8[4];                                  // E4M3: 4 bytes per (k-step, n-tile)
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t b[2][2];
                if constexpr (F8) {
                    // ldmatrix on byte pairs: row = one token's 16 dims of plane ks,
                    // lane (r, c) receives its bytes 4c..4c+3; matrices: (u, ks),
                    // (u, ks+1) for u = 0, 1, loaded every other k-step
                    if ((ks & 1) == 0) {
                        const int m = lane >> 3, rr = lane & 7;
                        const int u = m & 1, plane = ks + (m >> 1);
                        const int tok = 16 * h + 4 * (rr >> 1) + 2 * u + (rr & 1);
                        ldsm_x4(kbase + Lay::k_off(plane, tok), k8[0], k8[1], k8[2], k8[3]);
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t w4 = k8[(ks & 1) * 2 + u];
                        b[u][0] = e4m3x2_to_f16x2(w4);
                        b[u][1] = e4m3x2_to_f16x2(w4 >> 16);
                    }
                } else {
                    const int m = lane >> 3, rr = lane & 7;
                    const int plane = 2 * ks + (m & 1);
                    const int tok = 16 * h + 8 * (m >> 1) + rr;
                    ldsm_x4(kbase + Lay::k_off(plane, tok), b[0][0], b[0][1], b[1][0], b[1][1]);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float(&acc)[2][2] = (ks & 1) ? s2 : s;
                    mma16816(F8, acc[u][0], acc[u][1], st.qa[ks][0], st.qa[ks][1], b[u][0],
                             b[u][1], acc[u][0], acc[u][1]);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                s[u][0] += s2[u][0];
                s[u][1] += s2[u][1];
            }
            // ---- online softmax on this lane's 4 scores of head row r
            float mx = -INFINITY;
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = F8 ? 16 * h + 4 * c + 2 * u + e : 16 * h + 8 * u + 2 * c + e;
                    s[u][e] = (live && tok < ntok) ? s[u][e] * qscale : -INFINITY;
                    mx = fmaxf(mx, s[u][e]);
                }
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
            // a row with no live score yet keeps m = -inf; exponents are taken
            // against 0 then, so nothing becomes NaN and its weights stay 0
            const float m_new = fmaxf(st.m, mx);
            const float m_ref = (MASKED && m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = exp2f(st.m - m_ref);
            float pr[2][2];
            float psum = 0.f;
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    pr[u][e] = exp2f(s[u][e] - m_ref);
                    psum += pr[u][e];
                }
            st.l = st.l * alpha + psum;
            st.m = m_new;
            if (!__all_sync(kFull, alpha == 1.f)) {          // running max moved
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    st.o[nt][0] *= alpha;
                    st.o[nt][1] *= alpha;
                }
            }
            const uint32_t pa0 = F8 ? pack_f16(pr[0][0], pr[0][1]) : pack_bf16(pr[0][0], pr[0][1]);
            const uint32_t pa2 = F8 ? pack_f16(pr[1][0], pr[1][1]) : pack_bf16(pr[1][0], pr[1][1]);
            // ---- O += P V (V rows = dims); unwritten slots beyond ntok are zeroed
            const int tail = ntok - 16 * h;                  // valid tokens in this subtile
            uint32_t v8[4];                                  // E4M3: 4 bytes per n-tile
#pragma unroll
            for (int nt = 0; nt < NT; nt += 2) {
                uint32_t b[2][2];
                if constexpr (F8) {
                    // ldmatrix on byte pairs: row = one dim's 16 tokens of this
                    // subtile, lane (r, c) receives tokens 4c..4c+3 of dim 8nt'+r;
                    // matrices: n-tiles nt..nt+3, loaded every other pair
                    if ((nt & 2) == 0) {
                        const int m = lane >> 3, rr = lane & 7;
                        const int d = 8 * (nt + m) + rr;
                        ldsm_x4(vbase + Lay::v_off(d, h), v8[0], v8[1], v8[2], v8[3]);
                    }
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        uint32_t w4 = v8[(nt & 2) + x];
                        if (tail < 16) {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (4 * c + e >= tail) w4 &= ~(0xffu << (8 * e));
                        }
                        b[x][0] = e4m3x2_to_f16x2(w4);
                        b[x][1] = e4m3x2_to_f16x2(w4 >> 16);
                    }
                } else {
                    const int m = lane >> 3, rr = lane & 7;
                    const int d = 8 * (nt + (m >> 1)) + rr;
                    const int tok = 16 * h + 8 * (m & 1);
                    ldsm_x4(vbase + Lay::v_off(d, tok / 8), b[0][0], b[0][1], b[1][0], b[1][1]);
                    if (tail < 16) {                         // lane holds tokens 2c,2c+1 (+8)
#pragma unroll
                        for (int x = 0; x < 2; ++x)
#pragma unroll
                            for (int y = 0; y < 2; ++y) {
                                const int t0 = 8 * y + 2 * c;
                                if (t0 >= tail) b[x][y] = 0u;
                                else if (t0 + 1 >= tail) b[x][y] &= 0x0000ffffu;
                            }
                    }
                }
#pragma unroll
                for (int x = 0; x < 2; ++x)
                    mma16816(F8, st.o[nt + x][0], st.o[nt + x][1], pa0, pa2, b[x][0], b[x][1],
                             st.o[nt + x][0], st.o[nt + x][1]);
            }
        }
    }

    __device__ __forceinline__ static void finish(State& st, float* cm, float* cl, float* cacc,
                                                  int w, int lane, bool dead) {
        const int r = lane >> 2, c = lane & 3;
        float l = st.l;
        l += __shfl_xor_sync(kFull, l, 1);
        l += __shfl_xor_sync(kFull, l, 2);
        if (r < G) {
            if (c == 0) {
                cm[w * G + r] = dead ? -INFINITY : st.m;
                cl[w * G + r] = dead ? 0.f : l;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                cacc[(w * G + r) * D + 8 * nt + 2 * c] = dead ? 0.f : st.o[nt][0];
                cacc[(w * G + r) * D + 8 * nt + 2 * c + 1] = dead ? 0.f : st.o[nt][1];
            }
        }
    }
};

// ============================================================ pipeline skeleton
template <class Math, int D, int BS, int G, int NW>
struct Pipe {
    using Lay = typename Math::Lay;
    static constexpr int kTile = Lay::kTile;
    // about PKV_RING_BYTES of ring per CTA; at least one stage per warp (a 16 KB
    // tile, float32 D128 with 32-token blocks, gets a single stage)
    static constexpr int kStages = (PKV_RING_BYTES / (NW * 2 * kTile)) < 1 ? 1
                                   : (PKV_RING_BYTES / (NW * 2 * kTile)) > 8 ? 8
                                   : (PKV_RING_BYTES / (NW * 2 * kTile));
    static constexpr int kRingBytes = NW * kStages * 2 * kTile;
    // shared-memory carve-up: ring | mbarriers | stage block ids | q rows | per-warp
    // scratch; the q rows and the scratch start on 16-byte boundaries (float4 reads)
    static constexpr int kBarOff = kRingBytes;
    static constexpr int kIdOff = kBarOff + NW * kStages * 8;          // block id per stage
    static constexpr int kInfoOff = kIdOff + NW * kStages * 4;         // ntok | live rows << 8
    static constexpr int kQOff = (kInfoOff + NW * kStages * 4 + 15) / 16 * 16;
    static constexpr int kWarpOff = kQOff + (Math::kCtaSmemFloats * 4 + 15) / 16 * 16;
    static constexpr int kSmem = kWarpOff + NW * Math::kWarpSmemFloats * 4;
    static_assert(kRingBytes % 128 == 0 && kQOff % 16 == 0 && kWarpOff % 16 == 0 &&
                      (Math::kWarpSmemFloats * 4) % 16 == 0, "shared-memory alignment");
    static_assert(NW * G * (D + 2) * 4 <= kRingBytes, "combine area must fit in the ring");
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

// Query row r of the CTA: (sequence, head), or sequence -1 for an unused row.
// Regular launch: the G heads of kv head hk of sequence b. Group launch: row
// r = m * Gh + g is head hk * Gh + g of the group's m-th member (Gh = the
// model's query heads per kv head), so every member shares the loaded tiles.
template <bool PREFIX, int G>
__device__ __forceinline__ void row_target(const Params& p, int b_or_group, int hk, int r, int* seq,
                                           int* head) {
    if constexpr (!PREFIX) {
        *seq = b_or_group;
        *head = hk * G + r;
    } else {
        const int gh = p.num_heads / p.num_kv_heads;
        const int m = r / gh;
        int s = -1;
        if (m < p.max_members) {
            s = p.group_members[(size_t)b_or_group * p.max_members + m];
            if (s >= p.num_seqs) s = -1;
        }
        *seq = s;
        *head = hk * gh + r % gh;
    }
}

// Shared memory allows three CTAs per SM (about 66 KB each); the bound lets the
// compiler spend the registers that leaves.
// PAIR = 2 (regular launch only): each pipeline stage holds two consecutive
// cache blocks of BS/2 tokens, copied side by side, which is exactly the
// layout of one BS-token tile (K: whole 8-token groups; V: whole X-token
// chunks), so the tile math runs on BS tokens and the per-stage work (barrier,
// block ids, copy issue) is paid once per two blocks. BS is then the stage's
// token count and the cache's block size is BS / PAIR.
template <class Math, typename QT, int D, int BS, int G, int NW, bool PREFIX, int PAIR = 1>
__global__ void __launch_bounds__(NW * 32, 3) paged_decode_kernel(const Params p) {
    using P = Pipe<Math, D, BS, G, NW>;
    constexpr int TILE = P::kTile, ST = P::kStages;
    static_assert(ST <= 32, "prologue stages are taken from one warp-wide read");
    constexpr int PBS = BS / PAIR;                          // the cache's block size
    constexpr int PTILE = TILE / PAIR;                      // one cache block's tile
    static_assert(PAIR == 1 || (PAIR == 2 && !PREFIX), "paired stages: regular launch only");

    // launched with launch_pdl: wait for the previous launch before touching
    // memory, unless it is this call's own step writes (p.defer: then each warp
    // waits before copying an entry that holds a sequence's last block)
    if (p.defer) launch_dependents();
    else pdl_enter();
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::kBarOff);
    int32_t* stage_id = reinterpret_cast<int32_t*>(smem + P::kIdOff);
    float* qs = reinterpret_cast<float*>(smem + P::kQOff);
    float* wsm = reinterpret_cast<float*>(smem + P::kWarpOff);

    // Regular launch: CTA (partition, kv head, sequence b) over blocks
    // [part*PB, ...) of b. Group launch: CTA (partition, kv head, group g) over
    // g's block list -- the P shared prefix blocks (every member's rows live),
    // then each member's own blocks P.. (that member's rows live) -- so a group
    // reads its prompt once and needs no second launch for the members' tails.
    const int part = blockIdx.x, hk = blockIdx.y;
    const int key = (!PREFIX && p.seq_list) ? p.seq_list[blockIdx.z] : (int)blockIdx.z;
    // b, L, own start, own count per member; P, T (one copy per warp)
    __shared__ int grp_all[NW][4 * kMaxMembers + 4];
    int* grp = grp_all[threadIdx.x >> 5];
    int L = 0, nblk = 0;                       // regular launch: the sequence
    int total;                                 // blocks (or list entries) of this CTA's key
    int spec = -1, specP = 0;                  // group launch: see below
    if constexpr (PREFIX) {
        // Every warp reads the group itself (lane m: member m) and keeps its own
        // copy, so no warp waits for another before its first copies. In the
        // round trip of the members' lengths it also reads the table entries of
        // its first 32 list entries that the group's stated prefix covers (the
        // first member's row, as the list takes them): the shared blocks' ids
        // are in when the lengths are, one round trip before the list is known.
        const int ln = threadIdx.x & 31;
        int sb = -1;
        if (ln < kMaxMembers && ln < p.max_members)
            sb = p.group_members[(size_t)key * p.max_members + ln];
        const int P0 = max(p.group_prefix[key], 0);
        const bool ok = sb >= 0 && sb < p.num_seqs;
        const unsigned okm = __ballot_sync(kFull, ok);
        const int row0 = okm ? __shfl_sync(kFull, sb, __ffs(okm) - 1) : -1;
        const int j0 = part * p.part_blocks + (int)(threadIdx.x >> 5) + ln * NW;
        if (row0 >= 0 && j0 < min(P0, p.max_blocks))
            spec = p.block_tables[(size_t)row0 * p.max_blocks + j0];
        const int Lm = ok ? min(max(p.seq_lens[sb], 0), p.max_blocks * BS) : 0;
        // shared blocks are full for every member
        const int P = okm ? min(P0, __reduce_min_sync(kFull, ok ? Lm / BS : INT_MAX)) : 0;
        const int own = ok ? (Lm + BS - 1) / BS - P : 0;
        int incl = own;                                     // members' own blocks, inclusive scan
#pragma unroll
        for (int o = 1; o < kMaxMembers; o <<= 1) {
            const int t = __shfl_up_sync(kFull, incl, o);
            if (ln >= o) incl += t;
        }
        if (ln < kMaxMembers) {
            grp[4 * ln] = ok ? sb : -1;
            grp[4 * ln + 1] = Lm;
            grp[4 * ln + 2] = P + incl - own;               // list index of its first own block
            grp[4 * ln + 3] = own;
        }
        total = P + __shfl_sync(kFull, incl, kMaxMembers - 1);
        if (ln == 0) {
            grp[4 * kMaxMembers] = P;
            grp[4 * kMaxMembers + 1] = total;
        }
        __syncwarp();
        specP = P;
    } else {
        if (key < 0 || key >= p.num_seqs) {                 // a bad ungrouped-list entry
            if (part == 0 && hk == 0 && threadIdx.x == 0) flag_error(p.err, kErrOutOfRange);
            return;
        }
        if (p.seq_group && p.seq_group[key] >= 0) return;  // attended by its group's CTAs
        L = p.seq_lens[key];
        if (L < 0 || L > p.max_blocks * PBS) {              // length the table cannot hold
            if (part == 0 && hk == 0 && threadIdx.x == 0) flag_error(p.err, kErrOutOfRange);
            L = L < 0 ? 0 : p.max_blocks * PBS;
        }
        nblk = (L + BS - 1) / BS;
        total = nblk;
    }
    const int PB = p.part_blocks;
    int nparts = (total + PB - 1) / PB;
    if (PREFIX && nparts > (int)gridDim.x) {                // list longer than the caller said
        if (part == 0 && hk == 0 && threadIdx.x == 0) flag_error(p.err, kErrOutOfRange);
        nparts = gridDim.x;                                 // wrong result, flagged; in bounds
    }
    if (part >= (nparts > 0 ? nparts : 1)) return;          // beyond this key's list
    const int blk0 = part * PB;                             // first entry of this partition
    const int nbp = max(0, min(PB, total - blk0));          // entries in this partition
    const bool single = nparts <= 1;                        // the only contributor: write `out`

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < ST; ++s) mbar_init(smem_addr(&bars[w * ST + s]), 1);
        fence_mbar_init();
    }
    const int nk = nbp > w ? (nbp - w + NW - 1) / NW : 0;  // this warp's blocks
    // regular launch: this warp's entry holding the sequence's last block, or -1
    const int last_rel = nblk - 1 - blk0 - w;
    const int last_kk = (!PREFIX && last_rel >= 0 && last_rel % NW == 0) ? last_rel / NW : -1;
    const uint64_t pol = l2_evict_first();
    const int gh = p.num_heads / p.num_kv_heads;
    const int all_rows = G >= 32 ? -1 : (1 << G) - 1;

    // block id and (ntok | live rows << 8 | group launch: holds a member's last
    // block << 30) of the warp's kk-th entry; with paired stages also the id of
    // the entry's second block (-1 past the sequence)
    constexpr int kLastBit = 1 << 30;
    auto entry = [&](int kk, int* info, int* id2) -> int {
        const int j = blk0 + w + kk * NW;
        int row, blk, ntok, live;
        if constexpr (PREFIX) {
            const int P = grp[4 * kMaxMembers];
            if (j < P) {
                row = grp[0];                               // shared: the first member's table
                for (int m = 0; row < 0 && m + 1 < kMaxMembers; ++m) row = grp[4 * (m + 1)];
                blk = j;
                ntok = BS;
                live = all_rows;
            } else {
                int m = 0;
                while (m + 1 < kMaxMembers && j >= grp[4 * m + 2] + grp[4 * m + 3]) ++m;
                row = grp[4 * m];
                blk = P + (j - grp[4 * m + 2]);
                ntok = min(BS, grp[4 * m + 1] - blk * BS);
                live = ((1 << gh) - 1) << (m * gh);
                if (blk == (grp[4 * m + 1] + BS - 1) / BS - 1) live |= kLastBit >> 8;
            }
        } else {
            row = key;
            blk = j;
            ntok = 0;                                        // derived by the consumer
            live = all_rows;
        }
        *info = ntok | (live << 8);
        const int pb = PAIR * blk;                          // the entry's (first) cache block
        int id = p.block_tables[(size_t)row * p.max_blocks + pb];
        if (id < 0 || id >= p.num_blocks) {
            flag_error(p.err, kErrOutOfRange);
            id = -1;
        }
        *id2 = -1;
        if constexpr (PAIR == 2) {
            if ((pb + 1) * PBS < L) {                       // the sequence reaches the second
                const int i2 = p.block_tables[(size_t)row * p.max_blocks + pb + 1];
                if (i2 < 0 || i2 >= p.num_blocks) {
                    flag_error(p.err, kErrOutOfRange);
                    id = -1;                                // the whole stage is in error
                } else {
                    *id2 = i2;
                }
            }
        }
        return id;
    };
    // 32 entries per warp-wide load, double-buffered in registers; invalid id -> -1
    int info_cur = 0, info_nxt = 0, id2_cur = -1, id2_nxt = -1;
    auto load_chunk = [&](int chunk, int* info, int* id2) -> int {
        const int kk = chunk * 32 + lane;
        *info = 0;
        *id2 = -1;
        return kk < nk ? entry(kk, info, id2) : -1;
    };
    int id_cur = load_chunk(0, &info_cur, &id2_cur);
    int id_nxt = load_chunk(1, &info_nxt, &id2_nxt), chunk_cur = 0;
    auto get_id = [&](int kk, int* info, int* id2) -> int {   // warp-uniform call
        while ((kk >> 5) > chunk_cur) {
            id_cur = id_nxt;
            info_cur = info_nxt;
            id2_cur = id2_nxt;
            ++chunk_cur;
            id_nxt = load_chunk(chunk_cur + 1, &info_nxt, &id2_nxt);
        }
        *info = PREFIX ? __shfl_sync(kFull, info_cur, kk & 31) : 0;
        *id2 = PAIR == 2 ? __shfl_sync(kFull, id2_cur, kk & 31) : -1;
        return __shfl_sync(kFull, id_cur, kk & 31);
    };
    int32_t* stage_info = reinterpret_cast<int32_t*>(smem + P::kInfoOff);
    // the whole converged warp: one elected lane makes the copies and arrivals
    auto issue = [&](int kk, int id, int id2, int info) {
        const int s = kk % ST;
        const uint32_t bar = smem_addr(&bars[w * ST + s]);
        // this step's slot writes land in the sequences' last blocks only
        if (p.defer && (PREFIX ? (info & kLastBit) != 0 : kk == last_kk)) wait_prerequisites();
        if (lane == 0) {
            stage_id[w * ST + s] = id;
            if constexpr (PREFIX) stage_info[w * ST + s] = info & ~kLastBit;
        }
        __syncwarp();
        if (id >= 0) {
            const uint32_t dst = smem_addr(ring + (size_t)((w * ST + s) * 2) * TILE);
            const size_t off = ((size_t)id * p.num_kv_heads + hk) * PTILE;
            const bool two = PAIR == 2 && id2 >= 0;
            mbar_arrive_expect_tx_elect(bar, (two ? 4 : 2) * PTILE);
            bulk_g2s_elect(dst, p.k_pool + off, PTILE, bar, pol);
            bulk_g2s_elect(dst + TILE, p.v_pool + off, PTILE, bar, pol);
            if (two) {                                      // the second block right after
                const size_t off2 = ((size_t)id2 * p.num_kv_heads + hk) * PTILE;
                bulk_g2s_elect(dst + PTILE, p.k_pool + off2, PTILE, bar, pol);
                bulk_g2s_elect(dst + TILE + PTILE, p.v_pool + off2, PTILE, bar, pol);
            }
        } else {
            mbar_arrive_elect(bar);
        }
    };

    // the first stages' copies go out before the q rows are read (each warp
    // uses only its own barriers and ring)
    const int pro = nk < ST ? nk : ST;
    for (int kk = 0; kk < pro; ++kk) {
        int info, id2, id;
        if (PREFIX && blk0 + w + kk * NW < specP) {          // a shared block: read with the lengths
            id = __shfl_sync(kFull, spec, kk);
            if (id < 0 || id >= p.num_blocks) {
                if (lane == 0) flag_error(p.err, kErrOutOfRange);
                id = -1;
            }
            info = BS | (all_rows << 8);
            id2 = -1;
        } else {
            id = get_id(kk, &info, &id2);
        }
        issue(kk, id, id2, info);
    }

    for (int i = tid; i < G * D; i += NW * 32) {            // query rows of this CTA
        const int r = i / D;
        int seq, head;
        row_target<PREFIX, G>(p, key, hk, r, &seq, &head);
        float qv = 0.f;
        if (seq >= 0) qv = to_f(static_cast<const QT*>(p.q)[((size_t)seq * p.num_heads + head) * D + i % D]);
        qs[i] = Math::kPrescaledQ ? qv * p.qscale : qv;
    }
    __syncthreads();

    typename Math::State st;
    Math::init(st, qs, lane);
    float* pb = wsm + w * Math::kWarpSmemFloats;


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
            const int info = PREFIX ? stage_info[w * ST + s] : 0;
            const int ntok = PREFIX ? (info & 0xff) : min(BS, L - (blk0 + w + k * NW) * BS);
            const unsigned char* kt = ring + (size_t)((w * ST + s) * 2) * TILE;
            if constexpr (Math::kWarpSmemFloats > 0)
                Math::tile(st, kt, kt + TILE, ntok, lane, qs, pb);
            else
                Math::template tile<PREFIX>(st, kt, kt + TILE, ntok, lane, p.qscale, qs, pb, info >> 8);
        }
        __syncwarp();
        if (k + ST < nk) {
            int info, id2;
            const int id = get_id(k + ST, &info, &id2);
            fence_proxy_async_smem();
            issue(k + ST, id, id2, info);
        }
    }
    if (aborted) {
        // give up: record it, and let the copies already issued land before the
        // shared memory is reused or released. These waits have a bound of their
        // own and ignore the error word: the timeout bit set above (or by another
        // CTA) must not cut them short while a copy may still be landing.
        if (lane == 0) flag_error(p.err, kErrTimeout);
        const int last = min(nk, k + ST);
        for (int kk = k; kk < last; ++kk)
            (void)mbar_wait_bounded(smem_addr(&bars[w * ST + (kk % ST)]), (kk / ST) & 1, nullptr);
    }

    __syncthreads();                                        // every warp is done with its ring
    float* cm = reinterpret_cast<float*>(ring);             // [NW][G]
    float* cl = cm + NW * G;                                // [NW][G]
    float* cacc = cl + NW * G;                              // [NW][G][D]
    Math::finish(st, cm, cl, cacc, w, lane, aborted);
    __syncthreads();

    // ---- merge the warps (and write out, or the partition's partial)
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
        int seq, h;
        row_target<PREFIX, G>(p, key, hk, g, &seq, &h);
        if (seq < 0) continue;
        const float o = Ssum > 0.f ? O / Ssum : 0.f;
        if (single) {
            store_out(static_cast<QT*>(p.out) + ((size_t)seq * p.num_heads + h) * D + d, o * p.v_scale);
        } else {
            const size_t base = ((size_t)seq * p.num_heads + h) * p.slots + part;
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
// One warp per (sequence, head): lanes take the partitions' (m, l) 32 at a
// time, then the weighted rows are summed with each lane owning D/32 dims.
// A sequence of a prefix group has as many partitions as its group's list.
template <typename QT, int D>
__global__ void __launch_bounds__(256) split_reduce_kernel(const Params p, int BS, int max_len) {
    constexpr int DPL = D / 32;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= p.num_seqs * p.num_heads) return;
    const int b = row / p.num_heads, h = row % p.num_heads;
    int nparts;
    const int g = p.seq_group ? p.seq_group[b] : -1;
    if (g >= p.num_groups) {                               // not a group of this call
        if (h == 0 && lane == 0) flag_error(p.err, kErrOutOfRange);
        return;
    }
    if (g >= 0) {                                          // as the group CTA counts its list
        int P = max(p.group_prefix[g], 0), n = 0, sum = 0;
        for (int m = 0; m < p.max_members && m < kMaxMembers; ++m) {
            const int sb = p.group_members[(size_t)g * p.max_members + m];
            if (sb < 0 || sb >= p.num_seqs) continue;
            const int Lm = min(max(p.seq_lens[sb], 0), p.max_blocks * BS);
            P = min(P, Lm / BS);
            sum += (Lm + BS - 1) / BS;
            ++n;
        }
        if (n == 0) P = 0;
        nparts = (P + sum - n * P + p.group_part_blocks - 1) / p.group_part_blocks;
        nparts = min(nparts, p.group_parts);               // as the group CTAs clamp it
    } else {
        const int L = min(max(p.seq_lens[b], 0), max_len);   // as the decode kernel clamps
        nparts = ((L + BS - 1) / BS + p.part_blocks - 1) / p.part_blocks;
    }
    if (nparts <= 1) return;                               // written by the decode kernel
    // Launched as a programmatic dependent of the decode launch (see
    // launch_merge): everything above was written before that launch began;
    // the partials below only after it has completed.
    wait_prerequisites();
    launch_dependents();
    const size_t base = ((size_t)b * p.num_heads + h) * p.slots;
    const float* ml = p.ws_ml + 2 * base;
    const float* wo = p.ws_o + base * D;
    float M = -INFINITY;
    for (int q = lane; q < nparts; q += 32) M = fmaxf(M, ml[2 * q]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    float S = 0.f;
    if (M != -INFINITY) {
        for (int c = 0; c < nparts; c += 32) {
            const int q = c + lane;
            const float wq = q < nparts ? exp2f(ml[2 * q] - M) * ml[2 * q + 1] : 0.f;
            S += wq;
            const int n = min(32, nparts - c);
            for (int j = 0; j < n; ++j) {
                const float wj = __shfl_sync(kFull, wq, j);
                const float* src = wo + (size_t)(c + j) * D + lane * DPL;
                if constexpr (DPL == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(src);
                    acc[0] = fmaf(wj, v.x, acc[0]);
                    acc[1] = fmaf(wj, v.y, acc[1]);
                    acc[2] = fmaf(wj, v.z, acc[2]);
                    acc[3] = fmaf(wj, v.w, acc[3]);
                } else {
                    const float2 v = *reinterpret_cast<const float2*>(src);
                    acc[0] = fmaf(wj, v.x, acc[0]);
                    acc[1] = fmaf(wj, v.y, acc[1]);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) S += __shfl_xor_sync(kFull, S, o);
    const float inv = S > 0.f ? p.v_scale / S : 0.f;
    QT* dst = static_cast<QT*>(p.out) + ((size_t)b * p.num_heads + h) * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) store_out(dst + i, acc[i] * inv);
}

// ----------------------------------------------------------------- host launch
// The merge of a split call, launched right behind the decode launch(es) of
// the same call as a programmatic dependent: its CTAs may be scheduled (and
// read the lengths and groups) while the decode's last CTAs still run, and
// wait_prerequisites() holds every read of the partials until the decode
// launch has completed and its writes are visible.
template <typename QT, int D>
int launch_merge(const Params& p, int BS, int max_len, cudaStream_t stream) {
    note_launch();
    const unsigned rows = (unsigned)p.num_seqs * p.num_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, split_reduce_kernel<QT, D>, p, BS, max_len);
    return e == cudaSuccess ? PKV_OK : cuda_fail("decode: split merge launch", e);
}

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
    // prefix-grouped decode (all null / 0 for the plain call)
    const int32_t* seq_group;
    const int32_t* seq_list;
    int num_list;
    const int32_t* group_members;
    const int32_t* group_prefix;
    int num_groups, max_members;
    int max_group_blocks;          // longest group list (prefix + own blocks), <= 0: unknown
    int defer = 0;                 // see Params::defer
};

constexpr int kNumWarps = PKV_DECODE_WARPS;
constexpr int kMinPartBlocks = 2 * kNumWarps;   // finest split: 8 blocks per partition
constexpr int kPrefixRows = 8;                  // query rows of a prefix-group CTA

inline size_t workspace_need(int B, int Hq, int D, int slots) {
    return (size_t)B * Hq * slots * ((size_t)D + 2) * sizeof(float);
}

// Partition size: about PKV_PART_BYTES of K+V per CTA; smaller when that leaves
// fewer than ~2 waves of CTAs; never finer than kMinPartBlocks; coarser until the
// workspace holds `copies` sets of partials (2 for grouped decode: prefix and
// own range); one partition when even that does not fit (then *parts_out = 1).
inline int choose_part_blocks(const Args& a, int tile_bytes, int ctas_per_sm, int copies,
                              int* parts_out) {
    const int MB = a.max_blocks;
    int target = PKV_PART_BYTES / (2 * tile_bytes);
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
                         workspace_need(a.num_seqs, a.num_heads, a.head_dim, copies * parts) >
                             a.workspace_bytes)) {
        PB *= 2;
        if (PB >= MB) PB = MB;
        parts = (MB + PB - 1) / PB;
    }
    if (PB < 1) PB = 1;
    *parts_out = parts;
    return PB;
}

template <class Math, typename QT, int D, int BS, int G, bool PREFIX, int PAIR = 1>
int launch_kernel(const Params& p, dim3 grid, cudaStream_t stream) {
    using P = Pipe<Math, D, BS, G, kNumWarps>;
    auto kern = paged_decode_kernel<Math, QT, D, BS, G, kNumWarps, PREFIX, PAIR>;
    int occ = 0;
    const int st = kernel_setup(reinterpret_cast<const void*>(kern), P::kSmem, kNumWarps * 32, &occ);
    if (st != PKV_OK) return st;
    note_launch();
    const cudaError_t e = launch_pdl(kern, grid, dim3(kNumWarps * 32), P::kSmem, stream, p);
    return e == cudaSuccess ? PKV_OK : cuda_fail("decode: kernel launch", e);
}

// Regular launch with paired stages (see paged_decode_kernel): Math runs on
// 2 * the cache's block size; partitions and the merge count in stages.
template <class Math, typename QT, int D, int BS, int G>
int launch_paired(const Args& a) {
    using P = Pipe<Math, D, BS, G, kNumWarps>;
    int occ = 0;
    int st = kernel_setup(
        reinterpret_cast<const void*>(paged_decode_kernel<Math, QT, D, BS, G, kNumWarps, false, 2>),
        P::kSmem, kNumWarps * 32, &occ);
    if (st != PKV_OK) return st;
    Args av = a;
    av.max_blocks = (a.max_blocks + 1) / 2;                 // stages of the longest table
    int parts = 1;
    const int PB = choose_part_blocks(av, P::kTile, occ, 1, &parts);
    Params p{};
    p.out = a.out;
    p.q = a.q;
    p.k_pool = static_cast<const char*>(a.k_pool);
    p.v_pool = static_cast<const char*>(a.v_pool);
    p.block_tables = a.block_tables;
    p.seq_lens = a.seq_lens;
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
    p.slots = parts;
    p.defer = a.defer;
    const bool split = parts > 1;
    p.ws_o = split ? static_cast<float*>(a.workspace) : nullptr;
    p.ws_ml = split ? p.ws_o + (size_t)a.num_seqs * a.num_heads * parts * D : nullptr;
    st = launch_kernel<Math, QT, D, BS, G, false, 2>(p, dim3(parts, a.num_kv_heads, a.num_seqs),
                                                      a.stream);
    if (st != PKV_OK) return st;
    if (split) return launch_merge<QT, D>(p, BS, a.max_blocks * (BS / 2), a.stream);
    return PKV_OK;
}

template <class Math, typename QT, int D, int BS, int G>
int launch_variant(const Args& a) {
    using P = Pipe<Math, D, BS, G, kNumWarps>;
    using KV = typename Math::KVT;
    // grouped decode needs the tensor-core group kernel (bf16 / E4M3 caches) and
    // groups whose members fit the CTA's query rows
    constexpr bool kCanGroup = !std::is_same<KV, float>::value;
    const int gh = a.num_heads / a.num_kv_heads;
    const bool grouped = kCanGroup && a.group_members && a.group_prefix && a.seq_group &&
                         a.num_groups > 0 && a.max_members > 0 && a.max_members <= kMaxMembers &&
                         a.max_members * gh <= kPrefixRows;
    if constexpr (Math::kPairStages) {
        // no prefix groups (every sequence gets regular CTAs): two blocks per stage
        if (!grouped)
            return launch_paired<MmaMath<KV, D, 2 * BS, G>, QT, D, 2 * BS, G>(a);
    }
    int occ = 0;
    int st = kernel_setup(reinterpret_cast<const void*>(paged_decode_kernel<Math, QT, D, BS, G, kNumWarps, false>),
                          P::kSmem, kNumWarps * 32, &occ);
    if (st != PKV_OK) return st;
    int parts = 1;
    const int PB = choose_part_blocks(a, P::kTile, occ, 1, &parts);
    // A group's list is at most max_members tables long, or as long as the
    // caller's max_group_blocks says. Whole lists, one CTA each, while the group
    // CTAs fill ~4 waves and no list is longer than twice a sequence partition
    // (a split costs a merge). Otherwise cut the longest list into equal pieces
    // of about the sequence partition (finer while the group CTAs make fewer than
    // ~2 waves) when the workspace holds their partials.
    int group_list = 0, gPB = 0, gparts = 0;
    if (grouped) {
        group_list = a.max_members * a.max_blocks;
        if (a.max_group_blocks > 0 && a.max_group_blocks < group_list) group_list = a.max_group_blocks;
        const long long gunits = (long long)a.num_groups * a.num_kv_heads;
        const long long wave = (long long)num_sms() * (occ > 0 ? occ : 1);
        int target = PKV_GROUP_PART_BYTES / (2 * P::kTile);
        target = target < kMinPartBlocks ? kMinPartBlocks : target / kNumWarps * kNumWarps;
        if (gunits >= PKV_GROUP_WHOLE_WAVES * wave && group_list <= 2 * target) {
            gparts = 1;
        } else {
            gPB = target;
            while (gPB > kMinPartBlocks &&
                   gunits * ((group_list + gPB - 1) / gPB) < PKV_GROUP_MIN_WAVES * wave)
                gPB = gPB / 2 < kMinPartBlocks ? kMinPartBlocks : gPB / 2;
            gparts = (group_list + gPB - 1) / gPB;
        }
        gPB = ((group_list + gparts - 1) / gparts + kNumWarps - 1) / kNumWarps * kNumWarps;
        gparts = (group_list + gPB - 1) / gPB;
        if (gparts > 1 && (a.workspace == nullptr ||
                           workspace_need(a.num_seqs, a.num_heads, a.head_dim, gparts) >
                               a.workspace_bytes)) {
            gPB = group_list;
            gparts = 1;
        }
    }
    const int slots = gparts > parts ? gparts : parts;

    Params p{};
    p.out = a.out;
    p.q = a.q;
    p.k_pool = static_cast<const char*>(a.k_pool);
    p.v_pool = static_cast<const char*>(a.v_pool);
    p.block_tables = a.block_tables;
    p.seq_lens = a.seq_lens;
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
    p.seq_group = grouped ? a.seq_group : nullptr;
    p.seq_list = nullptr;
    p.group_members = grouped ? a.group_members : nullptr;
    p.group_prefix = grouped ? a.group_prefix : nullptr;
    p.num_groups = grouped ? a.num_groups : 0;
    p.max_members = grouped ? a.max_members : 0;
    p.group_part_blocks = gPB;
    p.group_parts = gparts;
    p.slots = slots;
    p.defer = a.defer;
    const bool split = slots > 1;
    p.ws_o = split ? static_cast<float*>(a.workspace) : nullptr;
    p.ws_ml = split ? p.ws_o + (size_t)a.num_seqs * a.num_heads * slots * D : nullptr;

    if constexpr (kCanGroup) {
        if (grouped) {                                       // shared prefixes, read once per group
            Params pg = p;
            pg.part_blocks = gPB;
            st = launch_kernel<MmaMath<KV, D, BS, kPrefixRows>, QT, D, BS, kPrefixRows, true>(
                pg, dim3(gparts, a.num_kv_heads, a.num_groups), a.stream);
            if (st != PKV_OK) return st;
            p.defer = 0;                                     // the next launch waits for this one
        }
    }
    // sequences of no group (all of them, or the caller's list in a grouped call)
    const bool listed = grouped && a.num_list >= 0;
    p.seq_list = listed ? a.seq_list : nullptr;
    const int n_regular = listed ? a.num_list : a.num_seqs;
    if (n_regular > 0) {
        st = launch_kernel<Math, QT, D, BS, G, false>(p, dim3(parts, a.num_kv_heads, n_regular), a.stream);
        if (st != PKV_OK) return st;
    }
    if (split) return launch_merge<QT, D>(p, BS, a.max_blocks * BS, a.stream);
    return PKV_OK;
}

// float32 caches: CUDA cores for every group size. bf16 / E4M3 caches: CUDA
// cores for MHA (G = 1, one flop per byte), tensor cores for G in {2, 4, 8}.
template <typename QT, typename KV, int D, int BS>
int dispatch_group(const Args& a) {
    constexpr bool simt_only = std::is_same<KV, float>::value;
    switch (a.num_heads / a.num_kv_heads) {
        case 1: return launch_variant<SimtMath<QT, KV, D, BS, 1>, QT, D, BS, 1>(a);
        case 2:
            if constexpr (simt_only) return launch_variant<SimtMath<QT, KV, D, BS, 2>, QT, D, BS, 2>(a);
            else return launch_variant<MmaMath<KV, D, BS, 2>, QT, D, BS, 2>(a);
        case 4:
            if constexpr (simt_only) return launch_variant<SimtMath<QT, KV, D, BS, 4>, QT, D, BS, 4>(a);
            else return launch_variant<MmaMath<KV, D, BS, 4>, QT, D, BS, 4>(a);
        case 8:
            if constexpr (simt_only) return launch_variant<SimtMath<QT, KV, D, BS, 8>, QT, D, BS, 8>(a);
            else return launch_variant<MmaMath<KV, D, BS, 8>, QT, D, BS, 8>(a);
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
