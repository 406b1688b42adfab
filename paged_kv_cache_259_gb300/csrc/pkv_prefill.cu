// Chunked-prefill attention over the paged KV cache on the fifth-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes: the feature list of "vLLM PagedAttention: uma revolução no
// throughput..." names chunked prefill, a long prompt's prefill split into
// chunks run as separate steps. Sequence b holds seq_lens[b] cached tokens after
// its chunk's own K/V were written; the chunk is its last C_b tokens, and chunk
// query i (position p = L_b - C_b + i) attends keys 0..p, the tokens already
// seen by the autoregressive model (upskillscore "KV cache paginado...", opening
// paragraph). The glossary "PagedAttention" ("Các kỹ thuật liên quan") has
// engines run FlashAttention-style kernels over the paged blocks: the score
// matrix is tiled and never written to memory.
//
// One CTA = one tile of 128 query rows (128/G chunk tokens x the G query heads
// of one KV head, so each K/V tile feeds every head that shares it) of one
// sequence; two CTAs share an SM (half its tensor memory, registers and shared
// memory each), so one CTA's set-up and epilogue overlap the other's tiles and
// the tensor cores alternate between two independent score pipelines. Keys go
// in tiles of 64, so that within its half of the SM a CTA double-buffers the
// scores (tensor memory) and the K and V tiles (shared memory): the scores of
// tile j+1 are computed while the softmax works on tile j. Warp roles:
// * warps 0-3 (softmax, one warpgroup with most of the registers): thread r
//   owns row r = TMEM lane r. Puts its q row into shared memory, then per KV
//   tile reads its 64 scores, applies the causal mask, keeps the running max /
//   sum (exp2 domain, scale * log2 e folded in), writes P (bf16) over the
//   scores it has just read, and finally normalises O;
// * warp 4 (MMA issuer, TMEM owner): one thread issues, in tile order, S = Q K^T
//   (A = Q, B = the K tile, both in shared memory, M = 128, N = 64) and O += P V
//   (A = P from TMEM, B = the V tile, K = 16 keys per instruction): S of tiles
//   0 and 1 at once, then per tile j, P.V(j) as soon as P is written and S of
//   tile j+2 right behind it, into the buffer P(j) has just been read from;
// * warps 5 and 6 (loaders, K and V): copy each tile of 64 keys block by block
//   (through the block table) with 1-D bulk copies, lane i copying block i of
//   the tile, into two K and two V buffers: K of tile j+2 as soon as S(j) is
//   computed, V of tile j+2 as soon as P.V(j) is done. The cache stores every
//   (block, head) tile as 128-byte core matrices, K [bs/8][D/8][8][8] and V
//   [bs/8][D/8][8][8] (8 dims x 8 tokens), which is the canonical no-swizzle
//   K-major operand layout, so a tile lands ready for the tensor cores (S with
//   N = 64 keys over 64/bs blocks, P.V with K = 16 keys per instruction); the q
//   rows are written in the same layout. Keys past the sequence in its last,
//   partly written block get zero V values.
// Tensor memory per CTA: O in columns 0-127, S of even tiles in 128-191, S of
// odd tiles in 192-255, P of a tile over the first 32 columns of its S. S of
// tile j+2 reuses the buffer of tile j and is issued after P.V(j) by the same
// thread; the tensor cores run one thread's MMAs in issue order, so it
// overwrites P(j) only after P.V(j) has read it. Warp 7 only hands its
// registers over.
// The running max is only moved (and O rescaled, after P.V of the previous tile
// has completed) when a tile's max exceeds it by more than 2^8, so O is rarely
// touched; the result is the same softmax.
#include <cmath>

#include <cuda_bf16.h>

#include "pkv_internal.cuh"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace prefill {

constexpr int kD = 128;            // head dim
constexpr int kRows = 128;         // query rows per CTA (M)
constexpr int kKeys = 64;          // keys per KV tile (N of S, K of P.V)
constexpr int kTileBytes = kKeys * kD * 2;         // one K (or V) tile, bf16: 16 KB
constexpr int kQBytes = kRows * kD * 2;            // the q rows: 32 KB
constexpr int kQOff = 0, kKOff = kQBytes, kVOff = kQBytes + 2 * kTileBytes;
constexpr int kSmem = kQBytes + 4 * kTileBytes;    // 96 KB: two CTAs per SM
constexpr int kCtasPerSm = 2;
constexpr int kMmaWarp = 4;                       // MMA issuer, TMEM owner
constexpr int kKLoadWarp = 5, kVLoadWarp = 6;     // warp 7: no role
constexpr int kThreads = 8 * 32;
constexpr int kGroupBytes = (kD / 8) * 128;         // Q, K: 8 rows x 128 dims
constexpr int kChunkBytes = (kD / 8) * 128;         // V: 128 dims x 8 tokens
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 0, kColS = 128;        // O | S of even tiles | S of odd tiles
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kRows, kKeys);   // S: M = 128, N = 64
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kRows, kD);      // P.V: M = N = 128
constexpr uint32_t kKDescHi = tc::desc_hi(kGroupBytes);           // Q, K: SBO = 8-row group
constexpr uint32_t kVDescHi = tc::desc_hi(128);                   // V: SBO = 8-dim group
// Registers: the launch gives every thread kLaunchRegs; the softmax warpgroup
// takes what the other warpgroup (issuers and loaders) gives back.
constexpr int kLaunchRegs = 65536 / (kThreads * kCtasPerSm);      // 128
constexpr uint32_t kSoftmaxRegs = 208, kOtherRegs = 48;

static_assert(kCtasPerSm * (kSmem + 1024) <= 228 * 1024, "two CTAs' shared memory per SM");
static_assert(kCtasPerSm * kTmemCols <= 512, "two CTAs' tensor memory per SM");
static_assert(kColS + 2 * kKeys == kTmemCols, "two score buffers after O");
static_assert(128 * kSoftmaxRegs + 128 * kOtherRegs == (uint32_t)(kThreads * kLaunchRegs),
              "the register split must add up to the launch's registers");

struct Params {
    __nv_bfloat16* out;
    const __nv_bfloat16* q;
    const __nv_bfloat16* k_pool;
    const __nv_bfloat16* v_pool;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* query_start;
    int max_blocks;
    int num_blocks;
    int num_heads;
    int num_kv_heads;
    int G;
    float scale_log2;   // softmax scale * log2(e)
    int* err;
    // Launched (with programmatic stream serialisation) right behind this call's
    // own block copies and chunk slot writes, which change only the chunk
    // positions L - C .. L - 1 of each sequence: the loaders wait for them only
    // before the first key tile holding one of those positions.
    int defer;
};

// 1-D bulk copy global -> shared (TMA engine), completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void st_shared16(uint32_t addr, const uint32_t (&w)[4]) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3])
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared16(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two-wide float32 arithmetic (one instruction for a pair of values) and a
// three-input max: the softmax is bound by instruction issue, so each element
// should cost as few instructions as possible.
__device__ __forceinline__ uint64_t f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Barriers (in this order in shared memory). Two of each for the buffers (K
// and V stages, S and P buffers: tile j uses buffer j % 2, one phase per use),
// so that no waiter can fall two phases behind a barrier: the softmax may
// write P(j+1) before the issuer has waited for P(j), never P(j+2).
enum : int { kBarKFull = 0, kBarVFull = 2, kBarS = 4, kBarPV = 6, kBarP = 8, kBarLand = 10,
             kBarDrain, kNumBars };

// kStageO (one query head per KV head): the output leaves through shared
// memory, see the epilogue.
template <int BS, bool kStageO>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) paged_prefill_kernel(const Params p) {
    constexpr int kBlocksPerTile = kKeys / BS;
    constexpr int kBlockBytes = BS * kD * 2;       // one (block, head) tile
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[kNumBars];
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (p.defer) launch_dependents();
    // grid (query tile, kv head, sequence), the query tile fastest: the tiles
    // of one (sequence, kv head) run side by side and share its K/V through L2
    // (launching every sequence's last tile first instead measured 0.35 / 0.46
    // of the bf16 peak against 0.47 / 0.68); within them the longest goes first
    const int b = blockIdx.z, hk = blockIdx.y;
    const int qtile = gridDim.x - 1 - blockIdx.x;
    const int G = p.G;
    const int tok_per_tile = kRows / G;
    // The loaders read the first two 32-entry windows of the table row before
    // the lengths (the row has max_blocks entries whatever the length), so the
    // first copies need one round trip less; entries past the sequence are
    // ignored as before.
    int pre_ids0 = 0, pre_ids1 = 0;
    if (warp == kKLoadWarp || warp == kVLoadWarp) {
        const int32_t* row = p.block_tables + (size_t)b * p.max_blocks;
        if (lane < p.max_blocks) pre_ids0 = row[lane];
        if (32 + lane < p.max_blocks) pre_ids1 = row[32 + lane];
    }
    const int L = p.seq_lens[b];
    const int q0 = p.query_start[b];
    const int q1 = p.query_start[b + 1];
    const int T = p.query_start[gridDim.z];                // rows of q and out
    const int C = q1 - q0;
    // the chunk's rows must lie inside q and out, and inside the sequence
    if (C < 0 || C > L || L > p.max_blocks * BS || q0 < 0 || q1 > T) {
        if (tid == 0 && C != 0) flag_error(p.err, kErrOutOfRange);
        return;
    }
    const int i0 = qtile * tok_per_tile;
    if (i0 >= C) return;                                   // uniform over the CTA
    const int i_last = min(C, i0 + tok_per_tile) - 1;
    const int p_min = L - C + i0;                          // first query's position
    const int p_max = L - C + i_last;                      // last query's position
    const int n_tiles = p_max / kKeys + 1;                 // tiles of keys 0..p_max
    const int first_masked = (p_min + 1) / kKeys;          // tiles before it need no mask
    const int blk_last = p_max / BS;                       // last block any query sees

    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar0 = smem_addr(bars);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    if (tid == 0) {                                        // the loaders init their own
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarS + i), 1);
            mbar_init(bar(kBarPV + i), 1);
            mbar_init(bar(kBarP + i), 128);
        }
        mbar_init(bar(kBarDrain), 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tc::alloc(smem_addr(&tmem_slot), kTmemCols);
        tc::relinquish_alloc_permit();
    }
    // Loader state (warps 5 and 6: K and V). Block ids come in windows of 32
    // blocks, one per lane, with the next window fetched a window ahead, so table
    // reads never wait on the copies.
    const bool is_v = warp == kVLoadWarp;
    const int bar_full = is_v ? kBarVFull : kBarKFull;
    const int bar_free = is_v ? kBarPV : kBarS;            // the buffer's last reader is done
    const __nv_bfloat16* pool = is_v ? p.v_pool : p.k_pool;
    const int32_t* bt = p.block_tables + (size_t)b * p.max_blocks;
    const int tail = L % BS;                               // tokens in a partly written last block
    int win = 0, win_ids = 0, next_ids = 0;
    int issued = 0;                                        // tiles whose copies went out
    bool land_pending = false;                             // the zero-fill tile's copies
    auto check_id = [&](int blk, int id) {
        if (blk > blk_last) return 0;
        if (id < 0 || id >= p.num_blocks) {
            flag_error(p.err, kErrOutOfRange);
            return 0;                                      // in bounds; the sequence is in error
        }
        return id;
    };
    auto fetch_id = [&](int blk) { return blk > blk_last ? 0 : check_id(blk, bt[blk]); };
    // Copies of tile j into buffer j % 2 (false: a wait timed out)
    const int chunk_tile = (L - C) / kKeys;                // first key tile with a chunk position
    bool waited = !p.defer;
    auto load_tile = [&](int j) -> bool {
        if (!waited && j >= chunk_tile) {                  // this call's slot writes land there
            wait_prerequisites();
            waited = true;
        }
        if ((j * kBlocksPerTile) / 32 != win) {
            ++win;
            win_ids = next_ids;
            next_ids = fetch_id((win + 1) * 32 + lane);
        }
        const int my_id = __shfl_sync(0xffffffffu, win_ids, (j * kBlocksPerTile) % 32 +
                                                                (lane % kBlocksPerTile));
        const int sb = j & 1;                              // buffer of this tile
        // the buffer is free once its previous tile's reader has completed
        if (j >= 2 && !mbar_wait_bounded(bar(bar_free + sb), ((j - 2) >> 1) & 1, p.err)) {
            flag_error(p.err, kErrTimeout);
            return false;
        }
        const uint32_t buf = sbase + (uint32_t)((is_v ? kVOff : kKOff) + sb * kTileBytes);
        const int blk0 = j * kBlocksPerTile;
        const int n_load = min(kBlocksPerTile, blk_last - blk0 + 1);
        // V of the block holding the sequence's last token is zero-filled past
        // it (K there only meets masked scores)
        const bool fix = is_v && tail != 0 && blk_last == (L - 1) / BS &&
                         blk_last < blk0 + kBlocksPerTile;
        const uint32_t land = fix ? bar(kBarLand) : bar(bar_full + sb);
        if (lane == 0) mbar_arrive_expect_tx(land, (uint32_t)(n_load * kBlockBytes));
        __syncwarp();
        if (lane < n_load) {                               // lane jb copies block jb of the tile
            const size_t off = ((size_t)my_id * p.num_kv_heads + hk) * (size_t)(BS * kD);
            bulk_load(buf + (uint32_t)(lane * kBlockBytes), pool + off, kBlockBytes, land);
        }
        issued = j + 1;
        land_pending = fix;
        if (fix) {
            if (!mbar_wait_bounded(bar(kBarLand), 0, p.err)) {
                flag_error(p.err, kErrTimeout);
                return false;
            }
            land_pending = false;
            // V of the last block: [BS/8 chunks][128 dims] rows of 8 tokens
            const uint32_t vb = buf + (uint32_t)((blk_last - blk0) * kBlockBytes);
            for (int row = lane; row < (BS / 8) * kD; row += 32) {
                const int valid = tail - (row / kD) * 8;   // tokens of this row's chunk kept
                if (valid >= 8) continue;
                uint4* v = reinterpret_cast<uint4*>(smem + (vb - sbase) + row * 16);
                uint4 x = *v;
                uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (2 * e >= valid) w[e] = 0u;
                    else if (2 * e + 1 >= valid) w[e] &= 0x0000ffffu;
                }
                *v = x;
            }
            fence_proxy_async_smem();                      // visible to the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bar_full + sb));
        }
        return true;
    };

    // The first DRAM reads go out before the set-up barrier: each softmax
    // thread's q row goes straight to shared memory (row r in the K-major core
    // matrix layout: 8-row groups 2 KB apart, 8-dim chunks 128 bytes apart), and
    // the loaders set up their own barriers and send the copies of the first
    // two tiles (they wait for no other warp; a row's first 64 table entries are
    // inside the table whatever the length, checked where they are used)
    bool load_ok = true;
    if (warp < 4) {
        const int il = tid / G;
        const bool v_ok = i0 + il < C;
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + ((size_t)(q0 + (v_ok ? i0 + il : 0)) * p.num_heads + hk * G + tid % G) * kD);
        uint4 qv[kD / 8];
#pragma unroll
        for (int c = 0; c < kD / 8; ++c) qv[c] = v_ok ? src[c] : make_uint4(0, 0, 0, 0);
        unsigned char* qrow = smem + kQOff + (tid >> 3) * kGroupBytes + (tid & 7) * 16;
#pragma unroll
        for (int c = 0; c < kD / 8; ++c) *reinterpret_cast<uint4*>(qrow + c * 128) = qv[c];
        fence_proxy_async_smem();   // visible to the tensor cores after the barrier below
    } else if (warp == kKLoadWarp || warp == kVLoadWarp) {
        if (lane == 0) {
            mbar_init(bar(bar_full), 1);
            mbar_init(bar(bar_full + 1), 1);
            if (is_v) mbar_init(bar(kBarLand), 1);
            fence_mbar_init();
        }
        __syncwarp();
        win_ids = check_id(lane, pre_ids0);
        next_ids = check_id(32 + lane, pre_ids1);
        for (int j = 0; j < min(2, n_tiles) && load_ok; ++j) load_ok = load_tile(j);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;

    // warpgroup 1 (issuer, loaders) hands registers to warpgroup 0 (softmax)
    if (warp >= 4) {
    tc::regs_dec<kOtherRegs>();
    if (warp == kKLoadWarp || warp == kVLoadWarp) {
        // ------------------------------------------------------------ loaders
        for (int j = 2; j < n_tiles && load_ok; ++j) load_ok = load_tile(j);
        // Every copy this warp issued lands before the CTA may exit, also after a
        // timeout here or in a consumer: wait, with a bound of its own, on the
        // last tile issued on each buffer (a buffer takes a tile only after the
        // previous one there landed and was read, so those phases are
        // unambiguous).
        for (int jj = max(0, issued - 2); jj < issued; ++jj) {
            if (land_pending && jj == issued - 1) continue;   // it lands on kBarLand
            (void)mbar_wait_bounded(bar(bar_full + (jj & 1)), (jj >> 1) & 1, nullptr);
        }
        if (land_pending) (void)mbar_wait_bounded(bar(kBarLand), 0, nullptr);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the issue loop (its descriptors are warp-uniform
        // values); one elected lane issues each MMA and commit.
        bool ok = true;
        auto wait_all = [&](uint32_t b, uint32_t parity) {
            ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(b, parity, p.err));
        };
        // S: A = 128 q rows (8-row groups 2 KB apart, SBO; 8-dim chunks 128
        // bytes apart, LBO); B = 64 keys, the same layout; each 16-dim step
        // starts 256 bytes on for both
        const uint32_t a_lo = tc::desc_lo(sbase + kQOff, 128);
        auto issue_s = [&](int j) {
            const int sb = j & 1;
            wait_all(bar(kBarKFull + sb), (j >> 1) & 1);
            if (!ok) return;
            tc::fence_after_sync();
            const uint32_t b_lo = tc::desc_lo(sbase + kKOff + sb * kTileBytes, 128);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
                tc::mma_ss2_elect(tmem + kColS + sb * kKeys, a_lo + kk * (256 / 16), kKDescHi,
                                  b_lo + kk * (256 / 16), kKDescHi, kIdescS, kk > 0);
            tc::commit_elect(bar(kBarS + sb));
        };
        issue_s(0);
        if (n_tiles > 1) issue_s(1);
        for (int j = 0; j < n_tiles && ok; ++j) {
            const int sb = j & 1;
            wait_all(bar(kBarP + sb), (j >> 1) & 1);
            wait_all(bar(kBarVFull + sb), (j >> 1) & 1);
            if (!ok) break;
            tc::fence_after_sync();
            // 16-key steps that hold a key some query sees (P is 0 past them)
            const int n16 = min(kKeys / 16, (p_max - j * kKeys) / 16 + 1);
            // B = V of 16 keys: two 8-token chunks 2 KB apart (LBO), 8-dim
            // core-matrix rows 128 bytes apart (SBO); each step 4 KB on
            const uint32_t v_lo = tc::desc_lo(sbase + kVOff + sb * kTileBytes, kChunkBytes);
#pragma unroll
            for (int jj = 0; jj < kKeys / 16; ++jj)
                if (jj < n16)
                    tc::mma_ts2_elect(tmem + kColO, tmem + kColS + sb * kKeys + jj * 8,
                                      v_lo + jj * (2 * kChunkBytes / 16), kVDescHi, kIdescO,
                                      (j > 0 || jj > 0));
            tc::commit_elect(bar(kBarPV + sb));
            if (j + 2 < n_tiles) issue_s(j + 2);           // into the buffer P(j) was read from
        }
        if (!ok && lane == 0) flag_error(p.err, kErrTimeout);
        // every MMA issued here is complete before tensor memory is released
        tc::commit_elect(bar(kBarDrain));
        mbar_wait_bounded(bar(kBarDrain), 0, nullptr);     // a real wait even after a timeout
        __syncwarp();
    }
    } else {
        // ------------------------------------------------------------ softmax
        tc::regs_inc<kSoftmaxRegs>();
        const int r = tid;
        const int il = r / G, g = r % G;
        const int i = i0 + il;
        const bool valid = i < C;
        const int pr = valid ? L - C + i : L - 1;
        const int h = hk * G + g;
        const uint32_t row = tmem + ((uint32_t)(warp * 32) << 16);
        bool ok = true;
        const float sc = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j & 1;
            const uint32_t scol = kColS + sb * kKeys;
            ok = ok && mbar_wait_bounded(bar(kBarS + sb), (j >> 1) & 1, p.err);
            ok = __all_sync(0xffffffffu, ok);              // the warp's tcgen05 ops stay converged
            if (!ok) break;
            tc::fence_after_sync();
            uint32_t sv[2][32];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) tc::ld32(row + scol + cb * 32, sv[cb]);
            tc::wait_ld();
            float s[kKeys];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb)
#pragma unroll
                for (int c = 0; c < 32; ++c) s[cb * 32 + c] = __uint_as_float(sv[cb][c]);
            if (j >= first_masked) {
                const int lim = pr - j * kKeys;            // keys 0..lim of this tile are visible
#pragma unroll
                for (int c = 0; c < kKeys; ++c) s[c] = c <= lim ? s[c] : -INFINITY;
            }
            float m8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) m8[c] = fmaxf(s[2 * c], s[2 * c + 1]);
#pragma unroll
            for (int c = 8; c < kKeys / 2; ++c) m8[c & 7] = max3(m8[c & 7], s[2 * c], s[2 * c + 1]);
            const float mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]),
                                  fmaxf(m8[6], m8[7]));
            const float mt = mx * sc;
            if (j == 0) {
                m_run = mt;
            } else if (__any_sync(0xffffffffu, mt > m_run + kRescaleLog2)) {
                // move the running max: O must hold P.V of every earlier tile
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarPV + ((j - 1) & 1)),
                                                               ((j - 1) >> 1) & 1, p.err));
                if (!ok) break;
                tc::fence_after_sync();
                const float m_new = fmaxf(m_run, mt);
                const float alpha = ex2(m_run - m_new);
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t v[32];
                    tc::ld32(row + kColO + cb * 32, v);
                    tc::wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
                    tc::st32(row + kColO + cb * 32, v);
                }
                l_run *= alpha;
                m_run = m_new;
            }
            // P over the scores just read, 32 keys (16 columns) at a time
            const uint64_t sc2 = f2(sc, sc), nm2 = f2(-m_run, -m_run);
            uint64_t l2[4] = {0ull, 0ull, 0ull, 0ull};       // pairs of partial row sums
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    float x0, x1;
                    f2_split(fma2(f2(s[cb * 32 + 2 * c], s[cb * 32 + 2 * c + 1]), sc2, nm2), x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    l2[c & 3] = add2(l2[c & 3], f2(p0, p1));
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                    pk[c] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                tc::st16(row + scol + cb * 16, pk);
            }
            {
                float a0, a1, b0, b1, c0, c1, d0, d1;
                f2_split(l2[0], a0, a1);
                f2_split(l2[1], b0, b1);
                f2_split(l2[2], c0, c1);
                f2_split(l2[3], d0, d1);
                l_run += ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
            }
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(bar(kBarP + sb));
        }
        if (ok) ok = mbar_wait_bounded(bar(kBarPV + ((n_tiles - 1) & 1)), ((n_tiles - 1) >> 1) & 1,
                                       p.err);
        ok = __all_sync(0xffffffffu, ok);
        tc::fence_after_sync();
        if (!ok) {
            flag_error(p.err, kErrTimeout);
        } else {
            const float inv = 1.f / l_run;
            if constexpr (kStageO) {
                // One head per KV head: a warp's 32 rows are 32 tokens, a token's
                // heads apart in memory. O leaves through shared memory (the K
                // stages, free once the last S has completed): each thread writes its
                // bf16 row there (16-byte chunk c at position c ^ (row % 8), so no two
                // lanes of a quarter-warp share banks), then the warp stores two whole
                // rows per instruction (256 contiguous bytes each) instead of 32 rows
                // x 16 bytes.
                const uint32_t stg = sbase + kKOff + warp * (32 * kD * 2);
                fence_proxy_async_smem();              // after the tensor cores' reads there
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t ov[32];
                    tc::ld32(row + kColO + cb * 32, ov);
                    tc::wait_ld();
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 h2 = __floats2bfloat162_rn(
                                __uint_as_float(ov[8 * u + 2 * e]) * inv,
                                __uint_as_float(ov[8 * u + 2 * e + 1]) * inv);
                            w[e] = *reinterpret_cast<const uint32_t*>(&h2);
                        }
                        st_shared16(stg + lane * 256 + (((cb * 4 + u) ^ (lane & 7)) << 4), w);
                    }
                }
                __syncwarp();
                const int half = lane >> 4, ch = lane & 15;
                uint4* const obase = reinterpret_cast<uint4*>(
                    p.out + ((size_t)(q0 + i0 + warp * 32) * p.num_heads + hk) * kD) + ch;
#pragma unroll 4
                for (int m = 0; m < 16; ++m) {
                    const int rr = 2 * m + half;                   // token within the warp's rows
                    const uint4 x = ld_shared16(stg + rr * 256 + ((ch ^ (rr & 7)) << 4));
                    if (i0 + warp * 32 + rr < C) obase[(size_t)rr * p.num_heads * (kD / 8)] = x;
                }
            } else {
                uint4* dst = reinterpret_cast<uint4*>(
                    p.out + ((size_t)(q0 + (valid ? i : 0)) * p.num_heads + h) * kD);
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t ov[32];
                    tc::ld32(row + kColO + cb * 32, ov);
                    tc::wait_ld();
                    if (valid) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 h2 = __floats2bfloat162_rn(
                                    __uint_as_float(ov[8 * u + 2 * e]) * inv,
                                    __uint_as_float(ov[8 * u + 2 * e + 1]) * inv);
                                w[e] = *reinterpret_cast<const uint32_t*>(&h2);
                            }
                            dst[cb * 4 + u] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::dealloc(tmem, kTmemCols);
    }
}

template <int BS, bool kStageO>
int launch(const Params& p, dim3 grid, cudaStream_t stream) {
    auto kern = paged_prefill_kernel<BS, kStageO>;
    int occ = 0;
    const int st = kernel_setup(reinterpret_cast<const void*>(kern), kSmem, kThreads, &occ);
    if (st != PKV_OK) return st;
    // The softmax warpgroup's register increase waits until the other warpgroup
    // has released enough: the split adds up only for the launch's register
    // count, so a build that launches with another count is refused here.
    static int regs_ok = -1;
    if (regs_ok < 0) {
        cudaFuncAttributes fa;
        const cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kern));
        if (e != cudaSuccess) return cuda_fail("prefill: kernel attributes", e);
        regs_ok = fa.numRegs == kLaunchRegs ? 1 : 0;
    }
    if (!regs_ok || occ < 1) return PKV_ERR_UNSUPPORTED;
    note_launch();
    cudaError_t e;
    if (p.defer) {
        e = launch_pdl(kern, grid, dim3(kThreads), kSmem, stream, p);
    } else {
        kern<<<grid, kThreads, kSmem, stream>>>(p);
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? PKV_OK : cuda_fail("prefill: kernel launch", e);
}

}  // namespace prefill
}  // namespace pkv

namespace {

int prefill_common(void* out, const void* q, const void* k_pool, const void* v_pool,
                   const int32_t* block_tables, const int32_t* seq_lens,
                   const int32_t* query_start, int num_seqs, int max_query_len,
                   int max_blocks_per_seq, int num_blocks, int num_heads, int num_kv_heads,
                   int head_dim, int block_size, float scale, int q_dtype, int kv_dtype,
                   void* stream, int defer, bool check_only) {
    using namespace pkv;
    if (num_seqs < 0 || num_seqs > 65535 || max_query_len < 0 || max_blocks_per_seq <= 0 ||
        num_blocks <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_kv_heads > 65535 ||
        head_dim <= 0 || block_size <= 0 || !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    const int G = num_heads / num_kv_heads;
    if (q_dtype != PKV_BF16 || kv_dtype != PKV_BF16 || head_dim != prefill::kD ||
        (block_size != 16 && block_size != 32) || prefill::kRows % G != 0)
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_query_len == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !query_start)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID_ARG;
    const long long rows = (long long)max_query_len * G;
    const long long tiles = (rows + prefill::kRows - 1) / prefill::kRows;
    if (tiles > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    if (check_only) return PKV_OK;
    int* err = error_word();
    if (!err) return PKV_ERR_CUDA;

    prefill::Params p;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
    p.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.query_start = query_start;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.G = G;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    p.defer = defer;
    const dim3 grid((unsigned)tiles, (unsigned)num_kv_heads, (unsigned)num_seqs);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (G == 1)
        return block_size == 16 ? prefill::launch<16, true>(p, grid, s)
                                : prefill::launch<32, true>(p, grid, s);
    return block_size == 16 ? prefill::launch<16, false>(p, grid, s)
                            : prefill::launch<32, false>(p, grid, s);
}

}  // namespace

extern "C" int paged_attention_prefill(void* out, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* seq_lens, const int32_t* query_start,
                                       int num_seqs, int max_query_len, int max_blocks_per_seq,
                                       int num_blocks, int num_heads, int num_kv_heads,
                                       int head_dim, int block_size, float scale, int q_dtype,
                                       int kv_dtype, void* stream) {
    return prefill_common(out, q, k_pool, v_pool, block_tables, seq_lens, query_start, num_seqs,
                          max_query_len, max_blocks_per_seq, num_blocks, num_heads, num_kv_heads,
                          head_dim, block_size, scale, q_dtype, kv_dtype, stream, 0, false);
}

extern "C" int paged_prefill_step(const int64_t* src_dst_pairs, int num_pairs, const void* k_new,
                                  const void* v_new, const int64_t* slot_mapping, int num_tokens,
                                  void* out, const void* q, void* k_pool, void* v_pool,
                                  const int32_t* block_tables, const int32_t* seq_lens,
                                  const int32_t* query_start, int num_seqs, int max_query_len,
                                  int max_blocks_per_seq, int num_blocks, int num_heads,
                                  int num_kv_heads, int head_dim, int block_size, float scale,
                                  int q_dtype, int kv_dtype, void* stream) {
    using namespace pkv;
    if (num_pairs < 0 || num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0 && num_tokens == 0 && (num_seqs == 0 || max_query_len == 0)) return PKV_OK;
    // every argument error is found before anything is launched
    int st = prefill_common(out, q, k_pool, v_pool, block_tables, seq_lens, query_start, num_seqs,
                            max_query_len, max_blocks_per_seq, num_blocks, num_heads,
                            num_kv_heads, head_dim, block_size, scale, q_dtype, kv_dtype, stream,
                            1, true);
    if (st != PKV_OK) return st;
    if (num_tokens > 0 && (!k_new || !v_new || !slot_mapping || !aligned16(k_new) ||
                           !aligned16(v_new) || !k_pool || !v_pool))
        return PKV_ERR_INVALID_ARG;
    if (num_pairs > 0 && (!src_dst_pairs || !k_pool || !v_pool)) return PKV_ERR_INVALID_ARG;
    if (num_pairs > (1 << 30)) return PKV_ERR_UNSUPPORTED;
    const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * 2;
    if (num_pairs > 0) {
        st = copy_blocks(k_pool, v_pool, src_dst_pairs, num_pairs, num_blocks, block_bytes, stream);
        if (st != PKV_OK) return st;
    }
    if (num_tokens > 0) {
        st = reshape_and_cache(k_new, v_new, k_pool, v_pool, slot_mapping, num_tokens,
                               num_kv_heads, head_dim, block_size, num_blocks, q_dtype, kv_dtype,
                               1.f, 1.f, stream);
        if (st != PKV_OK) return st;
    }
    // deferred waits only behind this call's own launches
    return prefill_common(out, q, k_pool, v_pool, block_tables, seq_lens, query_start, num_seqs,
                          max_query_len, max_blocks_per_seq, num_blocks, num_heads, num_kv_heads,
                          head_dim, block_size, scale, q_dtype, kv_dtype, stream,
                          (num_pairs > 0 || num_tokens > 0) ? 1 : 0, false);
}
