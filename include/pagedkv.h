/*
 * pagedkv.h -- C ABI of libpagedkv: decode-step and chunked-prefill attention
 * over a paged KV cache, the cache writes of a step (slot write, copy-on-write
 * copy, swap copy to and from host memory), and the host-side block manager
 * (with prefix caching, beam-search reshuffles and swapping).
 *
 * Sources, by page title and section:
 *   "PagedAttention" (Ultralytics glossary)
 *     - "Cách phân trang hoạt động" (how paging works): the KV cache is cut into
 *       blocks of a fixed number of tokens (16 by default) that sit anywhere in one
 *       shared pool; each request owns a block table listing its blocks in order; a
 *       block is taken only when the last one is full; the attention kernel reads
 *       keys and values back through that table.
 *     - "Chia sẻ block giữa các chuỗi" (sharing blocks): sequences may point at
 *       the same physical block, with a reference count per block; a block still
 *       used by another sequence is copied before a write (copy-on-write).
 *     - "Các kỹ thuật liên quan" (related techniques): FlashAttention-style
 *       tiling, grouped-query attention, FP8 cache quantisation.
 *   "KV cache paginado e batching contínuo para LLMs" (upskillscore), "Como
 *     funciona": block tables, waste confined to the last block, reference
 *     counts, block-level copy-on-write (allocate, copy, decrement the original),
 *     preemption of whole requests by swapping their blocks to CPU memory or by
 *     recomputation.
 *   "vLLM PagedAttention: uma revolução no throughput..." (news.hada.io), the
 *     feature list: chunked prefill, prefix caching.
 *
 * Conventions for every call
 *   - Device pointers are plain CUDA device addresses on the current device; the
 *     caller owns every buffer. The library allocates no device memory.
 *     swap_blocks alone also takes pinned host memory (see there).
 *   - Every device call is asynchronous on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream) and does not synchronise.
 *   - Arguments are checked on the host before any launch; a bad argument
 *     returns PKV_ERR_INVALID_ARG or PKV_ERR_UNSUPPORTED and launches nothing.
 *   - Data-dependent errors found on the device (a block id or slot outside the
 *     pool, a wait that gave up) never trap: the offending access is skipped and
 *     a sticky device error word is set; read it with pkv_get_device_error().
 *     pkv_check_wait_timeout() exercises the timeout path without a fault.
 *   - Per-device state (the error word's address, each kernel's shared-memory
 *     set-up, the address of paged_attention_decode_noalloc's scratch) is
 *     looked up once per device and kept for the process: do not use the
 *     library across a cudaDeviceReset of a device it has run on.
 *
 * KV pool layout. The pages show one head as key_pool[block, slot, dim] and
 * say no more; here each pool is [num_blocks][num_kv_heads][tile], one
 * contiguous tile of block_size*head_dim elements per (block, kv head), made of
 * 128-byte "core matrices" (8 rows of 16 bytes; X = 16 bytes of elements: 4
 * float32, 8 bfloat16, 16 E4M3):
 *     K tile: [block_size/8][head_dim/X][8][X]  core matrix (g, c) = tokens
 *             8g..8g+7 (rows) x dims cX..cX+X-1;
 *     V tile: [block_size/X][head_dim/8][8][X]  core matrix (c, g) = dims
 *             8g..8g+7 (rows) x tokens cX..cX+X-1 (V is stored transposed).
 * So K element (blk, h, t, d) is at
 *     (blk*Hkv + h)*bs*D + ((t/8)*(D/X) + d/X)*8X + (t%8)*X + d%X
 * and V element (blk, h, t, d) at
 *     (blk*Hkv + h)*bs*D + ((t/X)*(D/8) + d/8)*8X + (d%8)*X + t%X.
 * A core matrix is what one ldmatrix or tensor-core operand row group reads,
 * so every tile lands in shared memory with one 1-D bulk copy already in the
 * operand layout of the tensor cores. block_size must be a multiple of 16.
 * Element type:
 * float32, bfloat16, or E4M3 bytes (OCP FP8, value = code * per-tensor scale).
 * A whole block (every head, K and V) is num_kv_heads*block_size*head_dim
 * elements per pool, contiguous.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

/* Every entry point is exported; everything else in the library is hidden. */
#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every call. */
typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,    /* null/misaligned pointer, bad size or shape   */
    PKV_ERR_UNSUPPORTED = -2,    /* valid but not built (head_dim, dtype, group) */
    PKV_ERR_CUDA = -3,           /* a CUDA runtime call failed                   */
    PKV_ERR_OUT_OF_RANGE = -4,   /* block id / slot / sequence id outside range  */
    PKV_ERR_POOL_EXHAUSTED = -5, /* block manager: no free block left            */
    PKV_ERR_TIMEOUT = -6         /* a device-side wait gave up (see kernels)     */
} pkv_status;

/* Element types. */
typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_E4M3 = 2 } pkv_dtype;

/* Human-readable name of a status code (static string). */
PKV_API const char* pkv_status_string(int status);

/* Message of the last CUDA runtime failure behind a PKV_ERR_CUDA returned to
 * this thread (which call, the runtime's error string and code); "" if none.
 * The string belongs to the library and stays valid until the thread's next
 * failing call. */
PKV_API const char* pkv_last_error_string(void);

/* ------------------------------------------------------------------------
 * paged_attention_decode -- one decode query per sequence, attention over
 * that sequence's cached tokens gathered through its block table
 * (glossary "PagedAttention", "Cách phân trang hoạt động"; tiling and online
 * softmax as in the FlashAttention item of "Các kỹ thuật liên quan").
 *
 * For every sequence b < num_seqs and query head h < num_heads, with
 * G = num_heads / num_kv_heads and L = seq_lens[b]:
 *     K[t] = k_pool[block_tables[b*max_blocks_per_seq + t/block_size]]
 *                  [h/G][t % block_size][:]                         t < L
 *     s_t  = scale * k_scale * <q[b][h], K[t]>
 *     out[b][h] = v_scale * sum_t softmax(s)_t * V[t]
 * L counts every cached token including the one the step just wrote; L == 0
 * gives a zero row. Query head h reads KV head h/G.
 *
 *   out           device, [num_seqs][num_heads][head_dim], dtype q_dtype, written
 *   q             device, [num_seqs][num_heads][head_dim], dtype q_dtype
 *   k_pool/v_pool device, pool layouts above, dtype kv_dtype, 16-byte aligned
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                 ceil(L/block_size) are not read
 *   seq_lens      device int32 [num_seqs], 0 <= L <= max_blocks_per_seq*block_size
 *   num_blocks    number of blocks in each pool (bounds for table entries)
 *   scale         softmax scale (e.g. 1/sqrt(head_dim))
 *   q_dtype/kv_dtype  supported pairs: (F32,F32), (BF16,BF16), (BF16,E4M3)
 *   k_scale/v_scale   per-tensor FP8 scales; must be 1.0 unless kv_dtype is E4M3
 *   workspace     device scratch for split-KV partitions (float32), or NULL;
 *                 with NULL (or workspace_bytes too small for any split) every
 *                 (sequence, kv head) runs as one partition. Size it with
 *                 paged_attention_workspace_size(). Contents need no clearing.
 *   stream        cudaStream_t
 * Supported: head_dim in {64,128}, block_size in {16,32}, G in {1,2,4,8}.
 * A table entry outside [0, num_blocks) is skipped (its tokens get zero
 * weight) and sets the device error word to PKV_ERR_OUT_OF_RANGE.
 * Launches: the decode kernel, then (when it split) the merge. Both, like
 * the kernels of reshape_and_cache and copy_blocks, are launched with
 * programmatic stream serialisation: a kernel's CTAs may be scheduled while the
 * previous launch in the stream finishes, but each waits for that launch (and
 * so for all earlier work in the stream) to complete before touching memory,
 * the merge excepted, which reads only the lengths and groups before that
 * wait. A kernel the caller launches next with programmatic serialisation must
 * itself wait (griddepcontrol.wait) before reading these outputs; stream order
 * for every other kind of work is unchanged.
 * ---------------------------------------------------------------------- */
PKV_API int paged_attention_decode(void* out, const void* q,
                           const void* k_pool, const void* v_pool,
                           const int32_t* block_tables, const int32_t* seq_lens,
                           int num_seqs, int max_blocks_per_seq, int num_blocks,
                           int num_heads, int num_kv_heads, int head_dim, int block_size,
                           float scale, int q_dtype, int kv_dtype,
                           float k_scale, float v_scale,
                           void* workspace, size_t workspace_bytes,
                           void* stream);

/* ------------------------------------------------------------------------
 * paged_attention_decode_grouped -- the same result as paged_attention_decode,
 * with the K/V of shared prefixes read once per group of sequences instead of
 * once per sequence. Sharing is what the block tables allow ("Chia sẻ block giữa
 * các chuỗi": parallel samples of one prompt point at the same physical blocks;
 * "Como funciona": the prompt's KV is stored once); this call also reads it once.
 *
 * A group is up to max_members sequences (batch indices) whose block tables
 * begin with the same group_prefix_blocks[g] physical blocks, full for every
 * member. One CTA per (partition, group, kv head) walks the group's block list:
 * the shared blocks, loaded once and attended by every member's query heads (the
 * members' heads are the rows of the tensor-core tiles), then each member's own
 * blocks, attended by that member's rows only. Long lists are split like long
 * sequences and merged; the sequences in no group are decoded as usual.
 *
 *   seq_group            device int32 [num_seqs]: the sequence's group, -1 if none
 *   group_members        device int32 [num_groups][max_members], -1 padded
 *   group_prefix_blocks  device int32 [num_groups]
 *   max_group_blocks     host int: the longest group's block list (its prefix
 *                        once plus each member's blocks after it, as
 *                        bm_prefix_groups reports it); sizes the group CTAs'
 *                        partitions. <= 0: unknown, max_members *
 *                        max_blocks_per_seq is assumed. A list longer than
 *                        this is cut short and sets PKV_ERR_OUT_OF_RANGE in the
 *                        device error word (wrong outputs, no bad access).
 *   ungrouped_seqs       device int32 [num_ungrouped]: the batch indices in no
 *                        group (they get the regular CTAs); num_ungrouped < 0:
 *                        no list, every sequence is launched and the grouped
 *                        ones leave at once
 * Preconditions (the block manager's bm_prefix_groups meets them): a sequence
 * is in at most one group and seq_group names it; the prefix blocks are the same
 * ids in every member's table. The prefix is clamped to the blocks every member
 * has filled; any other violation gives wrong outputs, never out-of-range
 * accesses.
 * Needs max_members <= 8 and max_members * (num_heads / num_kv_heads) <= 8 and a
 * bf16 or E4M3 cache; otherwise (or with num_groups == 0) it computes exactly
 * what paged_attention_decode computes. Works with or without a workspace.
 * ---------------------------------------------------------------------- */
PKV_API int paged_attention_decode_grouped(void* out, const void* q,
                                   const void* k_pool, const void* v_pool,
                                   const int32_t* block_tables, const int32_t* seq_lens,
                                   int num_seqs, int max_blocks_per_seq, int num_blocks,
                                   int num_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, int q_dtype, int kv_dtype,
                                   float k_scale, float v_scale,
                                   const int32_t* seq_group,
                                   const int32_t* group_members,
                                   const int32_t* group_prefix_blocks,
                                   int num_groups, int max_members, int max_group_blocks,
                                   const int32_t* ungrouped_seqs, int num_ungrouped,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * paged_decode_step -- one decode step in one call: the step's copy-on-write
 * block copies, the slot write of every sequence's new token, then decode
 * attention (glossary "Cách phân trang hoạt động": a new token's K/V goes into
 * the sequence's last block, then the kernel reads every block back through the
 * table; "Chia sẻ block giữa các chuỗi": a write into a shared block copies it
 * first). The result is that of
 *     copy_blocks(k_pool, v_pool, src_dst_pairs, num_pairs, num_blocks, block bytes);
 *     reshape_and_cache(k_new, v_new, k_pool, v_pool, slot_mapping, num_seqs, ...,
 *                       q_dtype as the source dtype, kv_dtype as the cache dtype);
 *     paged_attention_decode_grouped(...)   (paged_attention_decode if num_groups == 0)
 * with the same arguments, k_new / v_new [num_seqs][num_kv_heads][head_dim] of
 * dtype q_dtype and slot_mapping int64 [num_seqs] (one new token per sequence).
 * Precondition (bm_append_slots and bm_plan_decode meet it): slot_mapping[b] is
 * sequence b's newest position, so the slot writes change only the sequences'
 * last blocks. The decode kernel then starts reading every other block while the
 * copies and slot writes finish, and waits for them only before it reads a
 * sequence's last block (the copies are complete by then too). A slot outside
 * that precondition may be read before it is written.
 * Errors: those of the three calls; argument errors come before any launch.
 * ---------------------------------------------------------------------- */
PKV_API int paged_decode_step(const int64_t* src_dst_pairs, int num_pairs, const void* k_new,
                              const void* v_new, const int64_t* slot_mapping, void* out,
                              const void* q, void* k_pool, void* v_pool,
                              const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                              int max_blocks_per_seq, int num_blocks, int num_heads,
                              int num_kv_heads, int head_dim, int block_size, float scale,
                              int q_dtype, int kv_dtype, float k_scale, float v_scale,
                              const int32_t* seq_group, const int32_t* group_members,
                              const int32_t* group_prefix_blocks, int num_groups, int max_members,
                              int max_group_blocks, const int32_t* ungrouped_seqs,
                              int num_ungrouped, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Bytes of workspace that lets paged_attention_decode use its finest split for
 * these sizes (an upper bound; any size works, smaller ones split less). A
 * grouped call splits long group lists too when it has max_members times this. */
PKV_API size_t paged_attention_workspace_size(int num_seqs, int num_heads, int head_dim,
                                      int block_size, int max_blocks_per_seq);

/* ------------------------------------------------------------------------
 * reshape_and_cache -- write each new token's K and V into its pool slot
 * (glossary worked example: token pos goes to block table[pos / block_size],
 * slot pos % block_size; the caller folds both into one slot number).
 *
 * For each token i < num_tokens with s = slot_mapping[i]:
 *     s < 0          : padding, skipped
 *     s >= num_blocks*block_size : skipped, device error PKV_ERR_OUT_OF_RANGE
 *     otherwise      : K and V of token i, every kv head h, are stored as
 *                      element (s/block_size, h, s%block_size, :) of the
 *                      pools (layouts above).
 * With cache_dtype E4M3 the stored byte is round-to-nearest-even, saturating
 * E4M3 of (x / k_scale) (resp. v_scale), the division in IEEE float32.
 *
 *   k, v          device [num_tokens][num_kv_heads][head_dim], dtype src_dtype
 *   k_pool/v_pool device pools, dtype cache_dtype (== src_dtype, or E4M3)
 *   slot_mapping  device int64 [num_tokens]
 * Supported: head_dim a multiple of 16; (src, cache) in {(F32,F32),
 * (BF16,BF16), (F32,E4M3), (BF16,E4M3)}.
 * ---------------------------------------------------------------------- */
PKV_API int reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                      const int64_t* slot_mapping, int num_tokens,
                      int num_kv_heads, int head_dim, int block_size, int num_blocks,
                      int src_dtype, int cache_dtype, float k_scale, float v_scale,
                      void* stream);

/* ------------------------------------------------------------------------
 * copy_blocks -- the copy half of block-level copy-on-write ("Como funciona";
 * glossary "Chia sẻ block giữa các chuỗi"): for each pair p < num_pairs,
 * block src = pairs[2p] is copied over block dst = pairs[2p+1], in both pools,
 * all kv heads (block_bytes bytes per pool).
 *
 *   src_dst_pairs device int64 [num_pairs][2]
 *   block_bytes   bytes of one block of one pool
 *                 (= num_kv_heads*block_size*head_dim*element size); a
 *                 multiple of 16
 * Preconditions (met by the block manager, whose dst is always a block it has
 * just taken from the free list): dst values are distinct and no dst is also a
 * src (of any pair, its own included); otherwise which bytes land is
 * unspecified. A launch of at most 4096 pairs checks this on the device (one
 * read of every pair per pair, while the copies' loads are in flight) and sets
 * PKV_ERR_INVALID_ARG in the device error word on a violation; the copies still
 * run, in bounds. Larger launches are not checked. A pair with an id outside
 * [0, num_blocks) is skipped and sets PKV_ERR_OUT_OF_RANGE on the device.
 * ---------------------------------------------------------------------- */
PKV_API int copy_blocks(void* k_pool, void* v_pool, const int64_t* src_dst_pairs,
                int num_pairs, int num_blocks, size_t block_bytes, void* stream);

/* ------------------------------------------------------------------------
 * paged_attention_prefill -- chunked prefill: several new query tokens per
 * sequence, each attending causally over that sequence's cached tokens
 * gathered through its block table. Chunked prefill (a long prompt's prefill
 * cut into chunks run as separate steps) is in the feature list of "vLLM
 * PagedAttention: uma revolução no throughput..."; a token attends to itself
 * and to every token before it ("KV cache paginado...", opening paragraph:
 * the autoregressive model keeps K/V of every token already seen); the tiled,
 * score-matrix-free kernel is the FlashAttention item of the glossary's
 * "Các kỹ thuật liên quan".
 *
 * Sequence b (b < num_seqs) holds L = seq_lens[b] cached tokens, its chunk's
 * own K/V already written (reshape_and_cache); the chunk is the last
 * C = query_start[b+1] - query_start[b] of them. For chunk query i < C
 * (position p = L - C + i) and query head h (KV head h/G, G = num_heads /
 * num_kv_heads):
 *     out[query_start[b] + i][h] = sum_{t <= p} softmax_t(scale * <q[.][h], K[t]>) V[t]
 *
 *   out           device, [query_start[num_seqs]][num_heads][head_dim] bf16, written
 *   q             device, [query_start[num_seqs]][num_heads][head_dim] bf16
 *   k_pool/v_pool device, pool layouts above, bf16, 16-byte aligned
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                 ceil(L/block_size) are not read
 *   seq_lens      device int32 [num_seqs], C <= L <= max_blocks_per_seq*block_size
 *   query_start   device int32 [num_seqs + 1], non-decreasing, query_start[0] = 0
 *   max_query_len an upper bound on every C (sizes the grid; queries past it
 *                 are not computed)
 *   q_dtype/kv_dtype  BF16 / BF16
 *   stream        cudaStream_t
 * Supported: head_dim 128, block_size in {16,32}, G dividing 128. Runs on the
 * tcgen05 tensor cores (one 128-row query tile per CTA); allocates nothing.
 * A sequence with C > L or L beyond its table, with rows outside
 * [0, query_start[num_seqs]) (offsets that are not non-decreasing), or a table
 * entry outside [0, num_blocks), sets PKV_ERR_OUT_OF_RANGE in the device error
 * word (the sequence's rows are left unwritten, or the block's keys get zero
 * values). query_start[num_seqs] itself must be the row count of q and out.
 * ---------------------------------------------------------------------- */
PKV_API int paged_attention_prefill(void* out, const void* q,
                            const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            const int32_t* query_start, int num_seqs, int max_query_len,
                            int max_blocks_per_seq, int num_blocks,
                            int num_heads, int num_kv_heads, int head_dim, int block_size,
                            float scale, int q_dtype, int kv_dtype, void* stream);

/* ------------------------------------------------------------------------
 * paged_prefill_step -- one chunked-prefill step in one call: the step's
 * copy-on-write block copies, the slot write of every chunk token, then the
 * chunked-prefill attention. The result is that of
 *     copy_blocks(k_pool, v_pool, src_dst_pairs, num_pairs, num_blocks, block bytes);
 *     reshape_and_cache(k_new, v_new, k_pool, v_pool, slot_mapping, num_tokens, ...,
 *                       BF16, BF16, 1, 1);
 *     paged_attention_prefill(...)
 * with the same arguments, k_new / v_new [num_tokens][num_kv_heads][head_dim]
 * bf16 and slot_mapping int64 [num_tokens].
 * Precondition (the engine's plan_prefill / plan_prompts meet it): the slots
 * are the chunk positions L - C .. L - 1 of their sequences, so the slot writes
 * change only those positions. The attention's loaders then read the key tiles
 * before a sequence's chunk while the copies and slot writes finish, and wait
 * for them only before the first tile holding a chunk position (the copies are
 * complete by then too). A slot outside that precondition may be read before
 * it is written.
 * Errors: those of the three calls; argument errors come before any launch.
 * ---------------------------------------------------------------------- */
PKV_API int paged_prefill_step(const int64_t* src_dst_pairs, int num_pairs, const void* k_new,
                               const void* v_new, const int64_t* slot_mapping, int num_tokens,
                               void* out, const void* q, void* k_pool, void* v_pool,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               const int32_t* query_start, int num_seqs, int max_query_len,
                               int max_blocks_per_seq, int num_blocks, int num_heads,
                               int num_kv_heads, int head_dim, int block_size, float scale,
                               int q_dtype, int kv_dtype, void* stream);

/* ------------------------------------------------------------------------
 * swap_blocks -- copy whole blocks between two pools, e.g. a device pool and a
 * pinned host pool of the same layout, for preemption by swapping
 * ("KV cache paginado e batching contínuo para LLMs", "Como funciona": when
 * physical blocks run out the newest requests are preempted and their blocks
 * swapped to the CPU). For every pair i:
 *     dst_pool[src_dst_pairs[2i+1]] = src_pool[src_dst_pairs[2i]]   (K and V)
 *   dst_k_pool/dst_v_pool, src_k_pool/src_v_pool: device memory or pinned host
 *                 memory (cudaHostAlloc / cudaHostRegister; the device reaches
 *                 it through its mapped address); anything else is
 *                 PKV_ERR_INVALID_ARG. 16-byte aligned.
 *   src_dst_pairs int64 [num_pairs][2], device or pinned host memory; the
 *                 destinations must be distinct and not also sources
 *   src_num_blocks/dst_num_blocks  bounds of the two pools
 *   block_bytes   bytes of one block in one pool (num_kv_heads*block_size*
 *                 head_dim*elt), a multiple of 16
 * A pair outside either pool is skipped and sets PKV_ERR_OUT_OF_RANGE in the
 * device error word. Asynchronous on `stream`.
 * ---------------------------------------------------------------------- */
PKV_API int swap_blocks(void* dst_k_pool, void* dst_v_pool, const void* src_k_pool,
                        const void* src_v_pool, const int64_t* src_dst_pairs, int num_pairs,
                        int src_num_blocks, int dst_num_blocks, size_t block_bytes,
                        void* stream);

/* ------------------------------------------------------------------------
 * paged_attention_decode_noalloc -- paged_attention_decode for callers that
 * cannot allocate device memory where they decode (e.g. a plug-in inside a
 * runtime that owns all device memory, or a serving loop whose memory plan is
 * fixed at start-up so nothing allocates -- and possibly synchronises or fails
 * -- while it serves). The pages have no counterpart: it is a deployment
 * variant of the same computation.
 *
 * Same arguments and result as paged_attention_decode, without workspace: the
 * split-KV scratch is a fixed array inside the library of
 * PKV_NOALLOC_WORKSPACE_BYTES per GPU, held by every GPU that loads the
 * library until the process exits. Nothing is allocated by the call.
 *   - Limit: when the batch can be split at all (that is, when
 *     paged_attention_workspace_size(num_seqs, num_heads, head_dim, block_size,
 *     max_blocks_per_seq) > 0), num_seqs * num_heads * 2 * (head_dim + 2) * 4
 *     bytes (the smallest split) must not exceed PKV_NOALLOC_WORKSPACE_BYTES,
 *     else the call returns PKV_ERR_INVALID_ARG and launches nothing. A batch
 *     that can never be split uses no scratch and has no limit here. Within
 *     the limit the split is chosen to fit the array.
 *   - The first call on a device looks up the array's device address on that
 *     device (once); make that first call before any stream capture.
 *   - All calls on a device share the array: calls that overlap on the GPU
 *     (other streams, other threads) race on it and must be serialised. It
 *     keeps the last call's contents; nothing in it needs clearing.
 * ---------------------------------------------------------------------- */
#define PKV_NOALLOC_WORKSPACE_BYTES (32u * 1024u * 1024u)
PKV_API int paged_attention_decode_noalloc(void* out, const void* q,
                                   const void* k_pool, const void* v_pool,
                                   const int32_t* block_tables, const int32_t* seq_lens,
                                   int num_seqs, int max_blocks_per_seq, int num_blocks,
                                   int num_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, int q_dtype, int kv_dtype,
                                   float k_scale, float v_scale, void* stream);

/* ------------------------------------------------------------------------
 * Stream plumbing of a pipelined step (no counterpart in the pages: it is how
 * a host loop feeds one step after another without spending its time on
 * runtime calls). Streams and events are cudaStream_t / cudaEvent_t passed as
 * void*; the caller creates and owns them and the buffers.
 *
 * pkv_stage_upload: copy `bytes` of a step's packed inputs from pinned host
 * memory to the device on `up_stream` and order the step's kernels (on
 * `compute_stream`) after that copy. When the buffers are being reused, pass
 * the events of their previous step: the copy then waits for
 * `reuse_computed_event` (the previous kernels have read the device buffer),
 * and the compute stream for `reuse_downloaded_event` (the previous output
 * has been read back); NULL otherwise. Records `uploaded_event` on up_stream.
 *
 * pkv_stage_download: record `computed_event` on compute_stream (the step's
 * kernels are enqueued), then copy `bytes` of output to pinned host memory on
 * `down_stream` after it and record `downloaded_event` there.
 *
 * Both are asynchronous and return PKV_OK, PKV_ERR_INVALID_ARG (null buffer or
 * event, zero bytes) or PKV_ERR_CUDA.
 * ---------------------------------------------------------------------- */
PKV_API int pkv_stage_upload(const void* host_src, void* dev_dst, size_t bytes, void* up_stream,
                             void* compute_stream, void* uploaded_event,
                             void* reuse_computed_event, void* reuse_downloaded_event);
PKV_API int pkv_stage_download(const void* dev_src, void* host_dst, size_t bytes,
                               void* compute_stream, void* down_stream, void* computed_event,
                               void* downloaded_event);

/* Kernels this library has launched in this process so far (all devices and
 * streams; for tracing and for counting the launches of a step). */
PKV_API unsigned long long pkv_kernel_launches(void);

/* Synchronise `stream`, then return (in *code) and clear the device error word
 * of the current device: PKV_OK if no kernel recorded an error since the last
 * read, else PKV_ERR_TIMEOUT if a device wait gave up, else PKV_ERR_OUT_OF_RANGE
 * if an id, slot or length was out of range, else PKV_ERR_INVALID_ARG
 * (copy_blocks pairs that break its preconditions).
 * The word is shared by every stream of the device. Once a wait has timed out,
 * every later wait on the device gives up at once until the word is cleared.
 * Returns PKV_OK or PKV_ERR_CUDA. */
PKV_API int pkv_get_device_error(int* code, void* stream);

/* A check of the timeout path on the current device: launches on `stream` one
 * kernel whose bounded wait cannot complete (a barrier nothing arrives at). The
 * wait gives up after its limit (about one second) and sets the device error
 * word, so the next pkv_get_device_error reports PKV_ERR_TIMEOUT; the context
 * stays usable. Until the word is read, every other wait of the library on the
 * device gives up at once, so run it while no other work of the library is in
 * flight on the device. Returns PKV_OK or PKV_ERR_CUDA (launch failed). */
PKV_API int pkv_check_wait_timeout(void* stream);

/* ------------------------------------------------------------------------
 * Host block manager ("Como funciona"; glossary "Cách phân trang hoạt động",
 * "Chia sẻ block giữa các chuỗi"). Host memory only, no CUDA calls; not
 * thread-safe (one manager per thread, or external locking).
 *
 * Rules: blocks are taken from the front of the free list; a sequence takes a
 * new block at its first token and whenever its length is a multiple of
 * block_size; appending into a last block whose reference count is above 1
 * first takes a new block dst, reports (src, dst) for copy_blocks, decrements
 * src and repoints the table; fork shares every block (counts + 1); freeing a
 * sequence decrements its blocks in table order and returns each block that
 * reaches 0 to the tail of the free list.
 * ---------------------------------------------------------------------- */
typedef struct pkv_block_manager pkv_block_manager;

/* free_order: the num_free initially free block ids, front first (distinct,
 * each in [0, num_blocks)). Returns NULL on a bad argument. */
PKV_API pkv_block_manager* bm_create(int num_blocks, int block_size,
                             const int32_t* free_order, int num_free);
PKV_API void bm_destroy(pkv_block_manager* bm);

PKV_API int bm_add_seq(pkv_block_manager* bm, int64_t seq_id);
/* Reserve the next token's slot: *slot = block*block_size + offset. If a
 * copy-on-write is needed *cow_src and *cow_dst get the pair, else both are -1.
 * PKV_ERR_POOL_EXHAUSTED leaves the manager unchanged. */
PKV_API int bm_append_slot(pkv_block_manager* bm, int64_t seq_id, int64_t* slot,
                   int32_t* cow_src, int32_t* cow_dst);
/* n appends to one sequence; the CoW pairs they raise are written as
 * (src, dst) int64 pairs into cow_pairs (capacity cow_cap pairs; n appends raise
 * at most one) and counted in *num_cow.
 *
 * Every batch append (this call, bm_append_slots, bm_append_tokens) is all or
 * nothing. The blocks and CoW pairs the whole batch needs are counted first,
 * without changing anything. PKV_ERR_POOL_EXHAUSTED if the free (plus, with
 * prefix caching, evictable) blocks cannot cover them. PKV_ERR_INVALID_ARG if
 * the pairs exceed cow_cap or a sequence is swapped out. PKV_ERR_OUT_OF_RANGE
 * for an unknown sequence. On any error nothing changes and *num_cow is 0. */
PKV_API int bm_append_n(pkv_block_manager* bm, int64_t seq_id, int n,
                int64_t* cow_pairs, int cow_cap, int* num_cow);
/* One append to each of n sequences (a decode step): slots[i] for seq_ids[i];
 * CoW pairs in order into cow_pairs (capacity n pairs), count in *num_cow. An
 * id may repeat: a chunked-prefill step lists a sequence once per token of its
 * chunk, and its appends then run in list order. All or nothing, as above. */
PKV_API int bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, int n,
                    int64_t* slots, int64_t* cow_pairs, int* num_cow);
PKV_API int bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child);
PKV_API int bm_free_seq(pkv_block_manager* bm, int64_t seq_id);
/* One beam-search step's reshuffle ("PagedAttention" glossary, "Chia sẻ block
 * giữa các chuỗi": beams share blocks through their tables, counted per block).
 * New beam new_ids[i] continues old beam old_ids[parents[i]]: it is forked from
 * it, in order of i; then every old beam is freed, in order (a beam nobody
 * continues returns the blocks only it held). The new beams' next appends copy
 * any shared partial last block (CoW pairs as usual).
 *   old_ids  host int64 [num_old], distinct, existing, not swapped out
 *   parents  host int32 [num_new], each in [0, num_old)
 *   new_ids  host int64 [num_new], distinct, not in use (so not among old_ids)
 * Returns PKV_ERR_OUT_OF_RANGE for an unknown old beam or a parent index out of
 * range, PKV_ERR_INVALID_ARG for a repeated or used id or a swapped-out beam;
 * on any error nothing changes. */
PKV_API int bm_beam_step(pkv_block_manager* bm, const int64_t* old_ids, int num_old,
                 const int32_t* parents, const int64_t* new_ids, int num_new);
/* The sequence's table into out[0..cap), its length in blocks in *n. */
PKV_API int bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* out,
                   int cap, int* n);
/* Dense int32 tables [n][max_blocks] (unused entries -1) and lengths [n] for
 * seq_ids, ready to copy to the device for paged_attention_decode. */
PKV_API int bm_build_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int n,
                    int max_blocks, int32_t* tables, int32_t* seq_lens);
PKV_API int bm_seq_len(const pkv_block_manager* bm, int64_t seq_id, int* len);
PKV_API int bm_refcount(const pkv_block_manager* bm, int block, int* count);
PKV_API int bm_num_free(const pkv_block_manager* bm);
/* Prefix groups for paged_attention_decode_grouped over the batch seq_ids[0..n):
 * sequences whose tables start with the same physical block form a bucket; the
 * buckets are taken in the order of their first member in the batch, and each
 * is cut, in batch order, into consecutive runs of max_members (the last may be
 * shorter). A run's prefix is the number of leading block ids common to all of
 * its members that are full for every member; a run with two or more members
 * and a prefix of at least one block is the next group.
 * Writes group_members [n][max_members] (batch indices, -1 padded; at most n
 * groups), group_prefix [n], seq_group [n] (the sequence's group or -1),
 * group_blocks [n] (may be null: the group's block list for the grouped decode,
 * its prefix once plus each member's blocks after it; the largest is that
 * call's max_group_blocks) and *num_groups. */
PKV_API int bm_prefix_groups(const pkv_block_manager* bm, const int64_t* seq_ids, int n,
                     int max_members, int32_t* group_members, int32_t* group_prefix,
                     int32_t* seq_group, int32_t* group_blocks, int* num_groups);
/* The host half of one decode step in one call, written into caller buffers
 * (e.g. a pinned upload slab) with nothing allocated for the caller: one
 * append per listed sequence (bm_append_slots: slots int64 [n], copy-on-write
 * pairs int64 [n][2], their count in *num_cow), dense tables and lengths
 * (bm_build_tables: int32 [n][max_blocks], int32 [n]) and, when max_members >=
 * 1, the prefix groups (bm_prefix_groups: members int32 [n][max_members],
 * prefixes, list blocks int32 [n], seq_group int32 [n], *num_groups) with the
 * batch indices in no group (ungrouped int32 [n], in batch order,
 * *num_ungrouped) and the longest group list (*max_group_blocks, 0 without
 * groups). Pass max_members <= 0 and null group buffers to skip the groups.
 * All or nothing: a table that would outgrow max_blocks
 * (PKV_ERR_INVALID_ARG), an unknown id (PKV_ERR_OUT_OF_RANGE) or a pool that
 * cannot hold the appends (PKV_ERR_POOL_EXHAUSTED) changes nothing. This is
 * the host work the pages' lazy allocation asks for at every step (glossary
 * "PagedAttention", "Cách phân trang hoạt động"). */
PKV_API int bm_plan_decode(pkv_block_manager* bm, const int64_t* seq_ids, int n, int max_blocks,
                           int64_t* slots, int64_t* cow_pairs, int* num_cow,
                           int32_t* tables, int32_t* seq_lens, int max_members,
                           int32_t* group_members, int32_t* group_prefix, int32_t* seq_group,
                           int32_t* group_blocks, int32_t* ungrouped, int* num_groups,
                           int* num_ungrouped, int* max_group_blocks);

/* ------------------------------------------------------------------------
 * pkv_decode_pipeline_step -- one pipelined decode step, host half and device
 * launches, in one call: bm_plan_decode into the step's pinned host slab
 * (slots, copy-on-write pairs, tables, lengths and, with max_members >= 1,
 * the prefix groups), pkv_stage_upload of the whole slab, paged_decode_step on
 * the slab's device copy with this step's counts (pairs; groups, 0 groups
 * being the plain decode), and pkv_stage_download of the output into
 * `host_out`. The same work as those four calls made one after another (the
 * results are the same, bit for bit), without the host time between them, so
 * a loop feeding short steps keeps up with the device (glossary
 * "PagedAttention", "Cách phân trang hoạt động": the host plans every step's
 * allocation as the sequences grow).
 *
 * `a` describes one buffer set of the pipeline and stays valid across calls:
 * the manager and the step's sequence ids; the host slab views the plan is
 * written to (h_*, sized for the most a step can raise: a pair and a group
 * row per sequence; group_blocks host scratch int32 [num_seqs]); the host and
 * device slabs (slab_bytes each) with the device views of q, k_new, v_new and
 * of the plan inside the device slab; the step's fixed arguments (those of
 * paged_decode_step); the output buffer (out_bytes) and the streams and
 * events of pkv_stage_upload / pkv_stage_download (cudaStream_t, cudaEvent_t).
 * `reuse` != 0 when this buffer set has run a step before: the upload then
 * waits for that step's kernels and the kernels for its read-back.
 * Precondition: the host slab is free, i.e. the caller has waited for the
 * buffer set's previous upload (its uploaded event) before writing q, k_new
 * and v_new there and before this call.
 * Outputs (each may be NULL): counts[4] = copy-on-write pairs, prefix groups,
 * sequences in no group, longest group list; *plan_us = host microseconds
 * spent in bm_plan_decode.
 * Errors: PKV_ERR_INVALID_ARG for a null `a` or `host_out`; otherwise those of
 * bm_plan_decode (before anything is enqueued; the manager is unchanged) and
 * of the three enqueueing calls.
 * ---------------------------------------------------------------------- */
typedef struct pkv_decode_pipeline_step_args {
    pkv_block_manager* bm;
    const int64_t* seq_ids;
    int num_seqs;
    int max_blocks;
    int max_members;
    int64_t* h_slots;
    int64_t* h_pairs;
    int32_t* h_tables;
    int32_t* h_lens;
    int32_t* h_group_members;
    int32_t* h_group_prefix;
    int32_t* h_seq_group;
    int32_t* h_ungrouped;
    int32_t* group_blocks;
    const void* host_slab;
    void* dev_slab;
    size_t slab_bytes;
    const void* q;
    const void* k_new;
    const void* v_new;
    const int64_t* slots;
    const int64_t* pairs;
    const int32_t* tables;
    const int32_t* lens;
    const int32_t* seq_group;
    const int32_t* group_members;
    const int32_t* group_prefix;
    const int32_t* ungrouped;
    void* out;
    void* k_pool;
    void* v_pool;
    int num_blocks;
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int block_size;
    float scale;
    int q_dtype;
    int kv_dtype;
    float k_scale;
    float v_scale;
    void* workspace;
    size_t workspace_bytes;
    size_t out_bytes;
    void* up_stream;
    void* compute_stream;
    void* down_stream;
    void* uploaded_event;
    void* computed_event;
    void* downloaded_event;
} pkv_decode_pipeline_step_args;

PKV_API int pkv_decode_pipeline_step(const pkv_decode_pipeline_step_args* a, int reuse,
                                     void* host_out, int* counts, double* plan_us);

/* Prefix caching (glossary "Chia sẻ block giữa các chuỗi": requests that begin
 * with the same system prompt reuse one copy of the common prefix, with a count
 * per block; "vLLM PagedAttention: uma revolução...": prefix caching).
 * A block filled by tokens whose ids are known is registered under its prefix
 * (every token id from the start of the sequence through the block). A new
 * request reuses, from the front, the registered blocks of its prompt, leaving
 * at least one prompt token to compute. A registered block whose count reaches 0
 * stays cached as "evictable" (a later hit revives it); when a block is needed
 * and the free list is empty, the oldest evictable block is evicted. One release
 * sends uncached blocks to the free list in table order and cached ones to the
 * evictable list in reverse table order. Lookups use a 64-bit hash of the whole
 * prefix and compare the block's own token ids and the hash of the prefix
 * before it (a false hit needs a 64-bit hash collision).
 *
 * bm_enable_prefix_caching: switch it on; only before any sequence is added
 *   (else PKV_ERR_INVALID_ARG). Appends through bm_append_slot / _n / _slots
 *   carry no token ids: their blocks are never registered.
 * bm_add_seq_prompt: create seq_id and reuse the cached blocks of prompt[0..n);
 *   *num_cached = prompt tokens already cached (a multiple of block_size). The
 *   caller appends prompt[*num_cached..n) with bm_append_tokens.
 * bm_append_tokens: n appends with token ids; slots[i] for tokens[i]; CoW pairs
 *   and errors as bm_append_n (all or nothing).
 * bm_cache_stats: blocks looked up / found by bm_add_seq_prompt so far, blocks
 *   registered, evictable blocks.
 * bm_evictable_list: evictable block ids, oldest first, into out[0..cap);
 *   returns their number. */
PKV_API int bm_enable_prefix_caching(pkv_block_manager* bm);
PKV_API int bm_add_seq_prompt(pkv_block_manager* bm, int64_t seq_id, const int32_t* prompt,
                              int n, int* num_cached);
PKV_API int bm_append_tokens(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens, int n,
                             int64_t* slots, int64_t* cow_pairs, int cow_cap, int* num_cow);
PKV_API int bm_cache_stats(const pkv_block_manager* bm, int64_t* hit_blocks,
                           int64_t* lookup_blocks, int* num_cached, int* num_evictable);
PKV_API int bm_evictable_list(const pkv_block_manager* bm, int32_t* out, int cap);

/* Swapping to a host block pool ("KV cache paginado...", "Como funciona":
 * preempted requests, all or nothing, swapped to the CPU).
 * bm_set_host_blocks: give the manager host blocks 0..n-1 (only before any
 *   sequence exists).
 * bm_swap_out: move seq_id to host blocks: pairs[i] = (device block, host block)
 *   for each table entry in order (*num_pairs of them; cap must hold them);
 *   its device blocks are released as by bm_free_seq. PKV_ERR_POOL_EXHAUSTED
 *   (nothing changed) if the host pool cannot take the whole sequence.
 * bm_swap_in: the reverse onto fresh device blocks, pairs = (host, device);
 *   PKV_ERR_POOL_EXHAUSTED if the device pool (free plus evictable blocks)
 *   cannot take it. A swapped-out sequence cannot be appended to, forked or put
 *   in a batch (PKV_ERR_INVALID_ARG); bm_free_seq returns its host blocks.
 * bm_is_swapped, bm_host_free_list: state queries. */
PKV_API int bm_set_host_blocks(pkv_block_manager* bm, int num_host_blocks);
PKV_API int bm_swap_out(pkv_block_manager* bm, int64_t seq_id, int64_t* pairs, int cap,
                        int* num_pairs);
PKV_API int bm_swap_in(pkv_block_manager* bm, int64_t seq_id, int64_t* pairs, int cap,
                       int* num_pairs);
PKV_API int bm_is_swapped(const pkv_block_manager* bm, int64_t seq_id, int* swapped);
PKV_API int bm_host_free_list(const pkv_block_manager* bm, int32_t* out, int cap);

/* The free list, front first, into out[0..cap); returns its length. */
PKV_API int bm_free_list(const pkv_block_manager* bm, int32_t* out, int cap);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
