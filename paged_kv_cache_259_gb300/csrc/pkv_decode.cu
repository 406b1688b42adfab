// C ABI entry points of decode attention: argument checks and dispatch.
#include <cmath>

#include "pkv_decode_impl.cuh"

namespace pkv {
namespace decode {
int dispatch_f32(const Args& a);
int dispatch_bf16(const Args& a);
int dispatch_e4m3(const Args& a);
}  // namespace decode
}  // namespace pkv

extern "C" {

size_t paged_attention_workspace_size(int num_seqs, int num_heads, int head_dim, int block_size,
                                      int max_blocks_per_seq) {
    using namespace pkv::decode;
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        max_blocks_per_seq <= 0)
        return 0;
    const int parts = (max_blocks_per_seq + kMinPartBlocks - 1) / kMinPartBlocks;
    return parts > 1 ? workspace_need(num_seqs, num_heads, head_dim, parts) : 0;
}

namespace {

int decode_common(void* out, const void* q, const void* k_pool, const void* v_pool,
                  const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                  int max_blocks_per_seq, int num_blocks, int num_heads, int num_kv_heads,
                  int head_dim, int block_size, float scale, int q_dtype, int kv_dtype,
                  float k_scale, float v_scale, const int32_t* seq_group,
                  const int32_t* group_members, const int32_t* group_prefix, int num_groups,
                  int max_members, int max_group_blocks, const int32_t* seq_list, int num_list,
                  void* workspace,
                  size_t workspace_bytes, void* stream, int defer = 0, bool check_only = false) {
    using namespace pkv;
    if (num_seqs < 0 || num_seqs > 65535 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        num_heads <= 0 || num_kv_heads <= 0 || num_kv_heads > 65535 || head_dim <= 0 ||
        block_size <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale) ||
        !(k_scale > 0.f) || !(v_scale > 0.f))
        return PKV_ERR_INVALID_ARG;
    if (kv_dtype != PKV_E4M3 && (k_scale != 1.f || v_scale != 1.f)) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(q) || !aligned16(out))
        return PKV_ERR_INVALID_ARG;
    if (workspace && !aligned16(workspace)) return PKV_ERR_INVALID_ARG;
    if ((head_dim != 64 && head_dim != 128) || (block_size != 16 && block_size != 32))
        return PKV_ERR_UNSUPPORTED;

    decode::Args a;
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.scale = scale;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.workspace = workspace;
    a.workspace_bytes = workspace ? workspace_bytes : 0;
    a.stream = static_cast<cudaStream_t>(stream);
    a.seq_group = seq_group;
    a.seq_list = seq_list;
    a.num_list = num_list;
    a.group_members = group_members;
    a.group_prefix = group_prefix;
    a.num_groups = num_groups;
    a.max_members = max_members;
    a.max_group_blocks = max_group_blocks;
    a.defer = defer;
    if (check_only) {
        const bool pair_ok = (q_dtype == PKV_F32 && kv_dtype == PKV_F32) ||
                             (q_dtype == PKV_BF16 && (kv_dtype == PKV_BF16 || kv_dtype == PKV_E4M3));
        return pair_ok ? PKV_OK : PKV_ERR_UNSUPPORTED;
    }
    a.err = error_word();
    if (!a.err) return PKV_ERR_CUDA;

    if (q_dtype == PKV_F32 && kv_dtype == PKV_F32) return decode::dispatch_f32(a);
    if (q_dtype == PKV_BF16 && kv_dtype == PKV_BF16) return decode::dispatch_bf16(a);
    if (q_dtype == PKV_BF16 && kv_dtype == PKV_E4M3) return decode::dispatch_e4m3(a);
    return PKV_ERR_UNSUPPORTED;
}

}  // namespace

int paged_attention_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                           int max_blocks_per_seq, int num_blocks, int num_heads, int num_kv_heads,
                           int head_dim, int block_size, float scale, int q_dtype, int kv_dtype,
                           float k_scale, float v_scale, void* workspace, size_t workspace_bytes,
                           void* stream) {
    return decode_common(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                         max_blocks_per_seq, num_blocks, num_heads, num_kv_heads, head_dim,
                         block_size, scale, q_dtype, kv_dtype, k_scale, v_scale, nullptr, nullptr,
                         nullptr, 0, 0, 0, nullptr, 0, workspace, workspace_bytes, stream);
}

int paged_attention_decode_grouped(void* out, const void* q, const void* k_pool,
                                   const void* v_pool, const int32_t* block_tables,
                                   const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq,
                                   int num_blocks, int num_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, int q_dtype, int kv_dtype,
                                   float k_scale, float v_scale, const int32_t* seq_group,
                                   const int32_t* group_members, const int32_t* group_prefix_blocks,
                                   int num_groups, int max_members, int max_group_blocks,
                                   const int32_t* ungrouped_seqs, int num_ungrouped,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    // num_ungrouped < 0: no list, every sequence gets a regular CTA (grouped ones
    // leave at once); otherwise the list names the ungrouped batch indices
    if ((num_ungrouped > 0 && !ungrouped_seqs) || num_ungrouped > num_seqs)
        return PKV_ERR_INVALID_ARG;
    if (num_groups < 0 || (num_groups > 0 && (max_members <= 0 || !seq_group ||
                                              !group_members || !group_prefix_blocks)))
        return PKV_ERR_INVALID_ARG;
    if (num_groups > 65535) return PKV_ERR_UNSUPPORTED;
    return decode_common(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                         max_blocks_per_seq, num_blocks, num_heads, num_kv_heads, head_dim,
                         block_size, scale, q_dtype, kv_dtype, k_scale, v_scale,
                         num_groups > 0 ? seq_group : nullptr,
                         num_groups > 0 ? group_members : nullptr,
                         num_groups > 0 ? group_prefix_blocks : nullptr, num_groups, max_members,
                         max_group_blocks, ungrouped_seqs, num_ungrouped, workspace, workspace_bytes, stream);
}

int paged_decode_step(const int64_t* src_dst_pairs, int num_pairs, const void* k_new,
                      const void* v_new, const int64_t* slot_mapping, void* out, const void* q,
                      void* k_pool, void* v_pool, const int32_t* block_tables,
                      const int32_t* seq_lens, int num_seqs, int max_blocks_per_seq,
                      int num_blocks, int num_heads, int num_kv_heads, int head_dim,
                      int block_size, float scale, int q_dtype, int kv_dtype, float k_scale,
                      float v_scale, const int32_t* seq_group, const int32_t* group_members,
                      const int32_t* group_prefix_blocks, int num_groups, int max_members,
                      int max_group_blocks, const int32_t* ungrouped_seqs, int num_ungrouped,
                      void* workspace, size_t workspace_bytes, void* stream) {
    using namespace pkv;
    if (num_pairs < 0 || num_seqs < 0) return PKV_ERR_INVALID_ARG;
    if ((num_ungrouped > 0 && !ungrouped_seqs) || num_ungrouped > num_seqs)
        return PKV_ERR_INVALID_ARG;
    if (num_groups < 0 || (num_groups > 0 && (max_members <= 0 || !seq_group ||
                                              !group_members || !group_prefix_blocks)))
        return PKV_ERR_INVALID_ARG;
    if (num_groups > 65535) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 && num_pairs == 0) return PKV_OK;
    if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
    // every argument error is found before anything is launched
    int st = decode_common(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                           max_blocks_per_seq, num_blocks, num_heads, num_kv_heads, head_dim,
                           block_size, scale, q_dtype, kv_dtype, k_scale, v_scale, nullptr,
                           nullptr, nullptr, 0, 0, 0, nullptr, 0, workspace, workspace_bytes,
                           stream, 1, /*check_only=*/true);
    if (st != PKV_OK) return st;
    if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)))
        return PKV_ERR_INVALID_ARG;
    if (num_pairs > 0 && (!src_dst_pairs || !k_pool || !v_pool)) return PKV_ERR_INVALID_ARG;
    if (num_pairs > (1 << 30)) return PKV_ERR_UNSUPPORTED;
    const size_t elt = kv_dtype == PKV_E4M3 ? 1 : kv_dtype == PKV_BF16 ? 2 : 4;
    const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * elt;
    if (num_pairs > 0) {
        st = copy_blocks(k_pool, v_pool, src_dst_pairs, num_pairs, num_blocks, block_bytes, stream);
        if (st != PKV_OK) return st;
    }
    if (num_seqs > 0) {
        st = reshape_and_cache(k_new, v_new, k_pool, v_pool, slot_mapping, num_seqs, num_kv_heads,
                               head_dim, block_size, num_blocks, q_dtype, kv_dtype, k_scale,
                               v_scale, stream);
        if (st != PKV_OK) return st;
    }
    return decode_common(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                         max_blocks_per_seq, num_blocks, num_heads, num_kv_heads, head_dim,
                         block_size, scale, q_dtype, kv_dtype, k_scale, v_scale,
                         num_groups > 0 ? seq_group : nullptr,
                         num_groups > 0 ? group_members : nullptr,
                         num_groups > 0 ? group_prefix_blocks : nullptr, num_groups, max_members,
                         max_group_blocks, num_groups > 0 ? ungrouped_seqs : nullptr,
                         num_groups > 0 ? num_ungrouped : 0, workspace, workspace_bytes, stream,
                         /*defer=*/1);
}

}  // extern "C"
