"""The binding refuses malformed arguments before any pointer reaches the
library: shapes, dtypes and layouts are checked first (so these tests need no
GPU), then that every tensor is a contiguous CUDA tensor on one device. A
wrong shape that slipped through would let a kernel index past a buffer."""
import pytest
import torch

from _lib import library, pkv

B, HQ, HKV, D, BS, NB, MB = 3, 4, 2, 64, 16, 8, 5


@pytest.fixture(scope="module", autouse=True)
def lib():
    return library()


def decode_args(**over):
    ks, vs = pkv.pool_shapes(NB, HKV, BS, D, torch.bfloat16)
    a = dict(out=torch.empty(B, HQ, D, dtype=torch.bfloat16),
             q=torch.empty(B, HQ, D, dtype=torch.bfloat16),
             k_pool=torch.empty(ks, dtype=torch.bfloat16),
             v_pool=torch.empty(vs, dtype=torch.bfloat16),
             block_tables=torch.zeros(B, MB, dtype=torch.int32),
             seq_lens=torch.zeros(B, dtype=torch.int32), scale=0.125)
    a.update(over)
    return a


def group_args(**over):
    a = decode_args()
    a.update(seq_group=torch.full((B,), -1, dtype=torch.int32),
             group_members=torch.full((1, 2), -1, dtype=torch.int32),
             group_prefix_blocks=torch.zeros(1, dtype=torch.int32))
    a.update(over)
    return a


DECODE_BAD = [
    ("block_tables short", dict(block_tables=torch.zeros(B - 1, MB, dtype=torch.int32)), ValueError),
    ("block_tables 1-D", dict(block_tables=torch.zeros(B * MB, dtype=torch.int32)), ValueError),
    ("seq_lens short", dict(seq_lens=torch.zeros(B - 1, dtype=torch.int32)), ValueError),
    ("seq_lens int64", dict(seq_lens=torch.zeros(B, dtype=torch.int64)), TypeError),
    ("out short", dict(out=torch.empty(B - 1, HQ, D, dtype=torch.bfloat16)), ValueError),
    ("out dtype", dict(out=torch.empty(B, HQ, D, dtype=torch.float32)), ValueError),
    ("q 2-D", dict(q=torch.empty(B, HQ * D, dtype=torch.bfloat16),
                   out=torch.empty(B, HQ * D, dtype=torch.bfloat16)), ValueError),
    ("head_dim", dict(q=torch.empty(B, HQ, 2 * D, dtype=torch.bfloat16),
                      out=torch.empty(B, HQ, 2 * D, dtype=torch.bfloat16)), ValueError),
    ("pool layout", dict(k_pool=torch.empty(NB, HKV, BS, D, dtype=torch.bfloat16)), ValueError),
    ("not a tensor", dict(seq_lens=[0] * B), TypeError),
]


@pytest.mark.parametrize("name,over,exc", DECODE_BAD, ids=[d[0] for d in DECODE_BAD])
@pytest.mark.parametrize("call", ["decode", "noalloc", "grouped"])
def test_decode_calls_refuse_malformed_arguments(call, name, over, exc):
    if call == "grouped":
        fn, a = pkv.paged_attention_decode_grouped, group_args(**over)
    else:
        fn = pkv.paged_attention_decode if call == "decode" else pkv.paged_attention_decode_noalloc
        a = decode_args(**over)
    with pytest.raises(exc):
        fn(**a)


GROUP_BAD = [
    ("seq_group short", dict(seq_group=torch.full((B - 1,), -1, dtype=torch.int32)), ValueError),
    ("members 1-D", dict(group_members=torch.full((2,), -1, dtype=torch.int32)), ValueError),
    ("prefix length", dict(group_prefix_blocks=torch.zeros(2, dtype=torch.int32)), ValueError),
    ("members int64", dict(group_members=torch.full((1, 2), -1, dtype=torch.int64)), TypeError),
    ("ungrouped 2-D", dict(ungrouped=torch.zeros(1, B, dtype=torch.int32)), ValueError),
    ("ungrouped int64", dict(ungrouped=torch.zeros(B, dtype=torch.int64)), TypeError),
]


@pytest.mark.parametrize("name,over,exc", GROUP_BAD, ids=[g[0] for g in GROUP_BAD])
def test_grouped_decode_refuses_malformed_group_arrays(name, over, exc):
    with pytest.raises(exc):
        pkv.paged_attention_decode_grouped(**group_args(**over))


def test_well_formed_host_tensors_are_refused_as_not_on_the_gpu():
    for fn, a in ((pkv.paged_attention_decode, decode_args()),
                  (pkv.paged_attention_decode_noalloc, decode_args()),
                  (pkv.paged_attention_decode_grouped, group_args())):
        with pytest.raises(TypeError, match="CUDA"):
            fn(**a)


def prefill_args(**over):
    a = decode_args()
    T = 7
    a.update(out=torch.empty(T, HQ, D, dtype=torch.bfloat16),
             q=torch.empty(T, HQ, D, dtype=torch.bfloat16),
             query_start=torch.tensor([0, 2, 5, T], dtype=torch.int32), max_query_len=3)
    a.update(over)
    return a


@pytest.mark.parametrize("over,exc", [
    (dict(query_start=torch.tensor([0, 2, 7], dtype=torch.int32)), ValueError),
    (dict(query_start=torch.tensor([0, 2, 5, 7], dtype=torch.int64)), TypeError),
    (dict(block_tables=torch.zeros(B + 1, MB, dtype=torch.int32)), ValueError),
    (dict(seq_lens=torch.zeros(1, B, dtype=torch.int32)), ValueError),
    (dict(out=torch.empty(6, HQ, D, dtype=torch.bfloat16)), ValueError),
    ({}, TypeError),                                   # well formed, but on the host
])
def test_prefill_refuses_malformed_arguments(over, exc):
    with pytest.raises(exc):
        pkv.paged_attention_prefill(**prefill_args(**over))


def cache_args(**over):
    ks, vs = pkv.pool_shapes(NB, HKV, BS, D, torch.bfloat16)
    a = dict(k=torch.empty(3, HKV, D, dtype=torch.bfloat16),
             v=torch.empty(3, HKV, D, dtype=torch.bfloat16),
             k_pool=torch.empty(ks, dtype=torch.bfloat16),
             v_pool=torch.empty(vs, dtype=torch.bfloat16),
             slot_mapping=torch.zeros(3, dtype=torch.int64))
    a.update(over)
    return a


@pytest.mark.parametrize("over,exc", [
    (dict(k=torch.empty(3, HKV * D, dtype=torch.bfloat16)), ValueError),
    (dict(v=torch.empty(2, HKV, D, dtype=torch.bfloat16)), ValueError),
    (dict(k=torch.empty(3, HKV + 1, D, dtype=torch.bfloat16),
          v=torch.empty(3, HKV + 1, D, dtype=torch.bfloat16)), ValueError),
    (dict(slot_mapping=torch.zeros(4, dtype=torch.int64)), ValueError),
    (dict(slot_mapping=torch.zeros(3, dtype=torch.int32)), TypeError),
    ({}, TypeError),
])
def test_reshape_and_cache_refuses_malformed_arguments(over, exc):
    with pytest.raises(exc):
        pkv.reshape_and_cache(**cache_args(**over))


@pytest.mark.parametrize("over,exc", [
    (dict(src_dst_pairs=torch.zeros(2, 3, dtype=torch.int64)), ValueError),
    (dict(src_dst_pairs=torch.zeros(2, 2, dtype=torch.int32)), ValueError),
    (dict(v_pool=torch.empty(4, dtype=torch.bfloat16)), ValueError),
    ({}, TypeError),
])
def test_copy_blocks_refuses_malformed_arguments(over, exc):
    a = cache_args()
    a = dict(k_pool=a["k_pool"], v_pool=a["v_pool"],
             src_dst_pairs=torch.zeros(2, 2, dtype=torch.int64))
    a.update(over)
    with pytest.raises(exc):
        pkv.copy_blocks(**a)


def _noalloc_batch(max_blocks):
    """1024 sequences x 32 heads, D 128: the smallest split (2 partitions of
    130 floats per sequence and head) needs 34 MB, more than the fixed scratch."""
    b, hq, hkv, d, bs = 1024, 32, 8, 128, 16
    ks, vs = pkv.pool_shapes(4, hkv, bs, d, torch.bfloat16)
    return dict(out=torch.empty(b, hq, d, dtype=torch.bfloat16),
                q=torch.empty(b, hq, d, dtype=torch.bfloat16),
                k_pool=torch.empty(ks, dtype=torch.bfloat16),
                v_pool=torch.empty(vs, dtype=torch.bfloat16),
                block_tables=torch.zeros(b, max_blocks, dtype=torch.int32),
                seq_lens=torch.zeros(b, dtype=torch.int32), scale=0.125)


def test_noalloc_wrapper_refuses_a_splittable_batch_beyond_its_scratch():
    a = _noalloc_batch(max_blocks=9)                # may span two 8-block partitions
    assert 1024 * 32 * 2 * 130 * 4 > pkv.NOALLOC_WORKSPACE_BYTES
    assert pkv.paged_attention_workspace_size(1024, 32, 128, 16, 9) > 0
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_attention_decode_noalloc(**a)
    assert e.value.status == -1 and "scratch" in str(e.value)


def test_noalloc_wrapper_lets_an_unsplittable_batch_through_the_size_check():
    """With at most 8 blocks per sequence the batch is never split and needs no
    scratch: the size check passes and the next check (CPU tensors) refuses."""
    a = _noalloc_batch(max_blocks=8)
    assert pkv.paged_attention_workspace_size(1024, 32, 128, 16, 8) == 0
    with pytest.raises(TypeError, match="CUDA tensor"):
        pkv.paged_attention_decode_noalloc(**a)
