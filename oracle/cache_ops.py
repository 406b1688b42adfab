"""Oracle: the two cache writes of a decode step (slot write, block copy).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

Pool layout (a reading; the glossary's example shows one head as
``key_pool[block, slot, dim]``): ``[num_blocks, num_kv_heads, block_size, head_dim]``.

* ``reshape_and_cache`` follows the worked example of "PagedAttention"
  (glossary, "Cách phân trang hoạt động"): the token at position ``pos`` is
  stored in block ``block_table[pos // block_size]`` at slot ``pos % block_size``.
  Here the caller has already folded block and offset into one slot number
  ``slot = block * block_size + offset``; a negative slot marks a padding token
  and is skipped (a reading). In the FP8 variant the stored byte is
  ``e4m3_quantize(x, scale)`` (see ``fp8_e4m3``).
* ``copy_blocks`` is the copy half of block-level copy-on-write ("KV cache
  paginado...", "Como funciona"; glossary, "Chia sẻ block giữa các chuỗi"):
  for each ``(src, dst)`` the whole block, every head, K and V, becomes a copy of
  ``src``.
* ``swap_blocks`` is the copy of swapping ("KV cache paginado...", "Como
  funciona": preempted requests' blocks go to CPU memory and come back): the
  same whole-block copy, but from one pool into another (device pool to host
  pool on swap-out, host to device on swap-in).

All functions take torch CPU tensors and write in place, copying stored bits
exactly (no arithmetic except the FP8 quantiser).
"""
import torch

from .fp8_e4m3 import e4m3_quantize


def reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, block_size,
                      k_scale=1.0, v_scale=1.0):
    """Write token ``i``'s K/V (``[T, Hkv, D]``) into the pools at ``slot_mapping[i]``.

    If the pools are uint8 they hold E4M3 codes and the values are quantised
    with the per-tensor scales; otherwise the pools must have the dtype of k/v
    and the bits are copied unchanged.
    """
    num_blocks = k_pool.shape[0]
    fp8 = k_pool.dtype == torch.uint8
    if not fp8 and (k.dtype != k_pool.dtype or v.dtype != v_pool.dtype):
        raise TypeError("pool dtype must equal the source dtype unless the pool is FP8")
    for i, s in enumerate(slot_mapping.tolist()):
        if s < 0:
            continue
        block, offset = s // block_size, s % block_size
        if block >= num_blocks:
            raise IndexError(f"slot {s} is outside the pool")
        if fp8:
            k_pool[block, :, offset, :] = torch.from_numpy(
                e4m3_quantize(k[i].float().numpy(), k_scale))
            v_pool[block, :, offset, :] = torch.from_numpy(
                e4m3_quantize(v[i].float().numpy(), v_scale))
        else:
            k_pool[block, :, offset, :] = k[i]
            v_pool[block, :, offset, :] = v[i]


def copy_blocks(k_pool, v_pool, pairs):
    """``pool[dst] = pool[src]`` for every ``(src, dst)`` pair, K and V, all heads."""
    num_blocks = k_pool.shape[0]
    for src, dst in pairs:
        if not (0 <= src < num_blocks and 0 <= dst < num_blocks):
            raise IndexError("block id outside the pool")
        k_pool[dst] = k_pool[src]
        v_pool[dst] = v_pool[src]


def swap_blocks(dst_k_pool, dst_v_pool, src_k_pool, src_v_pool, pairs):
    """``dst_pool[d] = src_pool[s]`` for every ``(s, d)`` pair, K and V, all heads."""
    ns, nd = src_k_pool.shape[0], dst_k_pool.shape[0]
    for src, dst in pairs:
        if not (0 <= src < ns and 0 <= dst < nd):
            raise IndexError("block id outside its pool")
        dst_k_pool[dst] = src_k_pool[src]
        dst_v_pool[dst] = src_v_pool[src]
