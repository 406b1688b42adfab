"""Oracle: decode-step attention over a paged KV cache, as the plain definition.

TEST INFRASTRUCTURE (see ``oracle/__init__``).

Paging changes where a sequence's keys and values live, not what attention
computes: the glossary "PagedAttention" ("Cách phân trang hoạt động") has the
kernel read the request's keys back through its block table and shows the
gathered keys equal to the originals, so the cache need not be contiguous. The
FlashAttention-style tiling of the related-techniques section only avoids
writing the score matrix to memory; it reaches the same softmax attention up to
rounding order. So, for one decode query per sequence:

    K_b[t] = k_pool[block_tables[b][t // bs], h_kv, t % bs]      t < L_b
    s_t    = scale * k_scale * <q[b, h], K_b[t]>
    p      = exp(s - max s) / sum exp(s - max s)
    out    = v_scale * sum_t p_t V_b[t]

Readings where the pages are silent:

* grouped-query attention (glossary, "Attention truy vấn theo nhóm": K/V heads
  shared between query heads): query head h reads KV head h // G with
  G = num_heads / num_kv_heads, i.e. consecutive query heads share a KV head;
* ``seq_lens`` counts every cached token of the sequence, including the one the
  step has just written;
* a sequence of length 0 yields a zero output;
* ``k_scale``/``v_scale`` are the per-tensor FP8 scales (1 otherwise): the
  stored code times the scale is the value attended over.

Stored values are widened exactly to float64 (bf16/fp32 values exactly, E4M3
codes through the spec decoder) and all arithmetic is float64.
"""
import numpy as np
import torch

from .fp8_e4m3 import e4m3_decode


def widen(rows):
    """Stored values -> exact float64 numpy array (uint8 tensors are E4M3 codes)."""
    if rows.dtype == torch.uint8:
        return e4m3_decode(rows.numpy())
    return rows.to(torch.float64).numpy()


def gather(pool, block_table, seq_len, kv_head, block_size):
    """``[seq_len, head_dim]`` stored rows of one KV head, in token order.

    Token t is read from physical block ``block_table[t // block_size]``, slot
    ``t % block_size``.
    """
    t = np.arange(seq_len)
    blocks = np.asarray(block_table, dtype=np.int64)[t // block_size]
    if seq_len and (blocks.min() < 0 or blocks.max() >= pool.shape[0]):
        raise IndexError("block table entry outside the pool")
    return pool[torch.from_numpy(blocks), kv_head, torch.from_numpy(t % block_size)]


def decode_one(q_vec, K, V, scale, k_scale=1.0, v_scale=1.0):
    """Softmax attention of one query vector over rows K, V (float64 arrays)."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64)
    s = scale * k_scale * (K @ q_vec)
    p = np.exp(s - s.max())
    p = p / p.sum()
    return v_scale * (p @ V)


def paged_decode(q, k_pool, v_pool, block_tables, seq_lens, scale, block_size,
                 k_scale=1.0, v_scale=1.0, units=None, widen_k=widen, widen_v=widen):
    """Decode attention through block tables.

    q: ``[B, Hq, D]`` tensor; pools: ``[NB, Hkv, bs, D]`` tensors (uint8 = E4M3
    codes); block_tables: ``[B, max_blocks]``; seq_lens: ``[B]``.

    With ``units=None`` returns a float64 array ``[B, Hq, D]``; otherwise
    ``units`` is a list of ``(b, h)`` pairs and the result is a dict mapping each
    pair to its float64 output row. ``widen_k``/``widen_v`` turn gathered stored
    rows into float64 values; they default to exact widening of what is stored.
    """
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    if Hq % Hkv:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    G = Hq // Hkv
    bt = np.asarray(block_tables)
    lens = np.asarray(seq_lens)
    todo = units if units is not None else [(b, h) for b in range(B) for h in range(Hq)]
    res = {}
    for b, h in todo:
        L = int(lens[b])
        hk = h // G
        K = widen_k(gather(k_pool, bt[b], L, hk, block_size))
        V = widen_v(gather(v_pool, bt[b], L, hk, block_size))
        qv = q[b, h].to(torch.float64).numpy()
        res[(b, h)] = decode_one(qv, K.reshape(L, D), V.reshape(L, D), scale, k_scale, v_scale)
    if units is not None:
        return res
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for (b, h), o in res.items():
        out[b, h] = o
    return out


def paged_prefill(q, k_pool, v_pool, block_tables, seq_lens, query_start, scale, block_size,
                  k_scale=1.0, v_scale=1.0, units=None):
    """Chunked-prefill attention through block tables: several query tokens per
    sequence, each attending causally over the paged cache.

    The feature list of "vLLM PagedAttention: uma revolução no throughput..."
    names chunked prefill: a long prompt's prefill is split into chunks that run
    as separate steps. The pages' autoregressive model keeps keys and values of
    every token already seen (upskillscore "KV cache paginado...", opening
    paragraph; glossary "Vấn đề bộ nhớ"), so a token attends to itself and to the
    tokens before it. Readings where the pages are silent: sequence ``b`` holds
    ``seq_lens[b]`` cached tokens after the chunk's own K/V were written; its
    chunk is the last ``C_b = query_start[b+1] - query_start[b]`` of them, so
    chunk query ``i`` sits at position ``p = seq_lens[b] - C_b + i`` and attends
    keys ``0..p``. Each query row is therefore exactly a decode over its own causal
    prefix:

        out[query_start[b] + i, h] = decode(q[query_start[b] + i, h], K_b[:p+1], V_b[:p+1])

    q: ``[T, Hq, D]`` (T = query_start[B]); pools ``[NB, Hkv, bs, D]``. With
    ``units=None`` returns float64 ``[T, Hq, D]``; otherwise ``units`` lists
    ``(token, h)`` pairs and a dict of their rows is returned.
    """
    T, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    if Hq % Hkv:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    G = Hq // Hkv
    bt = np.asarray(block_tables)
    lens = np.asarray(seq_lens)
    qs = np.asarray(query_start)
    B = len(lens)
    seq_of = np.zeros(T, dtype=np.int64)
    for b in range(B):
        if qs[b + 1] - qs[b] > lens[b]:
            raise ValueError("a chunk cannot be longer than its sequence")
        seq_of[qs[b]:qs[b + 1]] = b
    todo = units if units is not None else [(t, h) for t in range(T) for h in range(Hq)]
    res = {}
    cache = {}
    for t, h in todo:
        b = int(seq_of[t])
        L = int(lens[b])
        C = int(qs[b + 1] - qs[b])
        p = L - C + (t - int(qs[b]))
        hk = h // G
        if (b, hk) not in cache:
            cache = {(b, hk): (widen(gather(k_pool, bt[b], L, hk, block_size)).reshape(L, D),
                               widen(gather(v_pool, bt[b], L, hk, block_size)).reshape(L, D))}
        K, V = cache[(b, hk)]
        qv = q[t, h].to(torch.float64).numpy()
        res[(t, h)] = decode_one(qv, K[:p + 1], V[:p + 1], scale, k_scale, v_scale)
    if units is not None:
        return res
    out = np.zeros((T, Hq, D), dtype=np.float64)
    for (t, h), o in res.items():
        out[t, h] = o
    return out
