"""GB300-native paged KV-cache decode path.

Thin ctypes binding of ``libpagedkv.so`` (C ABI in ``include/pagedkv.h``). The
functions here only marshal arguments: torch tensors give device pointers,
shapes and the current CUDA stream; every step of the path runs in the
library's CUDA kernels. There is no CPU fallback: if the library is missing, or
a tensor is not on a CUDA device, the call raises.

Entry points (same names as the C ABI):

* ``paged_attention_decode`` -- decode attention through block tables.
* ``reshape_and_cache``      -- slot-mapped write of new K/V (optionally E4M3).
* ``copy_blocks``            -- whole-block copies for copy-on-write.
* ``paged_attention_workspace_size``, ``get_device_error``.
* ``BlockManager``           -- the host block manager (free list, tables,
                                reference counts, fork, copy-on-write).
"""
import ctypes
import os

import numpy as np
import torch

__all__ = [
    "PagedKVError", "paged_attention_decode", "paged_attention_workspace_size",
    "paged_attention_decode_noalloc", "NOALLOC_WORKSPACE_BYTES", "paged_attention_decode_grouped",
    "paged_attention_prefill", "swap_blocks",
    "reshape_and_cache", "copy_blocks", "get_device_error", "check_wait_timeout",
    "BoundCall", "bind_paged_attention_decode", "bind_paged_attention_decode_grouped",
    "bind_reshape_and_cache", "bind_copy_blocks", "paged_decode_step", "bind_paged_decode_step", "paged_prefill_step",
    "kernel_launches", "BlockManager",
    "library_path", "load_library", "pool_shapes", "pool_views", "pools_from_views", "PKV_F32",
    "PKV_BF16", "PKV_E4M3", "PKV_ERR_POOL_EXHAUSTED",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpagedkv.so")
_LIB = None

PKV_F32, PKV_BF16, PKV_E4M3 = 0, 1, 2
PKV_ERR_POOL_EXHAUSTED = -5
_STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported configuration",
           -3: "CUDA runtime error", -4: "index out of range", -5: "block pool exhausted",
           -6: "device wait timed out"}


class PagedKVError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {_STATUS.get(status, 'unknown status')} ({status})")


class DecodePipelineStepArgs(ctypes.Structure):
    """``pkv_decode_pipeline_step_args`` (include/pagedkv.h): one buffer set of a
    pipelined decode step, field for field."""
    _vp, _i32p, _i64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
    _fields_ = [
        ("bm", _vp), ("seq_ids", _i64p), ("num_seqs", ctypes.c_int), ("max_blocks", ctypes.c_int),
        ("max_members", ctypes.c_int),
        ("h_slots", _i64p), ("h_pairs", _i64p), ("h_tables", _i32p), ("h_lens", _i32p),
        ("h_group_members", _i32p), ("h_group_prefix", _i32p), ("h_seq_group", _i32p),
        ("h_ungrouped", _i32p), ("group_blocks", _i32p),
        ("host_slab", _vp), ("dev_slab", _vp), ("slab_bytes", ctypes.c_size_t),
        ("q", _vp), ("k_new", _vp), ("v_new", _vp), ("slots", _vp), ("pairs", _vp),
        ("tables", _vp), ("lens", _vp), ("seq_group", _vp), ("group_members", _vp),
        ("group_prefix", _vp), ("ungrouped", _vp),
        ("out", _vp), ("k_pool", _vp), ("v_pool", _vp),
        ("num_blocks", ctypes.c_int), ("num_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int), ("scale", ctypes.c_float),
        ("q_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int), ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("out_bytes", ctypes.c_size_t),
        ("up_stream", _vp), ("compute_stream", _vp), ("down_stream", _vp),
        ("uploaded_event", _vp), ("computed_event", _vp), ("downloaded_event", _vp),
    ]


def library_path():
    return _LIB_PATH


def load_library():
    """Load libpagedkv.so (built by ``paged_kv_cache_259_gb300.build``); raise if absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is not built; run "
                           "`python -m paged_kv_cache_259_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(_LIB_PATH)
    c_int, c_float, c_size, vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    ip = ctypes.POINTER(ctypes.c_int)
    sig = {
        "pkv_status_string": (ctypes.c_char_p, [c_int]),
        "pkv_last_error_string": (ctypes.c_char_p, []),
        "pkv_kernel_launches": (ctypes.c_ulonglong, []),
        "paged_attention_decode": (c_int, [vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int,
                                           c_int, c_int, c_int, c_float, c_int, c_int, c_float,
                                           c_float, vp, c_size, vp]),
        "paged_attention_workspace_size": (c_size, [c_int, c_int, c_int, c_int, c_int]),
        "paged_attention_decode_grouped": (c_int, [vp, vp, vp, vp, vp, vp, c_int, c_int, c_int,
                                                   c_int, c_int, c_int, c_int, c_float, c_int,
                                                   c_int, c_float, c_float, vp, vp, vp, c_int,
                                                   c_int, c_int, vp, c_int, vp, c_size, vp]),
        "paged_decode_step": (c_int, [vp, c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int,
                                      c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                      c_float, c_float, vp, vp, vp, c_int, c_int, c_int, vp,
                                      c_int, vp, c_size, vp]),
        "bm_prefix_groups": (c_int, [vp, i64p, c_int, c_int, i32p, i32p, i32p, i32p, ip]),
        "bm_plan_decode": (c_int, [vp, i64p, c_int, c_int, i64p, i64p, ip, i32p, i32p, c_int, i32p,
                                   i32p, i32p, i32p, i32p, ip, ip, ip]),
        "paged_attention_decode_noalloc": (c_int, [vp, vp, vp, vp, vp, vp, c_int, c_int, c_int,
                                                   c_int, c_int, c_int, c_int, c_float, c_int,
                                                   c_int, c_float, c_float, vp]),
        "paged_attention_prefill": (c_int, [vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int,
                                            c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                                            c_int, vp]),
        "paged_prefill_step": (c_int, [vp, c_int, vp, vp, vp, c_int, vp, vp, vp, vp, vp, vp, vp,
                                       c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                       c_float, c_int, c_int, vp]),
        "reshape_and_cache": (c_int, [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                      c_int, c_int, c_float, c_float, vp]),
        "copy_blocks": (c_int, [vp, vp, vp, c_int, c_int, c_size, vp]),
        "pkv_get_device_error": (c_int, [ip, vp]),
        "pkv_check_wait_timeout": (c_int, [vp]),
        "pkv_stage_upload": (c_int, [vp, vp, c_size, vp, vp, vp, vp, vp]),
        "pkv_stage_download": (c_int, [vp, vp, c_size, vp, vp, vp, vp]),
        "bm_create": (vp, [c_int, c_int, i32p, c_int]),
        "bm_destroy": (None, [vp]),
        "bm_add_seq": (c_int, [vp, ctypes.c_int64]),
        "bm_append_slot": (c_int, [vp, ctypes.c_int64, i64p, i32p, i32p]),
        "bm_append_n": (c_int, [vp, ctypes.c_int64, c_int, i64p, c_int, ip]),
        "bm_append_slots": (c_int, [vp, i64p, c_int, i64p, i64p, ip]),
        "bm_fork": (c_int, [vp, ctypes.c_int64, ctypes.c_int64]),
        "bm_free_seq": (c_int, [vp, ctypes.c_int64]),
        "bm_beam_step": (c_int, [vp, i64p, c_int, i32p, i64p, c_int]),
        "bm_block_table": (c_int, [vp, ctypes.c_int64, i32p, c_int, ip]),
        "bm_build_tables": (c_int, [vp, i64p, c_int, c_int, i32p, i32p]),
        "bm_seq_len": (c_int, [vp, ctypes.c_int64, ip]),
        "bm_refcount": (c_int, [vp, c_int, ip]),
        "bm_num_free": (c_int, [vp]),
        "bm_free_list": (c_int, [vp, i32p, c_int]),
        "bm_enable_prefix_caching": (c_int, [vp]),
        "bm_set_host_blocks": (c_int, [vp, c_int]),
        "bm_swap_out": (c_int, [vp, ctypes.c_int64, i64p, c_int, ip]),
        "bm_swap_in": (c_int, [vp, ctypes.c_int64, i64p, c_int, ip]),
        "bm_is_swapped": (c_int, [vp, ctypes.c_int64, ip]),
        "bm_host_free_list": (c_int, [vp, i32p, c_int]),
        "swap_blocks": (c_int, [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_size, vp]),
        "bm_add_seq_prompt": (c_int, [vp, ctypes.c_int64, i32p, c_int, ip]),
        "bm_append_tokens": (c_int, [vp, ctypes.c_int64, i32p, c_int, i64p, i64p, c_int, ip]),
        "bm_cache_stats": (c_int, [vp, i64p, i64p, ip, ip]),
        "bm_evictable_list": (c_int, [vp, i32p, c_int]),
        "pkv_decode_pipeline_step": (c_int, [ctypes.POINTER(DecodePipelineStepArgs), c_int, vp, ip,
                                             ctypes.POINTER(ctypes.c_double)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(status, what):
    if status != 0:
        if status == -3 and _LIB is not None:
            what = f"{what} [{_LIB.pkv_last_error_string().decode(errors='replace')}]"
        raise PagedKVError(status, what)


_DTYPES = {torch.float32: PKV_F32, torch.bfloat16: PKV_BF16, torch.uint8: PKV_E4M3}
if hasattr(torch, "float8_e4m3fn"):
    _DTYPES[torch.float8_e4m3fn] = PKV_E4M3


def _dt(t, what):
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"{what}: unsupported dtype {t.dtype}") from None


def _cuda(t, what, contiguous=True):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t


def _on_gpu(named):
    """Every (tensor, name) a contiguous CUDA tensor, all on one device; returns
    that device. Called after the shape checks, so those run without a GPU."""
    dev = None
    for t, n in named:
        _cuda(t, n)
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{n} is on {t.device}, the other tensors on {dev}")
    return dev


def _tensors(named):
    for t, n in named:
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{n} must be a tensor")


def _decode_shapes(out, q, k_pool, v_pool, block_tables, seq_lens):
    """(B, Hq, D, NB, Hkv, bs) of a decode call; raise on a mismatch."""
    _tensors(((out, "out"), (q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"),
              (block_tables, "block_tables"), (seq_lens, "seq_lens")))
    if q.dim() != 3 or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q and out must be [B, Hq, D] of the same dtype")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = _pool_dims(k_pool, v_pool)
    if D2 != D or block_tables.dim() != 2 or block_tables.shape[0] != B or \
            tuple(seq_lens.shape) != (B,):
        raise ValueError("inconsistent shapes: block_tables must be [B, max_blocks], "
                         "seq_lens [B], pools of q's head_dim")
    return B, Hq, D, NB, Hkv, bs


def _workspace(workspace, device):
    if workspace is None:
        return None, 0
    _on_gpu(((workspace, "workspace"),))
    if workspace.device != device:
        raise ValueError(f"workspace is on {workspace.device}, the other tensors on {device}")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def _stream_ptr(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


class _on_device:
    """Make ``device`` current for the call (the library works on the current device)."""

    def __init__(self, device):
        self.idx = device.index if device.index is not None else torch.cuda.current_device()
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.idx:
            self.prev = cur
            torch.cuda.set_device(self.idx)

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)


def pool_shapes(num_blocks, num_kv_heads, block_size, head_dim, dtype):
    """Tensor shapes of the K and V pools in the library's layout.

    Each (block, head) tile is contiguous and made of 128-byte core matrices
    (8 rows of 16 bytes; X = 16 bytes of elements): K ``[NB, Hkv, bs/8, D/X, 8,
    X]`` (8 tokens x X dims per core matrix), V ``[NB, Hkv, bs/X, D/8, 8, X]``
    (8 dims x X tokens per core matrix). See ``include/pagedkv.h``.
    """
    esize = torch.empty((), dtype=dtype).element_size()
    x = 16 // esize
    if head_dim % x or head_dim % 8 or block_size % 8 or block_size % x:
        raise ValueError(f"head_dim and block_size must be multiples of {max(x, 8)} for {dtype}")
    return ((num_blocks, num_kv_heads, block_size // 8, head_dim // x, 8, x),
            (num_blocks, num_kv_heads, block_size // x, head_dim // 8, 8, x))


def pool_views(k_pool, v_pool):
    """The pools as plain ``[NB, Hkv, bs, D]`` (block, head, slot, dim) copies."""
    NB, Hkv, bs, D = _pool_dims(k_pool, v_pool)
    k = k_pool.permute(0, 1, 2, 4, 3, 5).reshape(NB, Hkv, bs, D)
    v = v_pool.permute(0, 1, 2, 5, 3, 4).reshape(NB, Hkv, bs, D)
    return k, v


def pools_from_views(k, v):
    """Plain ``[NB, Hkv, bs, D]`` K/V -> pools in the library layout (copies)."""
    NB, Hkv, bs, D = k.shape
    x = 16 // k.element_size()
    kp = k.reshape(NB, Hkv, bs // 8, 8, D // x, x).permute(0, 1, 2, 4, 3, 5).contiguous()
    vp = v.reshape(NB, Hkv, bs // x, x, D // 8, 8).permute(0, 1, 2, 4, 5, 3).contiguous()
    return kp, vp


def _pool_dims(k_pool, v_pool):
    """(NB, Hkv, bs, D) of pools in the library layout; raise on a mismatch."""
    if k_pool.dim() != 6 or v_pool.dim() != 6 or k_pool.dtype != v_pool.dtype:
        raise ValueError("pools must be K [NB, Hkv, bs/8, D/X, 8, X] and V [NB, Hkv, bs/X, D/8, "
                         "8, X] of one dtype (see pool_shapes)")
    NB, Hkv, G8, P, r8, X = k_pool.shape
    bs, D = G8 * 8, P * X
    if X * k_pool.element_size() != 16 or r8 != 8 or bs % X or \
            tuple(v_pool.shape) != (NB, Hkv, bs // X, D // 8, 8, X):
        raise ValueError("pool shapes do not match the library layout (see pool_shapes)")
    return NB, Hkv, bs, D


def paged_attention_workspace_size(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq):
    """Bytes of split-KV workspace for the finest split of these sizes."""
    return int(load_library().paged_attention_workspace_size(
        num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq))


def paged_attention_decode(out, q, k_pool, v_pool, block_tables, seq_lens, scale,
                           k_scale=1.0, v_scale=1.0, workspace=None, stream=None):
    """out[b, h] = softmax attention of q[b, h] over sequence b's cached tokens.

    q, out: ``[B, Hq, D]`` (float32 or bfloat16, same dtype); pools in the
    library layout (``pool_shapes``; float32/bfloat16 like q, or uint8/
    float8_e4m3fn for the E4M3 cache with per-tensor ``k_scale``/``v_scale``); block_tables int32
    ``[B, max_blocks]``; seq_lens int32 ``[B]``; workspace: any CUDA tensor used
    as split-KV scratch (see ``paged_attention_workspace_size``) or None.
    """
    bind_paged_attention_decode(out, q, k_pool, v_pool, block_tables, seq_lens, scale, k_scale,
                                v_scale, workspace)(stream)
    return out


def bind_paged_attention_decode(out, q, k_pool, v_pool, block_tables, seq_lens, scale,
                                k_scale=1.0, v_scale=1.0, workspace=None):
    """``paged_attention_decode`` checked once and bound to these tensors
    (``BoundCall``): calling the result launches it on a stream."""
    lib = load_library()
    B, Hq, D, NB, Hkv, bs = _decode_shapes(out, q, k_pool, v_pool, block_tables, seq_lens)
    dev = _on_gpu(((out, "out"), (q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"),
                   (block_tables, "block_tables"), (seq_lens, "seq_lens")))
    ws_ptr, ws_bytes = _workspace(workspace, dev)
    args = [_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens)]
    args += _c_args([B, block_tables.shape[1], NB, Hq, Hkv, D, bs, float(scale), _dt(q, "q"),
                     _dt(k_pool, "k_pool"), float(k_scale), float(v_scale)])
    args += [ctypes.c_void_p(ws_ptr), ctypes.c_size_t(ws_bytes)]
    return BoundCall(lib.paged_attention_decode, args, "paged_attention_decode", dev)


def paged_attention_decode_grouped(out, q, k_pool, v_pool, block_tables, seq_lens, scale,
                                   seq_group, group_members, group_prefix_blocks,
                                   k_scale=1.0, v_scale=1.0, workspace=None, stream=None,
                                   ungrouped=None, max_group_blocks=0):
    """``paged_attention_decode`` reading each shared prefix once per group.

    seq_group int32 ``[B]`` (group or -1); group_members int32 ``[num_groups,
    max_members]`` (batch indices, -1 padded); group_prefix_blocks int32
    ``[num_groups]`` -- as ``BlockManager.prefix_groups`` returns them; ungrouped:
    int32 ``[n]`` batch indices in no group (None: every sequence is launched);
    max_group_blocks: the largest of ``prefix_groups``' list blocks (0: unknown).
    """
    bind_paged_attention_decode_grouped(
        out, q, k_pool, v_pool, block_tables, seq_lens, scale, seq_group, group_members,
        group_prefix_blocks, k_scale, v_scale, workspace, ungrouped, max_group_blocks)(stream)
    return out


def bind_paged_attention_decode_grouped(out, q, k_pool, v_pool, block_tables, seq_lens, scale,
                                        seq_group, group_members, group_prefix_blocks,
                                        k_scale=1.0, v_scale=1.0, workspace=None,
                                        ungrouped=None, max_group_blocks=0):
    """``paged_attention_decode_grouped`` checked once and bound to these
    tensors (``BoundCall``). ``group_members``, ``group_prefix_blocks`` and
    ``ungrouped`` may be sized for the most groups and ungrouped sequences a
    step can have: each call may then pass ``num_groups``, ``num_ungrouped`` and
    ``max_group_blocks`` for the rows actually filled."""
    lib = load_library()
    B, Hq, D, NB, Hkv, bs = _decode_shapes(out, q, k_pool, v_pool, block_tables, seq_lens)
    groups = [(seq_group, "seq_group"), (group_members, "group_members"),
              (group_prefix_blocks, "group_prefix_blocks")]
    if ungrouped is not None:
        groups.append((ungrouped, "ungrouped"))
    _tensors(groups)
    for t, n in groups:
        if t.dtype != torch.int32:
            raise TypeError(f"{n} must be int32")
    if tuple(seq_group.shape) != (B,) or group_members.dim() != 2 or \
            tuple(group_prefix_blocks.shape) != (group_members.shape[0],) or \
            (ungrouped is not None and ungrouped.dim() != 1):
        raise ValueError("inconsistent shapes: seq_group [B], group_members [G, max_members], "
                         "group_prefix_blocks [G], ungrouped [n]")
    dev = _on_gpu([(out, "out"), (q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"),
                   (block_tables, "block_tables"), (seq_lens, "seq_lens")] + groups)
    ws_ptr, ws_bytes = _workspace(workspace, dev)
    G, n_un = group_members.shape[0], -1 if ungrouped is None else ungrouped.numel()
    args = [_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens)]
    args += _c_args([B, block_tables.shape[1], NB, Hq, Hkv, D, bs, float(scale), _dt(q, "q"),
                     _dt(k_pool, "k_pool"), float(k_scale), float(v_scale)])
    args += [_ptr(seq_group), _ptr(group_members), _ptr(group_prefix_blocks)]
    args += _c_args([G, group_members.shape[1], int(max_group_blocks)])
    args += [_ptr(ungrouped), ctypes.c_int(n_un), ctypes.c_void_p(ws_ptr), ctypes.c_size_t(ws_bytes)]
    counts = {"num_groups": (21, G), "max_group_blocks": (23, 2 ** 31 - 1)}
    if ungrouped is not None:
        counts["num_ungrouped"] = (25, n_un)
    return BoundCall(lib.paged_attention_decode_grouped, args, "paged_attention_decode_grouped",
                     dev, counts)


def paged_decode_step(out, q, k_new, v_new, k_pool, v_pool, block_tables, seq_lens,
                      slot_mapping, src_dst_pairs, scale, k_scale=1.0, v_scale=1.0,
                      workspace=None, stream=None, seq_group=None, group_members=None,
                      group_prefix_blocks=None, ungrouped=None, max_group_blocks=0):
    """One decode step in one call: the copy-on-write pairs, the slot write of
    every sequence's new token (k_new / v_new ``[B, Hkv, D]`` like q, slot_mapping
    int64 ``[B]``: sequence b's newest position) and the attention, grouped when
    the group tensors are given (as ``paged_attention_decode_grouped`` takes
    them). The decode reads every block but the sequences' last ones while the
    copies and slot writes finish."""
    bind_paged_decode_step(out, q, k_new, v_new, k_pool, v_pool, block_tables, seq_lens,
                           slot_mapping, src_dst_pairs, scale, k_scale, v_scale, workspace,
                           seq_group, group_members, group_prefix_blocks, ungrouped,
                           max_group_blocks)(stream)
    return out


def bind_paged_decode_step(out, q, k_new, v_new, k_pool, v_pool, block_tables, seq_lens,
                           slot_mapping, src_dst_pairs, scale, k_scale=1.0, v_scale=1.0,
                           workspace=None, seq_group=None, group_members=None,
                           group_prefix_blocks=None, ungrouped=None, max_group_blocks=0):
    """``paged_decode_step`` checked once and bound to these tensors
    (``BoundCall``). ``src_dst_pairs`` and the group tensors may be sized for the
    most a step can raise: each call may then pass ``num_pairs``, ``num_groups``,
    ``max_group_blocks`` and ``num_ungrouped`` for the rows actually filled
    (``num_groups=0``: the plain decode)."""
    lib = load_library()
    B, Hq, D, NB, Hkv, bs = _decode_shapes(out, q, k_pool, v_pool, block_tables, seq_lens)
    named = [(k_new, "k_new"), (v_new, "v_new"), (slot_mapping, "slot_mapping"),
             (src_dst_pairs, "src_dst_pairs")]
    grouped = group_members is not None
    if grouped:
        named += [(seq_group, "seq_group"), (group_members, "group_members"),
                  (group_prefix_blocks, "group_prefix_blocks")]
        if ungrouped is not None:
            named.append((ungrouped, "ungrouped"))
    _tensors(named)
    if tuple(k_new.shape) != (B, Hkv, D) or v_new.shape != k_new.shape or \
            k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise ValueError("k_new and v_new must be [B, Hkv, D] in the dtype of q")
    if slot_mapping.dtype != torch.int64 or tuple(slot_mapping.shape) != (B,):
        raise ValueError("slot_mapping must be int64 [B]")
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or \
            src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be int64 [P, 2]")
    if grouped:
        for t, n in named[4:]:
            if t.dtype != torch.int32:
                raise TypeError(f"{n} must be int32")
        if tuple(seq_group.shape) != (B,) or group_members.dim() != 2 or \
                tuple(group_prefix_blocks.shape) != (group_members.shape[0],) or \
                (ungrouped is not None and ungrouped.dim() != 1):
            raise ValueError("inconsistent shapes: seq_group [B], group_members [G, max_members], "
                             "group_prefix_blocks [G], ungrouped [n]")
    dev = _on_gpu([(out, "out"), (q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"),
                   (block_tables, "block_tables"), (seq_lens, "seq_lens")] + named)
    ws_ptr, ws_bytes = _workspace(workspace, dev)
    P = src_dst_pairs.shape[0]
    G = group_members.shape[0] if grouped else 0
    M = group_members.shape[1] if grouped else 0
    n_un = -1 if ungrouped is None else ungrouped.numel()
    args = [_ptr(src_dst_pairs), ctypes.c_int(P), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
            _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens)]
    args += _c_args([B, block_tables.shape[1], NB, Hq, Hkv, D, bs, float(scale), _dt(q, "q"),
                     _dt(k_pool, "k_pool"), float(k_scale), float(v_scale)])
    args += [_ptr(seq_group if grouped else None), _ptr(group_members if grouped else None),
             _ptr(group_prefix_blocks if grouped else None)]
    args += _c_args([G, M, int(max_group_blocks)])
    args += [_ptr(ungrouped), ctypes.c_int(n_un), ctypes.c_void_p(ws_ptr), ctypes.c_size_t(ws_bytes)]
    counts = {"num_pairs": (1, P), "num_groups": (26, G), "max_group_blocks": (28, 2 ** 31 - 1)}
    if ungrouped is not None:
        counts["num_ungrouped"] = (30, n_un)
    return BoundCall(lib.paged_decode_step, args, "paged_decode_step", dev, counts)


# scratch bytes of paged_attention_decode_noalloc (PKV_NOALLOC_WORKSPACE_BYTES)
NOALLOC_WORKSPACE_BYTES = 32 * 1024 * 1024


def paged_attention_decode_noalloc(out, q, k_pool, v_pool, block_tables, seq_lens, scale,
                                   k_scale=1.0, v_scale=1.0, stream=None):
    """``paged_attention_decode`` for callers that cannot allocate device memory
    where they decode (a plug-in inside a runtime that owns all device memory, a
    serving loop whose memory plan is fixed at start-up): the split-KV scratch is
    a fixed 32 MiB array inside the library (per GPU), so no workspace is passed
    and nothing is allocated. Calls on one device share that array and must not
    overlap on the GPU; the first call on a device should come before any stream
    capture. A batch that can be split (``paged_attention_workspace_size`` > 0)
    is refused when ``B * Hq * 2 * (D + 2) * 4 > NOALLOC_WORKSPACE_BYTES``.
    """
    lib = load_library()
    B, Hq, D, NB, Hkv, bs = _decode_shapes(out, q, k_pool, v_pool, block_tables, seq_lens)
    need = B * Hq * 2 * (D + 2) * 4
    splittable = lib.paged_attention_workspace_size(B, Hq, D, bs, block_tables.shape[1]) > 0
    if splittable and need > NOALLOC_WORKSPACE_BYTES:
        raise PagedKVError(-1, f"paged_attention_decode_noalloc: batch needs {need} bytes of "
                               f"scratch, the fixed array holds {NOALLOC_WORKSPACE_BYTES}")
    dev = _on_gpu(((out, "out"), (q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"),
                   (block_tables, "block_tables"), (seq_lens, "seq_lens")))
    with _on_device(dev):
        st = lib.paged_attention_decode_noalloc(
            out.data_ptr(), q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
            block_tables.data_ptr(), seq_lens.data_ptr(), B, block_tables.shape[1], NB,
            Hq, Hkv, D, bs, float(scale), _dt(q, "q"), _dt(k_pool, "k_pool"),
            float(k_scale), float(v_scale), _stream_ptr(stream, dev))
    _check(st, "paged_attention_decode_noalloc")
    return out


def paged_attention_prefill(out, q, k_pool, v_pool, block_tables, seq_lens, query_start,
                            scale, max_query_len, stream=None):
    """Chunked prefill: for sequence b, the last ``C_b = query_start[b+1] -
    query_start[b]`` of its ``seq_lens[b]`` cached tokens are the chunk; chunk
    query i attends causally to keys ``0 .. seq_lens[b] - C_b + i``.

    q, out: bfloat16 ``[T, Hq, D]`` (T = query_start[-1]); pools bfloat16 in the
    library layout; block_tables int32 ``[B, max_blocks]``; seq_lens int32
    ``[B]``; query_start int32 ``[B + 1]``; ``max_query_len`` >= every C_b.
    """
    lib = load_library()
    named = ((out, "out"), (q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"),
             (block_tables, "block_tables"), (seq_lens, "seq_lens"), (query_start, "query_start"))
    _tensors(named)
    for t in (block_tables, seq_lens, query_start):
        if t.dtype != torch.int32:
            raise TypeError("block_tables, seq_lens and query_start must be int32")
    if q.dim() != 3 or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q and out must be [T, Hq, D] of the same dtype")
    if seq_lens.dim() != 1:
        raise ValueError("seq_lens must be [B]")
    B = seq_lens.shape[0]
    T, Hq, D = q.shape
    NB, Hkv, bs, D2 = _pool_dims(k_pool, v_pool)
    if D2 != D or block_tables.dim() != 2 or block_tables.shape[0] != B or \
            tuple(query_start.shape) != (B + 1,):
        raise ValueError("inconsistent shapes: block_tables [B, max_blocks], query_start "
                         "[B + 1], pools of q's head_dim")
    dev = _on_gpu(named)
    with _on_device(dev):
        st = lib.paged_attention_prefill(
            out.data_ptr(), q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
            block_tables.data_ptr(), seq_lens.data_ptr(), query_start.data_ptr(), B,
            int(max_query_len), block_tables.shape[1], NB, Hq, Hkv, D, bs, float(scale),
            _dt(q, "q"), _dt(k_pool, "k_pool"), _stream_ptr(stream, dev))
    _check(st, "paged_attention_prefill")
    return out


def paged_prefill_step(out, q, k_new, v_new, k_pool, v_pool, block_tables, seq_lens,
                       query_start, slot_mapping, src_dst_pairs, scale, max_query_len,
                       stream=None):
    """One chunked-prefill step in one call: the copy-on-write pairs (int64
    ``[P, 2]``), the chunk tokens' K/V (bfloat16 ``[T, Hkv, D]``) into their slots
    (int64 ``[T]``: the chunk positions of their sequences) and the attention of
    ``paged_attention_prefill``; the attention reads the key tiles before each
    chunk while the writes finish."""
    lib = load_library()
    named = ((out, "out"), (q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_pool, "k_pool"),
             (v_pool, "v_pool"), (block_tables, "block_tables"), (seq_lens, "seq_lens"),
             (query_start, "query_start"), (slot_mapping, "slot_mapping"),
             (src_dst_pairs, "src_dst_pairs"))
    _tensors(named)
    for t in (block_tables, seq_lens, query_start):
        if t.dtype != torch.int32:
            raise TypeError("block_tables, seq_lens and query_start must be int32")
    if q.dim() != 3 or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q and out must be [T, Hq, D] of the same dtype")
    if seq_lens.dim() != 1:
        raise ValueError("seq_lens must be [B]")
    B = seq_lens.shape[0]
    T, Hq, D = q.shape
    NB, Hkv, bs, D2 = _pool_dims(k_pool, v_pool)
    if D2 != D or block_tables.dim() != 2 or block_tables.shape[0] != B or \
            tuple(query_start.shape) != (B + 1,):
        raise ValueError("inconsistent shapes: block_tables [B, max_blocks], query_start "
                         "[B + 1], pools of q's head_dim")
    if k_new.dim() != 3 or k_new.shape[1:] != (Hkv, D) or v_new.shape != k_new.shape or \
            k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise ValueError("k_new and v_new must be [T, Hkv, D] in the dtype of q")
    if slot_mapping.dtype != torch.int64 or tuple(slot_mapping.shape) != (k_new.shape[0],):
        raise ValueError("slot_mapping must be int64 [T]")
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or \
            src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be int64 [P, 2]")
    dev = _on_gpu(named)
    with _on_device(dev):
        st = lib.paged_prefill_step(
            src_dst_pairs.data_ptr(), src_dst_pairs.shape[0], k_new.data_ptr(), v_new.data_ptr(),
            slot_mapping.data_ptr(), k_new.shape[0], out.data_ptr(), q.data_ptr(),
            k_pool.data_ptr(), v_pool.data_ptr(), block_tables.data_ptr(), seq_lens.data_ptr(),
            query_start.data_ptr(), B, int(max_query_len), block_tables.shape[1], NB, Hq, Hkv, D,
            bs, float(scale), _dt(q, "q"), _dt(k_pool, "k_pool"), _stream_ptr(stream, dev))
    _check(st, "paged_prefill_step")
    return out


def reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, k_scale=1.0, v_scale=1.0, stream=None):
    """Write k/v ``[T, Hkv, D]`` into the pools (library layout) at ``slot_mapping``
    (int64 ``[T]``)."""
    bind_reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, k_scale, v_scale)(stream)


def bind_reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, k_scale=1.0, v_scale=1.0):
    """``reshape_and_cache`` checked once and bound to these tensors (``BoundCall``)."""
    lib = load_library()
    named = ((k, "k"), (v, "v"), (k_pool, "k_pool"), (v_pool, "v_pool"),
             (slot_mapping, "slot_mapping"))
    _tensors(named)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if k.dim() != 3:
        raise ValueError("k and v must be [T, Hkv, D]")
    T, Hkv, D = k.shape
    NB, Hkv2, bs, D2 = _pool_dims(k_pool, v_pool)
    if v.shape != k.shape or v.dtype != k.dtype or (Hkv2, D2) != (Hkv, D) or \
            tuple(slot_mapping.shape) != (T,):
        raise ValueError("inconsistent shapes: k and v [T, Hkv, D] like the pools, "
                         "slot_mapping [T]")
    dev = _on_gpu(named)
    args = [_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool), _ptr(slot_mapping)]
    args += _c_args([T, Hkv, D, bs, NB, _dt(k, "k"), _dt(k_pool, "k_pool"), float(k_scale),
                     float(v_scale)])
    return BoundCall(lib.reshape_and_cache, args, "reshape_and_cache", dev)


class BoundCall:
    """One library call whose tensors, shapes and sizes were checked once, as the
    plain call checks them, with its arguments kept as C values: calling it
    launches on the given stream (default: the current stream of its device).
    Count arguments named at binding time (``counts``: name -> (argument index,
    largest allowed value)) may be given anew per call, e.g. the number of
    copy-on-write pairs held in a buffer sized for the most a step can raise.
    The tensors must stay alive and in place while the bound call is used."""

    __slots__ = ("_fn", "_args", "_what", "_idx", "_stream", "_sptr", "_counts")

    def __init__(self, fn, args, what, device, counts=None):
        self._fn = fn
        self._args = list(args)
        self._what = what
        self._idx = device.index if device.index is not None else torch.cuda.current_device()
        self._stream = None
        self._sptr = None
        self._counts = counts or {}

    def __call__(self, stream=None, **counts):
        if stream is None:
            stream = torch.cuda.current_stream(self._idx)
        if stream is not self._stream:
            self._stream, self._sptr = stream, ctypes.c_void_p(stream.cuda_stream)
        args = self._args
        if counts:
            args = list(args)
            for name, v in counts.items():
                i, top = self._counts[name]
                if not 0 <= int(v) <= top:
                    raise ValueError(f"{self._what}: {name}={v} outside [0, {top}]")
                args[i] = type(args[i])(int(v))
        if torch.cuda.current_device() != self._idx:
            with _on_device(torch.device("cuda", self._idx)):
                st = self._fn(*args, self._sptr)
        else:
            st = self._fn(*args, self._sptr)
        _check(st, self._what)


def _c_args(values):
    """C values of a call's arguments: pointers (ints from data_ptr or None)
    as void*, ints as int, floats as float; ``size_t`` values wrapped by the
    caller."""
    out = []
    for v in values:
        if isinstance(v, (ctypes.c_size_t, ctypes.c_void_p)):
            out.append(v)
        elif isinstance(v, bool):
            out.append(ctypes.c_int(int(v)))
        elif isinstance(v, int):
            out.append(ctypes.c_int(v))
        elif isinstance(v, float):
            out.append(ctypes.c_float(v))
        else:
            raise TypeError(f"unexpected argument {v!r}")
    return out


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(None)


def copy_blocks(k_pool, v_pool, src_dst_pairs, stream=None):
    """``pool[dst] = pool[src]`` for each row of int64 ``src_dst_pairs [P, 2]``.

    Destinations must be distinct and none may also be a source; a launch of at
    most 4096 pairs checks this on the device and reports a violation as
    ``PKV_ERR_INVALID_ARG`` through ``get_device_error``."""
    bind_copy_blocks(k_pool, v_pool, src_dst_pairs)(stream)


def bind_copy_blocks(k_pool, v_pool, src_dst_pairs):
    """``copy_blocks`` checked once and bound to these tensors (``BoundCall``);
    ``src_dst_pairs`` may be sized for the most pairs a step can raise, each call
    passing ``num_pairs`` for the rows filled."""
    lib = load_library()
    named = ((k_pool, "k_pool"), (v_pool, "v_pool"), (src_dst_pairs, "src_dst_pairs"))
    _tensors(named)
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or \
            src_dst_pairs.shape[1] != 2 or k_pool.dim() < 1 or v_pool.dim() < 1 or \
            k_pool.shape[0] != v_pool.shape[0] or k_pool.numel() != v_pool.numel() or \
            k_pool.dtype != v_pool.dtype:
        raise ValueError("src_dst_pairs must be int64 [P, 2]; pools of one shape and dtype")
    dev = _on_gpu(named)
    block_bytes = k_pool[0].numel() * k_pool.element_size()
    P = src_dst_pairs.shape[0]
    args = [_ptr(k_pool), _ptr(v_pool), _ptr(src_dst_pairs), ctypes.c_int(P),
            ctypes.c_int(k_pool.shape[0]), ctypes.c_size_t(block_bytes)]
    return BoundCall(lib.copy_blocks, args, "copy_blocks", dev, {"num_pairs": (3, P)})


def swap_blocks(dst_k_pool, dst_v_pool, src_k_pool, src_v_pool, src_dst_pairs, stream=None):
    """``dst_pool[d] = src_pool[s]`` for every (s, d) pair, K and V; each pool is a
    CUDA tensor or a pinned CPU tensor (``pin_memory()``) in the library layout."""
    lib = load_library()
    for t, n in ((dst_k_pool, "dst_k_pool"), (dst_v_pool, "dst_v_pool"),
                 (src_k_pool, "src_k_pool"), (src_v_pool, "src_v_pool")):
        if not t.is_contiguous() or (not t.is_cuda and not t.is_pinned()):
            raise ValueError(f"{n} must be a contiguous CUDA or pinned CPU tensor")
    if src_dst_pairs.dtype != torch.int64 or not src_dst_pairs.is_contiguous() or \
            (not src_dst_pairs.is_cuda and not src_dst_pairs.is_pinned()):
        raise TypeError("src_dst_pairs must be contiguous int64, on the GPU or pinned")
    NBd, Hkv, bs, D = _pool_dims(dst_k_pool, dst_v_pool)
    NBs, Hkv2, bs2, D2 = _pool_dims(src_k_pool, src_v_pool)
    if (Hkv, bs, D) != (Hkv2, bs2, D2) or dst_k_pool.dtype != src_k_pool.dtype:
        raise ValueError("pools of different layouts")
    block_bytes = Hkv * bs * D * dst_k_pool.element_size()
    dev = dst_k_pool.device if dst_k_pool.is_cuda else src_k_pool.device
    with _on_device(dev):
        st = lib.swap_blocks(dst_k_pool.data_ptr(), dst_v_pool.data_ptr(), src_k_pool.data_ptr(),
                             src_v_pool.data_ptr(), src_dst_pairs.data_ptr(),
                             src_dst_pairs.shape[0], NBs, NBd, block_bytes,
                             _stream_ptr(stream, dev))
    _check(st, "swap_blocks")


def kernel_launches():
    """Kernels this library has launched in this process so far."""
    return int(load_library().pkv_kernel_launches())


def get_device_error(device=None, stream=None):
    """Synchronise and return-and-clear the device error word (0 = no error)."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    code = ctypes.c_int(0)
    with _on_device(dev):
        _check(lib.pkv_get_device_error(ctypes.byref(code), _stream_ptr(stream, dev)),
               "pkv_get_device_error")
    return code.value


def check_wait_timeout(device=None, stream=None):
    """Launch the library's timeout check: a bounded wait that nothing completes
    gives up after about a second, so the next ``get_device_error`` returns
    ``PKV_ERR_TIMEOUT`` (-6). Run it with no other work of the library in flight
    on the device."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    with _on_device(dev):
        _check(lib.pkv_check_wait_timeout(_stream_ptr(stream, dev)), "pkv_check_wait_timeout")


def _i32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _i64p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


class BlockManager:
    """Host block manager of the C library (free list front-first, refcounts, CoW)."""

    def __init__(self, num_blocks, block_size, free_order, prefix_caching=False,
                 num_host_blocks=0):
        self._lib = load_library()
        fo = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
        h = self._lib.bm_create(num_blocks, block_size, _i32p(fo), len(fo))
        if not h:
            raise ValueError("bm_create: invalid arguments")
        self._h = ctypes.c_void_p(h)
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.prefix_caching = bool(prefix_caching)
        if prefix_caching:
            _check(self._lib.bm_enable_prefix_caching(self._h), "bm_enable_prefix_caching")
        self.num_host_blocks = int(num_host_blocks)
        if num_host_blocks:
            _check(self._lib.bm_set_host_blocks(self._h, int(num_host_blocks)), "bm_set_host_blocks")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.bm_destroy(h)
            self._h = None

    def add_seq(self, sid):
        _check(self._lib.bm_add_seq(self._h, sid), "bm_add_seq")

    def append_slot(self, sid):
        """Returns ``(slot, cow)``; ``cow`` is ``(src, dst)`` or None."""
        slot = ctypes.c_int64()
        s, d = ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.bm_append_slot(self._h, sid, ctypes.byref(slot), ctypes.byref(s),
                                        ctypes.byref(d)), "bm_append_slot")
        return slot.value, ((s.value, d.value) if s.value >= 0 else None)

    def append_n(self, sid, n):
        """n appends to one sequence; returns the CoW pairs raised, as a list. All
        or nothing: if the pool cannot take them all, ``PagedKVError`` (status
        ``PKV_ERR_POOL_EXHAUSTED``) and nothing changes."""
        cap = max(1, n)
        buf = np.zeros((cap, 2), dtype=np.int64)
        cnt = ctypes.c_int(0)
        _check(self._lib.bm_append_n(self._h, sid, n, _i64p(buf), cap, ctypes.byref(cnt)),
               "bm_append_n")
        return [tuple(map(int, r)) for r in buf[:cnt.value]]

    def append_slots(self, seq_ids):
        """One append per listed sequence, in list order (an id may repeat);
        returns (slots int64 array, pairs int64 [P, 2]). All or nothing, as
        ``append_n``."""
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        slots = np.zeros(len(ids), dtype=np.int64)
        pairs = np.zeros((max(1, len(ids)), 2), dtype=np.int64)
        cnt = ctypes.c_int(0)
        _check(self._lib.bm_append_slots(self._h, _i64p(ids), len(ids), _i64p(slots),
                                         _i64p(pairs), ctypes.byref(cnt)), "bm_append_slots")
        return slots, pairs[:cnt.value].copy()

    def plan_decode_into(self, ids_p, n, max_blocks, slots_p, pairs_p, tables_p, lens_p,
                         groups=None):
        """The host half of a decode step in one native call (``bm_plan_decode``),
        written straight into caller buffers given as ctypes pointers (e.g. views
        of a pinned upload slab), with no array allocated: one append per listed
        sequence (``slots_p`` int64 [n], ``pairs_p`` int64 [n, 2]: the
        copy-on-write pairs), dense ``tables_p`` int32 [n, max_blocks] and
        ``lens_p`` int32 [n], and, with ``groups = (max_members, members_p,
        prefix_p, seq_group_p, blocks_p, ungrouped_p)`` (int32 [n, max_members],
        [n], [n], [n], [n]), the prefix groups and the batch indices in no group.
        Returns (pairs, groups, ungrouped, longest group list). All or nothing:
        a refused step leaves the manager unchanged."""
        cnt, ng, nu, mgb = (ctypes.c_int(0) for _ in range(4))
        if groups is None:
            args = (0, None, None, None, None, None)
        else:
            args = groups
        _check(self._lib.bm_plan_decode(self._h, ids_p, n, max_blocks, slots_p, pairs_p,
                                        ctypes.byref(cnt), tables_p, lens_p, *args,
                                        ctypes.byref(ng), ctypes.byref(nu), ctypes.byref(mgb)),
               "bm_plan_decode")
        return cnt.value, ng.value, nu.value, mgb.value

    def fork(self, parent, child):
        _check(self._lib.bm_fork(self._h, parent, child), "bm_fork")

    def free_seq(self, sid):
        _check(self._lib.bm_free_seq(self._h, sid), "bm_free_seq")

    def beam_step(self, old_ids, parents, new_ids):
        """New beam ``new_ids[i]`` continues ``old_ids[parents[i]]`` (forked, in
        order), then the old beams are freed; nothing changes on an error."""
        old = np.ascontiguousarray(np.asarray(old_ids, dtype=np.int64))
        par = np.ascontiguousarray(np.asarray(parents, dtype=np.int32))
        new = np.ascontiguousarray(np.asarray(new_ids, dtype=np.int64))
        if len(par) != len(new):
            raise ValueError("parents and new_ids differ in length")
        _check(self._lib.bm_beam_step(self._h, _i64p(old), len(old), _i32p(par), _i64p(new),
                                      len(new)), "bm_beam_step")

    def block_table(self, sid):
        n = ctypes.c_int(0)
        st = self._lib.bm_block_table(self._h, sid, None, 0, ctypes.byref(n))
        if st not in (0, -1):
            _check(st, "bm_block_table")
        out = np.zeros(max(1, n.value), dtype=np.int32)
        _check(self._lib.bm_block_table(self._h, sid, _i32p(out), len(out), ctypes.byref(n)),
               "bm_block_table")
        return [int(x) for x in out[:n.value]]

    def build_tables(self, seq_ids, max_blocks):
        """int32 tables ``[n, max_blocks]`` (-1 padded) and int32 lengths ``[n]``."""
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        tables = np.empty((len(ids), max_blocks), dtype=np.int32)   # every entry written
        lens = np.empty(len(ids), dtype=np.int32)
        _check(self._lib.bm_build_tables(self._h, _i64p(ids), len(ids), max_blocks,
                                         _i32p(tables), _i32p(lens)), "bm_build_tables")
        return tables, lens

    def prefix_groups(self, seq_ids, max_members):
        """Groups of the batch that share leading full blocks (see bm_prefix_groups):
        (members int32 [g, max_members], prefix int32 [g], seq_group int32 [n],
        list blocks int32 [g])."""
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = len(ids)
        members = np.full((max(1, n), max_members), -1, dtype=np.int32)
        prefix = np.zeros(max(1, n), dtype=np.int32)
        seq_group = np.full(max(1, n), -1, dtype=np.int32)
        blocks = np.zeros(max(1, n), dtype=np.int32)
        ng = ctypes.c_int(0)
        _check(self._lib.bm_prefix_groups(self._h, _i64p(ids), n, max_members, _i32p(members),
                                          _i32p(prefix), _i32p(seq_group), _i32p(blocks),
                                          ctypes.byref(ng)), "bm_prefix_groups")
        g = ng.value
        return members[:g].copy(), prefix[:g].copy(), seq_group[:n].copy(), blocks[:g].copy()

    def seq_len(self, sid):
        n = ctypes.c_int(0)
        _check(self._lib.bm_seq_len(self._h, sid, ctypes.byref(n)), "bm_seq_len")
        return n.value

    def refcount(self, block):
        n = ctypes.c_int(0)
        _check(self._lib.bm_refcount(self._h, block, ctypes.byref(n)), "bm_refcount")
        return n.value

    def num_free(self):
        return int(self._lib.bm_num_free(self._h))

    def free_list(self):
        n = self._lib.bm_free_list(self._h, None, 0)
        out = np.zeros(max(1, n), dtype=np.int32)
        self._lib.bm_free_list(self._h, _i32p(out), len(out))
        return [int(x) for x in out[:n]]

    # ---- prefix caching (BlockManager(..., prefix_caching=True))
    def add_seq_prompt(self, sid, prompt):
        """New sequence reusing the cached full blocks of ``prompt``; returns the
        number of prompt tokens already cached (append the rest with
        ``append_tokens``)."""
        p = np.ascontiguousarray(np.asarray(prompt, dtype=np.int32))
        n = ctypes.c_int(0)
        _check(self._lib.bm_add_seq_prompt(self._h, sid, _i32p(p), len(p), ctypes.byref(n)),
               "bm_add_seq_prompt")
        return n.value

    def append_tokens(self, sid, tokens):
        """Appends with token ids; returns (slots int64 array, CoW pairs int64
        [P, 2]). All or nothing, as ``append_n``."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        slots = np.zeros(max(1, len(t)), dtype=np.int64)
        pairs = np.zeros((max(1, len(t)), 2), dtype=np.int64)
        cnt = ctypes.c_int(0)
        _check(self._lib.bm_append_tokens(self._h, sid, _i32p(t), len(t), _i64p(slots),
                                          _i64p(pairs), len(t), ctypes.byref(cnt)),
               "bm_append_tokens")
        return slots[:len(t)].copy(), pairs[:cnt.value].copy()

    def cache_stats(self):
        """(hit blocks, looked-up blocks, registered blocks, evictable blocks)."""
        h, l = ctypes.c_int64(), ctypes.c_int64()
        c, e = ctypes.c_int(), ctypes.c_int()
        _check(self._lib.bm_cache_stats(self._h, ctypes.byref(h), ctypes.byref(l), ctypes.byref(c),
                                        ctypes.byref(e)), "bm_cache_stats")
        return h.value, l.value, c.value, e.value

    # ---- swapping to host blocks (BlockManager(..., num_host_blocks=n))
    def _swap(self, fn, sid, what):
        n = ctypes.c_int(0)
        st = fn(self._h, sid, None, 0, ctypes.byref(n))
        if st == 0:                                      # a sequence without blocks
            return np.zeros((0, 2), dtype=np.int64)
        if st != -1 or n.value == 0:
            _check(st, what)
        pairs = np.zeros((max(1, n.value), 2), dtype=np.int64)
        _check(fn(self._h, sid, _i64p(pairs), n.value, ctypes.byref(n)), what)
        return pairs[:n.value].copy()

    def swap_out(self, sid):
        """Move the sequence to host blocks; returns (device, host) pairs [n, 2]."""
        return self._swap(self._lib.bm_swap_out, sid, "bm_swap_out")

    def swap_in(self, sid):
        """Move a swapped-out sequence back; returns (host, device) pairs [n, 2]."""
        return self._swap(self._lib.bm_swap_in, sid, "bm_swap_in")

    def is_swapped(self, sid):
        f = ctypes.c_int(0)
        _check(self._lib.bm_is_swapped(self._h, sid, ctypes.byref(f)), "bm_is_swapped")
        return bool(f.value)

    def host_free_list(self):
        n = self._lib.bm_host_free_list(self._h, None, 0)
        out = np.zeros(max(1, n), dtype=np.int32)
        self._lib.bm_host_free_list(self._h, _i32p(out), len(out))
        return [int(x) for x in out[:n]]

    def evictable_list(self):
        n = self._lib.bm_evictable_list(self._h, None, 0)
        out = np.zeros(max(1, n), dtype=np.int32)
        self._lib.bm_evictable_list(self._h, _i32p(out), len(out))
        return [int(x) for x in out[:n]]
