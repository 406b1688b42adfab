"""One decode step of paged attention, end to end, over the C ABI.

A ``PagedKVCache`` owns the two device pools (tiles of 128-byte core matrices,
see ``pool_shapes``; ``k_view``/``v_view`` give the plain ``[NB, Hkv, bs, D]``
view) and a host ``BlockManager``. A step is:

1. host: one ``append_slot`` per sequence -> slot numbers and copy-on-write
   pairs ("KV cache paginado...", "Como funciona": copy a shared block before
   writing into it); dense block tables and lengths for the batch;
2. device, in stream order: ``copy_blocks`` (CoW copies first), then
   ``reshape_and_cache`` (the new token's K/V into its slot), then
   ``paged_attention_decode`` (glossary "PagedAttention": attention reads the
   cache back through the block table).

Pools are allocated by torch (device memory is plumbing); all arithmetic runs in
the library's kernels.
"""
import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import (PKV_ERR_POOL_EXHAUSTED, BlockManager, DecodePipelineStepArgs, PagedKVError, _check,
               _decode_shapes, _dt, _workspace, bind_paged_decode_step, copy_blocks, paged_attention_decode, paged_prefill_step,
               paged_attention_decode_grouped, load_library, paged_attention_workspace_size, pool_shapes, pool_views,
               reshape_and_cache, swap_blocks)


@dataclass
class StepPlan:
    """Host-side inputs of one decode step."""
    seq_ids: np.ndarray      # int64 [B]
    slots: np.ndarray        # int64 [B]
    pairs: np.ndarray        # int64 [P, 2]
    tables: np.ndarray       # int32 [B, max_blocks]
    lens: np.ndarray         # int32 [B]
    seq_group: np.ndarray = None      # int32 [B]; shared-prefix groups (-1: none)
    group_members: np.ndarray = None  # int32 [g, max_members]
    group_prefix: np.ndarray = None   # int32 [g]
    group_blocks: np.ndarray = None   # int32 [g]; each group's block list (prefix once)

    @property
    def num_groups(self):
        return 0 if self.group_members is None else int(self.group_members.shape[0])

    def host_tensors(self, pin=True):
        t = {"slots": torch.from_numpy(self.slots), "pairs": torch.from_numpy(self.pairs),
             "tables": torch.from_numpy(self.tables), "lens": torch.from_numpy(self.lens)}
        if self.num_groups:
            t.update({"ungrouped": torch.from_numpy(
                          np.nonzero(self.seq_group < 0)[0].astype(np.int32)),
                      "seq_group": torch.from_numpy(self.seq_group),
                      "group_members": torch.from_numpy(self.group_members),
                      "group_prefix": torch.from_numpy(self.group_prefix)})
        if pin:
            t = {k: v.pin_memory() for k, v in t.items()}
        return t

    def device_tensors(self, device, non_blocking=False):
        """The host tensors on the device, plus (grouped plans) the host int
        ``max_group_blocks`` that sizes the group launch."""
        d = {k: v.to(device, non_blocking=non_blocking)
             for k, v in self.host_tensors(pin=non_blocking).items()}
        if self.num_groups:
            d["max_group_blocks"] = self.max_group_blocks
        return d

    @property
    def max_group_blocks(self):
        return int(self.group_blocks.max()) if self.num_groups else 0

    def nbytes(self):
        n = self.slots.nbytes + self.pairs.nbytes + self.tables.nbytes + self.lens.nbytes
        if self.num_groups:
            n += self.seq_group.nbytes + self.group_members.nbytes + self.group_prefix.nbytes
        return n


@dataclass
class PrefillPlan:
    """Host-side inputs of one chunked-prefill step."""
    seq_ids: np.ndarray      # int64 [B]
    chunks: np.ndarray       # int64 [B] new tokens per sequence
    slots: np.ndarray        # int64 [T] slot of every chunk token (sequence by sequence)
    pairs: np.ndarray        # int64 [P, 2]
    tables: np.ndarray       # int32 [B, max_blocks]
    lens: np.ndarray         # int32 [B]
    query_start: np.ndarray  # int32 [B + 1]

    @property
    def max_query_len(self):
        return int(self.chunks.max()) if len(self.chunks) else 0

    def host_tensors(self, pin=True):
        t = {"slots": torch.from_numpy(self.slots), "pairs": torch.from_numpy(self.pairs),
             "tables": torch.from_numpy(self.tables), "lens": torch.from_numpy(self.lens),
             "query_start": torch.from_numpy(self.query_start)}
        if pin:
            t = {k: v.pin_memory() for k, v in t.items()}
        return t

    def device_tensors(self, device, non_blocking=False):
        return {k: v.to(device, non_blocking=non_blocking)
                for k, v in self.host_tensors(pin=non_blocking).items()}


def host_runs(host_ids):
    """Runs of consecutive host block ids in a list: (start, stop, first id)
    triples, so block ``host_ids[i]`` for ``start <= i < stop`` is ``first id +
    i - start``."""
    ids = np.asarray(host_ids, dtype=np.int64).reshape(-1)
    runs, a = [], 0
    for i in range(1, len(ids) + 1):
        if i == len(ids) or ids[i] != ids[i - 1] + 1:
            runs.append((a, i, int(ids[a])))
            a = i
    return runs


def copy_waves(pairs):
    """Cut a list of (src, dst) block copies, meant to run in order, into
    consecutive [start, stop) waves that ``copy_blocks`` may run concurrently:
    within a wave no block is written twice and no block written is also read.
    A copy that reads or writes a block an earlier copy of the current wave
    wrote, or writes one it read, starts a new wave. The pairs of one step
    (fresh destinations) always form a single wave."""
    waves, start, written, read = [], 0, set(), set()
    for i, (src, dst) in enumerate(np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist()):
        if src in written or dst in written or dst in read:
            waves.append((start, i))
            start, written, read = i, set(), set()
        written.add(dst)
        read.add(src)
    if len(pairs) > start:
        waves.append((start, len(pairs)))
    return waves


class PagedKVCache:
    def __init__(self, num_blocks, num_heads, num_kv_heads, head_dim, block_size, kv_dtype,
                 free_order, device="cuda", prefix_caching=False, num_host_blocks=0):
        self.device = torch.device(device)
        self.num_blocks = num_blocks
        self.num_heads = num_heads
        self.num_kv_heads = num_kv_heads
        self.head_dim = head_dim
        self.block_size = block_size
        k_shape, v_shape = pool_shapes(num_blocks, num_kv_heads, block_size, head_dim, kv_dtype)
        self.k_pool = torch.empty(k_shape, dtype=kv_dtype, device=self.device)
        self.v_pool = torch.empty(v_shape, dtype=kv_dtype, device=self.device)
        self.bm = BlockManager(num_blocks, block_size, free_order, prefix_caching=prefix_caching,
                               num_host_blocks=num_host_blocks)
        self.num_host_blocks = num_host_blocks
        if num_host_blocks:
            hk, hv = pool_shapes(num_host_blocks, num_kv_heads, block_size, head_dim, kv_dtype)
            self.host_k = torch.empty(hk, dtype=kv_dtype).pin_memory()
            self.host_v = torch.empty(hv, dtype=kv_dtype).pin_memory()

    def load(self, k_vals, v_vals, k_scale=1.0, v_scale=1.0):
        """Fill every slot from values given as ``[NB, Hkv, bs, D]`` (block,
        head, slot, dim), through the library's slot write (which lays them out
        and, for an E4M3 cache, quantises them)."""
        NB, Hkv, bs, D = self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim
        slots = torch.arange(NB * bs, dtype=torch.int64, device=self.device)
        tok = lambda x: x.to(self.device).permute(0, 2, 1, 3).reshape(NB * bs, Hkv, D).contiguous()
        reshape_and_cache(tok(k_vals), tok(v_vals), self.k_pool, self.v_pool, slots, k_scale, v_scale)

    def k_view(self):
        """K pool as ``[NB, Hkv, bs, D]`` (a copy, for inspection and tests)."""
        return pool_views(self.k_pool, self.v_pool)[0]

    def v_view(self):
        """V pool as ``[NB, Hkv, bs, D]`` (a copy, for inspection and tests)."""
        return pool_views(self.k_pool, self.v_pool)[1]

    def replay(self, script):
        """Apply block-manager operations; returns the CoW pairs raised (in order)."""
        pairs = []
        for op in script:
            if op[0] == "add":
                self.bm.add_seq(op[1])
            elif op[0] == "append":
                pairs += self.bm.append_n(op[1], op[2])
            elif op[0] == "fork":
                self.bm.fork(op[1], op[2])
            elif op[0] == "free":
                self.bm.free_seq(op[1])
            elif op[0] == "beam":
                self.bm.beam_step(op[1], op[2], op[3])
            else:
                raise ValueError(f"unknown op {op[0]}")
        return pairs

    def apply_copies(self, pairs, stream=None):
        """Apply (src, dst) block copies in list order, e.g. the CoW pairs of a
        replayed script spanning many steps: one ``copy_blocks`` launch per wave
        of ``copy_waves``."""
        pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
        for a, b in copy_waves(pairs):
            t = torch.as_tensor(pairs[a:b], device=self.device)
            copy_blocks(self.k_pool, self.v_pool, t, stream=stream)

    def plan_step(self, seq_ids, max_blocks=None, group_prefixes=True):
        """Host half of a step: one slot per sequence (CoW pairs included), dense
        tables and, when sequences share leading full blocks (forks of one prompt),
        the prefix groups that let the decode read those blocks once per group."""
        ids = np.asarray(seq_ids, dtype=np.int64)
        slots, pairs = self.bm.append_slots(ids)
        if max_blocks is None:
            max_blocks = max(1, max((-(-self.bm.seq_len(int(s)) // self.block_size) for s in ids),
                                    default=0))
        tables, lens = self.bm.build_tables(ids, max_blocks)
        plan = StepPlan(ids, slots, pairs, tables, lens)
        if group_prefixes and self.k_pool.dtype != torch.float32:
            max_members = max(1, 8 // (self.num_heads // self.num_kv_heads))
            members, prefix, seq_group, blocks = self.bm.prefix_groups(ids, max_members)
            if len(members):
                plan.seq_group, plan.group_members, plan.group_prefix = seq_group, members, prefix
                plan.group_blocks = blocks
        return plan

    def plan_step_preempting(self, requests, preempt, max_blocks=None, group_prefixes=True):
        """``plan_step`` under the rule for running out of blocks ("KV cache
        paginado...", "Como funciona": the newest requests are preempted, all or
        nothing, and their blocks recovered by swapping or recomputation).

        ``requests``: the running requests, oldest first; each is a sequence id
        or a list of the ids of one request's sequences (its samples or beams).
        The step appends to every sequence of every request. While the manager
        refuses the whole step (it changes nothing then), the newest remaining
        request goes whole to ``preempt(ids)``, which must release its device
        blocks (``preempt_by_recompute``, or ``swap_out``), and the step is planned
        again without it. Returns ``(plan, preempted)``: ``preempted`` lists what
        each ``preempt`` call returned, newest request first; ``plan`` is None
        when no request was left."""
        reqs = [[int(r)] if np.isscalar(r) else [int(s) for s in r] for r in requests]
        preempted = []
        while reqs:
            ids = [s for r in reqs for s in r]
            try:
                return self.plan_step(ids, max_blocks, group_prefixes), preempted
            except PagedKVError as e:
                if e.status != PKV_ERR_POOL_EXHAUSTED:
                    raise
            preempted.append(preempt(reqs.pop()))
        return None, preempted

    def plan_prefill(self, seq_ids, chunks, max_blocks=None):
        """Host half of a chunked-prefill step: ``chunks[i]`` appends to sequence
        ``seq_ids[i]`` (slots in token order, CoW pairs), dense tables, lengths and
        the chunk offsets."""
        ids = np.asarray(seq_ids, dtype=np.int64)
        chunks = np.asarray(chunks, dtype=np.int64)
        slots, pairs = self.bm.append_slots(np.repeat(ids, chunks))
        if max_blocks is None:
            max_blocks = max(1, max((-(-self.bm.seq_len(int(s)) // self.block_size) for s in ids),
                                    default=0))
        tables, lens = self.bm.build_tables(ids, max_blocks)
        qs = np.zeros(len(ids) + 1, dtype=np.int32)
        qs[1:] = np.cumsum(chunks)
        return PrefillPlan(ids, chunks, slots, pairs, tables, lens, qs)

    def swap_out(self, seq_ids, stream=None, copy_engines=False):
        """Preempt sequences by swapping: each moves, all or nothing, to host blocks
        and its K/V is copied there; returns the (device, host) pairs.

        ``copy_engines``: the blocks are first gathered into a contiguous device
        staging buffer (one ``swap_blocks`` launch, HBM to HBM), then cross to the
        host on the copy engines, one copy per run of consecutive host blocks, so
        the SMs stay free for concurrent work; otherwise one ``swap_blocks``
        launch copies every block over the host link from the SMs."""
        pairs = [self.bm.swap_out(int(s)) for s in seq_ids]
        pairs = np.concatenate(pairs) if pairs else np.zeros((0, 2), np.int64)
        if len(pairs) and not copy_engines:
            swap_blocks(self.host_k, self.host_v, self.k_pool, self.v_pool,
                        torch.as_tensor(pairs, device=self.device), stream)
        elif len(pairs):
            sk, sv = self.staging_pools(len(pairs))
            gather = np.stack([pairs[:, 0], np.arange(len(pairs))], 1)
            swap_blocks(sk, sv, self.k_pool, self.v_pool,
                        torch.as_tensor(gather, device=self.device), stream)
            with torch.cuda.stream(stream or torch.cuda.current_stream(self.device)):
                for a, b, h in host_runs(pairs[:, 1]):
                    self.host_k[h:h + b - a].copy_(sk[a:b], non_blocking=True)
                    self.host_v[h:h + b - a].copy_(sv[a:b], non_blocking=True)
        return pairs

    def swap_in(self, seq_ids, stream=None, copy_engines=False):
        """Bring swapped-out sequences back onto fresh device blocks; returns the
        (host, device) pairs. ``copy_engines`` as for ``swap_out``, in reverse: the
        host runs land in the staging buffer, one launch scatters them."""
        pairs = [self.bm.swap_in(int(s)) for s in seq_ids]
        pairs = np.concatenate(pairs) if pairs else np.zeros((0, 2), np.int64)
        if len(pairs) and not copy_engines:
            swap_blocks(self.k_pool, self.v_pool, self.host_k, self.host_v,
                        torch.as_tensor(pairs, device=self.device), stream)
        elif len(pairs):
            sk, sv = self.staging_pools(len(pairs))
            with torch.cuda.stream(stream or torch.cuda.current_stream(self.device)):
                for a, b, h in host_runs(pairs[:, 0]):
                    sk[a:b].copy_(self.host_k[h:h + b - a], non_blocking=True)
                    sv[a:b].copy_(self.host_v[h:h + b - a], non_blocking=True)
            scatter = np.stack([np.arange(len(pairs)), pairs[:, 1]], 1)
            swap_blocks(self.k_pool, self.v_pool, sk, sv,
                        torch.as_tensor(scatter, device=self.device), stream)
        return pairs

    def preempt_by_recompute(self, seq_ids):
        """Preempt sequences by recomputation ("KV cache paginado...", "Como
        funciona": a preempted request's blocks are recovered by swapping or by
        recomputing them later): their blocks are freed now. Returns each one's
        token count, for ``plan_resume``."""
        lens = {int(s): self.bm.seq_len(int(s)) for s in seq_ids}
        for s in seq_ids:
            self.bm.free_seq(int(s))
        return lens

    def plan_resume(self, seq_ids, lens, max_blocks=None):
        """Host half of resuming sequences preempted by recomputation: each is
        added again and all of its ``lens[s]`` tokens form one chunk, so one
        chunked-prefill step (``prefill_step`` with their recomputed q, K, V)
        writes their K/V into fresh blocks and attends over them. If the pool
        cannot take them all, none is added and the error is raised."""
        added = []
        try:
            for s in seq_ids:
                self.bm.add_seq(int(s))
                added.append(int(s))
            return self.plan_prefill(seq_ids, [lens[int(s)] for s in seq_ids], max_blocks)
        except PagedKVError:
            for s in reversed(added):                # still preempted, nothing held
                self.bm.free_seq(s)
            raise

    def staging_pools(self, n):
        """Device staging pools of at least n blocks (grown on demand)."""
        have = getattr(self, "_stage", None)
        if have is None or have[0].shape[0] < n:
            ks, vs = pool_shapes(n, self.num_kv_heads, self.block_size, self.head_dim,
                                 self.k_pool.dtype)
            self._stage = (torch.empty(ks, dtype=self.k_pool.dtype, device=self.device),
                           torch.empty(vs, dtype=self.k_pool.dtype, device=self.device))
        return self._stage[0][:n], self._stage[1][:n]

    def plan_prompts(self, seq_ids, prompts, max_blocks=None):
        """Host half of a prefill step with prefix caching (the manager must have
        it on): each new sequence reuses the cached full blocks of its prompt and
        the rest of the prompt is its chunk. ``plan.cached[i]`` = prompt tokens of
        sequence i found in the cache.

        If the pool cannot take every prompt, the sequences this call added are
        freed again, newest first, and the error is raised: their blocks return
        as if they had finished (full prompt blocks stay cached)."""
        ids = np.asarray(seq_ids, dtype=np.int64)
        cached, slots, pairs = [], [], []
        added = []
        try:
            for sid, p in zip(ids, prompts):
                n = self.bm.add_seq_prompt(int(sid), p)
                added.append(int(sid))
                s, pr = self.bm.append_tokens(int(sid), np.asarray(p)[n:])
                cached.append(n)
                slots.append(s)
                pairs.append(pr)
        except PagedKVError:
            for s in reversed(added):
                self.bm.free_seq(s)
            raise
        chunks = np.array([len(p) - n for p, n in zip(prompts, cached)], dtype=np.int64)
        if max_blocks is None:
            max_blocks = max(1, max((-(-self.bm.seq_len(int(s)) // self.block_size) for s in ids),
                                    default=0))
        tables, lens = self.bm.build_tables(ids, max_blocks)
        qs = np.zeros(len(ids) + 1, dtype=np.int32)
        qs[1:] = np.cumsum(chunks)
        plan = PrefillPlan(ids, chunks, np.concatenate(slots) if slots else np.zeros(0, np.int64),
                           np.concatenate(pairs).reshape(-1, 2) if pairs else np.zeros((0, 2), np.int64),
                           tables, lens, qs)
        plan.cached = np.asarray(cached, dtype=np.int64)
        return plan

    def prefill_step(self, q, k_new, v_new, dev_plan, out, scale, max_query_len, stream=None):
        """Device half of a chunked-prefill step: CoW copies, the chunk's K/V into
        its slots, then causal attention of every chunk token (one
        ``paged_prefill_step`` call; the attention reads the tiles before each
        chunk while the writes finish)."""
        return paged_prefill_step(out, q, k_new, v_new, self.k_pool, self.v_pool,
                                  dev_plan["tables"], dev_plan["lens"], dev_plan["query_start"],
                                  dev_plan["slots"], dev_plan["pairs"], scale, max_query_len,
                                  stream)

    def workspace(self, batch, max_blocks):
        """Split-KV scratch, room for split group lists included."""
        n = paged_attention_workspace_size(batch, self.num_heads, self.head_dim, self.block_size,
                                           max_blocks)
        mult = max(1, 8 // (self.num_heads // self.num_kv_heads))
        return torch.empty(max(mult * n, 16), dtype=torch.uint8, device=self.device)

    def decode(self, q, dev_plan, out, scale, k_scale=1.0, v_scale=1.0, workspace=None,
               stream=None):
        """The attention of a step (grouped when the plan found shared prefixes)."""
        if "group_members" in dev_plan:
            return paged_attention_decode_grouped(
                out, q, self.k_pool, self.v_pool, dev_plan["tables"], dev_plan["lens"], scale,
                dev_plan["seq_group"], dev_plan["group_members"], dev_plan["group_prefix"],
                k_scale, v_scale, workspace, stream, dev_plan.get("ungrouped"),
                dev_plan.get("max_group_blocks", 0))
        return paged_attention_decode(out, q, self.k_pool, self.v_pool, dev_plan["tables"],
                                      dev_plan["lens"], scale, k_scale, v_scale, workspace, stream)

    def bind_step(self, q, k_new, v_new, dev_plan, out, scale, k_scale=1.0, v_scale=1.0,
                  workspace=None):
        """``step`` checked once and bound to these tensors: returns ``run(stream,
        num_pairs=None, groups=None)`` that launches the step's copies, slot
        writes and attention (one ``paged_decode_step`` call). ``num_pairs``
        (default: every row of the plan's pairs) counts the filled rows of a pairs
        buffer sized for the most a step can raise; with a grouped plan, ``groups
        = (num_groups, max_group_blocks, num_ungrouped)`` counts the filled rows
        of its group buffers (0 groups: the plain decode)."""
        grouped = "group_members" in dev_plan
        call = bind_paged_decode_step(
            out, q, k_new, v_new, self.k_pool, self.v_pool, dev_plan["tables"], dev_plan["lens"],
            dev_plan["slots"], dev_plan["pairs"], scale, k_scale, v_scale, workspace,
            dev_plan.get("seq_group"), dev_plan.get("group_members"),
            dev_plan.get("group_prefix"), dev_plan.get("ungrouped") if grouped else None,
            dev_plan.get("max_group_blocks", 0) if grouped else 0)

        def run(stream, num_pairs=None, groups=None):
            counts = {}
            if num_pairs is not None:
                counts["num_pairs"] = num_pairs
            if grouped and groups is not None:
                ng, mgb, nu = groups
                counts.update(num_groups=ng, max_group_blocks=mgb)
                if dev_plan.get("ungrouped") is not None:
                    counts["num_ungrouped"] = nu
            call(stream, **counts)
        return run

    def step(self, q, k_new, v_new, dev_plan, out, scale, k_scale=1.0, v_scale=1.0,
             workspace=None, stream=None):
        """The device half of a decode step: copies, slot writes, attention (one
        ``paged_decode_step`` call)."""
        self.bind_step(q, k_new, v_new, dev_plan, out, scale, k_scale, v_scale, workspace)(stream)
        return out


def slab_layout(templates, align=256):
    """Byte offsets of the tensors of ``templates`` packed one after another into
    one buffer, each start a multiple of ``align``: ({name: (offset, dtype,
    shape)}, total bytes). Non-tensor entries are left out."""
    layout, off = {}, 0
    for k, t in templates.items():
        if torch.is_tensor(t):
            layout[k] = (off, t.dtype, tuple(t.shape))
            off += -(-(t.numel() * t.element_size()) // align) * align
    return layout, max(off, align)


def slab_views(slab, layout):
    """Typed views of a uint8 buffer laid out by ``slab_layout``."""
    out = {}
    for k, (off, dtype, shape) in layout.items():
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        out[k] = slab[off:off + n].view(dtype).view(shape)
    return out


class StepPipeline:
    """Decode steps fed from host memory, with the copies overlapped.

    The inputs of a step (q, k_new, v_new and the plan's tensors) live in one
    pinned host slab per buffer set (``host_inputs(i)`` gives step i's views to
    fill in); ``submit`` uploads the slab with one copy on an upload stream, runs
    the step on the compute stream once it has landed, and reads the output back
    into the given pinned buffer on a download stream as soon as the step is
    done. Two buffer sets alternate, so step i+1's upload runs while step i
    computes and step i's download while step i+1 computes; steps run in
    submission order on the compute stream (the cache writes stay ordered).

    ``templates``: tensors shaped like q, k_new, v_new and every plan tensor (a
    first step's ``StepPlan.host_tensors`` plus q and the new K/V), and any host
    values the plan carries (``max_group_blocks``); ``out_template`` is shaped
    like the output. Step i's host views may be rewritten once step i-2's
    ``uploaded`` event has completed (``host_inputs`` waits for it), and its
    output read once its ``downloaded`` event has. ``run(q, k_new, v_new, plan,
    out, stream)`` is the device half of a step; by default a decode step
    (``PagedKVCache.step``; ``submit`` passes its scales and workspace), for a
    chunked-prefill step e.g. ``lambda q, k, v, plan, out, s:
    cache.prefill_step(q, k, v, plan, out, scale, max_query_len, stream=s)``.
    """

    _ALIGN = 256

    def __init__(self, cache, templates, out_template, stream=None, run=None):
        self.cache = cache
        self.run = run
        self.device = cache.device
        self.compute = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.up = torch.cuda.Stream(self.device)
        self.down = torch.cuda.Stream(self.device)
        self.extra = {k: v for k, v in templates.items() if not torch.is_tensor(v)}
        self.layout, self.slab_bytes = slab_layout(templates, self._ALIGN)
        self.host_slabs = [torch.empty(self.slab_bytes, dtype=torch.uint8).pin_memory()
                           for _ in range(2)]
        self.dev_slabs = [torch.empty(self.slab_bytes, dtype=torch.uint8, device=self.device)
                          for _ in range(2)]
        self.outs = [torch.empty_like(out_template, device=self.device) for _ in range(2)]
        self.steps = []                                   # per slab: (q, k_new, v_new, plan)
        for slab in self.dev_slabs:
            dev = self._views(slab)
            plan = {k: v for k, v in dev.items() if k not in ("q", "k_new", "v_new")}
            plan.update(self.extra)
            self.steps.append((dev["q"], dev["k_new"], dev["v_new"], plan))
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.uploaded, self.computed, self.downloaded = ev(), ev(), ev()
        for e in self.uploaded + self.computed + self.downloaded:
            e.record(self.compute)                        # creates the CUDA event now
        self.n = 0
        self._host_views = [self._views(h) for h in self.host_slabs]
        self._bound = [None, None]                        # per slab: (key, bound step)
        # raw handles for the library's stream plumbing (pkv_stage_upload/download)
        self._lib = load_library()
        vp = ctypes.c_void_p
        self._h = {"up": vp(self.up.cuda_stream), "down": vp(self.down.cuda_stream),
                   "compute": vp(self.compute.cuda_stream),
                   "uploaded": [vp(e.cuda_event) for e in self.uploaded],
                   "computed": [vp(e.cuda_event) for e in self.computed],
                   "downloaded": [vp(e.cuda_event) for e in self.downloaded],
                   "host": [vp(t.data_ptr()) for t in self.host_slabs],
                   "dev": [vp(t.data_ptr()) for t in self.dev_slabs],
                   "out": [vp(t.data_ptr()) for t in self.outs]}
        self._slab_size = ctypes.c_size_t(self.slab_bytes)

    def _views(self, slab):
        return slab_views(slab, self.layout)

    def host_inputs(self, i=None):
        """Pinned views to fill with step i's inputs (default: the next step)."""
        i = self.n if i is None else i
        if i >= 2:
            self.uploaded[i % 2].synchronize()            # step i-2's slab has been read
        return self._host_views[i % 2]

    def _bound_step(self, b, scale, k_scale, v_scale, workspace):
        """Slab b's decode step, bound once to its device views (rebound when the
        scales or workspace change)."""
        key = (scale, k_scale, v_scale, None if workspace is None else workspace.data_ptr())
        if self._bound[b] is None or self._bound[b][0] != key:
            q, k_new, v_new, plan = self.steps[b]
            self._bound[b] = (key, self.cache.bind_step(q, k_new, v_new, plan, self.outs[b],
                                                        scale, k_scale, v_scale, workspace))
        return self._bound[b][1]

    def submit(self, host_out, scale=None, k_scale=1.0, v_scale=1.0, workspace=None):
        """Run the next step from its filled host views; ``host_out`` = pinned
        buffer (contiguous, shaped like the output) the output is read back
        into. Returns the step's (uploaded, downloaded) events. The copies and
        the stream ordering are two library calls (pkv_stage_upload /
        pkv_stage_download); step n-2 used the same buffer set, so its events
        order the reuse."""
        b = self.n % 2
        h = self._h
        reuse = self.n >= 2
        _check(self._lib.pkv_stage_upload(
            h["host"][b], h["dev"][b], self._slab_size, h["up"], h["compute"], h["uploaded"][b],
            h["computed"][b] if reuse else None, h["downloaded"][b] if reuse else None),
            "pkv_stage_upload")
        if self.run is None:
            self._bound_step(b, scale, k_scale, v_scale, workspace)(self.compute, **self._counts())
        else:
            q, k_new, v_new, plan = self.steps[b]
            self.run(q, k_new, v_new, plan, self.outs[b], self.compute)
        out = self.outs[b]
        if not (host_out.is_contiguous() and host_out.numel() == out.numel() and
                host_out.dtype == out.dtype and not host_out.is_cuda):
            raise ValueError("host_out must be a contiguous CPU tensor shaped like the output")
        _check(self._lib.pkv_stage_download(
            h["out"][b], ctypes.c_void_p(host_out.data_ptr()),
            ctypes.c_size_t(out.numel() * out.element_size()), h["compute"], h["down"],
            h["computed"][b], h["downloaded"][b]), "pkv_stage_download")
        self.n += 1
        return self.uploaded[b], self.downloaded[b]

    def _counts(self):
        return {}


class LiveDecodePipeline(StepPipeline):
    """Decode steps planned on the host as they are submitted, fed from pinned
    memory and overlapped like ``StepPipeline``.

    Every ``submit`` first plans the step -- the native block manager appends a
    token to each of ``seq_ids`` (slots and copy-on-write pairs), builds dense
    tables and lengths and finds the prefix groups -- straight into the next
    pinned slab (no array is allocated on the way), then uploads that slab with
    the step's q, k_new and v_new (written by the caller into
    ``host_inputs()``, or left from an earlier step), runs the step's launches
    with that step's counts (pairs, groups) and reads the output back -- one
    library call (``pkv_decode_pipeline_step``) for all of it. The slab's plan
    buffers are sized for the most a step can raise (a pair and
    a group row per sequence). Planning ahead of the device work is what the
    pages' lazy allocation asks of the host every step ("Cách phân trang hoạt
    động" of the "PagedAttention" glossary)."""

    def __init__(self, cache, seq_ids, q, k_new, v_new, out_template, max_blocks, stream=None,
                 group_prefixes=True):
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        B = len(ids)
        t = {"q": q, "k_new": k_new, "v_new": v_new,
             "slots": torch.empty(B, dtype=torch.int64),
             "pairs": torch.empty(B, 2, dtype=torch.int64),
             "tables": torch.empty(B, max_blocks, dtype=torch.int32),
             "lens": torch.empty(B, dtype=torch.int32)}
        self.max_members = max(1, 8 // (cache.num_heads // cache.num_kv_heads))
        self.grouped = group_prefixes and cache.k_pool.dtype != torch.float32
        if self.grouped:
            t.update(seq_group=torch.empty(B, dtype=torch.int32),
                     group_members=torch.empty(B, self.max_members, dtype=torch.int32),
                     group_prefix=torch.empty(B, dtype=torch.int32),
                     ungrouped=torch.empty(B, dtype=torch.int32))
        super().__init__(cache, t, out_template, stream)
        self.ids = ids
        self.max_blocks = max_blocks
        self._ids_p = ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        self._blocks = np.zeros(max(1, B), dtype=np.int32)
        p64 = lambda x: ctypes.cast(x.data_ptr(), ctypes.POINTER(ctypes.c_int64))
        p32 = lambda x: ctypes.cast(x.data_ptr(), ctypes.POINTER(ctypes.c_int32))
        self._ptrs = []
        for v in self._host_views:
            g = None
            if self.grouped:
                g = (self.max_members, p32(v["group_members"]), p32(v["group_prefix"]),
                     p32(v["seq_group"]),
                     self._blocks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                     p32(v["ungrouped"]))
            self._ptrs.append((p64(v["slots"]), p64(v["pairs"]), p32(v["tables"]),
                               p32(v["lens"]), g))
        self._step_counts = {}
        self._native_args = [None, None]                  # per slab: (key, step arguments)
        self.last_plan_us = 0.0                           # host planning of the last submit
        self.last_counts = (0, 0, 0, 0)                   # its pairs, groups, ungrouped, longest list

    def plan(self):
        """Plan the next step into its slab with one native call (waits until
        that slab's previous upload has been read). Returns (pairs, groups) of
        the step."""
        self.host_inputs()
        slots_p, pairs_p, tables_p, lens_p, g = self._ptrs[self.n % 2]
        npairs, ng, nu, mgb = self.cache.bm.plan_decode_into(
            self._ids_p, len(self.ids), self.max_blocks, slots_p, pairs_p, tables_p, lens_p, g)
        if self.grouped:
            self._step_counts = {"num_pairs": npairs, "groups": (ng, mgb, nu)}
        else:
            self._step_counts = {"num_pairs": npairs}
        return npairs, ng

    def _native(self, b, scale, k_scale, v_scale, workspace):
        """Slab b's ``pkv_decode_pipeline_step`` arguments, built once per scales
        and workspace (after the bound step's argument checks)."""
        key = (scale, k_scale, v_scale, None if workspace is None else workspace.data_ptr())
        if self._native_args[b] is not None and self._native_args[b][0] == key:
            return self._native_args[b][1]
        self._bound_step(b, scale, k_scale, v_scale, workspace)
        q, k_new, v_new, plan = self.steps[b]
        out, c, h = self.outs[b], self.cache, self._h
        B, Hq, D, NB, Hkv, bs = _decode_shapes(out, q, c.k_pool, c.v_pool, plan["tables"],
                                               plan["lens"])
        ws_ptr, ws_bytes = _workspace(workspace, out.device)
        a = DecodePipelineStepArgs()
        a.seq_ids = self._ids_p
        a.num_seqs, a.max_blocks = len(self.ids), self.max_blocks
        slots_p, pairs_p, tables_p, lens_p, g = self._ptrs[b]
        a.h_slots, a.h_pairs, a.h_tables, a.h_lens = slots_p, pairs_p, tables_p, lens_p
        if g is not None:
            (a.max_members, a.h_group_members, a.h_group_prefix, a.h_seq_group, a.group_blocks,
             a.h_ungrouped) = g
            a.seq_group, a.group_members, a.group_prefix, a.ungrouped = (
                plan[k].data_ptr() for k in ("seq_group", "group_members", "group_prefix",
                                             "ungrouped"))
        a.host_slab, a.dev_slab, a.slab_bytes = h["host"][b], h["dev"][b], self.slab_bytes
        a.q, a.k_new, a.v_new = q.data_ptr(), k_new.data_ptr(), v_new.data_ptr()
        a.slots, a.pairs, a.tables, a.lens = (plan[k].data_ptr()
                                              for k in ("slots", "pairs", "tables", "lens"))
        a.out, a.k_pool, a.v_pool = out.data_ptr(), c.k_pool.data_ptr(), c.v_pool.data_ptr()
        a.num_blocks, a.num_heads, a.num_kv_heads, a.head_dim, a.block_size = NB, Hq, Hkv, D, bs
        a.scale, a.k_scale, a.v_scale = float(scale), float(k_scale), float(v_scale)
        a.q_dtype, a.kv_dtype = _dt(q, "q"), _dt(c.k_pool, "k_pool")
        a.workspace, a.workspace_bytes = ws_ptr, ws_bytes
        a.out_bytes = out.numel() * out.element_size()
        a.up_stream, a.compute_stream, a.down_stream = h["up"], h["compute"], h["down"]
        a.uploaded_event, a.computed_event, a.downloaded_event = (
            h["uploaded"][b], h["computed"][b], h["downloaded"][b])
        self._native_args[b] = (key, a)
        return a

    def submit(self, host_out, scale=None, k_scale=1.0, v_scale=1.0, workspace=None):
        """Plan and run the next step. Unless ``plan`` was called for it, the
        planning, the upload, the step's launches and the read-back are one
        library call (``pkv_decode_pipeline_step``; ``last_plan_us`` and
        ``last_counts`` then report its planning); after ``plan``, the step runs
        as ``StepPipeline.submit`` does."""
        if self._step_counts:
            try:
                return super().submit(host_out, scale, k_scale, v_scale, workspace)
            finally:
                self._step_counts = {}
        if not (host_out.is_contiguous() and host_out.numel() == self.outs[0].numel() and
                host_out.dtype == self.outs[0].dtype and not host_out.is_cuda):
            raise ValueError("host_out must be a contiguous CPU tensor shaped like the output")
        b = self.n % 2
        self.host_inputs()                                # the slab's previous upload is done
        a = self._native(b, scale, k_scale, v_scale, workspace)
        counts, us = (ctypes.c_int * 4)(), ctypes.c_double(0.0)
        a.bm = self.cache.bm._h                           # the manager may have been replaced
        st = self._lib.pkv_decode_pipeline_step(ctypes.byref(a), 1 if self.n >= 2 else 0,
                                                ctypes.c_void_p(host_out.data_ptr()), counts,
                                                ctypes.byref(us))
        self.last_plan_us, self.last_counts = us.value, tuple(counts)
        _check(st, "pkv_decode_pipeline_step")
        self.n += 1
        return self.uploaded[b], self.downloaded[b]

    def _counts(self):
        return self._step_counts
