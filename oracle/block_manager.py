"""Oracle: KV block manager (free list, block tables, reference counts, CoW).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

Each rule below is a step the pages state, taken in their order:

* "PagedAttention" glossary, "Cách phân trang hoạt động": the cache is split into
  blocks of a fixed number of tokens; a request receives a new block only when
  its last block is full, from wherever a free block is; its block table records
  the order. The worked example takes free blocks with ``pop(0)`` from a list of
  scattered ids, so the free list is consumed from its front.
* "KV cache paginado e batching contínuo para LLMs", "Como funciona": several
  logical blocks may point at one physical block, with a reference count; when a
  sequence must write into a shared block it copies at block level: allocate
  another block, copy, and decrement the original's count.
* Same page and the glossary's "Batching liên tục" item: a finished sequence's
  blocks go straight back to the free pool.

Readings where the pages are silent:

* the first block is taken at the first token, and a new one whenever the
  sequence length is a multiple of the block size before the append;
* a block is "shared" when its reference count is above 1; a sequence that
  writes into its last block while it is shared triggers the copy, and the last
  remaining owner (count 1) writes in place;
* a freed block (count reaching 0) is appended at the tail of the free list, and
  a sequence's blocks are released in table order;
* running out of free blocks is an error (``PoolExhausted``), never a silent
  overwrite.

Swapping ("KV cache paginado...", "Como funciona": when physical blocks run out
the newest requests are preempted, all or nothing, and their blocks recovered by
swapping them to the CPU or by recomputation). Readings: a second pool of
``num_cpu_blocks`` host blocks with its own free list (front first, freed blocks
to the tail); ``swap_out`` moves one sequence whole -- each block of its table,
in table order, gets a fresh host block and a (device, host) copy pair, and the
device blocks are released as on ``free_seq``; ``swap_in`` is the reverse with
(host, device) pairs and fresh device blocks. If either pool cannot take the
whole sequence nothing changes (``PoolExhausted``). A swapped-out sequence can
only be swapped in or freed (its host blocks return to the host free list).

Beam search (glossary, "Chia sẻ block giữa các chuỗi": beams share blocks
through their tables with a count per block, and a beam about to write into a
shared block copies it first). One step's reshuffle of the beams, a reading:
new beam ``i`` continues old beam ``parents[i]`` -- forked from it, in order of
``i`` -- and then every old beam is freed, in order, so an old beam nobody
continues returns the blocks only it held and a continued one hands its blocks
on. The new beams' next appends then copy any shared partial last block.
"""


class PoolExhausted(RuntimeError):
    pass


class BlockManager:
    def __init__(self, num_blocks, block_size, free_order, num_cpu_blocks=0):
        """``free_order``: the initially free block ids, front first (blocks not
        listed belong to someone else and are never handed out); host blocks
        0..num_cpu_blocks-1 start free in that order."""
        free_order = [int(b) for b in free_order]
        if len(set(free_order)) != len(free_order) or any(
                not 0 <= b < num_blocks for b in free_order):
            raise ValueError("free_order must list distinct block ids of the pool")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(free_order)
        self.ref = [0] * num_blocks
        self.tables = {}
        self.lens = {}
        self.num_cpu_blocks = num_cpu_blocks
        self.cpu_free = list(range(num_cpu_blocks))
        self.swapped = set()

    def _take(self):
        if not self.free:
            raise PoolExhausted("no free block")
        b = self.free.pop(0)
        self.ref[b] = 1
        return b

    def add_seq(self, sid):
        if sid in self.tables:
            raise ValueError("sequence exists")
        self.tables[sid] = []
        self.lens[sid] = 0

    def append_slot(self, sid):
        """Reserve the slot for the sequence's next token (not while swapped out).

        Returns ``(slot, cow)`` with ``slot = block * block_size + offset`` and
        ``cow`` either ``None`` or the pair ``(src, dst)`` of a block copy that
        must happen before the token is written.
        """
        if sid in self.swapped:
            raise ValueError("sequence is swapped out")
        table = self.tables[sid]
        n = self.lens[sid]
        cow = None
        if n % self.block_size == 0:
            table.append(self._take())
        else:
            last = table[-1]
            if self.ref[last] > 1:
                dst = self._take()
                self.ref[last] -= 1
                table[-1] = dst
                cow = (last, dst)
        block = table[n // self.block_size]
        slot = block * self.block_size + n % self.block_size
        self.lens[sid] = n + 1
        return slot, cow

    def fork(self, parent, child):
        """Child shares every block of the parent; counts go up by one."""
        if child in self.tables:
            raise ValueError("sequence exists")
        if parent in self.swapped:
            raise ValueError("sequence is swapped out")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def _release(self, table):
        """Drop one reference to each device block of ``table``, in order."""
        for b in table:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)

    def _device_blocks_available(self):
        return len(self.free)

    def free_seq(self, sid):
        table = self.tables.pop(sid)
        if sid in self.swapped:
            self.swapped.discard(sid)
            self.cpu_free.extend(table)
        else:
            self._release(table)
        del self.lens[sid]

    def swap_out(self, sid):
        """Move the sequence's blocks to the host pool; returns the (device,
        host) copy pairs, in table order."""
        if sid in self.swapped:
            raise ValueError("sequence is swapped out")
        table = self.tables[sid]
        if len(table) > len(self.cpu_free):
            raise PoolExhausted("host pool cannot take the sequence")
        host = [self.cpu_free.pop(0) for _ in table]
        pairs = list(zip(table, host))
        self._release(table)
        self.tables[sid] = host
        self.swapped.add(sid)
        return pairs

    def swap_in(self, sid):
        """Move a swapped-out sequence back to fresh device blocks; returns the
        (host, device) copy pairs, in table order."""
        if sid not in self.swapped:
            raise ValueError("sequence is not swapped out")
        host = self.tables[sid]
        if len(host) > self._device_blocks_available():
            raise PoolExhausted("device pool cannot take the sequence")
        dev = [self._take() for _ in host]
        self.tables[sid] = dev
        self.swapped.discard(sid)
        self.cpu_free.extend(host)
        return list(zip(host, dev))

    def block_table(self, sid):
        return list(self.tables[sid])

    def seq_len(self, sid):
        return self.lens[sid]

    def refcount(self, block):
        return self.ref[block]

    def num_free(self):
        return len(self.free)

    def beam_step(self, old_ids, parents, new_ids):
        """New beam ``new_ids[i]`` continues ``old_ids[parents[i]]``; then the old
        beams are freed. Nothing changes if an argument is invalid."""
        old_ids, new_ids = list(old_ids), list(new_ids)
        if len(parents) != len(new_ids) or len(set(old_ids)) != len(old_ids) or \
                len(set(new_ids)) != len(new_ids):
            raise ValueError("parents must match new_ids; ids must be distinct")
        if any(s not in self.tables or s in self.swapped for s in old_ids):
            raise ValueError("old beam unknown or swapped out")
        if any(s in self.tables for s in new_ids):
            raise ValueError("new beam id in use")
        if any(not 0 <= int(p) < len(old_ids) for p in parents):
            raise ValueError("parent index out of range")
        for p, sid in zip(parents, new_ids):
            self.fork(old_ids[int(p)], sid)
        for sid in old_ids:
            self.free_seq(sid)

    def blocks_in_use(self):
        """Physical device blocks with a nonzero count."""
        return sum(1 for c in self.ref if c > 0)


def replay(bm, script):
    """Apply a workload script's operations to ``bm``; returns the CoW pairs the
    appends raised, in order. Ops: ``("add", sid)``, ``("append", sid, n)``,
    ``("fork", parent, child)``, ``("free", sid)``, ``("beam", old_ids, parents,
    new_ids)``."""
    pairs = []
    for op in script:
        if op[0] == "add":
            bm.add_seq(op[1])
        elif op[0] == "append":
            for _ in range(op[2]):
                cow = bm.append_slot(op[1])[1]
                if cow is not None:
                    pairs.append(cow)
        elif op[0] == "fork":
            bm.fork(op[1], op[2])
        elif op[0] == "free":
            bm.free_seq(op[1])
        elif op[0] == "beam":
            bm.beam_step(op[1], op[2], op[3])
        else:
            raise ValueError(f"unknown op {op[0]}")
    return pairs
