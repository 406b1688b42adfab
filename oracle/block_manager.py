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
"""


class PoolExhausted(RuntimeError):
    pass


class BlockManager:
    def __init__(self, num_blocks, block_size, free_order):
        """``free_order``: the initially free block ids, front first (blocks not
        listed belong to someone else and are never handed out)."""
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
        """Reserve the slot for the sequence's next token.

        Returns ``(slot, cow)`` with ``slot = block * block_size + offset`` and
        ``cow`` either ``None`` or the pair ``(src, dst)`` of a block copy that
        must happen before the token is written.
        """
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
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_seq(self, sid):
        for b in self.tables.pop(sid):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        del self.lens[sid]

    def block_table(self, sid):
        return list(self.tables[sid])

    def seq_len(self, sid):
        return self.lens[sid]

    def refcount(self, block):
        return self.ref[block]

    def num_free(self):
        return len(self.free)
