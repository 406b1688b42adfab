"""Oracle: block manager with prefix caching (full blocks shared across requests).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

What the pages state: the block table lets several sequences point at one
physical block with a reference count per block; parallel samples, beam search
and requests that begin with the same system prompt can reuse one copy of the
common prefix ("PagedAttention" glossary, "Chia sẻ block giữa các chuỗi");
the vLLM feature list names prefix caching ("vLLM PagedAttention: uma revolução
no throughput...").

Readings where the pages are silent, taken in this order:

* a block is shareable across requests once it is full: its identity is the
  exact sequence of token ids from the start of the sequence up to the end of
  that block (its content depends on every earlier token, so only an equal
  prefix may reuse it);
* a new request reuses, from the front, every full block of its prompt whose
  prefix is cached, and stops at the first miss; it always leaves at least one
  prompt token to compute (the step after the prompt needs that token's output),
  so at most ``(len(prompt) - 1) // block_size`` blocks are reused;
* a block is registered when a sequence fills it; if its prefix is already
  registered to another block the new block stays unregistered (first wins);
* a registered block whose count drops to 0 is kept with its contents as
  "evictable" instead of returning to the free list, so a later request with the
  same prefix can revive it; within one sequence release, uncached blocks go to
  the free list in table order and cached ones to the evictable list in reverse
  table order (the end of a prefix becomes evictable before its beginning);
* a new block comes from the front of the free list; when that is empty the
  oldest evictable block is evicted (its registration dropped) and reused;
  running out of both is an error.
"""
from .block_manager import BlockManager, PoolExhausted


class PrefixCachingBlockManager(BlockManager):
    def __init__(self, num_blocks, block_size, free_order, num_cpu_blocks=0):
        super().__init__(num_blocks, block_size, free_order, num_cpu_blocks)
        self.tokens = {}          # sid -> token ids (None where unknown)
        self.key_of = {}          # registered block -> its prefix (tuple of ids)
        self.block_of = {}        # prefix -> registered block
        self.evictable = []       # registered blocks with count 0, oldest first
        self.hit_blocks = 0
        self.lookup_blocks = 0

    # ---- allocation
    def _take(self):
        if self.free:
            b = self.free.pop(0)
        elif self.evictable:
            b = self.evictable.pop(0)
            del self.block_of[self.key_of.pop(b)]
        else:
            raise PoolExhausted("no free or evictable block")
        self.ref[b] = 1
        return b

    # ---- sequences
    def add_seq(self, sid):
        super().add_seq(sid)
        self.tokens[sid] = []

    def add_seq_prompt(self, sid, prompt):
        """Create ``sid`` and reuse the cached full blocks of ``prompt``; returns
        the number of prompt tokens whose K/V is already cached (the caller
        appends the rest with ``append_token``)."""
        prompt = [int(t) for t in prompt]
        self.add_seq(sid)
        bs = self.block_size
        for i in range(max(0, (len(prompt) - 1) // bs)):
            key = tuple(prompt[:bs * (i + 1)])
            self.lookup_blocks += 1
            b = self.block_of.get(key)
            if b is None:
                break
            self.hit_blocks += 1
            if self.ref[b] == 0:
                self.evictable.remove(b)
            self.ref[b] += 1
            self.tables[sid].append(b)
        n = len(self.tables[sid]) * bs
        self.lens[sid] = n
        self.tokens[sid] = prompt[:n]
        return n

    def _append(self, sid, token):
        slot, cow = super().append_slot(sid)
        self.tokens[sid].append(token)
        n = self.lens[sid]
        if n % self.block_size == 0:                     # the last block is now full
            key = tuple(self.tokens[sid])
            b = self.tables[sid][-1]
            if None not in key and key not in self.block_of:
                self.block_of[key] = b
                self.key_of[b] = key
        return slot, cow

    def append_slot(self, sid):
        """Append a token whose id is not known (its block is never shared)."""
        return self._append(sid, None)

    def append_token(self, sid, token):
        return self._append(sid, int(token))

    def fork(self, parent, child):
        super().fork(parent, child)
        self.tokens[child] = list(self.tokens[parent])

    def _release(self, table):
        cached = []
        for b in table:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                if b in self.key_of:
                    cached.append(b)
                else:
                    self.free.append(b)
        self.evictable.extend(reversed(cached))

    def _device_blocks_available(self):
        return len(self.free) + len(self.evictable)

    def free_seq(self, sid):
        super().free_seq(sid)
        del self.tokens[sid]

    def num_evictable(self):
        return len(self.evictable)

    def num_cached(self):
        return len(self.key_of)
