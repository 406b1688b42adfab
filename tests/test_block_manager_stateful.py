"""The library's block manager against the oracle's under stateful random
testing: hypothesis interleaves every operation (sequences added plain or from
a prompt, single and batch appends, forks, frees, beam steps, swaps out and
in), compares the whole state after each one, checks the prefix groups of
random batches exactly, and shrinks a failing script to a short one. Prefix
caching and the host pool are drawn per run.
"""
import copy

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, settings, strategies as st  # noqa: E402
from hypothesis.stateful import (RuleBasedStateMachine, initialize, invariant,  # noqa: E402
                                 precondition, rule)

from _groups import assert_groups_exact  # noqa: E402
from _lib import library, pkv  # noqa: E402
from oracle.block_manager import BlockManager as OracleBM, PoolExhausted  # noqa: E402
from oracle.prefix_cache import PrefixCachingBlockManager  # noqa: E402

TOKENS = st.integers(0, 2)          # few token ids, so prompts repeat and hit the cache


class Managers(RuleBasedStateMachine):
    @initialize(nb=st.integers(2, 20), bs=st.sampled_from([1, 2, 4]),
                host=st.integers(0, 10), caching=st.booleans(), seed=st.integers(0, 1 << 16))
    def start(self, nb, bs, host, caching, seed):
        library()
        order = [int(b) for b in np.random.default_rng(seed).permutation(nb)]
        self.bs, self.caching = bs, caching
        self.nat = pkv.BlockManager(nb, bs, order, prefix_caching=caching, num_host_blocks=host)
        cls = PrefixCachingBlockManager if caching else OracleBM
        self.ora = cls(nb, bs, order, num_cpu_blocks=host)
        self.live, self.nxt = [], 0

    # ---------------------------------------------------------------- helpers
    def resident(self):
        return [s for s in self.live if s not in self.ora.swapped]

    def new_id(self):
        self.nxt += 1
        return self.nxt - 1

    def appends(self, steps, call):
        """Run the oracle's appends one by one on a copy; all fit -> the library
        must return the same slots and pairs; one does not -> the library must
        refuse the whole call and change nothing."""
        trial = copy.deepcopy(self.ora)
        try:
            exp = [f(trial) for f in steps]
        except PoolExhausted:
            with pytest.raises(pkv.PagedKVError) as e:
                call()
            assert e.value.status == -5
            return
        slots, pairs = call()
        if slots is not None:
            assert [int(s) for s in slots] == [s for s, _ in exp]
        assert [tuple(map(int, p)) for p in pairs] == [c for _, c in exp if c is not None]
        self.ora = trial

    # ---------------------------------------------------------------- rules
    @rule()
    def add(self):
        sid = self.new_id()
        self.nat.add_seq(sid)
        self.ora.add_seq(sid)
        self.live.append(sid)

    @precondition(lambda self: self.caching)
    @rule(prompt=st.lists(TOKENS, max_size=12))
    def add_prompt(self, prompt):
        sid = self.new_id()
        assert self.nat.add_seq_prompt(sid, prompt) == self.ora.add_seq_prompt(sid, prompt)
        self.live.append(sid)

    @precondition(lambda self: self.resident())
    @rule(data=st.data())
    def append(self, data):
        sid = data.draw(st.sampled_from(self.resident()))
        k = data.draw(st.integers(1, 3 * self.bs))
        if self.caching and data.draw(st.booleans()):
            toks = data.draw(st.lists(TOKENS, min_size=k, max_size=k))
            self.appends([(lambda o, t=t: o.append_token(sid, t)) for t in toks],
                         lambda: self.nat.append_tokens(sid, toks))
        else:
            self.appends([(lambda o: o.append_slot(sid))] * k,
                         lambda: (None, np.asarray(self.nat.append_n(sid, k)).reshape(-1, 2)))

    @precondition(lambda self: self.resident())
    @rule(data=st.data())
    def batch_append(self, data):
        ids = data.draw(st.lists(st.sampled_from(self.resident()), min_size=1, max_size=8))
        self.appends([(lambda o, s=s: o.append_slot(s)) for s in ids],
                     lambda: self.nat.append_slots(ids))

    @precondition(lambda self: self.resident())
    @rule(data=st.data())
    def fork(self, data):
        parent = data.draw(st.sampled_from(self.resident()))
        child = self.new_id()
        self.nat.fork(parent, child)
        self.ora.fork(parent, child)
        self.live.append(child)

    @precondition(lambda self: self.live)
    @rule(data=st.data())
    def free(self, data):
        sid = data.draw(st.sampled_from(self.live))
        self.nat.free_seq(sid)
        self.ora.free_seq(sid)
        self.live.remove(sid)

    @precondition(lambda self: self.resident())
    @rule(data=st.data())
    def beam_step(self, data):
        old = data.draw(st.lists(st.sampled_from(self.resident()), min_size=1, max_size=4,
                                 unique=True))
        parents = data.draw(st.lists(st.integers(0, len(old) - 1), min_size=0, max_size=5))
        new = [self.new_id() for _ in parents]
        self.nat.beam_step(old, parents, new)
        self.ora.beam_step(old, parents, new)
        self.live = [s for s in self.live if s not in old] + new

    @precondition(lambda self: self.ora.num_cpu_blocks and self.resident())
    @rule(data=st.data())
    def swap_out(self, data):
        sid = data.draw(st.sampled_from(self.resident()))
        try:
            exp = self.ora.swap_out(sid)
        except PoolExhausted:
            with pytest.raises(pkv.PagedKVError) as e:
                self.nat.swap_out(sid)
            assert e.value.status == -5
            return
        assert [tuple(map(int, p)) for p in self.nat.swap_out(sid)] == [tuple(p) for p in exp]

    @precondition(lambda self: self.ora.swapped)
    @rule(data=st.data())
    def swap_in(self, data):
        sid = data.draw(st.sampled_from(sorted(self.ora.swapped)))
        try:
            exp = self.ora.swap_in(sid)
        except PoolExhausted:
            with pytest.raises(pkv.PagedKVError) as e:
                self.nat.swap_in(sid)
            assert e.value.status == -5
            return
        assert [tuple(map(int, p)) for p in self.nat.swap_in(sid)] == [tuple(p) for p in exp]

    @precondition(lambda self: self.resident())
    @rule(data=st.data())
    def prefix_groups(self, data):
        ids = data.draw(st.lists(st.sampled_from(self.resident()), min_size=1, max_size=10,
                                 unique=True))
        maxm = data.draw(st.integers(1, 8))
        assert_groups_exact(self.ora, ids, maxm, self.nat.prefix_groups(ids, maxm))

    # ---------------------------------------------------------------- state
    @invariant()
    def same_state(self):
        if not hasattr(self, "nat"):
            return
        nat, ora = self.nat, self.ora
        assert nat.free_list() == ora.free
        assert [nat.refcount(b) for b in range(ora.num_blocks)] == ora.ref
        assert nat.host_free_list() == ora.cpu_free
        for sid in self.live:
            assert nat.block_table(sid) == ora.block_table(sid)
            assert nat.seq_len(sid) == ora.seq_len(sid)
            assert nat.is_swapped(sid) == (sid in ora.swapped)
        if self.caching:
            assert nat.evictable_list() == ora.evictable
            assert nat.cache_stats() == (ora.hit_blocks, ora.lookup_blocks, ora.num_cached(),
                                         ora.num_evictable())


Managers.TestCase.settings = settings(max_examples=150, stateful_step_count=40, deadline=None,
                                      suppress_health_check=list(HealthCheck), derandomize=True)
test_managers_agree = Managers.TestCase
