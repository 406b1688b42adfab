"""The library's C++ block manager against the oracle's, operation by operation.

Host logic, bit-exact: slots, copy-on-write pairs, block tables, reference counts
and the free list must agree after every operation of seeded random scripts and of
the benchmark workloads' set-up scripts.
"""
import copy
import ctypes

import numpy as np
import pytest

from _groups import assert_groups_exact
from _lib import library, pkv
import pkv_workloads as wl
from oracle.block_manager import BlockManager as OracleBM, PoolExhausted


def same_state(a, o):
    assert a.free_list() == o.free
    for sid in o.tables:
        assert a.block_table(sid) == o.tables[sid]
        assert a.seq_len(sid) == o.lens[sid]
    assert [a.refcount(b) for b in range(o.num_blocks)] == o.ref


def test_random_scripts_match_oracle():
    library()
    rng = np.random.default_rng(7)
    for trial in range(25):
        nb, bs = int(rng.integers(4, 80)), int(rng.choice([1, 2, 4, 16, 32]))
        free = rng.permutation(nb)
        a = pkv.BlockManager(nb, bs, free)
        o = OracleBM(nb, bs, free)
        nxt = 0
        for _ in range(300):
            live = sorted(o.tables)
            op = int(rng.integers(0, 10))
            if op == 0 or not live:
                a.add_seq(nxt)
                o.add_seq(nxt)
                nxt += 1
            elif op == 1:
                p = int(rng.choice(live))
                a.fork(p, nxt)
                o.fork(p, nxt)
                nxt += 1
            elif op == 2:
                s = int(rng.choice(live))
                a.free_seq(s)
                o.free_seq(s)
            else:
                s = int(rng.choice(live))
                try:
                    exp = o.append_slot(s)
                except PoolExhausted:
                    with pytest.raises(pkv.PagedKVError) as e:
                        a.append_slot(s)
                    assert e.value.status == -5
                else:
                    assert a.append_slot(s) == exp
            same_state(a, o)


def test_batch_append_and_tables_match_oracle():
    library()
    a = pkv.BlockManager(40, 4, range(40))
    o = OracleBM(40, 4, range(40))
    for s in range(3):
        a.add_seq(s)
        o.add_seq(s)
    assert a.append_n(0, 9) == []
    for _ in range(9):
        o.append_slot(0)
    a.fork(0, 3)
    o.fork(0, 3)
    slots, pairs = a.append_slots([0, 3, 1, 2])
    exp = [o.append_slot(s) for s in (0, 3, 1, 2)]
    assert list(slots) == [e[0] for e in exp]
    assert [tuple(p) for p in pairs] == [e[1] for e in exp if e[1] is not None]
    tables, lens = a.build_tables([0, 3, 1, 2], 5)
    for i, s in enumerate((0, 3, 1, 2)):
        t = o.tables[s]
        assert list(tables[i, :len(t)]) == t and all(tables[i, len(t):] == -1)
        assert lens[i] == o.lens[s]


@pytest.mark.parametrize("name", ["tiny_fp32", "llama13b_mha_bf16", "gqa_chat_bf16",
                                  "shared_prefix_bf16", "shared_prefix_fork_bf16",
                                  "beam_search_bf16"])
def test_workload_setup_and_step_match_oracle(name):
    library()
    w = wl.CONFIGS[name]()
    a = pkv.BlockManager(w.NB, w.bs, w.free_order)
    o = OracleBM(w.NB, w.bs, w.free_order)
    for op in w.script:
        if op[0] == "add":
            a.add_seq(op[1])
            o.add_seq(op[1])
        elif op[0] == "fork":
            a.fork(op[1], op[2])
            o.fork(op[1], op[2])
        elif op[0] == "append":
            got = a.append_n(op[1], op[2])
            exp = [c for c in (o.append_slot(op[1])[1] for _ in range(op[2])) if c is not None]
            assert got == exp
        elif op[0] == "beam":
            a.beam_step(*op[1:])
            o.beam_step(*op[1:])
        else:
            raise AssertionError(f"unexpected op {op[0]}")
    slots, pairs = a.append_slots(w.step_seqs)
    exp = [o.append_slot(s) for s in w.step_seqs]
    assert list(slots) == [e[0] for e in exp]
    assert [tuple(p) for p in pairs] == [e[1] for e in exp if e[1] is not None]
    assert [o.lens[s] for s in w.step_seqs] == list(w.final_lens)
    same_state(a, o)
    if name == "shared_prefix_fork_bf16":
        assert len(pairs) == 64 * 3          # 3 of 4 writers copy; the last writes in place
    maxm = max(1, 8 // (w.Hq // w.Hkv))      # as the engine plans a step
    assert_groups_exact(o, list(w.step_seqs), maxm, a.prefix_groups(w.step_seqs, maxm))


def test_prefix_groups_share_full_leading_blocks():
    """bm_prefix_groups against the oracle's tables: members share the group's
    leading block ids, those blocks are full for every member, the prefix is
    maximal, no sequence is in two groups, group sizes respect max_members."""
    library()
    rng = np.random.default_rng(5)
    for trial in range(30):
        bs = int(rng.choice([1, 2, 4, 16]))
        nb = 400
        free = rng.permutation(nb)
        a = pkv.BlockManager(nb, bs, free)
        o = OracleBM(nb, bs, free)
        seqs = []
        for p in range(int(rng.integers(1, 4))):
            sid = len(seqs)
            for m in (a, o):
                m.add_seq(sid)
            n0 = int(rng.integers(0, 40))
            a.append_n(sid, n0)
            for _ in range(n0):
                o.append_slot(sid)
            seqs.append(sid)
            for c in range(int(rng.integers(0, 6))):
                cid = max(seqs) + 1
                a.fork(sid, cid)
                o.fork(sid, cid)
                k = int(rng.integers(0, 12))
                a.append_n(cid, k)
                for _ in range(k):
                    o.append_slot(cid)
                seqs.append(cid)
        ids = list(rng.permutation(seqs))
        maxm = int(rng.choice([2, 3, 4, 8]))
        members, prefix, seq_group, blocks = a.prefix_groups(ids, maxm)
        seen = set()
        for gi, (row, pre, nlist) in enumerate(zip(members, prefix, blocks)):
            ms = [int(m) for m in row if m >= 0]
            assert 2 <= len(ms) <= maxm and pre >= 1
            tabs = [o.tables[ids[m]] for m in ms]
            # the group's list: the shared blocks once, then every member's others
            assert nlist == pre + sum(len(t) - pre for t in tabs)
            full = min(o.lens[ids[m]] // bs for m in ms)
            assert pre <= full
            assert all(t[:pre] == tabs[0][:pre] for t in tabs)
            if pre < full:                               # maximal
                assert len({t[pre] for t in tabs}) > 1
            for m in ms:
                assert m not in seen and seq_group[m] == gi
                seen.add(m)
        assert all(seq_group[i] == -1 for i in range(len(ids)) if i not in seen)
        assert_groups_exact(o, ids, maxm, (members, prefix, seq_group, blocks))


# ---------------------------------------------------------------- prefix caching
from oracle.prefix_cache import PrefixCachingBlockManager  # noqa: E402

BlockManager = pkv.BlockManager


def _same_state(nat, ora, live):
    for sid in live:
        assert nat.block_table(sid) == ora.block_table(sid)
        assert nat.seq_len(sid) == ora.seq_len(sid)
    assert nat.free_list() == ora.free
    assert nat.evictable_list() == ora.evictable
    assert [nat.refcount(b) for b in range(ora.num_blocks)] == ora.ref
    h, l, c, e = nat.cache_stats()
    assert (h, l, c, e) == (ora.hit_blocks, ora.lookup_blocks, ora.num_cached(), ora.num_evictable())


@pytest.mark.parametrize("seed", range(12))
def test_prefix_caching_matches_oracle_operation_by_operation(seed):
    rng = np.random.default_rng(100 + seed)
    bs = int(rng.choice([2, 4, 16]))
    nb = int(rng.integers(20, 60))
    order = list(rng.permutation(nb))
    nat = BlockManager(nb, bs, order, prefix_caching=True)
    ora = PrefixCachingBlockManager(nb, bs, order)
    prompts = [list(rng.integers(0, 4, size=rng.integers(1, 6 * bs))) for _ in range(4)]
    live, nxt = [], 0
    for step in range(120):
        op = int(rng.integers(0, 5))
        try:
            if op == 0 or not live:
                p = prompts[rng.integers(len(prompts))] + list(rng.integers(0, 4, size=rng.integers(0, 2 * bs)))
                n_o = ora.add_seq_prompt(nxt, p)
                n_n = nat.add_seq_prompt(nxt, p)
                assert n_n == n_o
                live.append(nxt)
                rest = [int(t) for t in p[n_o:]]
                slots, pairs = nat.append_tokens(nxt, rest)
                exp = [ora.append_token(nxt, t) for t in rest]
                assert list(slots) == [s for s, _ in exp]
                assert [tuple(x) for x in pairs] == [c for _, c in exp if c is not None]
                nxt += 1
            elif op == 1:
                sid = live[rng.integers(len(live))]
                toks = [int(t) for t in rng.integers(0, 4, size=rng.integers(1, 2 * bs))]
                slots, pairs = nat.append_tokens(sid, toks)
                exp = [ora.append_token(sid, t) for t in toks]
                assert list(slots) == [s for s, _ in exp]
                assert [tuple(x) for x in pairs] == [c for _, c in exp if c is not None]
            elif op == 2:
                sid = live[rng.integers(len(live))]
                nat.fork(sid, nxt)
                ora.fork(sid, nxt)
                live.append(nxt)
                nxt += 1
            elif op == 3:
                sid = live[rng.integers(len(live))]
                assert nat.append_slot(sid) == ora.append_slot(sid)     # token id unknown
            else:
                sid = live.pop(rng.integers(len(live)))
                nat.free_seq(sid)
                ora.free_seq(sid)
        except (pkv.PagedKVError, PoolExhausted) as e:
            # both must run out at the same point
            assert isinstance(e, PoolExhausted) or e.status == -5
            break
        _same_state(nat, ora, live)


def test_prefix_caching_must_be_enabled_before_sequences_exist():
    bm = BlockManager(8, 4, range(8))
    bm.add_seq(0)
    assert bm._lib.bm_enable_prefix_caching(bm._h) == -1
    with pytest.raises(pkv.PagedKVError):
        bm.add_seq_prompt(1, [1, 2, 3])              # caching is off


@pytest.mark.parametrize("seed,caching", [(s, c) for s in range(6) for c in (False, True)])
def test_swapping_matches_oracle_operation_by_operation(seed, caching):
    rng = np.random.default_rng(300 + seed)
    bs = int(rng.choice([2, 4, 16]))
    nb, ncpu = int(rng.integers(20, 50)), int(rng.integers(5, 40))
    order = list(rng.permutation(nb))
    nat = BlockManager(nb, bs, order, prefix_caching=caching, num_host_blocks=ncpu)
    ora = PrefixCachingBlockManager(nb, bs, order, ncpu)
    live, nxt = [], 0
    for step in range(150):
        op = int(rng.integers(0, 6))
        resident = [s for s in live if s not in ora.swapped]
        try:
            if op == 0 or not live:
                p = [int(t) for t in rng.integers(0, 3, size=rng.integers(1, 5 * bs))]
                if not caching:
                    n_o = 0
                    ora.add_seq(nxt)
                    nat.add_seq(nxt)
                    toks = [t + 10 * (nxt + 1) for t in p]
                else:
                    n_o = ora.add_seq_prompt(nxt, p)
                    assert nat.add_seq_prompt(nxt, p) == n_o
                    toks = p[n_o:]
                sid = nxt
                nxt += 1
                live.append(sid)
                slots, pairs = nat.append_tokens(sid, toks) if caching else (
                    np.array([nat.append_slot(sid)[0] for _ in toks]), None)
                exp = [ora.append_token(sid, t) if caching else ora.append_slot(sid) for t in toks]
                assert list(slots) == [s for s, _ in exp]
            elif op == 1 and resident:
                sid = resident[rng.integers(len(resident))]
                assert nat.append_slot(sid) == ora.append_slot(sid)
            elif op == 2 and resident:
                sid = resident[rng.integers(len(resident))]
                nat.fork(sid, nxt)
                ora.fork(sid, nxt)
                live.append(nxt)
                nxt += 1
            elif op == 3 and resident:
                sid = resident[rng.integers(len(resident))]
                try:
                    exp = ora.swap_out(sid)
                except PoolExhausted:
                    with pytest.raises(pkv.PagedKVError) as e:
                        nat.swap_out(sid)
                    assert e.value.status == -5
                    continue
                assert [tuple(x) for x in nat.swap_out(sid)] == exp
                assert nat.is_swapped(sid)
            elif op == 4 and ora.swapped:
                sid = sorted(ora.swapped)[rng.integers(len(ora.swapped))]
                try:
                    exp = ora.swap_in(sid)
                except PoolExhausted:
                    with pytest.raises(pkv.PagedKVError) as e:
                        nat.swap_in(sid)
                    assert e.value.status == -5
                    continue
                assert [tuple(x) for x in nat.swap_in(sid)] == exp
            elif op == 5:
                sid = live.pop(rng.integers(len(live)))
                nat.free_seq(sid)
                ora.free_seq(sid)
        except (PoolExhausted, pkv.PagedKVError) as e:
            assert isinstance(e, PoolExhausted) or e.status == -5
            break                                      # the device pool ran out
        for sid in live:
            assert nat.block_table(sid) == ora.block_table(sid)
            assert nat.is_swapped(sid) == (sid in ora.swapped)
        assert nat.free_list() == ora.free
        assert nat.host_free_list() == ora.cpu_free
        assert [nat.refcount(b) for b in range(nb)] == ora.ref
        if caching:
            assert nat.evictable_list() == ora.evictable


@pytest.mark.parametrize("seed", range(6))
def test_beam_steps_match_oracle(seed):
    """Requests of W beams reshuffled by seeded random parents every step, one
    append per beam, interleaved with whole-request frees and new requests."""
    library()
    rng = np.random.default_rng(100 + seed)
    nb, bs, W = 1200, int(rng.choice([2, 4, 16])), int(rng.choice([2, 3, 4, 8]))
    free = rng.permutation(nb)
    a, o = pkv.BlockManager(nb, bs, free), OracleBM(nb, bs, free)
    nxt, reqs = 0, []
    for step in range(120):
        if len(reqs) < 3 or rng.random() < 0.05:
            P = int(rng.integers(1, 40))
            a.add_seq(nxt)
            o.add_seq(nxt)
            assert a.append_n(nxt, P) == []
            for _ in range(P):
                o.append_slot(nxt)
            reqs.append([nxt])
            nxt += 1
        if rng.random() < 0.03 and len(reqs) > 1:
            for s in reqs.pop(int(rng.integers(len(reqs)))):
                a.free_seq(s)
                o.free_seq(s)
        for r, beams in enumerate(reqs):
            parents = rng.integers(0, len(beams), size=W).tolist()
            new = list(range(nxt, nxt + W))
            nxt += W
            a.beam_step(beams, parents, new)
            o.beam_step(beams, parents, new)
            reqs[r] = new
            try:
                exp = [o.append_slot(s) for s in new]
            except PoolExhausted:
                assert step > 30                        # the script ran long enough
                return                                  # pool full: the script ends here
            slots, pairs = a.append_slots(new)
            assert list(slots) == [s for s, _ in exp]
            assert [tuple(p) for p in pairs] == [c for _, c in exp if c is not None]
        same_state(a, o)


def test_beam_step_refusals_change_nothing():
    library()
    a = pkv.BlockManager(16, 4, range(16))
    a.add_seq(0)
    a.append_n(0, 6)
    a.beam_step([0], [0, 0], [1, 2])
    before = (a.free_list(), a.block_table(1), a.block_table(2))
    for old, par, new, st in (([1, 2], [0, 2], [3, 4], -4),      # parent out of range
                              ([1, 9], [0, 1], [3, 4], -4),      # unknown old beam
                              ([1, 2], [0, 1], [3, 3], -1),      # repeated new id
                              ([1, 2], [0, 1], [2, 4], -1),      # new id in use
                              ([1, 1], [0, 1], [3, 4], -1)):     # repeated old beam
        with pytest.raises(pkv.PagedKVError) as e:
            a.beam_step(old, par, new)
        assert e.value.status == st
        assert (a.free_list(), a.block_table(1), a.block_table(2)) == before
    with pytest.raises(ValueError):
        a.beam_step([1, 2], [0], [3, 4])


@pytest.mark.parametrize("seed", range(6))
def test_beam_steps_with_prefix_caching_match_oracle(seed):
    """Beam search on a caching manager: requests that share a prompt prefix
    (cached full blocks reused), beams reshuffled every step (forks carry their
    token history, freed beams' registered blocks become evictable), one token
    id appended per beam, requests finishing and new ones reviving cached
    blocks. The library's manager and the oracle's agree after every operation."""
    rng = np.random.default_rng(300 + seed)
    bs = int(rng.choice([2, 4, 16]))
    nb = int(rng.integers(60, 160))
    W = int(rng.choice([2, 3, 4]))
    order = list(rng.permutation(nb))
    nat = BlockManager(nb, bs, order, prefix_caching=True)
    ora = PrefixCachingBlockManager(nb, bs, order)
    system = [int(t) for t in rng.integers(0, 5, size=int(rng.integers(1, 4 * bs)))]
    reqs, nxt = [], 0
    try:
        for step in range(60):
            if len(reqs) < 2 or rng.random() < 0.1:
                p = system + [int(t) for t in rng.integers(0, 5, size=int(rng.integers(1, 2 * bs)))]
                n_o = ora.add_seq_prompt(nxt, p)
                assert nat.add_seq_prompt(nxt, p) == n_o
                rest = p[n_o:]
                slots, pairs = nat.append_tokens(nxt, rest)
                exp = [ora.append_token(nxt, t) for t in rest]
                assert list(slots) == [s for s, _ in exp]
                assert [tuple(x) for x in pairs] == [c for _, c in exp if c is not None]
                reqs.append([nxt])
                nxt += 1
            if rng.random() < 0.08 and len(reqs) > 1:
                for s in reqs.pop(int(rng.integers(len(reqs)))):
                    nat.free_seq(s)
                    ora.free_seq(s)
            old = [s for b in reqs for s in b]
            parents, new, base = [], [], 0
            for b in reqs:
                parents += [base + int(x) for x in rng.integers(0, len(b), size=W)]
                base += len(b)
            new = list(range(nxt, nxt + len(parents)))
            nxt += len(parents)
            nat.beam_step(old, parents, new)
            ora.beam_step(old, parents, new)
            reqs = [new[i:i + W] for i in range(0, len(new), W)]
            for s in new:
                t = int(rng.integers(0, 5))
                slots, pairs = nat.append_tokens(s, [t])
                slot, cow = ora.append_token(s, t)
                assert list(slots) == [slot]
                assert [tuple(x) for x in pairs] == ([cow] if cow is not None else [])
            _same_state(nat, ora, new)
    except (pkv.PagedKVError, PoolExhausted) as e:
        assert isinstance(e, PoolExhausted) or e.status == -5
        assert step > 10                                 # the script ran long enough


# ---------------------------------------------------------------- batch appends: all or nothing
def _snapshot(nat, ids):
    return (nat.free_list(), [nat.refcount(b) for b in range(nat.num_blocks)],
            {s: (nat.block_table(s), nat.seq_len(s)) for s in ids})


def test_batch_append_counts_a_shared_block_copied_once():
    """Two tables share a partial last block and one block is free: the first
    append copies it, which leaves the second table its only owner, so the batch
    needs one block and fits. A batch that needs one more block is refused whole."""
    library()
    nat = BlockManager(2, 4, [0, 1])
    ora = OracleBM(2, 4, [0, 1])
    for bm in (nat, ora):
        bm.add_seq(0)
    assert nat.append_n(0, 2) == []
    ora.append_slot(0), ora.append_slot(0)
    nat.fork(0, 1)
    ora.fork(0, 1)
    slots, pairs = nat.append_slots([0, 1])
    exp = [ora.append_slot(0), ora.append_slot(1)]
    assert list(slots) == [s for s, _ in exp] and [tuple(p) for p in pairs] == [(0, 1)]
    same_state(nat, ora)
    assert nat.free_list() == []
    nat.append_slots([0])
    ora.append_slot(0)
    before = _snapshot(nat, [0, 1])
    with pytest.raises(pkv.PagedKVError) as e:    # seq 1: one slot in place, then a new block
        nat.append_slots([1, 1])
    assert e.value.status == -5
    assert _snapshot(nat, [0, 1]) == before
    with pytest.raises(pkv.PagedKVError) as e:
        nat.append_n(1, 2)
    assert e.value.status == -5
    assert _snapshot(nat, [0, 1]) == before
    assert nat.append_n(1, 1) == []                  # the in-place slot alone fits
    ora.append_slot(1)
    same_state(nat, ora)


def test_append_with_too_small_cow_capacity_changes_nothing():
    lib = library()
    nat = BlockManager(4, 4, range(4))
    nat.add_seq(0)
    nat.append_n(0, 1)
    nat.fork(0, 1)
    before = _snapshot(nat, [0, 1])
    buf = np.zeros((2, 2), dtype=np.int64)
    cnt = ctypes.c_int(7)
    st = lib.bm_append_n(nat._h, 1, 3, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), 0,
                         ctypes.byref(cnt))
    assert st == -1 and cnt.value == 0             # PKV_ERR_INVALID_ARG
    assert _snapshot(nat, [0, 1]) == before
    st = lib.bm_append_n(nat._h, 1, 3, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), 1,
                         ctypes.byref(cnt))
    assert st == 0 and cnt.value == 1 and tuple(buf[0]) == (0, 1)


@pytest.mark.parametrize("caching", [False, True])
@pytest.mark.parametrize("seed", range(8))
def test_batch_appends_are_all_or_nothing_against_oracle(seed, caching):
    """Seeded scripts of forks, frees and batch appends (ids repeated in runs, as
    a chunked-prefill step lists them) on small pools. The oracle applies each
    batch one append at a time; where it runs out part-way, the library must
    refuse the whole batch and keep its state; otherwise slots, pairs and state
    must match."""
    rng = np.random.default_rng(900 + seed)
    bs = int(rng.choice([1, 2, 4, 16]))
    nb = int(rng.integers(6, 40))
    order = list(rng.permutation(nb))
    nat = BlockManager(nb, bs, order, prefix_caching=caching)
    ora = (PrefixCachingBlockManager if caching else OracleBM)(nb, bs, order)
    live, nxt = [], 0
    refused = done = cows = 0
    for _ in range(250):
        op = int(rng.integers(0, 6))
        if op == 0 or not live:
            nat.add_seq(nxt)
            ora.add_seq(nxt)
            live.append(nxt)
            nxt += 1
            continue
        if op == 1:
            sid = live[rng.integers(len(live))]
            nat.fork(sid, nxt)
            ora.fork(sid, nxt)
            live.append(nxt)
            nxt += 1
            continue
        if op == 2 and len(live) > 1:
            sid = live.pop(rng.integers(len(live)))
            nat.free_seq(sid)
            ora.free_seq(sid)
            continue
        snap = copy.deepcopy(ora)
        if op == 3:                                    # one sequence, k tokens with ids
            sid = live[rng.integers(len(live))]
            toks = [int(t) for t in rng.integers(0, 3, size=int(rng.integers(1, 3 * bs + 2)))]
            if caching:
                call = lambda: nat.append_tokens(sid, toks)
                step = [(lambda t=t: ora.append_token(sid, t)) for t in toks]
            else:
                call = lambda: (None, nat.append_n(sid, len(toks)))
                step = [(lambda: ora.append_slot(sid)) for _ in toks]
        else:                                          # a batch with runs of repeated ids
            k = int(rng.integers(1, len(live) + 1))
            pick = rng.choice(live, size=k, replace=False)
            ids = np.repeat(pick, rng.integers(1, bs + 2, size=k)).astype(np.int64)
            call = lambda: nat.append_slots(ids)
            step = [(lambda s=int(s): ora.append_slot(s)) for s in ids]
        try:
            exp = [f() for f in step]
        except PoolExhausted:
            ora = snap
            before = _snapshot(nat, live)
            with pytest.raises(pkv.PagedKVError) as e:
                call()
            assert e.value.status == -5
            assert _snapshot(nat, live) == before
            refused += 1
        else:
            slots, pairs = call()
            if slots is not None:
                assert list(slots) == [s for s, _ in exp]
            assert [tuple(map(int, p)) for p in pairs] == [c for _, c in exp if c is not None]
            done += 1
            cows += len(pairs)
        assert nat.free_list() == ora.free
        assert [nat.refcount(b) for b in range(nb)] == ora.ref
        for sid in live:
            assert nat.block_table(sid) == ora.block_table(sid)
            assert nat.seq_len(sid) == ora.seq_len(sid)
        if caching:
            assert nat.evictable_list() == ora.evictable
    assert refused > 0 and done > 0 and cows > 0


def test_swap_in_takes_evictable_blocks_when_the_free_list_is_short():
    """With prefix caching, cached blocks nobody holds count as available: a
    swap-in with an empty free list evicts them (oldest first), as the oracle
    does."""
    library()
    nat = BlockManager(6, 4, range(6), prefix_caching=True, num_host_blocks=4)
    ora = PrefixCachingBlockManager(6, 4, list(range(6)), num_cpu_blocks=4)
    prompt = list(range(12))                           # three full blocks, ids known
    for m in (nat, ora):
        assert m.add_seq_prompt(0, prompt) == 0
    nat.append_tokens(0, prompt)
    for t in prompt:
        ora.append_token(0, t)
    for m in (nat, ora):
        m.add_seq(1)
    nat.append_n(1, 8)
    for _ in range(8):
        ora.append_slot(1)
    assert [tuple(p) for p in nat.swap_out(1)] == [tuple(p) for p in ora.swap_out(1)]
    for m in (nat, ora):
        m.free_seq(0)                                  # its three blocks become evictable
        m.add_seq(2)
    nat.append_n(2, 12)
    for _ in range(12):
        ora.append_slot(2)
    assert nat.free_list() == ora.free == [] and len(ora.evictable) == 3
    assert [tuple(p) for p in nat.swap_in(1)] == [tuple(p) for p in ora.swap_in(1)]
    _same_state(nat, ora, [1, 2])


@pytest.mark.parametrize("name", ["shared_prefix_fork_bf16", "beam_search_bf16", "gqa_chat_bf16"])
def test_plan_into_buffers_matches_the_array_calls(name):
    """BlockManager.plan_decode_into (bm_plan_decode: the allocation-free host
    half of a step that engine.LiveDecodePipeline writes into its pinned slab)
    gives the slots, copy-on-write pairs, tables, lengths and prefix groups of
    append_slots, build_tables and prefix_groups on an identical manager, plus
    the batch indices in no group and the longest group list, step after step;
    a refused step changes nothing."""
    w = wl.CONFIGS[name]()
    a = pkv.BlockManager(w.NB, w.bs, w.free_order)
    b = pkv.BlockManager(w.NB, w.bs, w.free_order)
    for bm in (a, b):
        for op in w.script:
            if op[0] == "add":
                bm.add_seq(op[1])
            elif op[0] == "append":
                bm.append_n(op[1], op[2])
            elif op[0] == "fork":
                bm.fork(op[1], op[2])
            else:
                bm.beam_step(op[1], op[2], op[3])
    ids = np.ascontiguousarray(np.asarray(w.step_seqs, dtype=np.int64))
    n, mb, mm = len(ids), w.max_blocks_per_seq + 3, max(1, 8 // (w.Hq // w.Hkv))
    slots = np.zeros(n, np.int64)
    pairs = np.zeros((n, 2), np.int64)
    tables = np.zeros((n, mb), np.int32)
    lens = np.zeros(n, np.int32)
    members = np.zeros((n, mm), np.int32)
    prefix = np.zeros(n, np.int32)
    seq_group = np.zeros(n, np.int32)
    blocks = np.zeros(n, np.int32)
    ungrouped = np.zeros(n, np.int32)
    p64 = lambda x: x.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    p32 = lambda x: x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    groups = (mm, p32(members), p32(prefix), p32(seq_group), p32(blocks), p32(ungrouped))
    for step in range(20):
        np_, ng, nu, mgb = a.plan_decode_into(p64(ids), n, mb, p64(slots), p64(pairs),
                                              p32(tables), p32(lens), groups)
        s2, pr2 = b.append_slots(ids)
        t2, l2 = b.build_tables(ids, mb)
        m2, pf2, sg2, bl2 = b.prefix_groups(ids, mm)
        assert np.array_equal(slots, s2) and np.array_equal(pairs[:np_], pr2)
        assert np.array_equal(tables, t2) and np.array_equal(lens, l2)
        assert ng == len(m2) and np.array_equal(members[:ng], m2)
        assert np.array_equal(prefix[:ng], pf2) and np.array_equal(seq_group, sg2)
        assert np.array_equal(blocks[:ng], bl2)
        assert np.array_equal(ungrouped[:nu], np.flatnonzero(sg2 < 0))
        assert mgb == (int(bl2.max()) if ng else 0)
        if name == "shared_prefix_fork_bf16" and step == 0:
            assert np_ == 192 and ng > 0
    # without groups: the plain half of the step
    np_, ng, nu, mgb = a.plan_decode_into(p64(ids), n, mb, p64(slots), p64(pairs), p32(tables),
                                          p32(lens))
    b.append_slots(ids)
    t2, l2 = b.build_tables(ids, mb)
    assert (ng, nu, mgb) == (0, 0, 0) and np.array_equal(tables, t2) and np.array_equal(lens, l2)
    # refusals change nothing: tables that would outgrow max_blocks, a pool that
    # cannot hold the appends
    free = a.free_list()
    lens_before = [a.seq_len(int(s)) for s in ids]
    with pytest.raises(pkv.PagedKVError) as e:
        a.plan_decode_into(p64(ids), n, 1, p64(slots), p64(pairs), p32(tables), p32(lens))
    assert e.value.status == -1
    assert np.array_equal(a.free_list(), free)
    assert [a.seq_len(int(s)) for s in ids] == lens_before
    small = pkv.BlockManager(2, w.bs, np.arange(2))
    small.add_seq(0)
    small.append_n(0, 2 * w.bs)
    one = np.array([0], dtype=np.int64)
    with pytest.raises(pkv.PagedKVError) as e:
        small.plan_decode_into(p64(one), 1, 4, p64(slots), p64(pairs), p32(tables), p32(lens))
    assert e.value.status == pkv.PKV_ERR_POOL_EXHAUSTED and small.seq_len(0) == 2 * w.bs
