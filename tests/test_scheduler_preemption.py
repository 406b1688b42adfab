"""Planning a decode step when the pool runs out ("KV cache paginado e batching
contínuo para LLMs", "Como funciona": the newest requests are preempted, all or
nothing, and their blocks recovered by swapping or recomputation).

``PagedKVCache.plan_step_preempting`` is host logic over the library's block
manager: the pools sit in host memory here and no kernel runs. Each case is
checked against the oracle's manager driven by the same rule one append at a
time: run the step's appends in order; if the pool runs out, undo them, free
the newest request and try again.
"""
import copy

import numpy as np
import pytest
import torch

from _lib import library, pkv
from oracle.block_manager import BlockManager as OracleBM, PoolExhausted
from paged_kv_cache_259_gb300.engine import PagedKVCache


def host_cache(nb, bs, order, prefix_caching=False):
    library()
    return PagedKVCache(nb, 4, 4, 16, bs, torch.bfloat16, order, device="cpu",
                        prefix_caching=prefix_caching)


def oracle_step(ora, requests):
    """The rule on the oracle: returns (state after the step, slots, pairs, the
    preempted requests newest first)."""
    reqs = [list(r) for r in requests]
    gone = []
    while reqs:
        trial = copy.deepcopy(ora)
        try:
            got = [trial.append_slot(s) for r in reqs for s in r]
        except PoolExhausted:
            r = reqs.pop()
            gone.append(r)
            for s in r:
                ora.free_seq(s)
            continue
        return trial, [s for s, _ in got], [c for _, c in got if c is not None], gone
    return ora, [], [], gone


def check_same(cache, ora, live):
    bm = cache.bm
    assert bm.free_list() == ora.free
    assert [bm.refcount(b) for b in range(ora.num_blocks)] == ora.ref
    for s in live:
        assert bm.block_table(s) == ora.block_table(s)
        assert bm.seq_len(s) == ora.seq_len(s)


def test_newest_requests_go_first_and_whole():
    bs, nb = 8, 5
    cache = host_cache(nb, bs, range(nb))
    ora = OracleBM(nb, bs, range(nb))
    # request 0: one sequence of 16 tokens; request 1: two samples forked after
    # 12 tokens (they share a partial block); request 2: one sequence of 8 tokens
    for sid, n in ((0, 16), (1, 12), (3, 8)):
        cache.bm.add_seq(sid)
        ora.add_seq(sid)
        cache.bm.append_n(sid, n)
        for _ in range(n):
            ora.append_slot(sid)
    cache.bm.fork(1, 2)
    ora.fork(1, 2)
    assert cache.bm.free_list() == []                # 2 + 2 + 1 blocks held
    requests = [0, [1, 2], 3]                        # needs 1 + 1 (CoW) + 1 blocks
    seen = []
    plan, gone = cache.plan_step_preempting(
        requests, lambda ids: seen.append(list(ids)) or cache.preempt_by_recompute(ids))
    ora, slots, pairs, gone_o = oracle_step(ora, [[0], [1, 2], [3]])
    assert seen == gone_o == [[3], [1, 2]]
    assert gone == [{3: 8}, {1: 12, 2: 12}]
    assert list(plan.seq_ids) == [0]
    assert list(plan.slots) == slots and [tuple(p) for p in plan.pairs] == pairs
    check_same(cache, ora, [0])


def test_a_step_that_fits_preempts_nothing():
    cache = host_cache(8, 8, range(8))
    for sid in range(3):
        cache.bm.add_seq(sid)
    plan, gone = cache.plan_step_preempting([0, 1, 2], lambda ids: pytest.fail("preempted"))
    assert gone == [] and list(plan.seq_ids) == [0, 1, 2]


def test_when_nothing_fits_every_request_is_preempted():
    cache = host_cache(2, 8, [0, 1])
    cache.bm.add_seq(0)
    cache.bm.append_n(0, 16)                         # both blocks full
    plan, gone = cache.plan_step_preempting([0], cache.preempt_by_recompute)
    assert plan is None and gone == [{0: 16}]
    assert sorted(cache.bm.free_list()) == [0, 1]


def test_other_errors_are_not_preemption():
    cache = host_cache(4, 8, range(4))
    cache.bm.add_seq(0)
    with pytest.raises(pkv.PagedKVError) as e:
        cache.plan_step_preempting([0, 9], lambda ids: pytest.fail("preempted"))
    assert e.value.status == -4                      # unknown sequence
    assert cache.bm.seq_len(0) == 0


@pytest.mark.parametrize("seed", range(10))
def test_random_steps_match_the_oracle(seed):
    rng = np.random.default_rng(1300 + seed)
    bs = int(rng.choice([8, 16, 32]))
    nb = int(rng.integers(8, 40))
    order = list(rng.permutation(nb))
    cache = host_cache(nb, bs, order)
    ora = OracleBM(nb, bs, order)
    requests, nxt, preemptions = [], 0, 0
    for _ in range(60):
        if not requests or rng.random() < 0.3:       # a new request of 1-3 samples
            width = int(rng.integers(1, 4))
            cache.bm.add_seq(nxt)
            ora.add_seq(nxt)
            prompt = int(rng.integers(0, 2 * bs))
            try:
                for _ in range(prompt):
                    ora.append_slot(nxt)
            except PoolExhausted:
                ora.free_seq(nxt)
                cache.bm.free_seq(nxt)
                nxt += 1
                continue
            cache.bm.append_n(nxt, prompt)
            group = [nxt]
            for k in range(1, width):
                cache.bm.fork(nxt, nxt + k)
                ora.fork(nxt, nxt + k)
                group.append(nxt + k)
            requests.append(group)
            nxt += width
        plan, gone = cache.plan_step_preempting(requests, cache.preempt_by_recompute)
        ora, slots, pairs, gone_o = oracle_step(ora, requests)
        assert [sorted(g) for g in gone] == [sorted(r) for r in gone_o]
        requests = requests[:len(requests) - len(gone)]
        preemptions += len(gone)
        if plan is None:
            assert requests == [] and slots == []
        else:
            assert list(plan.slots) == slots
            assert [tuple(map(int, p)) for p in plan.pairs] == pairs
        check_same(cache, ora, [s for r in requests for s in r])
        if rng.random() < 0.1 and requests:          # a request finishes
            for s in requests.pop(int(rng.integers(len(requests)))):
                cache.bm.free_seq(s)
                ora.free_seq(s)
    assert preemptions > 0


def test_resume_that_does_not_fit_adds_nothing():
    cache = host_cache(4, 8, range(4))
    bm = cache.bm
    bm.add_seq(0)
    bm.append_n(0, 20)                               # 3 blocks
    lens = cache.preempt_by_recompute([0])
    bm.add_seq(1)
    bm.append_n(1, 9)                                # 2 blocks: 2 left, 0 needs 3
    free = bm.free_list()
    with pytest.raises(pkv.PagedKVError) as e:
        cache.plan_resume([0], lens)
    assert e.value.status == -5
    with pytest.raises(pkv.PagedKVError) as e:
        bm.seq_len(0)
    assert e.value.status == -4                      # still preempted
    assert bm.free_list() == free
    bm.free_seq(1)
    plan = cache.plan_resume([0], lens)
    assert list(plan.chunks) == [20] and bm.seq_len(0) == 20


def test_prompts_that_do_not_fit_are_freed_again():
    bs = 8
    cache = host_cache(6, bs, range(6), prefix_caching=True)
    bm = cache.bm
    system = list(range(100, 100 + 2 * bs))          # two full blocks
    cache.plan_prompts([0], [system + [1]])
    bm.free_seq(0)                                   # its full blocks stay cached
    assert bm.cache_stats()[2:] == (2, 2)
    before = (bm.free_list(), bm.evictable_list())
    with pytest.raises(pkv.PagedKVError) as e:       # 1 reuses both; 2 needs 5 of 4 left
        cache.plan_prompts([1, 2], [system + [2], list(range(200, 200 + 5 * bs))])
    assert e.value.status == -5
    for sid in (1, 2):
        with pytest.raises(pkv.PagedKVError):
            bm.seq_len(sid)
    assert [bm.refcount(b) for b in range(6)] == [0] * 6
    free, evictable = bm.free_list(), bm.evictable_list()
    assert sorted(free + evictable) == sorted(before[0] + before[1])
    assert sorted(evictable) == sorted(before[1])    # the system prompt is still cached
    plan = cache.plan_prompts([3], [system + [3]])
    assert list(plan.cached) == [2 * bs]


def test_empty_batches_plan_to_empty_steps():
    """An empty step plans to empty arrays (the library returns at once for zero
    sequences, tokens or pairs)."""
    cache = host_cache(4, 8, range(4), prefix_caching=True)
    plan = cache.plan_step([])
    assert plan.slots.shape == (0,) and plan.pairs.shape == (0, 2)
    assert plan.tables.shape == (0, 1) and plan.lens.shape == (0,) and plan.num_groups == 0
    pre = cache.plan_prefill([], [])
    assert pre.slots.shape == (0,) and list(pre.query_start) == [0] and pre.max_query_len == 0
    prompts = cache.plan_prompts([], [])
    assert prompts.slots.shape == (0,) and list(prompts.query_start) == [0]
    plan, gone = cache.plan_step_preempting([], lambda ids: pytest.fail("preempted"))
    assert plan is None and gone == []
    assert cache.bm.free_list() == [0, 1, 2, 3]
