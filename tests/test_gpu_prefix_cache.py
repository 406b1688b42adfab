"""GPU parity of prefill with prefix caching: requests that begin with a served
system prompt reuse its cached blocks and compute only the rest of their
prompts (chunked-prefill attention over the whole cached sequence).

The library's block manager (prefix caching on) and the oracle's
(`oracle.prefix_cache`) replay the same requests; cached token counts, slots,
tables and the pools after the slot writes are compared bit-exactly, the
attention outputs within |gpu - oracle| <= 2e-2 + 2e-2 |oracle|.
"""
import numpy as np
import pytest
import torch

import pkv_workloads as wl
from _lib import library, pkv
from _parity import assert_close, stored_bits
from paged_kv_cache_259_gb300.engine import PagedKVCache

from oracle import attention as oatt
from oracle import cache_ops as oops
from oracle.prefix_cache import PrefixCachingBlockManager

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_and_library():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    library()
    torch.cuda.set_device(0)


def phase_rows(w, phase, prompts, cached):
    """q, k, v of the computed (uncached) positions of each request, in order."""
    rows = [w.rows(phase, b, int(n), len(p)) for b, (p, n) in enumerate(zip(prompts, cached))]
    return tuple(torch.cat([r[i] for r in rows]) for i in range(3))


def run_gpu(w, warm_ids, step_ids):
    cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, torch.bfloat16, w.free_order, "cuda",
                         prefix_caching=True)
    k0, v0 = w.past_pools()
    cache.load(k0, v0)
    outs, plans = [], []
    for phase, ids, prompts in (("warm", warm_ids, w.warm), ("step", step_ids, w.prompts)):
        plan = cache.plan_prompts(ids, prompts, max_blocks=w.max_blocks_per_seq)
        q, k, v = phase_rows(w, phase, prompts, plan.cached)
        dev = plan.device_tensors("cuda")
        out = torch.full((int(plan.chunks.sum()), w.Hq, w.D), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        cache.prefill_step(q.cuda(), k.cuda(), v.cuda(), dev, out, w.scale, plan.max_query_len)
        outs.append(out.float().cpu())
        plans.append(plan)
        if phase == "warm":
            for sid in ids:
                cache.bm.free_seq(int(sid))            # its blocks stay cached, evictable
    return outs, plans, cache, pkv.get_device_error()


def run_oracle(w, warm_ids, step_ids, units=None):
    """``units``: None (every output row) or {phase: [(row, head), ...]}; then each
    phase's output is a dict of the sampled rows."""
    bm = PrefixCachingBlockManager(w.NB, w.bs, w.free_order)
    kp, vp = w.past_pools()
    outs, info = [], []
    for phase, ids, prompts in (("warm", warm_ids, w.warm), ("step", step_ids, w.prompts)):
        cached, slots, pairs = [], [], []
        for sid, p in zip(ids, prompts):
            n = bm.add_seq_prompt(sid, p)
            cached.append(n)
            for t in p[n:]:
                s, c = bm.append_token(sid, int(t))
                slots.append(s)
                if c is not None:
                    pairs.append(c)
        q, k, v = phase_rows(w, phase, prompts, cached)
        oops.copy_blocks(kp, vp, pairs)
        oops.reshape_and_cache(k, v, kp, vp, torch.tensor(slots, dtype=torch.int64), w.bs)
        tables = np.full((len(ids), w.max_blocks_per_seq), -1, dtype=np.int64)
        for i, sid in enumerate(ids):
            t = bm.block_table(sid)
            tables[i, :len(t)] = t
        lens = np.array([bm.seq_len(sid) for sid in ids])
        chunks = [len(p) - n for p, n in zip(prompts, cached)]
        qs = np.concatenate([[0], np.cumsum(chunks)])
        outs.append(oatt.paged_prefill(q, kp, vp, tables, lens, qs, w.scale, w.bs,
                                       units=None if units is None else units[phase]))
        info.append({"cached": cached, "slots": slots, "pairs": pairs, "tables": tables,
                     "lens": lens})
        if phase == "warm":
            for sid in ids:
                bm.free_seq(sid)
    return outs, info, kp, vp, bm


@pytest.mark.parametrize("system,bs,Hq,Hkv", [(40, 16, 8, 2), (64, 16, 8, 8), (70, 32, 16, 2)])
def test_system_prompt_prefix_cache_parity(system, bs, Hq, Hkv):
    w = wl.system_prompt(B=5, system=system, suffix=0, suffix_lens=[0, 1, 9, 30, 100], Hq=Hq,
                         Hkv=Hkv, D=128, bs=bs, seed=system + bs, vocab=50,
                         name="system_prompt_small")
    warm_ids, step_ids = [100], list(range(w.B))
    g_out, g_plans, cache, err = run_gpu(w, warm_ids, step_ids)
    o_out, o_info, kp, vp, obm = run_oracle(w, warm_ids, step_ids)
    assert err == 0
    for gp, oi in zip(g_plans, o_info):
        assert list(gp.cached) == oi["cached"]
        assert list(gp.slots) == oi["slots"]
        assert [tuple(x) for x in gp.pairs] == oi["pairs"]
        assert np.array_equal(gp.tables.astype(np.int64), oi["tables"])
        assert np.array_equal(gp.lens, oi["lens"])
    # every request of the step reused the system prompt's full blocks (at least
    # one prompt token is always left to compute)
    full = system // bs
    assert [min(full, (len(p) - 1) // bs) * bs for p in w.prompts] == o_info[1]["cached"]
    assert sum(o_info[1]["cached"]) > 0
    h, l, c, e = cache.bm.cache_stats()
    assert (h, l) == (obm.hit_blocks, obm.lookup_blocks)
    assert torch.equal(stored_bits(cache.k_view().cpu()), stored_bits(kp))
    assert torch.equal(stored_bits(cache.v_view().cpu()), stored_bits(vp))
    for g, o, what in zip(g_out, o_out, ("warm", "step")):
        assert_close(g.numpy(), o, "bf16", what)


def test_full_size_system_prompt_workload_sampled():
    """The benchmark's prompt workload at full size (a 1024-token system prompt
    served first, then 64 requests of it plus 256 tokens each), in the
    benchmark's launch configuration: cached counts, slots, pairs, tables and
    lengths bit for bit, every written slot bit for bit, sampled output rows
    of both phases against the oracle."""
    w = wl.PROMPT_CONFIGS["prefill_system_prompt_bf16"]()
    warm_ids, step_ids = [10_000], list(range(w.B))
    rng = np.random.default_rng(17)
    g_out, g_plans, cache, err = run_gpu(w, warm_ids, step_ids)
    assert err == 0
    T = [int(gp.chunks.sum()) for gp in g_plans]
    units = {}
    for phase, n in zip(("warm", "step"), T):
        u = {(0, 0), (n - 1, w.Hq - 1)}
        while len(u) < 24:
            u.add((int(rng.integers(n)), int(rng.integers(w.Hq))))
        units[phase] = sorted(u)
    o_out, o_info, kp, vp, obm = run_oracle(w, warm_ids, step_ids, units=units)
    for gp, oi in zip(g_plans, o_info):
        assert list(gp.cached) == oi["cached"]
        assert list(gp.slots) == oi["slots"]
        assert [tuple(x) for x in gp.pairs] == oi["pairs"]
        assert np.array_equal(gp.tables.astype(np.int64), oi["tables"])
        assert np.array_equal(gp.lens, oi["lens"])
    assert o_info[1]["cached"] == [1024] * w.B          # the whole system prompt was reused
    kview, vview = cache.k_view(), cache.v_view()
    for gv, ov in ((kview, kp), (vview, vp)):
        for oi in o_info:
            sl = torch.tensor(oi["slots"], dtype=torch.int64)
            b, off = sl // w.bs, sl % w.bs
            got = gv[b.cuda(), :, off.cuda()].cpu()
            assert torch.equal(stored_bits(got), stored_bits(ov[b, :, off]))
    for g, o, phase in zip(g_out, o_out, ("warm", "step")):
        got = np.stack([g[t, h].numpy() for t, h in units[phase]])
        ref = np.stack([o[u] for u in units[phase]])
        assert_close(got, ref, "bf16", f"full size, {phase}")
        assert torch.isfinite(g).all()
