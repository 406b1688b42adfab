"""GPU parity of preemption by swapping: sequences move to a pinned host pool
(device -> host block copies), a new sequence reuses their device blocks, then
they come back (host -> device copies onto fresh blocks) and decode.

The library's block manager and the oracle's replay the same operations; the
copy pairs, tables and both pools are compared bit-exactly, the decode outputs
within |gpu - oracle| <= 2e-2 + 2e-2 |oracle| (bf16).
"""
import math

import numpy as np
import pytest
import torch

import pkv_workloads as wl
from _lib import library, pkv
from _parity import assert_close, stored_bits
from paged_kv_cache_259_gb300.engine import PagedKVCache

from oracle import attention as oatt
from oracle import cache_ops as oops
from oracle.block_manager import BlockManager as OracleBM

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_and_library():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    library()
    torch.cuda.set_device(0)


def randn(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("copy_engines", [False, True])
@pytest.mark.parametrize("Hq,Hkv,bs", [(8, 8, 16), (16, 4, 32)])
def test_swap_out_reuse_swap_in_then_decode(Hq, Hkv, bs, copy_engines):
    NB, NH, D = 24, 16, 128
    lens = {0: 3 * bs + 5, 1: bs + 1, 2: 2 * bs}
    order = list(np.random.default_rng(bs).permutation(NB))
    cache = PagedKVCache(NB, Hq, Hkv, D, bs, torch.bfloat16, order, "cuda", num_host_blocks=NH)
    obm = OracleBM(NB, bs, order, num_cpu_blocks=NH)
    k0, v0 = randn((NB, Hkv, bs, D), 1), randn((NB, Hkv, bs, D), 2)
    cache.load(k0, v0)
    cache.host_k.zero_()
    cache.host_v.zero_()
    kp, vp = k0.clone(), v0.clone()                        # oracle device pools
    hk = torch.zeros(NH, Hkv, bs, D, dtype=torch.bfloat16)  # oracle host pools
    hv = torch.zeros_like(hk)
    for sid, L in lens.items():
        cache.bm.add_seq(sid)
        obm.add_seq(sid)
        assert cache.bm.append_n(sid, L) == []
        for _ in range(L):
            obm.append_slot(sid)
    # preempt 0 and 2 by swapping
    pairs = cache.swap_out([0, 2], copy_engines=copy_engines)
    exp = obm.swap_out(0) + obm.swap_out(2)
    assert [tuple(x) for x in pairs] == exp
    for d, h in exp:
        hk[h], hv[h] = kp[d], vp[d]
    # a new sequence takes their device blocks and writes its own K/V there
    cache.bm.add_seq(9)
    obm.add_seq(9)
    n9 = 4 * bs
    slots, cows = cache.bm.append_slots([9] * n9)
    exp_slots = [obm.append_slot(9)[0] for _ in range(n9)]
    assert list(slots) == exp_slots and not len(cows)
    k9, v9 = randn((n9, Hkv, D), 3), randn((n9, Hkv, D), 4)
    pkv.reshape_and_cache(k9.cuda(), v9.cuda(), cache.k_pool, cache.v_pool,
                          torch.as_tensor(slots, device="cuda"))
    oops.reshape_and_cache(k9, v9, kp, vp, torch.tensor(exp_slots), bs)
    # bring 0 and 2 back onto fresh device blocks
    pairs = cache.swap_in([0, 2], copy_engines=copy_engines)
    exp = obm.swap_in(0) + obm.swap_in(2)
    assert [tuple(x) for x in pairs] == exp
    for h, d in exp:
        kp[d], vp[d] = hk[h], hv[h]
    assert pkv.get_device_error() == 0
    kv, vv = cache.k_view().cpu(), cache.v_view().cpu()
    assert torch.equal(stored_bits(kv), stored_bits(kp))
    assert torch.equal(stored_bits(vv), stored_bits(vp))
    hkv, hvv = pkv.pool_views(cache.host_k, cache.host_v)
    assert torch.equal(stored_bits(hkv), stored_bits(hk))
    assert torch.equal(stored_bits(hvv), stored_bits(hv))
    # decode every sequence over the restored cache
    ids = [0, 1, 2, 9]
    MB = max(-(-cache.bm.seq_len(s) // bs) for s in ids)
    tables, slens = cache.bm.build_tables(ids, MB)
    q = randn((len(ids), Hq, D), 5)
    out = torch.empty(len(ids), Hq, D, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attention_decode(out, q.cuda(), cache.k_pool, cache.v_pool,
                               torch.as_tensor(tables, device="cuda"),
                               torch.as_tensor(slens, device="cuda"), 1 / math.sqrt(D))
    otables = np.full((len(ids), MB), -1, dtype=np.int64)
    for i, s in enumerate(ids):
        t = obm.block_table(s)
        otables[i, :len(t)] = t
    assert np.array_equal(tables.astype(np.int64), otables)
    ref = oatt.paged_decode(q, kp, vp, otables, [obm.seq_len(s) for s in ids], 1 / math.sqrt(D), bs)
    assert_close(out.float().cpu().numpy(), ref, "bf16", "decode after swap-in")
    assert pkv.get_device_error() == 0


def test_swap_blocks_rejects_pageable_host_memory_and_flags_bad_pairs():
    ks, vs = pkv.pool_shapes(4, 2, 16, 64, torch.bfloat16)
    dk = torch.zeros(ks, dtype=torch.bfloat16, device="cuda")
    dv = torch.zeros(vs, dtype=torch.bfloat16, device="cuda")
    hk = torch.zeros(ks, dtype=torch.bfloat16)             # pageable: not reachable
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    with pytest.raises(ValueError):
        pkv.swap_blocks(hk, hk.clone(), dk, dv, pairs)
    ph = hk.pin_memory()
    pv = torch.zeros(vs, dtype=torch.bfloat16).pin_memory()
    bad = torch.tensor([[0, 9], [1, 2]], dtype=torch.int64, device="cuda")
    dk.fill_(1.0)
    dv.fill_(2.0)
    pkv.swap_blocks(ph, pv, dk, dv, bad)
    assert pkv.get_device_error() == -4                  # (0, 9): outside the host pool
    assert torch.all(ph[2] == 1) and torch.all(pv[2] == 2)
    assert torch.count_nonzero(ph[0]) == 0 and torch.count_nonzero(pv[[0, 1, 3]]) == 0


@pytest.mark.parametrize("copy_engines", [False, True])
def test_full_size_swap_workload_two_round_trips_bit_exact(copy_engines):
    """The benchmarked workload (the newest 16 of 64 LLaMA-13B-shaped sequences,
    1105 blocks) swapped out and in twice, block ids changing every time; pairs
    equal the oracle's, and sampled blocks of both pools equal the oracle's pools."""
    sw = wl.swap_llama13b_bf16()
    w = sw.base
    cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, torch.bfloat16, w.free_order, "cuda",
                         num_host_blocks=sw.num_host_blocks)
    kp, vp = w.past_pools()                                # also the oracle's device pools
    cache.load(kp, vp)
    cache.replay(w.script)
    obm = OracleBM(w.NB, w.bs, list(w.free_order), num_cpu_blocks=sw.num_host_blocks)
    for op in w.script:
        if op[0] == "add":
            obm.add_seq(op[1])
        else:
            for _ in range(op[2]):
                obm.append_slot(op[1])
    hk = torch.zeros((sw.num_host_blocks,) + tuple(kp.shape[1:]), dtype=kp.dtype)
    hv = torch.zeros_like(hk)
    for _ in range(2):
        g = cache.swap_out(sw.victims, copy_engines=copy_engines)
        o = [p for s in sw.victims for p in obm.swap_out(s)]
        assert [tuple(x) for x in g] == o and len(o) == sw.victim_blocks
        oops.swap_blocks(hk, hv, kp, vp, o)
        g = cache.swap_in(sw.victims, copy_engines=copy_engines)
        o = [p for s in sw.victims for p in obm.swap_in(s)]
        assert [tuple(x) for x in g] == o
        oops.swap_blocks(kp, vp, hk, hv, o)
    assert pkv.get_device_error() == 0
    rng = np.random.default_rng(0)
    victim_blocks = [b for s in sw.victims for b in obm.block_table(s)]
    other = [b for s in range(w.B) if s not in sw.victims for b in obm.block_table(s)]
    idx = torch.tensor(sorted(set(rng.choice(victim_blocks, 64).tolist() +
                                  rng.choice(other, 32).tolist())))
    kv, vv = cache.k_view(), cache.v_view()
    assert torch.equal(stored_bits(kv[idx.cuda()].cpu()), stored_bits(kp[idx]))
    assert torch.equal(stored_bits(vv[idx.cuda()].cpu()), stored_bits(vp[idx]))
    del kv, vv
    hidx = torch.tensor(sorted(set(rng.choice(sw.num_host_blocks, 64).tolist())))
    hkv, hvv = pkv.pool_views(cache.host_k, cache.host_v)
    assert torch.equal(stored_bits(hkv[hidx]), stored_bits(hk[hidx]))
    assert torch.equal(stored_bits(hvv[hidx]), stored_bits(hv[hidx]))


def test_preempt_by_recompute_then_resume_decodes_as_before():
    """Two sequences are preempted by recomputation (blocks freed), another
    sequence takes every free block, overwrites it and finishes, then they
    resume: one
    chunked-prefill step over all their tokens rewrites their K/V (the values
    the model would recompute: here the original ones) into fresh blocks. The
    next decode step gives bit for bit the outputs it gave before, and the
    resumed tables read back the original K/V."""
    Hq, Hkv, bs, D, NB = 8, 2, 16, 128, 40
    lens = {0: 3 * bs + 5, 1: bs + 1, 2: 2 * bs}
    order = list(np.random.default_rng(3).permutation(NB))
    cache = PagedKVCache(NB, Hq, Hkv, D, bs, torch.bfloat16, order, "cuda")
    k0, v0 = randn((NB, Hkv, bs, D), 11), randn((NB, Hkv, bs, D), 12)
    cache.load(k0, v0)
    for sid, L in lens.items():
        cache.bm.add_seq(sid)
        assert cache.bm.append_n(sid, L) == []
    ids = [0, 1, 2]
    MB = max(-(-L // bs) for L in lens.values()) + 1
    q = randn((len(ids), Hq, D), 13)

    def decode():
        tables, slens = cache.bm.build_tables(ids, MB)
        out = torch.empty(len(ids), Hq, D, dtype=torch.bfloat16, device="cuda")
        pkv.paged_attention_decode(out, q.cuda(), cache.k_pool, cache.v_pool,
                                   torch.as_tensor(tables, device="cuda"),
                                   torch.as_tensor(slens, device="cuda"), 1 / math.sqrt(D))
        return out.cpu()

    def rows(sid):                                        # [L, Hkv, D] through the table
        kv, vv = cache.k_view().cpu(), cache.v_view().cpu()
        t = cache.bm.block_table(sid)
        k = torch.cat([kv[b].transpose(0, 1) for b in t])[:cache.bm.seq_len(sid)]
        v = torch.cat([vv[b].transpose(0, 1) for b in t])[:cache.bm.seq_len(sid)]
        return k, v

    before = decode()
    saved = {s: rows(s) for s in (0, 2)}
    old_tables = {s: cache.bm.block_table(s) for s in (0, 2)}
    n = cache.preempt_by_recompute([0, 2])
    assert n == {0: lens[0], 2: lens[2]}
    # another sequence takes every free block (theirs included), overwrites them
    # all and finishes: whatever blocks the resumed sequences get hold garbage
    cache.bm.add_seq(9)
    n9 = cache.bm.num_free() * bs
    slots = np.concatenate([cache.bm.append_slots([9])[0] for _ in range(n9)])
    assert cache.bm.num_free() == 0 and set(old_tables[0] + old_tables[2]) <= set(
        cache.bm.block_table(9))
    pkv.reshape_and_cache(randn((n9, Hkv, D), 14).cuda(), randn((n9, Hkv, D), 15).cuda(),
                          cache.k_pool, cache.v_pool, torch.as_tensor(slots, device="cuda"))
    cache.bm.free_seq(9)
    plan = cache.plan_resume([0, 2], n)
    k = torch.cat([saved[0][0], saved[2][0]])
    v = torch.cat([saved[0][1], saved[2][1]])
    qp = randn((k.shape[0], Hq, D), 16)
    out = torch.empty(k.shape[0], Hq, D, dtype=torch.bfloat16, device="cuda")
    cache.prefill_step(qp.cuda(), k.cuda(), v.cuda(), plan.device_tensors("cuda"), out,
                       1 / math.sqrt(D), plan.max_query_len)
    assert pkv.get_device_error() == 0
    for s in (0, 2):
        kk, vv = rows(s)
        assert torch.equal(stored_bits(kk), stored_bits(saved[s][0]))
        assert torch.equal(stored_bits(vv), stored_bits(saved[s][1]))
    assert torch.equal(decode(), before)
