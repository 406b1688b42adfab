"""The one-call steps against the same steps as separate calls: outputs and
both whole pools bit for bit.

paged_decode_step (copy-on-write copies, slot writes, attention, with the
attention reading every block but the sequences' last ones while the writes
finish) on regular, split, grouped (fork step with its copies), beam-search and
paired-stage E4M3 steps; paged_prefill_step (the attention reading the key tiles
before each chunk while the writes finish) on ragged MHA, GQA with 32-token
blocks, the LLaMA-13B chunk shape and a chunk after a fork (copy-on-write). The
separate calls are themselves held to the oracle by test_gpu_parity.py and
test_gpu_prefill.py; the one-call steps are also what cache.step and
cache.prefill_step run there."""
import numpy as np
import pytest
import torch

import paged_kv_cache_259_gb300 as pkv
import pkv_workloads as wl
from paged_kv_cache_259_gb300.engine import PagedKVCache

from _parity import KV_TORCH, Inputs

pytestmark = pytest.mark.gpu

CASES = {
    "mha_bf16_split": lambda: wl.llama13b_mha_bf16(B=6),
    "gqa_bf16": lambda: wl.gqa_chat_bf16(B=24),
    "e4m3_bs16_paired": lambda: wl.long_fp8(16, B=2, L=3000),
    "e4m3_bs32": lambda: wl.long_fp8(32, B=2, L=3000),
    "fork_step_grouped": lambda: wl.shared_prefix_bf16(True, groups=5),
    "shared_prefix_grouped": lambda: wl.shared_prefix_bf16(False, groups=5),
    "beam_search": lambda: wl.beam_search_bf16(requests=3),
}


def _prepared(inp):
    w = inp.w
    cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, KV_TORCH[w.kv_dtype], w.free_order, "cuda")
    cache.load(inp.k_src, inp.v_src, inp.ks, inp.vs)
    cache.apply_copies(cache.replay(w.script))
    plan = cache.plan_step(w.step_seqs, max_blocks=w.max_blocks_per_seq)
    return cache, plan


@pytest.mark.parametrize("name", sorted(CASES))
def test_one_call_step_equals_separate_calls(name):
    w = CASES[name]()
    inp = Inputs(w)
    results = []
    for fused in (False, True):
        cache, plan = _prepared(inp)
        dev = plan.device_tensors("cuda")
        q, k, v = inp.q.cuda(), inp.k_new.cuda(), inp.v_new.cuda()
        out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=w.src_dtype, device="cuda")
        ws = cache.workspace(w.B, w.max_blocks_per_seq)
        if fused:
            cache.step(q, k, v, dev, out, w.scale, inp.ks, inp.vs, ws)
        else:
            if dev["pairs"].shape[0]:
                pkv.copy_blocks(cache.k_pool, cache.v_pool, dev["pairs"])
            pkv.reshape_and_cache(k, v, cache.k_pool, cache.v_pool, dev["slots"], inp.ks, inp.vs)
            cache.decode(q, dev, out, w.scale, inp.ks, inp.vs, ws)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        results.append((out.cpu(), cache.k_pool.cpu(), cache.v_pool.cpu(), plan))
    (o1, k1, v1, p1), (o2, k2, v2, p2) = results
    if name.startswith(("fork", "beam")):
        assert len(p1.pairs) > 0                        # the step copies blocks
    if name.startswith(("fork", "shared", "beam")):
        assert p1.num_groups > 0
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert not torch.isnan(o2.float()).any()
    assert torch.equal(o1, o2)


def test_one_call_step_repeated_is_idempotent_and_counts_its_launches():
    """The step re-run on its own output state gives the same output (the slot
    write and the copies are idempotent), with copy_blocks, reshape_and_cache,
    the decode and the merge as its launches."""
    w = wl.shared_prefix_bf16(True, groups=3)
    inp = Inputs(w)
    cache, plan = _prepared(inp)
    dev = plan.device_tensors("cuda")
    q, k, v = inp.q.cuda(), inp.k_new.cuda(), inp.v_new.cuda()
    ws = cache.workspace(w.B, w.max_blocks_per_seq)
    outs = []
    for _ in range(3):
        out = torch.empty(w.B, w.Hq, w.D, dtype=w.src_dtype, device="cuda")
        n0 = pkv.kernel_launches()
        cache.step(q, k, v, dev, out, w.scale, inp.ks, inp.vs, ws)
        torch.cuda.synchronize()
        assert pkv.kernel_launches() - n0 >= 3
        outs.append(out.cpu())
    assert pkv.get_device_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def _prefill_workload(name):
    if name == "fork_cow":
        # two samples share a 40-token prompt whose last block is partial: the
        # second one's chunk copies that block first (copy-on-write)
        w = wl.chunked_prefill("one_call_fork", 77, [0, 0], [1, 1], 8, 2, 128, 16, NB=40)
        w.script = [("add", 0), ("append", 0, 40), ("fork", 0, 1)]
        w.chunks = np.array([20, 150])
        w.final_lens = np.array([60, 190])
        return w
    return {
        "mha_ragged": lambda: wl.chunked_prefill("one_call_mha", 5, [0, 300, 77], [200, 64, 129],
                                                 8, 8, 128, 16),
        "gqa_bs32": lambda: wl.chunked_prefill("one_call_gqa", 6, [900, 0, 64], [96, 300, 5],
                                               32, 8, 128, 32),
        "llama13b_shape": lambda: wl.prefill_llama13b_bf16(B=2),
    }[name]()


@pytest.mark.parametrize("name", ["mha_ragged", "gqa_bs32", "llama13b_shape", "fork_cow"])
def test_one_call_prefill_step_equals_separate_calls(name):
    """paged_prefill_step (the attention reading the tiles before each chunk
    while the chunk's slot writes and the step's copies finish) against copy_blocks,
    reshape_and_cache and paged_attention_prefill made one after another: outputs
    and both whole pools bit for bit."""
    w = _prefill_workload(name)
    k_src, v_src = w.past_pools()
    q, k_new, v_new = w.step_inputs()
    results = []
    for fused in (False, True):
        cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, torch.bfloat16, w.free_order, "cuda")
        cache.load(k_src, v_src)
        cache.apply_copies(cache.replay(w.script))
        plan = cache.plan_prefill(w.step_seqs, w.chunks, max_blocks=w.max_blocks_per_seq)
        dev = plan.device_tensors("cuda")
        out = torch.full((w.T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        qd, kd, vd = q.cuda(), k_new.cuda(), v_new.cuda()
        if fused:
            cache.prefill_step(qd, kd, vd, dev, out, w.scale, plan.max_query_len)
        else:
            if dev["pairs"].shape[0]:
                pkv.copy_blocks(cache.k_pool, cache.v_pool, dev["pairs"])
            pkv.reshape_and_cache(kd, vd, cache.k_pool, cache.v_pool, dev["slots"])
            pkv.paged_attention_prefill(out, qd, cache.k_pool, cache.v_pool, dev["tables"],
                                        dev["lens"], dev["query_start"], w.scale,
                                        plan.max_query_len)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        results.append((out.cpu(), cache.k_pool.cpu(), cache.v_pool.cpu(), plan))
    (o1, k1, v1, p1), (o2, k2, v2, _) = results
    if name == "fork_cow":
        assert len(p1.pairs) > 0
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert not torch.isnan(o2.float()).any()
    assert torch.equal(o1, o2)
