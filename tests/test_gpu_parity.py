"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

* indexing (slots, copy-on-write pairs, block tables, lengths): bit-exact;
* cache writes (reshape_and_cache incl. E4M3 bytes, copy_blocks): bit-exact;
* attention outputs: |gpu - oracle| <= atol + rtol |oracle| elementwise, with
  (atol, rtol) = (2e-2, 2e-2) for bf16 caches, (6e-2, 6e-2) for E4M3 and
  (1e-5, 1e-5) for float32.

Small cases compare every output and the whole pools; the full-size workloads
(the benchmark's sizes and launch configuration, i.e. with a split-KV
workspace) compare sampled (sequence, head) outputs that the oracle computes one
by one.
"""
import math

import numpy as np
import pytest
import torch

import bench
import pkv_workloads as wl
from oracle import fp8_e4m3 as ofp8
from _lib import library, pkv
from _parity import (Inputs, assert_close, check_cache_writes, check_indexing,
                     run_gpu, run_oracle, sample_units)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_and_library():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    library()
    torch.cuda.set_device(0)


def small(name, seed, lens, Hq, Hkv, D, bs, kv, NB=None):
    src = torch.float32 if kv == "f32" else torch.bfloat16
    return wl.prefill_workload(name, seed, lens, Hq, Hkv, D, bs, src, kv, 1.0 / math.sqrt(D), NB=NB)


def ragged_lens(bs):
    return [1, 2, bs - 1, bs, bs + 1, 100, 777, 2500]


VARIANTS = [  # (kv dtype, G, head_dim, block_size)
    ("f32", 1, 64, 16), ("f32", 2, 128, 32), ("f32", 4, 64, 16), ("f32", 8, 128, 16),
    ("bf16", 1, 128, 16), ("bf16", 1, 64, 32), ("bf16", 2, 128, 16), ("bf16", 4, 128, 16),
    ("bf16", 4, 128, 32), ("bf16", 8, 64, 16), ("bf16", 8, 128, 32),
    ("e4m3", 4, 128, 16), ("e4m3", 4, 128, 32), ("e4m3", 1, 128, 16), ("e4m3", 2, 64, 16),
    ("e4m3", 8, 64, 32),
]


@pytest.mark.parametrize("kv,G,D,bs", VARIANTS)
@pytest.mark.parametrize("workspace", [True, False])
def test_small_variant_matches_oracle(kv, G, D, bs, workspace):
    Hkv = 2
    w = small(f"{kv}_g{G}_d{D}_bs{bs}", 100 + G * 7 + D + bs, ragged_lens(bs), G * Hkv, Hkv, D, bs, kv)
    inp = Inputs(w)
    g = run_gpu(inp, workspace=workspace)
    assert g["err"] == 0
    o = run_oracle(inp)
    check_indexing(g, o)
    check_cache_writes(inp, g, o, whole_pool=True)
    assert_close(g["out"].numpy(), o["out"], kv, w.name)


def test_tiny_fp32_config_all_outputs():
    inp = Inputs(wl.tiny_fp32())
    g = run_gpu(inp)
    assert g["err"] == 0
    o = run_oracle(inp)
    check_indexing(g, o)
    check_cache_writes(inp, g, o, whole_pool=True)
    assert_close(g["out"].numpy(), o["out"], "f32", "tiny_fp32")
    # seq_len 1: the output is exactly the value just written
    np.testing.assert_array_equal(g["out"][0].numpy(), inp.v_new[0].float().numpy())


FULL = ["llama13b_mha_bf16", "gqa_chat_bf16", "shared_prefix_bf16", "shared_prefix_fork_bf16",
        "long_fp8_bs16", "long_fp8_bs32", "beam_search_bf16"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled(name):
    w = wl.CONFIGS[name]()
    inp = Inputs(w)
    g = run_gpu(inp, workspace=True)
    assert g["err"] == 0
    units = sample_units(w, 128 if w.kv_dtype == "e4m3" else 96, seed=1)
    o = run_oracle(inp, units=[])                 # the oracle's state: slots, tables, pools
    check_indexing(g, o)
    check_cache_writes(inp, g, o)
    # the sampled rows through the bench's multi-process oracle runner (one
    # single-threaded float64 oracle process per host core)
    per_tok = 2 * w.Hkv * w.D * {"e4m3": 1, "bf16": 2, "f32": 4}[w.kv_dtype]
    _, _, _, note, rows = bench.oracle_timing(
        w, (inp.q, o["k_pool"], o["v_pool"], inp.ks, inp.vs), o["tables"], o["lens"], per_tok,
        0.0, 1, check_units=units)
    assert sorted(rows) == sorted(units), note
    got = np.stack([g["out"][b, h].numpy() for b, h in units])
    ref = np.stack([rows[u] for u in units])
    assert_close(got, ref, w.kv_dtype, name)
    assert torch.isfinite(g["out"]).all()
    if name == "shared_prefix_fork_bf16":
        assert len(o["pairs"]) == 192
    # the unsplit launch agrees with the split one on every output
    g1 = run_gpu(inp, workspace=False)
    assert g1["err"] == 0
    assert_close(g1["out"].numpy(), g["out"].numpy().astype(np.float64), w.kv_dtype,
                 name + " split vs unsplit")


def test_relabelling_physical_blocks_is_bitwise_invariant():
    w = small("relabel", 5, ragged_lens(16), 8, 2, 128, 16, "bf16")
    inp = Inputs(w)
    a = run_gpu(inp)
    perm = np.random.default_rng(3).permutation(w.NB)
    b = run_gpu(inp, relabel=perm)
    assert a["err"] == 0 and b["err"] == 0
    assert torch.equal(a["out"], b["out"])


def test_repeated_step_is_idempotent():
    w = wl.shared_prefix_bf16(fork_step=True, groups=4)
    inp = Inputs(w)
    g = run_gpu(inp)
    cache, plan = g["cache"], g["plan"]
    dev = plan.device_tensors("cuda")
    out2 = torch.empty(w.B, w.Hq, w.D, dtype=w.src_dtype, device="cuda")
    ws = cache.workspace(w.B, w.max_blocks_per_seq)
    for _ in range(3):
        cache.step(inp.q.cuda(), inp.k_new.cuda(), inp.v_new.cuda(), dev, out2, w.scale,
                   workspace=ws)
    assert pkv.get_device_error() == 0
    assert torch.equal(out2.float().cpu(), g["out"])


def to_layout(kc, vc):
    """Canonical ``[NB, Hkv, bs, D]`` K/V -> the library's pool layout (plain copies)."""
    return pkv.pools_from_views(kc, vc)


def _decode_args(B, Hq, Hkv, D, bs, NB, MB, dtype=torch.bfloat16, seed=0):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, D, generator=gen).to(dtype).cuda()
    kc = torch.randn(NB, Hkv, bs, D, generator=gen).to(dtype)
    vc = torch.randn(NB, Hkv, bs, D, generator=gen).to(dtype)
    kp, vp = to_layout(kc.cuda(), vc.cuda())
    bt = torch.arange(B * MB, dtype=torch.int32).reshape(B, MB).remainder(NB).cuda()
    return q, kp, vp, bt, kc, vc


def test_zero_length_sequences_give_zero_rows():
    q, kp, vp, bt, _, _ = _decode_args(4, 4, 4, 128, 16, 32, 8)
    lens = torch.tensor([0, 5, 0, 128], dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    pkv.paged_attention_decode(out, q, kp, vp, bt, lens, 0.1)
    assert pkv.get_device_error() == 0
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
    assert torch.isfinite(out).all() and torch.count_nonzero(out[1]) > 0


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])   # CUDA-core (MHA) and tensor-core (GQA)
def test_largest_batch_of_65535_sequences(Hq, Hkv):
    """The largest batch the decode takes (the sequence index is a grid
    dimension): 65,535 short sequences over a small shared pool, zero lengths
    included; sampled rows against the oracle, the first and last sequences among
    them."""
    from oracle import attention as oatt
    B, D, bs, NB, MB = 65535, 128, 16, 256, 4
    q, kp, vp, _, kc, vc = _decode_args(B, Hq, Hkv, D, bs, NB, MB, seed=Hq)
    rng = np.random.default_rng(Hq)
    tables = rng.integers(0, NB, size=(B, MB)).astype(np.int32)
    lens = rng.integers(0, MB * bs + 1, size=B).astype(np.int32)
    lens[0], lens[-1] = MB * bs, 1
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode(out, q, kp, vp, torch.from_numpy(tables).cuda(),
                               torch.from_numpy(lens).cuda(), 1 / math.sqrt(D))
    assert pkv.get_device_error() == 0
    got = out.float().cpu()
    assert torch.isfinite(got).all()
    assert torch.count_nonzero(got[torch.from_numpy(lens == 0)]) == 0
    picks = zip(rng.integers(0, B, 400), rng.integers(0, Hq, 400))
    units = sorted({(0, 0), (B - 1, Hq - 1)} | {(int(b), int(h)) for b, h in picks})
    ref = oatt.paged_decode(q.cpu(), kc, vc, tables, lens, 1 / math.sqrt(D), bs, units=units)
    for (b, h), row in ref.items():
        assert_close(got[b, h].numpy(), row, "bf16", f"sequence {b} head {h}")


def test_an_empty_step_launches_nothing():
    """No sequences: the engine plans empty arrays and every call returns at once."""
    from paged_kv_cache_259_gb300.engine import PagedKVCache
    cache = PagedKVCache(8, 8, 2, 128, 16, torch.bfloat16, range(8), "cuda")
    n0 = pkv.kernel_launches()
    plan = cache.plan_step([])
    out = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    cache.step(q, kv, kv, plan.device_tensors("cuda"), out, 0.1,
               workspace=cache.workspace(1, plan.tables.shape[1]))
    pre = cache.plan_prefill([], [])
    cache.prefill_step(q, kv, kv, pre.device_tensors("cuda"), out, 0.1, pre.max_query_len)
    torch.cuda.synchronize()
    assert pkv.kernel_launches() == n0 and pkv.get_device_error() == 0


@pytest.mark.parametrize("Hq", [4, 16])          # CUDA-core (MHA) and tensor-core (GQA) paths
def test_bad_block_id_sets_error_word_and_skips(Hq):
    q, kp, vp, bt, kc, vc = _decode_args(3, Hq, 4, 128, 16, 32, 8)
    bt[1, 2] = 32          # == num_blocks: outside the pool
    bt[2, 0] = -7
    lens = torch.tensor([100, 100, 20], dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    assert pkv.get_device_error() == 0
    pkv.paged_attention_decode(out, q, kp, vp, bt, lens, 0.1)
    assert pkv.get_device_error() == -4
    assert pkv.get_device_error() == 0       # read-and-clear
    # sequence 0 is untouched by the bad entries: compare with the oracle
    from oracle import attention as oatt
    from _parity import assert_close as ac
    ref = oatt.paged_decode(q.cpu()[:1], kc, vc, bt.cpu().numpy()[:1], [100], 0.1, 16)
    ac(out[:1].float().cpu().numpy(), ref, "bf16", "seq 0")


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_paired_stage_with_a_bad_second_block_is_flagged_and_skipped(kv):
    """A bad id in the second block of a stage (block 3 of sequence 1; the E4M3
    decode over 16-token blocks stages two blocks at a time) is flagged and its
    stage skipped; the other sequences, whose last stages hold one block (a
    40-token sequence) or a second block of one token (17 tokens), match the
    oracle. The bf16 case runs the one-block stages of the same path."""
    q, kp, vp, bt, kc, vc = _decode_args(3, 16, 4, 128, 16, 32, 8)
    if kv == "e4m3":
        kc8 = torch.from_numpy(ofp8.e4m3_quantize(kc.float().numpy(), 0.05))
        vc8 = torch.from_numpy(ofp8.e4m3_quantize(vc.float().numpy(), 0.05))
        kp, vp = to_layout(kc8.cuda(), vc8.cuda())
    bt[1, 3] = 32          # == num_blocks: outside the pool
    lens = torch.tensor([40, 100, 17], dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    assert pkv.get_device_error() == 0
    s = 0.05 if kv == "e4m3" else 1.0
    pkv.paged_attention_decode(out, q, kp, vp, bt, lens, 0.1, s, s)
    assert pkv.get_device_error() == -4
    from oracle import attention as oatt
    from _parity import assert_close as ac
    keep = [0, 2]                          # the oracle reads only valid tables
    tk, tv = (kc8, vc8) if kv == "e4m3" else (kc, vc)
    ref = oatt.paged_decode(q.cpu()[keep], tk, tv, bt.cpu().numpy()[keep], [40, 17], 0.1, 16, s, s)
    ac(out[keep].float().cpu().numpy(), ref, kv, "sequences 0 and 2")


def test_a_wait_nothing_completes_times_out_and_the_context_stays_usable():
    """The library's timeout check: one bounded wait on a barrier nothing arrives
    at gives up after its one-second limit and reports PKV_ERR_TIMEOUT (then the
    word is clear); a decode right after it still matches the oracle."""
    import time
    from oracle import attention as oatt
    assert pkv.get_device_error() == 0
    t0 = time.perf_counter()
    pkv.check_wait_timeout()
    assert pkv.get_device_error() == -6
    assert 0.9 < time.perf_counter() - t0 < 60
    assert pkv.get_device_error() == 0
    q, kp, vp, bt, kc, vc = _decode_args(2, 8, 2, 128, 16, 16, 4, seed=6)
    lens = torch.tensor([50, 64], dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    pkv.paged_attention_decode(out, q, kp, vp, bt, lens, 0.1)
    assert pkv.get_device_error() == 0
    ref = oatt.paged_decode(q.cpu(), kc, vc, bt.cpu().numpy(), [50, 64], 0.1, 16)
    assert_close(out.float().cpu().numpy(), ref, "bf16", "decode after the timeout check")


def test_reshape_and_cache_bad_and_padding_slots():
    ks, vs = pkv.pool_shapes(4, 2, 16, 64, torch.bfloat16)
    kp = torch.zeros(ks, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros(vs, dtype=torch.bfloat16, device="cuda")
    k = torch.ones(3, 2, 64, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([-1, 64, 5], dtype=torch.int64, device="cuda")   # pad, outside, ok
    pkv.reshape_and_cache(k, k, kp, vp, slots)
    assert pkv.get_device_error() == -4
    kv, vv = pkv.pool_views(kp, vp)
    assert torch.count_nonzero(kp) == 2 * 64 and torch.all(kv[0, :, 5] == 1)
    assert torch.count_nonzero(vp) == 2 * 64 and torch.all(vv[0, :, 5] == 1)


def test_copy_blocks_bad_pair_sets_error_word():
    ks, vs = pkv.pool_shapes(4, 2, 16, 64, torch.bfloat16)
    kp = torch.randn(ks, device="cuda").to(torch.bfloat16)
    vp = torch.randn(vs, device="cuda").to(torch.bfloat16)
    k0 = kp.clone()
    pairs = torch.tensor([[0, 9], [1, 2]], dtype=torch.int64, device="cuda")
    pkv.copy_blocks(kp, vp, pairs)
    assert pkv.get_device_error() == -4
    assert torch.equal(kp[2], k0[1]) and torch.equal(kp[0], k0[0])


@pytest.mark.parametrize("pairs", [[[0, 2], [1, 2]],          # a destination written twice
                                   [[0, 2], [2, 3]],          # a destination also read
                                   [[1, 1]]],                 # a block copied onto itself
                         ids=["dst_twice", "dst_is_src", "self_copy"])
def test_copy_blocks_conflicting_pairs_set_error_word(pairs):
    """copy_blocks' preconditions (distinct destinations, none also a source) are
    checked on the device: a launch that breaks them reports PKV_ERR_INVALID_ARG
    through the device error word. Every id is inside the pool, so the copies
    stay in bounds; only which bytes land is unspecified."""
    ks, vs = pkv.pool_shapes(4, 2, 16, 64, torch.bfloat16)
    kp = torch.randn(ks, device="cuda").to(torch.bfloat16)
    vp = torch.randn(vs, device="cuda").to(torch.bfloat16)
    assert pkv.get_device_error() == 0
    pkv.copy_blocks(kp, vp, torch.tensor(pairs, dtype=torch.int64, device="cuda"))
    assert pkv.get_device_error() == -1
    # a valid launch right after leaves the word clear
    pkv.copy_blocks(kp, vp, torch.tensor([[0, 2], [0, 3]], dtype=torch.int64, device="cuda"))
    assert pkv.get_device_error() == 0
    assert torch.equal(kp[2], kp[0]) and torch.equal(vp[3], vp[0])


def test_host_checks_reject_bad_arguments():
    q, kp, vp, bt, _, _ = _decode_args(2, 4, 4, 96, 16, 8, 4)       # head_dim 96 not built
    lens = torch.tensor([3, 4], dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_attention_decode(torch.empty_like(q), q, kp, vp, bt, lens, 0.1)
    assert e.value.status == -2
    q, kp, vp, bt, _, _ = _decode_args(2, 6, 4, 64, 16, 8, 4)       # 6 heads over 4 kv heads
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_attention_decode(torch.empty_like(q), q, kp, vp, bt, lens, 0.1)
    assert e.value.status == -1


# ------------------------------------------------------------ prefix-grouped decode
GROUPED = [  # (kv, Hq, Hkv, D, bs, per_group, prompt, fork_step)
    ("bf16", 8, 8, 128, 16, 4, 200, False),     # MHA, 4 members
    ("bf16", 8, 8, 64, 32, 6, 333, False),      # 6 forks: groups of 6 (8 rows allow it)
    ("bf16", 16, 8, 128, 16, 5, 97, False),     # GQA 2: 5 forks -> groups of 4 and 1
    ("bf16", 16, 4, 128, 16, 3, 150, True),     # GQA 4: groups of 2 and 1, CoW step
    ("e4m3", 16, 4, 128, 16, 2, 300, False),    # E4M3 cache
    ("e4m3", 8, 8, 128, 32, 4, 64, True),       # prompt fills its blocks exactly
    ("bf16", 64, 8, 128, 16, 3, 150, False),    # GQA 8: one member per group -> plain path
]


@pytest.mark.parametrize("kv,Hq,Hkv,D,bs,per_group,prompt,fork", GROUPED)
def test_grouped_prefix_decode_matches_oracle(kv, Hq, Hkv, D, bs, per_group, prompt, fork):
    w = wl.shared_prefix(fork_step=fork, groups=3, per_group=per_group, prompt=prompt,
                         max_suffix=70, Hq=Hq, Hkv=Hkv, D=D, bs=bs, kv=kv,
                         seed=per_group * 13 + prompt, name=f"grouped_{kv}_{Hq}_{Hkv}")
    inp = Inputs(w)
    g = run_gpu(inp)
    assert g["err"] == 0
    plan = g["plan"]
    G = Hq // Hkv
    if 8 // G >= 2:
        assert plan.num_groups > 0
        # every group: members share the prefix's block ids, full for all of them
        for gi, (members, pre) in enumerate(zip(plan.group_members, plan.group_prefix)):
            ms = [m for m in members if m >= 0]
            assert 2 <= len(ms) <= 8 // G and pre >= 1
            for m in ms:
                assert plan.seq_group[m] == gi and plan.lens[m] >= pre * bs
                assert np.array_equal(plan.tables[m, :pre], plan.tables[ms[0], :pre])
    else:
        assert plan.num_groups == 0
    o = run_oracle(inp)
    check_indexing(g, o)
    check_cache_writes(inp, g, o, whole_pool=True)
    assert_close(g["out"].numpy(), o["out"], kv, w.name)
    # the plain (ungrouped) decode agrees with the grouped one
    cache = g["cache"]
    dev = g["plan"].device_tensors("cuda")
    for k in ("seq_group", "group_members", "group_prefix", "ungrouped"):
        dev.pop(k, None)
    out2 = torch.empty(w.B, w.Hq, w.D, dtype=w.src_dtype, device="cuda")
    cache.decode(inp.q.cuda(), dev, out2, w.scale, inp.ks, inp.vs,
                 cache.workspace(w.B, w.max_blocks_per_seq))
    assert pkv.get_device_error() == 0
    assert_close(out2.float().cpu().numpy(), o["out"], kv, w.name + " plain")
    if plan.num_groups:
        # without the ungrouped list every sequence gets a regular CTA; grouped
        # ones leave at once
        dev = plan.device_tensors("cuda")
        out3 = torch.empty_like(out2)
        pkv.paged_attention_decode_grouped(
            out3, inp.q.cuda(), cache.k_pool, cache.v_pool, dev["tables"], dev["lens"], w.scale,
            dev["seq_group"], dev["group_members"], dev["group_prefix"], inp.ks, inp.vs,
            cache.workspace(w.B, w.max_blocks_per_seq), None, None)
        assert pkv.get_device_error() == 0
        assert_close(out3.float().cpu().numpy(), o["out"], kv, w.name + " no list")


BEAMS = [  # (kv, Hq, Hkv, D, bs, requests, width, prompt range, generated)
    ("bf16", 8, 8, 128, 16, 3, 4, (1, 60), 40),      # MHA: beams grouped (up to 8 rows)
    ("bf16", 16, 4, 128, 16, 3, 2, (20, 300), 70),   # GQA 4: groups of 2
    ("bf16", 8, 8, 64, 32, 2, 8, (1, 33), 50),       # 8 beams, block size 32
    ("e4m3", 8, 8, 128, 16, 2, 4, (100, 200), 33),   # E4M3 cache
    ("f32", 4, 4, 64, 16, 2, 3, (5, 40), 20),        # float32 cache: no grouping
]


@pytest.mark.parametrize("kv,Hq,Hkv,D,bs,requests,width,prompt,gen", BEAMS)
def test_beam_search_step_matches_oracle(kv, Hq, Hkv, D, bs, requests, width, prompt, gen):
    """A beam-search state (beams reshuffled every step: forks of the chosen
    parents, frees of the old beams, CoW of shared partial blocks) and the next
    step (CoW, slot write, grouped decode): pairs, tables, the whole pools and
    every output against the oracle."""
    src = torch.float32 if kv == "f32" else torch.bfloat16
    w = wl.beam_search(f"beam_{kv}_{Hq}_{width}", requests, width, prompt, gen, Hq, Hkv, D, bs,
                       seed=gen + width, src_dtype=src, kv_dtype=kv)
    inp = Inputs(w)
    g = run_gpu(inp)
    assert g["err"] == 0
    o = run_oracle(inp)
    check_indexing(g, o)
    check_cache_writes(inp, g, o, whole_pool=True)
    assert_close(g["out"].numpy(), o["out"], kv, w.name)
    if kv != "f32" and 8 // (Hq // Hkv) >= 2:
        assert g["plan"].num_groups > 0                # beams of a request share their prefix


def test_group_list_hint_sizes_the_launch_and_a_short_hint_is_flagged():
    """The engine passes the longest group list (bm_prefix_groups' count); the
    grouped decode without it (bound max_members x max_blocks) gives the same
    outputs; a hint shorter than a list cuts it, and the device error says so."""
    w = wl.beam_search("beam_hint", 3, 4, (300, 900), 40, 8, 8, 128, 16, seed=5)
    inp = Inputs(w)
    g = run_gpu(inp)
    assert g["err"] == 0
    plan, cache = g["plan"], g["cache"]
    assert plan.num_groups == 3
    assert plan.max_group_blocks < plan.group_members.shape[1] * plan.tables.shape[1]
    o = run_oracle(inp)
    assert_close(g["out"].numpy(), o["out"], "bf16", "engine (hint)")
    dev = plan.device_tensors("cuda")
    ws = cache.workspace(w.B, w.max_blocks_per_seq)
    q = inp.q.cuda()
    for hint in (0, plan.max_group_blocks, 1):
        out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        pkv.paged_attention_decode_grouped(
            out, q, cache.k_pool, cache.v_pool, dev["tables"], dev["lens"], w.scale,
            dev["seq_group"], dev["group_members"], dev["group_prefix"], 1.0, 1.0, ws, None,
            dev["ungrouped"], hint)
        err = pkv.get_device_error()
        if hint == 1:
            assert err == -4                           # lists longer than the hint
        else:
            assert err == 0
            assert_close(out.float().cpu().numpy(), o["out"], "bf16", f"hint {hint}")


@pytest.mark.parametrize("prompt,suffix", [(100, 40), (1200, 900)])
def test_grouped_decode_without_workspace(prompt, suffix):
    """No workspace: every group list and sequence runs as one partition."""
    w = wl.shared_prefix(groups=2, per_group=4, prompt=prompt, max_suffix=suffix, Hq=8, Hkv=8,
                         seed=prompt)
    inp = Inputs(w)
    g = run_gpu(inp, workspace=False)
    assert g["err"] == 0 and g["plan"].num_groups == 2
    o = run_oracle(inp)
    assert_close(g["out"].numpy(), o["out"], "bf16", "grouped, no workspace")


def test_grouped_decode_long_lists_are_split_and_merged():
    """Group lists longer than a partition (long prompt, long tails) go through
    the split merge."""
    w = wl.shared_prefix(groups=3, per_group=4, prompt=2000, max_suffix=1500, Hq=8, Hkv=8,
                         seed=77)
    inp = Inputs(w)
    g = run_gpu(inp)
    assert g["err"] == 0 and g["plan"].num_groups == 3
    o = run_oracle(inp)
    assert_close(g["out"].numpy(), o["out"], "bf16", "grouped, split lists")


def test_grouped_decode_bad_group_index_is_flagged_not_followed():
    """A seq_group entry naming no group of the call (>= num_groups) on a call
    whose group lists are split and merged: the merge's bounds check flags it
    (PKV_ERR_OUT_OF_RANGE) instead of reading past the group arrays; the context
    stays usable and the same call with the right groups is clean again."""
    w = wl.shared_prefix(groups=3, per_group=4, prompt=2000, max_suffix=1500, Hq=8, Hkv=8,
                         seed=77)
    inp = Inputs(w)
    g = run_gpu(inp)
    assert g["err"] == 0 and g["plan"].num_groups == 3
    cache, dev = g["cache"], g["plan"].device_tensors("cuda")
    ws = cache.workspace(w.B, w.max_blocks_per_seq)
    q = inp.q.cuda()
    out = torch.empty(w.B, w.Hq, w.D, dtype=w.src_dtype, device="cuda")
    bad = dev["seq_group"].clone()
    bad[0] = 1000
    for sg, want in ((bad, -4), (dev["seq_group"], 0)):
        pkv.paged_attention_decode_grouped(
            out, q, cache.k_pool, cache.v_pool, dev["tables"], dev["lens"], w.scale, sg,
            dev["group_members"], dev["group_prefix"], 1.0, 1.0, ws, None, dev["ungrouped"],
            dev["max_group_blocks"])
        assert pkv.get_device_error() == want


def test_reshape_and_cache_large_batch_runs_and_ragged_slots():
    """A batch large enough for the grouped slot write (>= 512 tokens): aligned
    runs of 8 consecutive slots (written as whole core matrices), runs that start
    off a multiple of 8, scattered slots, padding and one slot outside the pool;
    the pools must equal the oracle's slot writes bit for bit."""
    from oracle import cache_ops as oops
    NB, Hkv, bs, D = 96, 3, 16, 128
    rng = np.random.default_rng(5)
    slots = list(range(0, 256))                      # aligned runs
    slots += list(range(261, 261 + 203))             # a run off the 8-slot grid
    slots += [-1] * 5                                 # padding
    slots += [int(x) for x in rng.choice(np.arange(600, NB * bs), 100, replace=False)]
    slots += [NB * bs + 3]                            # outside the pool
    slots += list(range(520, 560))                    # another aligned run
    T = len(slots)
    assert T >= 512
    g = torch.Generator().manual_seed(9)
    k = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    k0 = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16)
    v0 = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16)
    kp, vp = pkv.pools_from_views(k0.cuda(), v0.cuda())
    st = torch.tensor(slots, dtype=torch.int64)
    assert pkv.get_device_error() == 0
    pkv.reshape_and_cache(k.cuda(), v.cuda(), kp, vp, st.cuda())
    assert pkv.get_device_error() == -4               # the slot outside the pool
    ok_slots = st.clone()
    ok_slots[st >= NB * bs] = -1
    kr, vr = k0.clone(), v0.clone()
    oops.reshape_and_cache(k, v, kr, vr, ok_slots, bs)
    kv, vv = pkv.pool_views(kp, vp)
    assert torch.equal(kv.cpu().view(torch.int16), kr.view(torch.int16))
    assert torch.equal(vv.cpu().view(torch.int16), vr.view(torch.int16))


def test_step_pipeline_matches_serial_steps():
    """engine.StepPipeline (uploads and downloads overlapped with the compute of
    neighbouring steps, two device buffer sets) gives, step by step, exactly the
    outputs of the same steps run one after another with device inputs."""
    from paged_kv_cache_259_gb300.engine import StepPipeline
    w = wl.shared_prefix(fork_step=True, groups=3, per_group=4, prompt=150, max_suffix=40,
                         Hq=8, Hkv=8, seed=9)
    n = 4
    gen = torch.Generator().manual_seed(4)
    qs = [torch.randn(w.B, w.Hq, w.D, generator=gen).to(torch.bfloat16) for _ in range(n)]
    ks = [torch.randn(w.B, w.Hkv, w.D, generator=gen).to(torch.bfloat16) for _ in range(n)]
    vs = [torch.randn(w.B, w.Hkv, w.D, generator=gen).to(torch.bfloat16) for _ in range(n)]
    outs = {}
    for mode in ("serial", "pipelined"):
        inp = Inputs(w)
        g = run_gpu(inp)                                   # same set-up and first step
        cache, plan = g["cache"], g["plan"]
        assert plan.num_groups > 0
        ws = cache.workspace(w.B, w.max_blocks_per_seq)
        res = []
        if mode == "serial":
            dev = plan.device_tensors("cuda")
            for i in range(n):
                o = torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16, device="cuda")
                cache.step(qs[i].cuda(), ks[i].cuda(), vs[i].cuda(), dev, o, w.scale, workspace=ws)
                res.append(o.cpu())
        else:
            host = plan.host_tensors(pin=False)
            tmpl = dict(host, q=qs[0], k_new=ks[0], v_new=vs[0],
                        max_group_blocks=plan.max_group_blocks)
            pipe = StepPipeline(cache, tmpl, torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16,
                                                         device="cuda"))
            houts = [torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16).pin_memory()
                     for _ in range(n)]
            for i in range(n):
                views = pipe.host_inputs()
                for k, t in dict(host, q=qs[i], k_new=ks[i], v_new=vs[i]).items():
                    views[k].copy_(t)
                pipe.submit(houts[i], w.scale, workspace=ws)
            torch.cuda.synchronize()
            res = houts
        assert pkv.get_device_error() == 0
        outs[mode] = res
    for a, b in zip(outs["serial"], outs["pipelined"]):
        assert torch.equal(a, b)
    assert not torch.equal(outs["serial"][0], outs["serial"][1])


@pytest.mark.parametrize("fork", [True, False], ids=["fork_step", "steady"])
def test_live_decode_pipeline_matches_planned_serial_steps(fork):
    """engine.LiveDecodePipeline (each step planned by the native manager
    straight into the pinned slab, copy-on-write pairs and prefix groups counted
    per step, uploads and downloads overlapped) gives, step by step, exactly the
    outputs and pools of plan_step + step run one after another: both as one
    library call per step (pkv_decode_pipeline_step, whose reported counts
    match the serial plans) and as plan() followed by the separate calls."""
    from paged_kv_cache_259_gb300.engine import LiveDecodePipeline, PagedKVCache
    w = wl.shared_prefix(fork_step=fork, groups=3, per_group=4, prompt=150, max_suffix=40,
                         Hq=16, Hkv=8, seed=11)
    n, mb = 6, w.max_blocks_per_seq + 2
    gen = torch.Generator().manual_seed(5)
    qs = [torch.randn(w.B, w.Hq, w.D, generator=gen).to(torch.bfloat16) for _ in range(n)]
    ks = [torch.randn(w.B, w.Hkv, w.D, generator=gen).to(torch.bfloat16) for _ in range(n)]
    vs = [torch.randn(w.B, w.Hkv, w.D, generator=gen).to(torch.bfloat16) for _ in range(n)]
    k_src, v_src = w.past_pools()
    outs, pools, counts, native_counts = {}, {}, [], []
    for mode in ("serial", "live", "live_planned"):
        cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, torch.bfloat16, w.free_order, "cuda")
        cache.load(k_src, v_src)
        cache.apply_copies(cache.replay(w.script))
        ws = cache.workspace(w.B, mb)
        if mode == "serial":
            res = []
            for i in range(n):
                plan = cache.plan_step(w.step_seqs, max_blocks=mb)
                counts.append((len(plan.pairs), plan.num_groups))
                o = torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16, device="cuda")
                cache.step(qs[i].cuda(), ks[i].cuda(), vs[i].cuda(), plan.device_tensors("cuda"),
                           o, w.scale, workspace=ws)
                res.append(o.cpu())
        else:
            pipe = LiveDecodePipeline(cache, w.step_seqs, qs[0], ks[0], vs[0],
                                      torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16,
                                                  device="cuda"), mb)
            res = [torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16).pin_memory()
                   for _ in range(n)]
            for i in range(n):
                views = pipe.host_inputs()
                views["q"].copy_(qs[i])
                views["k_new"].copy_(ks[i])
                views["v_new"].copy_(vs[i])
                if mode == "live_planned":
                    pipe.plan()
                pipe.submit(res[i], w.scale, workspace=ws)
                if mode == "live":
                    native_counts.append(pipe.last_counts[:2])
            torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        outs[mode] = res
        pools[mode] = (cache.k_pool.cpu(), cache.v_pool.cpu())
    for mode in ("live", "live_planned"):
        for a, b in zip(outs["serial"], outs[mode]):
            assert torch.equal(a, b)
        assert torch.equal(pools["serial"][0], pools[mode][0])
        assert torch.equal(pools["serial"][1], pools[mode][1])
    assert native_counts == counts
    assert all(g > 0 for _, g in counts)
    if fork:
        assert counts[0][0] == 9 and all(p == 0 for p, _ in counts[1:])
