"""The seeded synthetic workloads follow their stated recipes, so the benchmark
measures what its description says. Each test checks one workload: shapes,
length distributions, pool sizes, seeds, scales and script structure.
Distribution checks allow four standard errors of sampling.
"""
import math

import numpy as np

import pkv_workloads as wl


def blocks(lens, bs):
    return int(sum(-(-int(L) // bs) for L in lens))


def appended(w):
    """Tokens each sequence holds before the step, from the script's appends."""
    n = {}
    for op in w.script:
        if op[0] == "add":
            n[op[1]] = 0
        elif op[0] == "append":
            n[op[1]] += op[2]
        elif op[0] == "fork":
            n[op[2]] = n[op[1]]
    return n


def is_permutation(order, n):
    return sorted(np.asarray(order).tolist()) == list(range(n))


def test_tiny_fp32():
    w = wl.tiny_fp32()
    assert (w.B, w.Hq, w.Hkv, w.D, w.bs, w.NB, w.seed, w.kv_dtype) == \
        (4, 4, 4, 64, 16, 64, 0, "f32")
    assert list(w.final_lens) == [1, 17, 40, 100] and w.scale == 1 / 8
    assert is_permutation(w.free_order, 64)


def test_llama13b_lengths_uniform_and_pool_ten_percent_over():
    w = wl.llama13b_mha_bf16()
    assert (w.B, w.Hq, w.Hkv, w.D, w.bs, w.seed, w.kv_dtype) == (64, 40, 40, 128, 16, 1, "bf16")
    L = w.final_lens
    assert L.min() >= 128 and L.max() <= 2048
    se = (2048 - 128) / math.sqrt(12) / math.sqrt(w.B)
    assert abs(L.mean() - (128 + 2048) / 2) < 4 * se
    assert w.NB == math.ceil(1.1 * blocks(L, 16)) and is_permutation(w.free_order, w.NB)
    assert math.isclose(w.scale, 1 / math.sqrt(128))
    n = appended(w)
    assert all(n[s] + 1 == L[i] for i, s in enumerate(w.step_seqs))   # the step adds one


def test_gqa_chat_lognormal_median_400_clipped():
    w = wl.gqa_chat_bf16()
    assert (w.B, w.Hq, w.Hkv, w.D, w.bs, w.seed) == (256, 32, 8, 128, 16, 2)
    L = w.final_lens
    assert L.min() >= 16 and L.max() <= 4096
    se_log_median = 1.2533 / math.sqrt(w.B)              # sigma 1 in log space
    assert abs(math.log(np.median(L)) - math.log(400)) < 4 * se_log_median
    assert w.NB == math.ceil(1.1 * blocks(L, 16))


def test_shared_prefix_groups_share_a_520_token_prompt():
    for fork in (False, True):
        w = wl.shared_prefix_bf16(fork_step=fork)
        assert (w.B, w.Hq, w.Hkv, w.D, w.bs, w.seed) == (256, 40, 40, 128, 16, 3)
        forks = [op for op in w.script if op[0] == "fork"]
        assert len(forks) == 64 * 3
        assert all(op[1] % 4 == 0 and op[2] // 4 == op[1] // 4 for op in forks)
        L = w.final_lens
        if fork:
            assert (L == 521).all()                          # the step writes token 521
        else:
            assert L.min() >= 521 and L.max() <= 520 + 256 + 1
            se = 256 / math.sqrt(12) / math.sqrt(w.B)
            assert abs((L - 521).mean() - 128) < 4 * se


def test_long_fp8_contexts():
    for bs in (16, 32):
        w = wl.CONFIGS[f"long_fp8_bs{bs}"]()
        assert (w.B, w.Hq, w.Hkv, w.D, w.bs, w.seed, w.kv_dtype) == (16, 32, 8, 128, bs, 4, "e4m3")
        assert (w.final_lens == 32768).all()


def test_beam_search_requests_and_steps():
    w = wl.beam_search_bf16()
    assert (w.B, w.Hq, w.Hkv, w.D, w.bs, w.seed) == (64, 40, 40, 128, 16, 8)
    P = w.notes["prompt_lens"]
    assert len(P) == 16 and P.min() >= 128 and P.max() <= 2048
    assert list(w.final_lens) == list(np.repeat(P + 128 + 1, 4))
    beams = [op for op in w.script if op[0] == "beam"]
    assert len(beams) == 128 + 1                             # every generated token, then the step
    for _, old, parents, new in beams:
        assert len(new) == 64 and len(parents) == 64
        for i, p in enumerate(parents):                      # a beam's parent is of its request
            assert (i // 4) * (len(old) // 16) <= p < (i // 4 + 1) * (len(old) // 16)


def test_swap_victims_are_the_newest_sequences():
    sw = wl.swap_llama13b_bf16()
    assert sw.victims == list(range(48, 64))
    assert sw.num_host_blocks == math.ceil(1.1 * sw.victim_blocks)


def test_prefill_contexts_and_chunks():
    for name, ctx_max, Hq, Hkv, seed in (("prefill_llama13b_bf16", 1536, 40, 40, 5),
                                          ("prefill_gqa_bf16", 3584, 32, 8, 6)):
        w = wl.PREFILL_CONFIGS[name]()
        assert (w.B, w.Hq, w.Hkv, w.D, w.bs, w.seed) == (16, Hq, Hkv, 128, 16, seed)
        assert (w.chunks == 512).all() and w.T == 16 * 512
        ctx = w.final_lens - w.chunks
        assert ctx.min() >= 0 and ctx.max() <= ctx_max
        assert [appended(w)[b] for b in range(w.B)] == list(ctx)


def test_system_prompt_workload():
    w = wl.PROMPT_CONFIGS["prefill_system_prompt_bf16"]()
    assert (w.B, w.Hq, w.Hkv, w.D, w.bs, w.seed) == (64, 40, 40, 128, 16, 7)
    assert len(w.warm) == 1 and len(w.warm[0]) == 1024
    assert all(len(p) == 1024 + 256 and np.array_equal(p[:1024], w.warm[0]) for p in w.prompts)
    ids = np.concatenate(w.prompts)
    assert ids.min() >= 0 and ids.max() < 32000
