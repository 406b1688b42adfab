"""The bench's algorithmic byte and FLOP counts (the numerators of every
roofline figure), checked on small cases against counts made the plain way:
token by token, block by block. Host logic only."""
import math

import numpy as np
import torch

import bench
import pkv_workloads as wl


def test_decode_step_bytes_count_each_token_and_each_shared_block_once():
    w = wl.tiny_fp32()                                  # f32: 4 bytes per element
    B, Hq, Hkv, D, bs = w.B, w.Hq, w.Hkv, w.D, w.bs
    lens = np.array([1, 17, 40, 100])
    MB = 7
    tables = np.full((B, MB), -1, dtype=np.int32)
    nxt = 0
    for b, L in enumerate(lens):
        for j in range(-(-int(L) // bs)):
            tables[b, j] = nxt
            nxt += 1
    nb = bench.step_bytes(w, tables, lens, num_pairs=0)
    per_tok = 2 * Hkv * D * 4                           # one token's K and V
    plain = 0
    for b in range(B):
        for t in range(int(lens[b])):
            plain += per_tok                             # every cached token once
    plain += 2 * B * Hq * D * 4 + tables.size * 4 + B * 4   # q, out, tables, lengths
    assert nb["decode"] == plain == nb["decode_logical"]
    assert nb["reshape"] == B * Hkv * D * 2 * (4 + 4) + B * 8
    assert nb["copy"] == 0 and nb["total"] == nb["decode"] + nb["reshape"]
    # two sequences pointing at the same physical block 0 (full) and their own
    # partial block: the shared block's bytes count once in `decode`
    t2 = np.array([[0, 1], [0, 2]], dtype=np.int32)
    l2 = np.array([bs + 3, bs + 5])
    w2 = wl.prefill_workload("x", 0, l2, Hq, Hkv, D, bs, torch.float32, "f32", 1.0)
    nb2 = bench.step_bytes(w2, t2, l2, num_pairs=1)
    unique = bs + 3 + 5
    qo = 2 * 2 * Hq * D * 4 + t2.size * 4 + 2 * 4
    assert nb2["decode"] == unique * per_tok + qo
    assert nb2["decode_logical"] == int(l2.sum()) * per_tok + qo
    assert nb2["copy"] == 2 * 2 * Hkv * bs * D * 4 + 16   # one pair: both pools read + written


def test_prefill_flops_count_every_visible_key():
    w = wl.chunked_prefill("acct", 3, [0, 5, 40], [7, 1, 30], 8, 2, 64, 16)
    plain = 0
    for L, C in zip(w.final_lens, w.chunks):
        for i in range(int(C)):
            p = int(L) - int(C) + i                      # the token's position
            plain += (p + 1) * 4 * w.D * w.Hq             # Q.K and P.V: 2*D multiply-adds each
    assert math.isclose(bench.prefill_flops(w), plain, rel_tol=0, abs_tol=0.5)


def test_kernel_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """bench.code_hash: comments and blank lines do not change it, code does."""
    csrc = tmp_path / "paged_kv_cache_259_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "k.cu").write_text("// a kernel\nint f(int x) {\n  return x + 1;  // one\n}\n")
    h0 = bench.code_hash(["k.cu"])
    (csrc / "k.cu").write_text("/* the same kernel,\n   described */\n\nint f(int x) {\n  return x + 1;\n}\n")
    assert bench.code_hash(["k.cu"]) == h0
    (csrc / "k.cu").write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.code_hash(["k.cu"]) != h0
