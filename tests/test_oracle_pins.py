"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it does not compute itself: the
worked example of the glossary page "PagedAttention" and its printed result,
a library implementation of attention on contiguous K/V (torch's
scaled_dot_product_attention in float64), closed forms, brute force over every
block table of a tiny pool, torch's own float8_e4m3fn conversion, and the
reference-count / copy-on-write invariants the pages state.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as oatt
from oracle import cache_ops as oops
from oracle import fp8_e4m3 as ofp8
from oracle.block_manager import BlockManager, PoolExhausted

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [int(x) for x in rest]
    return vals


# ---------------------------------------------------------------- worked example
def test_snippet_replay():
    """The glossary's 40-token example: table [41, 7, 19], keys intact, 8 vs 2,008."""
    g = read_golden("snippet_40_tokens.txt")
    bs, d, nb, n = g["block_size"][0], g["head_dim"][0], g["pool_blocks"][0], g["tokens"][0]
    bm = BlockManager(nb, bs, g["free_blocks"])
    bm.add_seq(0)
    slots = [bm.append_slot(0)[0] for _ in range(n)]
    table = bm.block_table(0)
    assert table == g["expected_block_table"]
    assert bm.num_free() == len(g["free_blocks"]) - len(table)

    keys = torch.randn(n, d, generator=torch.Generator().manual_seed(0))
    pool = torch.zeros(nb, 1, bs, d)
    vpool = torch.zeros(nb, 1, bs, d)
    oops.reshape_and_cache(keys[:, None, :], keys[:, None, :], pool, vpool,
                           torch.tensor(slots), bs)
    # the example's layout, read off directly: consecutive 16-token chunks of the
    # request sit in blocks 41, 7 and 19, in order
    assert torch.equal(pool[41, 0], keys[0:16])
    assert torch.equal(pool[7, 0], keys[16:32])
    assert torch.equal(pool[19, 0, :8], keys[32:40])
    assert torch.count_nonzero(pool[19, 0, 8:]) == 0
    gathered = oatt.gather(pool, table, n, 0, bs)
    assert torch.equal(gathered, keys) == bool(g["expected_keys_intact"][0])
    assert len(table) * bs - n == g["expected_unused_slots"][0]
    assert g["reservation_tokens"][0] - n == g["expected_unused_reserved"][0]


# ---------------------------------------------------------------- helpers
def scatter_blockwise(Kc, table, pool, bs):
    """Place contiguous rows ``Kc [L, Hkv, D]`` into ``pool`` chunk by chunk:
    chunk j (rows j*bs .. j*bs+bs-1) goes to physical block table[j]."""
    L = Kc.shape[0]
    for j in range(-(-L // bs)):
        rows = Kc[j * bs:(j + 1) * bs]
        pool[table[j], :, :rows.shape[0], :] = rows.transpose(0, 1)


def sdpa_reference(q, Kc, Vc, scale):
    """torch SDPA in float64 on contiguous K/V; query head h uses KV head h // G."""
    Hq, D = q.shape
    L, Hkv, _ = Kc.shape
    G = Hq // Hkv
    if L == 0:
        return torch.zeros(Hq, D, dtype=torch.float64)
    K = Kc.to(torch.float64).transpose(0, 1).repeat_interleave(G, dim=0)  # [Hq, L, D]
    V = Vc.to(torch.float64).transpose(0, 1).repeat_interleave(G, dim=0)
    o = F.scaled_dot_product_attention(q.to(torch.float64)[:, None, :], K, V, scale=scale)
    return o[:, 0, :]


def random_case(seed, lens, Hq, Hkv, D, bs, extra_blocks=5, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    need = sum(-(-L // bs) for L in lens)
    NB = need + extra_blocks
    perm = rng.permutation(NB)
    MB = max(1, max(-(-L // bs) for L in lens))
    tables = np.full((len(lens), MB), -1, dtype=np.int64)
    kpool = torch.randn(NB, Hkv, bs, D, generator=g).to(dtype)
    vpool = torch.randn(NB, Hkv, bs, D, generator=g).to(dtype)
    conts = []
    pos = 0
    for b, L in enumerate(lens):
        nb = -(-L // bs)
        tables[b, :nb] = perm[pos:pos + nb]
        pos += nb
        Kc = torch.randn(L, Hkv, D, generator=g).to(dtype)
        Vc = torch.randn(L, Hkv, D, generator=g).to(dtype)
        scatter_blockwise(Kc, tables[b], kpool, bs)
        scatter_blockwise(Vc, tables[b], vpool, bs)
        conts.append((Kc, Vc))
    q = torch.randn(len(lens), Hq, D, generator=g).to(dtype)
    return q, kpool, vpool, tables, np.array(lens), conts


# ---------------------------------------------------------------- paged == contiguous
@pytest.mark.parametrize("Hq,Hkv,D,bs", [(4, 4, 64, 16), (8, 2, 32, 4), (6, 3, 16, 1),
                                          (8, 1, 64, 32), (4, 4, 128, 2)])
def test_paged_equals_contiguous_sdpa(Hq, Hkv, D, bs):
    lens = [1, 2, bs - 1 if bs > 1 else 3, bs, bs + 1, 3 * bs + 5, 0, 57]
    q, kp, vp, tables, sl, conts = random_case(Hq * 100 + D + bs, lens, Hq, Hkv, D, bs)
    scale = 1.0 / math.sqrt(D)
    out = oatt.paged_decode(q, kp, vp, tables, sl, scale, bs)
    for b, (Kc, Vc) in enumerate(conts):
        ref = sdpa_reference(q[b], Kc, Vc, scale).numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_paged_equals_contiguous_bf16_values():
    q, kp, vp, tables, sl, conts = random_case(7, [40, 100, 17], 8, 2, 128, 16,
                                               dtype=torch.bfloat16)
    out = oatt.paged_decode(q, kp, vp, tables, sl, 0.125, 16)
    for b, (Kc, Vc) in enumerate(conts):
        np.testing.assert_allclose(out[b], sdpa_reference(q[b], Kc, Vc, 0.125).numpy(),
                                   rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- closed forms
def test_single_token_returns_its_value():
    q, kp, vp, tables, sl, conts = random_case(3, [1, 1], 4, 2, 64, 16)
    out = oatt.paged_decode(q, kp, vp, tables, sl, 0.3, 16, v_scale=1.0)
    for b, (Kc, Vc) in enumerate(conts):
        for h in range(4):
            assert np.array_equal(out[b, h], Vc[0, h // 2].double().numpy())


def test_zero_query_and_equal_keys_give_mean_of_values():
    q, kp, vp, tables, sl, conts = random_case(4, [37, 16], 2, 2, 32, 8)
    zero_q = torch.zeros_like(q)
    out = oatt.paged_decode(zero_q, kp, vp, tables, sl, 1.0, 8)
    for b, (Kc, Vc) in enumerate(conts):
        np.testing.assert_allclose(out[b], Vc.double().mean(0).numpy(), rtol=0, atol=1e-14)
    # all keys equal: scores equal, uniform weights, whatever q is
    K_eq = torch.randn(1, 2, 32).expand(37, 2, 32).contiguous()
    table = list(range(5))
    kpool = torch.zeros(5, 2, 8, 32)
    scatter_blockwise(K_eq, table, kpool, 8)
    Vc = conts[0][1]
    vpool = torch.zeros(5, 2, 8, 32)
    scatter_blockwise(Vc, table, vpool, 8)
    out = oatt.paged_decode(q[:1], kpool, vpool, [table], [37], 0.7, 8)
    np.testing.assert_allclose(out[0], Vc.double().mean(0).numpy(), rtol=0, atol=1e-14)


def test_two_tokens_logistic_weight():
    """Two tokens: out = sigma(s0 - s1) v0 + sigma(s1 - s0) v1."""
    D = 8
    k = np.array([[0.5] * D, [-0.25] * D])
    v = np.array([[1.0] * D, [3.0] * D])
    qv = np.linspace(-1, 1, D)
    qv = qv + 0.3
    s = 0.5 * (k @ qv)
    w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    out = oatt.decode_one(qv, k, v, 0.5)
    np.testing.assert_allclose(out, w0 * v[0] + (1 - w0) * v[1], rtol=1e-15)


def test_scales_fold_linearly():
    """k_scale multiplies the logits, v_scale the output (value = code * scale)."""
    q, kp, vp, tables, sl, conts = random_case(11, [23], 2, 2, 16, 4)
    a = oatt.paged_decode(q, kp * 2.0, vp * 4.0, tables, sl, 0.25, 4)
    b = oatt.paged_decode(q, kp, vp, tables, sl, 0.25, 4, k_scale=2.0, v_scale=4.0)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- brute force
def test_every_block_table_of_a_tiny_pool_gives_the_same_result():
    """Pool of 4 blocks of 2 slots, 3-token sequence: all 12 ordered choices of 2
    distinct blocks hold the same contiguous K/V and must give identical output,
    equal to SDPA on the contiguous rows."""
    g = torch.Generator().manual_seed(5)
    Kc = torch.randn(3, 1, 4, generator=g)
    Vc = torch.randn(3, 1, 4, generator=g)
    q = torch.randn(1, 2, 4, generator=g)
    ref = sdpa_reference(q[0], Kc, Vc, 0.5).numpy()
    outs = []
    for a in range(4):
        for b in range(4):
            if a == b:
                continue
            kp = torch.randn(4, 1, 2, 4, generator=g)   # junk everywhere else
            vp = torch.randn(4, 1, 2, 4, generator=g)
            scatter_blockwise(Kc, [a, b], kp, 2)
            scatter_blockwise(Vc, [a, b], vp, 2)
            outs.append(oatt.paged_decode(q, kp, vp, [[a, b]], [3], 0.5, 2))
    assert len(outs) == 12
    for o in outs:
        assert np.array_equal(o, outs[0])
    np.testing.assert_allclose(outs[0][0], ref, rtol=1e-13, atol=1e-14)


def test_relabelling_physical_blocks_changes_nothing():
    q, kp, vp, tables, sl, conts = random_case(9, [50, 3, 31], 4, 4, 32, 8)
    NB = kp.shape[0]
    perm = np.random.default_rng(1).permutation(NB)        # new id of old block i
    kp2 = torch.empty_like(kp)
    vp2 = torch.empty_like(vp)
    kp2[torch.from_numpy(perm)] = kp
    vp2[torch.from_numpy(perm)] = vp
    t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1)
    a = oatt.paged_decode(q, kp, vp, tables, sl, 0.2, 8)
    b = oatt.paged_decode(q, kp2, vp2, t2, sl, 0.2, 8)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- FP8 E4M3
def test_e4m3_decode_all_codes_match_torch_and_spec_anchors():
    codes = np.arange(256, dtype=np.uint8)
    mine = ofp8.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(mine[ok], lib[ok])
    assert np.isnan(mine[0x7F]) and np.isnan(mine[0xFF]) and np.isnan(mine).sum() == 2
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6 and mine[0x07] == 7 * 2.0 ** -9
    assert mine[0x38] == 1.0 and mine[0x00] == 0.0 and math.copysign(1, mine[0x80]) < 0


def test_e4m3_encode_roundtrip_ties_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = ofp8.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(ofp8.e4m3_encode(vals), codes)
    # every midpoint between neighbouring magnitudes rounds to the even code
    mags = ofp8.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (mags[:-1] + mags[1:]) / 2)  # exact
    got = ofp8.e4m3_encode(mids).astype(np.int64)
    lo = np.arange(126)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1))
    # just off the midpoint goes to the nearer one
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(-np.inf))
    assert np.array_equal(ofp8.e4m3_encode(up).astype(np.int64), lo + 1)
    assert np.array_equal(ofp8.e4m3_encode(dn).astype(np.int64), lo)
    # saturation (satfinite): 448 and beyond stay 448
    big = np.array([448.0, 449.0, 463.9, 464.0, 1e6, 3e38, -500.0], dtype=np.float32)
    assert list(ofp8.e4m3_encode(big)) == [0x7E] * 6 + [0xFE]
    # negative values rounding to zero keep their sign
    assert list(ofp8.e4m3_encode(np.array([-1e-9, 1e-9, -0.0, 0.0], np.float32))) == \
        [0x80, 0x00, 0x80, 0x00]


def test_e4m3_encode_matches_torch_rne_cast_below_overflow():
    g = torch.Generator().manual_seed(0)
    x = torch.cat([torch.randn(200000, generator=g) * s for s in (1e-3, 0.05, 1, 30, 150)])
    x = x.clamp(-463.0, 463.0)
    lib = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ofp8.e4m3_encode(x.numpy()), lib)


def test_e4m3_quantize_divides_in_float32():
    x = np.array([1.0, -3.0, 0.1], dtype=np.float32)
    s = 0.0123
    q = (x / np.float32(s)).astype(np.float32)
    assert np.array_equal(ofp8.e4m3_quantize(x, s), ofp8.e4m3_encode(q))
    lib = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ofp8.e4m3_quantize(x, s), lib)


def test_e4m3_quantize_rounds_the_scale_to_float32_like_torch():
    """The kernel receives a float32 scale and divides in float32. Inputs a few
    float32 steps from tie points, with a scale float32 cannot hold exactly
    (0.1), tell that apart from dividing by the exact scale. Every code must
    equal torch's float32 divide followed by its float8_e4m3fn cast."""
    s = 0.1
    s32 = torch.tensor(s, dtype=torch.float32)
    mags = ofp8.e4m3_decode(np.arange(127, dtype=np.uint8))
    ties = (mags[:-1] + mags[1:]) / 2
    base = torch.from_numpy(ties[1:]).float() * s32                 # rounded to float32
    xs = [base]
    for _ in range(3):                                            # 3 steps either way
        xs.append(torch.nextafter(xs[-1], torch.full_like(base, float("inf"))))
    lo = base
    for _ in range(3):
        lo = torch.nextafter(lo, torch.full_like(base, float("-inf")))
        xs.append(lo)
    x = torch.cat(xs)
    lib = (x / s32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ofp8.e4m3_quantize(x.numpy(), s), lib)
    exact = ofp8.e4m3_encode((x.double().numpy() / s).astype(np.float32))
    assert (exact != lib).sum() > 0          # the cases do tell the two apart


def test_fp8_paged_attention_equals_sdpa_on_library_dequantised_values():
    q, kp, vp, tables, sl, conts = random_case(13, [40, 77], 8, 2, 64, 16)
    ks, vs = 4.5 / 448, 4.2 / 448
    kq = torch.from_numpy(ofp8.e4m3_quantize(kp.numpy(), ks))
    vq = torch.from_numpy(ofp8.e4m3_quantize(vp.numpy(), vs))
    out = oatt.paged_decode(q, kq, vq, tables, sl, 0.125, 16, k_scale=ks, v_scale=vs)
    kd = kq.view(torch.float8_e4m3fn).to(torch.float64) * ks
    vd = vq.view(torch.float8_e4m3fn).to(torch.float64) * vs
    for b in range(2):
        L = int(sl[b])
        nbk = -(-L // 16)
        Kc = torch.cat([kd[tables[b][j]].transpose(0, 1) for j in range(nbk)])[:L]
        Vc = torch.cat([vd[tables[b][j]].transpose(0, 1) for j in range(nbk)])[:L]
        np.testing.assert_allclose(out[b], sdpa_reference(q[b], Kc, Vc, 0.125).numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_reshape_and_cache_fp8_bytes_match_torch_cast():
    g = torch.Generator().manual_seed(2)
    k = torch.randn(5, 2, 32, generator=g).to(torch.bfloat16)
    v = torch.randn(5, 2, 32, generator=g).to(torch.bfloat16)
    kp = torch.zeros(4, 2, 4, 32, dtype=torch.uint8)
    vp = torch.zeros(4, 2, 4, 32, dtype=torch.uint8)
    slots = torch.tensor([3, 9, -1, 14, 0])
    ks, vs = 0.01, 0.02
    oops.reshape_and_cache(k, v, kp, vp, slots, 4, ks, vs)
    for i, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        ref = (k[i].float() / ks).to(torch.float8_e4m3fn).view(torch.uint8)
        assert torch.equal(kp[s // 4, :, s % 4], ref)
        ref = (v[i].float() / vs).to(torch.float8_e4m3fn).view(torch.uint8)
        assert torch.equal(vp[s // 4, :, s % 4], ref)
    # the padding token (slot -1) wrote nothing: only the 4 real slots are set
    written = (kp.permute(0, 2, 1, 3).reshape(16, -1) != 0).any(1)
    assert sorted(torch.nonzero(written).flatten().tolist()) == [0, 3, 9, 14]


# ---------------------------------------------------------------- cache ops
def test_copy_blocks_copies_whole_blocks_only():
    g = torch.Generator().manual_seed(1)
    kp = torch.randn(6, 2, 4, 8, generator=g).to(torch.bfloat16)
    vp = torch.randn(6, 2, 4, 8, generator=g).to(torch.bfloat16)
    k0, v0 = kp.clone(), vp.clone()
    oops.copy_blocks(kp, vp, [(1, 4), (2, 5)])
    assert torch.equal(kp[4], k0[1]) and torch.equal(vp[5], v0[2])
    for i in (0, 1, 2, 3):
        assert torch.equal(kp[i], k0[i]) and torch.equal(vp[i], v0[i])
    with pytest.raises(IndexError):
        oops.copy_blocks(kp, vp, [(0, 6)])


def test_reshape_and_cache_rejects_slot_outside_pool():
    kp = torch.zeros(2, 1, 4, 8)
    with pytest.raises(IndexError):
        oops.reshape_and_cache(torch.ones(1, 1, 8), torch.ones(1, 1, 8), kp, kp.clone(),
                               torch.tensor([8]), 4)


# ---------------------------------------------------------------- block manager
def check_invariants(bm):
    used = {b for b in range(bm.num_blocks) if bm.ref[b] > 0}
    free = set(bm.free)
    assert len(free) == len(bm.free)                       # no duplicates
    assert not (used & free)
    assert all(r >= 0 for r in bm.ref)
    assert sum(bm.ref) == sum(len(t) for t in bm.tables.values())
    for sid, t in bm.tables.items():
        L = bm.lens[sid]
        assert len(t) == -(-L // bm.block_size)
        assert len(t) * bm.block_size - L < bm.block_size   # waste below one block


def test_block_manager_random_ops_keep_invariants():
    rng = np.random.default_rng(123)
    for trial in range(20):
        nb, bs = int(rng.integers(8, 64)), int(rng.choice([1, 2, 4, 16]))
        bm = BlockManager(nb, bs, rng.permutation(nb))
        all_ids = set(range(nb))
        next_id = 0
        for _ in range(400):
            op = rng.integers(0, 10)
            live = list(bm.tables)
            try:
                if op == 0 or not live:
                    bm.add_seq(next_id)
                    next_id += 1
                elif op == 1:
                    bm.fork(int(rng.choice(live)), next_id)
                    next_id += 1
                elif op == 2:
                    bm.free_seq(int(rng.choice(live)))
                else:
                    sid = int(rng.choice(live))
                    free_before = list(bm.free)
                    last = bm.tables[sid][-1] if bm.tables[sid] else None
                    ref_last = bm.ref[last] if last is not None else None
                    slot, cow = bm.append_slot(sid)
                    blk = slot // bs
                    assert blk in bm.tables[sid]
                    assert bm.ref[blk] == 1          # never write into a shared block
                    if cow is not None:
                        src, dst = cow
                        assert src == last and dst == free_before[0] and src != dst
                        assert bm.ref[src] == ref_last - 1 and blk == dst
            except PoolExhausted:
                assert bm.num_free() == 0
            check_invariants(bm)
            used = {b for b in all_ids if bm.ref[b] > 0}
            assert used | set(bm.free) == all_ids


def test_block_manager_fork_then_write_copies_only_the_partial_block():
    bm = BlockManager(16, 4, range(16))
    bm.add_seq(0)
    for _ in range(10):                     # blocks 0, 1, 2 (2 holds 2 tokens)
        bm.append_slot(0)
    bm.fork(0, 1)
    assert [bm.refcount(b) for b in (0, 1, 2)] == [2, 2, 2]
    slot, cow = bm.append_slot(1)           # child writes into shared block 2
    assert cow == (2, 3) and slot == 3 * 4 + 2
    assert bm.block_table(1) == [0, 1, 3] and bm.block_table(0) == [0, 1, 2]
    assert bm.refcount(2) == 1 and bm.refcount(3) == 1
    slot, cow = bm.append_slot(0)           # last owner writes in place
    assert cow is None and slot == 2 * 4 + 2
    bm.free_seq(0)
    assert bm.refcount(0) == 1 and bm.refcount(2) == 0 and bm.free[-1] == 2


def test_block_manager_exhaustion_is_an_error():
    bm = BlockManager(2, 2, [1, 0])
    bm.add_seq(0)
    for _ in range(4):
        bm.append_slot(0)
    with pytest.raises(PoolExhausted):
        bm.append_slot(0)


def test_llama13b_kv_bytes_per_sequence_closed_form():
    """The glossary's "up to 1.7 GB" for one LLaMA-13B sequence: 40 layers x 40
    heads x 128 dims x (K, V) x 2 bytes per token, 2,048 tokens."""
    per_token = 40 * 40 * 128 * 2 * 2
    assert per_token == 819200
    assert abs(per_token * 2048 / 1e9 - 1.7) < 0.05


# ---------------------------------------------------------------- chunked prefill
def prefill_case(seed, lens, chunks, Hq, Hkv, D, bs, dtype=torch.float32):
    """random_case plus a query chunk per sequence: q [sum(chunks), Hq, D]."""
    q1, kp, vp, tables, sl, conts = random_case(seed, lens, Hq, Hkv, D, bs, dtype=dtype)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn(int(sum(chunks)), Hq, D, generator=g).to(dtype)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int64)
    return q, kp, vp, tables, sl, qs, conts


def sdpa_causal_reference(qc, Kc, Vc, scale):
    """torch SDPA in float64 with an explicit mask: the chunk's C queries are the
    last C positions of the L keys (query i may see keys 0 .. L - C + i)."""
    C, Hq, D = qc.shape
    L, Hkv, _ = Kc.shape
    G = Hq // Hkv
    K = Kc.to(torch.float64).transpose(0, 1).repeat_interleave(G, dim=0)   # [Hq, L, D]
    V = Vc.to(torch.float64).transpose(0, 1).repeat_interleave(G, dim=0)
    Q = qc.to(torch.float64).transpose(0, 1)                                 # [Hq, C, D]
    allowed = torch.arange(L)[None, :] <= (L - C + torch.arange(C))[:, None]
    o = F.scaled_dot_product_attention(Q, K, V, attn_mask=allowed, scale=scale)
    return o.transpose(0, 1)                                                 # [C, Hq, D]


@pytest.mark.parametrize("Hq,Hkv,D,bs", [(4, 4, 64, 16), (8, 2, 32, 4), (6, 3, 16, 1),
                                          (8, 1, 64, 32)])
def test_prefill_equals_contiguous_causal_sdpa(Hq, Hkv, D, bs):
    lens = [1, 7, bs + 3, 3 * bs + 5, 57, 40]
    chunks = [1, 7, 2, 3 * bs + 5, 20, 1]          # whole prompts, partial chunks, single tokens
    q, kp, vp, tables, sl, qs, conts = prefill_case(Hq * 10 + D + bs, lens, chunks, Hq, Hkv, D, bs)
    scale = 1.0 / math.sqrt(D)
    out = oatt.paged_prefill(q, kp, vp, tables, sl, qs, scale, bs)
    for b, (Kc, Vc) in enumerate(conts):
        ref = sdpa_causal_reference(q[qs[b]:qs[b + 1]], Kc, Vc, scale).numpy()
        np.testing.assert_allclose(out[qs[b]:qs[b + 1]], ref, rtol=1e-12, atol=1e-12)


def test_prefill_of_one_token_per_sequence_is_decode():
    lens = [1, 17, 40, 100]
    q, kp, vp, tables, sl, qs, _ = prefill_case(3, lens, [1, 1, 1, 1], 8, 2, 64, 16)
    np.testing.assert_array_equal(oatt.paged_prefill(q, kp, vp, tables, sl, qs, 0.2, 16),
                                  oatt.paged_decode(q, kp, vp, tables, sl, 0.2, 16))


def test_prefill_equal_keys_give_running_mean_of_values():
    """All keys equal: query at position p weights keys 0..p equally, so its
    output is the mean of V over 0..p (an off-by-one in the causal bound fails)."""
    L, C, bs, D = 37, 29, 4, 8
    q, kp, vp, tables, sl, qs, conts = prefill_case(11, [L], [C], 2, 2, D, bs,
                                                    dtype=torch.float64)
    kp[:] = 0.25
    out = oatt.paged_prefill(q, kp, vp, tables, sl, qs, 1.0, bs)
    Vc = conts[0][1].to(torch.float64).numpy()                 # [L, Hkv, D]
    for i in range(C):
        p = L - C + i
        np.testing.assert_allclose(out[i], Vc[:p + 1].mean(axis=0), rtol=1e-13, atol=1e-13)


def test_prefill_first_prompt_token_returns_its_value():
    q, kp, vp, tables, sl, qs, conts = prefill_case(5, [9], [9], 4, 2, 16, 4, dtype=torch.float64)
    out = oatt.paged_prefill(q, kp, vp, tables, sl, qs, 0.5, 4)
    Vc = conts[0][1]
    np.testing.assert_array_equal(out[0], Vc[0].repeat_interleave(2, dim=0).numpy())


def test_prefill_in_chunks_equals_prefill_in_one_pass():
    """Causal attention over a prompt does not depend on how the prompt is cut
    into chunks: chunks [11, 1, 20] against the same cache, each with the
    sequence length it would have after its own write, give the rows of one
    32-token pass."""
    L, bs = 32, 8
    q, kp, vp, tables, sl, qs, _ = prefill_case(21, [L], [L], 6, 3, 32, bs)
    whole = oatt.paged_prefill(q, kp, vp, tables, sl, qs, 0.17, bs)
    start = 0
    for c in (11, 1, 20):
        part = oatt.paged_prefill(q[start:start + c], kp, vp, tables, np.array([start + c]),
                                  np.array([0, c]), 0.17, bs)
        np.testing.assert_allclose(part, whole[start:start + c], rtol=1e-13, atol=1e-13)
        start += c


def test_prefill_rejects_chunk_longer_than_sequence():
    q, kp, vp, tables, sl, qs, _ = prefill_case(2, [5], [5], 2, 2, 8, 4)
    with pytest.raises(ValueError):
        oatt.paged_prefill(q, kp, vp, tables, np.array([4]), qs, 1.0, 4)


# ---------------------------------------------------------------- prefix caching
from oracle.prefix_cache import PrefixCachingBlockManager  # noqa: E402


class Shadow:
    """What every slot of the pool holds (the token whose K/V was written
    there), updated by the slot writes and block copies a manager asks for."""

    def __init__(self, num_blocks, bs):
        self.bs = bs
        self.slot = [None] * (num_blocks * bs)

    def write(self, slot, token):
        self.slot[slot] = token

    def copy(self, src, dst):
        bs = self.bs
        self.slot[dst * bs:(dst + 1) * bs] = self.slot[src * bs:(src + 1) * bs]

    def gather(self, table, n):
        bs = self.bs
        return [self.slot[table[t // bs] * bs + t % bs] for t in range(n)]


def pc_append(bm, sh, sid, token):
    slot, cow = bm.append_token(sid, token)
    if cow is not None:
        sh.copy(*cow)
    sh.write(slot, token)


def pc_check(bm, sh, live):
    """Every live sequence reads back exactly its own tokens through its table;
    counts equal table references; free, evictable and used blocks partition
    the pool; every registered block holds the last block of its prefix."""
    refs = [0] * bm.num_blocks
    for sid in live:
        t = bm.block_table(sid)
        for b in t:
            refs[b] += 1
        assert sh.gather(t, bm.seq_len(sid)) == bm.tokens[sid]
    assert refs == bm.ref
    used = {b for b in range(bm.num_blocks) if bm.ref[b] > 0}
    free, ev = set(bm.free), set(bm.evictable)
    assert not (free & ev) and not (free & used) and not (ev & used)
    assert len(bm.free) == len(free) and len(bm.evictable) == len(ev)
    assert all(bm.ref[b] == 0 and b in bm.key_of for b in ev)
    for key, b in bm.block_of.items():
        assert bm.key_of[b] == key
        assert sh.slot[b * sh.bs:(b + 1) * sh.bs] == list(key[-sh.bs:])


def test_prefix_cache_reuses_common_system_prompt_blocks():
    bs = 16
    bm = PrefixCachingBlockManager(64, bs, range(64))
    sh = Shadow(64, bs)
    system = list(range(1000, 1100))                   # 100-token system prompt
    p1 = system + [1, 2, 3]
    assert bm.add_seq_prompt("a", p1) == 0             # nothing cached yet
    assert (bm.hit_blocks, bm.lookup_blocks) == (0, 1)  # the first lookup misses: stop
    for t in p1:
        pc_append(bm, sh, "a", t)
    assert bm.num_cached() == 6                        # its 6 full blocks registered
    p2 = system + list(range(50, 80))
    n = bm.add_seq_prompt("b", p2)
    assert n == 96 and bm.hit_blocks == 6              # 6 full blocks of the common 100
    assert bm.lookup_blocks == 1 + 7                   # 6 hits, then the miss that stops it
    for t in p2[n:]:
        pc_append(bm, sh, "b", t)
    assert bm.block_table("b")[:6] == bm.block_table("a")[:6]
    assert bm.block_table("b")[6] != bm.block_table("a")[6]
    pc_check(bm, sh, ["a", "b"])


def test_prefix_cache_leaves_one_prompt_token_to_compute():
    bs = 16
    bm = PrefixCachingBlockManager(32, bs, range(32))
    sh = Shadow(32, bs)
    p = list(range(64))                                # exactly 4 blocks
    bm.add_seq_prompt(0, p)
    for t in p:
        pc_append(bm, sh, 0, t)
    assert bm.add_seq_prompt(1, p) == 48               # 3 blocks reused, 16 tokens left
    for t in p[48:]:
        pc_append(bm, sh, 1, t)
    pc_check(bm, sh, [0, 1])


def test_prefix_cache_never_shares_blocks_of_different_prefixes():
    """Block 1 of both prompts holds the same 16 ids, but their first tokens
    differ: the second request must not reuse either block."""
    bs = 16
    bm = PrefixCachingBlockManager(32, bs, range(32))
    sh = Shadow(32, bs)
    a = [7] + list(range(1, 40))
    b = [8] + list(range(1, 40))
    bm.add_seq_prompt("a", a)
    for t in a:
        pc_append(bm, sh, "a", t)
    assert bm.add_seq_prompt("b", b) == 0
    for t in b:
        pc_append(bm, sh, "b", t)
    assert not set(bm.block_table("a")) & set(bm.block_table("b"))
    pc_check(bm, sh, ["a", "b"])


def test_prefix_cache_never_registers_blocks_of_unknown_tokens():
    """A block's K/V depends on its token ids. Where they are not known
    (appends without ids) no later prompt can be shown to match, so the block
    is never registered. Freed, it goes back to the free list, not the
    evictable one, and a known block after it starts no chain."""
    bs = 4
    bm = PrefixCachingBlockManager(8, bs, range(8))
    bm.add_seq(0)
    for _ in range(2 * bs):
        bm.append_slot(0)                                # two full blocks, ids unknown
    for t in range(bs):
        bm.append_token(0, t)                            # a third, ids known
    assert bm.num_cached() == 0 and bm.block_table(0) == [0, 1, 2]
    bm.free_seq(0)                                       # to the tail, in table order
    assert bm.num_evictable() == 0 and bm.free == [3, 4, 5, 6, 7, 0, 1, 2]
    assert bm.add_seq_prompt(1, list(range(3 * bs + 1))) == 0


def test_prefix_cache_revives_freed_blocks_and_evicts_oldest_first():
    bs = 4
    bm = PrefixCachingBlockManager(8, bs, range(8))
    sh = Shadow(8, bs)
    p = list(range(12))                                # 3 full blocks
    bm.add_seq_prompt(0, p)
    for t in p:
        pc_append(bm, sh, 0, t)
    t0 = bm.block_table(0)
    bm.free_seq(0)
    assert bm.evictable == t0[::-1] and bm.num_free() == 5   # cached, kept, end first
    assert bm.add_seq_prompt(1, p + [99]) == 12        # revived: all 3 blocks reused
    assert bm.block_table(1) == t0 and bm.num_evictable() == 0
    pc_append(bm, sh, 1, 99)
    bm.free_seq(1)                                     # 4th block holds 1 token: uncached
    assert bm.evictable == t0[::-1]
    # fill the 5 free blocks with an unrelated 20-token prompt, then one more block
    q = list(range(500, 520))
    bm.add_seq_prompt(2, q)
    for t in q:
        pc_append(bm, sh, 2, t)
    assert bm.num_free() == 0
    pc_append(bm, sh, 2, 520)                          # needs a block: evicts the oldest
    assert bm.block_table(2)[-1] == t0[2]              # the end of the old prefix went first
    assert tuple(p) not in bm.block_of and tuple(p[:8]) in bm.block_of
    assert bm.add_seq_prompt(3, p + [1]) == 8          # only 2 blocks still cached
    pc_check(bm, sh, [2, 3])


def test_prefix_cache_random_scripts_keep_content_and_count_invariants():
    bs = 4
    rng = np.random.default_rng(11)
    for trial in range(30):
        nb = 40
        bm = PrefixCachingBlockManager(nb, bs, list(rng.permutation(nb)))
        sh = Shadow(nb, bs)
        prompts = [list(rng.integers(0, 3, size=rng.integers(1, 20))) for _ in range(4)]
        live, nxt = [], 0
        for step in range(60):
            op = rng.integers(0, 4)
            try:
                if op == 0 or not live:
                    base = prompts[rng.integers(len(prompts))]
                    p = base + list(rng.integers(0, 3, size=rng.integers(0, 6)))
                    n = bm.add_seq_prompt(nxt, p)
                    live.append(nxt)
                    for t in p[n:]:
                        pc_append(bm, sh, nxt, int(t))
                    nxt += 1
                elif op == 1:
                    sid = live[rng.integers(len(live))]
                    pc_append(bm, sh, sid, int(rng.integers(0, 3)))
                elif op == 2:
                    sid = live[rng.integers(len(live))]
                    bm.fork(sid, nxt)
                    live.append(nxt)
                    nxt += 1
                else:
                    sid = live.pop(rng.integers(len(live)))
                    bm.free_seq(sid)
            except PoolExhausted:
                break
            pc_check(bm, sh, live)


# ---------------------------------------------------------------- swapping to host memory
class Shadow2:
    """Slot contents of the device pool and of the host pool."""

    def __init__(self, nb, ncpu, bs):
        self.dev, self.host = Shadow(nb, bs), Shadow(ncpu, bs)

    def swap(self, pairs, to_host):
        bs = self.dev.bs
        src, dst = (self.dev, self.host) if to_host else (self.host, self.dev)
        for a, b in pairs:
            dst.slot[b * bs:(b + 1) * bs] = src.slot[a * bs:(a + 1) * bs]


def swap_check(bm, sh, live):
    for sid in live:
        pool = sh.host if sid in bm.swapped else sh.dev
        assert pool.gather(bm.tables[sid], bm.lens[sid]) == bm.tokens[sid]
    host_used = [b for sid in bm.swapped for b in bm.tables[sid]]
    assert len(host_used) == len(set(host_used))
    assert sorted(host_used + bm.cpu_free) == list(range(bm.num_cpu_blocks))
    refs = [0] * bm.num_blocks
    for sid in live:
        if sid not in bm.swapped:
            for b in bm.tables[sid]:
                refs[b] += 1
    assert refs == bm.ref


def test_swap_round_trip_preserves_content_while_device_blocks_are_reused():
    bs = 4
    bm = PrefixCachingBlockManager(6, bs, range(6), num_cpu_blocks=4)
    sh = Shadow2(6, 4, bs)
    bm.add_seq("a")
    for t in range(10):                                # 3 blocks
        slot, _ = bm.append_token("a", t)
        sh.dev.write(slot, t)
    dev_table = bm.block_table("a")
    pairs = bm.swap_out("a")
    assert pairs == list(zip(dev_table, [0, 1, 2])) and bm.block_table("a") == [0, 1, 2]
    sh.swap(pairs, to_host=True)
    bm.add_seq("b")                                    # b takes the freed device blocks
    for t in range(100, 124):
        slot, _ = bm.append_token("b", t)
        sh.dev.write(slot, t)
    swap_check(bm, sh, ["a", "b"])
    with pytest.raises(PoolExhausted):                 # all or nothing: device pool is full
        bm.swap_in("a")
    swap_check(bm, sh, ["a", "b"])
    bm.free_seq("b")
    pairs = bm.swap_in("a")
    sh.swap(pairs, to_host=False)
    assert [h for h, _ in pairs] == [0, 1, 2] and bm.cpu_free == [3, 0, 1, 2]
    swap_check(bm, sh, ["a"])
    for t in range(10, 14):                            # and it keeps growing
        slot, _ = bm.append_token("a", t)
        sh.dev.write(slot, t)
    swap_check(bm, sh, ["a"])


def test_swap_out_is_all_or_nothing_and_a_swapped_sequence_is_frozen():
    bm = BlockManager(8, 2, range(8), num_cpu_blocks=2)
    bm.add_seq(0)
    for _ in range(5):                                 # 3 blocks
        bm.append_slot(0)
    before = (list(bm.free), list(bm.cpu_free), bm.block_table(0))
    with pytest.raises(PoolExhausted):
        bm.swap_out(0)
    assert (list(bm.free), list(bm.cpu_free), bm.block_table(0)) == before
    bm2 = BlockManager(8, 2, range(8), num_cpu_blocks=4)
    bm2.add_seq(0)
    bm2.append_slot(0)
    bm2.swap_out(0)
    with pytest.raises(ValueError):
        bm2.append_slot(0)
    with pytest.raises(ValueError):
        bm2.fork(0, 1)
    bm2.free_seq(0)
    assert sorted(bm2.cpu_free) == [0, 1, 2, 3] and bm2.num_free() == 8


@pytest.mark.parametrize("caching", [False, True])
def test_swap_random_scripts_keep_content_and_partitions(caching):
    bs = 4
    rng = np.random.default_rng(21 + caching)
    for trial in range(25):
        nb, ncpu = 30, 20
        bm = PrefixCachingBlockManager(nb, bs, list(rng.permutation(nb)), ncpu)
        sh = Shadow2(nb, ncpu, bs)
        live, nxt = [], 0
        for step in range(80):
            op = int(rng.integers(0, 6))
            try:
                resident = [s for s in live if s not in bm.swapped]
                if op == 0 or not live:
                    p = list(rng.integers(0, 3, size=rng.integers(1, 14)))
                    if not caching:                    # ids of one sequence only: no hits
                        p = [t + 10 * (nxt + 1) for t in p]
                    sid = nxt
                    nxt += 1
                    n = bm.add_seq_prompt(sid, p)
                    live.append(sid)
                    for t in p[n:]:
                        slot, cow = bm.append_token(sid, int(t))
                        if cow:
                            sh.dev.copy(*cow)
                        sh.dev.write(slot, int(t))
                elif op == 1 and resident:
                    sid = resident[rng.integers(len(resident))]
                    t = int(rng.integers(0, 3)) + (0 if caching else 10 * (sid + 1))
                    slot, cow = bm.append_token(sid, t)
                    if cow:
                        sh.dev.copy(*cow)
                    sh.dev.write(slot, t)
                elif op == 2 and resident:
                    sid = resident[rng.integers(len(resident))]
                    bm.fork(sid, nxt)
                    live.append(nxt)
                    nxt += 1
                elif op == 3 and resident:
                    sid = resident[rng.integers(len(resident))]
                    sh.swap(bm.swap_out(sid), to_host=True)
                elif op == 4 and bm.swapped:
                    sid = sorted(bm.swapped)[rng.integers(len(bm.swapped))]
                    sh.swap(bm.swap_in(sid), to_host=False)
                elif op == 5:
                    sid = live.pop(rng.integers(len(live)))
                    bm.free_seq(sid)
            except PoolExhausted:
                pass                                   # all or nothing: state unchanged
            swap_check(bm, sh, live)

            if not caching:
                assert bm.hit_blocks == 0

def test_oracle_swap_blocks_round_trip_restores_every_sequence_through_its_table():
    """Pool values tagged by token id: after swapping a sequence out, letting
    another overwrite its freed device blocks and swapping it back, gathering
    through its new table gives back exactly the rows written for its tokens."""
    bs, Hkv, D, nb, ncpu = 4, 2, 3, 8, 6
    bm = BlockManager(nb, bs, [5, 2, 7, 0, 3, 6, 1, 4], num_cpu_blocks=ncpu)
    kp = torch.full((nb, Hkv, bs, D), -1.0, dtype=torch.float64)
    vp = kp.clone()
    hk = torch.full((ncpu, Hkv, bs, D), -1.0, dtype=torch.float64)
    hv = hk.clone()

    def write(sid, tok):
        s, _ = bm.append_slot(sid)
        row = torch.full((Hkv, D), float(tok), dtype=torch.float64)
        oops.reshape_and_cache(row[None], -row[None], kp, vp, torch.tensor([s]), bs)

    def rows(sid, kpool, vpool):
        t = bm.block_table(sid)
        k = torch.cat([kpool[b] for b in t], dim=1)[:, :bm.seq_len(sid)]
        v = torch.cat([vpool[b] for b in t], dim=1)[:, :bm.seq_len(sid)]
        return k[0, :, 0].tolist(), v[1, :, 2].tolist()

    for s, n in ((0, 10), (1, 5)):
        bm.add_seq(s)
        for i in range(n):
            write(s, 100 * s + i)
    want0 = [float(i) for i in range(10)]
    oops.swap_blocks(hk, hv, kp, vp, bm.swap_out(0))
    assert rows(0, hk, hv) == (want0, [-x for x in want0])
    bm.add_seq(2)
    for i in range(12):                                # 3 blocks: reuses 0's freed blocks
        write(2, 200 + i)
    oops.swap_blocks(hk, hv, kp, vp, bm.swap_out(2))   # 2 out as well, then 0 back in
    oops.swap_blocks(kp, vp, hk, hv, bm.swap_in(0))
    assert rows(0, kp, vp) == (want0, [-x for x in want0])
    assert rows(1, kp, vp)[0] == [100.0 + i for i in range(5)]
    assert rows(2, hk, hv)[0] == [200.0 + i for i in range(12)]
    with pytest.raises(IndexError):
        oops.swap_blocks(kp, vp, hk, hv, [(ncpu, 0)])


# ---------------------------------------------------------------- beam search
class Beams:
    """Beam search on the oracle's manager with a slot-content shadow and each
    beam's token history kept apart from the manager (its lineage)."""

    def __init__(self, P, bs, nb=600):
        self.bm = BlockManager(nb, bs, list(range(nb)))
        self.sh = Shadow(nb, bs)
        self.hist = {"p": []}
        self.bm.add_seq("p")
        for t in range(P):
            self.append("p", t)
        self.beams = ["p"]

    def append(self, sid, token):
        slot, cow = self.bm.append_slot(sid)
        if cow is not None:
            self.sh.copy(*cow)
        self.sh.write(slot, token)
        self.hist[sid].append(token)

    def step(self, g, parents):
        new = [(g, i) for i in range(len(parents))]
        self.bm.beam_step(self.beams, parents, new)
        hist = {n: self.hist[self.beams[p]] + [] for n, p in zip(new, parents)}
        self.hist = hist
        self.beams = new
        for i, sid in enumerate(new):
            self.append(sid, 10000 * (g + 1) + i)      # each beam's own new token

    def check(self):
        bm = self.bm
        refs = [0] * bm.num_blocks
        for sid in self.beams:
            t = bm.block_table(sid)
            assert self.sh.gather(t, bm.seq_len(sid)) == self.hist[sid]
            for b in t:
                refs[b] += 1
        assert refs == bm.ref
        assert sorted(bm.free + [b for b in range(bm.num_blocks) if bm.ref[b]]) == \
            list(range(bm.num_blocks))


@pytest.mark.parametrize("P,W,bs", [(40, 4, 16), (48, 4, 16), (47, 3, 16), (5, 2, 4), (1, 8, 16)])
def test_beams_collapsing_onto_one_parent_share_all_but_their_last_blocks(P, W, bs):
    """Every step, all W new beams continue old beam 0. After the step's appends
    the beams share every block except the one holding their last token, so the
    pool holds ceil(L/bs) - 1 + W blocks (W * ceil(L/bs) without sharing)."""
    b = Beams(P, bs)
    for g in range(40):
        b.step(g, [0] * W)
        L = P + g + 1
        assert b.bm.blocks_in_use() == -(-L // bs) - 1 + W
        b.check()


@pytest.mark.parametrize("P,W,bs", [(40, 4, 16), (48, 4, 16), (5, 3, 4)])
def test_beams_that_never_merge_share_only_the_prompts_full_blocks(P, W, bs):
    """The first step forks W beams off the prompt; after that beam i always
    continues beam i. Only the prompt's full blocks stay shared: the pool holds
    floor(P/bs) + W * (ceil(L/bs) - floor(P/bs)) blocks."""
    b = Beams(P, bs)
    b.step(0, [0] * W)
    for g in range(1, 40):
        b.step(g, list(range(W)))
        L = P + g + 1
        assert b.bm.blocks_in_use() == P // bs + W * (-(-L // bs) - P // bs)
        b.check()


def test_beam_step_copies_a_shared_partial_block_for_all_but_its_last_writer():
    b = Beams(20, 16)                                  # block 1 partial (4 tokens)
    b.bm.beam_step(["p"], [0, 0, 0], ["a", "b", "c"])
    pairs = [b.bm.append_slot(s)[1] for s in ("a", "b", "c")]
    shared = b.bm.block_table("c")[1]                  # c, the last writer, keeps it
    assert pairs[2] is None and pairs[0][0] == pairs[1][0] == shared
    assert len({pairs[0][1], pairs[1][1], shared}) == 3
    assert [b.bm.refcount(x) for x in (shared, pairs[0][1], pairs[1][1])] == [1, 1, 1]


@pytest.mark.parametrize("W,seed", [(2, 0), (4, 1), (4, 2), (8, 3)])
def test_random_beam_steps_keep_each_beams_history_and_the_counts(W, seed):
    rng = np.random.default_rng(seed)
    b = Beams(int(rng.integers(1, 60)), 4)
    b.step(0, [0] * W)
    for g in range(1, 60):
        b.step(g, sorted(rng.integers(0, W, size=W).tolist()))
        b.check()
    used = b.bm.blocks_in_use()
    assert used <= sum(-(-b.bm.seq_len(s) // 4) for s in b.beams)


def test_beam_step_rejects_bad_arguments_and_changes_nothing():
    b = Beams(10, 4)
    b.step(0, [0, 0])
    before = (dict(b.bm.tables), list(b.bm.ref), list(b.bm.free))
    for old, parents, new in ((b.beams, [0, 2], ["x", "y"]),        # parent out of range
                              (b.beams, [0, 1], ["x", "x"]),        # duplicate new id
                              (b.beams, [0, 1], [b.beams[0], "y"]),  # new id in use
                              (b.beams + ["zz"], [0, 1], ["x", "y"])):  # unknown old beam
        with pytest.raises(ValueError):
            b.bm.beam_step(old, parents, new)
        assert (dict(b.bm.tables), list(b.bm.ref), list(b.bm.free)) == before
