"""GPU parity of chunked-prefill attention (tcgen05 kernel, through the C ABI)
against the CPU oracle.

A step appends each sequence's chunk (slots and copy-on-write pairs from the
block manager), writes the chunk's K/V with reshape_and_cache, and runs
paged_attention_prefill. Indexing and cache writes are compared bit-exactly;
attention outputs elementwise within |gpu - oracle| <= 2e-2 + 2e-2 |oracle|
(bf16 cache, f32 accumulation). Small ragged cases compare every row; the
full-size workloads compare sampled (token, head) rows in the benchmark's
launch configuration.
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
from oracle.block_manager import BlockManager as OracleBM

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_and_library():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    library()
    torch.cuda.set_device(0)


class Case:
    def __init__(self, w):
        self.w = w
        self.k_src, self.v_src = w.past_pools()
        self.q, self.k_new, self.v_new = w.step_inputs()


def run_gpu(c, max_query_len=None, bad=None, device="cuda"):
    w = c.w
    cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, torch.bfloat16, w.free_order, device)
    cache.load(c.k_src, c.v_src)
    setup_pairs = cache.replay(w.script)
    cache.apply_copies(setup_pairs)
    plan = cache.plan_prefill(w.step_seqs, w.chunks, max_blocks=w.max_blocks_per_seq)
    dev = plan.device_tensors(device)
    if bad is not None:
        bad(dev)
    out = torch.full((w.T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=device)
    mql = plan.max_query_len if max_query_len is None else max_query_len
    cache.prefill_step(c.q.to(device), c.k_new.to(device), c.v_new.to(device), dev, out, w.scale,
                       mql)
    err = pkv.get_device_error()
    return {"out": out.float().cpu(), "cache": cache, "plan": plan, "setup_pairs": setup_pairs,
            "err": err}


def run_oracle(c, units=None):
    w = c.w
    bm = OracleBM(w.NB, w.bs, w.free_order)
    setup_pairs = []
    for op in w.script:
        if op[0] == "add":
            bm.add_seq(op[1])
        elif op[0] == "fork":
            bm.fork(op[1], op[2])
        else:
            for _ in range(op[2]):
                cow = bm.append_slot(op[1])[1]
                if cow is not None:
                    setup_pairs.append(cow)
    kp, vp = c.k_src.clone(), c.v_src.clone()
    oops.copy_blocks(kp, vp, setup_pairs)
    slots, pairs = [], []
    for s, n in zip(w.step_seqs, w.chunks):
        for _ in range(int(n)):
            slot, cow = bm.append_slot(s)
            slots.append(slot)
            if cow is not None:
                pairs.append(cow)
    oops.copy_blocks(kp, vp, pairs)
    oops.reshape_and_cache(c.k_new, c.v_new, kp, vp, torch.tensor(slots, dtype=torch.int64), w.bs)
    MB = w.max_blocks_per_seq
    tables = np.full((w.B, MB), -1, dtype=np.int64)
    for i, s in enumerate(w.step_seqs):
        t = bm.block_table(s)
        tables[i, :len(t)] = t
    lens = np.array([bm.seq_len(s) for s in w.step_seqs])
    qs = [0]
    for n in w.chunks:
        qs.append(qs[-1] + int(n))
    out = oatt.paged_prefill(c.q, kp, vp, tables, lens, np.array(qs), w.scale, w.bs,
                             units=units)
    return {"out": out, "slots": slots, "pairs": pairs, "setup_pairs": setup_pairs,
            "tables": tables, "lens": lens, "k_pool": kp, "v_pool": vp}


def check_indexing_and_writes(g, o):
    plan = g["plan"]
    assert list(plan.slots) == o["slots"]
    assert [tuple(p) for p in plan.pairs] == o["pairs"]
    assert g["setup_pairs"] == o["setup_pairs"]
    assert np.array_equal(plan.tables.astype(np.int64), o["tables"])
    assert np.array_equal(plan.lens, o["lens"])
    cache = g["cache"]
    assert torch.equal(stored_bits(cache.k_view().cpu()), stored_bits(o["k_pool"]))
    assert torch.equal(stored_bits(cache.v_view().cpu()), stored_bits(o["v_pool"]))


CTX = [0, 5, 16, 200, 0, 1000, 37, 3]
CHUNK = [1, 7, 128, 129, 300, 17, 64, 0]

SMALL = [
    ("mha_bs16", 8, 8, 16),
    ("gqa4_bs16", 16, 4, 16),
    ("gqa8_bs32", 16, 2, 32),
    ("gqa2_bs32", 8, 4, 32),
    ("gqa16_bs16", 16, 1, 16),
]


@pytest.mark.parametrize("name,Hq,Hkv,bs", SMALL, ids=[s[0] for s in SMALL])
def test_prefill_small_ragged_every_row(name, Hq, Hkv, bs):
    w = wl.chunked_prefill(f"prefill_{name}", 40 + Hq + bs, CTX, CHUNK, Hq, Hkv, 128, bs)
    c = Case(w)
    g = run_gpu(c)
    o = run_oracle(c)
    assert g["err"] == 0
    check_indexing_and_writes(g, o)
    assert_close(g["out"].numpy(), o["out"], "bf16", name)


def test_prefill_after_fork_copies_the_shared_partial_block():
    """Two samples share a 40-token prompt (last block partial); the second one's
    chunk first copies that block (copy-on-write), then attends over it."""
    w = wl.chunked_prefill("prefill_fork", 77, [0, 0], [1, 1], 8, 2, 128, 16, NB=40)
    w.script = [("add", 0), ("append", 0, 40), ("fork", 0, 1)]
    w.chunks = np.array([20, 150])
    w.final_lens = np.array([60, 190])
    c = Case(w)
    g = run_gpu(c)
    o = run_oracle(c)
    assert g["err"] == 0
    assert len(o["pairs"]) == 1 and not o["setup_pairs"]
    check_indexing_and_writes(g, o)
    assert_close(g["out"].numpy(), o["out"], "bf16", "fork")


def test_prefill_larger_max_query_len_changes_nothing():
    w = wl.chunked_prefill("prefill_mql", 9, [30, 0], [33, 100], 8, 8, 128, 16)
    c = Case(w)
    a = run_gpu(c)
    b = run_gpu(c, max_query_len=1000)
    assert a["err"] == 0 and b["err"] == 0
    assert torch.equal(a["out"], b["out"])
    assert_close(a["out"].numpy(), run_oracle(c)["out"], "bf16", "mql")


def test_prefill_bad_block_id_is_flagged_not_followed():
    w = wl.chunked_prefill("prefill_bad", 13, [100, 20], [40, 10], 8, 8, 128, 16)
    c = Case(w)

    def corrupt(dev):
        dev["tables"][0, 2] = w.NB + 1000
    g = run_gpu(c, bad=corrupt)
    assert g["err"] == -4
    # the other sequence is unaffected
    o = run_oracle(c)
    assert_close(g["out"][40:].numpy(), o["out"][40:], "bf16", "unaffected sequence")


def test_prefill_chunk_longer_than_sequence_is_flagged():
    w = wl.chunked_prefill("prefill_bad_len", 14, [10, 20], [5, 10], 8, 8, 128, 16)
    c = Case(w)

    def corrupt(dev):
        dev["lens"][0] = 3          # shorter than its 5-token chunk
    g = run_gpu(c, bad=corrupt)
    assert g["err"] == -4
    assert torch.isnan(g["out"][:5]).all()              # its rows are not written
    o = run_oracle(c)
    assert_close(g["out"][5:].numpy(), o["out"][5:], "bf16", "unaffected sequence")


def test_prefill_rows_outside_the_output_are_flagged_not_followed():
    """query_start entries that put a chunk past query_start[num_seqs] (the rows
    of q and out) or out of order: every affected sequence is flagged
    (PKV_ERR_OUT_OF_RANGE) and left unwritten -- nothing is read or written past
    the buffers -- and the same step with the right offsets is clean."""
    w = wl.chunked_prefill("prefill_bad_rows", 15, [500, 300], [10, 20], 8, 8, 128, 16)
    c = Case(w)

    def corrupt(dev):
        dev["query_start"][1] = w.T + 10        # chunk 0 would run past the 30 rows
    g = run_gpu(c, bad=corrupt)
    assert g["err"] == -4
    assert torch.isnan(g["out"]).all()          # sequence 1's offsets are out of order too
    g = run_gpu(c)
    assert g["err"] == 0
    o = run_oracle(c)
    assert_close(g["out"].numpy(), o["out"], "bf16", "the same step, right offsets")


def sample_rows(w, n, seed=0):
    rng = np.random.default_rng(seed)
    qs = w.query_start
    units = set()
    for b in (0, w.B - 1):
        units.add((int(qs[b]), 0))                           # first chunk token
        units.add((int(qs[b + 1]) - 1, w.Hq - 1))            # last chunk token
    while len(units) < n:
        units.add((int(rng.integers(w.T)), int(rng.integers(w.Hq))))
    return sorted(units)


@pytest.mark.parametrize("config", sorted(wl.PREFILL_CONFIGS))
def test_prefill_full_size_sampled(config):
    w = wl.PREFILL_CONFIGS[config]()
    c = Case(w)
    g = run_gpu(c)
    assert g["err"] == 0
    assert torch.isfinite(g["out"]).all()
    units = sample_rows(w, 512)
    o = run_oracle(c, units=units)
    got = np.stack([g["out"][t, h].numpy() for t, h in units])
    ref = np.stack([o["out"][u] for u in units])
    assert_close(got, ref, "bf16", config)
    assert list(g["plan"].slots) == o["slots"]


def test_prefill_through_step_pipeline_matches_serial_steps():
    """Chunked-prefill steps fed from pinned host memory through
    engine.StepPipeline (one packed upload per step, overlapped with the
    neighbouring steps) give exactly the outputs of the same steps run one after
    another with device inputs."""
    from paged_kv_cache_259_gb300.engine import StepPipeline
    w = wl.chunked_prefill("pipe", 11, [0, 37, 150], [64, 9, 130], 8, 2, 128, 16)
    c = Case(w)
    gen = torch.Generator().manual_seed(12)
    n = 3
    ins = [tuple(torch.randn(w.T, hh, w.D, generator=gen).to(torch.bfloat16)
                 for hh in (w.Hq, w.Hkv, w.Hkv)) for _ in range(n)]
    outs = {}
    for mode in ("serial", "pipelined"):
        g = run_gpu(c)
        cache, plan = g["cache"], g["plan"]
        mql = plan.max_query_len
        if mode == "serial":
            dev = plan.device_tensors("cuda")
            res = []
            for q, k, v in ins:
                o = torch.empty(w.T, w.Hq, w.D, dtype=torch.bfloat16, device="cuda")
                cache.prefill_step(q.cuda(), k.cuda(), v.cuda(), dev, o, w.scale, mql)
                res.append(o.cpu())
        else:
            host = plan.host_tensors(pin=False)
            tmpl = dict(host, q=ins[0][0], k_new=ins[0][1], v_new=ins[0][2])
            pipe = StepPipeline(cache, tmpl, torch.empty(w.T, w.Hq, w.D, dtype=torch.bfloat16,
                                                         device="cuda"),
                                run=lambda q_, k_, v_, pl, o, s: cache.prefill_step(
                                    q_, k_, v_, pl, o, w.scale, mql, stream=s))
            res = [torch.empty(w.T, w.Hq, w.D, dtype=torch.bfloat16).pin_memory() for _ in ins]
            for (q, k, v), ho in zip(ins, res):
                views = pipe.host_inputs()
                for key, t in dict(host, q=q, k_new=k, v_new=v).items():
                    views[key].copy_(t)
                pipe.submit(ho)
            torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        outs[mode] = res
    for a, b in zip(outs["serial"], outs["pipelined"]):
        assert torch.equal(a, b)


# ------------------------------------------------------------ running-max moves
# The kernel keeps a running row max m and moves it (rescaling O in tensor
# memory and the row sum by 2^(m_old - m_new)) only when a 128-key tile's max of
# the scaled log2 scores exceeds m by more than 8; otherwise it exponentiates
# against the old max. With N(0, 1) inputs a later tile almost never beats the
# first by 8, so these cases build keys whose size grows tile by tile along the
# query's direction: K[pos] = a(tile of pos) * u + noise, q = +/-u + noise with u
# a +/-1 vector per KV head. Query heads with +u see their scores rise from tile
# to tile (the move is taken, often on consecutive tiles and on diagonal tiles
# where the row sees a single key), heads with -u see them fall (never taken),
# so most warps mix rows that move with rows that do not.
RISE_LEVEL_STEPS = (0.75, 0.2, 0.75, 0.75, -0.3)   # a(tile) walks by these, in turn
KEY_TILE = 128
MOVE_LOG2 = 8.0


def _positions_to_slots(w):
    """(sequence, position) -> pool slot of every token cached before the step,
    from the oracle's block manager replaying the workload's script."""
    bm = OracleBM(w.NB, w.bs, w.free_order)
    for op in w.script:
        if op[0] == "add":
            bm.add_seq(op[1])
        else:
            for _ in range(op[2]):
                bm.append_slot(op[1])
    return {b: [bm.block_table(b)[t // w.bs] * w.bs + t % w.bs for t in range(bm.seq_len(b))]
            for b in w.step_seqs}


def rising_case(name, seed, context, chunks, Hq, Hkv, bs):
    w = wl.chunked_prefill(name, seed, context, chunks, Hq, Hkv, 128, bs)
    c = Case(w)
    rng = np.random.default_rng(seed)
    G = Hq // Hkv
    u = torch.from_numpy(rng.choice([-1.0, 1.0], size=(Hkv, w.D)))
    sign = torch.from_numpy(np.where(np.arange(Hq) % 3 == 2, -1.0, 1.0))   # 1 head in 3 falls
    n_tiles = int(max(w.final_lens)) // KEY_TILE + 1
    steps = [RISE_LEVEL_STEPS[j % len(RISE_LEVEL_STEPS)] for j in range(n_tiles - 1)]
    level = np.concatenate([[0.0], np.cumsum(steps)])
    level = torch.from_numpy(level)

    def keys(noise, pos):                     # noise [n, Hkv, D], pos [n]
        a = level[torch.as_tensor(pos) // KEY_TILE].view(-1, 1, 1)
        return (a * u.unsqueeze(0) + 0.25 * noise.double()).to(torch.bfloat16)

    # cached context tokens, in the pool at the slots the script gives them
    slots = _positions_to_slots(w)
    for b in w.step_seqs:
        sl = torch.tensor(slots[b], dtype=torch.int64)
        if len(sl) == 0:
            continue
        blk, off = sl // w.bs, sl % w.bs
        c.k_src[blk, :, off] = keys(c.k_src[blk, :, off], np.arange(len(sl)))
    # the chunk tokens (written by the step), then the queries
    pos = np.concatenate([np.arange(cx, cx + n) for cx, n in zip(context, chunks)])
    c.k_new = keys(c.k_new, pos)
    qdir = (sign.view(1, Hq, 1) * u[torch.arange(Hq) // G].unsqueeze(0))
    c.q = (qdir + 0.25 * c.q.double()).to(torch.bfloat16)
    return c


def running_max_moves(c, o):
    """Per query row (token, head): how many tiles move the running max, and how
    many of those moves happen on a tile where the row sees at most 2 keys --
    the kernel's rule replayed in float64 on the stored bf16 values (a move is
    counted only with a margin of 0.05 over the threshold, so float32 rounding in
    the kernel cannot undo it)."""
    w = c.w
    G = w.Hq // w.Hkv
    sc = w.scale * np.log2(np.e)
    qs = w.query_start
    moves = np.zeros((w.T, w.Hq), dtype=np.int64)
    sparse_moves = 0
    for b in range(w.B):
        L, C = int(o["lens"][b]), int(qs[b + 1] - qs[b])
        for hk in range(w.Hkv):
            K = oatt.widen(oatt.gather(o["k_pool"], o["tables"][b], L, hk, w.bs)).reshape(L, w.D)
            for h in range(hk * G, (hk + 1) * G):
                Q = c.q[qs[b]:qs[b + 1], h].to(torch.float64).numpy()
                S = (Q @ K.T) * sc                                   # [C, L]
                for i in range(C):
                    p = L - C + i
                    m = None
                    for j in range(p // KEY_TILE + 1):
                        seen = S[i, j * KEY_TILE:min(p + 1, (j + 1) * KEY_TILE)]
                        mt = seen.max()
                        if m is None:
                            m = mt
                        elif mt > m + MOVE_LOG2 + 0.05:
                            moves[qs[b] + i, h] += 1
                            sparse_moves += len(seen) <= 2
                            m = mt
    return moves, sparse_moves


RISING = [  # (name, Hq, Hkv, bs, context, chunks)
    ("small_mha_bs16", 8, 8, 16, [0, 300], [420, 90]),
    ("mid_mha_bs32", 8, 8, 32, [0, 700, 333], [520, 300, 250]),
    ("mid_gqa4_bs16", 16, 4, 16, [0, 450, 1000], [400, 333, 129]),
    ("mid_gqa8_bs32", 16, 2, 32, [5, 640], [260, 384]),
]


@pytest.mark.parametrize("name,Hq,Hkv,bs,context,chunks", RISING, ids=[r[0] for r in RISING])
def test_prefill_running_max_moves_every_row(name, Hq, Hkv, bs, context, chunks):
    """Inputs whose tile maxima rise by more than 8 log2 units (shown on the CPU
    from the stored values) take the kernel's O-rescale branch on most rows;
    every output row still equals the oracle's."""
    c = rising_case(f"rising_{name}", 91 + Hq + bs, context, chunks, Hq, Hkv, bs)
    w = c.w
    g = run_gpu(c)
    assert g["err"] == 0
    G = Hq // Hkv
    seq_of = np.repeat(np.arange(w.B), w.chunks)
    units = sorted(((t, h) for t in range(w.T) for h in range(w.Hq)),
                   key=lambda th: (seq_of[th[0]], th[1] // G, th[0], th[1]))
    o = run_oracle(c, units=units)
    check_indexing_and_writes(g, o)
    # the input forces moves of the running max
    moves, sparse = running_max_moves(c, o)
    rising = np.arange(w.Hq) % 3 != 2
    long_rows = np.array([[L - C + i >= KEY_TILE for h in range(w.Hq)]
                          for b, (L, C) in enumerate(zip(o["lens"], w.chunks))
                          for i in range(int(C))])
    assert (moves[:, rising][long_rows[:, rising]] >= 1).mean() > 0.9
    assert (moves >= 2).any()                          # moves on more than one tile
    assert not moves[:, ~rising].any()
    assert sparse > 0
    got = g["out"].numpy()
    ref = np.stack([o["out"][(t, h)] for t in range(w.T) for h in range(w.Hq)]).reshape(got.shape)
    assert_close(got, ref, "bf16", name)
