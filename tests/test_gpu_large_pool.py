"""GPU parity on a pool larger than 2 GiB, with sequences in blocks whose byte
offsets pass 2^31.

Every pool access computes its offset in 64 bits, but the benchmark workloads
keep each pool under 1 GB. Here each pool is 2.46 GB (300,000 blocks of 8 KiB).
One sequence holds block 0, the last block below a 2^31-byte offset and blocks
near the end of the pool. The others hold only blocks near the end.

The path checked is a whole-prompt prefill step, the next decode step, and a
block copy between two high blocks. The oracle runs on compact pools holding
only the used blocks, with tables relabelled to match. A relabelling of
physical blocks leaves attention unchanged.
"""
import math

import numpy as np
import pytest
import torch

from _lib import library, pkv
from _parity import assert_close, stored_bits
from paged_kv_cache_259_gb300.engine import PagedKVCache

from oracle import attention as oatt
from oracle import cache_ops as oops
from oracle.block_manager import BlockManager as OracleBM

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS = 8, 2, 128, 16
BLOCK_BYTES = HKV * BS * D * 2                    # 8 KiB of K (or V) per block
NB = 300_000                                      # 2.46 GB per pool
HIGH = (1 << 31) // BLOCK_BYTES                   # first block at a 2^31-byte offset
LENS = [40, 300, 17, 129]


@pytest.fixture(scope="module", autouse=True)
def gpu_and_library():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    library()
    torch.cuda.set_device(0)


def compact(tables, used):
    """Tables relabelled onto 0..len(used)-1 (-1 stays -1)."""
    remap = {b: i for i, b in enumerate(used)}
    return np.array([[remap[b] if b >= 0 else -1 for b in row] for row in tables], np.int64)


def compact_slots(slots, used):
    remap = {b: i for i, b in enumerate(used)}
    return torch.tensor([remap[s // BS] * BS + s % BS for s in slots], dtype=torch.int64)


def test_blocks_past_two_gib_prefill_decode_and_copy():
    assert NB > HIGH + 3000
    rng = np.random.default_rng(31)
    top = rng.permutation(np.arange(NB - 3000, NB))
    order = [0, HIGH - 1] + [int(b) for b in top[:200]]
    ids = list(range(len(LENS)))
    cache = PagedKVCache(NB, HQ, HKV, D, BS, torch.bfloat16, order, "cuda")
    ora = OracleBM(NB, BS, order)
    for s in ids:
        cache.bm.add_seq(s)
        ora.add_seq(s)
    g = torch.Generator().manual_seed(31)
    scale = 1.0 / math.sqrt(D)

    # ---- prefill: each prompt is one chunk
    T = sum(LENS)
    q = torch.randn(T, HQ, D, generator=g).to(torch.bfloat16)
    k = torch.randn(T, HKV, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, HKV, D, generator=g).to(torch.bfloat16)
    plan = cache.plan_prefill(ids, LENS)
    out = torch.full((T, HQ, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    cache.prefill_step(q.cuda(), k.cuda(), v.cuda(), plan.device_tensors("cuda"), out, scale,
                       plan.max_query_len)
    assert pkv.get_device_error() == 0
    slots = [ora.append_slot(s)[0] for s, n in zip(ids, LENS) for _ in range(n)]
    assert list(plan.slots) == slots and plan.pairs.shape[0] == 0
    MB = plan.tables.shape[1]
    tables = np.full((len(ids), MB), -1, np.int64)
    for i, s in enumerate(ids):
        t = ora.block_table(s)
        tables[i, :len(t)] = t
    assert np.array_equal(plan.tables.astype(np.int64), tables)
    assert ora.block_table(0)[:2] == [0, HIGH - 1] and tables.max() >= NB - 3000
    used = sorted({b for row in tables for b in row if b >= 0})

    kp = torch.zeros(len(used), HKV, BS, D, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    oops.reshape_and_cache(k, v, kp, vp, compact_slots(slots, used), BS)
    qs = np.concatenate([[0], np.cumsum(LENS)])
    ref = oatt.paged_prefill(q, kp, vp, compact(tables, used), np.array(LENS), qs, scale, BS)
    assert_close(out.float().cpu().numpy(), ref, "bf16", "prefill, high blocks")

    # the written slots, read back through the library layout, bit for bit
    idx = torch.tensor(used, dtype=torch.int64, device="cuda")
    kv, vv = pkv.pool_views(cache.k_pool[idx], cache.v_pool[idx])
    cs = compact_slots(slots, used)
    b, off = cs // BS, cs % BS
    assert torch.equal(stored_bits(kv.cpu()[b, :, off]), stored_bits(k))
    assert torch.equal(stored_bits(vv.cpu()[b, :, off]), stored_bits(v))

    # ---- the next decode step (no new blocks: every last block has room)
    q2 = torch.randn(len(ids), HQ, D, generator=g).to(torch.bfloat16)
    k2 = torch.randn(len(ids), HKV, D, generator=g).to(torch.bfloat16)
    v2 = torch.randn(len(ids), HKV, D, generator=g).to(torch.bfloat16)
    plan2 = cache.plan_step(ids)
    out2 = torch.full((len(ids), HQ, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    cache.step(q2.cuda(), k2.cuda(), v2.cuda(), plan2.device_tensors("cuda"), out2, scale,
               workspace=cache.workspace(len(ids), plan2.tables.shape[1]))
    assert pkv.get_device_error() == 0
    slots2 = [ora.append_slot(s)[0] for s in ids]
    assert list(plan2.slots) == slots2 and plan2.pairs.shape[0] == 0
    assert {s // BS for s in slots2} <= set(used)
    oops.reshape_and_cache(k2, v2, kp, vp, compact_slots(slots2, used), BS)
    lens2 = np.array([ora.seq_len(s) for s in ids])
    ref2 = oatt.paged_decode(q2, kp, vp, compact(tables, used), lens2, scale, BS)
    assert_close(out2.float().cpu().numpy(), ref2, "bf16", "decode, high blocks")

    # ---- a block copy between two blocks past the 2^31-byte offset
    src, dst = ora.block_table(1)[-1], int(top[-1])
    assert min(src, dst) >= HIGH and dst not in used
    pkv.copy_blocks(cache.k_pool, cache.v_pool,
                    torch.tensor([[src, dst]], dtype=torch.int64, device="cuda"))
    assert pkv.get_device_error() == 0
    for pool in (cache.k_pool, cache.v_pool):
        assert torch.equal(stored_bits(pool[dst].cpu()), stored_bits(pool[src].cpu()))
