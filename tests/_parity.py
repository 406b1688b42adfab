"""Shared helpers of the GPU parity tests: run one workload's decode step through
the library (CUDA path, C ABI) and through the oracle (CPU, float64) on the same
seeded inputs, and compare.

Both sides start from ``pkv_workloads``' values and replay the workload's
block-manager script with their own block manager; nothing computed on the GPU is
ever fed to the oracle.

FP8 cache: the oracle keeps the *source* values in its pools and quantises what
it gathers (quantisation is elementwise, so it commutes with the copies and slot
writes); the library quantises when it writes (reshape_and_cache).
"""
import numpy as np
import torch

import paged_kv_cache_259_gb300 as pkv
from paged_kv_cache_259_gb300.engine import PagedKVCache

from oracle import attention as oatt
from oracle import cache_ops as oops
from oracle import fp8_e4m3 as ofp8
from oracle.block_manager import BlockManager as OracleBM, replay as oracle_replay

KV_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}
# |gpu - oracle| <= ATOL + RTOL * |oracle|, elementwise (the stated max-abs 2e-2 /
# max-rel 2e-2 bound read per element; 6e-2 for the E4M3 cache). float32 caches
# are also held to 1e-5, well above fp32 rounding of a softmax over <= 1e5 terms.
TOL = {"bf16": (2e-2, 2e-2), "e4m3": (6e-2, 6e-2), "f32": (1e-5, 1e-5)}


class Inputs:
    def __init__(self, w):
        self.w = w
        self.k_src, self.v_src = w.past_pools()
        self.q, self.k_new, self.v_new = w.step_inputs()
        if w.kv_dtype == "e4m3":
            self.ks, self.vs = w.fp8_scales(self.k_src, self.v_src, self.k_new, self.v_new)
        else:
            self.ks, self.vs = 1.0, 1.0


def run_gpu(inp, workspace=True, relabel=None, device="cuda"):
    """The decode step through the C ABI. ``relabel``: optional permutation applied
    to physical block ids (old id i -> relabel[i]) before anything is stored."""
    w = inp.w
    free_order = w.free_order if relabel is None else relabel[w.free_order]
    cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, KV_TORCH[w.kv_dtype], free_order, device)
    k_src, v_src = inp.k_src, inp.v_src
    if relabel is not None:
        perm = torch.from_numpy(relabel)
        k_src = torch.empty_like(k_src)
        v_src = torch.empty_like(v_src)
        k_src[perm] = inp.k_src
        v_src[perm] = inp.v_src
    # fill the pools with the library's own slot write (layout, E4M3 quantising)
    cache.load(k_src, v_src, inp.ks, inp.vs)
    setup_pairs = cache.replay(w.script)
    cache.apply_copies(setup_pairs)
    plan = cache.plan_step(w.step_seqs, max_blocks=w.max_blocks_per_seq)
    dev = plan.device_tensors(device)
    out = torch.empty(w.B, w.Hq, w.D, dtype=w.src_dtype, device=device)
    ws = cache.workspace(w.B, w.max_blocks_per_seq) if workspace else None
    cache.step(inp.q.to(device), inp.k_new.to(device), inp.v_new.to(device), dev, out,
               w.scale, inp.ks, inp.vs, ws)
    err = pkv.get_device_error()
    return {"out": out.float().cpu(), "cache": cache, "plan": plan, "setup_pairs": setup_pairs,
            "err": err}


def run_oracle(inp, units=None):
    w = inp.w
    bm = OracleBM(w.NB, w.bs, w.free_order)
    setup_pairs = oracle_replay(bm, w.script)
    kp, vp = inp.k_src.clone(), inp.v_src.clone()
    oops.copy_blocks(kp, vp, setup_pairs)
    step = [bm.append_slot(s) for s in w.step_seqs]
    slots = [s for s, _ in step]
    pairs = [c for _, c in step if c is not None]
    oops.copy_blocks(kp, vp, pairs)
    oops.reshape_and_cache(inp.k_new, inp.v_new, kp, vp, torch.tensor(slots), w.bs)
    MB = w.max_blocks_per_seq
    tables = np.full((w.B, MB), -1, dtype=np.int64)
    for i, s in enumerate(w.step_seqs):
        t = bm.block_table(s)
        tables[i, :len(t)] = t
    lens = np.array([bm.seq_len(s) for s in w.step_seqs])
    if w.kv_dtype == "e4m3":
        wk = lambda rows: ofp8.e4m3_decode(ofp8.e4m3_quantize(rows.float().numpy(), inp.ks))
        wv = lambda rows: ofp8.e4m3_decode(ofp8.e4m3_quantize(rows.float().numpy(), inp.vs))
    else:
        wk = wv = oatt.widen
    out = oatt.paged_decode(inp.q, kp, vp, tables, lens, w.scale, w.bs, inp.ks, inp.vs,
                            units=units, widen_k=wk, widen_v=wv)
    return {"out": out, "slots": slots, "pairs": pairs, "setup_pairs": setup_pairs,
            "tables": tables, "lens": lens, "k_pool": kp, "v_pool": vp}


def stored_bits(t):
    """Exact stored bits of a pool slice (for bit-exact comparison)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


def oracle_stored(inp, x, which):
    """What the cache must hold for oracle source values x (quantised if FP8)."""
    if inp.w.kv_dtype == "e4m3":
        scale = inp.ks if which == "k" else inp.vs
        return torch.from_numpy(ofp8.e4m3_quantize(x.float().numpy(), scale))
    return x


def check_indexing(g, o):
    """Bit-exact: slots, CoW pairs, block tables and lengths."""
    assert list(g["plan"].slots) == o["slots"]
    assert [tuple(p) for p in g["plan"].pairs] == o["pairs"]
    assert g["setup_pairs"] == o["setup_pairs"]
    MB = o["tables"].shape[1]
    assert np.array_equal(g["plan"].tables.astype(np.int64), o["tables"][:, :MB])
    assert np.array_equal(g["plan"].lens, o["lens"])


def check_cache_writes(inp, g, o, whole_pool=False):
    """Bit-exact: the pools at every CoW destination block and every written slot
    (or the whole pools)."""
    w = inp.w
    cache = g["cache"]
    kview, vview = cache.k_view(), cache.v_view()          # [NB, Hkv, bs, D]
    if whole_pool:
        for which, gp, op in (("k", kview, o["k_pool"]), ("v", vview, o["v_pool"])):
            assert torch.equal(stored_bits(gp.cpu()), stored_bits(oracle_stored(inp, op, which)))
        return
    blocks = sorted({d for _, d in o["setup_pairs"] + o["pairs"]})
    for which, gp, op in (("k", kview, o["k_pool"]), ("v", vview, o["v_pool"])):
        if blocks:
            idx = torch.tensor(blocks)
            assert torch.equal(stored_bits(gp[idx.to(gp.device)].cpu()),
                               stored_bits(oracle_stored(inp, op[idx], which)))
        for s in o["slots"]:
            b, off = s // w.bs, s % w.bs
            assert torch.equal(stored_bits(gp[b, :, off].cpu()),
                               stored_bits(oracle_stored(inp, op[b, :, off], which)))


def assert_close(got, ref, kv_dtype, what=""):
    atol, rtol = TOL[kv_dtype]
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: got {got[i]}, oracle {ref[i]}; "
                             f"max abs err {err.max():.3e}")
    return float(err.max())


def sample_units(w, n, seed=0):
    """n (sequence, query head) pairs: seeded, plus the longest and shortest sequences."""
    rng = np.random.default_rng(seed)
    units = {(int(np.argmax(w.final_lens)), 0), (int(np.argmin(w.final_lens)), w.Hq - 1)}
    while len(units) < n:
        units.add((int(rng.integers(w.B)), int(rng.integers(w.Hq))))
    return sorted(units)
