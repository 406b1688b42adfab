"""Benchmark: one decode step of paged attention (copy_blocks -> reshape_and_cache ->
paged_attention_decode, as one paged_decode_step call) on a seeded synthetic
workload, timed on the GPU.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints ONE JSON line (rank 0). ``value`` is achieved algorithmic HBM bytes of the
whole step per second (GB/s), with every input resident in HBM; ``e2e`` is the
same metric through the engine (``LiveDecodePipeline``): every step is planned
on the host by the native block manager straight into a pinned slab, the slab
is uploaded and the output read back inside the timed region, overlapped with
the neighbouring steps. ``roofline`` covers the decode attention op alone (its
kernel plus the split-KV merge), timed with CUDA events on its stream in a
second pass of the same steps made as separate calls.
``cpu_baseline`` times the CPU oracle on a bounded sample of the same workload,
and ``check`` compares the timed steps' output with the oracle rows that run
computed first. The default workload's line also carries ``others``: every
other decode workload timed the same way, each with its own check. With
``--impl reference`` the oracle alone is timed (the reference arm; a slow CPU
program, not a target).

Other workloads (``--config``): ``prefill_*`` time a chunked-prefill step
(TFLOP/s of the causal attention, tensor-bound roofline), the prompt workload a
prefill step with prefix caching, ``swap_*`` a swap step of preempted sequences
to and from pinned host memory (GB/s of block bytes against the copy engines'
rate measured in the same run, plus the copy-engine path and its overlap with
decode), ``beam_search_bf16`` a beam-search decode step.

Multi-GPU (torchrun): every rank runs its own copy of the workload (independent
sequences; decode attention needs no exchange), so scaling is weak; the NCCL
process group is used only for the barrier and the max-over-ranks time.
"""
import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")   # each oracle process: one thread
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse
import json
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import pkv_workloads as wl  # noqa: E402

METRIC = "paged decode attention: achieved HBM GB/s (% of peak) and seq-steps/s"
DEFAULT_CONFIG = "llama13b_mha_bf16"
KV_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}
KV_ELT = {"f32": 4, "bf16": 2, "e4m3": 1}
L2_BYTES = 129 * 2 ** 20


KERNEL_SOURCES = ["pkv_decode_impl.cuh", "pkv_decode.cu", "pkv_decode_bf16.cu",
                  "pkv_decode_e4m3.cu", "pkv_decode_f32.cu"]


def code_hash(files):
    """Hash of kernel sources with their comments and blank lines removed, so
    that documentation edits do not orphan counters captured on the same code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_259_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("\n".join(line.rstrip() for line in src.splitlines() if line.strip()).encode())
    return h.hexdigest()[:16]


def kernel_source_hash():
    return code_hash(KERNEL_SOURCES)


def measured_traffic(config):
    """DRAM bytes per decode launch from profiles/decode_traffic.json (an ncu
    capture), or None when it was taken on other kernel sources or workloads."""
    try:
        with open(os.path.join(ROOT, "profiles", "decode_traffic.json")) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("kernel_source_sha") != kernel_source_hash():
        return None
    e = t.get("workloads", {}).get(config)
    return None if e is None else e.get("dram_bytes_per_decode")


def load_tensor_peak():
    """Dense bf16 tensor peak in TFLOP/s: the measured burst figure (a kernel
    timed alone), else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- byte accounting
def step_bytes(w, tables, lens, num_pairs):
    """Algorithmic HBM bytes of one step, by op.

    decode: K and V of every cached token a sequence attends over (shared blocks
    counted once: the unique bytes the method must move; ``logical`` counts them
    per sequence), plus q, out, block tables and lengths. reshape: new K/V read,
    cache slots written, slot numbers. copy: each CoW block read and written in
    both pools, plus the pairs.
    """
    elt, src = KV_ELT[w.kv_dtype], (4 if w.src_dtype == torch.float32 else 2)
    per_tok = 2 * w.Hkv * w.D * elt
    used = {}
    for b in range(len(lens)):
        L = int(lens[b])
        nb = -(-L // w.bs)
        for j in range(nb):
            blk = int(tables[b, j])
            n = min(w.bs, L - j * w.bs)
            used[blk] = max(used.get(blk, 0), n)
    unique_tok = sum(used.values())
    logical_tok = int(np.sum(lens))
    qo = 2 * w.B * w.Hq * w.D * src + tables.size * 4 + len(lens) * 4
    decode = unique_tok * per_tok + qo
    reshape = w.B * w.Hkv * w.D * 2 * (src + elt) + w.B * 8
    block_bytes = w.Hkv * w.bs * w.D * elt
    copy = num_pairs * 2 * 2 * block_bytes + num_pairs * 16
    return {"decode": decode, "decode_logical": logical_tok * per_tok + qo, "reshape": reshape,
            "copy": copy, "total": decode + reshape + copy, "per_token": per_tok,
            "unique_tokens": unique_tok, "logical_tokens": logical_tok}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle timing
def _oracle_loop(p, inp, tables, lens, run_s, seed, check=()):
    """The oracle over random (sequence, head) units for about run_s seconds, one
    thread; returns the finish time (s from the start) and algorithmic K/V bytes
    of every unit, and the output rows of the ``check`` units, which it computes
    first (they count as timed units like the others)."""
    from oracle import attention as oatt
    from oracle import fp8_e4m3 as ofp8
    q, kp, vp, ks, vs = inp
    if p["kv"] == "e4m3":
        # the oracle takes source values and quantises the rows it gathers
        wk = lambda r: ofp8.e4m3_decode(ofp8.e4m3_quantize(r.float().numpy(), ks))
        wv = lambda r: ofp8.e4m3_decode(ofp8.e4m3_quantize(r.float().numpy(), vs))
    else:
        wk = wv = oatt.widen
    rng = np.random.default_rng(seed)
    fin, nbytes, outs = [], [], {}
    todo = [tuple(int(x) for x in u) for u in check]
    t0 = time.perf_counter()
    if p.get("mode") == "prefill":
        # units are (chunk token, head); the amount is the token's attention FLOPs
        qs = np.asarray(p["query_start"])
        seq_of = np.searchsorted(qs, np.arange(int(qs[-1])), side="right") - 1
        while todo or time.perf_counter() - t0 < run_s:
            t, h = todo.pop(0) if todo else (int(rng.integers(int(qs[-1]))),
                                             int(rng.integers(p["Hq"])))
            r = oatt.paged_prefill(q, kp, vp, tables, lens, qs, p["scale"], p["bs"],
                                   units=[(t, h)])
            fin.append(time.perf_counter() - t0)
            if len(outs) < len(check):
                outs[(t, h)] = r[(t, h)]
            b = int(seq_of[t])
            pos = int(lens[b]) - int(qs[b + 1] - qs[b]) + (t - int(qs[b]))
            nbytes.append(4.0 * p["D"] * (pos + 1))
        return np.array(fin), np.array(nbytes), outs
    while todo or time.perf_counter() - t0 < run_s:
        b, h = todo.pop(0) if todo else (int(rng.integers(p["B"])), int(rng.integers(p["Hq"])))
        r = oatt.paged_decode(q, kp, vp, tables, lens, p["scale"], p["bs"], ks, vs,
                              units=[(b, h)], widen_k=wk, widen_v=wv)
        fin.append(time.perf_counter() - t0)
        if len(outs) < len(check):
            outs[(b, h)] = r[(b, h)]
        # per (b, h) unit the oracle reads the sequence's K and V for one query head
        nbytes.append(int(lens[b]) * p["per_tok"] / p["Hkv"])
    return np.array(fin), np.array(nbytes), outs


def _oracle_worker(idx, spec, barrier, results):
    """One host core of the oracle timing (a spawned process): maps the pools the
    parent wrote (copy-on-write, nothing is copied), waits for the other cores,
    then runs the oracle for the whole timing window."""
    torch.set_num_threads(1)
    try:
        def load(name):
            path, shape, dtype = spec[name]
            m = np.memmap(path, dtype=np.uint8, mode="c")
            return torch.from_numpy(m).view(dtype).reshape(shape)
        inp = (load("q"), load("k"), load("v"), spec["ks"], spec["vs"])
        barrier.wait(timeout=600)
        results.put((idx,) + _oracle_loop(spec["p"], inp, spec["tables"], spec["lens"],
                                          spec["run_s"], 1000 + idx, spec["check"][idx]))
    except Exception as e:           # reported to the parent, which then times in-process
        results.put((-1, repr(e)))


def oracle_timing(w, inp, tables, lens, per_tok, slice_s, slices, cores=None, extra=None,
                  check_units=()):
    """Times the unmodified oracle on the host cores: one spawned single-threaded
    process per core, all started together and run for ``slices * slice_s``
    seconds over random (sequence, head) units of the workload. Each unit counts
    in the time slice it finishes in. The ``check_units`` are computed first
    (spread over the cores) and their output rows kept, so that the timed GPU
    run can be compared with them. Returns (GB/s of each slice, units of each
    slice, cores used, note, {check unit: oracle row}). Falls back to one
    in-process thread when the processes cannot be set up (cores 1, the note
    says why)."""
    import multiprocessing as mp
    import shutil
    import tempfile
    p = {"kv": w.kv_dtype, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "bs": w.bs, "scale": w.scale,
         "per_tok": per_tok, "D": w.D, **(extra or {})}
    run_s = slice_s * slices
    cores = cores or len(os.sched_getaffinity(0))
    note, runs = "", None
    if cores > 1:
        tmp, procs = None, []
        try:
            tmp = tempfile.mkdtemp(prefix=".oracle_timing_", dir=ROOT)
            spec = {"p": p, "tables": np.asarray(tables), "lens": np.asarray(lens),
                    "ks": inp[3], "vs": inp[4], "run_s": run_s,
                    "check": [list(check_units)[i::cores] for i in range(cores)]}
            for name, t in (("q", inp[0]), ("k", inp[1]), ("v", inp[2])):
                path = os.path.join(tmp, name)
                t.contiguous().view(torch.uint8).reshape(-1).numpy().tofile(path)
                spec[name] = (path, tuple(t.shape), t.dtype)
            ctx = mp.get_context("spawn")
            barrier, results = ctx.Barrier(cores), ctx.Queue()
            procs = [ctx.Process(target=_oracle_worker, args=(i, spec, barrier, results),
                                 daemon=True) for i in range(cores)]
            for pr in procs:
                pr.start()
            runs = []
            for _ in range(cores):
                r = results.get(timeout=900 + 2 * run_s)
                if r[0] < 0:
                    raise RuntimeError(r[1])
                runs.append(r[1:])
        except Exception as e:
            runs, note = None, f"; host processes unavailable ({e!r}), one thread instead"
        finally:
            for pr in procs:
                pr.join(timeout=10)
                if pr.is_alive():
                    pr.terminate()
            if tmp:
                shutil.rmtree(tmp, ignore_errors=True)
    if runs is None:
        cores = 1
        prev = torch.get_num_threads()
        torch.set_num_threads(1)
        try:
            runs = [_oracle_loop(p, inp, tables, lens, run_s, 7, list(check_units))]
        finally:
            torch.set_num_threads(prev)
    fin = np.concatenate([r[0] for r in runs])
    nb = np.concatenate([r[1] for r in runs])
    outs = {u: row for r in runs for u, row in r[2].items()}
    # the window ends when the last unit does (units started before run_s finish)
    width = max(run_s, float(fin.max()) if fin.size else run_s) / slices
    idx = np.minimum((fin / width).astype(np.int64), slices - 1)
    gbs = np.bincount(idx, weights=nb, minlength=slices) / width / 1e9
    units = np.bincount(idx, minlength=slices)
    return gbs, units, cores, note, outs


# Elementwise bound |gpu - oracle| <= atol + rtol |oracle| of the parity tests:
# the stated max-abs 2e-2 / max-rel 2e-2 read per element (6e-2 with the E4M3
# cache; float32 caches are held to 1e-5).
CHECK_TOL = {"bf16": (2e-2, 2e-2), "e4m3": (6e-2, 6e-2), "f32": (1e-5, 1e-5)}


def check_units_decode(w, n, seed=0):
    """(sequence, query head) units for the run's self-check: the longest and
    the shortest sequence, then seeded random ones."""
    rng = np.random.default_rng(seed)
    L = np.asarray(w.final_lens)
    units = [(int(np.argmax(L)), 0), (int(np.argmin(L)), w.Hq - 1)]
    while len(units) < min(n, w.B * w.Hq):
        u = (int(rng.integers(w.B)), int(rng.integers(w.Hq)))
        if u not in units:
            units.append(u)
    return units


def check_units_prefill(T, Hq, query_start, n, seed=0):
    """(chunk token, head) units: each sequence's first and last chunk token of
    the first and last sequence, then seeded random ones."""
    rng = np.random.default_rng(seed)
    qs = np.asarray(query_start)
    units = []
    for b in (0, len(qs) - 2):
        for u in ((int(qs[b]), 0), (int(qs[b + 1]) - 1, Hq - 1)):
            if qs[b + 1] > qs[b] and u not in units:
                units.append(u)
    while len(units) < min(n, T * Hq):
        u = (int(rng.integers(T)), int(rng.integers(Hq)))
        if u not in units:
            units.append(u)
    return units


def self_check(got, ref_rows, kv):
    """The GPU rows of the timed run against the oracle rows the CPU baseline
    computed: max abs error, max relative error over |oracle| > 1e-3, and whether
    every element is inside the parity tests' bound."""
    atol, rtol = CHECK_TOL[kv]
    units = sorted(ref_rows)
    g = np.stack([np.asarray(got[u[0], u[1]], dtype=np.float64) for u in units])
    r = np.stack([ref_rows[u] for u in units])
    err = np.abs(g - r)
    big = np.abs(r) > 1e-3
    return {"units": len(units), "max_abs_err": float(err.max()),
            "max_rel_err": float((err[big] / np.abs(r[big])).max()) if big.any() else 0.0,
            "atol": atol, "rtol": rtol,
            "pass": bool(np.all(np.isfinite(g)) and np.all(err <= atol + rtol * np.abs(r)))}


# ---------------------------------------------------------------- setup
def build_state(w, device):
    import paged_kv_cache_259_gb300 as pkv
    from paged_kv_cache_259_gb300.engine import PagedKVCache
    k_src, v_src = w.past_pools()
    q, k_new, v_new = w.step_inputs()
    ks = vs = 1.0
    if w.kv_dtype == "e4m3":
        ks, vs = w.fp8_scales(k_src, v_src, k_new, v_new)
    cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, KV_TORCH[w.kv_dtype], w.free_order, device)
    cache.load(k_src, v_src, ks, vs)
    cache.apply_copies(cache.replay(w.script))
    plan = cache.plan_step(w.step_seqs, max_blocks=w.max_blocks_per_seq)
    torch.cuda.synchronize()
    return cache, plan, (q, k_new, v_new, ks, vs), (k_src, v_src)


def time_steps(cache, dev, qd, kd, vd, out, w, ks, vs, ws, K, stream, has_copy):
    """K device-resident steps, twice, back to back on ``stream``. First as one
    ``paged_decode_step`` call each (copy_blocks when the step has CoW pairs,
    reshape_and_cache and the decode; the decode reads every block but the
    sequences' last ones while the writes finish): returns that pass's whole time
    (ms) and the library's launches in it. Then as separate calls with CUDA
    events around each step's decode op: returns its time per step (ms), the
    roofline's kernel time."""
    import paged_kv_cache_259_gb300 as pkv
    run = cache.bind_step(qd, kd, vd, dev, out, w.scale, ks, vs, ws)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = pkv.kernel_launches()
    t_start.record(stream)
    for _ in range(K):
        run(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = pkv.kernel_launches() - launches0
    ev_dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    for i in range(K):
        if has_copy:
            pkv.copy_blocks(cache.k_pool, cache.v_pool, dev["pairs"], stream=stream)
        pkv.reshape_and_cache(kd, vd, cache.k_pool, cache.v_pool, dev["slots"], ks, vs, stream=stream)
        ev_dec[i][0].record(stream)
        cache.decode(qd, dev, out, w.scale, ks, vs, ws, stream=stream)
        ev_dec[i][1].record(stream)
    torch.cuda.synchronize()
    return (t_start.elapsed_time(t_end), np.array([a.elapsed_time(b) for a, b in ev_dec]),
            launches)


def rewind(cache, w, max_blocks):
    """A fresh block manager in the state after the measured step's appends: the
    workload's script replayed, then that step planned (its K/V already sit in
    the pools; the script's copies were applied when the cache was built)."""
    import paged_kv_cache_259_gb300 as pkv
    cache.bm = pkv.BlockManager(w.NB, w.bs, w.free_order)
    cache.replay(w.script)
    return cache.plan_step(w.step_seqs, max_blocks=max_blocks)


def e2e_live_planning(cache, w, q, k_new, v_new, out, ks, vs, ws, stream, steps, warmup, world,
                      nb):
    """End to end through the public API, host planning included
    (``engine.LiveDecodePipeline``): every step the native block manager
    appends one token to every sequence (slots and copy-on-write pairs), builds
    the tables and finds the prefix groups straight into a pinned slab; the slab
    (plan, q, k_new, v_new) is uploaded, the step runs with that step's counts
    and its output is read back -- each step's planning and copies overlapped
    with the neighbouring steps' device work. Sequences grow by one token per
    step; the manager is rewound to the measured step's state between passes
    (outside the timed passes), and a pass ends early when the pool has no room
    for a further step. Returns ms per step, bytes per step (each step's
    algorithmic bytes at its lengths), h2d/d2h bytes per step, the median host
    planning time per step (us) and the pass length."""
    from paged_kv_cache_259_gb300 import PKV_ERR_POOL_EXHAUSTED, PagedKVError
    from paged_kv_cache_259_gb300.engine import LiveDecodePipeline
    free = w.NB - int(sum(-(-int(L) // w.bs) for L in w.final_lens))
    per_pass = max(1, min(steps, w.bs * max(1, free // w.B)))
    mb = w.max_blocks_per_seq + -(-per_pass // w.bs) + 1
    rewind(cache, w, mb)
    hq, hk, hv = q.pin_memory(), k_new.pin_memory(), v_new.pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    pipe = LiveDecodePipeline(cache, w.step_seqs, hq, hk, hv, out, mb, stream=stream)
    for i in range(2):
        v = pipe.host_inputs(i)
        v["q"].copy_(hq)
        v["k_new"].copy_(hk)
        v["v_new"].copy_(hv)

    def one_step(plan_us):
        # planning, upload, launches and read-back: one library call
        # (pkv_decode_pipeline_step), which times its planning
        try:
            pipe.submit(hout, w.scale, ks, vs, ws)
        except PagedKVError as e:
            if e.status != PKV_ERR_POOL_EXHAUSTED:
                raise
            return False                   # no room for another step in this pass
        plan_us.append(pipe.last_plan_us)
        return True

    warm_us = []
    for _ in range(min(warmup, per_pass)):
        if not one_step(warm_us):
            break
    torch.cuda.synchronize()
    total_ms, total_bytes, done, plan_us = 0.0, 0.0, 0, []
    while done < steps:
        rewind(cache, w, mb)
        n = min(per_pass, steps - done)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0.record(pipe.up)
        k = 0
        for _ in range(n):
            if not one_step(plan_us):
                break
            k += 1
            # the pass's k-th step attends over k more tokens per sequence than
            # the measured step (one appended per sequence per step)
            total_bytes += nb["total"] + k * w.B * nb["per_token"]
        e1.record(pipe.down)
        torch.cuda.synchronize()
        if k == 0:
            raise RuntimeError("e2e: the pool has no room for a single further step")
        total_ms += e0.elapsed_time(e1)
        done += k
    return {"ms": total_ms / done, "bytes": total_bytes / done, "h2d": pipe.slab_bytes,
            "d2h": hout.numel() * hout.element_size(),
            "host_plan_us": float(np.median(plan_us)), "steps": done, "per_pass": per_pass}


def run_gpu(args, rank, world, device):
    import paged_kv_cache_259_gb300 as pkv
    w = make_workload(args)
    cache, plan, (q, k_new, v_new, ks, vs), (k_src, v_src) = build_state(w, device)
    stream = torch.cuda.current_stream(device)
    dev = plan.device_tensors(device)
    qd, kd, vd = q.to(device), k_new.to(device), v_new.to(device)
    out = torch.empty(w.B, w.Hq, w.D, dtype=w.src_dtype, device=device)
    ws = cache.workspace(w.B, w.max_blocks_per_seq)
    nbytes = step_bytes(w, plan.tables, plan.lens, len(plan.pairs))
    has_copy = len(plan.pairs) > 0

    def step():
        cache.step(qd, kd, vd, dev, out, w.scale, ks, vs, ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    # ---- device-resident timing: whole step, plus the decode op alone per step
    K = args.steps
    clocks = ClockSampler(device.index if device.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    total_ms, dec_ms, launches_timed = time_steps(cache, dev, qd, kd, vd, out, w, ks, vs, ws, K,
                                                  stream, has_copy)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    out_timed = out.float().cpu()                        # the timed steps' result (self-check)
    launches_per_step = count_launches(step)

    # ---- end to end through the public API, host planning included
    e2e = e2e_live_planning(cache, w, q, k_new, v_new, out, ks, vs, ws, stream,
                            max(50, K // 4), max(4, args.warmup // 4), world, nbytes)
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error in the end-to-end steps")

    res = {"w": w, "nbytes": nbytes, "ms_per_step": total_ms / K, "dec_ms": float(dec_ms.mean()),
           "dec_ms_median": float(np.median(dec_ms)), "e2e": e2e,
           "clocks": clk, "launches": launches_timed, "groups": plan.num_groups,
           "launches_per_step": launches_per_step, "out": out_timed,
           "cpu": (q, k_src, v_src, ks, vs, plan)}
    return res


OTHER_DECODE = ["gqa_chat_bf16", "shared_prefix_bf16", "shared_prefix_fork_bf16",
                "long_fp8_bs16", "long_fp8_bs32", "beam_search_bf16"]


def run_other(name, steps, warmup, device, peak):
    """Another decode workload, timed like the headline's device-resident steps
    (fewer of them), with its self-check: the GPU rows of the timed steps
    against oracle rows computed on one host core (the check units of a
    one-core oracle timing run with no time budget beyond them)."""
    import paged_kv_cache_259_gb300 as pkv
    w = wl.CONFIGS[name]()
    cache, plan, (q, k_new, v_new, ks, vs), (k_src, v_src) = build_state(w, device)
    stream = torch.cuda.current_stream(device)
    dev = plan.device_tensors(device)
    qd, kd, vd = q.to(device), k_new.to(device), v_new.to(device)
    out = torch.empty(w.B, w.Hq, w.D, dtype=w.src_dtype, device=device)
    ws = cache.workspace(w.B, w.max_blocks_per_seq)
    nb = step_bytes(w, plan.tables, plan.lens, len(plan.pairs))
    has_copy = len(plan.pairs) > 0
    for _ in range(warmup):
        cache.step(qd, kd, vd, dev, out, w.scale, ks, vs, ws)
    torch.cuda.synchronize()
    if pkv.get_device_error() != 0:
        raise RuntimeError(f"{name}: device error during warm-up")
    total_ms, dec_ms, _ = time_steps(cache, dev, qd, kd, vd, out, w, ks, vs, ws, steps, stream,
                                     has_copy)
    if pkv.get_device_error() != 0:
        raise RuntimeError(f"{name}: device error in the timed region")
    got = out.float().cpu()
    groups = plan.num_groups
    del cache, dev, qd, kd, vd, out, ws
    torch.cuda.empty_cache()
    kp, vp, tables, lens = oracle_inputs_for_step(w, q, k_src, v_src, plan)
    n_check = 8 if w.kv_dtype == "e4m3" else 24
    _, _, _, _, ref_rows = oracle_timing(w, (q, kp, vp, ks, vs), tables, lens, nb["per_token"],
                                         0.0, 1, cores=1,
                                         check_units=check_units_decode(w, n_check))
    ms = total_ms / steps
    dgbs = nb["decode"] / (float(dec_ms.mean()) * 1e-3) / 1e9
    return {"workload": workload_desc(w), "kv": w.kv_dtype, "steps": steps,
            "decode_gbs": round(dgbs, 2), "frac": round(dgbs / peak, 4),
            "decode_ms": round(float(dec_ms.mean()), 5),
            "decode_bytes": nb["decode"], "decode_logical_bytes": nb["decode_logical"],
            "step_gbs": round(nb["total"] / (ms * 1e-3) / 1e9, 2), "ms_per_step": round(ms, 5),
            "seq_steps_per_s": round(w.B / (ms * 1e-3), 1), "cow_pairs": int(len(plan.pairs)),
            "prefix_groups": groups, "traffic": measured_traffic(name),
            "check": self_check(got, ref_rows, w.kv_dtype)}


def count_launches(step, reps=3):
    """Kernels of this library one step launches (the library counts them)."""
    import paged_kv_cache_259_gb300 as pkv
    n0 = pkv.kernel_launches()
    for _ in range(reps):
        step()
    torch.cuda.synchronize()
    return (pkv.kernel_launches() - n0) // reps


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def oracle_inputs_for_step(w, q, k_src, v_src, plan):
    """CPU pools after the step's writes, as the oracle sees them (source values;
    no GPU data). Built with the oracle's own block manager and cache ops."""
    from oracle import cache_ops as oops
    from oracle.block_manager import BlockManager as OBM, replay
    bm = OBM(w.NB, w.bs, w.free_order)
    pairs = replay(bm, w.script)
    step = [bm.append_slot(s) for s in w.step_seqs]
    kp, vp = k_src, v_src                   # in place: the bench's copies are not reused
    oops.copy_blocks(kp, vp, pairs + [c for _, c in step if c is not None])
    _, k_new, v_new = w.step_inputs()
    oops.reshape_and_cache(k_new, v_new, kp, vp, torch.tensor([s for s, _ in step]), w.bs)
    MB = w.max_blocks_per_seq
    tables = np.full((w.B, MB), -1, dtype=np.int64)
    for i, s in enumerate(w.step_seqs):
        t = bm.block_table(s)
        tables[i, :len(t)] = t
    lens = np.array([bm.seq_len(s) for s in w.step_seqs])
    return kp, vp, tables, lens


# ---------------------------------------------------------------- chunked prefill
PREFILL_METRIC = ("paged chunked-prefill attention: achieved TFLOP/s (% of bf16 tensor peak) "
                  "and chunk tokens/s")


def prefill_flops(w, lens=None, chunks=None):
    """Algorithmic FLOPs of the step's attention: chunk token i of sequence b sees
    p + 1 keys (p = L_b - C_b + i), and per (token, head, key) Q.K and P.V are
    2 * D multiply-adds each."""
    L = np.asarray(w.final_lens if lens is None else lens, dtype=np.float64)
    C = np.asarray(w.chunks if chunks is None else chunks, dtype=np.float64)
    keys = C * (L - C) + C * (C + 1) / 2
    return float(keys.sum()) * w.Hq * 4 * w.D


def prefill_oracle_inputs(w, k_src, v_src, k_new, v_new):
    """CPU pools after the step's writes (the oracle's own block manager and
    cache ops; no GPU data), block tables and lengths."""
    from oracle import cache_ops as oops
    from oracle.block_manager import BlockManager as OBM
    bm = OBM(w.NB, w.bs, w.free_order)
    pairs = []
    for op in w.script:
        if op[0] == "add":
            bm.add_seq(op[1])
        elif op[0] == "fork":
            bm.fork(op[1], op[2])
        else:
            for _ in range(op[2]):
                c = bm.append_slot(op[1])[1]
                if c is not None:
                    pairs.append(c)
    slots = []
    for sid, n in zip(w.step_seqs, w.chunks):
        for _ in range(int(n)):
            slot, c = bm.append_slot(sid)
            slots.append(slot)
            if c is not None:
                pairs.append(c)
    kp, vp = k_src, v_src
    oops.copy_blocks(kp, vp, pairs)
    oops.reshape_and_cache(k_new, v_new, kp, vp, torch.tensor(slots, dtype=torch.int64), w.bs)
    tables = np.full((w.B, w.max_blocks_per_seq), -1, dtype=np.int64)
    for i, sid in enumerate(w.step_seqs):
        t = bm.block_table(sid)
        tables[i, :len(t)] = t
    lens = np.array([bm.seq_len(sid) for sid in w.step_seqs])
    return kp, vp, tables, lens


PREFILL_SOURCES = ["pkv_prefill.cu", "pkv_tcgen05.cuh"]


def prefill_source_hash():
    return code_hash(PREFILL_SOURCES)


def prefill_traffic(config):
    """DRAM bytes per prefill launch from profiles/prefill_traffic.json (one ncu
    capture at full size), or None for other kernel sources or workloads."""
    try:
        with open(os.path.join(ROOT, "profiles", "prefill_traffic.json")) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("kernel_source_sha") != prefill_source_hash():
        return None
    e = t.get("workloads", {}).get(config)
    return None if e is None else e.get("dram_bytes_per_launch")


def prefill_workload(args):
    make = {**wl.PREFILL_CONFIGS, **wl.PROMPT_CONFIGS}[args.config]
    return make() if args.batch is None else make(B=args.batch)


def run_prefill(args, rank, world, device):
    """One chunked-prefill step (CoW copies, the chunk's K/V into the cache,
    causal attention of every chunk token), timed like the decode step."""
    import paged_kv_cache_259_gb300 as pkv
    from paged_kv_cache_259_gb300.engine import PagedKVCache
    w = prefill_workload(args)
    k_src, v_src = w.past_pools()
    prompts = isinstance(w, wl.PromptWorkload)
    cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, torch.bfloat16, w.free_order, device,
                         prefix_caching=prompts)
    cache.load(k_src, v_src)
    plan_s = 0.0
    if prompts:
        # serve the system prompt first (its blocks are then cached), then plan
        # the batch: each request reuses them and computes only the rest
        warm = cache.plan_prompts([10 ** 9], w.warm, max_blocks=w.max_blocks_per_seq)
        wq, wk, wv = (t.to(device) for t in w.rows("warm", 0, 0, len(w.warm[0])))
        wout = torch.empty(wq.shape, dtype=torch.bfloat16, device=device)
        cache.prefill_step(wq, wk, wv, warm.device_tensors(device), wout, w.scale,
                           warm.max_query_len)
        cache.bm.free_seq(10 ** 9)
        t_plan = time.perf_counter()
        plan = cache.plan_prompts(list(range(w.B)), w.prompts, max_blocks=w.max_blocks_per_seq)
        plan_s = time.perf_counter() - t_plan
        rows = [w.rows("step", b, int(n), len(p)) for b, (p, n) in enumerate(zip(w.prompts, plan.cached))]
        q, k_new, v_new = (torch.cat([r[i] for r in rows]) for i in range(3))
    else:
        q, k_new, v_new = w.step_inputs()
        cache.apply_copies(cache.replay(w.script))
        plan = cache.plan_prefill(w.step_seqs, w.chunks, max_blocks=w.max_blocks_per_seq)
    mql = plan.max_query_len
    stream = torch.cuda.current_stream(device)
    dev = plan.device_tensors(device)
    qd, kd, vd = q.to(device), k_new.to(device), v_new.to(device)
    out = torch.empty(int(plan.chunks.sum()), w.Hq, w.D, dtype=torch.bfloat16, device=device)
    torch.cuda.synchronize()

    def step():
        cache.prefill_step(qd, kd, vd, dev, out, w.scale, mql, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device.index if device.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    # the step as one paged_prefill_step call (step time, launches), then as
    # separate calls with CUDA events around the attention (the roofline's time)
    launches0 = pkv.kernel_launches()
    t0.record(stream)
    for i in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    launches = pkv.kernel_launches() - launches0
    for i in range(K):
        if dev["pairs"].shape[0]:
            pkv.copy_blocks(cache.k_pool, cache.v_pool, dev["pairs"], stream=stream)
        pkv.reshape_and_cache(kd, vd, cache.k_pool, cache.v_pool, dev["slots"], stream=stream)
        ev[i][0].record(stream)
        pkv.paged_attention_prefill(out, qd, cache.k_pool, cache.v_pool, dev["tables"],
                                    dev["lens"], dev["query_start"], w.scale, mql, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    att_ms = np.array([a.elapsed_time(b) for a, b in ev])
    out_timed = out.float().cpu()                        # the timed steps' result (self-check)
    launches_per_step = count_launches(step)

    host = plan.host_tensors(pin=True)
    hq, hk, hv = q.pin_memory(), k_new.pin_memory(), v_new.pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    # end to end: every step's inputs uploaded from one pinned slab and its
    # output read back, overlapped with the neighbouring steps (StepPipeline)
    from paged_kv_cache_259_gb300.engine import StepPipeline
    host.update(q=hq, k_new=hk, v_new=hv)
    pipe = StepPipeline(cache, host, out, stream=stream,
                        run=lambda q_, k_, v_, pl, o, s: cache.prefill_step(
                            q_, k_, v_, pl, o, w.scale, mql, stream=s))
    for i in range(2):
        for k, view in pipe.host_inputs(i).items():
            view.copy_(host[k])
    h2d = pipe.slab_bytes
    d2h = hout.numel() * hout.element_size()
    for _ in range(4):
        pipe.submit(hout)
    torch.cuda.synchronize()
    K2 = max(4, K // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    e0.record(pipe.up)
    for _ in range(K2):
        pipe.submit(hout)
    e1.record(pipe.down)
    torch.cuda.synchronize()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error in the end-to-end steps")
    return {"w": w, "ms_per_step": t0.elapsed_time(t1) / K, "att_ms": float(att_ms.mean()),
            "att_ms_median": float(np.median(att_ms)), "e2e_ms": e0.elapsed_time(e1) / K2,
            "h2d": h2d, "d2h": d2h, "clocks": clk, "launches": launches,
            "launches_per_step": launches_per_step, "pairs": int(plan.pairs.shape[0]),
            "plan": plan, "plan_s": plan_s, "T": int(plan.chunks.sum()), "out": out_timed,
            "cpu": (q, k_src, v_src, k_new, v_new)}


def prompt_stats(w, plan, r, ms, world):
    """Prefix-cache figures of a prompt workload's step."""
    served = int(np.sum(plan.lens))
    cached = int(np.sum(plan.cached))
    return {"prompt_tokens_per_s": round(world * served / (ms * 1e-3), 1),
            "cached_fraction": round(cached / served, 4),
            "host_plan_us_per_request": round(1e6 * r["plan_s"] / w.B, 2)}


def prefill_workload_desc(w):
    if isinstance(w, wl.PromptWorkload):
        L = np.asarray(w.final_lens)
        return (f"{w.name}: B={w.B} requests of {int(L.min())}..{int(L.max())} prompt tokens that "
                f"all begin with one {len(w.warm[0])}-token system prompt, served first (prefix "
                f"caching: its full blocks are reused), Hq={w.Hq}, Hkv={w.Hkv}, D={w.D}, "
                f"block_size={w.bs}, NB={w.NB}, bf16")
    ctx = np.asarray(w.final_lens) - np.asarray(w.chunks)
    return (f"{w.name}: B={w.B}, chunk={int(w.chunks[0])} tokens per sequence (T={w.T}), "
            f"context {int(ctx.min())}..{int(ctx.max())} cached tokens, Hq={w.Hq}, Hkv={w.Hkv}, "
            f"D={w.D}, block_size={w.bs}, NB={w.NB}, bf16")


def prompt_oracle_inputs(w, k_src, v_src):
    """Oracle pools, tables, lengths and chunk offsets of a prompt workload's step:
    the oracle's prefix-caching manager serves the warm prompt, releases it, then
    plans the batch (no GPU data)."""
    from oracle import cache_ops as oops
    from oracle.prefix_cache import PrefixCachingBlockManager as OPC
    bm = OPC(w.NB, w.bs, w.free_order)
    kp, vp = k_src, v_src
    for phase, ids, prompts in (("warm", [10 ** 9], w.warm), ("step", list(range(w.B)), w.prompts)):
        cached, slots, pairs = [], [], []
        for sid, p in zip(ids, prompts):
            n = bm.add_seq_prompt(sid, p)
            cached.append(n)
            for t in p[n:]:
                s_, c = bm.append_token(sid, int(t))
                slots.append(s_)
                if c is not None:
                    pairs.append(c)
        rows = [w.rows(phase, b, int(n), len(p)) for b, (p, n) in enumerate(zip(prompts, cached))]
        oops.copy_blocks(kp, vp, pairs)
        oops.reshape_and_cache(torch.cat([r[1] for r in rows]), torch.cat([r[2] for r in rows]),
                               kp, vp, torch.tensor(slots, dtype=torch.int64), w.bs)
        if phase == "warm":
            for sid in ids:
                bm.free_seq(sid)
    tables = np.full((w.B, w.max_blocks_per_seq), -1, dtype=np.int64)
    for i in range(w.B):
        t = bm.block_table(i)
        tables[i, :len(t)] = t
    lens = np.array([bm.seq_len(i) for i in range(w.B)])
    chunks = [len(p) - n for p, n in zip(w.prompts, cached)]
    return kp, vp, tables, lens, np.concatenate([[0], np.cumsum(chunks)])


def prefill_cpu_inputs(w, cpu):
    q, k_src, v_src, k_new, v_new = cpu
    if isinstance(w, wl.PromptWorkload):
        kp, vp, tables, lens, qs = prompt_oracle_inputs(w, k_src, v_src)
        return (q, kp, vp, 1.0, 1.0), tables, lens, qs
    kp, vp, tables, lens = prefill_oracle_inputs(w, k_src, v_src, k_new, v_new)
    return (q, kp, vp, 1.0, 1.0), tables, lens, w.query_start


def prefill_main(args, rank, world, device):
    r = run_prefill(args, rank, world, device)
    w, plan = r["w"], r["plan"]
    ms = max_over_ranks(r["ms_per_step"], world, device)
    att_ms = max_over_ranks(r["att_ms"], world, device)
    e2e_ms = max_over_ranks(r["e2e_ms"], world, device)
    fl = prefill_flops(w, plan.lens, plan.chunks)
    peak, kind = load_tensor_peak()
    if rank != 0:
        return
    cpu_line, check = None, None
    if args.cpu_budget > 0:                           # <= 0: profiling runs skip the CPU leg
        inp, tables, lens, qs = prefill_cpu_inputs(w, r["cpu"])
        extra = {"mode": "prefill", "query_start": qs}
        gf, units, cores, note, ref_rows = oracle_timing(
            w, inp, tables, lens, 0, args.cpu_budget, 1, extra=extra,
            check_units=check_units_prefill(r["T"], w.Hq, qs, 48))
        cpu_line = {
            "value": round(float(gf[0]) / 1e3, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{int(units[0])} random (chunk token, head) rows of this workload in "
                      f"{args.cpu_budget:.1f} s on {cores} host cores (one single-threaded "
                      f"float64 oracle process per core){note}"}
        check = {**self_check(r["out"], ref_rows, "bf16"),
                 "of": "the timed steps' output rows against the oracle rows of the "
                       "cpu_baseline run (its first units)"}
    att_tf = fl / (att_ms * 1e-3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": round(world * fl / (ms * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": prefill_workload_desc(w),
            "step": ("paged_prefill_step: copy_blocks (CoW pairs: %d) + reshape_and_cache of %d "
                     "chunk tokens + paged_attention_prefill; %d kernel launches per step"
                     % (r["pairs"], r["T"], r["launches_per_step"])),
            "l2": "K/V of the step's sequences %.2f GB vs %d MB L2; the chunk's K/V "
                  "(%.0f MB) is rewritten every step" % (
                      float(np.sum(w.final_lens)) * 2 * w.Hkv * w.D * 2 / 1e9, L2_BYTES >> 20,
                      r["T"] * 2 * w.Hkv * w.D * 2 / 1e6),
            "flops_per_step": fl,
            "chunk_tokens_per_s": round(world * r["T"] / (ms * 1e-3), 1),
            **(prompt_stats(w, plan, r, ms, world) if isinstance(w, wl.PromptWorkload) else {}),
            "step_frac_of_peak": round(fl / (ms * 1e-3) / 1e12 / peak, 4),
        },
        "roofline": {
            "kernel": "paged_attention_prefill (tcgen05)", "bound": "tensor",
            "achieved": round(att_tf, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(att_tf / peak, 4),
            "traffic": prefill_traffic(args.config) if args.batch is None else None,
            "peak_source": f"{kind} bf16_tflops (dense bf16 GEMM burst, MEASURED_PEAKS.json)",
            "flops_per_launch": fl, "ms_per_launch": round(att_ms, 5),
            "ms_per_launch_median": round(r["att_ms_median"], 5),
        },
        "cpu_baseline": cpu_line,
        "e2e": {"value": round(world * fl / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": round(e2e_ms, 5),
                "note": "engine.StepPipeline: each step's q/k/v and plan uploaded from one "
                        "pinned slab and its output read back inside the timed region, "
                        "overlapped with the neighbouring steps (bound by the host link)"},
        "check": check,
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    print(json.dumps(line), flush=True)


def run_reference_prefill(args):
    """Reference arm for a chunked-prefill workload: the oracle on the host cores."""
    w = prefill_workload(args)
    k_src, v_src = w.past_pools()
    if isinstance(w, wl.PromptWorkload):
        kp, vp, tables, lens, qs = prompt_oracle_inputs(w, k_src, v_src)
        cached = np.asarray(lens) - np.diff(qs)
        rows = [w.rows("step", b, int(n), len(p)) for b, (p, n) in enumerate(zip(w.prompts, cached))]
        inp = (torch.cat([r[0] for r in rows]), kp, vp, 1.0, 1.0)
    else:
        q, k_new, v_new = w.step_inputs()
        inp, tables, lens, qs = prefill_cpu_inputs(w, (q, k_src, v_src, k_new, v_new))
    slice_s = 120.0 / (args.steps + args.warmup)
    gf, units, cores, note, _ = oracle_timing(w, inp, tables, lens, 0, slice_s,
                                              args.warmup + args.steps,
                                              extra={"mode": "prefill", "query_start": qs})
    value = float(gf[args.warmup:].mean()) / 1e3
    line = {
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6),
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * slice_s, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": prefill_workload_desc(w)},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{int(units[args.warmup:].sum())} random (chunk token, head) "
                                   f"rows finished in {args.steps} time slices of {slice_s:.3f} s "
                                   f"on {cores} host cores{note}"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- swapping
SWAP_METRIC = ("swap of preempted sequences' KV blocks between HBM and pinned host memory: "
               "achieved GB/s of block bytes moved (% of the measured copy-engine rate)")


def swap_plans(bm, victims, n):
    """Host half of n swap steps: every victim swapped out, then every victim
    swapped back in; returns [(out pairs, in pairs)] as int64 [P, 2] arrays."""
    plans = []
    for _ in range(n):
        o = np.concatenate([bm.swap_out(int(s)) for s in victims])
        i = np.concatenate([bm.swap_in(int(s)) for s in victims])
        plans.append((np.asarray(o, dtype=np.int64).reshape(-1, 2),
                      np.asarray(i, dtype=np.int64).reshape(-1, 2)))
    return plans


def copy_engine_rate(nbytes, device, reps=5):
    """GB/s of one contiguous device->pinned-host copy plus one pinned-host->device
    copy of ``nbytes`` each (cudaMemcpyAsync on the copy engines), best of reps."""
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d.fill_(1)
    stream = torch.cuda.current_stream(device)
    best = {}
    for name, dst, src in (("d2h", h, d), ("h2d", d, h)):
        ts = []
        for _ in range(reps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        best[name] = min(ts[1:])
    return 2 * nbytes / ((best["d2h"] + best["h2d"]) * 1e-3) / 1e9, best


def swap_copy_engine_path(cache, sw, stream, n):
    """The same swap steps with the host link crossed by the copy engines: a
    gather launch (HBM to HBM) into a contiguous staging buffer, one
    cudaMemcpyAsync per run of consecutive host blocks each way, a scatter
    launch. Pairs and runs planned beforehand; returns GB/s over n steps and a
    callable that issues the next planned step on a stream."""
    import paged_kv_cache_259_gb300 as pkv
    from paged_kv_cache_259_gb300.engine import host_runs
    dev = cache.device
    P = sw.victim_blocks
    sk, sv = cache.staging_pools(P)
    idx = np.arange(P)
    plans = []
    for o, i in swap_plans(cache.bm, sw.victims, n + 3 + 64):
        plans.append((torch.as_tensor(np.stack([o[:, 0], idx], 1), device=dev), host_runs(o[:, 1]),
                      torch.as_tensor(np.stack([idx, i[:, 1]], 1), device=dev), host_runs(i[:, 0])))
    state = {"next": 0}

    def step(st):
        go, ro, si, ri = plans[state["next"]]
        state["next"] += 1
        pkv.swap_blocks(sk, sv, cache.k_pool, cache.v_pool, go, st)
        with torch.cuda.stream(st):
            for a, b, h in ro:
                cache.host_k[h:h + b - a].copy_(sk[a:b], non_blocking=True)
                cache.host_v[h:h + b - a].copy_(sv[a:b], non_blocking=True)
            for a, b, h in ri:
                sk[a:b].copy_(cache.host_k[h:h + b - a], non_blocking=True)
                sv[a:b].copy_(cache.host_v[h:h + b - a], non_blocking=True)
        pkv.swap_blocks(cache.k_pool, cache.v_pool, sk, sv, si, st)

    for _ in range(3):
        step(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error in the copy-engine swap steps")
    ms = e0.elapsed_time(e1) / n
    runs = np.mean([len(p_[1]) + len(p_[3]) for p_ in plans[:n]])
    return {"gbs": round(2 * P * 2 * cache.k_pool[0].numel() * cache.k_pool.element_size() /
                         (ms * 1e-3) / 1e9, 2),
            "ms_per_step": round(ms, 5), "host_runs_per_step": float(runs), "step": step}


def swap_overlap(cache, sw, w, device, ce_path, others, plan):
    """Decode steps of the sequences that stay on the device (``others``, their
    step ``plan``), on one stream, while one swap step (all victims out, then
    in) runs on another: the time of the two together against each alone, for
    the SM-kernel swap and for the copy-engine one."""
    import paged_kv_cache_259_gb300 as pkv
    dev = plan.device_tensors(device)
    q, k_new, v_new = (t[others].to(device) for t in w.step_inputs())
    out = torch.empty(len(others), w.Hq, w.D, dtype=torch.bfloat16, device=device)
    ws = cache.workspace(len(others), w.max_blocks_per_seq)
    sa, sb = torch.cuda.Stream(device), torch.cuda.Stream(device)
    P = sw.victim_blocks
    kplans = [(torch.as_tensor(o, device=device), torch.as_tensor(i, device=device))
              for o, i in swap_plans(cache.bm, sw.victims, 8)]
    kstate = {"next": 0}

    def kernel_swap(st):
        o, i = kplans[kstate["next"]]
        kstate["next"] += 1
        pkv.swap_blocks(cache.host_k, cache.host_v, cache.k_pool, cache.v_pool, o, st)
        pkv.swap_blocks(cache.k_pool, cache.v_pool, cache.host_k, cache.host_v, i, st)

    def decode(st, m):
        for _ in range(m):
            cache.step(q, k_new, v_new, dev, out, w.scale, workspace=ws, stream=st)

    def timed(fn):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(sa)
        sb.wait_event(e0)
        fn()
        done = torch.cuda.Event()
        done.record(sb)
        sa.wait_event(done)
        e1.record(sa)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    decode(sa, 5)
    t1 = timed(lambda: decode(sa, 20)) / 20
    ts_k = timed(lambda: kernel_swap(sb))
    ts_c = timed(lambda: ce_path["step"](sb))
    m = max(1, int(round(ts_c / t1)))
    alone = timed(lambda: decode(sa, m))
    both_k = timed(lambda: (kernel_swap(sb), decode(sa, m)))
    both_c = timed(lambda: (ce_path["step"](sb), decode(sa, m)))
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error in the overlap steps")
    return {"decode_batch": len(others), "decode_steps": m, "decode_ms": round(alone, 4),
            "swap_ms_kernel": round(ts_k, 4), "swap_ms_copy_engines": round(ts_c, 4),
            "together_ms_kernel": round(both_k, 4), "together_ms_copy_engines": round(both_c, 4)}


def swap_oracle_state(sw, k_src, v_src):
    """The oracle's block manager after the workload's script, with its pools."""
    from oracle.block_manager import BlockManager as OracleBM
    w = sw.base
    bm = OracleBM(w.NB, w.bs, list(w.free_order), num_cpu_blocks=sw.num_host_blocks)
    for op in w.script:
        if op[0] == "add":
            bm.add_seq(op[1])
        else:
            for _ in range(op[2]):
                bm.append_slot(op[1])
    hk = torch.zeros((sw.num_host_blocks,) + tuple(k_src.shape[1:]), dtype=k_src.dtype)
    return bm, k_src, v_src, hk, torch.zeros_like(hk)


def swap_oracle_timing(sw, k_src, v_src, slice_s, slices):
    """The oracle (block manager swap + whole-block copies on host tensors), one
    thread, for ``slices`` windows of ``slice_s`` s; a step (all victims out,
    then in) counts in the window it finishes in. Returns GB/s per window and
    steps per window."""
    from oracle import cache_ops as oops
    bm, kp, vp, hk, hv = swap_oracle_state(sw, k_src, v_src)
    step_bytes = 2 * sw.victim_blocks * 2 * kp[0].numel() * kp.element_size()
    prev = torch.get_num_threads()
    torch.set_num_threads(1)
    fin = []
    try:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < slice_s * slices:
            for s in sw.victims:
                oops.swap_blocks(hk, hv, kp, vp, bm.swap_out(s))
            for s in sw.victims:
                oops.swap_blocks(kp, vp, hk, hv, bm.swap_in(s))
            fin.append(time.perf_counter() - t0)
    finally:
        torch.set_num_threads(prev)
    fin = np.array(fin)
    width = max(slice_s * slices, float(fin.max()) if fin.size else 0.0) / slices
    idx = np.minimum((fin / width).astype(np.int64), slices - 1)
    steps = np.bincount(idx, minlength=slices)
    return steps * step_bytes / width / 1e9, steps


def swap_workload_desc(sw):
    w = sw.base
    L = np.asarray(w.final_lens) - 1
    Lv = L[sw.victims]
    return (f"{sw.name}: B={w.B} sequences holding L in [{L.min()}, {L.max()}] tokens "
            f"(LLaMA-13B layer: Hkv={w.Hkv}, D={w.D}, block_size={w.bs}, bf16, NB={w.NB}); "
            f"the newest {len(sw.victims)} (L mean {Lv.mean():.1f}, {sw.victim_blocks} blocks) "
            f"swapped out to a pinned host pool of {sw.num_host_blocks} blocks and back in "
            f"each step")


def swap_main(args, rank, world, device):
    import paged_kv_cache_259_gb300 as pkv
    from paged_kv_cache_259_gb300.engine import PagedKVCache
    sw = wl.SWAP_CONFIGS[args.config]()
    w = sw.base
    cache = PagedKVCache(w.NB, w.Hq, w.Hkv, w.D, w.bs, torch.bfloat16, w.free_order, device,
                         num_host_blocks=sw.num_host_blocks)
    k_src, v_src = w.past_pools()
    cache.load(k_src, v_src)
    cache.replay(w.script)
    stream = torch.cuda.current_stream(device)
    block_bytes = w.Hkv * w.bs * w.D * 2
    P = sw.victim_blocks
    dir_bytes = P * 2 * block_bytes                         # K and V blocks, one direction
    step_bytes = 2 * dir_bytes
    K, W = args.steps, args.warmup
    plans = [(torch.as_tensor(o, device=device), torch.as_tensor(i, device=device))
             for o, i in swap_plans(cache.bm, sw.victims, W + K)]

    def step(o, i):
        pkv.swap_blocks(cache.host_k, cache.host_v, cache.k_pool, cache.v_pool, o, stream)
        pkv.swap_blocks(cache.k_pool, cache.v_pool, cache.host_k, cache.host_v, i, stream)

    for o, i in plans[:W]:
        step(o, i)
    torch.cuda.synchronize()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device.index if device.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = pkv.kernel_launches()
    t_start.record(stream)
    for k in range(K):
        o, i = plans[W + k]
        ev[k][0].record(stream)
        pkv.swap_blocks(cache.host_k, cache.host_v, cache.k_pool, cache.v_pool, o, stream)
        ev[k][1].record(stream)
        pkv.swap_blocks(cache.k_pool, cache.v_pool, cache.host_k, cache.host_v, i, stream)
        ev[k][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = pkv.kernel_launches() - launches0
    clk = clocks.stop()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    ms = max_over_ranks(t_start.elapsed_time(t_end) / K, world, device)
    out_ms = float(np.mean([a.elapsed_time(b) for a, b, _ in ev]))
    in_ms = float(np.mean([b.elapsed_time(c) for _, b, c in ev]))

    # end to end through the engine: block-manager swaps on the host, pair
    # upload, both copies; wall clock around whole steps
    for _ in range(3):
        cache.swap_out(sw.victims, stream)
        cache.swap_in(sw.victims, stream)
    torch.cuda.synchronize()
    K2 = max(3, K // 2)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(K2):
        cache.swap_out(sw.victims, stream)
        cache.swap_in(sw.victims, stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / K2, world, device)
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error in the end-to-end steps")
    peak, ce = copy_engine_rate(dir_bytes, device)
    # the staying sequences' decode plan first: their blocks are then never a
    # destination of the swaps planned after it
    others = [s_ for s_ in range(w.B) if s_ not in sw.victims]
    dplan = cache.plan_step(others, max_blocks=w.max_blocks_per_seq)
    ce_path = swap_copy_engine_path(cache, sw, stream, max(3, K // 2))
    overlap = swap_overlap(cache, sw, w, device, ce_path, others, dplan)
    if rank != 0:
        return
    gbs, steps = swap_oracle_timing(sw, k_src, v_src, args.cpu_budget, 1)
    achieved = step_bytes / ((out_ms + in_ms) * 1e-3) / 1e9
    line = {
        "metric": SWAP_METRIC, "value": round(world * step_bytes / (ms * 1e-3) / 1e9, 2),
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": swap_workload_desc(sw),
            "step": ("swap_blocks device->host (%d block pairs, K and V) + swap_blocks "
                     "host->device (%d pairs); pairs planned by the block manager beforehand "
                     "and resident on the device" % (P, P)),
            "l2": "inputs larger than L2: %.0f MB of device blocks read per step vs %d MB L2"
                  % (dir_bytes / 1e6, L2_BYTES >> 20),
            "bytes_per_step": step_bytes,
            "swap_out_gbs": round(dir_bytes / (out_ms * 1e-3) / 1e9, 2),
            "swap_in_gbs": round(dir_bytes / (in_ms * 1e-3) / 1e9, 2),
            "copy_engine_ms": {k: round(v, 5) for k, v in ce.items()},
            "sequences_swapped_per_s": round(world * 2 * len(sw.victims) / (ms * 1e-3), 1),
            "copy_engine_path": {k: v for k, v in ce_path.items() if k != "step"},
            "overlap_with_decode": overlap,
        },
        "roofline": {
            "kernel": "swap_blocks (out + in)", "bound": "host-link",
            "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": None,
            "peak_source": ("measured in this run: one contiguous cudaMemcpyAsync of the same "
                            "bytes device->pinned host plus one back (copy engines)"),
            "traffic_note": "null: the bound is the host link; the device side reads and "
                            "writes the same block bytes once",
            "bytes_per_launch": dir_bytes,
            "ms_per_launch": round((out_ms + in_ms) / 2, 5),
        },
        "cpu_baseline": {
            "value": round(float(gbs[0]), 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{int(steps[0])} whole swap steps (block-manager swaps plus whole-block "
                      f"copies of host tensors) of this workload in {args.cpu_budget:.1f} s on "
                      f"one host thread",
        },
        "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": dir_bytes + 2 * P * 16, "d2h_bytes_per_step": dir_bytes,
                "ms_per_step": round(e2e_ms, 5),
                "note": "wall clock around engine swap_out + swap_in (host block manager, "
                        "pair upload, both copies)"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_reference_swap(args):
    """Reference arm for the swap workload: the oracle on one host thread."""
    sw = wl.SWAP_CONFIGS[args.config]()
    k_src, v_src = sw.base.past_pools()
    slice_s = 120.0 / (args.steps + args.warmup)
    gbs, steps = swap_oracle_timing(sw, k_src, v_src, slice_s, args.warmup + args.steps)
    value = float(gbs[args.warmup:].mean())
    line = {
        "impl": "reference", "metric": SWAP_METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * slice_s, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": swap_workload_desc(sw)},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{int(steps[args.warmup:].sum())} whole swap steps finished "
                                   f"in {args.steps} time slices of {slice_s:.3f} s on one host "
                                   f"thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def make_workload(args):
    if args.batch is None:
        return wl.CONFIGS[args.config]()
    scaled = {"llama13b_mha_bf16": lambda B: wl.llama13b_mha_bf16(B=B),
              "gqa_chat_bf16": lambda B: wl.gqa_chat_bf16(B=B),
              "long_fp8_bs16": lambda B: wl.long_fp8(16, B=B),
              "long_fp8_bs32": lambda B: wl.long_fp8(32, B=B),
              "shared_prefix_bf16": lambda B: wl.shared_prefix_bf16(groups=max(1, B // 4)),
              "shared_prefix_fork_bf16": lambda B: wl.shared_prefix_bf16(True, groups=max(1, B // 4)),
              "beam_search_bf16": lambda B: wl.beam_search_bf16(requests=max(1, B // 4))}
    if args.config not in scaled:
        raise SystemExit(f"--batch is not supported for {args.config}")
    return scaled[args.config](args.batch)


def beam_stats(w, steps=50, seed=0):
    """Beam workloads: blocks held with sharing vs one copy per beam after the
    measured step, and the host half of further real beam steps on the library's
    block manager (every request's beams reshuffled by seeded random parents,
    one append per beam, dense tables, prefix groups), in us per step."""
    import paged_kv_cache_259_gb300 as pkv
    bm = pkv.BlockManager(w.NB, w.bs, w.free_order)
    for op in w.script:
        if op[0] == "add":
            bm.add_seq(op[1])
        elif op[0] == "append":
            bm.append_n(op[1], op[2])
        elif op[0] == "beam":
            bm.beam_step(op[1], op[2], op[3])
        else:
            raise ValueError(f"unexpected op {op[0]}")
    bm.append_slots(w.step_seqs)
    held = w.NB - bm.num_free()
    unshared = int(sum(-(-int(L) // w.bs) for L in w.final_lens))
    W = w.notes["width"]
    beams = [list(w.step_seqs[i:i + W]) for i in range(0, w.B, W)]
    nxt = max(w.step_seqs) + 1
    rng = np.random.default_rng(seed)
    parents = rng.integers(0, W, size=(steps, len(beams), W))
    MB = w.max_blocks_per_seq + -(-steps // w.bs) + 1
    max_members = max(1, 8 // (w.Hq // w.Hkv))
    t0 = time.perf_counter()
    for k in range(steps):
        old = [s for b in beams for s in b]
        par = (parents[k] + W * np.arange(len(beams))[:, None]).reshape(-1)
        ids = list(range(nxt, nxt + len(old)))
        nxt += len(old)
        bm.beam_step(old, par, ids)
        beams = [ids[i:i + W] for i in range(0, len(ids), W)]
        bm.append_slots(ids)
        bm.build_tables(ids, MB)
        bm.prefix_groups(ids, max_members)
    us = (time.perf_counter() - t0) * 1e6 / steps
    return {"requests": w.notes["requests"], "width": W, "generated": w.notes["generated"],
            "blocks_held": held, "blocks_unshared": unshared,
            "memory_saving": round(1 - held / unshared, 4),
            "host_beam_step_us": round(us, 1)}


def kv_utilisation(w, plan):
    """Tokens held over slots allocated: per sequence (its own table, the waste of
    its last block) and over the distinct physical blocks of the batch (shared
    prefix blocks counted once, so sharing shows as a value above 1)."""
    lens = np.asarray(plan.lens, dtype=np.int64)
    nblk = -(-lens // w.bs)
    t = np.asarray(plan.tables)
    used = np.unique(np.concatenate([t[i, :nblk[i]] for i in range(len(lens))]))
    return {"per_sequence": round(float(lens.sum() / (nblk.sum() * w.bs)), 4),
            "physical": round(float(lens.sum() / (used.size * w.bs)), 4)}


def workload_desc(w):
    L = np.asarray(w.final_lens)
    return (f"{w.name}: B={w.B}, Hq={w.Hq}, Hkv={w.Hkv}, D={w.D}, block_size={w.bs}, "
            f"NB={w.NB}, kv={w.kv_dtype}, L in [{L.min()}, {L.max()}] mean {L.mean():.1f}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default=DEFAULT_CONFIG,
                    choices=sorted(wl.CONFIGS) + sorted(wl.PREFILL_CONFIGS) +
                    sorted(wl.PROMPT_CONFIGS) + sorted(wl.SWAP_CONFIGS))
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's sequence count (profiling small cases)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle timing")
    ap.add_argument("--no-others", dest="others", action="store_false",
                    help="default workload only: skip timing the other decode workloads")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        if args.config in wl.PREFILL_CONFIGS or args.config in wl.PROMPT_CONFIGS:
            run_reference_prefill(args)
        elif args.config in wl.SWAP_CONFIGS:
            run_reference_swap(args)
        else:
            run_reference(args)
        return

    import paged_kv_cache_259_gb300 as pkv
    pkv.load_library()                       # fails loudly if the library is not built
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)

    modes = {**{c: prefill_main for c in wl.PREFILL_CONFIGS},
             **{c: prefill_main for c in wl.PROMPT_CONFIGS},
             **{c: swap_main for c in wl.SWAP_CONFIGS}}
    if args.config in modes:
        modes[args.config](args, rank, world, device)
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return

    r = run_gpu(args, rank, world, device)
    w, nb = r["w"], r["nbytes"]
    ms = max_over_ranks(r["ms_per_step"], world, device)
    dec_ms = max_over_ranks(r["dec_ms"], world, device)
    e2e = r["e2e"]
    e2e_ms = max_over_ranks(e2e["ms"], world, device)
    peak, peak_kind = load_peaks()
    value = world * nb["total"] / (ms * 1e-3) / 1e9
    dec_gbs = nb["decode"] / (dec_ms * 1e-3) / 1e9
    others = {}
    if world == 1 and args.others and args.config == DEFAULT_CONFIG and args.batch is None:
        n_other = max(20, min(args.steps, 200))
        for name in OTHER_DECODE:
            others[name] = run_other(name, n_other, args.warmup, device, peak)

    line = None
    if rank == 0:
        cpu_line, check = None, None
        if args.cpu_budget > 0:                       # <= 0: profiling runs skip the CPU leg
            q, k_src, v_src, ks, vs, plan = r["cpu"]
            kp, vp, tables, lens = oracle_inputs_for_step(w, q, k_src, v_src, plan)
            gbs, units, cores, note, ref_rows = oracle_timing(
                w, (q, kp, vp, ks, vs), tables, lens, nb["per_token"], args.cpu_budget, 1,
                check_units=check_units_decode(w, 48))
            cpu_line = {
                "value": round(float(gbs[0]), 4), "unit": "GB/s", "cores": cores,
                "kind": "oracle",
                "sample": f"{int(units[0])} random (sequence, head) units of this workload in "
                          f"{args.cpu_budget:.1f} s on {cores} host cores (one single-threaded "
                          f"float64 oracle process per core){note}"}
            check = {**self_check(r["out"], ref_rows, w.kv_dtype),
                     "of": "the timed steps' output rows against the oracle rows of the "
                           "cpu_baseline run (its first units)"}
        plan = r["cpu"][5]
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.kv_dtype, "data": "synthetic",
            "config": {
                "workload": workload_desc(w),
                "step": ("paged_decode_step: copy_blocks (CoW pairs: %d) + reshape_and_cache + "
                         "%s; %d kernel launches per step" % (
                             len(plan.pairs),
                             "paged_attention_decode_grouped (%d prefix groups)" % r["groups"]
                             if r["groups"] else "paged_attention_decode",
                             r["launches_per_step"])),
                "l2": "inputs larger than L2: %.2f GB of K/V read per step vs %d MB L2"
                      % (nb["decode"] / 1e9, L2_BYTES >> 20),
                "bytes_per_step": nb["total"], "decode_bytes_per_step": nb["decode"],
                "decode_logical_bytes_per_step": nb["decode_logical"],
                "seq_steps_per_s": round(world * w.B / (ms * 1e-3), 1),
                "kv_utilisation": kv_utilisation(w, plan),
                **({"beam": beam_stats(w)} if "width" in w.notes else {}),
                "step_frac_of_peak": round(value / world / peak, 4),
            },
            "roofline": {
                "kernel": "paged_attention_decode (decode kernel + split merge)",
                "bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peak, "unit": "GB/s",
                "frac": round(dec_gbs / peak, 4), "traffic": measured_traffic(args.config),
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                "bytes_per_launch": nb["decode"], "ms_per_launch": round(dec_ms, 5),
                "ms_per_launch_median": round(r["dec_ms_median"], 5),
            },
            "cpu_baseline": cpu_line,
            "e2e": {
                "value": round(world * e2e["bytes"] / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_ms, 5), "steps": e2e["steps"],
                "host_plan_us_per_step": round(e2e["host_plan_us"], 1),
                "note": ("public API with host planning (engine.LiveDecodePipeline): every "
                         "step the native block manager appends a token to every sequence, "
                         "builds the tables and finds the prefix groups straight into a "
                         "pinned slab; the slab (plan, q, k, v) is uploaded, the step runs "
                         "and its output is read back, overlapped with the neighbouring "
                         "steps, all of it one library call per step "
                         "(pkv_decode_pipeline_step); sequences grow by one token per step (bytes counted at each "
                         "step's lengths), the manager rewound every %d steps outside the "
                         "timed passes" % e2e["per_pass"])},
            "check": check,
            **({"others": others} if others else {}),
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on this workload's config."""
    w = make_workload(args)
    k_src, v_src = w.past_pools()
    q, k_new, v_new = w.step_inputs()
    ks = vs = 1.0
    if w.kv_dtype == "e4m3":
        ks, vs = w.fp8_scales(k_src, v_src, k_new, v_new)
    kp, vp, tables, lens = oracle_inputs_for_step(w, q, k_src, v_src, None)
    per_tok = 2 * w.Hkv * w.D * KV_ELT[w.kv_dtype]
    slice_s = 120.0 / (args.steps + args.warmup)       # whole run within ~2 minutes
    gbs, units, cores, note, _ = oracle_timing(w, (q, kp, vp, ks, vs), tables, lens, per_tok,
                                               slice_s, args.warmup + args.steps)
    value = float(gbs[args.warmup:].mean())
    units_done = int(units[args.warmup:].sum())
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * slice_s, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype, "data": "synthetic",
        "config": {"workload": workload_desc(w)},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{units_done} random (sequence, head) units finished in "
                                   f"{args.steps} time slices of {slice_s:.3f} s (after "
                                   f"{args.warmup} warm-up slices) on {cores} host cores (one "
                                   f"single-threaded float64 oracle process per core){note}"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
