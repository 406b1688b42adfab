"""The oracle's pins catch plausible mistakes in it.

Each case plants one mistake in a copy of the oracle and runs
tests/test_oracle_pins.py against that copy. Nothing is written to the
repository's own oracle: the copy and the pins live in a temporary directory.
Each run must fail the pins. The mistakes cover head mapping, scales,
softmax normalisation, causal positions, block and slot indexing, E4M3
rounding, sign, NaN, bias, subnormals and scaling, and copy and swap
direction. They also cover copy-on-write, fork counts, free-list order, beam
parents and their order against the frees, swap pairs and capacity, and
prefix-cache keys, registration, revival, counters and eviction order. A
control run of the unchanged copy
must pass, so a broken set-up cannot pass for a caught mistake.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (what, file, original text, planted text)
MUTANTS = [
    ("decode GQA head mapping", "oracle/attention.py",
     "        hk = h // G\n        K = widen_k", "        hk = h % Hkv\n        K = widen_k"),
    ("prefill GQA head mapping", "oracle/attention.py",
     "        p = L - C + (t - int(qs[b]))\n        hk = h // G",
     "        p = L - C + (t - int(qs[b]))\n        hk = h % Hkv"),
    ("softmax scale dropped", "oracle/attention.py",
     "s = scale * k_scale * (K @ q_vec)", "s = k_scale * (K @ q_vec)"),
    ("v_scale dropped", "oracle/attention.py", "return v_scale * (p @ V)", "return (p @ V)"),
    ("causal mask off by one", "oracle/attention.py", "K[:p + 1], V[:p + 1]", "K[:p], V[:p]"),
    ("logical block read as physical", "oracle/attention.py",
     "blocks = np.asarray(block_table, dtype=np.int64)[t // block_size]",
     "blocks = (t // block_size)"),
    ("slot within the block off by one", "oracle/attention.py",
     "torch.from_numpy(t % block_size)]", "torch.from_numpy((t + 1) % block_size)]"),
    ("E4M3 ties to the odd code", "oracle/fp8_e4m3.py",
     "((d_hi == d_lo) & (hi % 2 == 0))", "((d_hi == d_lo) & (hi % 2 == 1))"),
    ("E4M3 exponent bias 8", "oracle/fp8_e4m3.py",
     "normal = np.ldexp(1.0 + m / 8.0, e - 7)", "normal = np.ldexp(1.0 + m / 8.0, e - 8)"),
    ("E4M3 subnormal step", "oracle/fp8_e4m3.py",
     "subnormal = np.ldexp(m / 8.0, -6)", "subnormal = np.ldexp(m / 8.0, -7)"),
    ("quantisation multiplies by the scale", "oracle/fp8_e4m3.py",
     "/ np.float32(scale)", "* np.float32(scale)"),
    ("copy_blocks copies K only", "oracle/cache_ops.py",
     "        k_pool[dst] = k_pool[src]\n        v_pool[dst] = v_pool[src]",
     "        k_pool[dst] = k_pool[src]"),
    ("reshape_and_cache writes K into V", "oracle/cache_ops.py",
     "            v_pool[block, :, offset, :] = v[i]", "            v_pool[block, :, offset, :] = k[i]"),
    ("swap_blocks copies the wrong way", "oracle/cache_ops.py",
     "        dst_k_pool[dst] = src_k_pool[src]\n        dst_v_pool[dst] = src_v_pool[src]",
     "        src_k_pool[src] = dst_k_pool[dst]\n        src_v_pool[src] = dst_v_pool[dst]"),
    ("copy-on-write of an unshared block", "oracle/block_manager.py",
     "            if self.ref[last] > 1:", "            if self.ref[last] >= 1:"),
    ("free list taken from the back", "oracle/block_manager.py",
     "        b = self.free.pop(0)", "        b = self.free.pop()"),
    ("freed blocks go to the front", "oracle/block_manager.py",
     "            if self.ref[b] == 0:\n                self.free.append(b)",
     "            if self.ref[b] == 0:\n                self.free.insert(0, b)"),
    ("copy-on-write keeps the source count", "oracle/block_manager.py",
     "                self.ref[last] -= 1\n", ""),
    ("every new beam forks the first parent", "oracle/block_manager.py",
     "            self.fork(old_ids[int(p)], sid)", "            self.fork(old_ids[0], sid)"),
    ("swap-out pairs reversed", "oracle/block_manager.py",
     "        pairs = list(zip(table, host))", "        pairs = list(zip(host, table))"),
    ("swap-in frees host blocks to the front", "oracle/block_manager.py",
     "        self.cpu_free.extend(host)", "        self.cpu_free[:0] = host"),
    ("prefix reuse leaves no prompt token", "oracle/prefix_cache.py",
     "for i in range(max(0, (len(prompt) - 1) // bs)):", "for i in range(len(prompt) // bs):"),
    ("prefix key is the block's own tokens", "oracle/prefix_cache.py",
     "            key = tuple(prompt[:bs * (i + 1)])",
     "            key = tuple(prompt[bs * i:bs * (i + 1)])"),
    ("evictable blocks in table order", "oracle/prefix_cache.py",
     "        self.evictable.extend(reversed(cached))", "        self.evictable.extend(cached)"),
    ("prefill position counted from the chunk start", "oracle/attention.py",
     "        p = L - C + (t - int(qs[b]))", "        p = (t - int(qs[b]))"),
    ("softmax normalised by its largest term", "oracle/attention.py",
     "    p = p / p.sum()", "    p = p / p.max()"),
    ("E4M3 sign lost", "oracle/fp8_e4m3.py",
     "    sign = np.signbit(x32).astype(np.int64) << 7",
     "    sign = np.zeros_like(x32, dtype=np.int64)"),
    ("E4M3 NaN for the whole top exponent", "oracle/fp8_e4m3.py",
     "np.where((e == 15) & (m == 7), np.nan, out)", "np.where((e == 15), np.nan, out)"),
    ("fork leaves the counts alone", "oracle/block_manager.py",
     "        for b in self.tables[child]:\n            self.ref[b] += 1\n", ""),
    ("swap-out accepts one block too many", "oracle/block_manager.py",
     "        if len(table) > len(self.cpu_free):", "        if len(table) > len(self.cpu_free) + 1:"),
    ("new block one token late", "oracle/block_manager.py",
     "        if n % self.block_size == 0:", "        if n % self.block_size == 1 or n == 0:"),
    ("revived block stays evictable", "oracle/prefix_cache.py",
     "                self.evictable.remove(b)", "                pass"),
    ("blocks of unknown tokens registered", "oracle/prefix_cache.py",
     "            if None not in key and key not in self.block_of:",
     "            if key not in self.block_of:"),
    ("a later registration wins", "oracle/prefix_cache.py",
     "            if None not in key and key not in self.block_of:", "            if None not in key:"),
    ("decode length one short", "oracle/attention.py",
     "        L = int(lens[b])\n        hk = h // G\n        K = widen_k",
     "        L = int(lens[b]) - 1\n        hk = h // G\n        K = widen_k"),
    ("chunk rows mapped to the next sequence", "oracle/attention.py",
     "        seq_of[qs[b]:qs[b + 1]] = b", "        seq_of[qs[b]:qs[b + 1]] = min(b + 1, B - 1)"),
    ("quantisation divides by the unrounded scale", "oracle/fp8_e4m3.py",
     "    q = np.asarray(x, dtype=np.float32) / np.float32(scale)",
     "    q = (np.asarray(x, dtype=np.float64) / float(scale)).astype(np.float32)"),
    ("swap-in pairs reversed", "oracle/block_manager.py",
     "        return list(zip(host, dev))", "        return list(zip(dev, host))"),
    ("old beams freed before the forks", "oracle/block_manager.py",
     "        for p, sid in zip(parents, new_ids):\n            self.fork(old_ids[int(p)], sid)\n"
     "        for sid in old_ids:\n            self.free_seq(sid)",
     "        keep = {s: (list(self.tables[s]), self.lens[s]) for s in old_ids}\n"
     "        for sid in old_ids:\n            self.free_seq(sid)\n"
     "        for p, sid in zip(parents, new_ids):\n"
     "            t, n = keep[old_ids[int(p)]]\n"
     "            self.tables[sid] = list(t)\n            self.lens[sid] = n\n"
     "            for b in t:\n                self.ref[b] += 1"),
    ("prefix lookups not counted", "oracle/prefix_cache.py", "            self.lookup_blocks += 1\n", ""),
    ("prefix hits not counted", "oracle/prefix_cache.py", "            self.hit_blocks += 1\n", ""),
    ("caching manager frees to the front", "oracle/prefix_cache.py",
     "                else:\n                    self.free.append(b)",
     "                else:\n                    self.free.insert(0, b)"),
]


def copy_tree(dst):
    """The oracle and the pins (with their fixtures) under ``dst``."""
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


def run_pins(root):
    env = dict(os.environ, OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")   # runs go side by side
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=root, capture_output=True, text=True,
                       timeout=900, env=env)
    return r.returncode, r.stdout[-2000:]


def plant(root, mutant):
    _, f, old, new = mutant
    path = os.path.join(root, f)
    with open(path) as fh:
        src = fh.read()
    assert src.count(old) == 1, f"{mutant[0]}: the original text is not in {f} exactly once"
    with open(path, "w") as fh:
        fh.write(src.replace(old, new))


def test_the_unchanged_copy_passes_the_pins(tmp_path):
    copy_tree(str(tmp_path))
    code, out = run_pins(str(tmp_path))
    assert code == 0, out


def test_every_planted_mistake_fails_the_pins(tmp_path):
    roots = []
    for i, m in enumerate(MUTANTS):
        root = str(tmp_path / f"m{i}")
        copy_tree(root)
        plant(root, m)
        roots.append(root)
    workers = max(1, min(8, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(run_pins, roots))
    # exit code 1: tests ran and failed (not a collection or usage error)
    missed = [(m[0], code) for m, (code, _) in zip(MUTANTS, results) if code != 1]
    assert not missed, f"mistakes the pins did not catch (pytest exit code): {missed}"
