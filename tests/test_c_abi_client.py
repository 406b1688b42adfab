"""The C ABI from plain C: tests/c_abi/host_block_manager.c, compiled with the
system C compiler against include/pagedkv.h and linked to the built library,
drives the host block manager (appends, fork, copy-on-write, a beam step, a
batch step, a refused chunk, frees), then a second manager with prefix caching
and a host pool (a served prompt, a request reusing its blocks, cache
statistics, a swap out and back in), with no Python or torch in between. Its
output must equal the oracle's managers on the same operations."""
import os
import shutil
import subprocess

import pytest

from _lib import library
from oracle.block_manager import BlockManager as OracleBM
from oracle.prefix_cache import PrefixCachingBlockManager

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def expected():
    bm = OracleBM(12, 4, [5, 2, 7, 0, 3, 6, 1, 4, 11, 9, 10, 8])
    out = []
    bm.add_seq(0)
    for _ in range(6):
        slot, cow = bm.append_slot(0)
        s, d = cow if cow else (-1, -1)
        out.append(f"slot 0 {slot} cow {s} {d}")
    bm.fork(0, 1)
    for sid in (1, 0):
        slot, cow = bm.append_slot(sid)
        s, d = cow if cow else (-1, -1)
        out.append(f"slot {sid} {slot} cow {s} {d}")
    for sid in (0, 1):
        out.append(" ".join(["table", str(sid)] + [str(b) for b in bm.block_table(sid)]))
    bm.beam_step([0, 1], [1, 1], [2, 3])
    for sid in (2, 3):
        out.append(" ".join(["table", str(sid)] + [str(b) for b in bm.block_table(sid)]))
    out.append(" ".join(["free"] + [str(b) for b in bm.free]))
    line = ["step"]
    cows = []
    for sid in (2, 3):
        slot, cow = bm.append_slot(sid)
        line.append(str(slot))
        if cow:
            cows += ["cow", str(cow[0]), str(cow[1])]
    out.append(" ".join(line + cows))
    nf, n2 = len(bm.free), bm.seq_len(2)
    out.append(f"refused -5 cow 0 len {n2} {n2} free {nf} {nf}")
    out.append("unknown -4")
    pc = PrefixCachingBlockManager(8, 4, list(range(8)), num_cpu_blocks=4)
    prompt = [5, 6, 7, 8, 9, 10, 11, 12, 13]
    n = pc.add_seq_prompt(0, prompt)
    slots = [pc.append_token(0, t)[0] for t in prompt[n:]]
    out.append(" ".join(["prompt", "0", "cached", str(n)] + [str(x) for x in slots]))
    out.append(f"prompt 1 cached {pc.add_seq_prompt(1, prompt)}")
    out.append(f"stats {pc.hit_blocks} {pc.lookup_blocks} {pc.num_cached()} {pc.num_evictable()}")
    out.append(" ".join(["out"] + [str(x) for p in pc.swap_out(0) for x in p]))
    out.append(" ".join(["in"] + [str(x) for p in pc.swap_in(0) for x in p]))
    return out


def test_plain_c_client_matches_the_oracle(tmp_path):
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = library()
    libdir = os.path.dirname(lib._name)
    exe = str(tmp_path / "host_block_manager")
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "host_block_manager.c"),
                    "-L", libdir, "-lpagedkv", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    got = subprocess.run([exe], capture_output=True, text=True, timeout=60, check=True).stdout
    assert got.strip().splitlines() == expected()
