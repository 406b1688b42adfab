"""The C-ABI library loads without a GPU and exports every function pagedkv.h declares."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import paged_kv_cache_259_gb300 as pkv
from _lib import ROOT, library

HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = re.sub(r"#[^\n]*", " ", text)
    names = set()
    for stmt in text.split(";"):
        stmt = " ".join(stmt.split())
        if "typedef" in stmt or "(" not in stmt:
            continue
        m = re.match(r"^(?:extern \"C\" \{ )?[\w\s\*]*?\b(\w+)\s*\(", stmt)
        if m:
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("paged_attention_decode", "reshape_and_cache", "copy_blocks",
              "paged_attention_workspace_size", "pkv_get_device_error", "bm_create",
              "bm_append_slot", "bm_fork", "bm_free_seq"):
        assert n in names, n


def test_library_exports_every_declared_symbol():
    lib = library()
    raw = ctypes.CDLL(lib._name)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_status_strings_and_host_side_argument_checks():
    lib = library()
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(-5) == b"block pool exhausted"
    # argument errors are caught on the host before any CUDA call
    assert lib.paged_attention_decode(None, None, None, None, None, None, 4, 8, 64, 3, 2, 64,
                                      16, 0.1, 0, 0, 1.0, 1.0, None, 0, None) == -1  # Hq % Hkv
    assert lib.paged_attention_decode(None, None, None, None, None, None, 0, 8, 64, 4, 4, 64,
                                      16, 0.1, 0, 0, 1.0, 1.0, None, 0, None) == 0   # empty batch
    assert lib.paged_attention_decode(None, None, None, None, None, None, 4, 8, 64, 4, 4, 64,
                                      16, 0.1, 1, 1, 2.0, 1.0, None, 0, None) == -1  # k_scale w/o fp8
    assert lib.reshape_and_cache(None, None, None, None, None, 0, 4, 64, 16, 8, 0, 0, 1.0, 1.0,
                                 None) == 0
    assert lib.reshape_and_cache(None, None, None, None, None, 3, 4, 72, 16, 8, 0, 0, 1.0, 1.0,
                                 None) == -2                                          # head_dim % 16
    assert lib.copy_blocks(None, None, None, 0, 8, 4096, None) == 0
    assert lib.copy_blocks(None, None, None, 1, 8, 4100, None) == -1                  # bytes % 16
    assert lib.paged_attention_workspace_size(64, 40, 128, 16, 128) == 64 * 40 * 16 * 130 * 4
    assert lib.paged_attention_workspace_size(4, 4, 64, 16, 8) == 0                  # never split


@pytest.mark.parametrize("dtype,bs,D", [(torch.bfloat16, 16, 128), (torch.bfloat16, 32, 64),
                                         (torch.float32, 16, 64), (torch.uint8, 32, 128)])
def test_pool_layout_helpers_follow_the_header_formula(dtype, bs, D):
    """pools_from_views / pool_views against the element offsets the header states:
    K (blk, h, t, d) at (blk*Hkv + h)*bs*D + ((t/8)*(D/X) + d/X)*8X + (t%8)*X + d%X,
    V (blk, h, t, d) at (blk*Hkv + h)*bs*D + ((t/X)*(D/8) + d/8)*8X + (d%8)*X + t%X."""
    NB, Hkv = 3, 2
    X = 16 // torch.empty((), dtype=dtype).element_size()
    n = NB * Hkv * bs * D
    ids = torch.arange(n, dtype=torch.int64)
    k = (ids % 251).to(dtype).reshape(NB, Hkv, bs, D) if dtype == torch.uint8 else \
        ids.to(torch.float32).to(dtype).reshape(NB, Hkv, bs, D)
    v = (k.to(torch.float32) + 1).to(dtype) if dtype != torch.uint8 else (k + 1)
    kp, vp = pkv.pools_from_views(k, v)
    ks, vs = pkv.pool_shapes(NB, Hkv, bs, D, dtype)
    assert tuple(kp.shape) == ks and tuple(vp.shape) == vs
    kf, vf = kp.reshape(-1), vp.reshape(-1)
    rng = np.random.default_rng(0)
    for _ in range(300):
        blk, h, t, d = (int(rng.integers(NB)), int(rng.integers(Hkv)), int(rng.integers(bs)),
                        int(rng.integers(D)))
        base = (blk * Hkv + h) * bs * D
        ko = base + ((t // 8) * (D // X) + d // X) * 8 * X + (t % 8) * X + d % X
        vo = base + ((t // X) * (D // 8) + d // 8) * 8 * X + (d % 8) * X + t % X
        assert kf[ko] == k[blk, h, t, d] and vf[vo] == v[blk, h, t, d]
    k2, v2 = pkv.pool_views(kp, vp)
    assert torch.equal(k2, k) and torch.equal(v2, v)


def test_copy_waves_run_concurrently_give_the_in_order_result():
    """Host logic of PagedKVCache.apply_copies: pairs cut into waves, each wave
    applied at once (every destination gets its source as the wave began), must
    give what applying the pairs one by one gives."""
    import numpy as np
    from paged_kv_cache_259_gb300.engine import copy_waves
    rng = np.random.default_rng(0)
    for trial in range(200):
        nb = int(rng.integers(2, 12))
        pairs = [tuple(rng.choice(nb, 2, replace=False).tolist())
                 for _ in range(int(rng.integers(0, 20)))]
        seq = list(range(nb))
        for s, d in pairs:
            seq[d] = seq[s]
        par = list(range(nb))
        waves = copy_waves(pairs)
        assert [i for a, b in waves for i in range(a, b)] == list(range(len(pairs)))
        for a, b in waves:
            w = pairs[a:b]
            dsts = [d for _, d in w]
            assert len(set(dsts)) == len(dsts) and not set(dsts) & {s for s, _ in w}
            snap = list(par)
            for s, d in w:
                par[d] = snap[s]
        assert par == seq
    assert copy_waves([(0, 5), (1, 6), (2, 7)]) == [(0, 3)]
    assert copy_waves([(0, 5), (5, 6)]) == [(0, 1), (1, 2)]


def test_step_pipeline_slab_layout_packs_every_input_once_aligned():
    """Host logic of engine.StepPipeline: a step's inputs share one slab; each
    view starts on a 256-byte boundary, keeps its dtype and shape, and no two
    views overlap (empty tensors included); values round-trip."""
    import torch
    from paged_kv_cache_259_gb300.engine import slab_layout, slab_views
    t = {"q": torch.randn(3, 5, 8).to(torch.bfloat16), "slots": torch.arange(3, dtype=torch.int64),
         "pairs": torch.zeros((0, 2), dtype=torch.int64),
         "tables": torch.arange(21, dtype=torch.int32).view(3, 7), "lens": torch.ones(3, dtype=torch.int32),
         "max_group_blocks": 9}
    layout, nbytes = slab_layout(t)
    assert set(layout) == {"q", "slots", "pairs", "tables", "lens"}
    spans = []
    for k, (off, dtype, shape) in layout.items():
        assert off % 256 == 0 and dtype == t[k].dtype and shape == tuple(t[k].shape)
        spans.append((off, off + t[k].numel() * t[k].element_size()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:])) and spans[-1][1] <= nbytes
    slab = torch.zeros(nbytes, dtype=torch.uint8)
    views = slab_views(slab, layout)
    for k, v in views.items():
        v.copy_(t[k])
    again = slab_views(slab, layout)
    for k in layout:
        assert torch.equal(again[k], t[k])


def test_host_runs_cover_the_ids_in_order():
    import numpy as np
    from paged_kv_cache_259_gb300.engine import host_runs
    assert host_runs([]) == []
    assert host_runs([5]) == [(0, 1, 5)]
    assert host_runs([3, 4, 5, 9, 10, 2]) == [(0, 3, 3), (3, 5, 9), (5, 6, 2)]
    rng = np.random.default_rng(1)
    for _ in range(50):
        ids = rng.permutation(40)[:int(rng.integers(0, 40))]
        rebuilt = [h + i for a, b, h in host_runs(ids) for i in range(b - a)]
        assert rebuilt == list(ids)


def test_noalloc_refuses_a_splittable_batch_beyond_its_scratch():
    """65535 sequences x 64 heads x 2 partitions x 130 floats is far above the
    fixed 32 MiB scratch: with 9 blocks per sequence (the batch may be split)
    the call is refused on the host before any pointer is used or anything is
    launched; the GPU is never touched."""
    lib = library()
    st = lib.paged_attention_decode_noalloc(None, None, None, None, None, None, 65535, 9, 64, 64,
                                            8, 128, 16, 0.1, 1, 1, 1.0, 1.0, None)
    assert st == -1
    assert lib.paged_attention_workspace_size(65535, 64, 128, 16, 9) > 0



def test_stage_calls_refuse_missing_buffers_before_any_cuda_call():
    """pkv_stage_upload / pkv_stage_download check their arguments on the host:
    a null buffer or event, or zero bytes, is PKV_ERR_INVALID_ARG and nothing
    reaches the CUDA runtime (so this runs without a GPU)."""
    lib = library()
    vp = ctypes.c_void_p
    some = vp(0x1000)
    assert lib.pkv_stage_upload(None, some, 64, None, None, some, None, None) == -1
    assert lib.pkv_stage_upload(some, None, 64, None, None, some, None, None) == -1
    assert lib.pkv_stage_upload(some, some, 0, None, None, some, None, None) == -1
    assert lib.pkv_stage_upload(some, some, 64, None, None, None, None, None) == -1
    assert lib.pkv_stage_download(None, some, 64, None, None, some, some) == -1
    assert lib.pkv_stage_download(some, some, 64, None, None, None, some) == -1
    assert lib.pkv_stage_download(some, some, 64, None, None, some, None) == -1
    assert lib.pkv_stage_download(some, some, 0, None, None, some, some) == -1


def test_decode_step_refuses_bad_arguments_before_any_launch():
    """paged_decode_step checks every argument on the host before it launches
    anything (so these run without a GPU): negative counts, group arrays
    missing, an ungrouped list longer than the batch, decode arguments the
    plain decode refuses (query heads not a multiple of the kv heads), a missing
    slot mapping; an empty step is a no-op."""
    lib = library()
    vp = ctypes.c_void_p
    some = vp(0x1000)

    def step(pairs=None, num_pairs=0, k=some, v=some, slots=some, B=4, Hq=4, Hkv=4,
             groups=(None, None, None, 0, 0), ungrouped=(None, -1)):
        sg, gm, gp, ng, mm = groups
        return lib.paged_decode_step(pairs, num_pairs, k, v, slots, some, some, some, some, some,
                                     some, B, 8, 64, Hq, Hkv, 64, 16, 0.1, 1, 1, 1.0, 1.0,
                                     sg, gm, gp, ng, mm, 0, ungrouped[0], ungrouped[1], None, 0,
                                     None)

    assert step(num_pairs=-1) == -1
    assert step(groups=(None, None, None, 1, 4)) == -1          # groups without arrays
    assert step(ungrouped=(some, 5)) == -1                      # longer than the batch
    assert step(Hq=6) == -1                                     # Hq % Hkv
    assert step(slots=None) == -1                               # no slot mapping
    assert step(num_pairs=2, pairs=None) == -1                  # pairs missing
    assert step(B=0) == 0                                       # nothing to do


def test_prefill_step_refuses_bad_arguments_before_any_launch():
    """paged_prefill_step checks every argument on the host before it launches
    anything (so these run without a GPU)."""
    lib = library()
    vp = ctypes.c_void_p
    some = vp(0x1000)

    def step(num_pairs=0, pairs=None, T=8, slots=some, Hq=8, Hkv=8, D=128, bs=16):
        return lib.paged_prefill_step(pairs, num_pairs, some, some, slots, T, some, some, some,
                                      some, some, some, some, 2, 8, 8, 64, Hq, Hkv, D, bs, 0.1, 1,
                                      1, None)

    assert step(num_pairs=-1) == -1
    assert step(Hq=12) == -1                                    # Hq % Hkv
    assert step(D=64) == -2                                     # head_dim 128 only
    assert step(slots=None) == -1                               # no slot mapping
    assert step(num_pairs=1) == -1                              # pairs missing


def test_decode_pipeline_step_args_match_the_header_layout(tmp_path):
    """The binding's ctypes mirror of pkv_decode_pipeline_step_args has the C
    struct's size and every field at the C offset (a C program built from the
    header prints them)."""
    import shutil
    import subprocess
    import paged_kv_cache_259_gb300 as pkv
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    S = pkv.DecodePipelineStepArgs
    names = [f[0] for f in S._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include <stdint.h>\n"
                   '#include "pagedkv.h"\nint main(void) {\n'
                   '    printf("%zu\\n", sizeof(pkv_decode_pipeline_step_args));\n' +
                   "".join(f'    printf("%zu\\n", offsetof(pkv_decode_pipeline_step_args, {n}));\n'
                           for n in names) + "    return 0;\n}\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run([cc, "-I", inc, "-o", str(exe), str(src)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(S)
    assert got[1:] == [getattr(S, n).offset for n in names]


def test_decode_pipeline_step_refuses_before_any_cuda_call():
    """pkv_decode_pipeline_step: a null argument block or output buffer is
    PKV_ERR_INVALID_ARG, and a step the block manager refuses (an unknown
    sequence id) returns its status from the planning, before anything is
    enqueued (so this runs without a GPU), leaving the manager unchanged."""
    import paged_kv_cache_259_gb300 as pkv
    lib = library()
    S = pkv.DecodePipelineStepArgs
    some = ctypes.c_void_p(0x1000)
    assert lib.pkv_decode_pipeline_step(None, 0, some, None, None) == -1
    bm = pkv.BlockManager(8, 16, np.arange(8))
    bm.add_seq(0)
    ids = np.array([7], dtype=np.int64)                   # never added
    slots = np.zeros(1, dtype=np.int64)
    pairs = np.zeros(2, dtype=np.int64)
    tables = np.zeros(4, dtype=np.int32)
    lens = np.zeros(1, dtype=np.int32)
    a = S()
    a.bm = bm._h
    a.seq_ids = ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    a.num_seqs, a.max_blocks, a.max_members = 1, 4, 0
    a.h_slots = slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    a.h_pairs = pairs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    a.h_tables = tables.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    a.h_lens = lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    assert lib.pkv_decode_pipeline_step(ctypes.byref(a), 0, None, None, None) == -1
    counts, us = (ctypes.c_int * 4)(), ctypes.c_double(-1.0)
    assert lib.pkv_decode_pipeline_step(ctypes.byref(a), 0, some, counts,
                                        ctypes.byref(us)) == -4
    assert us.value >= 0.0 and list(counts) == [0, 0, 0, 0]
    assert bm.seq_len(0) == 0 and bm.num_free() == 8

