"""Whole outputs against the oracle at the benchmark's sizes (GPU).

The other full-size tests compare sampled rows; here every output row of a
mid-size E4M3 decode workload (4 sequences of the 32,768-token E4M3 batch, in
its launch configuration: all 128 (sequence, head) rows) and of a mid-size
chunked-prefill workload (4 sequences of the GQA prefill batch: 2,048 chunk
tokens x 32 heads = 65,536 rows over up to 4,096 keys) is compared element by
element with the float64 oracle. The oracle rows
come from the benchmark's multi-process oracle runner (one spawned
single-threaded process per host core, pools shared read-only through
memory-mapped files), so the whole outputs take seconds, not minutes.

Tolerance as in the parity tests: |gpu - oracle| <= 6e-2 + 6e-2 |oracle| with
the E4M3 cache, 2e-2 + 2e-2 |oracle| with bf16.
"""
import numpy as np
import pytest
import torch

import bench
import pkv_workloads as wl
from _lib import library, pkv
from _parity import Inputs, assert_close, check_indexing, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_and_library():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    library()
    torch.cuda.set_device(0)


def test_long_fp8_bs16_mid_size_every_row():
    w = wl.long_fp8(16, B=4)
    inp = Inputs(w)
    g = run_gpu(inp, workspace=True)
    assert g["err"] == 0
    o = run_oracle(inp, units=[])                 # the oracle's state: slots, tables, pools
    check_indexing(g, o)
    units = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    per_tok = 2 * w.Hkv * w.D
    _, _, cores, note, rows = bench.oracle_timing(
        w, (inp.q, o["k_pool"], o["v_pool"], inp.ks, inp.vs), o["tables"], o["lens"], per_tok,
        0.0, 1, check_units=units)
    assert sorted(rows) == units, note
    got = g["out"].numpy()
    ref = np.stack([rows[u] for u in units]).reshape(got.shape)
    assert_close(got, ref, "e4m3", f"long_fp8_bs16 B=4, every row ({cores} oracle processes)")


def test_prefill_gqa_mid_size_every_row():
    import test_gpu_prefill as tp
    w = wl.prefill_gqa_bf16(B=4)
    c = tp.Case(w)
    g = tp.run_gpu(c)
    assert g["err"] == 0
    o = tp.run_oracle(c, units=[])
    tp.check_indexing_and_writes(g, o)
    G = w.Hq // w.Hkv
    seq_of = np.repeat(np.arange(w.B), w.chunks)
    # sorted by (sequence, KV head) so each oracle process keeps its gathered K/V
    units = sorted(((t, h) for t in range(w.T) for h in range(w.Hq)),
                   key=lambda th: (seq_of[th[0]], th[1] // G, th[0], th[1]))
    _, _, cores, note, rows = bench.oracle_timing(
        w, (c.q, o["k_pool"], o["v_pool"], 1.0, 1.0), o["tables"], o["lens"], 0, 0.0, 1,
        extra={"mode": "prefill", "query_start": w.query_start}, check_units=units)
    assert len(rows) == len(units), note
    got = g["out"].numpy()
    ref = np.stack([rows[(t, h)] for t in range(w.T) for h in range(w.Hq)]).reshape(got.shape)
    assert_close(got, ref, "bf16", f"prefill_gqa_bf16 B=4, every row ({cores} oracle processes)")
