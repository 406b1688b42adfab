"""The allocation-free decode entry point, checked against the regular one (GPU).

paged_attention_decode_noalloc serves callers that cannot allocate device memory
where they decode -- a plug-in inside a runtime that owns all device memory, or
a serving loop whose memory plan is fixed at start-up -- by using a fixed
scratch array inside the library instead of a caller-provided workspace. It must
give the regular entry point's result. Both are called through the C ABI.

The file name makes pytest collect it last, so a failure here comes after every
other test has run.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from _lib import library

pytestmark = pytest.mark.gpu

PKV_BF16 = 1
ATOL = RTOL = 2e-2          # the bf16 tolerance of the parity tests


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _regular(lib, out, q, kp, vp, bt, lens, scale, ws):
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = kp.shape
    return lib.paged_attention_decode(
        _ptr(out), _ptr(q), _ptr(kp), _ptr(vp), _ptr(bt), _ptr(lens), B, bt.shape[1], NB, Hq,
        Hkv, D, bs, scale, PKV_BF16, PKV_BF16, 1.0, 1.0, _ptr(ws), ws.numel(), _stream())


def _noalloc(lib, out, q, kp, vp, bt, lens, scale):
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = kp.shape
    return lib.paged_attention_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(kp), _ptr(vp), _ptr(bt), _ptr(lens), B, bt.shape[1], NB, Hq,
        Hkv, D, bs, scale, PKV_BF16, PKV_BF16, 1.0, 1.0, _stream())


def test_noalloc_matches_regular_entry_point_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    lib = library()
    torch.cuda.set_device(0)
    g = torch.Generator().manual_seed(21)
    B, Hq, Hkv, D, bs = 8, 16, 4, 128, 16
    lens_list = [1, 17, 300, 1024, 2047, 3000, 5, 999]
    MB = max(-(-L // bs) for L in lens_list)
    NB = sum(-(-L // bs) for L in lens_list) + 7
    kp = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16).cuda()
    vp = torch.randn(NB, Hkv, bs, D, generator=g).to(torch.bfloat16).cuda()
    perm = torch.randperm(NB, generator=g)
    bt = torch.full((B, MB), -1, dtype=torch.int32)
    pos = 0
    for b, L in enumerate(lens_list):
        n = -(-L // bs)
        bt[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    bt = bt.cuda()
    lens = torch.tensor(lens_list, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    ws_bytes = lib.paged_attention_workspace_size(B, Hq, D, bs, MB)
    assert ws_bytes > 0                       # this batch is split across partitions
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for call in range(2):                     # the second call meets the first call's leftovers
        q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16).cuda()
        ref = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        assert _regular(lib, ref, q, kp, vp, bt, lens, scale, ws) == 0
        assert _noalloc(lib, got, q, kp, vp, bt, lens, scale) == 0
        torch.cuda.synchronize()
        code = ctypes.c_int(-1)
        assert lib.pkv_get_device_error(ctypes.byref(code), None) == 0 and code.value == 0
        r = ref.float().cpu().numpy()
        o = got.float().cpu().numpy()
        assert np.all(np.isfinite(o)), f"call {call}: non-finite output"
        err = np.abs(o - r)
        assert np.all(err <= ATOL + RTOL * np.abs(r)), f"call {call}: max abs err {err.max()}"


def test_noalloc_refuses_a_batch_beyond_its_scratch():
    lib = library()
    # 65535 sequences x 64 heads x 2 partitions x 130 floats is far above 32 MiB:
    # refused on the host before any pointer is used or anything is launched
    st = lib.paged_attention_decode_noalloc(None, None, None, None, None, None, 65535, 8, 64, 64,
                                            8, 128, 16, 0.1, PKV_BF16, PKV_BF16, 1.0, 1.0, None)
    assert st == -1
