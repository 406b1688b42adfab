"""The allocation-free decode entry point, checked against the regular one and
the oracle (GPU).

paged_attention_decode_noalloc serves callers that cannot allocate device memory
where they decode -- a plug-in inside a runtime that owns all device memory, or
a serving loop whose memory plan is fixed at start-up -- by using a fixed
scratch array inside the library instead of a caller-provided workspace. It must
give the regular entry point's result and the float64 oracle's (within the bf16
tolerance of the parity tests). Both entry points are called through the C ABI;
the binding's wrapper is called too.

The file name makes pytest collect it last, so a failure here comes after every
other test has run.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from _lib import library, pkv

from oracle import attention as oatt

pytestmark = pytest.mark.gpu

PKV_BF16 = 1
ATOL = RTOL = 2e-2          # the bf16 tolerance of the parity tests


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _regular(lib, out, q, kp, vp, bt, lens, scale, ws):
    B, Hq, D = q.shape
    NB, Hkv, bs = kp.shape[0], kp.shape[1], 8 * kp.shape[2]      # K [NB, Hkv, bs/8, D/X, 8, X]
    return lib.paged_attention_decode(
        _ptr(out), _ptr(q), _ptr(kp), _ptr(vp), _ptr(bt), _ptr(lens), B, bt.shape[1], NB, Hq,
        Hkv, D, bs, scale, PKV_BF16, PKV_BF16, 1.0, 1.0, _ptr(ws), ws.numel(), _stream())


def _noalloc(lib, out, q, kp, vp, bt, lens, scale):
    B, Hq, D = q.shape
    NB, Hkv, bs = kp.shape[0], kp.shape[1], 8 * kp.shape[2]
    return lib.paged_attention_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(kp), _ptr(vp), _ptr(bt), _ptr(lens), B, bt.shape[1], NB, Hq,
        Hkv, D, bs, scale, PKV_BF16, PKV_BF16, 1.0, 1.0, _stream())


SHAPES = [  # (B, Hq, Hkv, D, bs, lengths)
    (8, 16, 4, 128, 16, [1, 17, 300, 1024, 2047, 3000, 5, 999]),
    (5, 8, 8, 64, 32, [4000, 33, 1, 640, 2500]),
]


def _batch(g, B, Hq, Hkv, D, bs, lens_list):
    MB = max(-(-L // bs) for L in lens_list)
    NB = sum(-(-L // bs) for L in lens_list) + 7
    ks, vs = pkv.pool_shapes(NB, Hkv, bs, D, torch.bfloat16)
    kp = torch.randn(ks, generator=g).to(torch.bfloat16).cuda()
    vp = torch.randn(vs, generator=g).to(torch.bfloat16).cuda()
    perm = torch.randperm(NB, generator=g)
    bt = torch.full((B, MB), -1, dtype=torch.int32)
    pos = 0
    for b, L in enumerate(lens_list):
        n = -(-L // bs)
        bt[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    return kp, vp, bt.cuda(), torch.tensor(lens_list, dtype=torch.int32, device="cuda")


def _close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert np.all(err <= ATOL + RTOL * np.abs(ref)), f"{what}: max abs err {err.max()}"


@pytest.mark.parametrize("B,Hq,Hkv,D,bs,lens_list", SHAPES, ids=["gqa4_d128_bs16", "mha_d64_bs32"])
def test_noalloc_matches_regular_entry_point_on_two_calls_in_a_row(B, Hq, Hkv, D, bs, lens_list):
    """Two calls in a row through the C ABI (the second meets the first call's
    leftovers in the shared scratch) give the regular entry point's result; the
    first is also checked against the float64 oracle directly."""
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    lib = library()
    torch.cuda.set_device(0)
    g = torch.Generator().manual_seed(21 + D)
    kp, vp, bt, lens = _batch(g, B, Hq, Hkv, D, bs, lens_list)
    scale = 1.0 / math.sqrt(D)
    ws_bytes = lib.paged_attention_workspace_size(B, Hq, D, bs, bt.shape[1])
    assert ws_bytes > 0                       # this batch is split across partitions
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for call in range(2):
        q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16).cuda()
        ref = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        assert _regular(lib, ref, q, kp, vp, bt, lens, scale, ws) == 0
        assert _noalloc(lib, got, q, kp, vp, bt, lens, scale) == 0
        torch.cuda.synchronize()
        code = ctypes.c_int(-1)
        assert lib.pkv_get_device_error(ctypes.byref(code), None) == 0 and code.value == 0
        _close(got.float().cpu().numpy(), ref.float().cpu().numpy().astype(np.float64),
               f"call {call} vs the regular entry point")
        if call == 0:
            kv, vv = pkv.pool_views(kp.cpu(), vp.cpu())
            want = oatt.paged_decode(q.cpu(), kv, vv, bt.cpu().numpy(), lens.cpu().numpy(),
                                     scale, bs)
            _close(got.float().cpu().numpy(), want, "call 0 vs the oracle")


def test_noalloc_python_wrapper_matches_the_oracle():
    """The binding's paged_attention_decode_noalloc (its size pre-check, shape
    checks and argument marshalling) against the float64 oracle."""
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    library()
    torch.cuda.set_device(0)
    B, Hq, Hkv, D, bs, lens_list = SHAPES[0]
    g = torch.Generator().manual_seed(5)
    kp, vp, bt, lens = _batch(g, B, Hq, Hkv, D, bs, lens_list)
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16).cuda()
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode_noalloc(out, q, kp, vp, bt, lens, 1.0 / math.sqrt(D))
    assert pkv.get_device_error() == 0
    kv, vv = pkv.pool_views(kp.cpu(), vp.cpu())
    want = oatt.paged_decode(q.cpu(), kv, vv, bt.cpu().numpy(), lens.cpu().numpy(),
                             1.0 / math.sqrt(D), bs)
    _close(out.float().cpu().numpy(), want, "wrapper vs the oracle")
