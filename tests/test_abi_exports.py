"""The C-ABI library loads without a GPU and exports every function pagedkv.h declares."""
import ctypes
import os
import re

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
