"""Build-on-demand access to the product library for tests (no GPU needed to load)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import paged_kv_cache_259_gb300 as pkv  # noqa: E402
from paged_kv_cache_259_gb300 import build as pkv_build  # noqa: E402


def library():
    """Build libpagedkv.so if it is missing or stale, then load it."""
    pkv_build.build_library()
    return pkv.load_library()
