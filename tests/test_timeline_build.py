"""The instrumented library behind ``paged_kv_gqa_attn_gb300.timeline`` (-DPA_TIMELINE, built into
its own directory, never loaded by the product path) still compiles and exports its readers."""

import shutil
import subprocess
import sys

import pytest

from paged_kv_gqa_attn_gb300 import build

READERS = ("paged_attn_timeline_read_verify", "paged_attn_timeline_read_verify_steps",
           "paged_attn_timeline_read_prefill")


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="needs nvcc")
def test_instrumented_library_builds_and_exports_its_readers():
    path = build.build(timeline=True)
    assert path == build.TIMELINE_LIB_PATH and path != build.LIB_PATH
    # a separate process: the product library may already be loaded in this one
    code = ("import ctypes, sys; lib = ctypes.CDLL(sys.argv[1]); "
            "print(' '.join(n for n in sys.argv[2:] if not hasattr(lib, n)))")
    res = subprocess.run([sys.executable, "-c", code, path, *READERS], capture_output=True, text=True,
                         timeout=120)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == "", "missing: " + res.stdout
