"""Every C-ABI entry point that does work opens an NVTX range named after
itself in the "fp8q" domain and closes it on return.

Checked without a GPU: a small NVTX tool (tests/nvtx_recorder.c, loaded
through NVTX_INJECTION64_PATH) logs the ranges while a child process calls
entry points whose host-side checks fail before any CUDA work."""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"

CHILD = textwrap.dedent("""
    import ctypes, sys
    sys.path.insert(0, {root!r})
    from tensor_scaling_cast_gb300 import fp8q
    L = fp8q.load()
    h = ctypes.c_void_p()
    assert L.fp8q_create(7, 16, 0, 0, ctypes.byref(h)) == -3            # bad format
    assert L.fp8q_cast(None, None, 1, 0, None, None, None, None, None) == -5
    assert L.mx_cast(None, 1, 4, 48, 0, 0, None, None, None, None) == -1
    assert L.fp8q_error_stats_noalloc(None, 9, 16, None, 0, None, None, None) == -3
    assert L.fp8q_strerror(-1) == b"invalid argument"                 # not traced
""")


@pytest.fixture(scope="module")
def recorder(tmp_path_factory):
    if not os.path.exists(os.path.join(CUDA_INC, "nvtx3", "nvToolsExt.h")):
        pytest.skip("NVTX headers not installed")
    out = str(tmp_path_factory.mktemp("nvtx") / "librec.so")
    subprocess.check_call(["gcc", "-O1", "-shared", "-fPIC", f"-I{CUDA_INC}", "-o", out,
                           os.path.join(ROOT, "tests", "nvtx_recorder.c")])
    return out


def test_entry_points_open_and_close_named_ranges(recorder, tmp_path):
    from tensor_scaling_cast_gb300 import build
    build.build()
    log = tmp_path / "ranges.txt"
    env = dict(os.environ, NVTX_INJECTION64_PATH=recorder, FP8Q_NVTX_LOG=str(log))
    subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], env=env, check=True, timeout=300)
    lines = log.read_text().splitlines()
    assert lines[0] == "domain fp8q"
    pushes = [ln.split()[1] for ln in lines if ln.startswith("push ")]
    # fp8q_create and mx_cast forward to their _ex forms: nested ranges
    assert pushes == ["fp8q_create", "fp8q_create_ex", "fp8q_cast", "mx_cast", "mx_cast_ex",
                      "fp8q_error_stats_noalloc"]
    depth = 0
    for ln in lines[1:]:
        depth += 1 if ln.startswith("push ") else -1
        assert depth >= 0
    assert depth == 0
