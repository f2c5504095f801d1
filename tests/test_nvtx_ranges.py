"""NVTX ranges around every exported call that launches work (CPU test, no GPU needed).

The library opens an NVTX range named after the call for the host-side part of each such call.
This test compiles a minimal NVTX injection library (tests/nvtx_probe.c, which records each
range push and pop), points NVTX_INJECTION64_PATH at it in a child process, calls every entry
point with a null descriptor or error word (each returns an error before touching the device),
and checks that each call opened its own range and closed it again.
"""
import os
import subprocess
import sys
import textwrap

import pytest

from recurrent_state_update_gb300 import build as bld

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

TRACED = [
    "mamba_state_update", "mamba_conv_update", "mamba_spec_commit", "mamba_conv_varlen", "mamba_chunk_scan",
    "mamba_chunk_scan_noalloc", "mamba_slot_copy", "mamba_ckpt_store_int8", "mamba_ckpt_load_int8",
    "mamba1_conv_update", "mamba1_state_update", "mamba_selftest_wait_timeout",
]


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("nvtx") / "libnvtx_probe.so")
    subprocess.run(["gcc", "-O1", "-shared", "-fPIC", "-Wall", os.path.join(HERE, "nvtx_probe.c"), "-o", out],
                   check=True)
    return out


def test_every_launching_call_opens_and_closes_its_range(probe):
    lib = bld.build()
    if os.environ.get("MAMBA_NVTX", "1") == "0":
        pytest.skip("library built without NVTX ranges")
    script = textwrap.dedent(f"""
        import ctypes
        lib = ctypes.CDLL({lib!r})
        zeros = [ctypes.c_void_p(0)] * 32   # null descriptor / error word, zero sizes
        codes = {{}}
        for name in {TRACED!r}:
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            codes[name] = fn(*zeros)
        probe = ctypes.CDLL({probe!r})
        probe.nvtx_probe_log.restype = ctypes.c_char_p
        print("CODES", codes)
        print(probe.nvtx_probe_log().decode())
    """)
    env = dict(os.environ, NVTX_INJECTION64_PATH=probe)
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.splitlines()
    codes = eval(lines[0][len("CODES "):])  # noqa: S307 - our own child's dict literal
    assert all(c < 0 for c in codes.values()), codes  # every call refused its arguments
    events = [ln for ln in lines[1:] if ln]
    assert events == [e for name in TRACED for e in ("+" + name, "-")], events
