"""The C-ABI from a plain C99 host: tests/c_host_calls.c includes dsa.h as C
(strict C99, warnings as errors), links libdsa.so and makes every call that
needs no GPU. No GPU: the device calls it makes only get NULL arguments,
which the library refuses on the host."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_host_compiles_and_runs(dsa_lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = dsa_lib.LIB_PATH
    exe = tmp_path / "c_host_calls"
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_host_calls.c"),
           "-o", str(exe), lib, "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    # the C compiler's struct layouts must equal the binding's ctypes mirrors
    sizes = [ctypes.sizeof(dsa_lib.dsa_config_t), dsa_lib.dsa_config_t.score_buffer_bytes.offset,
             ctypes.sizeof(dsa_lib.dsa_step_args_t), ctypes.sizeof(dsa_lib.dsa_workspace_layout_t)]
    r = subprocess.run([str(exe), *map(str, sizes)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
