"""The C interface used from C: tests/c_api_host.c compiled with gcc as C99
against include/kvattn.h and linked to the in-tree library, run without a GPU
(host-only calls: split, prepare, sequence copy and removal, the batching
loop)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "continuous_batching_kv_gb300", "libkvattn.so")


def test_c_program_drives_the_host_calls(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(LIB):
        pytest.skip("library not built")
    exe = str(tmp_path / "c_api_host")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_api_host.c"), LIB,
                        "-Wl,-rpath," + os.path.dirname(LIB), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")   # host calls only
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok fixed_passes=4096 continuous_passes=")
