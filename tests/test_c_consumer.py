"""The boundary is a C ABI: a plain C program (tests/c_consumer/consumer.c),
compiled with gcc against include/adaln.h and linked to the library, calls the
host-only entry points and the argument validation.  No GPU is needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_include():
    for d in ("/usr/local/cuda/include", os.path.join(os.environ.get("CUDA_HOME", ""), "include")):
        if d and os.path.exists(os.path.join(d, "cuda_runtime_api.h")):
            return d
    return None


def test_c_program_uses_the_abi(tmp_path):
    import modulation_adaln_fwd_gb300 as m
    cc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include()
    if cc is None or inc is None:
        pytest.skip("no C compiler or CUDA headers")
    exe = str(tmp_path / "consumer")
    libdir = os.path.dirname(m.lib_path)
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", inc, os.path.join(ROOT, "tests", "c_consumer", "consumer.c"), "-o", exe,
           m.lib_path, "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    env = dict(os.environ, CUDA_VISIBLE_DEVICES=os.environ.get("CUDA_VISIBLE_DEVICES", ""))
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failure(s)" in r.stdout, r.stdout


@pytest.mark.gpu
def test_c_program_runs_the_chain_on_the_gpu(tmp_path):
    """The same from C with device memory: forward and backward through the C ABI,
    checked in the program against double-precision sums."""
    import modulation_adaln_fwd_gb300 as m
    cc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include()
    if cc is None or inc is None:
        pytest.skip("no C compiler or CUDA headers")
    cudalib = os.path.join(os.path.dirname(inc), "lib64")
    exe = str(tmp_path / "consumer_gpu")
    libdir = os.path.dirname(m.lib_path)
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", inc, os.path.join(ROOT, "tests", "c_consumer", "consumer_gpu.c"), "-o", exe,
           m.lib_path, "-L", cudalib, "-lcudart", "-lm", "-Wl,-rpath," + libdir,
           "-Wl,-rpath," + cudalib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failure(s)" in r.stdout, r.stdout
