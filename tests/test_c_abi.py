"""The C ABI used from C.  ``tests/c/abi_closed_form.c`` includes only
``include/ls.h`` and the CUDA runtime header, links ``libls.so``, and checks
three decode tokens of every variant and gate whose outputs and states have
closed forms (its header derives them), through ``ls_decode_step``,
``ls_decode_step_host`` and ``ls_decode_step_split_static``, then
``ls_window_commit``, ``ls_pool_read`` and ``ls_pool_status``."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_closed_form.c")
PKG = os.path.join(ROOT, "recurrent_state_quantization_gb300")


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME")
    if home:
        return home
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _build(tmp_path) -> str:
    import __graft_entry__
    __graft_entry__.build()
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("needs gcc")
    cuda = _cuda_home()
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
               if os.path.isdir(d)]
    exe = str(tmp_path / "abi_closed_form")
    cmd = [gcc, "-std=c11", "-O2", "-Wall", "-Wextra", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), SRC, "-L", PKG, "-lls",
           *[f"-L{d}" for d in libdirs], "-lcudart", "-lm", f"-Wl,-rpath,{PKG}",
           *[f"-Wl,-rpath,{d}" for d in libdirs], "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "warning" not in r.stderr, r.stderr
    return exe


def test_c_program_builds_against_the_header(tmp_path):
    """Plain C11 against include/ls.h compiles without warnings and links
    libls.so (no GPU needed)."""
    _build(tmp_path)


@pytest.mark.gpu
def test_c_program_closed_forms(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_closed_form: ok" in r.stdout
