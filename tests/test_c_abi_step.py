"""The shard step through the C ABI alone: tests/c_abi/step_check.c uses
include/vsf.h with plain cudaMalloc buffers (no Python, no torch) for two
steps and compares every buffer with the oracle's C entry points byte for
byte. On CPU it must compile and link (the header is valid C); on the GPU it
must run and report bit-exact results."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "step_check.c")


def _compile(out):
    import oracle
    from fsdp_buffer_layout_gb300 import _build
    lib, orc = _build.build(), oracle.build()
    libdir, orcdir = os.path.dirname(lib), os.path.dirname(orc)
    cmd = [_build.nvcc(), "-O2", SRC, "-I", _build.INCLUDE, "-L", libdir, "-lvsf", "-L", orcdir,
           "-loracle", "-lcudart", "-Xlinker", "-rpath=" + libdir, "-Xlinker", "-rpath=" + orcdir,
           "-o", str(out)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def test_c_program_compiles_against_the_header(tmp_path):
    assert os.path.exists(_compile(tmp_path / "step_check"))


@pytest.mark.gpu
def test_shard_step_through_the_c_abi_is_bit_exact(tmp_path):
    exe = _compile(tmp_path / "step_check")
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("bit-exact"), r.stdout
