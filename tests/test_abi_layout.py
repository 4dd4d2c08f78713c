"""The Python binding's ctypes structures against the C header: a C program
compiled here (gcc, include/vsf.h only) prints sizeof of every public struct
and offsetof of every field the binding declares. Names, order, sizes and
padding must agree, or a field read through the binding would return another
field's bytes."""
import ctypes
import shutil
import subprocess

import pytest

from fsdp_buffer_layout_gb300 import _build, vsf as V

STRUCTS = [V.vsf_tensor_desc, V.vsf_adam_hparams, V.vsf_plan_info, V.vsf_muon_hparams]


def _c_layout(tmp_path):
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "vsf.h"', "int main(void) {"]
    for st in STRUCTS:
        t = st.__name__
        lines.append(f'  printf("{t} %zu\\n", sizeof({t}));')
        for name, _ in st._fields_:
            lines.append(f'  printf("{t}.{name} %zu\\n", offsetof({t}, {name}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", _build.INCLUDE, str(src),
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    return dict(line.rsplit(" ", 1) for line in out.splitlines())


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_ctypes_structs_match_the_header(tmp_path):
    c = _c_layout(tmp_path)
    for st in STRUCTS:
        t = st.__name__
        assert int(c[t]) == ctypes.sizeof(st), t
        for name, _ in st._fields_:
            assert int(c[f"{t}.{name}"]) == getattr(st, name).offset, f"{t}.{name}"
