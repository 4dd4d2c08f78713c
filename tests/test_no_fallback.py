"""The product path has no fallback: without its compiled library it fails
loudly, and no product source imports, links or calls the oracle."""
import ast
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fsdp_buffer_layout_gb300")


def test_missing_library_raises(tmp_path):
    code = ("from fsdp_buffer_layout_gb300 import vsf as V\n"
            "try:\n"
            "    V.vsf_plan_create([V.make_desc((4, 8), V.VSF_GRAN_ROWS, 1, 0)], 2, 8)\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n"
            "else:\n"
            "    print('no error')\n")
    env = dict(os.environ, VSF_LIBRARY=str(tmp_path / "absent" / "libvsf.so"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, check=True)
    assert r.stdout.startswith("raised:") and "not built" in r.stdout, r.stdout


def _product_files(exts):
    for d, _, files in os.walk(PKG):
        if "_build" in d or "__pycache__" in d:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_product_python_never_imports_the_oracle():
    for path in _product_files((".py",)):
        tree = ast.parse(open(path).read(), path)
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            else:
                continue
            assert not any(n == "oracle" or n.startswith("oracle.") for n in names), path


def test_product_native_code_never_names_the_oracle():
    for path in _product_files((".cu", ".cuh", ".cpp", ".h")):
        src = open(path).read()
        for word in ("liboracle", "orc_", "oracle.cpp"):
            assert word not in src, f"{path} names {word}"
    for path in _product_files((".py",)):
        assert "liboracle" not in open(path).read(), path
