"""The product path stands apart from the oracle and has no fallback: no
module of the package imports the oracle or another implementation of the
method, and the binding refuses to run without the compiled library. No GPU."""

import ast
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "attention_neo_qknorm_gb300")


def _imports(path):
    tree = ast.parse(open(path).read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            yield from (a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            yield node.module or ""


def test_package_modules_do_not_import_the_oracle():
    for name in os.listdir(PKG):
        if name.endswith(".py"):
            mods = list(_imports(os.path.join(PKG, name)))
            assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), f"{name} imports the oracle"
            assert not any(m.split(".")[0] in ("triton", "numpy") for m in mods if name == "neo.py"), \
                "the binding marshals arguments only"


def test_cuda_sources_have_no_host_compute_path():
    for name in os.listdir(os.path.join(PKG, "csrc")):
        text = open(os.path.join(PKG, "csrc", name)).read()
        assert "oracle" not in text.lower(), name


def test_binding_fails_loudly_without_the_library(tmp_path):
    """A fresh interpreter pointed at a missing library raises on the first
    call instead of computing anything another way."""
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from attention_neo_qknorm_gb300 import neo\n"
        "neo.LIB_PATH = %r\n"
        "try:\n"
        "    neo.load_library(neo.LIB_PATH)\n"
        "except FileNotFoundError:\n"
        "    print('refused')\n"
    ) % (ROOT, str(tmp_path / "libneo_missing.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "refused"
