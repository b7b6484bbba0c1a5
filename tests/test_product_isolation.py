"""The product path and the oracle stay apart: importing the package and loading its library pulls in no part of
oracle/ (no module, no shared object), no product source imports or includes it, and the oracle shares no code
with the CUDA sources. Only tests/, smoke() and the bench's baseline legs may load the oracle."""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_decoding_tree_top_gb300")


def _sources(top, exts):
    for d, _, files in os.walk(top):
        if "__pycache__" in d:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_loading_the_product_loads_no_oracle(dtlib):  # dtlib: the library is built first
    code = (
        "import sys\n"
        "import speculative_decoding_tree_top_gb300 as pkg\n"
        "from speculative_decoding_tree_top_gb300 import dominotree, synth, buildlib\n"
        "dominotree.lib()\n"
        "assert not any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules), 'oracle module imported'\n"
        "maps = open('/proc/self/maps').read()\n"
        "assert 'liboracle' not in maps, 'oracle library mapped'\n"
        "assert 'libdominotree' in maps, 'product library not mapped'\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]


def test_no_product_source_imports_or_includes_the_oracle():
    for path in _sources(PKG, (".py",)):
        text = open(path).read()
        assert not re.search(r"^\s*(from\s+oracle\b|import\s+oracle\b)", text, re.M), path
    for path in list(_sources(PKG, (".cu", ".cuh", ".h"))) + list(_sources(os.path.join(ROOT, "include"), (".h",))):
        text = open(path).read()
        assert not re.search(r'#\s*include\s*[<"][^>"]*oracle', text), path
        assert "orc_" not in text, path  # the oracle's C entry points


def test_oracle_includes_nothing_of_the_product():
    text = open(os.path.join(ROOT, "oracle", "oracle.cpp")).read()
    includes = re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', text)
    assert includes and all("/" not in i and not i.endswith((".cuh", ".cu")) and i != "dominotree.h"
                            for i in includes), includes
    assert "dt_" not in re.sub(r"//.*|/\*.*?\*/", "", text, flags=re.S).replace("std::", ""), "calls into the product"


def test_the_binding_fails_loudly_without_its_library():
    """No fallback: with the compiled library absent, the first call raises instead of computing anything else."""
    code = (
        "import pathlib\n"
        "from speculative_decoding_tree_top_gb300 import buildlib, dominotree\n"
        "buildlib.LIB = pathlib.Path('/nonexistent/libdominotree.so')\n"
        "try:\n"
        "    dominotree.lib()\n"
        "except RuntimeError as e:\n"
        "    assert 'must be built' in str(e)\n"
        "else:\n"
        "    raise SystemExit('no error without the library')\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:] + r.stdout[-500:]
