"""The CUDA path and the oracle stay apart: the package never imports, includes
or names the oracle, the oracle never uses the package, the shared input
generators import neither, importing the package loads no oracle module, and a
missing library fails loudly instead of falling back to anything."""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "bit_row_speculative_gb300")


def _sources(folder, exts):
    for dirpath, dirnames, files in os.walk(folder):
        dirnames[:] = [d for d in dirnames if not d.startswith(("_build", "__pycache__"))]
        for f in files:
            if f.endswith(exts):
                yield os.path.join(dirpath, f)


def _text(path):
    with open(path, encoding="utf-8") as fh:
        return fh.read()


def test_package_never_uses_the_oracle():
    pat = re.compile(r"\boracle\b")
    hits = [p for p in _sources(PKG, (".py", ".cu", ".cuh", ".h", ".c")) if pat.search(_text(p))]
    hits += [p for p in _sources(os.path.join(ROOT, "include"), (".h",)) if pat.search(_text(p))]
    assert not hits, f"the CUDA path names the oracle: {hits}"


def test_oracle_never_uses_the_package():
    # imports of the package, includes of its headers, paths into its sources or its library
    pat = re.compile(r"^\s*(import|from)\s+bit_row_speculative_gb300\b|#include\s+[\"<][^\">]*(q4|csrc)|"
                     r"[\"']csrc[\"']|libq4\.so|include[\"'/]", re.M)
    for planted in ("import bit_row_speculative_gb300 as q4", "from bit_row_speculative_gb300 import build",
                    '#include "q4.h"', '#include "../bit_row_speculative_gb300/csrc/q4_tm.cuh"',
                    'os.path.join(ROOT, "bit_row_speculative_gb300", "csrc")', 'ctypes.CDLL("libq4.so")'):
        assert pat.search(planted), planted          # the check is not vacuous
    hits = [p for p in _sources(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")) if pat.search(_text(p))]
    assert not hits, f"the oracle uses the CUDA path: {hits}"


def test_input_generators_import_neither():
    src = _text(os.path.join(ROOT, "synth_inputs.py"))
    assert not re.search(r"^\s*(import|from)\s+(oracle|bit_row_speculative_gb300)\b", src, re.M)


def test_importing_the_package_loads_no_oracle_module():
    code = ("import sys, bit_row_speculative_gb300 as q4; q4.lib(); "
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]; "
            "assert not bad, bad")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]


def test_missing_library_fails_loudly(monkeypatch):
    import bit_row_speculative_gb300 as q4
    monkeypatch.setattr(q4, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libq4.so"))
    monkeypatch.setattr(q4, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        q4.lib()
    with pytest.raises(RuntimeError, match="not built"):
        q4.packed_bytes(128, 512)
