"""The library and the oracle stay apart.

No source file of the package or its public header names the oracle; no oracle file names the
package, its headers or its CUDA sources; the seeded input generators (``synth/``) import neither;
and the package refuses to import when its compiled library is missing, so no call can fall back
to anything else.
"""
import ast
import os
import re
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE_EXT = (".py", ".cu", ".cuh", ".h", ".c", ".cpp", ".hpp")


def _sources(*dirs):
    for d in dirs:
        for base, subdirs, files in os.walk(os.path.join(ROOT, d)):
            subdirs[:] = [s for s in subdirs if s != "__pycache__" and not s.startswith("_build")]
            for f in files:
                if f.endswith(SOURCE_EXT):
                    yield os.path.join(base, f)


def test_package_never_names_the_oracle():
    files = list(_sources("request_token_sampling_gb300", "include"))
    assert len(files) >= 8
    for p in files:
        text = open(p, encoding="utf-8").read()
        assert not re.search(r"\boracle\b", text, re.IGNORECASE), f"{os.path.relpath(p, ROOT)} names the oracle"


def test_oracle_never_names_the_package():
    files = list(_sources("oracle"))
    assert files
    for p in files:
        text = open(p, encoding="utf-8").read()
        for word in ("request_token_sampling_gb300", "strata_", "csrc", "include/"):
            assert word not in text, f"{os.path.relpath(p, ROOT)} names {word!r}"


def test_input_generators_import_neither_side():
    for p in _sources("synth"):
        if not p.endswith(".py"):
            continue
        tree = ast.parse(open(p, encoding="utf-8").read())
        for node in ast.walk(tree):
            names = []
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            for n in names:
                top = n.split(".")[0]
                assert top not in ("oracle", "request_token_sampling_gb300"), f"{p} imports {n}"


def test_package_import_fails_without_its_library(tmp_path):
    """The package's Python files without the compiled library: importing it raises ImportError."""
    pkg = tmp_path / "request_token_sampling_gb300"
    pkg.mkdir()
    src = os.path.join(ROOT, "request_token_sampling_gb300")
    for f in os.listdir(src):
        if f.endswith(".py"):
            shutil.copy(os.path.join(src, f), pkg / f)
    r = subprocess.run([sys.executable, "-c", "import request_token_sampling_gb300"], cwd=tmp_path,
                       capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, PYTHONPATH=str(tmp_path)))
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "not built" in r.stderr
