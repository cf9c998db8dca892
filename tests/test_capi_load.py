"""The C-ABI library builds, loads without a GPU and exports every declared symbol."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("spec_draft", "spec_verify", "spec_accept", "kv_commit", "spec_model_create", "spec_kv_create",
              "spec_prefill", "spec_schedule_k"):
        assert n in names


def test_library_exports_every_declared_symbol():
    from speculative_decoding_verify_04_gb300 import build, spec
    path = build.build()
    lib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(spec.EXPORTS) == declared_functions()
    spec.load(path)
    assert spec.load().spec_last_error() == b""


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "speculative_decoding_verify_04_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_header_compiles_as_plain_c():
    """The ABI header needs no C++: a C99 compiler accepts it alone."""
    import shutil
    import subprocess
    import pytest
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", "c", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the compiled library the binding raises: there is no fallback."""
    import pytest
    from speculative_decoding_verify_04_gb300 import spec
    monkeypatch.setattr(spec, "_lib", None)
    with pytest.raises(spec.SpecError, match="missing"):
        spec.load(str(tmp_path / "libspec.so"))
