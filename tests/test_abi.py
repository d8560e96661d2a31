"""The C ABI library: it builds for sm_103a and exports every declared symbol.
No compute calls here (no GPU on the CPU test runner)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^(?:int|void|const char \*)\s*\*?(jet_\w+)\s*\(", text, re.M))
    return sorted(names)


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="CUDA toolkit not available")
def test_library_builds_and_exports_all_declared_symbols():
    from candidate_answer_scoring_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    names = declared_symbols()
    assert "jet_score_sets" in names and "jet_score_tokens" in names and "jet_create" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    lib.jet_status_string.restype = ctypes.c_char_p
    assert lib.jet_status_string(0) == b"ok"
    assert lib.jet_status_string(-9) == b"device-side wait timed out"


def test_host_checks_reject_bad_arguments_without_a_device():
    """Argument checks that run before any CUDA call."""
    from candidate_answer_scoring_gb300 import build
    lib = ctypes.CDLL(build.build())
    out = ctypes.c_void_p()
    assert lib.jet_create(ctypes.byref(out), 63, 1000, 10, 10, 0) == -1     # d not a multiple of 64
    assert lib.jet_create(ctypes.byref(out), 64, 0, 10, 10, 0) == -1        # V < 1
    assert lib.jet_create(None, 64, 1000, 10, 10, 0) == -1
    assert lib.jet_score_sets(None, None, None, 1, None, None, 1, None, 1, None, None, 1,
                              ctypes.c_float(1.0), 0, None, 0, None, None) == -1


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    import candidate_answer_scoring_gb300.jetscore as js
    monkeypatch.setattr(js, "_lib", None)
    monkeypatch.setattr(js, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        js.load()
