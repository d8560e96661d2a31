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


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "jetscore.h"

int main(void) {
  jet_ctx *ctx = NULL;
  jet_set_out out;
  memset(&out, 0, sizeof out);
  /* host checks run before any CUDA call: no device needed */
  if (jet_create(&ctx, 63, 1000, 16, 16, 0) != JET_ERR_ARG) return 1;      /* d % 64 != 0 */
  if (jet_score_sets(NULL, NULL, NULL, 1, NULL, NULL, 1, NULL, 1, NULL, NULL, 1, 1.0f,
                     JET_MODE_FULL, NULL, 0, &out, NULL) != JET_ERR_ARG) return 2;
  if (strcmp(jet_status_string(JET_OK), "ok") != 0) return 3;
  printf("%s|%s\n", jet_status_string(JET_ERR_TOKEN_RANGE), jet_status_string(JET_ERR_TIMEOUT));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_compiles_as_c99_and_links_from_c(tmp_path):
    """include/jetscore.h is plain C (C99, -pedantic, warnings as errors) and a
    C program links against libjetscore.so and runs its host-side checks."""
    import subprocess
    from candidate_answer_scoring_gb300 import build
    lib = build.build()
    src = tmp_path / "use_abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{ROOT}/include", str(src),
                    f"-L{libdir}", "-l:" + os.path.basename(lib), f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip() == "token id or row index out of range|device-side wait timed out"
