"""The oracle's pins are strong enough: each test here plants one plausible
mistake in a temporary copy of the oracle's C source (a dropped term, a wrong
sign or index, a transposed operand, a wrong tie-break, ...), compiles it,
binds the oracle wrapper to the mutant, and checks that at least one pin of
tests/test_oracle_pins.py fails.  The mistakes are planted in the oracle, on
the CPU; the real oracle is untouched.
"""
import ctypes
import inspect
import os
import shutil

import pytest

import oracle
import test_oracle_pins as pins
from conftest import cached_workload

SRC = os.path.join(os.path.dirname(oracle.__file__), "jet_oracle.c")

# name: (exact text in jet_oracle.c, replacement)
MUTANTS = {
    "transposed-W": ("acc += h[k] * bf16_to_double(w[k]);",
                     "acc += h[k] * bf16_to_double(W[k * v_count + i]);"),
    "lse-sign": ("return M + log(sum);", "return M - log(sum);"),
    "lse-drops-last-entry": ("for (int64_t i = 0; i < n; ++i) sum += exp(z[i] - M);",
                             "for (int64_t i = 0; i + 1 < n; ++i) sum += exp(z[i] - M);"),
    "gather-token-off-by-one": ("logp[j] = z[pos] - lse_r;", "logp[j] = z[pos > 0 ? pos - 1 : pos] - lse_r;"),
    "chain-drops-first-token": ("for (int64_t t = cand_offsets[c]; t < cand_offsets[c + 1]; ++t) acc += logp[t];",
                                "for (int64_t t = cand_offsets[c] + 1; t < cand_offsets[c + 1]; ++t) acc += logp[t];"),
    "temperature-multiplies": ("s[c] / T - amax", "s[c] * T - amax"),
    "tie-goes-to-last": ("if (s[c] > s[best]) best = c;", "if (s[c] >= s[best]) best = c;"),
    "expected-index-off-by-one": ("ex += (double)(c - c0) * q[c];", "ex += (double)(c - c0 + 1) * q[c];"),
    "entropy-sign": ("if (q[c] > 0.0) ent -= q[c] * log(q[c]);", "if (q[c] > 0.0) ent += q[c] * log(q[c]);"),
    "confidence-wrong-normaliser": ("1.0 - ent / log((double)K)", "1.0 - ent / log(2.0)"),
    "mass-counts-duplicates": ("if (first) m += exp(s[c]);", "m += exp(s[c]);"),
    "mass-uses-temperature": ("if (first) m += exp(s[c]);", "if (first) m += exp(s[c] / T);"),
    "q-equiv-self-only": ("qe += q[c2];", "qe += (c2 == c) ? q[c2] : 0.0;"),
    "union-position-shifted": ("if (union_ids[u] == tok_ids[j]) pos = u;",
                               "if (union_ids[u] == tok_ids[j]) pos = (u + 1) % n_union;"),
    "union-normaliser-is-vocab": ("row_logits(h, W, d, n_norm, union_ids, z);\n      const double lse_r = logsumexp(z, n_norm);",
                                  "row_logits(h, W, d, n_norm, union_ids, z);\n      const double lse_r = logsumexp(z, n_norm) + (union_ids ? 0.25 : 0.0);"),
    "margin-counts-winner-copy": ("if (!same_sequence(tok_ids, cand_offsets, c, best) && q[c] > other) other = q[c];",
                                  "if (c != best && q[c] > other) other = q[c];"),
}


def _pin_functions():
    return [(n, f) for n, f in inspect.getmembers(pins, inspect.isfunction) if n.startswith("test_")]


def _run_pins():
    """Run every pin against the currently bound oracle library; return the
    names of the pins that failed."""
    failed = []
    for name, fn in _pin_functions():
        params = inspect.signature(fn).parameters
        calls = [dict()]
        if "case" in params:
            calls = [dict(case=c) for c in ("tiny", "ragged")]
        for kw in calls:
            if "wl_cache" in params:
                kw = dict(kw, wl_cache=cached_workload)
            try:
                fn(**kw)
            except Exception:            # assertion or oracle error: the pin caught it
                failed.append(name)
                break
    return failed


@pytest.fixture
def bind_mutant(tmp_path, monkeypatch):
    def bind(name):
        old, new = MUTANTS[name]
        text = open(SRC).read()
        assert text.count(old) >= 1, f"mutation site for {name} not found in the oracle source"
        src = tmp_path / f"mutant_{name}.c"
        src.write_text(text.replace(old, new))
        lib = oracle.configure(ctypes.CDLL(oracle.compile_library(str(src), str(tmp_path / f"{name}.so"))))
        monkeypatch.setattr(oracle, "_lib", lib)
    return bind


def test_pins_pass_on_the_real_oracle():
    assert _run_pins() == []


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc needed to build mutants")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_planted_mistake_fails_a_pin(bind_mutant, name):
    bind_mutant(name)
    failed = _run_pins()
    assert failed, f"no pin caught the planted mistake '{name}'"
