"""fp64 CPU oracle of the candidate-set scoring head -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``jet_oracle.c`` (plain C,
double precision, OpenMP over rows) through ctypes; see that file for the
equations it follows and the page sections it cites.  It shares no code with
the CUDA library and never imports it.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jet_oracle.c")
_LIB = os.path.join(_HERE, "libjetoracle.so")

ORC_OK, ORC_ERR_ARG, ORC_ERR_TOKEN, ORC_ERR_OFFSETS, ORC_ERR_UNION = 0, -1, -2, -3, -5


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, OpenMP, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        compile_library(_SRC, tmp)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def configure(lib: C.CDLL) -> C.CDLL:
    """Declare the C signatures on a loaded oracle library."""
    P = C.c_void_p
    i64 = C.c_int64
    lib.orc_log_softmax_at.argtypes = [P, i64, i64, P]
    lib.orc_logits.argtypes = [P, P, i64, i64, i64, P, i64, P]
    lib.orc_score_tokens.argtypes = [P, P, i64, i64, i64, P, P, i64, P, P, P, C.c_int]
    lib.orc_score_tokens_restricted.argtypes = [P, P, i64, i64, i64, P, i64, P, P, i64, P, P, P, C.c_int]
    lib.orc_set_rules.argtypes = [P, P, i64, P, i64, P, P, i64, C.c_double] + [P] * 8
    lib.orc_score_sets.argtypes = ([P, P, i64, i64, i64, P, P, i64, P, i64, P, P, i64,
                                    C.c_double, C.c_int, P, i64] + [P] * 10 + [C.c_int])
    lib.orc_max_threads.argtypes = []
    return lib


def compile_library(src: str, out: str) -> str:
    """Compile an oracle source file (used by the build and by mutation tests)."""
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-ffp-contract=off",
                           "-Wall", "-shared", "-o", out, src, "-lm"])
    return out


def _load():
    global _lib
    if _lib is None:
        _lib = configure(C.CDLL(build()))
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dt)


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != ORC_OK:
        raise OracleError(f"{what}: oracle status {rc}")


def max_threads() -> int:
    return int(_load().orc_max_threads())


def log_softmax_at(z: np.ndarray, tok: int) -> float:
    """l = z[tok] - logsumexp(z) for a given logit vector (fp64)."""
    z = _c(z, np.float64)
    out = np.zeros(1, np.float64)
    _check(_load().orc_log_softmax_at(_p(z), z.size, int(tok), _p(out)), "log_softmax_at")
    return float(out[0])


def logits(H: np.ndarray, W: np.ndarray, rows) -> np.ndarray:
    """Full fp64 logit vectors z[r, :] for the listed rows."""
    H = _c(H, np.uint16); W = _c(W, np.uint16)
    rows = _c(rows, np.int64)
    out = np.zeros((rows.size, W.shape[0]), np.float64)
    _check(_load().orc_logits(_p(H), _p(W), H.shape[0], H.shape[1], W.shape[0], _p(rows), rows.size,
                              _p(out)), "logits")
    return out


def score_tokens(H, W, tok_row, tok_ids, want=None, union_ids=None, threads: int = 0):
    """Per-token log-probabilities and per-row log-sum-exp (NaN where not asked)."""
    H = _c(H, np.uint16); W = _c(W, np.uint16)
    tok_row = _c(tok_row, np.int32); tok_ids = _c(tok_ids, np.int32)
    n_tok = tok_ids.size
    wantb = None if want is None else _c(want, np.uint8)
    logp = np.empty(n_tok, np.float64)
    lse = np.empty(H.shape[0], np.float64)
    lib = _load()
    if union_ids is None:
        rc = lib.orc_score_tokens(_p(H), _p(W), H.shape[0], H.shape[1], W.shape[0], _p(tok_row),
                                  _p(tok_ids), n_tok, _p(wantb), _p(logp), _p(lse), int(threads))
    else:
        u = _c(union_ids, np.int32)
        rc = lib.orc_score_tokens_restricted(_p(H), _p(W), H.shape[0], H.shape[1], W.shape[0], _p(u),
                                             u.size, _p(tok_row), _p(tok_ids), n_tok, _p(wantb),
                                             _p(logp), _p(lse), int(threads))
    _check(rc, "score_tokens")
    return logp, lse


@dataclass
class SetResult:
    s: np.ndarray
    q: np.ndarray
    q_equiv: np.ndarray
    decision: np.ndarray
    expected: np.ndarray
    confidence: np.ndarray
    mass: np.ndarray
    margin: np.ndarray
    logp: Optional[np.ndarray] = None
    lse: Optional[np.ndarray] = None


def _set_outputs(n_cand: int, n_sets: int):
    f = lambda n: np.empty(n, np.float64)
    return (f(n_cand), f(n_cand), f(n_cand), np.empty(n_sets, np.int32), f(n_sets), f(n_sets),
            f(n_sets), f(n_sets))


def set_rules(logp, tok_ids, cand_offsets, set_offsets, kind, T: float) -> SetResult:
    """Chain rule and set rules from given per-token log-probabilities."""
    logp = _c(logp, np.float64); tok_ids = _c(tok_ids, np.int32)
    co = _c(cand_offsets, np.int32); so = _c(set_offsets, np.int32); kd = _c(kind, np.uint8)
    outs = _set_outputs(co.size - 1, so.size - 1)
    rc = _load().orc_set_rules(_p(logp), _p(tok_ids), tok_ids.size, _p(co), co.size - 1, _p(so), _p(kd),
                               so.size - 1, float(T), *[_p(o) for o in outs])
    _check(rc, "set_rules")
    return SetResult(*outs)


def score_sets(H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T: float, mode: int = 0,
               union_ids=None, threads: int = 0) -> SetResult:
    """The whole path for one batch (full vocabulary, or the union when mode == 1)."""
    H = _c(H, np.uint16); W = _c(W, np.uint16)
    tok_row = _c(tok_row, np.int32); tok_ids = _c(tok_ids, np.int32)
    co = _c(cand_offsets, np.int32); so = _c(set_offsets, np.int32); kd = _c(kind, np.uint8)
    u = None if union_ids is None else _c(union_ids, np.int32)
    logp = np.empty(tok_ids.size, np.float64)
    lse = np.empty(H.shape[0], np.float64)
    outs = _set_outputs(co.size - 1, so.size - 1)
    rc = _load().orc_score_sets(_p(H), _p(W), H.shape[0], H.shape[1], W.shape[0], _p(tok_row), _p(tok_ids),
                                tok_ids.size, _p(co), co.size - 1, _p(so), _p(kd), so.size - 1, float(T),
                                int(mode), _p(u), 0 if u is None else u.size, _p(logp), _p(lse),
                                *[_p(o) for o in outs], int(threads))
    _check(rc, "score_sets")
    r = SetResult(*outs)
    r.logp, r.lse = logp, lse
    return r


def score_workload(wl, threads: int = 0) -> SetResult:
    """Convenience: run the whole path on a ``workloads.Workload``."""
    return score_sets(wl.H, wl.W, wl.tok_row, wl.tok_ids, wl.cand_offsets, wl.set_offsets, wl.kind,
                      wl.T, wl.mode, wl.union_ids, threads)
