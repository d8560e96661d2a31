"""Shared helpers of the GPU parity tests: run the CUDA path and the fp64
oracle on the same seeded inputs and compare element by element.

Tolerances (the scoring benchmark's parity bar, with the remaining ones derived
from the fp32 arithmetic of the GPU path):
  logp, lse           2e-3 absolute
  q, expected         1e-4 absolute
  confidence, q_equiv 1e-4 absolute
  s                   2e-3 * (tokens in the candidate) absolute (sum of logp errors)
  mass                1e-4 absolute, and 1e-3 relative where the oracle's mass >= 1e-30
  decision            exact wherever the oracle's top-two margin exceeds 1e-3
  duplicates          identical token sequences tie bit for bit and resolve to
                      the lowest index
"""
from __future__ import annotations

import numpy as np

import workloads as wk

LOGP_ATOL = 2e-3
LSE_ATOL = 2e-3
Q_ATOL = 1e-4
EXPECTED_ATOL = 1e-4
CONF_ATOL = 1e-4
QEQ_ATOL = 1e-4
MASS_ATOL = 1e-4
MASS_RTOL = 1e-3
MASS_RTOL_FLOOR = 1e-30
MARGIN = 1e-3


def subset(wl: wk.Workload, set_ids) -> tuple:
    """A workload holding only the given sets (rows renumbered), plus the token
    and candidate indices of those sets in the original layout."""
    set_ids = sorted(int(s) for s in set_ids)
    cands = np.concatenate([np.arange(wl.set_offsets[k], wl.set_offsets[k + 1]) for k in set_ids])
    toks = np.concatenate([np.arange(wl.cand_offsets[c], wl.cand_offsets[c + 1]) for c in cands])
    rows, new_row = np.unique(wl.tok_row[toks], return_inverse=True)
    lens = wl.cand_offsets[cands + 1] - wl.cand_offsets[cands]
    ks = wl.set_offsets[np.array(set_ids) + 1] - wl.set_offsets[np.array(set_ids)]
    sub = wk.Workload(wl.name + "-subset", wl.d, wl.V, np.ascontiguousarray(wl.H[rows]), wl.W,
                      new_row.astype(np.int32), wl.tok_ids[toks].astype(np.int32),
                      np.concatenate([[0], np.cumsum(lens)]).astype(np.int32),
                      np.concatenate([[0], np.cumsum(ks)]).astype(np.int32),
                      wl.kind[set_ids].astype(np.uint8), wl.T, wl.mode, wl.union_ids, dict(wl.info))
    return sub, np.asarray(set_ids), cands, toks, rows


def duplicate_groups(wl: wk.Workload):
    """Per set, lists of candidate indices with identical token sequences."""
    out = []
    for k in range(wl.n_sets):
        seen = {}
        for c in range(wl.set_offsets[k], wl.set_offsets[k + 1]):
            key = tuple(wl.tok_ids[wl.cand_offsets[c]:wl.cand_offsets[c + 1]])
            seen.setdefault(key, []).append(c)
        out.extend(v for v in seen.values() if len(v) > 1)
    return out


def compare(wl: wk.Workload, gpu: dict, orc, set_ids=None, cands=None, toks=None, rows=None,
            check_lse=True) -> dict:
    """Assert GPU outputs agree with the oracle's; gpu holds full-batch numpy
    arrays, orc the oracle result of ``wl`` (or of its subset, with the index
    maps from ``subset``).  Returns error statistics."""
    if set_ids is None:
        set_ids = np.arange(wl.n_sets)
        cands = np.arange(wl.n_cand)
        toks = np.arange(wl.n_tok)
        rows = np.arange(wl.N)
    stats = {}
    g_logp = gpu["logp"][toks].astype(np.float64)
    err = np.abs(g_logp - orc.logp)
    stats["logp_max_abs"] = float(err.max())
    assert err.max() <= LOGP_ATOL, f"logp differs by {err.max():.3e} at token {toks[int(err.argmax())]}"
    if check_lse and "lse" in gpu:
        e = np.abs(gpu["lse"][rows].astype(np.float64) - orc.lse)
        e = e[np.isfinite(orc.lse)]
        stats["lse_max_abs"] = float(e.max()) if e.size else 0.0
        assert e.size == 0 or e.max() <= LSE_ATOL, f"lse differs by {e.max():.3e}"
    sub_co = np.concatenate([[0], np.cumsum(wl.cand_offsets[cands + 1] - wl.cand_offsets[cands])])
    m = np.diff(sub_co)
    e = np.abs(gpu["s"][cands].astype(np.float64) - orc.s)
    stats["s_max_abs"] = float(e.max())
    assert np.all(e <= LOGP_ATOL * m), "s differs beyond the summed logp tolerance"
    for key, tol in (("q", Q_ATOL), ("q_equiv", QEQ_ATOL)):
        e = np.abs(gpu[key][cands].astype(np.float64) - getattr(orc, key))
        stats[f"{key}_max_abs"] = float(e.max())
        assert e.max() <= tol, f"{key} differs by {e.max():.3e} at candidate {cands[int(e.argmax())]}"
    for key, tol in (("expected", EXPECTED_ATOL), ("confidence", CONF_ATOL)):
        e = np.abs(gpu[key][set_ids].astype(np.float64) - getattr(orc, key))
        stats[f"{key}_max_abs"] = float(e.max())
        assert e.max() <= tol, f"{key} differs by {e.max():.3e} at set {set_ids[int(e.argmax())]}"
    gm = gpu["mass"][set_ids].astype(np.float64)
    e = np.abs(gm - orc.mass)
    assert e.max() <= MASS_ATOL, f"mass differs by {e.max():.3e}"
    big = orc.mass >= MASS_RTOL_FLOOR
    if big.any():
        rel = e[big] / orc.mass[big]
        stats["mass_max_rel"] = float(rel.max())
        assert rel.max() <= MASS_RTOL, f"mass relative error {rel.max():.3e}"
    clear = orc.margin > MARGIN
    stats["decisions_checked"] = int(clear.sum())
    stats["decisions_total"] = int(len(set_ids))
    bad = np.nonzero(clear & (gpu["decision"][set_ids] != orc.decision))[0]
    assert bad.size == 0, f"decision differs on sets {set_ids[bad][:10]}"
    # within tolerance sets, the GPU decision must still be a maximum of its own s
    for i, k in enumerate(set_ids):
        c0, c1 = wl.set_offsets[k], wl.set_offsets[k + 1]
        s = gpu["s"][c0:c1]
        dgpu = int(gpu["decision"][k])
        assert 0 <= dgpu < c1 - c0 and s[dgpu] == s.max() and np.all(s[:dgpu] < s.max())
    return stats


def check_duplicates(wl: wk.Workload, gpu: dict) -> int:
    """Identical token sequences: bit-identical s and q, and the set's decision
    never points at a later copy of the first maximum."""
    n = 0
    for group in duplicate_groups(wl):
        s = gpu["s"][group]
        q = gpu["q"][group]
        assert np.all(s.view(np.uint32) == s[0].view(np.uint32)), f"duplicates {group} differ in s"
        assert np.all(q.view(np.uint32) == q[0].view(np.uint32)), f"duplicates {group} differ in q"
        qe = gpu["q_equiv"][group]
        assert np.all(qe.view(np.uint32) == qe[0].view(np.uint32))
        n += 1
    for k in range(wl.n_sets):
        c0, c1 = wl.set_offsets[k], wl.set_offsets[k + 1]
        d = int(gpu["decision"][k])
        s = gpu["s"][c0:c1]
        assert s[d] == s.max() and not np.any(s[:d] == s.max()), f"set {k}: tie not resolved to lowest index"
    return n
