"""fp64 oracle of temperature fitting -- TEST INFRASTRUCTURE (see oracle/__init__.py).

The Gemma/MLX architecture page ("Output contracts") fits the set-softmax
temperature on labelled data.  The plain definition used here:

  q_c(T)   = exp(s_c / T) / sum_{c' in set} exp(s_c' / T)          (JET Eq. 4)
  NLL(T)   = mean over sets k of  -log sum_{c in G_k} q_c(T)
  G_k      = candidates of set k whose token sequence equals the gold one's
             (the gold probability is summed over labels with identical text,
             JET Eq. 5 discussion)
  T*       = argmin NLL(T) over [T_min, T_max]

NLL is convex in 1/T (a difference of log-sum-exps whose second term has zero
variance, since equivalent candidates share their score), hence unimodal in
log T; the oracle minimises it with a bounded scalar method (a library
routine) on log T, evaluating NLL straight from the definition.
"""
from __future__ import annotations

import math
from typing import Tuple

import numpy as np
import scipy.optimize
import scipy.special


def gold_classes(tok_ids, cand_offsets, set_offsets, gold) -> list:
    """Per set, the indices (global candidate ids) equivalent to the gold one."""
    out = []
    for k in range(len(set_offsets) - 1):
        c0, c1 = int(set_offsets[k]), int(set_offsets[k + 1])
        g = c0 + int(gold[k])
        if not (c0 <= g < c1):
            raise ValueError(f"gold index {gold[k]} outside set {k}")
        seq = tuple(tok_ids[cand_offsets[g]:cand_offsets[g + 1]])
        out.append([c for c in range(c0, c1) if tuple(tok_ids[cand_offsets[c]:cand_offsets[c + 1]]) == seq])
    return out


def nll(T: float, s, set_offsets, classes) -> float:
    """Mean gold negative log-likelihood at temperature T (fp64)."""
    s = np.asarray(s, np.float64)
    total = 0.0
    for k, G in enumerate(classes):
        c0, c1 = int(set_offsets[k]), int(set_offsets[k + 1])
        a = s[c0:c1] / T
        total += scipy.special.logsumexp(a) - scipy.special.logsumexp(s[G] / T)
    return total / len(classes)


def fit_temperature(s, tok_ids, cand_offsets, set_offsets, gold, T_min: float = 0.05,
                    T_max: float = 100.0) -> Tuple[float, float]:
    """(T*, NLL(T*)) minimising the gold NLL over [T_min, T_max]."""
    classes = gold_classes(tok_ids, cand_offsets, set_offsets, gold)
    f = lambda lt: nll(math.exp(lt), s, set_offsets, classes)
    r = scipy.optimize.minimize_scalar(f, bounds=(math.log(T_min), math.log(T_max)), method="bounded",
                                       options=dict(xatol=1e-10, maxiter=500))
    T = math.exp(r.x)
    # a minimum at the boundary: report the boundary itself
    for Tb in (T_min, T_max):
        if nll(Tb, s, set_offsets, classes) <= nll(T, s, set_offsets, classes):
            T = Tb
    return T, nll(T, s, set_offsets, classes)
