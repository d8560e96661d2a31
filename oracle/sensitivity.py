"""fp64 oracle of decision-guided layer sensitivity -- TEST INFRASTRUCTURE.

"FastJEV: Understanding Redundancy for Compact JEV Inference", section 3.4,
Eq. 5-6, written out:

  ctr(v)    = v - mean(v) 1                    (removes a common logit shift)
  rms(v)    = ||v||_2 / sqrt(m)                 (v has m entries)
  d_l(x)    = rms(ctr(z^(-l)(x) - z(x))) / max(eps, rms(ctr(z(x)))),  eps = 1e-8
  J_l       = mean over the calibration inputs x of d_l(x)
  selection = the k layers with the smallest J_l, ties resolved by layer index

Each input x has its own logit vector (candidate logits; the lengths may
differ), given in CSR layout: entries offsets[x] .. offsets[x+1].
"""
from __future__ import annotations

import numpy as np

EPS = 1e-8


def _rms_ctr(v: np.ndarray) -> float:
    c = v - v.mean()
    return float(np.sqrt(np.sum(c * c) / v.size))


def layer_sensitivity(z, z_skip, offsets, k: int):
    """z [total], z_skip [L, total], offsets [n+1] -> (d [L, n], J [L], selected [k])."""
    z = np.asarray(z, np.float64)
    z_skip = np.asarray(z_skip, np.float64)
    offsets = np.asarray(offsets)
    L, n = z_skip.shape[0], offsets.size - 1
    d = np.empty((L, n))
    for l in range(L):
        for x in range(n):
            a, b = int(offsets[x]), int(offsets[x + 1])
            d[l, x] = _rms_ctr(z_skip[l, a:b] - z[a:b]) / max(EPS, _rms_ctr(z[a:b]))
    J = d.mean(axis=1)
    order = sorted(range(L), key=lambda l: (J[l], l))
    return d, J, np.asarray(order[:k], np.int64)
