"""Pins of the temperature-fitting oracle: a closed form, brute force, the
boundary cases and the gold-class rule."""
import math

import numpy as np

from oracle import calibration as cal


def _binary_sets(margins_gold):
    """Binary sets with scores (0, -a); gold index per set."""
    s, tok, co, so, gold = [], [], [0], [0], []
    t = 0
    for a, g in margins_gold:
        for v in (0.0, -a):
            s.append(v); tok.append(t); t += 1; co.append(len(tok))
        so.append(len(co) - 1)
        gold.append(g)
    return (np.array(s), np.array(tok, np.int32), np.array(co, np.int32), np.array(so, np.int32),
            np.array(gold, np.int32))


def test_closed_form_optimum():
    """n1 sets right by margin a, n2 wrong by margin a: exp(a/T*) = n1/n2."""
    for n1, n2, a in ((3, 1, 2.0), (5, 2, 0.7), (9, 4, 3.3)):
        s, tok, co, so, gold = _binary_sets([(a, 0)] * n1 + [(a, 1)] * n2)
        T, val = cal.fit_temperature(s, tok, co, so, gold)
        T_star = a / math.log(n1 / n2)
        assert abs(T - T_star) < 1e-6 * T_star
        p = n1 / (n1 + n2)          # optimum: q(gold) = p on right sets, 1 - p on wrong ones
        ref = -(n1 * math.log(p) + n2 * math.log(1 - p)) / (n1 + n2)
        assert abs(val - ref) < 1e-10


def test_grid_brute_force():
    rng = np.random.default_rng(3)
    margins = [(float(rng.uniform(0.1, 4.0)), int(rng.random() < 0.3)) for _ in range(40)]
    s, tok, co, so, gold = _binary_sets(margins)
    T, val = cal.fit_temperature(s, tok, co, so, gold)
    classes = cal.gold_classes(tok, co, so, gold)
    grid = np.exp(np.linspace(math.log(0.05), math.log(100.0), 400))
    assert val <= min(cal.nll(t, s, so, classes) for t in grid) + 1e-12


def test_boundaries():
    s, tok, co, so, gold = _binary_sets([(2.0, 0)] * 5)          # always right: sharpen to T_min
    T, _ = cal.fit_temperature(s, tok, co, so, gold, 0.1, 10.0)
    assert T == 0.1
    s, tok, co, so, gold = _binary_sets([(2.0, 0), (2.0, 1)])   # half right: flatten to T_max
    T, _ = cal.fit_temperature(s, tok, co, so, gold, 0.1, 10.0)
    assert T == 10.0


def test_gold_probability_summed_over_identical_text():
    # set: candidates A, B, A' (A' copies A), gold = A' : the class is {A, A'}
    s = np.array([-1.0, -0.5, -1.0])
    tok = np.array([7, 8, 7], np.int32)
    co = np.array([0, 1, 2, 3], np.int32)
    so = np.array([0, 3], np.int32)
    classes = cal.gold_classes(tok, co, so, np.array([2], np.int32))
    assert classes == [[0, 2]]
    T = 1.3
    q = np.exp(s / T) / np.exp(s / T).sum()
    assert abs(cal.nll(T, s, so, classes) + math.log(q[0] + q[2])) < 1e-14
