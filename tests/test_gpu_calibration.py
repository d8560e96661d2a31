"""jet_fit_temperature against the fp64 oracle (oracle/calibration.py).

Tolerance: the fitted T within 1e-4 relative and the mean NLL within 1e-5
absolute of the oracle's (the GPU sums per-set terms in fp32 and the sets in
fp64; the optimum is flat, so T is the sensitive output)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wk
from oracle import calibration as cal

pytestmark = pytest.mark.gpu

T_RTOL = 1e-4
NLL_ATOL = 1e-5


@pytest.fixture(scope="module")
def jet():
    import candidate_answer_scoring_gb300 as jet
    jet.load()
    return jet


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_fit(jet, s, tok, co, so, gold, T_min=0.05, T_max=100.0):
    sc = jet.JetScorer(64, 100, 4, max(4, tok.size))
    return sc.fit_temperature(dev(np.asarray(s, np.float32)), dev(tok), dev(co), dev(so), dev(gold), T_min, T_max)


def labelled_sets(n_sets, T_true, seed, dup_prob=0.15):
    """Scores of a scored workload and gold labels drawn from q(T_true)."""
    wl = wk.custom(64, 700, n_sets, K=(2, 12), length=(1, 5), dup_prob=dup_prob, peak=(0.3, 0.9), seed=seed)
    r = oracle.score_workload(wl)
    s = r.s.astype(np.float32)                      # both sides see the same fp32 scores
    rng = np.random.default_rng(seed)
    gold = []
    for k in range(wl.n_sets):
        c0, c1 = wl.set_offsets[k], wl.set_offsets[k + 1]
        a = s[c0:c1].astype(np.float64) / T_true
        p = np.exp(a - a.max()); p /= p.sum()
        gold.append(int(rng.choice(c1 - c0, p=p)))
    return s, wl.tok_ids, wl.cand_offsets, wl.set_offsets, np.asarray(gold, np.int32)


def check(jet, s, tok, co, so, gold, T_min=0.05, T_max=100.0):
    T_ref, nll_ref = cal.fit_temperature(s.astype(np.float64), tok, co, so, gold, T_min, T_max)
    T, nll = gpu_fit(jet, s, tok, co, so, gold, T_min, T_max)
    assert abs(T - T_ref) <= T_RTOL * T_ref, (T, T_ref)
    assert abs(nll - nll_ref) <= NLL_ATOL, (nll, nll_ref)
    return T


def test_closed_form(jet):
    n1, n2, a = 3, 1, 2.0
    s, tok, co, so, gold = [], [], [0], [0], []
    for i in range(n1 + n2):
        s += [0.0, -a]; tok += [2 * i, 2 * i + 1]; co += [len(tok) - 1, len(tok)]; so.append(len(co) - 1)
        gold.append(0 if i < n1 else 1)
    args = (np.array(s, np.float32), np.array(tok, np.int32), np.array(co, np.int32), np.array(so, np.int32),
            np.array(gold, np.int32))
    T = check(jet, *args)
    assert abs(T - a / math.log(n1 / n2)) < 1e-4


@pytest.mark.parametrize("T_true,seed", [(0.7, 1), (1.0, 2), (2.179, 3), (4.0, 4)])
def test_labelled_sets(jet, T_true, seed):
    check(jet, *labelled_sets(60, T_true, seed))


def test_boundaries(jet):
    s = np.array([0.0, -2.0] * 5, np.float32)
    tok = np.arange(10, dtype=np.int32)
    co = np.arange(11, dtype=np.int32)
    so = np.arange(0, 11, 2, dtype=np.int32)
    T, _ = gpu_fit(jet, s, tok, co, so, np.zeros(5, np.int32), 0.1, 10.0)        # always right
    assert abs(T - 0.1) < 1e-6
    gold = np.array([0, 1, 0, 1, 0], np.int32)
    s2 = np.array([0.0, -2.0, 0.0, -2.0, 0.0, -2.0, 0.0, -2.0, 0.0, -2.0], np.float32)
    check(jet, s2, tok, co, so, gold, 0.1, 10.0)


def test_rejects_gold_outside_its_set(jet):
    import candidate_answer_scoring_gb300 as j
    s, tok, co, so, gold = labelled_sets(10, 1.0, 5)
    gold = gold.copy()
    gold[3] = np.diff(so)[3]
    with pytest.raises(j.JetError) as e:
        gpu_fit(jet, s, tok, co, so, gold)
    assert e.value.status == -3


def test_bound_call_matches_fit_temperature(jet):
    """bind_fit_temperature marshals once; call() is the bare C call and
    returns the same (T, nll) as fit_temperature, bit for bit, on every call."""
    s, tok, co, so, gold = labelled_sets(60, 1.7, seed=41)
    sc = jet.JetScorer(64, 100, 4, max(4, tok.size))
    args = (dev(s), dev(tok), dev(co), dev(so), dev(gold))
    ref = sc.fit_temperature(*args)
    call = sc.bind_fit_temperature(*args)
    assert call() == ref and call() == ref


def test_large_problem():
    """1500 sets of 20-40 candidates (about 45k, some sets with a repeated
    text in the gold class): each of the CTA's threads takes one or two sets
    per Newton step; the fit matches the oracle."""
    import candidate_answer_scoring_gb300 as jet
    n_sets = 1500
    rng = np.random.default_rng(52)
    K = rng.integers(20, 41, size=n_sets)
    so = np.concatenate([[0], np.cumsum(K)]).astype(np.int32)
    n_cand = int(so[-1])
    tok = np.empty(n_cand, np.int32)
    for k in range(n_sets):
        ids = rng.choice(1000, size=K[k], replace=False)
        if rng.random() < 0.2:
            ids[-1] = ids[0]                        # a duplicate text: its gold class has two labels
        tok[so[k]:so[k + 1]] = ids
    co = np.arange(n_cand + 1, dtype=np.int32)       # one token per candidate
    s = (rng.normal(size=n_cand) * 3).astype(np.float32)
    for k in range(n_sets):                         # equal texts carry equal scores
        c0, c1 = so[k], so[k + 1]
        s[c0:c1][tok[c0:c1] == tok[c0]] = s[c0]
    gold = np.empty(n_sets, np.int32)
    for k in range(n_sets):
        a = s[so[k]:so[k + 1]].astype(np.float64) / 1.6
        p = np.exp(a - a.max()); p /= p.sum()
        gold[k] = rng.choice(K[k], p=p)
    check(jet, s, tok, co, so, gold)
