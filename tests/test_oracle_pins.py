"""Pins of the fp64 oracle against what the pages and mathematics fix.

Every check compares the oracle with something other than itself: a value the
pages print, a closed form, an invariant, a library routine or brute force.
Chosen so that a dropped term, a wrong sign or index, or a transposed operand
anywhere in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
import workloads as wk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _single_token_sets(s_lists, kinds=None):
    """Layout where every candidate is one token with log-prob = the given s."""
    logp, tok, co, so, kd = [], [], [0], [0], []
    tid = 0
    for i, s_list in enumerate(s_lists):
        for s in s_list:
            logp.append(s)
            tok.append(tid)
            tid += 1
            co.append(len(logp))
        so.append(len(co) - 1)
        kd.append(0 if kinds is None else kinds[i])
    return (np.array(logp), np.array(tok, np.int32), np.array(co, np.int32),
            np.array(so, np.int32), np.array(kd, np.uint8))


# --------------------------------------------------------------------------
# values printed on the pages
# --------------------------------------------------------------------------
def test_worked_example_from_page():
    ex = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    s = [math.log(p) for p in ex["likelihoods"]]
    logp, tok, co, so, kd = _single_token_sets([s])
    r = oracle.set_rules(logp, tok, co, so, kd, ex["temperature"])
    np.testing.assert_allclose(r.q, ex["normalized"], rtol=0, atol=1e-12)
    assert r.decision[0] == 0
    # mass of the allowed set = summed complete-candidate likelihoods
    np.testing.assert_allclose(r.mass[0], sum(ex["likelihoods"]), rtol=1e-12)


def test_worked_example_through_full_vocab_softmax():
    """Token probabilities 0.06 / 0.02 produced by a logit vector: l = ln p
    exactly (Eq. 1-2), then Eq. 4 gives 0.75 / 0.25."""
    p = np.array([0.06, 0.02, 0.5, 0.42])
    z = np.log(p) + 3.7  # any common shift
    l0 = oracle.log_softmax_at(z, 0)
    l1 = oracle.log_softmax_at(z, 1)
    assert abs(l0 - math.log(0.06)) < 1e-14
    assert abs(l1 - math.log(0.02)) < 1e-14
    logp, tok, co, so, kd = _single_token_sets([[l0, l1]])
    r = oracle.set_rules(logp, tok, co, so, kd, 1.0)
    np.testing.assert_allclose(r.q, [0.75, 0.25], atol=1e-12)


# --------------------------------------------------------------------------
# normalisation, temperature, binary rule
# --------------------------------------------------------------------------
def test_q_sums_to_one_and_matches_scipy_softmax():
    rng = np.random.default_rng(1)
    sets = [list(rng.normal(-10, 4, size=k)) for k in (1, 2, 3, 7, 26, 64)]
    for T in (1.0, wk.T_FITTED, 0.3):
        logp, tok, co, so, kd = _single_token_sets(sets)
        r = oracle.set_rules(logp, tok, co, so, kd, T)
        for i, s_list in enumerate(sets):
            q = r.q[so[i]:so[i + 1]]
            assert abs(q.sum() - 1.0) < 1e-12
            np.testing.assert_allclose(q, scipy.special.softmax(np.array(s_list) / T), atol=1e-13)


def test_binary_closed_form_and_threshold():
    rng = np.random.default_rng(2)
    for T in (1.0, wk.T_FITTED):
        pairs = [list(rng.normal(-8, 3, size=2)) for _ in range(50)] + [[-3.0, -3.0]]
        logp, tok, co, so, kd = _single_token_sets(pairs, kinds=[1] * len(pairs))
        r = oracle.set_rules(logp, tok, co, so, kd, T)
        for i, (s0, s1) in enumerate(pairs):
            qt = scipy.special.expit((s1 - s0) / T)
            assert abs(r.q[2 * i + 1] - qt) < 1e-13
            assert abs(r.expected[i] - qt) < 1e-13          # binary returns q(true)
            assert r.decision[i] == (1 if s1 > s0 else 0)   # exact tie -> false (index 0)


def test_temperature_is_a_power_of_likelihoods():
    """q(c) is proportional to P(c)**(1/T) (Eq. 4 with temperature)."""
    P = np.array([0.3, 0.05, 0.001, 0.2])
    for T in (0.5, 1.0, wk.T_FITTED, 7.0):
        logp, tok, co, so, kd = _single_token_sets([list(np.log(P))])
        r = oracle.set_rules(logp, tok, co, so, kd, T)
        ref = P ** (1.0 / T) / np.sum(P ** (1.0 / T))
        np.testing.assert_allclose(r.q, ref, rtol=1e-12)


def test_decision_and_mass_do_not_depend_on_temperature():
    rng = np.random.default_rng(3)
    sets = [list(rng.normal(-5, 2, size=k)) for k in (2, 5, 9)]
    logp, tok, co, so, kd = _single_token_sets(sets)
    base = oracle.set_rules(logp, tok, co, so, kd, 1.0)
    for T in (0.2, wk.T_FITTED, 11.0):
        r = oracle.set_rules(logp, tok, co, so, kd, T)
        np.testing.assert_array_equal(r.decision, base.decision)
        np.testing.assert_allclose(r.mass, base.mass, rtol=1e-15)
        np.testing.assert_array_equal(r.s, base.s)


# --------------------------------------------------------------------------
# duplicates, equivalence classes, ties
# --------------------------------------------------------------------------
def test_duplicate_candidate_shifts_distribution_and_ties_to_lowest_index():
    T = 1.7
    P = np.array([0.1, 0.4, 0.05])
    # candidates 0..2 with token sequences (10,), (11, 12), (13,); then a copy of 1
    logp = np.array([math.log(P[0]), math.log(P[1]), 0.0, math.log(P[2]), math.log(P[1]), 0.0])
    tok = np.array([10, 11, 12, 13, 11, 12], np.int32)
    co = np.array([0, 1, 3, 4, 6], np.int32)
    so = np.array([0, 4], np.int32)
    r = oracle.set_rules(logp, tok, co, so, np.array([0], np.uint8), T)
    Pt = P ** (1 / T)
    denom = Pt.sum() + Pt[1]
    np.testing.assert_allclose(r.q[:3], Pt / denom, rtol=1e-12)
    np.testing.assert_allclose(r.q[3], Pt[1] / denom, rtol=1e-12)
    assert r.s[1] == r.s[3]
    assert r.decision[0] == 1                       # first of the tied pair
    np.testing.assert_allclose(r.q_equiv[[1, 3]], 2 * Pt[1] / denom, rtol=1e-12)
    np.testing.assert_allclose(r.q_equiv[[0, 2]], r.q[[0, 2]], rtol=0)
    # distinct sequences counted once in the mass
    np.testing.assert_allclose(r.mass[0], P.sum(), rtol=1e-12)
    # margin ignores the winner's own duplicate
    np.testing.assert_allclose(r.margin[0], r.q[1] - r.q[0], rtol=1e-12)


def test_all_equivalent_set_has_infinite_margin_and_k1_rules():
    logp = np.array([-2.0, -2.0, -0.5])
    tok = np.array([4, 4, 9], np.int32)
    co = np.array([0, 1, 2, 3], np.int32)
    so = np.array([0, 2, 3], np.int32)
    r = oracle.set_rules(logp, tok, co, so, np.array([0, 0], np.uint8), 1.0)
    assert math.isinf(r.margin[0])
    np.testing.assert_allclose(r.q[:2], [0.5, 0.5], atol=1e-15)
    assert r.decision[0] == 0
    # K = 1: q = 1, decision 0, expected 0, confidence 1
    assert r.q[2] == 1.0 and r.decision[1] == 0 and r.expected[1] == 0.0 and r.confidence[1] == 1.0
    np.testing.assert_allclose(r.mass[1], math.exp(-0.5), rtol=1e-15)


# --------------------------------------------------------------------------
# ordinal expectation and confidence
# --------------------------------------------------------------------------
def test_uniform_and_dominant_sets():
    for K in (2, 5, 26):
        logp, tok, co, so, kd = _single_token_sets([[-4.0] * K], kinds=[2])
        r = oracle.set_rules(logp, tok, co, so, kd, 1.3)
        assert abs(r.expected[0] - (K - 1) / 2) < 1e-12
        assert abs(r.confidence[0]) < 1e-12
        for i_star in (0, K // 2, K - 1):
            T = 1.5
            s = [-100.0] * K
            s[i_star] = -100.0 + 50 * T + 40 * T
            logp, tok, co, so, kd = _single_token_sets([s], kinds=[2])
            r = oracle.set_rules(logp, tok, co, so, kd, T)
            assert abs(r.expected[0] - i_star) < 1e-10
            assert 1.0 - r.confidence[0] < 1e-10
            assert r.decision[0] == i_star


def test_confidence_matches_scipy_entropy():
    rng = np.random.default_rng(4)
    for K in (2, 3, 8, 26, 64):
        s = list(rng.normal(-6, 2.5, size=K))
        logp, tok, co, so, kd = _single_token_sets([s])
        r = oracle.set_rules(logp, tok, co, so, kd, wk.T_FITTED)
        ref = 1.0 - scipy.stats.entropy(r.q) / math.log(K)
        assert abs(r.confidence[0] - ref) < 1e-12


def test_expected_index_is_probability_weighted_level():
    """Ordinal contract: distribution over level indices and its mean; checked
    on a two-point distribution whose mean is known in closed form."""
    # only levels 1 and 3 carry mass, in ratio 1:3  ->  mean = 1*0.25 + 3*0.75
    s = [-1e4, math.log(1.0), -1e4, math.log(3.0), -1e4]
    logp, tok, co, so, kd = _single_token_sets([s], kinds=[2])
    r = oracle.set_rules(logp, tok, co, so, kd, 1.0)
    assert abs(r.expected[0] - 2.5) < 1e-12


# --------------------------------------------------------------------------
# token-level log-probabilities
# --------------------------------------------------------------------------
def test_log_prob_invariant_to_constant_logit_shift():
    rng = np.random.default_rng(5)
    z = rng.normal(0, 3, size=1000)
    for tok in (0, 17, 999):
        base = oracle.log_softmax_at(z, tok)
        for c in (-50.0, 1e-3, 80.0):
            assert abs(oracle.log_softmax_at(z + c, tok) - base) < 1e-12
    # and the pin is not vacuous: scaling the row does change it
    assert abs(oracle.log_softmax_at(2 * z, 17) - oracle.log_softmax_at(z, 17)) > 1e-3


@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_token_log_probs_match_torch_log_softmax(case, wl_cache):
    if case == "tiny":
        wl = wl_cache("tiny")
    else:
        wl = wl_cache("custom", 128, 777, 6, seed=11)
    H = torch.from_numpy(wk.bf16_bits_to_f32(wl.H).astype(np.float64))
    W = torch.from_numpy(wk.bf16_bits_to_f32(wl.W).astype(np.float64))
    ref = torch.log_softmax(H @ W.T, dim=-1)
    ref_lse = torch.logsumexp(H @ W.T, dim=-1).numpy()
    logp, lse = oracle.score_tokens(wl.H, wl.W, wl.tok_row, wl.tok_ids)
    want = ref[torch.from_numpy(wl.tok_row.astype(np.int64)), torch.from_numpy(wl.tok_ids.astype(np.int64))]
    np.testing.assert_allclose(logp, want.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_single_token_candidate_equals_first_position_log_prob(wl_cache):
    """Tiny workload: candidates 0 (one token) and 1 (three tokens) share their
    first token and its row, so l agrees exactly (prefix output supplies the
    first-token probability)."""
    wl = wl_cache("tiny")
    r = oracle.score_workload(wl)
    c0, c1 = wl.cand_offsets[0], wl.cand_offsets[1]
    assert wl.tok_ids[c0] == wl.tok_ids[c1]
    assert r.logp[c0] == r.logp[c1]
    assert r.s[0] == r.logp[c0]
    # candidate 3 copies candidate 2: identical s, tie goes to index 2
    assert r.s[2] == r.s[3]
    assert r.q_equiv[2] == r.q_equiv[3] == r.q[2] + r.q[3]


def test_common_prefix_can_be_factored_out():
    """Gemma/MLX architecture page, "Candidate likelihoods": dropping a common
    candidate-token prefix leaves the normalised distribution unchanged."""
    rng = np.random.default_rng(6)
    d, V = 32, 50
    W = wk.to_bf16_bits(rng.normal(0, d ** -0.5, size=(V, d)).astype(np.float32))
    shared = (7, 3)
    cands = [shared + (1,), shared + (2, 9), shared + (40,)]
    rows, toks, co, hist = [], [], [0], {}
    H = []
    for c in cands:
        for t in range(len(c)):
            key = c[:t]
            if key not in hist:
                hist[key] = len(H)
                H.append(wk.to_bf16_bits(rng.normal(size=d).astype(np.float32)))
            rows.append(hist[key])
            toks.append(c[t])
        co.append(len(toks))
    H = np.stack(H)
    rows, toks, co = np.array(rows, np.int32), np.array(toks, np.int32), np.array(co, np.int32)
    so, kd = np.array([0, 3], np.int32), np.array([0], np.uint8)
    logp, _ = oracle.score_tokens(H, W, rows, toks)
    full = oracle.set_rules(logp, toks, co, so, kd, 1.4)
    dropped = logp.copy()
    for c in range(3):
        dropped[co[c]:co[c] + len(shared)] = 0.0
    fac = oracle.set_rules(dropped, toks, co, so, kd, 1.4)
    np.testing.assert_allclose(fac.q, full.q, atol=1e-13)
    assert fac.decision[0] == full.decision[0]
    # the shared positions really do carry probability (pin not vacuous)
    assert np.all(logp[:len(shared)] < -0.01)


def test_brute_force_chain_rule_sums_to_one():
    """V=8, d=16, one hidden row per history: the probabilities of all 8**3
    length-3 continuations sum to 1 (chain rule, Eq. 3 over Eq. 1)."""
    rng = np.random.default_rng(7)
    V, d, L = 8, 16, 3
    W = wk.to_bf16_bits(rng.normal(0, 1.5 * d ** -0.5, size=(V, d)).astype(np.float32))
    hist = {}
    H = []
    for n in range(L):
        for h in np.ndindex(*([V] * n)):
            hist[tuple(h)] = len(H)
            H.append(wk.to_bf16_bits(rng.normal(size=d).astype(np.float32)))
    H = np.stack(H)
    rows, toks, co = [], [], [0]
    for seq in np.ndindex(*([V] * L)):
        for t in range(L):
            rows.append(hist[tuple(seq[:t])])
            toks.append(seq[t])
        co.append(len(toks))
    rows, toks, co = np.array(rows, np.int32), np.array(toks, np.int32), np.array(co, np.int32)
    so = np.array([0, V ** L], np.int32)
    r = oracle.score_sets(H, W, rows, toks, co, so, np.array([0], np.uint8), 1.0)
    assert abs(np.exp(r.s).sum() - 1.0) < 1e-12
    assert abs(r.mass[0] - 1.0) < 1e-12
    np.testing.assert_allclose(r.q, np.exp(r.s), atol=1e-14)   # normaliser is already 1
    # first-position marginal: summing over the tail gives the one-token probability
    lp0, _ = oracle.score_tokens(H, W, np.zeros(V, np.int32), np.arange(V, dtype=np.int32))
    marg = np.exp(r.s).reshape(V, V * V).sum(axis=1)
    np.testing.assert_allclose(marg, np.exp(lp0), atol=1e-13)


# --------------------------------------------------------------------------
# restricted (union) normaliser
# --------------------------------------------------------------------------
def test_restricted_with_union_equal_to_vocab_is_full_mode():
    wl = workloads_small_binary()
    rng = np.random.default_rng(8)
    U = rng.permutation(wl.V).astype(np.int32)           # order must not matter
    full = oracle.score_sets(wl.H, wl.W, wl.tok_row, wl.tok_ids, wl.cand_offsets, wl.set_offsets,
                             wl.kind, 1.3, 0)
    rest = oracle.score_sets(wl.H, wl.W, wl.tok_row, wl.tok_ids, wl.cand_offsets, wl.set_offsets,
                             wl.kind, 1.3, 1, U)
    for a in ("logp", "s", "q", "q_equiv", "expected", "confidence", "mass"):
        np.testing.assert_allclose(getattr(rest, a), getattr(full, a), rtol=1e-11, atol=1e-13)
    np.testing.assert_array_equal(rest.decision, full.decision)


def test_restricted_q_equals_full_q_for_single_token_sets():
    wl = workloads_small_binary()
    U = wl.info["codes"]
    for T in (1.0, wk.T_FITTED):
        full = oracle.score_sets(wl.H, wl.W, wl.tok_row, wl.tok_ids, wl.cand_offsets, wl.set_offsets,
                                 wl.kind, T, 0)
        rest = oracle.score_sets(wl.H, wl.W, wl.tok_row, wl.tok_ids, wl.cand_offsets, wl.set_offsets,
                                 wl.kind, T, 1, U)
        np.testing.assert_allclose(rest.q, full.q, atol=1e-12)
        np.testing.assert_array_equal(rest.decision, full.decision)
        # union-relative mass is larger than the full-vocabulary mass
        assert np.all(rest.mass > full.mass)
        assert np.all(rest.mass <= 1.0 + 1e-12)
    # restricted l = z - lse over the union, checked on the raw logits
    z = oracle.logits(wl.H, wl.W, np.arange(3))
    for r in range(3):
        zu = z[r, U]
        want = zu - scipy.special.logsumexp(zu)
        j = np.nonzero(wl.tok_row == r)[0]
        pos = [int(np.nonzero(U == t)[0][0]) for t in wl.tok_ids[j]]
        np.testing.assert_allclose(rest.logp[j], want[pos], atol=1e-12)


def workloads_small_binary():
    return wk.binary_batch(n_questions=12, random_pairs=True, d=64, V=300)


# --------------------------------------------------------------------------
# the oracle rejects what the method does not define
# --------------------------------------------------------------------------
def test_oracle_rejects_invalid_layouts():
    logp, tok, co, so, kd = _single_token_sets([[-1.0, -2.0]])
    with pytest.raises(oracle.OracleError):
        oracle.set_rules(logp, tok, co, so, kd, 0.0)                    # T must be > 0
    with pytest.raises(oracle.OracleError):                              # sets must cover all
        oracle.set_rules(logp, tok, co, np.array([0, 1], np.int32), kd, 1.0)
    bad_co = np.array([0, 1, 1], np.int32)                                # empty candidate
    with pytest.raises(oracle.OracleError):
        oracle.set_rules(logp[:1], tok[:1], bad_co, so, kd, 1.0)
    with pytest.raises(oracle.OracleError):                              # binary needs K = 2
        oracle.set_rules(*_single_token_sets([[-1.0, -2.0, -3.0]], kinds=[1])[:4],
                         np.array([1], np.uint8), 1.0)
    wl = workloads_small_binary()
    with pytest.raises(oracle.OracleError):                              # token outside union
        oracle.score_sets(wl.H, wl.W, wl.tok_row, wl.tok_ids, wl.cand_offsets, wl.set_offsets,
                          wl.kind, 1.0, 1, wl.info["codes"][:3])
