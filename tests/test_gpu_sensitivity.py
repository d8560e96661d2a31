"""jet_layer_sensitivity against the fp64 oracle (oracle/sensitivity.py).

Tolerance (fp32 two-pass statistics): d and J within 1e-4 relative; the
selection exact wherever neighbouring J values differ by more than 1e-4
relative, and otherwise a valid ordering."""
import numpy as np
import pytest
import torch

from oracle import sensitivity as sens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def scorer():
    import candidate_answer_scoring_gb300 as jet
    return jet.JetScorer(64, 100, 4, 4)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def case(seed, n=40, L=36, const_input=False, len_range=(2, 66)):
    rng = np.random.default_rng(seed)
    lens = rng.integers(len_range[0], len_range[1], size=n)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(offsets[-1])
    z = rng.normal(-20, 6, size=total).astype(np.float32)
    if const_input:                       # flat logit vectors: rms(ctr(z)) = 0, d = rd / eps
        z[offsets[0]:offsets[1]] = -7.0
        z[offsets[1]:offsets[2]] = -7.3   # fp32 sums of -7.3 are inexact: flatness must be exact
    scale = np.exp(rng.normal(-2, 1.5, size=L))           # layers differ in how much they move the logits
    z_skip = (z[None, :] + scale[:, None] * rng.normal(size=(L, total)) + rng.normal(size=(L, 1)) * 3).astype(np.float32)
    return z, z_skip, offsets


@pytest.mark.parametrize("seed,const_input,L,len_range", [
    (0, False, 36, (2, 66)), (1, False, 36, (2, 66)), (2, True, 36, (2, 66)),
    (4, False, 9, (200, 600)),     # segments held 8 per lane and, past 256 logits, read in two passes
])
def test_matches_oracle(scorer, seed, const_input, L, len_range):
    z, z_skip, offsets = case(seed, L=L, const_input=const_input, len_range=len_range)
    k = 6
    d, J, sel = scorer.layer_sensitivity(dev(z), dev(z_skip), dev(offsets), k)
    torch.cuda.synchronize()
    d_ref, J_ref, sel_ref = sens.layer_sensitivity(z.astype(np.float64), z_skip.astype(np.float64), offsets, k)
    np.testing.assert_allclose(d.cpu().numpy(), d_ref, rtol=1e-4, atol=0)
    np.testing.assert_allclose(J.cpu().numpy(), J_ref, rtol=1e-4, atol=0)
    order = np.argsort(J_ref, kind="stable")
    gaps = np.diff(J_ref[order]) / np.maximum(J_ref[order][1:], 1e-30)
    if np.all(gaps[:k] > 1e-4):
        assert list(sel.cpu().numpy()) == list(sel_ref)
    else:
        Jg = J.cpu().numpy()
        s = sel.cpu().numpy()
        assert len(set(s)) == k and np.all(np.diff(Jg[s]) >= 0)


def test_rejects_empty_input(scorer):
    import candidate_answer_scoring_gb300 as jet
    z, z_skip, offsets = case(3, n=5, L=4)
    bad = offsets.copy()
    bad[2] = bad[1]
    with pytest.raises(jet.JetError) as e:
        scorer.layer_sensitivity(dev(z), dev(z_skip), dev(bad), 2)
    assert e.value.status == -3


def test_bound_call_matches_layer_sensitivity(scorer):
    """bind_layer_sensitivity marshals once into caller buffers; call() is the
    bare C call: bit-identical d, J and selection to layer_sensitivity."""
    z, z_skip, offsets = case(5, n=64, L=40)
    a = (dev(z), dev(z_skip), dev(offsets))
    d_ref, J_ref, sel_ref = scorer.layer_sensitivity(*a, 7)
    d = torch.empty_like(d_ref)
    J = torch.empty_like(J_ref)
    sel = torch.empty(7, dtype=torch.int32, device="cuda")
    call = scorer.bind_layer_sensitivity(*a, 7, d, J, sel)
    for _ in range(2):
        call()
        assert torch.equal(d, d_ref) and torch.equal(J, J_ref) and torch.equal(sel, sel_ref)
