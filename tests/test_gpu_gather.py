"""jet_score_sets_gather: hidden rows read from a larger source array (the
answer positions of a right-padded backbone output): copied once into the
context's staging rows for the tcgen05 head, or read in place by the small
restricted kernel.  The gathered call must reproduce the compact call on the
same rows bit for bit (same bytes reach the same arithmetic), and match the
oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wk
from parity import compare

pytestmark = pytest.mark.gpu

OUT = ("logp", "lse", "s", "q", "q_equiv", "decision", "expected", "confidence", "mass")


@pytest.fixture(scope="module")
def jet():
    import candidate_answer_scoring_gb300 as jet
    jet.load()
    return jet


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def padded_source(wl, seed, L=None):
    """Right-padded [B, L, d] source: row i of the workload sits at the last
    valid position of sequence i; every other position holds unrelated rows."""
    rng = np.random.default_rng(seed)
    N, d = wl.N, wl.d
    L = L or 9
    lengths = rng.integers(1, L + 1, size=N)
    src = wk.to_bf16_bits(rng.standard_normal((N * L, d)).astype(np.float32))
    row_index = (np.arange(N) * L + lengths - 1).astype(np.int32)
    src[row_index] = wl.H
    return src, row_index


def run_both(jet, wl, src, row_index, scorer=None):
    sc = scorer or jet.JetScorer(wl.d, wl.V, max(1, wl.N), max(1, wl.n_tok))
    W = dev(wl.W.view(np.int16)).view(torch.bfloat16)
    args = (dev(wl.tok_row), dev(wl.tok_ids), dev(wl.cand_offsets), dev(wl.set_offsets), dev(wl.kind), wl.T, wl.mode,
            None if wl.union_ids is None else dev(wl.union_ids))
    compact = sc.score_sets(dev(wl.H.view(np.int16)).view(torch.bfloat16), W, *args)
    gathered = sc.score_sets_gather(dev(src.view(np.int16)).view(torch.bfloat16), dev(row_index), W, *args)
    torch.cuda.synchronize()
    return ({k: v.cpu().numpy() for k, v in compact.items()}, {k: v.cpu().numpy() for k, v in gathered.items()})


def assert_bitwise(a, b):
    for k in OUT:
        np.testing.assert_array_equal(a[k].view(np.uint32) if a[k].dtype == np.float32 else a[k],
                                      b[k].view(np.uint32) if b[k].dtype == np.float32 else b[k], err_msg=k)


@pytest.mark.parametrize("case", ["single-cta", "paired-ragged", "binary-256"])
def test_gather_full_matches_compact_and_oracle(jet, case):
    if case == "single-cta":          # N <= 128: the one-CTA head
        wl = wk.custom(128, 3000, 20, K=(2, 6), length=(1, 5), dup_prob=0.2, seed=61)
    elif case == "paired-ragged":     # N > 128, not a multiple of the 256-row pair tile
        wl = wk.custom(192, 2600, 70, K=(2, 8), length=(1, 4), dup_prob=0.2, seed=62)
    else:
        wl = wk.binary_batch(256, random_pairs=True, d=256, V=4000)
    src, row_index = padded_source(wl, 7)
    compact, gathered = run_both(jet, wl, src, row_index)
    assert_bitwise(compact, gathered)
    compare(wl, gathered, oracle.score_workload(wl))


def test_gather_restricted_matches_compact_and_oracle(jet):
    base = wk.binary_batch(200, random_pairs=True, d=256, V=3000)
    wl = wk.binary_restricted(base=base)
    src, row_index = padded_source(wl, 8, L=5)
    compact, gathered = run_both(jet, wl, src, row_index)
    assert_bitwise(compact, gathered)
    compare(wl, gathered, oracle.score_workload(wl))


def test_gather_repeated_source_rows(jet):
    """Several problem rows may read the same source row."""
    wl = wk.custom(64, 900, 12, K=(2, 5), length=(1, 3), seed=63)
    rng = np.random.default_rng(3)
    src = wk.to_bf16_bits(rng.standard_normal((5, wl.d)).astype(np.float32))
    row_index = rng.integers(0, 5, size=wl.N).astype(np.int32)
    H = src[row_index]
    wl2 = wk.Workload(wl.name + "-rep", wl.d, wl.V, H, wl.W, wl.tok_row, wl.tok_ids, wl.cand_offsets,
                      wl.set_offsets, wl.kind, wl.T, wl.mode, wl.union_ids, dict(wl.info))
    compact, gathered = run_both(jet, wl2, src, row_index)
    assert_bitwise(compact, gathered)
    compare(wl2, gathered, oracle.score_workload(wl2))


def test_gather_rejects_bad_indices(jet):
    import candidate_answer_scoring_gb300 as j
    wl = wk.custom(64, 700, 8, K=(2, 4), length=(1, 3), seed=64)
    rest = wk.binary_restricted(base=wk.binary_batch(16, random_pairs=True, d=64, V=700))
    sc = j.JetScorer(64, 700, max(wl.N, rest.N), max(wl.n_tok, rest.n_tok))
    for w in (wl, rest):
        src, row_index = padded_source(w, 9)
        W = dev(w.W.view(np.int16)).view(torch.bfloat16)
        args = (dev(w.tok_row), dev(w.tok_ids), dev(w.cand_offsets), dev(w.set_offsets), dev(w.kind), w.T, w.mode,
                None if w.union_ids is None else dev(w.union_ids))
        S = dev(src.view(np.int16)).view(torch.bfloat16)
        for bad in (src.shape[0], -1):
            ri = row_index.copy()
            ri[w.N // 2] = bad
            with pytest.raises(j.JetError) as e:
                sc.score_sets_gather(S, dev(ri), W, *args)
            assert e.value.status == -2
        out = sc.score_sets_gather(S, dev(row_index), W, *args)      # the context still works
        torch.cuda.synchronize()
        compare(w, {k: v.cpu().numpy() for k, v in out.items()}, oracle.score_workload(w))


def test_bound_gather_call_matches_gather(jet):
    """bind_gather_call marshals once; each call() is the bare asynchronous
    gather call, bit-identical to score_sets_gather."""
    wl = wk.binary_batch(n_questions=200, random_pairs=True, d=128, V=1500)
    src, row_index = padded_source(wl, 5, L=8)
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    args = (dev(src.view(np.int16)).view(torch.bfloat16), dev(row_index), dev(wl.W.view(np.int16)).view(torch.bfloat16),
            dev(wl.tok_row), dev(wl.tok_ids), dev(wl.cand_offsets), dev(wl.set_offsets), dev(wl.kind), wl.T)
    ref = sc.score_sets_gather(*args)
    call, out = sc.bind_gather_call(*args)
    call()
    assert sc.sync_status() == 0
    assert_bitwise({k: v.cpu().numpy() for k, v in out.items()}, {k: v.cpu().numpy() for k, v in ref.items()})
