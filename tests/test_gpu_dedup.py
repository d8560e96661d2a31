"""jet_dedup_rows: distinct rows in order of first occurrence, exact remapping,
and unchanged scoring results on the compacted layout (the candidate-preserving
readout of FastJEV section 3.3)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wk
from parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jet():
    import candidate_answer_scoring_gb300 as jet
    jet.load()
    return jet


def first_occurrence(H):
    """Reference: index of the first row equal to each row, distinct rows in order."""
    seen, rep, order = {}, np.empty(H.shape[0], np.int64), []
    for r in range(H.shape[0]):
        key = H[r].tobytes()
        if key not in seen:
            seen[key] = len(order)
            order.append(r)
        rep[r] = seen[key]
    return rep, np.asarray(order, np.int64)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_dedup(jet, sc, wl):
    H = dev(wl.H.view(np.int16)).view(torch.bfloat16)
    Hu, tok_u, row_map = sc.dedup_rows(H, dev(wl.tok_row), want_row_map=True)
    torch.cuda.synchronize()
    return Hu.view(torch.int16).cpu().numpy().view(np.uint16), tok_u.cpu().numpy(), row_map.cpu().numpy()


@pytest.mark.parametrize("case", ["custom-dups", "multitoken", "no-dups", "all-equal", "large"])
def test_dedup_is_exact(jet, case):
    if case == "large":                 # 20026 rows of d = 4096: 20 rank tiles of 1024 rows
        wl = wk.large_choice()
    elif case == "custom-dups":
        wl = wk.custom(128, 900, 40, K=(2, 8), length=(1, 6), dup_prob=0.3, seed=31)
    elif case == "multitoken":
        wl = wk.multi_token_choice()
    elif case == "no-dups":
        wl = wk.binary_batch(64, d=128, V=500)
    else:
        wl = wk.custom(64, 300, 5, K=(2, 4), length=(1, 3), seed=2)
        wl.H[:] = wl.H[0]
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    Hu, tok_u, row_map = run_dedup(jet, sc, wl)
    rep, order = first_occurrence(wl.H)
    assert Hu.shape[0] == order.size
    np.testing.assert_array_equal(Hu, wl.H[order])                 # distinct rows, first-occurrence order
    np.testing.assert_array_equal(row_map, rep)
    np.testing.assert_array_equal(Hu[tok_u], wl.H[wl.tok_row])      # every token keeps its row's bytes
    if case == "no-dups":
        assert Hu.shape[0] == wl.N
    if case == "all-equal":
        assert Hu.shape[0] == 1


def test_scoring_on_deduplicated_rows_matches_oracle(jet):
    wl = wk.custom(192, 2500, 30, K=(2, 10), length=(1, 7), dup_prob=0.25, peak=(0.5, 0.9), T=1.7, seed=41)
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    Hu, tok_u, _ = run_dedup(jet, sc, wl)
    assert Hu.shape[0] < wl.N
    W = dev(wl.W.view(np.int16)).view(torch.bfloat16)
    out = sc.score_sets(dev(Hu.view(np.int16)).view(torch.bfloat16), W, dev(tok_u), dev(wl.tok_ids),
                        dev(wl.cand_offsets), dev(wl.set_offsets), dev(wl.kind), wl.T)
    torch.cuda.synchronize()
    gpu = {k: v.cpu().numpy() for k, v in out.items()}
    orc = oracle.score_workload(wl)          # the oracle scores the original, un-deduplicated layout
    rows = np.arange(wl.N)
    rep, _ = first_occurrence(wl.H)
    gpu["lse"] = gpu["lse"][rep]             # lse of each original row = lse of its distinct row
    compare(wl, gpu, orc, np.arange(wl.n_sets), np.arange(wl.n_cand), np.arange(wl.n_tok), rows)


def test_dedup_rejects_bad_input(jet):
    import candidate_answer_scoring_gb300 as j
    wl = wk.custom(64, 300, 6, K=(2, 4), length=(1, 3), seed=9)
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    H = dev(wl.H.view(np.int16)).view(torch.bfloat16)
    bad = wl.tok_row.copy()
    bad[2] = wl.N
    with pytest.raises(j.JetError) as e:
        sc.dedup_rows(H, dev(bad))
    assert e.value.status == -2
    with pytest.raises(j.JetError) as e:
        sc.dedup_rows(H, dev(wl.tok_row), H_unique=H)                # output overlaps input
    assert e.value.status == -1
    Hu, tok_u, _ = sc.dedup_rows(H, dev(wl.tok_row))                   # context still works
    assert Hu.shape[0] >= 1


@pytest.mark.parametrize("n", [1023, 1024, 1025, 2048, 2049])
def test_dedup_rank_tile_edges(jet, n):
    """Row counts at and around the rank pass's 1024-row tiles: the leading n
    rows of the multitoken batch (shared histories repeat rows across tiles),
    one token per row."""
    base = wk.multi_token_choice()
    H = np.ascontiguousarray(base.H[:n])
    sc = jet.JetScorer(base.d, base.V, n, n)
    Hd = dev(H.view(np.int16)).view(torch.bfloat16)
    Hu, tok_u, row_map = sc.dedup_rows(Hd, dev(np.arange(n, dtype=np.int32)), want_row_map=True)
    torch.cuda.synchronize()
    rep, order = first_occurrence(H)
    assert order.size < n                                  # the prefix holds duplicates
    np.testing.assert_array_equal(Hu.view(torch.int16).cpu().numpy().view(np.uint16), H[order])
    np.testing.assert_array_equal(row_map.cpu().numpy(), rep)
    np.testing.assert_array_equal(tok_u.cpu().numpy(), rep)


def test_dedup_without_tokens(jet):
    """No token rows to remap (n_tok = 0): rows are still compacted."""
    wl = wk.custom(64, 300, 5, K=(2, 4), length=(1, 3), dup_prob=0.5, seed=4)
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    H = dev(wl.H.view(np.int16)).view(torch.bfloat16)
    Hu, tok_u, row_map = sc.dedup_rows(H, torch.empty(0, dtype=torch.int32, device="cuda"), want_row_map=True)
    torch.cuda.synchronize()
    rep, order = first_occurrence(wl.H)
    np.testing.assert_array_equal(Hu.view(torch.int16).cpu().numpy().view(np.uint16), wl.H[order])
    np.testing.assert_array_equal(row_map.cpu().numpy(), rep)
    assert tok_u.numel() == 0


def test_bound_call_matches_dedup_rows(jet):
    """bind_dedup_rows marshals once; each call() is the bare C call: the same
    count and bit-identical rows and remapped token rows as dedup_rows, new
    contents written into H are deduplicated, and a bad token row raises."""
    wl = wk.custom(128, 900, 40, K=(2, 8), length=(1, 6), dup_prob=0.3, seed=33)
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    H = dev(wl.H.view(np.int16)).view(torch.bfloat16)
    tok_row = dev(wl.tok_row)
    Hu_ref, tok_ref, map_ref = sc.dedup_rows(H, tok_row, want_row_map=True)
    Hu, tok_u, row_map = torch.empty_like(H), torch.empty_like(tok_row), torch.empty(wl.N, dtype=torch.int32,
                                                                                       device="cuda")
    call = sc.bind_dedup_rows(H, tok_row, Hu, tok_u, row_map)
    for _ in range(2):
        n = call()
        assert n == Hu_ref.shape[0]
        assert torch.equal(Hu[:n].view(torch.int16), Hu_ref.view(torch.int16))
        assert torch.equal(tok_u, tok_ref) and torch.equal(row_map, map_ref)
    H.copy_(H[torch.zeros(wl.N, dtype=torch.long, device="cuda")])     # every row now equals row 0
    assert call() == 1 and torch.all(tok_u == 0)
    tok_row[0] = wl.N
    with pytest.raises(jet.JetError) as e:
        call()
    assert e.value.status == jet.JET_ERR_TOKEN_RANGE
