"""Seeded random configurations against the oracle: hidden sizes, vocabulary
sizes (ragged against the 256-column tiles), set counts and sizes, candidate
lengths, kinds, duplicate rates, temperatures and row layouts in full mode;
unions of 1 to 150 codes (one to five 32-code groups of the restricted head)
and of 192 to 4096 codes (the tcgen05 head over the staged union) in
restricted mode.  Every case is fixed by its seed, so a failure reproduces."""
import numpy as np
import pytest

import oracle
import workloads as wk
from parity import check_duplicates, compare
from test_gpu_parity import run_gpu

pytestmark = pytest.mark.gpu

D_CHOICES = (64, 128, 192, 256, 512, 1024)
T_CHOICES = (0.5, 1.0, 2.179, 5.0)


@pytest.fixture(scope="module")
def jet():
    import candidate_answer_scoring_gb300 as jet
    jet.load()
    return jet


def full_case(seed):
    rng = np.random.default_rng(1000 + seed)
    d = int(rng.choice(D_CHOICES))
    V = int(rng.integers(50, 5000))
    n_sets = int(rng.integers(1, 60))
    k_hi = int(rng.integers(1, 12))
    len_hi = int(rng.integers(1, 7))
    kinds = tuple(int(k) for k in rng.choice(3, size=int(rng.integers(1, 4)), replace=False))
    row_mode = "per_token" if rng.random() < 0.6 else "per_key"
    peak = (0.3, 0.9) if rng.random() < 0.4 else None
    return wk.custom(d, V, n_sets, K=(1, max(1, k_hi)), length=(1, len_hi), kinds=kinds, row_mode=row_mode,
                     peak=peak, dup_prob=float(rng.uniform(0, 0.4)), T=float(rng.choice(T_CHOICES)),
                     seed=5000 + seed)


def restricted_case(seed):
    rng = np.random.default_rng(2000 + seed)
    d = int(rng.choice(D_CHOICES))
    V = int(rng.integers(200, 6000))
    n_union = int(rng.integers(1, 151))
    union = rng.choice(V, size=n_union, replace=False).astype(np.int32)
    sets = []
    for _ in range(int(rng.integers(1, 50))):
        K = int(rng.integers(1, min(n_union, 10) + 1))
        codes = rng.choice(union, size=K, replace=False)
        if K > 1 and rng.random() < 0.3:
            codes[-1] = codes[0]                    # a duplicated code within the set
        sets.append(wk._SetSpec(wk.KIND_CHOICE, [(int(t),) for t in codes]))
    T = float(rng.choice(T_CHOICES))
    W = wk.gen_W(7000 + seed, V, d)
    wl = wk._build(f"fuzz-restricted-{seed}", 7000 + seed, d, V, W, sets, T, row_mode="per_key")
    return wl.with_mode(wk.MODE_RESTRICTED, T, union)


def restricted_union_case(seed):
    """Unions the tcgen05 head serves: 192 to 4096 codes (ragged against the
    256-column tiles), sets of up to 40 codes with duplicates, rows shared by
    a set's codes."""
    rng = np.random.default_rng(3000 + seed)
    d = int(rng.choice(D_CHOICES))
    n_union = int(rng.integers(192, 4097))
    V = int(rng.integers(n_union + 1, n_union + 6000))
    union = rng.choice(V, size=n_union, replace=False).astype(np.int32)
    sets = []
    for _ in range(int(rng.integers(1, 120))):
        K = int(rng.integers(1, 41))
        codes = rng.choice(union, size=K, replace=False)
        if K > 1 and rng.random() < 0.3:
            codes[-1] = codes[0]                    # a duplicated code within the set
        sets.append(wk._SetSpec(wk.KIND_CHOICE, [(int(t),) for t in codes]))
    T = float(rng.choice(T_CHOICES))
    W = wk.gen_W(8000 + seed, V, d)
    wl = wk._build(f"fuzz-union-{seed}", 8000 + seed, d, V, W, sets, T, row_mode="per_key")
    return wl.with_mode(wk.MODE_RESTRICTED, T, union)


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_restricted_large_union(jet, seed):
    wl = restricted_union_case(seed)
    gpu = run_gpu(jet, wl)
    compare(wl, gpu, oracle.score_workload(wl))
    check_duplicates(wl, gpu)


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_full(jet, seed):
    wl = full_case(seed)
    gpu = run_gpu(jet, wl)
    compare(wl, gpu, oracle.score_workload(wl))
    check_duplicates(wl, gpu)


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_restricted(jet, seed):
    wl = restricted_case(seed)
    gpu = run_gpu(jet, wl)
    compare(wl, gpu, oracle.score_workload(wl))
    check_duplicates(wl, gpu)


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_score_tokens(jet, seed):
    """jet_score_tokens (one token per row) on random shapes against the oracle's
    per-token log-probabilities and row log-sum-exps."""
    import torch
    rng = np.random.default_rng(3000 + seed)
    d = int(rng.choice(D_CHOICES))
    V = int(rng.integers(20, 6000))
    n = int(rng.integers(1, 700))
    W = wk.gen_W(8000 + seed, V, d)
    H = wk.to_bf16_bits((rng.normal(size=(n, d)) * rng.uniform(0.5, 3.0)).astype(np.float32))
    tok = rng.integers(0, V, size=n).astype(np.int32)
    sc = jet.JetScorer(d, V, n, n)
    logp, lse = sc.score_tokens(_dev(H.view(np.int16)).view(torch.bfloat16), _dev(W.view(np.int16)).view(torch.bfloat16),
                                _dev(tok), want_lse=True)
    torch.cuda.synchronize()
    ref_lp, ref_lse = oracle.score_tokens(H, W, np.arange(n, dtype=np.int32), tok)
    assert np.abs(logp.cpu().numpy() - ref_lp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 2e-3


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_gather_rows(jet, seed):
    """jet_score_sets_gather: the problem rows scattered at random positions of a
    larger source array (padding rows between them hold other values); results
    equal the compact call's bit for bit, full or restricted."""
    import torch
    restricted = seed % 3 == 2
    wl = restricted_case(seed) if restricted else full_case(100 + seed)
    rng = np.random.default_rng(4000 + seed)
    n_src = wl.N + int(rng.integers(0, 3 * wl.N + 2))
    pos = np.sort(rng.choice(n_src, size=wl.N, replace=False)).astype(np.int32)
    src = wk.to_bf16_bits(rng.normal(size=(n_src, wl.d)).astype(np.float32))
    src[pos] = wl.H
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    W = _dev(wl.W.view(np.int16)).view(torch.bfloat16)
    rest = (_dev(wl.tok_row), _dev(wl.tok_ids), _dev(wl.cand_offsets), _dev(wl.set_offsets), _dev(wl.kind), wl.T,
            wl.mode, None if wl.union_ids is None else _dev(wl.union_ids))
    got = sc.score_sets_gather(_dev(src.view(np.int16)).view(torch.bfloat16), _dev(pos), W, *rest)
    got = {k: v.cpu().numpy() for k, v in got.items()}
    compact = sc.score_sets(_dev(wl.H.view(np.int16)).view(torch.bfloat16), W, *rest)
    for k, v in compact.items():
        assert np.array_equal(got[k].view(np.uint32), v.cpu().numpy().view(np.uint32)), k
