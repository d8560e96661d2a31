"""Tiled weights (jet_tile_weights / jet_set_weights_layout): the tiled copy
holds W's elements where the header says, and every path that reads W — the
full-vocabulary head (one-CTA and paired), the restricted head, and the
restricted set kernel's recomputation when the union logits do not fit the
scratch — gives the same bits as with row-major W."""
import os

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


def test_tiled_layout_matches_definition(jet):
    d, V = 192, 300                                   # V not a multiple of 128: padded rows are zero
    W = np.random.default_rng(1).integers(0, 65536, size=(V, d), dtype=np.uint16)
    sc = jet.JetScorer(d, V, 8, 8)
    Wt = sc.tile_weights(dev(W.view(np.int16)).view(torch.bfloat16), use=False)
    torch.cuda.synchronize()
    got = Wt.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
    Vp = -(-V // 128) * 128
    ref = np.zeros((Vp, d), np.uint16)
    ref[:V] = W
    ref = ref.reshape(Vp // 128, 128, d // 64, 64).transpose(0, 2, 1, 3).reshape(-1)
    assert got.size == ref.size
    np.testing.assert_array_equal(got, ref)


def scored(jet, wl, tiled, scorer_rows=None):
    sc = jet.JetScorer(wl.d, wl.V, scorer_rows or wl.N, wl.n_tok)
    W = dev(wl.W.view(np.int16)).view(torch.bfloat16)
    if tiled:
        W = sc.tile_weights(W)
    out = sc.score_sets(dev(wl.H.view(np.int16)).view(torch.bfloat16), W, dev(wl.tok_row), dev(wl.tok_ids),
                        dev(wl.cand_offsets), dev(wl.set_offsets), dev(wl.kind), wl.T, wl.mode,
                        None if wl.union_ids is None else dev(wl.union_ids))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def restricted_recompute_case():
    """N x |U| above the union-logit scratch: the set kernel recomputes logits."""
    rng = np.random.default_rng(29)
    d, V, n_union = 128, 5000, 4000
    union = rng.choice(V, size=n_union, replace=False).astype(np.int32)
    sets = [wk._SetSpec(wk.KIND_CHOICE, [(int(t),) for t in rng.choice(union, size=int(rng.integers(2, 6)),
                                                                            replace=False)]) for _ in range(300)]
    W = wk.gen_W(2929, V, d)
    wl = wk._build("tiled-recompute", 2929, d, V, W, sets, 1.1, row_mode="per_key")
    return wl.with_mode(wk.MODE_RESTRICTED, 1.1, union)


@pytest.mark.parametrize("case", ["one-cta", "paired", "restricted", "restricted-recompute"])
def test_tiled_weights_give_the_same_bits(jet, case):
    if case == "one-cta":
        wl = wk.custom(128, 1100, 20, K=(2, 6), length=(1, 4), seed=71)                # V not a multiple of 256
    elif case == "paired":
        wl = wk.binary_batch(200, random_pairs=True, d=256, V=2300)
    elif case == "restricted":
        wl = wk.binary_restricted(base=wk.binary_batch(100, random_pairs=True, d=256, V=2000))
    else:
        wl = restricted_recompute_case()
        assert wl.N * wl.union_ids.size > max(128 * wl.N, 1 << 20)
    a, b = scored(jet, wl, False), scored(jet, wl, True)
    for k in OUT:
        np.testing.assert_array_equal(a[k].view(np.uint32), b[k].view(np.uint32), err_msg=k)
    compare(wl, b, oracle.score_workload(wl))


def test_tiled_weights_reject_bad_arguments(jet):
    import ctypes as C
    import candidate_answer_scoring_gb300 as j
    sc = j.JetScorer(64, 200, 4, 4)
    with pytest.raises(j.JetError):
        sc.set_weights_layout(7)
    W = torch.zeros(200, 64, dtype=torch.bfloat16, device="cuda")
    p = C.c_void_p(W.data_ptr())
    assert sc.lib.jet_tile_weights(sc._h, p, p, None) == -1         # the tiled copy may not overlap W
    assert sc.lib.jet_tile_weights(sc._h, None, p, None) == -1


def test_tiled_weights_in_score_tokens_and_many_waves(jet):
    """The per-position entry, and a paired head running several waves of units
    in counter order, read the tiled copy with the same bits as row-major W."""
    import torch
    rng = np.random.default_rng(37)
    d, V, n = 128, 3000, 22000           # 86 paired row tiles, more than the 76 pairs: several waves
    W = wk.gen_W(3737, V, d)
    H = wk.to_bf16_bits(rng.normal(size=(n, d)).astype(np.float32))
    tok = rng.integers(0, V, size=n).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    Wd = dev(W.view(np.int16)).view(torch.bfloat16)
    Hd = dev(H.view(np.int16)).view(torch.bfloat16)
    sc = jet.JetScorer(d, V, n, n)
    info = sc.plan_info(n)
    if "JETSCORE_HEAD_PAIR" not in os.environ:   # a suite-wide variant override picks the head itself
        assert info["tile_rows"] == 256 and info["units"] > info["ctas"] // 2, info
    lp_row, lse_row = sc.score_tokens(Hd, Wd, dev(tok), want_lse=True)
    Wt = sc.tile_weights(Wd)
    lp_t, lse_t = sc.score_tokens(Hd, Wt, dev(tok), want_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(lp_row, lp_t) and torch.equal(lse_row, lse_t)
    ref_lp, ref_lse = oracle.score_tokens(H, W, np.arange(n, dtype=np.int32), tok)
    assert np.abs(lp_t.cpu().numpy() - ref_lp).max() <= 2e-3
    assert np.abs(lse_t.cpu().numpy() - ref_lse).max() <= 2e-3
