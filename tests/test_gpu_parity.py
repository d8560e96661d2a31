"""GPU parity: the CUDA path against the fp64 oracle on the same seeded inputs,
through the C ABI (via the thin ctypes binding).

Small and mid-size cases are compared element by element; they span several
row and vocabulary tiles with ragged tails.  The five named workloads run at
full size in the launch configuration the benchmark times, and are compared
on sampled sets (the oracle computes only those) plus properties that hold at
any size.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads as wk
from parity import check_duplicates, compare, subset

pytestmark = pytest.mark.gpu

OUT_KEYS = ("logp", "lse", "s", "q", "q_equiv", "decision", "expected", "confidence", "mass")


@pytest.fixture(scope="module")
def jet():
    import candidate_answer_scoring_gb300 as jet
    jet.load()
    return jet


def to_dev(wl, dev="cuda:0"):
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(dt) if dt is torch.bfloat16 \
        else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d = dict(H=t(wl.H.view(np.int16), torch.bfloat16), W=t(wl.W.view(np.int16), torch.bfloat16),
             tok_row=t(wl.tok_row, None), tok_ids=t(wl.tok_ids, None), cand_offsets=t(wl.cand_offsets, None),
             set_offsets=t(wl.set_offsets, None), kind=t(wl.kind, None))
    d["union_ids"] = None if wl.union_ids is None else t(wl.union_ids, None)
    return d


def run_gpu(jet, wl, scorer=None, dev_inputs=None):
    if scorer is None:
        scorer = jet.JetScorer(wl.d, wl.V, max(1, wl.N), max(1, wl.n_tok))
    x = dev_inputs if dev_inputs is not None else to_dev(wl)
    out = scorer.score_sets(x["H"], x["W"], x["tok_row"], x["tok_ids"], x["cand_offsets"], x["set_offsets"],
                            x["kind"], wl.T, wl.mode, x["union_ids"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


# ---------------------------------------------------------------------------
# element-by-element parity on small / mid-size cases
# ---------------------------------------------------------------------------
def test_tiny_workload(jet):
    wl = wk.tiny()
    gpu = run_gpu(jet, wl)
    orc = oracle.score_workload(wl)
    compare(wl, gpu, orc)
    assert check_duplicates(wl, gpu) >= 1


CASES = {
    # name: (d, V, n_sets, kwargs)
    "ragged-rows-and-vocab": (128, 1000, 40, dict(K=(2, 8), length=(1, 6))),
    "shared-rows-multitile": (256, 3000, 60, dict(K=(2, 10), length=(1, 5), row_mode="per_key")),
    "peaked-temperature": (192, 2051, 30, dict(K=(2, 12), length=(1, 8), peak=(0.9, 0.99), T=wk.T_FITTED)),
    "vocab-below-one-tile": (64, 7, 25, dict(K=(2, 5), length=(1, 3), dup_prob=0.3)),
    "vocab-exact-tiles": (64, 2048, 50, dict(K=(1, 6), length=(1, 4), kinds=(0,))),
    "long-k": (128, 1500, 6, dict(K=(60, 70), length=(1, 3), kinds=(0,))),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_custom_parity(jet, case):
    d, V, n_sets, kw = CASES[case]
    wl = wk.custom(d, V, n_sets, seed=zlib.crc32(case.encode()) % 1000, **kw)
    gpu = run_gpu(jet, wl)
    orc = oracle.score_workload(wl)
    compare(wl, gpu, orc)
    check_duplicates(wl, gpu)


def test_score_tokens(jet):
    rng = np.random.default_rng(0)
    d, V, n = 128, 5000, 700
    W = wk.gen_W(99, V, d)
    H = wk.to_bf16_bits(rng.normal(size=(n, d)).astype(np.float32))
    tok = rng.integers(0, V, size=n).astype(np.int32)
    sc = jet.JetScorer(d, V, n, n)
    Hd = torch.from_numpy(H.view(np.int16)).cuda().view(torch.bfloat16)
    Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    logp, lse = sc.score_tokens(Hd, Wd, torch.from_numpy(tok).cuda(), want_lse=True)
    ref_lp, ref_lse = oracle.score_tokens(H, W, np.arange(n, dtype=np.int32), tok)
    assert np.abs(logp.cpu().numpy() - ref_lp).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 2e-3


def test_restricted_parity(jet):
    base = wk.binary_batch(n_questions=40, random_pairs=True, d=128, V=3000)
    wl = wk.binary_restricted(base=base)
    gpu = run_gpu(jet, wl)
    orc = oracle.score_workload(wl)
    compare(wl, gpu, orc)


def test_restricted_union_larger_than_one_chunk(jet):
    """Single-token sets over a 600-code union, d=1024: the restricted head
    runs 19 groups of 32 codes (the last one ragged); rows shared by all codes
    of a set."""
    rng = np.random.default_rng(5)
    d, V = 1024, 20000
    union = rng.choice(V, size=600, replace=False).astype(np.int32)
    sets = []
    for _ in range(50):
        K = int(rng.integers(2, 9))
        sets.append(wk._SetSpec(wk.KIND_CHOICE, [(int(t),) for t in rng.choice(union, size=K, replace=False)]))
    W = wk.gen_W(1234, V, d)
    wl = wk._build("restricted-600", 1234, d, V, W, sets, 1.5, row_mode="per_key")
    wl = wl.with_mode(wk.MODE_RESTRICTED, 1.5, union)
    gpu = run_gpu(jet, wl)
    orc = oracle.score_workload(wl)
    compare(wl, gpu, orc)


def test_restricted_without_union_logit_scratch(jet):
    """N x |U| above the context's union-logit scratch (max(128 max_rows, 2^20)
    floats): the set kernel recomputes each scored logit with the head's dot
    product.  300 rows (one per set) x a 4000-code union, d=128."""
    rng = np.random.default_rng(17)
    d, V, n_union = 128, 6000, 4000
    union = rng.choice(V, size=n_union, replace=False).astype(np.int32)
    sets = []
    for _ in range(300):
        K = int(rng.integers(2, 7))
        sets.append(wk._SetSpec(wk.KIND_CHOICE, [(int(t),) for t in rng.choice(union, size=K, replace=False)]))
    W = wk.gen_W(4321, V, d)
    wl = wk._build("restricted-4000", 4321, d, V, W, sets, 1.3, row_mode="per_key")
    wl = wl.with_mode(wk.MODE_RESTRICTED, 1.3, union)
    assert wl.N * n_union > max(128 * wl.N, 1 << 20)
    gpu = run_gpu(jet, wl)
    orc = oracle.score_workload(wl)
    compare(wl, gpu, orc)
    # the same sets through the scratch (a union cut to the codes in use) agree
    used = np.unique(wl.tok_ids).astype(np.int32)
    small = run_gpu(jet, wl.with_mode(wk.MODE_RESTRICTED, 1.3, used))
    orc_small = oracle.score_workload(wl.with_mode(wk.MODE_RESTRICTED, 1.3, used))
    compare(wl.with_mode(wk.MODE_RESTRICTED, 1.3, used), small, orc_small)


def test_restricted_wide_rows(jet):
    """d = 16384, 300 rows (a ragged last tile of 16): each of the restricted
    head's 16 warps takes 32 of the 512 chunks of d."""
    rng = np.random.default_rng(23)
    d, V = 16384, 700
    union = rng.choice(V, size=120, replace=False).astype(np.int32)
    sets = []
    for _ in range(300):
        K = int(rng.integers(2, 6))
        sets.append(wk._SetSpec(wk.KIND_CHOICE, [(int(t),) for t in rng.choice(union, size=K, replace=False)]))
    W = wk.gen_W(777, V, d)
    wl = wk._build("restricted-wide", 777, d, V, W, sets, 0.9, row_mode="per_key")
    wl = wl.with_mode(wk.MODE_RESTRICTED, 0.9, union)
    gpu = run_gpu(jet, wl)
    compare(wl, gpu, oracle.score_workload(wl))


def test_full_equals_restricted_when_union_is_vocab(jet):
    base = wk.binary_batch(n_questions=30, random_pairs=True, d=64, V=1500)
    full = run_gpu(jet, base)
    rest = run_gpu(jet, base.with_mode(wk.MODE_RESTRICTED, base.T, np.arange(1500, dtype=np.int32)))
    for k in ("logp", "s", "q", "expected", "confidence", "mass"):
        np.testing.assert_allclose(rest[k], full[k], atol=2e-5, rtol=1e-4)
    np.testing.assert_array_equal(rest["decision"], full["decision"])


def test_edge_cases(jet):
    # one row, one single-token candidate (K = 1)
    wl = wk.custom(64, 300, 1, K=(1, 1), length=(1, 1), kinds=(0,), seed=3)
    gpu = run_gpu(jet, wl)
    orc = oracle.score_workload(wl)
    compare(wl, gpu, orc)
    assert gpu["q"][0] == 1.0 and gpu["decision"][0] == 0 and gpu["confidence"][0] == 1.0
    # empty batch: nothing launched, status ok
    sc = jet.JetScorer(64, 300, 4, 4)
    x = to_dev(wl)
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    sc.score_sets(x["H"], x["W"], e, e, z, z, torch.empty(0, dtype=torch.uint8, device="cuda"), 1.0,
                  out={k: torch.empty(1, device="cuda") for k in ("s",)})
    # batch exactly at the workspace limit
    wl = wk.custom(64, 500, 12, K=(2, 4), length=(1, 3), seed=8)
    sc = jet.JetScorer(64, 500, wl.N, wl.n_tok)
    gpu = run_gpu(jet, wl, scorer=sc)
    compare(wl, gpu, oracle.score_workload(wl))


@pytest.mark.parametrize("case", ["vocab-below-one-tile", "one-token-vocab", "widest-rows", "single-code-union",
                                  "million-vocab"])
def test_shape_extremes(jet, case):
    """A vocabulary smaller than one 256-column tile (every column ragged), a
    vocabulary of one token (lse = z, so every logp is 0, every candidate
    scores 0 and each set's q is uniform), the widest rows the library accepts
    (d = 16384: 256 k-blocks per tile) through the full-vocabulary head with
    both head variants' row counts, and a restricted union of one code
    (lse_U = z, so logp = 0 and q = 1)."""
    if case == "vocab-below-one-tile":
        wls = [wk.custom(64, 100, 6, K=(1, 5), length=(1, 3), seed=91)]
    elif case == "one-token-vocab":
        sets = [wk._SetSpec(wk.KIND_CHOICE, [(0,), (0, 0), (0, 0, 0)]), wk._SetSpec(wk.KIND_BINARY, [(0,), (0,)]),
                wk._SetSpec(wk.KIND_ORDINAL, [(0,)] * 5), wk._SetSpec(wk.KIND_CHOICE, [(0,)])]
        wls = [wk._build("one-token-vocab", 55, 64, 1, wk.gen_W(55, 1, 64), sets, 1.0, row_mode="per_token")]
        single = wk._build("one-token-vocab-single", 56, 64, 1, wk.gen_W(56, 1, 64), sets[1:], 1.0)
        wls += [single, single.with_mode(wk.MODE_RESTRICTED, 2.0, np.zeros(1, dtype=np.int32))]
    elif case == "widest-rows":
        wls = [wk.custom(16384, 700, 4, K=(2, 4), length=(1, 2), seed=92),      # N <= 128: one-CTA head
               wk.binary_batch(150, random_pairs=True, d=16384, V=600)]          # N > 128: paired head
    elif case == "million-vocab":     # 4097 vocabulary tiles, the last ragged; ids near the top of the range
        V = 1048583
        wls = [wk.custom(64, V, 8, K=(2, 5), length=(1, 3), seed=94),                  # one-CTA head
               wk.binary_batch(140, random_pairs=True, d=64, V=V)]                     # paired head
        top = np.arange(V - 40, V, dtype=np.int32)
        rest = wk.binary_batch(30, random_pairs=True, d=64, V=V)
        wls.append(rest.with_mode(wk.MODE_RESTRICTED, 2.179, np.unique(np.concatenate([rest.tok_ids, top]))))
    else:
        base = wk.custom(64, 400, 5, K=(1, 1), length=(1, 1), kinds=(0,), seed=93)
        wls = [base.with_mode(wk.MODE_RESTRICTED, 1.0, np.unique(base.tok_ids)[:1])]
        wls[0].tok_ids[:] = wls[0].union_ids[0]
    for wl in wls:
        gpu = run_gpu(jet, wl)
        compare(wl, gpu, oracle.score_workload(wl))
        if case == "single-code-union":
            assert np.all(gpu["logp"] == 0.0) and np.all(gpu["q"] == 1.0)
        if case == "one-token-vocab":
            assert np.abs(gpu["logp"]).max() <= 1e-6
            np.testing.assert_array_equal(gpu["decision"], 0)       # all tied: the first candidate


@pytest.mark.parametrize("T", [0.02, 0.25, 50.0])
def test_temperature_extremes(jet, T):
    """Set rules at temperatures from one-hot (0.02: most q underflow to 0) to
    flat (50); mass stays at T = 1.

    T = 50 meets the standard tolerances.  Below T = 1 the set softmax
    magnifies the score error: with da = max |s_gpu - s_oracle| / T over a set
    of K, the softmax Jacobian bounds |dq_i| by da / 2, |d expected| by
    (K - 1) da, |d q_equiv| by da (a group's q changes by at most the total
    variation, da), and |d confidence| by 2 da (1 + ln K) / ln K
    (d(-q ln q) = -(1 + ln q) dq with dq_i = q_i (da_i - <da>)).  Those bounds
    replace the fixed ones; decisions stay exact wherever the oracle's margin
    exceeds 1e-3."""
    wl = wk.custom(128, 2300, 60, K=(2, 8), length=(1, 4), dup_prob=0.15, T=T, seed=31)
    gpu = run_gpu(jet, wl)
    orc = oracle.score_workload(wl)
    if T > 1:
        compare(wl, gpu, orc)
        return
    from parity import LOGP_ATOL, MARGIN, MASS_ATOL
    assert np.abs(gpu["logp"].astype(np.float64) - orc.logp).max() <= LOGP_ATOL
    lens = np.diff(wl.cand_offsets)
    ds = np.abs(gpu["s"].astype(np.float64) - orc.s)
    assert np.all(ds <= LOGP_ATOL * lens)
    assert np.abs(gpu["mass"].astype(np.float64) - orc.mass).max() <= MASS_ATOL
    for k in range(wl.n_sets):
        c0, c1 = wl.set_offsets[k], wl.set_offsets[k + 1]
        K = c1 - c0
        da = ds[c0:c1].max() / T + 1e-5          # + fp32 rounding of q itself
        assert np.abs(gpu["q"][c0:c1] - orc.q[c0:c1]).max() <= da / 2, k
        assert np.abs(gpu["q_equiv"][c0:c1] - orc.q_equiv[c0:c1]).max() <= da, k
        assert abs(gpu["expected"][k] - orc.expected[k]) <= (K - 1) * da, k
        if K > 1:
            assert abs(gpu["confidence"][k] - orc.confidence[k]) <= 2 * da * (1 + np.log(K)) / np.log(K), k
        if orc.margin[k] > MARGIN:
            assert gpu["decision"][k] == orc.decision[k], k
    assert np.all(np.isfinite(gpu["q"])) and np.all(np.abs(gpu["q"].reshape(-1)).max() <= 1.0)


def test_repeat_calls_are_bitwise_deterministic(jet):
    wl = wk.custom(128, 2500, 30, K=(2, 8), length=(1, 5), seed=21)
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    x = to_dev(wl)
    a = run_gpu(jet, wl, sc, x)
    b = run_gpu(jet, wl, sc, x)
    for k in OUT_KEYS:
        assert np.array_equal(a[k].view(np.uint32), b[k].view(np.uint32)), k


def test_host_entry_matches_device_entry(jet):
    wl = wk.custom(128, 1200, 20, K=(2, 6), length=(1, 4), seed=17)
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    x = to_dev(wl)
    dev = run_gpu(jet, wl, sc, x)
    cpu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    host = sc.score_sets_host(cpu(wl.H.view(np.int16)).view(torch.bfloat16), x["W"], cpu(wl.tok_row),
                              cpu(wl.tok_ids), cpu(wl.cand_offsets), cpu(wl.set_offsets), cpu(wl.kind), wl.T)
    for k in OUT_KEYS:
        assert np.array_equal(host[k].numpy().view(np.uint32), dev[k].view(np.uint32)), k


def test_bound_host_call_matches_host_entry(jet):
    """bind_host_call marshals once; each call() is the bare C call on the
    same buffers, so new contents written into them are scored (here the
    new hidden rows copied over the first batch's)."""
    import dataclasses
    a = wk.custom(128, 1200, 20, K=(2, 6), length=(1, 4), seed=17)
    rng = np.random.default_rng(18)
    b = dataclasses.replace(a, H=wk.to_bf16_bits(rng.normal(size=a.H.shape).astype(np.float32)))
    sc = jet.JetScorer(a.d, a.V, a.N, a.n_tok)
    W = to_dev(a)["W"]
    cpu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    H = cpu(a.H.view(np.int16)).view(torch.bfloat16)
    args = (H, W, cpu(a.tok_row), cpu(a.tok_ids), cpu(a.cand_offsets), cpu(a.set_offsets), cpu(a.kind), a.T)
    call, out = sc.bind_host_call(*args)
    ref = sc.score_sets_host(*args)
    call()
    for k in OUT_KEYS:
        assert np.array_equal(out[k].numpy().view(np.uint32), ref[k].numpy().view(np.uint32)), k
    H.copy_(torch.from_numpy(b.H.view(np.int16)).view(torch.bfloat16))   # new rows, same shapes
    call()
    got = {k: v.numpy() for k, v in out.items()}
    compare(b, got, oracle.score_workload(b))


def test_pipelined_host_calls_match_host_entry(jet):
    """jet_score_sets_host_async: six calls alternating two batches (two
    staging slots, so each slot is reused while the other call's kernels may
    run), each into its own pinned outputs, equal the synchronous host entry
    bit for bit after one jet_host_wait; a device-side rejection among them is
    returned by the wait, and the context works afterwards."""
    import dataclasses
    a = wk.custom(128, 1200, 20, K=(2, 6), length=(1, 4), seed=23)
    rng = np.random.default_rng(24)
    b = dataclasses.replace(a, H=wk.to_bf16_bits(rng.normal(size=a.H.shape).astype(np.float32)))
    sc = jet.JetScorer(a.d, a.V, a.N, a.n_tok)
    W = to_dev(a)["W"]
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    batches = []
    for wl in (a, b):
        args = (pin(wl.H.view(np.int16)).view(torch.bfloat16), W, pin(wl.tok_row), pin(wl.tok_ids),
                pin(wl.cand_offsets), pin(wl.set_offsets), pin(wl.kind), wl.T)
        batches.append((args, sc.score_sets_host(*args)))
    calls = []
    for i in range(6):
        args, _ = batches[i % 2]
        calls.append(sc.bind_host_call(*args, pipelined=True))
    for call, _ in calls:
        call()
    assert sc.host_wait() == 0
    for i, (_, out) in enumerate(calls):
        ref = batches[i % 2][1]
        for k in OUT_KEYS:
            assert np.array_equal(out[k].numpy().view(np.uint32), ref[k].numpy().view(np.uint32)), (i, k)
    # a rejected call among valid ones
    args, _ = batches[0]
    bad_ids = args[3].clone().pin_memory()
    bad_ids[1] = a.V
    bad, _ = sc.bind_host_call(args[0], W, args[2], bad_ids, *args[4:], pipelined=True)
    calls[0][0]()
    bad()
    calls[1][0]()
    assert sc.host_wait() == -2
    calls[2][0]()
    calls[3][0]()
    assert sc.host_wait() == 0
    for k in OUT_KEYS:
        assert np.array_equal(calls[3][1][k].numpy().view(np.uint32), batches[1][1][k].numpy().view(np.uint32)), k


def test_pipelined_host_calls_past_the_status_ring(jet):
    """More pipelined calls between two waits than the context keeps status
    words for (4096): the call past the ring waits for the earlier ones and
    keeps their first rejection, which the wait still returns; a clean run of
    the same length returns JET_OK and the last call's outputs equal the
    synchronous host entry bit for bit."""
    a = wk.custom(64, 300, 6, K=(2, 3), length=(1, 2), seed=31)
    sc = jet.JetScorer(a.d, a.V, a.N, a.n_tok)
    W = to_dev(a)["W"]
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    args = (pin(a.H.view(np.int16)).view(torch.bfloat16), W, pin(a.tok_row), pin(a.tok_ids),
            pin(a.cand_offsets), pin(a.set_offsets), pin(a.kind), a.T)
    ref = sc.score_sets_host(*args)
    good, out = sc.bind_host_call(*args, pipelined=True)
    bad_ids = args[3].clone().pin_memory()
    bad_ids[0] = a.V
    bad, _ = sc.bind_host_call(args[0], W, args[2], bad_ids, *args[4:], pipelined=True)
    n = 4096 + 5
    for i in range(n):
        (bad if i == 3 else good)()
    assert sc.host_wait() == -2                # JET_ERR_TOKEN_RANGE, from before the ring filled
    for _ in range(n):
        good()
    assert sc.host_wait() == 0
    for k in OUT_KEYS:
        assert np.array_equal(out[k].numpy().view(np.uint32), ref[k].numpy().view(np.uint32)), k


def test_bound_device_call_matches_score_sets(jet):
    """bind_call marshals once; each call() is the bare asynchronous C call on
    the same device buffers: bit-identical to score_sets in full and
    restricted mode, new contents written into the inputs are scored, and a
    device-side rejection surfaces through the synchronous form."""
    import dataclasses
    a = wk.custom(128, 1200, 20, K=(2, 6), length=(1, 4), seed=19)
    r = wk.binary_restricted(base=wk.binary_batch(n_questions=60, random_pairs=True, d=128, V=1200))
    for wl in (a, r):
        sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
        x = to_dev(wl)
        args = (x["H"], x["W"], x["tok_row"], x["tok_ids"], x["cand_offsets"], x["set_offsets"], x["kind"], wl.T,
                wl.mode, x["union_ids"])
        call, out = sc.bind_call(*args)
        ref = sc.score_sets(*args)
        call()
        assert sc.sync_status() == 0
        for k in OUT_KEYS:
            assert torch.equal(out[k].view(torch.int32), ref[k].view(torch.int32)), k
    rng = np.random.default_rng(20)
    b = dataclasses.replace(a, H=wk.to_bf16_bits(rng.normal(size=a.H.shape).astype(np.float32)))
    sc = jet.JetScorer(a.d, a.V, a.N, a.n_tok)
    x = to_dev(a)
    call, out = sc.bind_call(x["H"], x["W"], x["tok_row"], x["tok_ids"], x["cand_offsets"], x["set_offsets"],
                             x["kind"], a.T, sync=True)
    x["H"].copy_(to_dev(b)["H"])   # new rows, same shapes
    call()
    compare(b, {k: v.cpu().numpy() for k, v in out.items()}, oracle.score_workload(b))
    x["tok_ids"][0] = a.V          # rejected by the pre-pass
    with pytest.raises(jet.JetError) as e:
        call()
    assert e.value.status == -2


def test_host_entry_restricted_subset_and_errors(jet):
    """The host entry packs the index arrays into one copy in and the requested
    outputs (behind the status words) into one copy out: restricted mode, a
    subset of outputs, and an error status all come back through it."""
    import candidate_answer_scoring_gb300 as j
    base = wk.binary_batch(n_questions=48, random_pairs=True, d=128, V=2000)
    wl = wk.binary_restricted(base=base)
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    x = to_dev(wl)
    dev = run_gpu(jet, wl, sc, x)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    args = [pin(wl.H.view(np.int16)).view(torch.bfloat16), x["W"], pin(wl.tok_row), pin(wl.tok_ids),
            pin(wl.cand_offsets), pin(wl.set_offsets), pin(wl.kind), wl.T, wl.mode, pin(wl.union_ids)]
    want = {"q": torch.full((wl.n_cand,), -7.0), "decision": torch.full((wl.n_sets,), -7, dtype=torch.int32),
            "mass": torch.full((wl.n_sets,), -7.0)}
    host = sc.score_sets_host(*args, out=want)
    for k in want:
        assert np.array_equal(host[k].numpy().view(np.uint32), dev[k].view(np.uint32)), k
    bad = wl.tok_ids.copy()
    bad[5] = wl.V
    args[3] = pin(bad)
    with pytest.raises(j.JetError) as e:
        sc.score_sets_host(*args, out=want)
    assert e.value.status == -2
    args[3] = pin(wl.tok_ids)
    host = sc.score_sets_host(*args)                                      # the context still works
    compare(wl, {k: v.numpy() for k, v in host.items()}, oracle.score_workload(wl))


def test_outputs_leave_guard_bands_untouched(jet):
    wl = wk.custom(64, 900, 15, K=(2, 6), length=(1, 4), seed=4)
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    x = to_dev(wl)
    G = 64
    sizes = dict(logp=wl.n_tok, lse=wl.N, s=wl.n_cand, q=wl.n_cand, q_equiv=wl.n_cand, decision=wl.n_sets,
                 expected=wl.n_sets, confidence=wl.n_sets, mass=wl.n_sets)
    bufs, out = {}, {}
    for k, n in sizes.items():
        dt = torch.int32 if k == "decision" else torch.float32
        b = torch.full((n + 2 * G,), -7777, dtype=dt, device="cuda")
        bufs[k] = b
        out[k] = b[G:G + n]
    sc.score_sets(x["H"], x["W"], x["tok_row"], x["tok_ids"], x["cand_offsets"], x["set_offsets"], x["kind"],
                  wl.T, out=out)
    torch.cuda.synchronize()
    for k, b in bufs.items():
        h = b.cpu().numpy()
        assert np.all(h[:G] == -7777) and np.all(h[-G:] == -7777), f"{k}: guard band overwritten"
        assert not np.any(h[G:-G] == -7777), f"{k}: output element not written"


# ---------------------------------------------------------------------------
# the five named workloads at full size (launch configuration of the bench)
# ---------------------------------------------------------------------------
def _full_size(jet, wl, sample_sets, threads=0):
    gpu = run_gpu(jet, wl)
    sub, set_ids, cands, toks, rows = subset(wl, sample_sets)
    orc = oracle.score_workload(sub, threads=threads)
    stats = compare(wl, gpu, orc, set_ids, cands, toks, rows)
    check_duplicates(wl, gpu)
    # properties at full size
    for k in range(wl.n_sets):
        c0, c1 = wl.set_offsets[k], wl.set_offsets[k + 1]
        assert abs(gpu["q"][c0:c1].astype(np.float64).sum() - 1.0) < 1e-5
    assert np.all(np.isfinite(gpu["logp"])) and np.all(gpu["logp"] <= 1e-6)
    s_from_logp = np.add.reduceat(gpu["logp"].astype(np.float64), wl.cand_offsets[:-1])
    np.testing.assert_allclose(gpu["s"], s_from_logp, rtol=1e-5, atol=1e-4)
    return gpu, stats


def test_full_size_tiny(jet):
    wl = wk.tiny()
    _full_size(jet, wl, range(wl.n_sets))


def test_full_size_binary(jet):
    wl = wk.binary_batch()
    _full_size(jet, wl, [0, 1, 2, 77, 128, 200, 254, 255])
    rest = wk.binary_restricted(base=wl)
    _full_size(jet, rest, range(0, 256, 3))


def test_full_size_binary_random_pairs_restricted(jet):
    wl = wk.binary_restricted(random_pairs=True)
    _full_size(jet, wl, range(0, 256, 5))


def test_full_size_multitoken(jet):
    wl = wk.multi_token_choice()
    _full_size(jet, wl, [0, 63])


def test_full_size_wideschema(jet):
    wl = wk.wide_schema()
    sizes = np.diff(wl.set_offsets)
    pick = [int(np.argmin(sizes)), 1, 2, int(np.nonzero(wl.kind == wk.KIND_ORDINAL)[0][0])]
    _full_size(jet, wl, sorted(set(pick)))


def test_full_size_large(jet):
    wl = wk.large_choice()
    gpu = run_gpu(jet, wl)
    # sampled tokens: every 700th token's log-probability and its row's lse
    idx = np.arange(0, wl.n_tok, 700)
    want = np.zeros(wl.n_tok, np.uint8)
    want[idx] = 1
    lp, lse = oracle.score_tokens(wl.H, wl.W, wl.tok_row, wl.tok_ids, want=want)
    assert np.abs(gpu["logp"][idx] - lp[idx]).max() <= 2e-3
    rows = wl.tok_row[idx]
    assert np.abs(gpu["lse"][rows] - lse[rows]).max() <= 2e-3
    assert check_duplicates(wl, gpu) >= 16 * 3 - 16   # copies per request (a copy may repeat a copy)
    for k in range(wl.n_sets):
        c0, c1 = wl.set_offsets[k], wl.set_offsets[k + 1]
        assert abs(gpu["q"][c0:c1].astype(np.float64).sum() - 1.0) < 1e-5


# ---------------------------------------------------------------------------
# whole sets of the full-size workloads against stored oracle outputs
# (written by tests/golden/make_oracle_golden.py, which calls only the oracle)
# ---------------------------------------------------------------------------
GOLDEN_GEN = {"multitoken": wk.multi_token_choice, "wideschema": wk.wide_schema, "large": wk.large_choice}


@pytest.mark.parametrize("name", sorted(GOLDEN_GEN))
def test_full_size_against_stored_oracle_sets(jet, name):
    import json
    import os
    from types import SimpleNamespace
    path = os.path.join(os.path.dirname(__file__), "golden", f"oracle_{name}.json")
    g = json.load(open(path))
    wl = GOLDEN_GEN[name]()
    assert wl.checksum() == g["generator_checksum"], \
        "the seeded generator produced different inputs on this platform; stored oracle values do not apply"
    gpu = run_gpu(jet, wl)
    orc = SimpleNamespace(**{k: np.asarray(g[k], np.float64) for k in
                             ("logp", "lse", "s", "q", "q_equiv", "expected", "confidence", "mass", "margin")})
    orc.decision = np.asarray(g["decision"], np.int32)
    compare(wl, gpu, orc, np.asarray(g["sets"]), np.asarray(g["cands"]), np.asarray(g["tokens"]),
            np.asarray(g["rows"]))


def test_two_contexts_on_two_streams_run_concurrently(jet):
    """Contexts share no device state: a full-vocabulary batch on one stream
    and a restricted batch on another, enqueued alternately without waiting,
    give the same bits as each run alone."""
    full = wk.custom(128, 2600, 50, K=(2, 8), length=(1, 5), seed=61)
    rest = wk.binary_restricted(base=wk.binary_batch(n_questions=300, random_pairs=True, d=128, V=2600))
    jobs = []
    for wl in (full, rest):
        sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
        x = to_dev(wl)
        alone = run_gpu(jet, wl, sc, x)
        jobs.append((wl, sc, x, alone, torch.cuda.Stream()))
    outs = [None, None]
    for _ in range(5):
        for i, (wl, sc, x, alone, st) in enumerate(jobs):
            with torch.cuda.stream(st):
                outs[i] = sc.score_sets(x["H"], x["W"], x["tok_row"], x["tok_ids"], x["cand_offsets"],
                                        x["set_offsets"], x["kind"], wl.T, wl.mode, x.get("union_ids"), sync=False)
    torch.cuda.synchronize()
    for (wl, sc, x, alone, st), out in zip(jobs, outs):
        assert sc.sync_status() == 0
        for k in OUT_KEYS:
            got = out[k].cpu().numpy()
            assert np.array_equal(got.view(np.uint32), alone[k].view(np.uint32)), (wl.name, k)


def test_async_calls_capture_into_a_cuda_graph(jet):
    """score_sets(sync=False) records into a CUDA graph (host checks and
    tensor-map encoding happen at capture; every launch is a graph node), and
    each replay reproduces the stream-launched results bit for bit, full and
    restricted mode in one graph."""
    full = wk.custom(128, 2600, 40, K=(2, 8), length=(1, 5), seed=71)
    rest = wk.binary_restricted(base=wk.binary_batch(n_questions=100, random_pairs=True, d=128, V=2600))
    sc = jet.JetScorer(128, 2600, max(full.N, rest.N), max(full.n_tok, rest.n_tok))
    xs = [to_dev(full), to_dev(rest)]
    wls = [full, rest]
    outs = [sc.alloc_outputs(w.N, w.n_tok, w.n_cand, w.n_sets) for w in wls]
    st = torch.cuda.Stream()

    def step():
        for w, x, o in zip(wls, xs, outs):
            sc.score_sets(x["H"], x["W"], x["tok_row"], x["tok_ids"], x["cand_offsets"], x["set_offsets"],
                          x["kind"], w.T, w.mode, x["union_ids"], out=o, sync=False)

    with torch.cuda.stream(st):
        step()
    torch.cuda.synchronize()
    ref = [{k: v.clone() for k, v in o.items()} for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        step()
    for _ in range(2):
        for o in outs:
            for v in o.values():
                v.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert sc.sync_status() == 0
        for o, r in zip(outs, ref):
            for k in o:
                assert torch.equal(o[k], r[k]), k
    for w, o in zip(wls, outs):
        compare(w, {k: v.cpu().numpy() for k, v in o.items()}, oracle.score_workload(w))
