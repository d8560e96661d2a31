"""The C ABI's error conventions on the GPU: every status code is produced by a
bad argument made on the host (invalid sizes, temperature, mode, alignment) or
by an index the device pre-pass rejects; nothing faults, and the context keeps
working after each error."""
import numpy as np
import pytest
import torch

import workloads as wk

pytestmark = pytest.mark.gpu

OK, ARG, TOKEN, OFFSETS, MODE, UNION, WORKSPACE = 0, -1, -2, -3, -4, -5, -6


@pytest.fixture(scope="module")
def env():
    import candidate_answer_scoring_gb300 as jet
    wl = wk.custom(64, 500, 10, K=(2, 5), length=(1, 3), seed=13)
    rest = wk.binary_restricted(base=wk.binary_batch(8, random_pairs=True, d=64, V=500))
    sc = jet.JetScorer(64, 500, max(wl.N, rest.N) + 4, max(wl.n_tok, rest.n_tok) + 4)
    return jet, sc, wl, rest


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def args_of(wl, **over):
    a = dict(H=dev(wl.H.view(np.int16)).view(torch.bfloat16), W=dev(wl.W.view(np.int16)).view(torch.bfloat16),
             tok_row=dev(wl.tok_row), tok_ids=dev(wl.tok_ids), cand_offsets=dev(wl.cand_offsets),
             set_offsets=dev(wl.set_offsets), kind=dev(wl.kind), T=wl.T, mode=wl.mode,
             union_ids=None if wl.union_ids is None else dev(wl.union_ids))
    a.update(over)
    return a


def call(sc, a):
    import candidate_answer_scoring_gb300 as jet
    try:
        sc.score_sets(a["H"], a["W"], a["tok_row"], a["tok_ids"], a["cand_offsets"], a["set_offsets"], a["kind"],
                      a["T"], a["mode"], a["union_ids"])
        return OK
    except jet.JetError as e:
        return e.status


def still_works(sc, wl):
    a = args_of(wl)
    assert call(sc, a) == OK


def test_host_checks(env):
    jet, sc, wl, _ = env
    for T in (0.0, -1.0, float("nan"), float("inf")):
        assert call(sc, args_of(wl, T=T)) == ARG
    assert call(sc, args_of(wl, mode=7)) == MODE
    H = args_of(wl)["H"]
    flat = H.view(-1)
    mis = flat[1:1 + H.numel() - 64].view(H.shape[0] - 1, 64) if H.shape[0] > 1 else None
    if mis is not None:       # 2-byte offset: not 16-byte aligned
        a = args_of(wl, H=mis)
        assert call(sc, a) == ARG
    big = wk.custom(64, 500, 40, K=(4, 8), length=(2, 4), seed=2)
    assert call(sc, args_of(big)) == WORKSPACE
    still_works(sc, wl)


def test_token_and_row_ranges(env):
    jet, sc, wl, _ = env
    for bad in (wl.V, -1, 10 ** 9):
        t = wl.tok_ids.copy(); t[3] = bad
        assert call(sc, args_of(wl, tok_ids=dev(t))) == TOKEN
        still_works(sc, wl)
    r = wl.tok_row.copy(); r[0] = wl.N
    assert call(sc, args_of(wl, tok_row=dev(r))) == TOKEN
    r[0] = -5
    assert call(sc, args_of(wl, tok_row=dev(r))) == TOKEN
    still_works(sc, wl)


def test_offsets_and_kinds(env):
    jet, sc, wl, _ = env
    co = wl.cand_offsets.copy(); co[2], co[3] = co[3], co[2]           # not monotone
    assert call(sc, args_of(wl, cand_offsets=dev(co))) == OFFSETS
    co = wl.cand_offsets.copy(); co[1] = co[0]                            # empty candidate
    assert call(sc, args_of(wl, cand_offsets=dev(co))) == OFFSETS
    so = wl.set_offsets.copy(); so[-1] -= 1                               # sets do not cover candidates
    so2 = np.concatenate([so[:-1], [so[-1]]]).astype(np.int32)
    assert call(sc, args_of(wl, set_offsets=dev(so2))) == OFFSETS
    kd = wl.kind.copy(); kd[0] = 9
    assert call(sc, args_of(wl, kind=dev(kd))) == ARG
    # a set with K != 2 declared binary, and a one-candidate ordinal set
    Ks = np.diff(wl.set_offsets)
    k3 = int(np.nonzero(Ks != 2)[0][0])
    kd = wl.kind.copy(); kd[k3] = wk.KIND_BINARY
    assert call(sc, args_of(wl, kind=dev(kd))) == OFFSETS
    one = wk.custom(64, 500, 3, K=(1, 1), length=(1, 2), kinds=(0,), seed=5)
    kd = one.kind.copy(); kd[1] = wk.KIND_ORDINAL
    assert call(sc, args_of(one, kind=dev(kd))) == OFFSETS
    still_works(sc, wl)


def test_restricted_mode_checks(env):
    jet, sc, wl, rest = env
    assert call(sc, args_of(rest)) == OK
    u = rest.union_ids.copy(); u[1] = u[0]                                # repeated union id
    assert call(sc, args_of(rest, union_ids=dev(u))) == UNION
    u = rest.union_ids.copy(); u[5] = rest.V + 3                          # union id out of range
    assert call(sc, args_of(rest, union_ids=dev(u))) == TOKEN
    used = set(rest.tok_ids.tolist())
    missing = [i for i, x in enumerate(rest.union_ids) if int(x) in used][0]
    u = rest.union_ids.copy()
    u[missing] = [v for v in range(rest.V) if v not in set(u.tolist())][0]   # a candidate token not in U
    assert call(sc, args_of(rest, union_ids=dev(u))) == UNION
    assert call(sc, args_of(rest, union_ids=dev(rest.union_ids[:0]))) == ARG     # empty union
    assert call(sc, args_of(rest, union_ids=dev(np.arange(5000, dtype=np.int32)))) == ARG   # > JET_MAX_UNION
    # a multi-token candidate in restricted mode
    assert call(sc, args_of(wl, mode=wk.MODE_RESTRICTED, union_ids=dev(np.arange(500, dtype=np.int32)))) == MODE
    still_works(sc, rest)
    still_works(sc, wl)


def test_restricted_mode_ranges_and_offsets(env):
    """The restricted path validates in its own set kernel: same status codes."""
    jet, sc, wl, rest = env
    t = rest.tok_ids.copy(); t[3] = rest.V
    assert call(sc, args_of(rest, tok_ids=dev(t))) == TOKEN
    r = rest.tok_row.copy(); r[0] = rest.N
    assert call(sc, args_of(rest, tok_row=dev(r))) == TOKEN
    so = rest.set_offsets.copy(); so[-1] -= 1                             # sets do not cover candidates
    assert call(sc, args_of(rest, set_offsets=dev(so))) == OFFSETS
    co = rest.cand_offsets.copy(); co[-1] += 1                            # candidates do not cover tokens
    assert call(sc, args_of(rest, cand_offsets=dev(co))) == OFFSETS
    kd = rest.kind.copy(); kd[2] = 9
    assert call(sc, args_of(rest, kind=dev(kd))) == ARG
    still_works(sc, rest)


def test_score_tokens_checks(env):
    jet, sc, wl, _ = env
    a = args_of(wl)
    n = wl.N
    tok = wl.tok_ids[:n].copy(); tok[0] = wl.V
    with pytest.raises(jet.JetError) as e:
        sc.score_tokens(a["H"], a["W"], dev(tok))
    assert e.value.status == TOKEN
    lp = sc.score_tokens(a["H"], a["W"], dev(wl.tok_ids[:n]))
    assert torch.isfinite(lp).all()


def test_bounded_wait_runs_out_and_context_survives(env):
    """A device wait on a barrier nothing completes gives up after its limit,
    reports JET_ERR_TIMEOUT through the error word, and the context keeps
    working (failure handled on the device without a fault or a hang)."""
    import time
    jet, sc, wl, _ = env
    t0 = time.perf_counter()
    assert sc.selftest_wait_timeout(50_000) == -9        # 50 ms limit
    assert time.perf_counter() - t0 < 5.0
    still_works(sc, wl)
