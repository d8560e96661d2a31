"""The allocation-free entry point, jet_score_tokens_noalloc, called through
the C ABI and checked against jet_score_tokens on two calls in a row.

It serves callers that may not allocate device memory (their process's device
memory belongs to another framework's pool), so its scratch is a static device
array shared by all calls; the second call, smaller and on other data, checks
that what the first call left there does not leak into the result.  This file
is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads as wk

pytestmark = pytest.mark.gpu

TOL = 2e-3   # the per-token log-probability tolerance of the parity tests


def _noalloc_fn():
    import candidate_answer_scoring_gb300 as jet
    lib = jet.load()
    fn = lib.jet_score_tokens_noalloc
    P = C.c_void_p
    fn.argtypes = [P, P, C.c_int, C.c_int, P, C.c_int, P, P, P]
    fn.restype = C.c_int
    return jet, fn


def test_noalloc_matches_score_tokens_on_two_calls():
    jet, fn = _noalloc_fn()
    dev = torch.device("cuda", 0)
    stream = C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    for call, (d, V, n, seed) in enumerate([(256, 7000, 900, 1), (128, 3001, 333, 2)]):
        rng = np.random.default_rng(seed)
        W = torch.from_numpy(wk.gen_W(500 + seed, V, d).view(np.int16)).to(dev).view(torch.bfloat16)
        H = torch.from_numpy(wk.to_bf16_bits(rng.normal(size=(n, d)).astype(np.float32)).view(np.int16))
        H = H.to(dev).view(torch.bfloat16)
        tok = torch.from_numpy(rng.integers(0, V, size=n).astype(np.int32)).to(dev)
        ref_lp, ref_lse = jet.JetScorer(d, V, n, n).score_tokens(H, W, tok, want_lse=True)
        logp = torch.full((n,), float("nan"), device=dev)
        lse = torch.full((n,), float("nan"), device=dev)
        rc = fn(C.c_void_p(H.data_ptr()), C.c_void_p(W.data_ptr()), d, V, C.c_void_p(tok.data_ptr()), n,
                C.c_void_p(logp.data_ptr()), C.c_void_p(lse.data_ptr()), stream)
        assert rc == 0, f"call {call}: status {rc} ({jet.status_string(rc)})"
        assert torch.isfinite(logp).all() and torch.isfinite(lse).all()
        assert (logp - ref_lp).abs().max().item() <= TOL, f"call {call}: logp differs"
        assert (lse - ref_lse).abs().max().item() <= TOL, f"call {call}: lse differs"


def test_noalloc_rejects_batches_beyond_its_static_scratch():
    jet, fn = _noalloc_fn()
    lib = jet.load()
    dev = torch.device("cuda", 0)
    n = 4097                                   # JET_NOALLOC_MAX_POS + 1
    H = torch.zeros((n, 64), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((100, 64), dtype=torch.bfloat16, device=dev)
    tok = torch.zeros(n, dtype=torch.int32, device=dev)
    out = torch.empty(n, device=dev)
    rc = fn(C.c_void_p(H.data_ptr()), C.c_void_p(W.data_ptr()), 64, 100, C.c_void_p(tok.data_ptr()), n,
            C.c_void_p(out.data_ptr()), None, C.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert rc == -6, f"expected JET_ERR_WORKSPACE, got {rc}"


def test_noalloc_many_waves_matches_fp32_torch():
    """4096 positions over V = 30000: 16 paired row tiles and several waves of
    units (taken in counter order), against logits formed with torch in fp32
    from the same bf16 values."""
    jet, fn = _noalloc_fn()
    dev = torch.device("cuda", 0)
    d, V, n = 128, 30000, 4096
    rng = np.random.default_rng(11)
    W = torch.from_numpy(wk.gen_W(611, V, d).view(np.int16)).to(dev).view(torch.bfloat16)
    H = torch.from_numpy(wk.to_bf16_bits(rng.normal(size=(n, d)).astype(np.float32)).view(np.int16))
    H = H.to(dev).view(torch.bfloat16)
    tok = torch.from_numpy(rng.integers(0, V, size=n).astype(np.int32)).to(dev)
    info = jet.JetScorer(d, V, n, n).plan_info(n)
    assert info["units"] > info["ctas"] // 2, info      # more than one wave
    logp = torch.full((n,), float("nan"), device=dev)
    lse = torch.full((n,), float("nan"), device=dev)
    rc = fn(C.c_void_p(H.data_ptr()), C.c_void_p(W.data_ptr()), d, V, C.c_void_p(tok.data_ptr()), n,
            C.c_void_p(logp.data_ptr()), C.c_void_p(lse.data_ptr()),
            C.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert rc == 0, jet.status_string(rc)
    z = H.float() @ W.float().T
    ref_lse = torch.logsumexp(z, dim=1)
    ref_lp = z.gather(1, tok.long()[:, None])[:, 0] - ref_lse
    assert (lse - ref_lse).abs().max().item() <= TOL
    assert (logp - ref_lp).abs().max().item() <= TOL


def test_noalloc_call_after_a_rejected_call():
    """A call the device pre-pass rejects (a token id equal to V) leaves its
    error word and, for a plan with several waves of units, the unit counter
    in the shared static array; the next valid call over several waves must
    start clean and match jet_score_tokens."""
    jet, fn = _noalloc_fn()
    dev = torch.device("cuda", 0)
    stream = C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    d, V, n = 128, 30000, 4096
    rng = np.random.default_rng(12)
    W = torch.from_numpy(wk.gen_W(612, V, d).view(np.int16)).to(dev).view(torch.bfloat16)
    H = torch.from_numpy(wk.to_bf16_bits(rng.normal(size=(n, d)).astype(np.float32)).view(np.int16))
    H = H.to(dev).view(torch.bfloat16)
    tok = torch.from_numpy(rng.integers(0, V, size=n).astype(np.int32)).to(dev)
    bad = tok.clone()
    bad[n // 2] = V
    logp = torch.full((n,), float("nan"), device=dev)
    lse = torch.full((n,), float("nan"), device=dev)
    args = lambda t: (C.c_void_p(H.data_ptr()), C.c_void_p(W.data_ptr()), d, V, C.c_void_p(t.data_ptr()), n,
                      C.c_void_p(logp.data_ptr()), C.c_void_p(lse.data_ptr()), stream)
    rc = fn(*args(bad))
    assert rc == -2, f"expected JET_ERR_TOKEN_RANGE, got {rc} ({jet.status_string(rc)})"
    sc = jet.JetScorer(d, V, n, n)
    info = sc.plan_info(n)
    assert info["units"] > info["ctas"] // 2, info      # the counter path
    rc = fn(*args(tok))
    assert rc == 0, f"status {rc} ({jet.status_string(rc)}) after a rejected call"
    ref_lp, ref_lse = sc.score_tokens(H, W, tok, want_lse=True)
    assert (logp - ref_lp).abs().max().item() <= TOL
    assert (lse - ref_lse).abs().max().item() <= TOL
