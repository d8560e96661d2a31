"""The head's two variants and the launch chain without programmatic dependent
launch, each forced through its diagnostic environment variable in a fresh
process (the library reads them once): the one-CTA head on several row tiles,
the paired head on a single partial row tile, and every kernel launched with
plain stream ordering.  Each run is compared with the oracle, full and
restricted mode."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
import oracle, workloads as wk
import candidate_answer_scoring_gb300 as jet
from parity import compare
cases = [wk.custom(128, 2100, {n_sets}, K=(2, 6), length=(1, 4), dup_prob=0.2, seed={seed}),
         wk.binary_restricted(base=wk.binary_batch({n_q}, random_pairs=True, d=128, V=1800))]
for wl in cases:
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    sc = jet.JetScorer(wl.d, wl.V, wl.N, wl.n_tok)
    out = sc.score_sets(t(wl.H.view(np.int16)).view(torch.bfloat16), t(wl.W.view(np.int16)).view(torch.bfloat16),
                        t(wl.tok_row), t(wl.tok_ids), t(wl.cand_offsets), t(wl.set_offsets), t(wl.kind), wl.T,
                        wl.mode, None if wl.union_ids is None else t(wl.union_ids))
    torch.cuda.synchronize()
    compare(wl, {{k: v.cpu().numpy() for k, v in out.items()}}, oracle.score_workload(wl))
    print("N", wl.N, "ok")
"""


@pytest.mark.parametrize("env,n_sets,n_q", [
    ({"JETSCORE_HEAD_PAIR": "0"}, 60, 300),    # one-CTA head, several 128-row tiles
    ({"JETSCORE_HEAD_PAIR": "1"}, 12, 40),     # paired head, one partial 256-row tile
    ({"JETSCORE_NO_PDL": "1"}, 40, 200),       # plain stream ordering between launches
])
def test_forced_variant_matches_oracle(env, n_sets, n_q):
    code = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"), n_sets=n_sets, seed=n_sets + 7, n_q=n_q)
    r = subprocess.run([sys.executable, "-c", code], env={**os.environ, **env}, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count(" ok") == 2, r.stdout
