"""Write oracle outputs for whole sampled sets of the full-size workloads.

The fp64 oracle needs minutes per set at full size (a large-workload set has
~1,300 hidden rows, each a 4096 x 152064 projection), too slow to recompute
inside a GPU test.  This script calls only ``oracle`` and ``workloads`` and
stores, per workload, the generator checksum and the oracle's outputs for the
chosen sets; the GPU test regenerates the inputs from the seed, checks the
checksum, and compares.

  python tests/golden/make_oracle_golden.py [workload ...]
"""
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
import workloads as wk  # noqa: E402
from parity import subset  # noqa: E402

# workload -> (generator, sets to store)
PLAN = {
    "multitoken": (wk.multi_token_choice, [5, 40]),
    "wideschema": (wk.wide_schema, None),          # chosen below: largest enum + an ordinal set
    "large": (wk.large_choice, None),              # chosen below: a set copying candidate 0 + one other
}


def choose_sets(name, wl):
    if name == "wideschema":
        sizes = np.diff(wl.set_offsets)
        return sorted({int(np.argmax(sizes)), int(np.nonzero(wl.kind == wk.KIND_ORDINAL)[0][0])})
    if name == "large":
        # a request in which a later candidate copies candidate 0 (the planted winner)
        for k in range(wl.n_sets):
            c0, c1 = wl.set_offsets[k], wl.set_offsets[k + 1]
            first = tuple(wl.tok_ids[wl.cand_offsets[c0]:wl.cand_offsets[c0 + 1]])
            if any(tuple(wl.tok_ids[wl.cand_offsets[c]:wl.cand_offsets[c + 1]]) == first for c in range(c0 + 1, c1)):
                return [k]
    return PLAN[name][1]


def main(names):
    for name in names:
        gen, sets = PLAN[name]
        wl = gen()
        sets = choose_sets(name, wl) if sets is None else sets
        sub, set_ids, cands, toks, rows = subset(wl, sets)
        t0 = time.time()
        r = oracle.score_workload(sub)
        dt = time.time() - t0
        rec = {
            "workload": name,
            "generator_checksum": wl.checksum(),
            "note": "fp64 oracle outputs for whole sets of the full-size workload; written by "
                    "tests/golden/make_oracle_golden.py (oracle and workloads only)",
            "oracle_seconds": round(dt, 1), "oracle_threads": oracle.max_threads(),
            "sets": [int(x) for x in set_ids], "cands": [int(x) for x in cands],
            "tokens": [int(x) for x in toks], "rows": [int(x) for x in rows],
            "logp": [float(x) for x in r.logp], "lse": [float(x) for x in r.lse],
            "s": [float(x) for x in r.s], "q": [float(x) for x in r.q], "q_equiv": [float(x) for x in r.q_equiv],
            "decision": [int(x) for x in r.decision], "expected": [float(x) for x in r.expected],
            "confidence": [float(x) for x in r.confidence], "mass": [float(x) for x in r.mass],
            "margin": [float(x) if np.isfinite(x) else 1e300 for x in r.margin],
        }
        with open(os.path.join(HERE, f"oracle_{name}.json"), "w") as f:
            json.dump(rec, f, separators=(",", ":"))
        print(f"{name}: sets {rec['sets']} ({len(toks)} tokens, {len(rows)} rows) in {dt:.0f}s", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:] or list(PLAN))
