"""Seeded synthetic workloads for the candidate-set scoring head.

This module only *draws inputs*: the output-embedding matrix ``W[V, d]``, the
hidden rows ``H[N, d]`` at teacher-forced candidate positions, candidate token
sequences and the CSR index arrays that describe candidate sets.  It holds none
of the scoring arithmetic (no projection, normaliser, chain rule or set rule);
both the fp64 CPU oracle and the CUDA library consume what it returns.

Conventions (the five named workloads follow the workload list of the scoring
benchmark; readings are listed in the design notes):

* bf16 values are stored as ``uint16`` bit patterns, rounded from fp32 with
  round-to-nearest-even.
* ``W``: i.i.d. N(0, 1) * d**-0.5, so a unit-RMS row gives logits of about unit
  variance.
* A hidden row is keyed by (set id, token history); identical keys give
  bit-identical rows, so duplicated candidates and shared prefixes see the same
  hidden states, as teacher forcing over one shared context would give them
  (JET: Justification Evaluation in Transformer, section on hybrid models:
  the prefix output supplies first-token probabilities; Gemma/MLX architecture
  page, "Candidate likelihoods").
* Row value: g ~ N(0, I_d) from a substream seeded by the key, h0 = g / rms(g).
  "Peaked" rows add gamma * W[t] / ||W[t]||^2 with gamma = logit(p) + ln V + 1/2,
  which puts roughly probability p on token t.
* RNG: numpy PCG64; base seed 20261202 + workload number; substreams via
  ``SeedSequence`` spawn keys so that results do not depend on draw order.
"""
from __future__ import annotations

import hashlib
import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

BASE_SEED = 20261202
# Fitted temperature of one checkpoint family (PARALLEL_SCORING page,
# "V2 probability default").
T_FITTED = 2.179078721266035

KIND_CHOICE, KIND_BINARY, KIND_ORDINAL = 0, 1, 2
MODE_FULL, MODE_RESTRICTED = 0, 1


# --------------------------------------------------------------------------
# bf16 helpers (bit-level conversions only)
# --------------------------------------------------------------------------
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (round-to-nearest-even); uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = (u >> 16) & 1          # finite inputs: u + 0x8000 stays below 2**32
    r += 0x7FFF
    r += u
    r >>= 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# workload container
# --------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    d: int
    V: int
    H: np.ndarray            # uint16 [N, d]   bf16 bits
    W: np.ndarray            # uint16 [V, d]   bf16 bits
    tok_row: np.ndarray      # int32 [n_tok]   row of H that predicts each token
    tok_ids: np.ndarray      # int32 [n_tok]   supplied candidate token ids
    cand_offsets: np.ndarray  # int32 [n_cand+1]  CSR: tokens of each candidate
    set_offsets: np.ndarray  # int32 [n_sets+1]  CSR: candidates of each set
    kind: np.ndarray         # uint8 [n_sets]  0 choice, 1 binary, 2 ordinal
    T: float
    mode: int = MODE_FULL
    union_ids: Optional[np.ndarray] = None   # int32 [n_union], restricted mode
    info: Dict[str, object] = field(default_factory=dict)

    @property
    def N(self) -> int:
        return int(self.H.shape[0])

    @property
    def n_tok(self) -> int:
        return int(self.tok_ids.shape[0])

    @property
    def n_cand(self) -> int:
        return int(self.cand_offsets.shape[0] - 1)

    @property
    def n_sets(self) -> int:
        return int(self.set_offsets.shape[0] - 1)

    def with_mode(self, mode: int, T: float, union_ids: Optional[np.ndarray]) -> "Workload":
        return Workload(self.name + ("-restricted" if mode == MODE_RESTRICTED else ""),
                        self.d, self.V, self.H, self.W, self.tok_row, self.tok_ids,
                        self.cand_offsets, self.set_offsets, self.kind, T, mode,
                        None if union_ids is None else np.ascontiguousarray(union_ids, np.int32),
                        dict(self.info))

    def checksum(self) -> str:
        h = hashlib.sha256()
        for a in (self.H, self.W, self.tok_row, self.tok_ids, self.cand_offsets,
                  self.set_offsets, self.kind):
            h.update(np.ascontiguousarray(a).tobytes())
        if self.union_ids is not None:
            h.update(self.union_ids.tobytes())
        h.update(repr((self.d, self.V, float(self.T), int(self.mode))).encode())
        return h.hexdigest()[:16]


# --------------------------------------------------------------------------
# random streams
# --------------------------------------------------------------------------
def _rng(seed: int, *key: int) -> np.random.Generator:
    # SeedSequence ignores trailing zero words, so a constant non-zero word
    # closes every key: keys that differ only by trailing zeros stay distinct.
    words = [seed, *[int(k) for k in key], 0x5EED]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(words)))


def gen_W(seed: int, V: int, d: int, chunk: int = 2048) -> np.ndarray:
    """Output embedding W[V, d]: N(0,1) * d**-0.5 in fp32, rounded to bf16.

    Each block of ``chunk`` rows has its own substream, so blocks are drawn in
    parallel threads and the result does not depend on the thread count."""
    scale = np.float32(1.0 / math.sqrt(d))
    W = np.empty((V, d), np.uint16)

    def block(i: int) -> None:
        v0 = i * chunk
        n = min(chunk, V - v0)
        g = _rng(seed, 0, i).standard_normal((n, d), dtype=np.float32)
        g *= scale
        W[v0:v0 + n] = to_bf16_bits(g)

    n_blocks = (V + chunk - 1) // chunk
    workers = max(1, min(32, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        list(ex.map(block, range(n_blocks)))
    return W


@dataclass
class _SetSpec:
    kind: int
    cands: List[Tuple[int, ...]]
    planted_first: bool = False     # config-5 style: candidate 0 is the planted path


def _continuations(spec: _SetSpec, prefix: Tuple[int, ...]) -> List[Tuple[int, int]]:
    """(candidate index, next token) of candidates that continue ``prefix``."""
    L = len(prefix)
    out = []
    for ci, c in enumerate(spec.cands):
        if len(c) > L and c[:L] == prefix:
            out.append((ci, c[L]))
    return out


def _build(name: str, seed: int, d: int, V: int, W: np.ndarray, sets: Sequence[_SetSpec],
           T: float, row_mode: str = "per_token",
           peak: Optional[Tuple[float, float]] = None, plant_prob: float = 0.8) -> Workload:
    """Lay out candidate sets as CSR arrays and draw the keyed hidden rows.

    row_mode "per_token": one hidden row per scored token (rows with equal keys
    are bit-identical copies).  "per_key": one row per distinct (set, history)
    key, shared by every token it predicts.
    """
    tok_row: List[int] = []
    tok_ids: List[int] = []
    cand_off = [0]
    set_off = [0]
    kinds: List[int] = []
    keys: List[Tuple[int, Tuple[int, ...]]] = []
    key_index: Dict[Tuple[int, Tuple[int, ...]], int] = {}
    key_of_row: List[int] = []
    for si, spec in enumerate(sets):
        kinds.append(spec.kind)
        for c in spec.cands:
            assert len(c) >= 1
            for t in range(len(c)):
                k = (si, tuple(c[:t]))
                if k not in key_index:
                    key_index[k] = len(keys)
                    keys.append(k)
                if row_mode == "per_token":
                    tok_row.append(len(key_of_row))
                    key_of_row.append(key_index[k])
                else:
                    tok_row.append(key_index[k])
                tok_ids.append(c[t])
            cand_off.append(len(tok_ids))
        set_off.append(len(cand_off) - 1)
    if row_mode != "per_token":
        key_of_row = list(range(len(keys)))

    # one value per distinct key
    vals = np.empty((len(keys), d), np.uint16)
    planted_p: List[float] = []
    for ki, (si, prefix) in enumerate(keys):
        rng = _rng(seed, 2, si, len(prefix), *prefix)
        g = rng.standard_normal(d)
        h = g / math.sqrt(float(np.mean(g * g)))
        if peak is not None:
            p = float(rng.uniform(peak[0], peak[1]))
            cont = _continuations(sets[si], prefix)
            u = float(rng.random())
            if sets[si].planted_first and cont and cont[0][0] == 0:
                t = cont[0][1]
            elif cont and u < plant_prob:
                t = cont[int(rng.integers(len(cont)))][1]
            else:
                t = int(rng.integers(V))
            w = bf16_bits_to_f32(W[t]).astype(np.float64)
            gamma = math.log(p / (1.0 - p)) + math.log(V) + 0.5
            h = h + gamma * w / float(np.sum(w * w))
            planted_p.append(p)
        vals[ki] = to_bf16_bits(h.astype(np.float32))
    H = vals[np.asarray(key_of_row, np.int64)] if key_of_row else np.zeros((0, d), np.uint16)
    wl = Workload(name, d, V, np.ascontiguousarray(H), W,
                  np.asarray(tok_row, np.int32), np.asarray(tok_ids, np.int32),
                  np.asarray(cand_off, np.int32), np.asarray(set_off, np.int32),
                  np.asarray(kinds, np.uint8), float(T))
    wl.info.update(distinct_rows=len(keys), seed=seed,
                   planted_p_mean=(float(np.mean(planted_p)) if planted_p else None))
    return wl


def _distinct_firsts(rng: np.random.Generator, V: int, n: int) -> List[int]:
    return [int(x) for x in rng.choice(V, size=n, replace=False)]


def _rand_tail(rng: np.random.Generator, V: int, n: int) -> Tuple[int, ...]:
    return tuple(int(x) for x in rng.integers(0, V, size=n))


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------
def tiny(seed_offset: int = 0) -> Workload:
    """d=64, V=1000: one choice set K=4 (lengths 1-3; candidates 0 and 1 share
    their first token; candidate 3 copies candidate 2), one binary set and one
    ordinal set of K=5 single-token levels.  T=1, full vocabulary."""
    seed = BASE_SEED + 1 + seed_offset
    d, V = 64, 1000
    W = gen_W(seed, V, d)
    rng = _rng(seed, 1)
    f = _distinct_firsts(rng, V, 2 + 2 + 5)
    lens = [int(x) for x in rng.integers(1, 4, size=3)]
    if lens[0] == 1 and lens[1] == 1:
        lens[1] = 2
    c0 = (f[0],) + _rand_tail(rng, V, lens[0] - 1)
    c1 = (f[0],) + _rand_tail(rng, V, lens[1] - 1)
    while c1 == c0:
        c1 = (f[0],) + _rand_tail(rng, V, lens[1] - 1)
    c2 = (f[1],) + _rand_tail(rng, V, lens[2] - 1)
    sets = [
        _SetSpec(KIND_CHOICE, [c0, c1, c2, c2]),
        _SetSpec(KIND_BINARY, [(f[2],), (f[3],)]),
        _SetSpec(KIND_ORDINAL, [(f[4 + i],) for i in range(5)]),
    ]
    return _build("tiny-d64-V1000", seed, d, V, W, sets, 1.0, row_mode="per_token")


def binary_batch(n_questions: int = 256, random_pairs: bool = False,
                 d: int = 2560, V: int = 248320, seed_offset: int = 0) -> Workload:
    """256 independent binary questions, one hidden row each (the last prefix
    position); candidates are the answer codes for A and B = (false, true).
    The 26 code ids A..Z are distinct and drawn once; ``info['codes']`` holds
    them (the restricted-mode union)."""
    seed = BASE_SEED + 2 + seed_offset
    W = gen_W(seed, V, d)
    rng = _rng(seed, 1)
    codes = _distinct_firsts(rng, V, 26)
    sets = []
    for _ in range(n_questions):
        if random_pairs:
            a, b = rng.choice(26, size=2, replace=False)
            pair = ((codes[int(a)],), (codes[int(b)],))
        else:
            pair = ((codes[0],), (codes[1],))
        sets.append(_SetSpec(KIND_BINARY, list(pair)))
    wl = _build(f"binary-d{d}-V{V}-q{n_questions}", seed, d, V, W, sets, 1.0, row_mode="per_key")
    wl.info["codes"] = np.asarray(codes, np.int32)
    return wl


def binary_restricted(n_questions: int = 256, random_pairs: bool = False,
                      d: int = 2560, V: int = 248320, base: Optional[Workload] = None) -> Workload:
    wl = base if base is not None else binary_batch(n_questions, random_pairs, d, V)
    return wl.with_mode(MODE_RESTRICTED, T_FITTED, wl.info["codes"])


def _shared_prefix_set(rng: np.random.Generator, V: int, K: int, len_lo: int, len_hi: int,
                       pair_lo: float, pair_hi: float) -> List[Tuple[int, ...]]:
    """K candidates; group members share an initial token run.  Group sizes are
    resampled until the fraction of candidate pairs inside a group lies in
    [pair_lo, pair_hi]."""
    n_pairs = K * (K - 1) // 2
    while True:
        G = int(rng.integers(2, K))
        labels = rng.integers(0, G, size=K)
        counts = np.bincount(labels, minlength=G)
        pairs = int(sum(c * (c - 1) // 2 for c in counts))
        if pair_lo * n_pairs <= pairs <= pair_hi * n_pairs:
            break
    groups = sorted(set(int(x) for x in labels))
    firsts = dict(zip(groups, _distinct_firsts(rng, V, len(groups))))
    cands: List[Optional[Tuple[int, ...]]] = [None] * K
    for gi in groups:
        members = [i for i in range(K) if labels[i] == gi]
        if len(members) == 1:
            L = int(rng.integers(len_lo, len_hi + 1))
            cands[members[0]] = (firsts[gi],) + _rand_tail(rng, V, L - 1)
            continue
        lens = [int(rng.integers(max(2, len_lo), len_hi + 1)) for _ in members]
        share = int(rng.integers(1, min(lens)))            # 1 .. min(m) - 1
        prefix = (firsts[gi],) + _rand_tail(rng, V, share - 1)
        made: List[Tuple[int, ...]] = []
        for i, L in zip(members, lens):
            c = prefix + _rand_tail(rng, V, L - share)
            while c in made:
                c = prefix + _rand_tail(rng, V, L - share)
            made.append(c)
            cands[i] = c
    return [c for c in cands if c is not None]


def multi_token_choice(n_questions: int = 64, K: int = 8, d: int = 1536, V: int = 262144,
                       seed_offset: int = 0) -> Workload:
    """64 questions x K=8 candidates of 1-12 tokens, one row per scored token;
    about 30% of candidate pairs share initial tokens; peaked rows with planted
    top-1 probability U(0.3, 0.9).  T=1."""
    seed = BASE_SEED + 3 + seed_offset
    W = gen_W(seed, V, d)
    rng = _rng(seed, 1)
    sets = [_SetSpec(KIND_CHOICE, _shared_prefix_set(rng, V, K, 1, 12, 0.25, 0.36))
            for _ in range(n_questions)]
    return _build(f"multitoken-d{d}-V{V}-q{n_questions}", seed, d, V, W, sets, 1.0,
                  row_mode="per_token", peak=(0.3, 0.9))


def wide_schema(n_requests: int = 16, n_fields: int = 32, d: int = 2560, V: int = 248320,
                seed_offset: int = 0) -> Workload:
    """16 requests x 32 fields; each field is, by a fair coin, an enum of
    K ~ U{2..26} candidates of 1-6 tokens or an ordinal set of K=5 single-token
    levels.  Unpeaked rows; T=2.179."""
    seed = BASE_SEED + 4 + seed_offset
    W = gen_W(seed, V, d)
    rng = _rng(seed, 1)
    sets = []
    for _ in range(n_requests * n_fields):
        if rng.random() < 0.5:
            K = int(rng.integers(2, 27))
            firsts = _distinct_firsts(rng, V, K)
            cands = [(f,) + _rand_tail(rng, V, int(rng.integers(1, 7)) - 1) for f in firsts]
            sets.append(_SetSpec(KIND_CHOICE, cands))
        else:
            sets.append(_SetSpec(KIND_ORDINAL, [(f,) for f in _distinct_firsts(rng, V, 5)]))
    return _build(f"wideschema-d{d}-V{V}-f{n_requests * n_fields}", seed, d, V, W, sets,
                  T_FITTED, row_mode="per_token")


def large_choice(n_requests: int = 16, K: int = 64, d: int = 4096, V: int = 152064,
                 len_lo: int = 8, len_hi: int = 32, seed_offset: int = 0) -> Workload:
    """16 requests x K=64 candidates of 8-32 tokens, one row per scored token;
    rows peaked (planted top-1 about 0.95) along candidate 0's path; 3 candidates
    per request are exact copies of earlier ones, and at least 4 requests copy
    candidate 0 to a later index.  T=1."""
    seed = BASE_SEED + 5 + seed_offset
    W = gen_W(seed, V, d)
    rng = _rng(seed, 1)
    copy0 = set(int(x) for x in rng.choice(n_requests, size=min(4, n_requests), replace=False))
    sets = []
    for r in range(n_requests):
        firsts = _distinct_firsts(rng, V, K)
        cands = [(f,) + _rand_tail(rng, V, int(rng.integers(len_lo, len_hi + 1)) - 1) for f in firsts]
        n_copy = min(3, K - 1)
        targets = sorted(int(x) for x in rng.choice(np.arange(1, K), size=n_copy, replace=False))
        for ti, t in enumerate(targets):
            src = 0 if (ti == 0 and r in copy0) else int(rng.integers(0, t))
            cands[t] = cands[src]
        sets.append(_SetSpec(KIND_CHOICE, cands, planted_first=True))
    return _build(f"large-d{d}-V{V}-r{n_requests}", seed, d, V, W, sets, 1.0,
                  row_mode="per_token", peak=(0.93, 0.97))


# --------------------------------------------------------------------------
# mid-size cases for element-by-element parity tests
# --------------------------------------------------------------------------
def custom(d: int, V: int, n_sets: int, K: Tuple[int, int] = (2, 8), length: Tuple[int, int] = (1, 6),
           kinds: Sequence[int] = (KIND_CHOICE, KIND_BINARY, KIND_ORDINAL), row_mode: str = "per_token",
           peak: Optional[Tuple[float, float]] = None, dup_prob: float = 0.1, T: float = 1.0,
           seed: int = 7) -> Workload:
    """Mixed sets at sizes the oracle finishes in seconds.  Binary sets get two
    single-token candidates; ordinal sets K single-token levels; choice sets
    K candidates with shared prefixes and occasional exact duplicates."""
    seed = BASE_SEED + 100 + seed
    W = gen_W(seed, V, d)
    rng = _rng(seed, 1)
    sets = []
    for _ in range(n_sets):
        kd = int(kinds[int(rng.integers(len(kinds)))])
        if kd == KIND_BINARY:
            a, b = _distinct_firsts(rng, V, 2)
            sets.append(_SetSpec(kd, [(a,), (b,)]))
        elif kd == KIND_ORDINAL:
            k = max(2, int(rng.integers(K[0], K[1] + 1)))
            sets.append(_SetSpec(kd, [(f,) for f in _distinct_firsts(rng, V, k)]))
        else:
            k = int(rng.integers(K[0], K[1] + 1))
            if k >= 3 and length[1] >= 2:
                cands = _shared_prefix_set(rng, V, k, length[0], length[1], 0.0, 1.0)
            else:
                cands = [(f,) + _rand_tail(rng, V, int(rng.integers(length[0], length[1] + 1)) - 1)
                         for f in _distinct_firsts(rng, V, k)]
            for i in range(1, k):
                if rng.random() < dup_prob:
                    cands[i] = cands[int(rng.integers(0, i))]
            sets.append(_SetSpec(kd, cands, planted_first=peak is not None))
    return _build(f"custom-d{d}-V{V}-s{n_sets}", seed, d, V, W, sets, T, row_mode=row_mode, peak=peak)


def union_choice(n_questions: int = 256, n_union: int = 600, K: Tuple[int, int] = (2, 2),
                 d: int = 2560, V: int = 248320, T: float = T_FITTED, seed_offset: int = 0) -> Workload:
    """Restricted mode over a larger union of single-token codes: n_union
    distinct ids drawn once; each question is a set of K ~ U{K[0]..K[1]}
    distinct codes of the union (binary when K = 2, else choice), one hidden
    row per question (shared by its codes)."""
    seed = BASE_SEED + 200 + seed_offset
    W = gen_W(seed, V, d)
    rng = _rng(seed, 1)
    union = np.asarray(_distinct_firsts(rng, V, n_union), np.int32)
    sets = []
    for _ in range(n_questions):
        k = min(int(rng.integers(K[0], K[1] + 1)), n_union)
        codes = [(int(t),) for t in rng.choice(union, size=k, replace=False)]
        sets.append(_SetSpec(KIND_BINARY if k == 2 else KIND_CHOICE, codes))
    wl = _build(f"union{n_union}-d{d}-V{V}-q{n_questions}", seed, d, V, W, sets, 1.0, row_mode="per_key")
    return wl.with_mode(MODE_RESTRICTED, T, union)


NAMED = {
    "tiny": tiny,
    "binary": binary_batch,
    "binary-restricted": binary_restricted,
    "multitoken": multi_token_choice,
    "wideschema": wide_schema,
    "large": large_choice,
}
