"""The seeded generator: determinism and the structure each workload promises."""
import numpy as np

import workloads as wk


def _sets(wl):
    for k in range(wl.n_sets):
        c0, c1 = wl.set_offsets[k], wl.set_offsets[k + 1]
        yield k, [tuple(wl.tok_ids[wl.cand_offsets[c]:wl.cand_offsets[c + 1]]) for c in range(c0, c1)]


def test_bf16_rounding_is_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], np.float32)
    got = wk.bf16_bits_to_f32(wk.to_bf16_bits(x))
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 3*2^-8 is a tie -> even (1 + 2^-6)
    np.testing.assert_array_equal(got, np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0], np.float32))


def test_generation_is_deterministic():
    a, b = wk.tiny(), wk.tiny()
    assert a.checksum() == b.checksum()
    c = wk.custom(64, 500, 5, seed=3)
    assert c.checksum() == wk.custom(64, 500, 5, seed=3).checksum()
    assert c.checksum() != wk.custom(64, 500, 5, seed=4).checksum()


def test_tiny_structure(wl_cache):
    wl = wl_cache("tiny")
    assert (wl.d, wl.V, wl.n_sets) == (64, 1000, 3)
    assert list(wl.kind) == [wk.KIND_CHOICE, wk.KIND_BINARY, wk.KIND_ORDINAL]
    sets = dict(_sets(wl))
    c = sets[0]
    assert len(c) == 4 and c[0][0] == c[1][0] and c[0] != c[1] and c[2] == c[3]
    assert all(1 <= len(x) <= 3 for x in c)
    assert len(sets[1]) == 2 and len(set(sets[1])) == 2
    assert len(sets[2]) == 5 and all(len(x) == 1 for x in sets[2])
    assert wl.N == wl.n_tok and np.array_equal(wl.tok_row, np.arange(wl.n_tok))
    # identical histories -> bit-identical rows
    assert np.array_equal(wl.H[0], wl.H[1])


def test_custom_structure_and_row_keys():
    wl = wk.custom(64, 700, 20, K=(2, 6), length=(1, 5), seed=9)
    assert wl.cand_offsets[-1] == wl.n_tok and wl.set_offsets[-1] == wl.n_cand
    for k, cands in _sets(wl):
        if wl.kind[k] == wk.KIND_BINARY:
            assert len(cands) == 2
        if wl.kind[k] == wk.KIND_ORDINAL:
            assert len(cands) >= 2 and all(len(c) == 1 for c in cands)
    per_key = wk.custom(64, 700, 20, K=(2, 6), length=(1, 5), seed=9, row_mode="per_key")
    assert per_key.N < wl.N and per_key.n_tok == wl.n_tok
    # each token sees the same row value in both layouts
    np.testing.assert_array_equal(per_key.H[per_key.tok_row], wl.H[wl.tok_row])
