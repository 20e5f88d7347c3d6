"""Oracle pins: greedy accept (speculative verify) and beam cache reorder. CPU only."""

import itertools
import json
import os

import numpy as np
import pytest

from workloads import gen_accept_inputs, gen_cache, gen_parents, make_rng

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _logits_with_tops(tops, vocab, rng, margin=3.0):
    """Rows whose unique largest logit sits at ``tops[i]``."""
    x = rng.standard_normal((len(tops), vocab)).astype(np.float32)
    for i, t in enumerate(tops):
        x[i, t] = x[i].max() + margin
    return x


def test_worked_example_sock_fox(oracle_mod):
    fx = json.load(open(os.path.join(GOLDEN, "sock_fox.json")))
    ids = {w: i for i, w in enumerate(fx["vocab"])}
    rng = make_rng(0)
    logits = _logits_with_tops([ids[w] for w in fx["main_top"]], len(ids), rng)[None]
    draft = np.array([[ids[w] for w in fx["draft"]]], np.int32)
    n, nxt, nmin, _, err = oracle_mod.greedy_accept(logits, draft)
    assert not err
    assert int(n[0]) == fx["expected"]["n_accepted"]
    assert fx["vocab"][int(nxt[0])] == fx["expected"]["next_token"]
    emitted = [fx["vocab"][t] for t in list(draft[0, : n[0]]) + [int(nxt[0])]]
    assert emitted == fx["expected"]["emitted"]


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
def test_every_agreement_pattern(oracle_mod, k):
    """All 2^k match/mismatch patterns: n is the position of the first mismatch (k if
    none) and the emitted token at n is the main model's token there."""
    rng = make_rng(20 + k)
    V = 11
    for pattern in itertools.product([True, False], repeat=k):
        tops = rng.integers(0, V, size=k + 1)
        logits = _logits_with_tops(tops, V, rng)[None]
        draft = np.array([[t if ok else (t + 1 + rng.integers(0, V - 1)) % V
                           for t, ok in zip(tops[:k], pattern)]], np.int32)
        n, nxt, _, amax, err = oracle_mod.greedy_accept(logits, draft)
        want_n = next((i for i, ok in enumerate(pattern) if not ok), k)
        assert not err
        assert list(amax[0]) == list(tops)
        assert int(n[0]) == want_n
        assert int(nxt[0]) == tops[want_n]


def test_argmax_matches_numpy_on_random_rows(oracle_mod):
    rng = make_rng(30)
    logits, draft = gen_accept_inputs(rng, 8, 5, 4099)
    _, _, _, amax, err = oracle_mod.greedy_accept(logits, draft)
    assert not err
    assert np.array_equal(amax, np.argmax(logits, axis=-1))


def test_ties_take_the_lowest_index(oracle_mod):
    V = 9
    row = np.zeros((1, 2, V), np.float32)
    row[0, 0, [2, 5, 7]] = 4.0
    row[0, 1, :] = -np.inf  # an all -inf row: every value ties, index 0 wins
    _, nxt, _, amax, err = oracle_mod.greedy_accept(row, np.array([[3]], np.int32))
    assert not err
    assert list(amax[0]) == [2, 0]
    assert int(nxt[0]) == 2


def test_nan_ranks_first_and_is_flagged(oracle_mod):
    V = 9
    x = np.zeros((1, 2, V), np.float32)
    x[0, 0, 1] = 100.0
    x[0, 0, [4, 6]] = np.nan
    _, _, _, amax, err = oracle_mod.greedy_accept(x, np.array([[1]], np.int32))
    assert amax[0, 0] == 4
    assert err == {19}


def test_out_of_vocab_draft_is_a_mismatch_and_flagged(oracle_mod):
    rng = make_rng(31)
    logits = _logits_with_tops([1, 2, 3, 4], 6, rng)[None]
    n, nxt, _, _, err = oracle_mod.greedy_accept(logits, np.array([[1, 6, 3]], np.int32))
    assert int(n[0]) == 1 and int(nxt[0]) == 2
    assert err == {18}
    n, nxt, _, _, err = oracle_mod.greedy_accept(logits, np.array([[1, 2, -1]], np.int32))
    assert int(n[0]) == 2 and int(nxt[0]) == 3
    assert err == {18}


def test_batch_minimum(oracle_mod):
    rng = make_rng(32)
    tops = [[1, 2, 3], [4, 4, 4], [0, 1, 2]]
    logits = np.stack([_logits_with_tops(t, 7, rng) for t in tops])
    draft = np.array([[1, 2], [4, 0], [5, 1]], np.int32)
    n, nxt, nmin, _, _ = oracle_mod.greedy_accept(logits, draft)
    assert list(n) == [2, 1, 0]
    assert list(nxt) == [3, 4, 0]
    assert nmin == 0


def test_accept_length_distribution_closed_form(oracle_mod):
    """With each draft matching independently with p = 0.75, P(n >= i) = 0.75^i, so
    E[n] = sum_{i=1..5} 0.75^i = 2.2880859375 and tokens per round = E[n] + 1."""
    rng = make_rng(33)
    trials, k = 4000, 5
    logits, draft = gen_accept_inputs(rng, trials, k, 997, p_match=0.75)
    n, _, nmin, _, err = oracle_mod.greedy_accept(logits, draft)
    assert not err
    e_n = sum(0.75 ** i for i in range(1, k + 1))
    sd = np.std(n) / np.sqrt(trials)
    assert abs(n.mean() - e_n) < 4 * sd
    for i in range(k):
        p_i = 0.75 ** i * 0.25
        assert abs(np.mean(n == i) - p_i) < 4 * np.sqrt(p_i * (1 - p_i) / trials)
    assert abs(np.mean(n == k) - 0.75 ** k) < 4 * np.sqrt(0.75 ** k * (1 - 0.75 ** k) / trials)
    assert nmin == n.min()


# --------------------------------------------------------------------------------- beam ----

def _expected_reorder(cache, parent, length):
    out = cache.copy()
    out[:, :, :length] = cache[parent][:, :, :length]
    return out


def test_identity_parents_change_nothing(oracle_mod):
    rng = make_rng(40)
    C, _ = gen_cache(rng, 10, 2, 12, 8, "f16", 1.0)
    got, err = oracle_mod.beam_reorder(C, np.arange(10, dtype=np.int32), 5, 12, "f16")
    assert not err and np.array_equal(got, C)


def test_all_parent_maps_beam3(oracle_mod):
    rng = make_rng(41)
    C, _ = gen_cache(rng, 3, 2, 9, 8, "bf16", 1.0)
    for parent in itertools.product(range(3), repeat=3):
        parent = np.array(parent, np.int32)
        for L in (0, 4, 9):
            got, err = oracle_mod.beam_reorder(C, parent, 3, L, "bf16")
            assert not err
            assert np.array_equal(got, _expected_reorder(C, parent, L))


def test_permutation_then_inverse_restores(oracle_mod):
    rng = make_rng(42)
    C, _ = gen_cache(rng, 10, 3, 7, 8, "f16", 1.0)
    perm = np.concatenate([rng.permutation(5), 5 + rng.permutation(5)]).astype(np.int32)
    inv = np.argsort(perm).astype(np.int32)
    a, _ = oracle_mod.beam_reorder(C, perm, 5, 7, "f16")
    b, _ = oracle_mod.beam_reorder(a, inv, 5, 7, "f16")
    assert np.array_equal(b, C)


def test_uniform_parents_match_fancy_indexing(oracle_mod):
    rng = make_rng(43)
    C, _ = gen_cache(rng, 40, 2, 16, 8, "f16", 1.0)
    parent = gen_parents(rng, 8, 5)
    got, err = oracle_mod.beam_reorder(C, parent, 5, 11, "f16")
    assert not err and np.array_equal(got, _expected_reorder(C, parent, 11))


def test_parent_outside_window_is_flagged_and_row_kept(oracle_mod):
    rng = make_rng(44)
    C, _ = gen_cache(rng, 6, 1, 5, 8, "f16", 1.0)
    parent = np.array([1, 1, 4, 3, 3, 4], np.int32)  # row 2 points into window 1
    got, err = oracle_mod.beam_reorder(C, parent, 3, 5, "f16")
    assert err == {17}
    assert np.array_equal(got[2], C[2])
    assert np.array_equal(got[0], C[1])
