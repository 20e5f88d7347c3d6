"""Pins of the oracle's temperature sampling and stochastic speculative acceptance
(oracle.sample_accept).

Fixed by the definitions and by the property the rejection rule exists for: inverse-CDF
draws at chosen uniforms (including the strict boundary of equal probabilities), the
tempered distribution p^(1/T) of a worked example, a hand-worked accept/reject case with
its residual, acceptance of every draft when draft and target agree, and -- the theorem
of speculative sampling -- that the first emitted token is distributed as the target
distribution whatever the draft distribution, checked by Monte Carlo over seeded
uniforms. A dropped clamp, an inverted ratio, a non-strict CDF test, an ignored
temperature or the bonus token drawn from the wrong row fails one of them.
"""

import math

import numpy as np
import pytest

import oracle


def _logits(*rows):
    return np.log(np.array(rows, dtype=np.float64)).astype(np.float32)


def test_inverse_cdf_draws():
    t = _logits([0.1, 0.2, 0.3, 0.4])[None]
    for u, want in [(0.05, 0), (0.15, 1), (0.35, 2), (0.65, 3), (0.999, 3)]:
        n, nxt, err = oracle.sample_accept(t, 1.0, np.array([u], np.float32))
        assert n.tolist() == [0] and nxt.tolist() == [want] and not err


def test_strict_boundary_of_equal_probabilities():
    # p = 1/4 each, exactly; u = 1/4 lies on the first boundary: the running sum must
    # exceed u, so the draw is id 1
    t = np.zeros((1, 1, 4), np.float32)
    for u, want in [(0.0, 0), (0.25, 1), (0.5, 2), (0.75, 3)]:
        assert oracle.sample_accept(t, 1.0, np.array([u], np.float32))[1].tolist() == [want]


def test_temperature_sharpens():
    # T = 0.5 turns p into p^2 / sum p^2 = (1, 4, 9, 16) / 30: the running sums are
    # 0.033, 0.167, 0.467, 1, so u = 0.5 draws id 3 (at T = 1 it draws id 2)
    t = _logits([0.1, 0.2, 0.3, 0.4])[None]
    u = np.array([0.5], np.float32)
    assert oracle.sample_accept(t, 1.0, u)[1].tolist() == [2]
    assert oracle.sample_accept(t, 0.5, u)[1].tolist() == [3]
    assert oracle.sample_accept(t, 0.5, np.array([0.1], np.float32))[1].tolist() == [1]


def test_worked_accept_and_reject():
    # p = (0.5, 0.5), q = (0.9, 0.1), draft id 0: accepted iff r < 0.5 / 0.9 = 0.556;
    # after a rejection the residual max(0, p - q) = (0, 0.4) always gives id 1
    target = np.stack([np.zeros(2), np.log([0.2, 0.8])]).astype(np.float32)[None]
    draft = _logits([0.9, 0.1])[None]
    drafts = np.array([[0]], np.int32)
    for r, u, want_n, want_next in [(0.5, 0.1, 1, 0), (0.5, 0.3, 1, 1), (0.5, 0.5, 1, 1),
                                    (0.6, 0.1, 0, 1), (0.99, 0.9, 0, 1)]:
        n, nxt, err = oracle.sample_accept(target, 1.0, np.array([u], np.float32), draft=draft,
                                           drafts=drafts, r=np.array([[r]], np.float32))
        # accepted: the bonus token comes from target row 1 = (0.2, 0.8), so u = 0.3
        # gives id 1 (row 0 would give id 0)
        assert (n.tolist(), nxt.tolist()) == ([want_n], [want_next]) and not err


def test_matching_draft_is_always_accepted():
    rng = np.random.default_rng(5)
    k, V = 4, 30
    x = rng.standard_normal((2, k + 1, V)).astype(np.float32)
    drafts = rng.integers(0, V, (2, k)).astype(np.int32)
    r = np.full((2, k), 0.999, np.float32)
    n, _, err = oracle.sample_accept(x, 0.7, np.array([0.3, 0.6], np.float32), draft=x[:, :k],
                                     drafts=drafts, r=r)
    assert n.tolist() == [k, k] and not err


@pytest.mark.parametrize("k", [1, 3])
def test_first_token_follows_the_target_distribution(k):
    # speculative sampling's guarantee: whatever q is, the first emitted token (the
    # draft if accepted, else the residual draw) is distributed as p
    rng = np.random.default_rng(11 + k)
    V, N, T = 6, 20000, 1.3
    target_row = rng.standard_normal(V).astype(np.float32) * 2
    draft_row = rng.standard_normal(V).astype(np.float32) * 2
    p = np.exp(target_row.astype(np.float64) / T)
    p /= p.sum()
    q = np.exp(draft_row.astype(np.float64) / T)
    q /= q.sum()
    target = np.broadcast_to(target_row, (N, k + 1, V)).copy()
    draft = np.broadcast_to(draft_row, (N, k, V)).copy()
    drafts = np.stack([rng.choice(V, size=N, p=q) for _ in range(k)], axis=1).astype(np.int32)
    r = rng.random((N, k)).astype(np.float32)
    u = rng.random(N).astype(np.float32)
    n, nxt, err = oracle.sample_accept(target, T, u, draft=draft, drafts=drafts, r=r)
    assert not err
    first = np.where(n > 0, drafts[:, 0], nxt)
    freq = np.bincount(first, minlength=V) / N
    sigma = np.sqrt(p * (1 - p) / N)
    assert np.all(np.abs(freq - p) < 5 * sigma + 1e-4), (freq, p)
    # and the acceptance rate of the first draft is sum_v min(p, q)
    acc = np.mean(n > 0)
    want = np.minimum(p, q).sum()
    assert abs(acc - want) < 5 * math.sqrt(want * (1 - want) / N)


def test_bad_draft_nan_and_empty_residual():
    t = np.zeros((1, 2, 4), np.float32)
    # a drafted id outside the vocabulary is rejected; p == q leaves an empty residual,
    # so the draw falls back to p
    n, nxt, err = oracle.sample_accept(t, 1.0, np.array([0.6], np.float32), draft=t[:, :1],
                                       drafts=np.array([[9]], np.int32),
                                       r=np.array([[0.1]], np.float32))
    assert n.tolist() == [0] and nxt.tolist() == [2] and err == {18}
    t2 = t.copy()
    t2[0, 0, 1] = np.nan
    n, nxt, err = oracle.sample_accept(t2[:, :1], 1.0, np.array([0.4], np.float32))
    assert err == {19} and nxt.tolist() == [2]  # (1/3, 0, 1/3, 1/3): 0.4 -> id 2


def test_low_temperature_picks_the_maximum():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 1, 100)).astype(np.float32) * 3
    n, nxt, err = oracle.sample_accept(x, 0.01, np.array([0.2, 0.5, 0.8], np.float32))
    assert nxt.tolist() == np.argmax(x[:, 0], axis=1).tolist()
