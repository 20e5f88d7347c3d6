"""Pins of the oracle's logit filters and beam-search step (oracle.beam_select).

The pins come from outside the oracle's own loops: a hand-worked two-beam example
whose log-probabilities are logs of chosen probabilities, the normalisation of a
log-softmax, scipy's log_softmax on the filtered logits, numpy's argmax for the
filtered greedy token, and a brute-force walk over every (beam, token) continuation of
the whole vocabulary -- which also checks that keeping only each beam's beam+1 best
tokens loses nothing. A dropped filter, a filter applied at the wrong step, a missing
cumulative score, a wrong tie rule or EOT kept as a live beam fails one of them.
"""

import math

import numpy as np
import pytest
from scipy.special import log_softmax

import oracle
from workloads import gen_beam_select_inputs, make_rng


def _logits(*rows):
    return np.log(np.array(rows, dtype=np.float64)).astype(np.float32)


def test_worked_example_two_beams():
    # beam 2, vocabulary {0, 1, 2, 3 = EOT}; logits are logs of probabilities, so the
    # log-softmax returns them (up to fp32 rounding of the inputs)
    x = _logits([0.5, 0.25, 0.125, 0.125], [0.1, 0.2, 0.3, 0.4])
    cum = np.array([-1.0, -0.5], np.float32)
    r = oracle.beam_select(x, 2, cum=cum, eot=3)
    # row 0: tokens 0, 1 and 2 (2 and 3 tie, the lower id wins); row 1: tokens 3, 2, 1
    assert r["row_token"].tolist() == [[0, 1, 2], [3, 2, 1]]
    lx = x.astype(np.float64)
    assert np.allclose(r["row_logprob"], [[lx[0, 0], lx[0, 1], lx[0, 2]],
                                          [lx[1, 3], lx[1, 2], lx[1, 1]]], atol=1e-7)
    # scores: (1,EOT) -1.416 > (0,0) -1.693 > (1,2) -1.704: EOT finishes, two beams kept
    assert r["n_fin"].tolist() == [1]
    assert r["fin_parent"].tolist() == [1, -1]
    assert r["fin_score"][0] == pytest.approx(-0.5 + math.log(0.4), abs=1e-6)
    assert r["fin_score"][1] == -np.inf
    assert r["parent"].tolist() == [0, 1] and r["token"].tolist() == [0, 2]
    assert np.allclose(r["new_cum"], [-1.0 + math.log(0.5), -0.5 + math.log(0.3)], atol=1e-6)
    assert not r["errors"]


def test_worked_example_first_step_masks_eot_and_blank():
    x = _logits([0.5, 0.25, 0.125, 0.125], [0.1, 0.2, 0.3, 0.4])
    cum = np.array([-1.0, -0.5], np.float32)
    # first position: EOT is masked, the other probabilities renormalise
    r = oracle.beam_select(x, 2, cum=cum, eot=3, first_step=True)
    assert r["n_fin"].tolist() == [0]
    assert r["parent"].tolist() == [1, 0] and r["token"].tolist() == [2, 0]
    assert np.allclose(r["new_cum"], [-0.5 + math.log(0.5), -1.0 + math.log(4 / 7)], atol=1e-6)
    # ... and with blank id 2: row 1 keeps {0, 1}, row 0 keeps {0, 1}
    r = oracle.beam_select(x, 2, cum=cum, eot=3, blank=[2], first_step=True)
    assert r["row_token"].tolist() == [[0, 1, 2], [1, 0, 2]]
    assert r["row_logprob"][0, 2] == -np.inf and r["row_logprob"][1, 2] == -np.inf
    assert np.allclose(r["row_logprob"][1, :2], [math.log(2 / 3), math.log(1 / 3)], atol=1e-6)
    assert r["parent"].tolist() == [1, 0] and r["token"].tolist() == [1, 0]
    # blank ids are only masked at the first position
    r = oracle.beam_select(x, 2, cum=cum, eot=3, blank=[2], first_step=False)
    assert r["row_token"][1, 1] == 2


def test_log_softmax_normalises():
    # vocab = beam + 1: every token comes back, and the probabilities sum to one
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((6, 4)) * 3).astype(np.float32)
    r = oracle.beam_select(x, 3, walk=False)
    p = np.exp(r["row_logprob"])
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12)
    # log-probability differences are the logit differences
    got = r["row_logprob"] - r["row_logprob"][:, :1]
    xs = np.take_along_axis(x.astype(np.float64), r["row_token"], axis=1)
    assert np.allclose(got, xs - xs[:, :1], atol=1e-12)
    # suppressed ids get probability 0, the rest renormalise
    r = oracle.beam_select(x, 3, suppress=[1], walk=False)
    lp = r["row_logprob"]
    assert np.all(r["row_token"][:, 3] == 1) and np.all(lp[:, 3] == -np.inf)
    assert np.allclose(np.exp(lp[:, :3]).sum(axis=1), 1.0, atol=1e-12)


def _brute_force(x, beam, cum, suppress, blank, eot, first_step):
    """Every (row, token) continuation of the whole vocabulary, ranked by score."""
    rows, V = x.shape
    f = x.astype(np.float64).copy()
    f[np.isnan(f)] = -np.inf
    f[:, list(suppress)] = -np.inf
    if first_step:
        f[:, list(blank) + [eot]] = -np.inf
    lp = log_softmax(f, axis=1)
    out = []
    for w in range(rows // beam):
        cont = []
        for j in range(beam):
            r = w * beam + j
            order = sorted(range(V), key=lambda v: (-f[r, v], v))  # rank in the row
            for rank, v in enumerate(order):
                cont.append((cum[r] + lp[r, v], j, rank, v))
        cont.sort(key=lambda c: (-c[0], c[1], c[2]))
        kept, fin = [], []
        for s, j, _, v in cont:
            if len(kept) == beam:
                break
            (fin if v == eot else kept).append((w * beam + j, v, s))
        out.append((kept, fin))
    return out, lp


@pytest.mark.parametrize("seed,beam,vocab,first", [(1, 2, 13, False), (2, 3, 40, True),
                                                    (3, 5, 64, False), (4, 4, 9, False)])
def test_brute_force_over_the_whole_vocabulary(seed, beam, vocab, first):
    rng = make_rng(seed)
    eot = vocab - 1
    x, cum, sup = gen_beam_select_inputs(rng, 3, beam, vocab, p_eot=0.6, eot=eot, n_suppress=2,
                                         cum_range=(0.0, 3.0))
    blank = [int(sup[0]) + 1 if sup[0] + 1 != eot else 0]
    want, lp = _brute_force(x, beam, cum.astype(np.float64), sup, blank, eot, first)
    r = oracle.beam_select(x, beam, cum=cum, suppress=sup, blank=blank, eot=eot,
                           first_step=first)
    assert not r["errors"]
    n_fin_total = 0
    for w, (kept, fin) in enumerate(want):
        sl = slice(w * beam, (w + 1) * beam)
        assert r["parent"][sl].tolist() == [k[0] for k in kept]
        assert r["token"][sl].tolist() == [k[1] for k in kept]
        assert np.allclose(r["new_cum"][sl], [k[2] for k in kept], atol=1e-12)
        assert r["n_fin"][w] == len(fin)
        assert r["fin_parent"][sl][:len(fin)].tolist() == [f[0] for f in fin]
        assert np.allclose(r["fin_score"][sl][:len(fin)], [f[2] for f in fin], atol=1e-12)
        n_fin_total += len(fin)
    # step 1 against scipy's log_softmax at the returned tokens
    assert np.allclose(np.take_along_axis(lp, r["row_token"], axis=1), r["row_logprob"],
                       atol=1e-12)
    if first:
        assert n_fin_total == 0
    elif seed == 3:
        assert n_fin_total > 0  # the case exercises finished continuations


def test_ties_across_and_within_beams():
    # two identical beams: equal scores keep the row order; equal logits the id order
    x = np.zeros((2, 6), np.float32)
    x[:, 4] = 1.0
    r = oracle.beam_select(x, 2, cum=np.zeros(2, np.float32), eot=5)
    assert r["row_token"].tolist() == [[4, 0, 1], [4, 0, 1]]
    assert r["parent"].tolist() == [0, 1] and r["token"].tolist() == [4, 4]


def test_greedy_token_is_the_filtered_argmax():
    rng = make_rng(11)
    x, _, sup = gen_beam_select_inputs(rng, 4, 1, 500, n_suppress=20, eot=499)
    sup = np.concatenate([sup, np.argmax(x, axis=1)[:2]]).astype(np.int32)  # mask 2 maxima
    r = oracle.beam_select(x, 1, suppress=sup, eot=499, walk=False)
    f = x.copy()
    f[:, sup] = -np.inf
    assert r["row_token"][:, 0].tolist() == np.argmax(f, axis=1).tolist()


def test_nan_and_bad_ids_are_flagged():
    x = _logits([0.5, 0.25, 0.125, 0.125], [0.1, 0.2, 0.3, 0.4])
    x[0, 0] = np.nan
    r = oracle.beam_select(x, 2, cum=np.zeros(2, np.float32), eot=3)
    assert r["errors"] == {19}
    assert 0 not in r["row_token"][0].tolist()[:2]  # NaN ranks as -inf
    r = oracle.beam_select(x[1:].repeat(2, axis=0), 2, suppress=[7, -1], eot=3)
    assert r["errors"] == {18}
    r = oracle.beam_select(x[1:].repeat(2, axis=0), 2, cum=np.array([np.nan, 0], np.float32),
                           eot=3)
    assert r["errors"] == {19} and np.all(r["parent"] == 1)


def test_invariants_on_the_beam_workload():
    rng = make_rng(12)
    x, cum, sup = gen_beam_select_inputs(rng, 2, 5, 51865)
    r = oracle.beam_select(x, 5, cum=cum, suppress=sup, blank=[220], eot=50257)
    for w in range(2):
        sl = slice(w * 5, (w + 1) * 5)
        assert np.all((r["parent"][sl] >= w * 5) & (r["parent"][sl] < w * 5 + 5))
        assert np.all(np.diff(r["new_cum"][sl]) <= 0)
        assert not np.isin(r["token"][sl], np.append(sup, 50257)).any()
        nf = r["n_fin"][w]
        assert np.all(r["fin_score"][sl][:nf] >= r["new_cum"][sl][-1])
        # a kept continuation never scores above its parent's cumulative score
        assert np.all(r["new_cum"][sl] <= cum[r["parent"][sl]])
