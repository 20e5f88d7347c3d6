"""Logit filters + beam-search selection on the GPU (kvd_beam_select) against the oracle.

Integer results are compared exactly where the oracle's fp64 scores leave a margin
larger than the fp32 rounding of the kernel (TOL); where two continuations of
different beams score closer than that, both orders are correct, and the kernel's
choice is checked for validity instead: every kept or finished continuation must be
one of its row's beam+1 best tokens, score within TOL of the oracle's score, and
outrank (within TOL) every continuation not chosen. Per-row tokens are decided by
exact comparisons of the fp32 logits and always match exactly; log-probabilities and
scores match the oracle within TOL.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev_i32, new_err, require_gpu
from workloads import WORKLOADS, gen_beam_select_inputs, make_rng

pytestmark = pytest.mark.gpu
WL = WORKLOADS["beam_select"]


def TOL(x):
    return 2e-5 + 2e-6 * np.abs(x)


def close(a, b):
    """Equal within TOL, or both -inf."""
    return (np.isneginf(a) and np.isneginf(b)) or abs(a - b) <= TOL(b)


def at_most(a, b):
    """a <= b within TOL (b may be -inf)."""
    return a == -np.inf if np.isneginf(b) else a <= b + TOL(b)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_gpu(logits, beam, *, cum=None, suppress=(), blank=(), eot=0, first=False, walk=True,
            flags=0, err=None, logits_dev=None):
    import kv_cached_decode_gb300 as kvd

    rows, V = logits.shape
    W, K = rows // beam, beam + 1
    e = new_err() if err is None else err
    f32 = dict(dtype=torch.float32, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    out = {"row_token": torch.full((rows, K), -7, **i32),
           "row_logprob": torch.full((rows, K), 7.0, **f32)}
    if walk:
        out.update(parent=torch.full((rows,), -7, **i32), token=torch.full((rows,), -7, **i32),
                   new_cum=torch.full((rows,), 7.0, **f32), n_finished=torch.full((W,), -7, **i32),
                   fin_parent=torch.full((rows,), -7, **i32),
                   fin_score=torch.full((rows,), 7.0, **f32))
    if logits_dev is None:
        logits_dev = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    kvd.kvd_beam_select(logits_dev, beam,
                        cum=None if cum is None else torch.from_numpy(cum).cuda(),
                        suppress=dev_i32(np.asarray(suppress, np.int32)) if len(suppress) else None,
                        blank=dev_i32(np.asarray(blank, np.int32)) if len(blank) else None,
                        eot=eot, first_step=first, flags=flags, dev_err=e, **out)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in out.items()}
    got["err"] = e.item()
    return got


def check(got, want, beam, cum_len_hint=""):
    """Compare a GPU result with the oracle's (see the module docstring)."""
    rt, wlp = want["row_token"], want["row_logprob"]
    assert np.array_equal(got["row_token"], rt)
    glp = got["row_logprob"]
    both_inf = np.isneginf(glp) & np.isneginf(wlp)
    assert np.all(both_inf | (np.abs(glp - wlp) <= TOL(wlp))), np.max(np.abs(glp - wlp))
    if "parent" not in want:
        return 0
    rows, K = rt.shape
    n_exact = 0
    for w in range(rows // beam):
        sl = slice(w * beam, (w + 1) * beam)
        # the oracle's continuation scores (cum + logprob), candidate c = j*K + k
        sc = (want["cum"][sl, None] + wlp[sl]).ravel()
        tok = rt[sl].ravel()
        order = sorted(range(beam * K), key=lambda c: (-sc[c], c))
        m = beam + int(want["n_fin"][w])
        top = sc[order[:m + 1]]
        fin_ok = np.isfinite(top)
        gaps = np.diff(top[fin_ok])
        if np.all(np.abs(gaps) > TOL(top[fin_ok][1:])) and fin_ok.all():
            assert np.array_equal(got["parent"][sl], want["parent"][sl])
            assert np.array_equal(got["token"][sl], want["token"][sl])
            assert got["n_finished"][w] == want["n_fin"][w]
            assert np.array_equal(got["fin_parent"][sl], want["fin_parent"][sl])
            n_exact += 1
        # validity, in every case
        nf = int(got["n_finished"][w])
        chosen = []
        for s in range(beam):
            j = got["parent"][w * beam + s] - w * beam
            assert 0 <= j < beam
            k = list(rt[w * beam + j]).index(got["token"][w * beam + s])
            c = j * K + k
            assert tok[c] != want["eot"]
            assert close(got["new_cum"][w * beam + s], sc[c])
            chosen.append(c)
        lowest_kept = min(sc[c] for c in chosen)
        for f in range(nf):
            j = got["fin_parent"][w * beam + f] - w * beam
            k = list(rt[w * beam + j]).index(want["eot"])
            c = j * K + k
            assert close(got["fin_score"][w * beam + f], sc[c])
            assert at_most(lowest_kept, sc[c])
            chosen.append(c)
        assert len(set(chosen)) == len(chosen)
        # nothing left out outranks the last kept continuation
        assert all(at_most(sc[c], lowest_kept) for c in range(beam * K) if c not in chosen)
        assert np.all(got["fin_parent"][w * beam + nf:(w + 1) * beam] == -1)
        assert np.all(np.isneginf(got["fin_score"][w * beam + nf:(w + 1) * beam]))
        assert np.all(np.diff(got["new_cum"][sl]) <= TOL(got["new_cum"][sl][1:]))
    return n_exact


def oracle_run(logits, beam, *, cum=None, suppress=(), blank=(), eot=0, first=False,
               walk=True):
    r = oracle.beam_select(logits, beam, cum=cum, suppress=suppress, blank=blank, eot=eot,
                           first_step=first, walk=walk)
    r["cum"] = np.zeros(logits.shape[0]) if cum is None else cum.astype(np.float64)
    r["eot"] = eot
    return r


@pytest.mark.parametrize("first", [False, True])
def test_whisper_beam_step(first):
    # 8 audio windows x beam 5 over the 51865-id vocabulary
    rng = make_rng(1000 + first)
    x, cum, sup = gen_beam_select_inputs(rng, WL["windows"], WL["beam"], WL["vocab"])
    args = dict(cum=cum, suppress=sup, blank=WL["blank"], eot=WL["eot"], first=first)
    want = oracle_run(x, WL["beam"], **args)
    got = run_gpu(x, WL["beam"], **args)
    assert got["err"] == 0 and not want["errors"]
    n_exact = check(got, want, WL["beam"])
    assert n_exact >= WL["windows"] - 1
    if first:
        assert np.all(got["n_finished"] == 0)
    else:
        assert got["n_finished"].sum() > 0


@pytest.mark.parametrize("windows,beam,vocab", [(3, 1, 37), (2, 2, 1000), (5, 3, 2049),
                                                (4, 4, 5000), (2, 8, 4097), (1, 4, 152064),
                                                (1, 8, 400000), (64, 5, 51865),
                                                (2, 8, 524288)])
def test_shapes(windows, beam, vocab):
    # one piece per row (37 and 1000 ids), a piece boundary + 1, several pieces per row,
    # a large vocabulary, pieces staged in several passes (400000 ids, 2 pieces of 200000),
    # many windows (64 clusters), the largest vocabulary and beam the call takes
    rng = make_rng(1100 + vocab + beam)
    eot = vocab - 3
    x, cum, sup = gen_beam_select_inputs(rng, windows, beam, vocab, eot=eot,
                                         n_suppress=min(20, vocab // 4), p_eot=0.5)
    want = oracle_run(x, beam, cum=cum, suppress=sup, eot=eot)
    got = run_gpu(x, beam, cum=cum, suppress=sup, eot=eot)
    assert got["err"] == 0
    check(got, want, beam)


def test_greedy_mode_is_the_filtered_argmax():
    # beam 1, no walk: row_token[:, 0] is the filtered argmax of each of 64 rows
    rng = make_rng(1200)
    x, _, sup = gen_beam_select_inputs(rng, 64, 1, 51865, n_suppress=88)
    x[5, sup[3]] = 100.0  # a suppressed id above everything else
    want = oracle_run(x, 1, suppress=sup, blank=[220], eot=50257, first=True, walk=False)
    got = run_gpu(x, 1, suppress=sup, blank=[220], eot=50257, first=True, walk=False)
    assert got["err"] == 0
    check(got, want, 1)
    assert got["row_token"][5, 0] != sup[3]


def test_exact_ties_follow_the_index_order():
    # identical rows and equal cumulative scores: the kernel's fp32 scores tie exactly,
    # so the order is (row, rank in the row); logits quantised to 4 values, so the best
    # ids of a row tie and rank by id: every window keeps its first row's three best
    rng = make_rng(1300)
    row = rng.integers(0, 4, size=7000).astype(np.float32)
    x = np.tile(row, (6, 1))
    cum = np.zeros(6, np.float32)
    want = oracle_run(x, 3, cum=cum, eot=6999)
    got = run_gpu(x, 3, cum=cum, eot=6999)
    assert got["err"] == 0
    assert np.array_equal(got["row_token"], want["row_token"])
    assert np.array_equal(got["parent"], want["parent"])
    assert np.array_equal(got["token"], want["token"])
    assert got["parent"].tolist() == [0, 0, 0, 3, 3, 3]
    assert got["token"][:3].tolist() == np.flatnonzero(row == 3)[:3].tolist()


def test_masked_rows_nan_and_bad_ids():
    import kv_cached_decode_gb300 as kvd

    rng = make_rng(1400)
    x, cum, _ = gen_beam_select_inputs(rng, 2, 2, 3000, eot=2999, p_eot=0.0)
    x[0, :] = -np.inf          # a row with nothing left: all log-probabilities -inf
    x[1, 10:20] = np.nan       # NaNs rank as -inf
    x[2, 2999] = 1e3           # EOT on top
    want = oracle_run(x, 2, cum=cum, eot=2999)
    got = run_gpu(x, 2, cum=cum, eot=2999)
    assert got["err"] == 19
    assert want["errors"] == {19}
    check(got, want, 2)
    assert got["row_token"][0].tolist() == [0, 1, 2]
    assert np.all(np.isneginf(got["row_logprob"][0]))
    assert got["n_finished"][1] == 1 and got["fin_parent"][2] == 2
    # an id outside the vocabulary in the suppression list is skipped and flagged
    y = x[2:].copy()
    want = oracle_run(y, 2, cum=cum[2:], suppress=[5, 3000], eot=2999)
    got = run_gpu(y, 2, cum=cum[2:], suppress=[5, 3000], eot=2999)
    assert got["err"] == 18 and want["errors"] == {18}
    check(got, want, 2)


def test_repeated_calls_pdl_and_unaligned_rows():
    import kv_cached_decode_gb300 as kvd

    rng = make_rng(1500)
    x, cum, sup = gen_beam_select_inputs(rng, 4, 5, 51865)
    want = oracle_run(x, 5, cum=cum, suppress=sup, eot=50257)
    for flags in (0, kvd.KVD_FLAG_PDL, kvd.KVD_FLAG_PDL):
        got = run_gpu(x, 5, cum=cum, suppress=sup, eot=50257, flags=flags)
        assert got["err"] == 0
        check(got, want, 5)
    # logits starting 4, 8 and 12 bytes past a 16-byte boundary (rows of an odd vocabulary
    # start at every alignment anyway)
    for off in (1, 2, 3):
        big = torch.empty(x.size + 4, dtype=torch.float32, device="cuda")
        view = big[off:off + x.size].view(x.shape)
        view.copy_(torch.from_numpy(x))
        got = run_gpu(x, 5, cum=cum, suppress=sup, eot=50257, logits_dev=view)
        assert got["err"] == 0
        check(got, want, 5)


def test_select_then_reorder():
    # the parents feed the cache reorder directly
    import kv_cached_decode_gb300 as kvd
    from gpu_util import dev16, host16
    from workloads import gen_cache

    rng = make_rng(1600)
    x, cum, sup = gen_beam_select_inputs(rng, 2, 5, 51865)
    got = run_gpu(x, 5, cum=cum, suppress=sup, eot=50257)
    K, V = gen_cache(rng, 10, 4, 64, 64, "f16", 0.125, lens=np.full(10, 40, np.int32))
    Kd, Vd = dev16(K, "f16"), dev16(V, "f16")
    kvd.kvd_beam_reorder_kv([kvd.make_cache(Kd, Vd)], 10, 5, dev_i32(got["parent"]),
                            fixed_len=40)
    torch.cuda.synchronize()
    want, err = oracle.beam_reorder(K, got["parent"], 5, 40, "f16")
    assert not err and np.array_equal(host16(Kd), want)
