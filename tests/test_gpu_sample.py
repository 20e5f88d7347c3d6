"""Temperature sampling and stochastic speculative acceptance on the GPU
(kvd_sample_accept) against the oracle.

The kernel computes in fp32, the oracle in fp64, and both take integer decisions from
floating-point comparisons. So the decisions are compared exactly wherever the
oracle's margin exceeds the fp32 error, and checked for validity elsewhere.

- Acceptance test. The margin is |r*q - p| at the deciding draft. The tolerance is
  2e-5 * max(p, q) + 1e-7.
- Draw. The margin is the distance of u from the nearest boundary of the normalised
  CDF. The tolerance is 5e-6: each fp32 weight is good to about 1e-6 relative, and so
  is a running sum of positive terms.
- Validity. A differing acceptance count must sit at a near-tie. A differing draw must
  lie within the tolerance of u on the fp64 CDF of the branch the kernel took.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import new_err, require_gpu
from workloads import gen_sample_inputs, make_rng

pytestmark = pytest.mark.gpu
ACC_TOL, CDF_TOL = 2e-5, 5e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _dist(row, T):
    x = row.astype(np.float64) / T
    x[np.isnan(x)] = -np.inf
    if not np.isfinite(x.max()):
        return np.zeros_like(x)
    e = np.exp(x - x.max())
    return e / e.sum()


def run_gpu(target, T, u, draft=None, drafts=None, r=None, flags=0):
    import kv_cached_decode_gb300 as kvd

    B = target.shape[0]
    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    e = new_err()
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_SAMPLE_ACCEPT, B,
                                                  qlen=target.shape[1] - 1,
                                                  vocab=target.shape[2]))
    kvd.kvd_sample_accept(dev(target), dev(u), n, nxt, ws, temperature=T, draft=dev(draft),
                          drafts=dev(drafts), r=dev(r), flags=flags, dev_err=e)
    torch.cuda.synchronize()
    return n.cpu().numpy(), nxt.cpu().numpy(), e.item()


def check(target, T, u, draft, drafts, r, got_n, got_next):
    """Compare with the oracle (exact where the margins allow, valid everywhere)."""
    want_n, want_next, _ = oracle.sample_accept(target, T, u, draft=draft, drafts=drafts, r=r)
    B, k1, V = target.shape
    k = k1 - 1
    n_exact = 0
    for b in range(B):
        # the acceptance count
        if got_n[b] != want_n[b]:
            j = min(got_n[b], want_n[b])
            assert j < k
            p = _dist(target[b, j], T)
            q = _dist(draft[b, j], T)
            x = drafts[b, j]
            assert 0 <= x < V
            assert abs(r[b, j] * q[x] - p[x]) <= ACC_TOL * max(p[x], q[x]) + 1e-7, b
        # the draw, in the branch the kernel took
        n = got_n[b]
        p = _dist(target[b, n], T)
        w = np.maximum(p - _dist(draft[b, n], T), 0.0) if n < k else p
        if n < k and w.sum() == 0:
            w = p
        cdf = np.cumsum(w) / w.sum()
        t = int(got_next[b])
        lo = cdf[t - 1] if t > 0 else 0.0
        assert lo <= u[b] + CDF_TOL and cdf[t] >= u[b] - CDF_TOL and w[t] > 0, (b, t)
        if got_n[b] == want_n[b] and np.min(np.abs(cdf - u[b])) > CDF_TOL:
            assert t == want_next[b], b
            n_exact += 1
    return n_exact


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_temperature_sampling_whisper_vocab(T):
    rng = make_rng(1700)
    target, _, _, _, u = gen_sample_inputs(rng, 64, 0, 51865)
    n, nxt, err = run_gpu(target, T, u)
    assert err == 0 and np.all(n == 0)
    assert check(target, T, u, None, None, None, n, nxt) >= 48


@pytest.mark.parametrize("k", [1, 5, 7])
def test_speculative_acceptance(k):
    rng = make_rng(1710 + k)
    target, draft, drafts, r, u = gen_sample_inputs(rng, 24, k, 51865)
    n, nxt, err = run_gpu(target, 1.0, u, draft, drafts, r)
    assert err == 0
    assert check(target, 1.0, u, draft, drafts, r, n, nxt) >= 18
    assert len(set(n.tolist())) > 1  # the case mixes accept counts


@pytest.mark.parametrize("V", [37, 2049, 4097, 152064, 524288])
def test_vocab_sizes(V):
    # one CTA, a slice boundary + 1, three slices, sixteen slices of 9504 ids, a
    # 524288-id vocabulary (the largest the beam selection takes)
    rng = make_rng(1720 + V)
    target, draft, drafts, r, u = gen_sample_inputs(rng, 6, 3, V)
    n, nxt, err = run_gpu(target, 0.8, u, draft, drafts, r, flags=1)
    assert err == 0
    check(target, 0.8, u, draft, drafts, r, n, nxt)


def test_bad_draft_and_nan():
    rng = make_rng(1730)
    target, draft, drafts, r, u = gen_sample_inputs(rng, 4, 2, 3000)
    drafts[1, 0] = 3000      # outside the vocabulary: rejected, flagged
    target[2, 0, 5] = np.nan  # counted as -inf, flagged
    n, nxt, err = run_gpu(target, 1.0, u, draft, drafts, r)
    assert err in (18, 19)   # the first flag wins
    assert n[1] == 0
    want_n, want_next, errs = oracle.sample_accept(target, 1.0, u, draft=draft, drafts=drafts,
                                                   r=r)
    assert errs == {18, 19}
    assert n[1] == want_n[1]


def test_first_token_follows_the_target_distribution():
    # the guarantee of speculative sampling, end to end on the GPU: over 8192 rows with
    # the same p and q (drafts drawn from q), the first emitted token is distributed as p
    rng = np.random.default_rng(1740)
    B, V, k, T = 8192, 6, 2, 1.0
    trow = (rng.standard_normal(V) * 2).astype(np.float32)
    drow = (rng.standard_normal(V) * 2).astype(np.float32)
    p, q = _dist(trow, T), _dist(drow, T)
    target = np.broadcast_to(trow, (B, k + 1, V)).copy()
    draft = np.broadcast_to(drow, (B, k, V)).copy()
    drafts = np.stack([rng.choice(V, size=B, p=q) for _ in range(k)], axis=1).astype(np.int32)
    r = rng.random((B, k)).astype(np.float32)
    u = rng.random(B).astype(np.float32)
    n, nxt, err = run_gpu(target, T, u, draft, drafts, r)
    assert err == 0
    first = np.where(n > 0, drafts[:, 0], nxt)
    freq = np.bincount(first, minlength=V) / B
    assert np.all(np.abs(freq - p) < 5 * np.sqrt(p * (1 - p) / B) + 1e-4), (freq, p)
