"""GPU parity, bit-exact, of the cache append, greedy accept and beam cache reorder
against the oracle, through the C ABI."""

import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev16, dev_i32, host16, new_err, require_gpu
from workloads import gen_accept_inputs, gen_cache, gen_new_kv, gen_parents, make_rng

pytestmark = pytest.mark.gpu
D = 64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _kvd():
    import kv_cached_decode_gb300 as kvd

    return kvd


# --------------------------------------------------------------------------- append -----

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("q", [1, 5])
def test_append_bit_exact(dtype, q):
    kvd = _kvd()
    rng = make_rng(200 + q)
    B, H, cap = 6, 4, 70
    lens = np.array([0, cap - q, 1, 33, 63, 64], np.int32)
    K, V = gen_cache(rng, B, H, cap, D, dtype, 0.125, lens=lens)
    kn, vn = gen_new_kv(rng, B, H, q, D, dtype, 0.125)
    Kd, Vd = dev16(K, dtype), dev16(V, dtype)
    lens_out = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    e = new_err()
    kvd.kvd_kv_append(kvd.make_cache(Kd, Vd), dev16(kn, dtype), dev16(vn, dtype), dev_i32(lens),
                      lens_out, dev_err=e)
    want_lens, err = oracle.kv_append(K, V, kn, vn, lens, dtype)
    torch.cuda.synchronize()
    assert not err and e.item() == 0
    assert np.array_equal(lens_out.cpu().numpy(), want_lens)
    assert np.array_equal(host16(Kd), K) and np.array_equal(host16(Vd), V)


def test_append_into_padded_cache_and_overflow_row():
    kvd = _kvd()
    rng = make_rng(210)
    B, H, cap_alloc, cap = 3, 2, 96, 80
    lens = np.array([78, 10, 79], np.int32)  # rows 0 and 2 cannot take 3 more
    Kbig, Vbig = gen_cache(rng, B, H, cap_alloc, D, "f16", 0.125)
    kn, vn = gen_new_kv(rng, B, H, 3, D, "f16", 0.125)
    Kd, Vd = dev16(Kbig, "f16"), dev16(Vbig, "f16")
    lens_out = torch.zeros(B, dtype=torch.int32, device="cuda")
    e = new_err()
    kvd.kvd_kv_append(kvd.make_cache(Kd[:, :, :cap], Vd[:, :, :cap]), dev16(kn, "f16"),
                      dev16(vn, "f16"), dev_i32(lens), lens_out, dev_err=e)
    K, V = Kbig[:, :, :cap].copy(), Vbig[:, :, :cap].copy()
    want_lens, err = oracle.kv_append(K, V, kn, vn, lens, "f16")
    torch.cuda.synchronize()
    assert err == {16} and e.item() == 16
    assert np.array_equal(lens_out.cpu().numpy(), want_lens)
    got = host16(Kd)
    assert np.array_equal(got[:, :, :cap], K)
    assert np.array_equal(got[:, :, cap:], Kbig[:, :, cap:])  # padding untouched


# --------------------------------------------------------------------------- accept -----

def run_accept(logits, draft, want_nmin=True):
    kvd = _kvd()
    B, k1, V = logits.shape
    ld = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    dd = dev_i32(draft)
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    amax = torch.full((B, k1), -1, dtype=torch.int32, device="cuda")
    nmin = torch.full((1,), -1, dtype=torch.int32, device="cuda") if want_nmin else None
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_GREEDY_ACCEPT, B, qlen=k1 - 1,
                                                  vocab=V))
    e = new_err()
    kvd.kvd_greedy_accept(ld, dd, n, nxt, ws, n_min=nmin, argmax=amax, dev_err=e)
    torch.cuda.synchronize()
    assert int(ws[: kvd.KVD_WS_COUNTER_BYTES].sum().item()) == 0
    return (n.cpu().numpy(), nxt.cpu().numpy(), None if nmin is None else int(nmin.item()),
            amax.cpu().numpy(), e.item())


def _check_against_oracle(logits, draft, codes=()):
    n, nxt, nmin, amax, e = run_accept(logits, draft)
    wn, wnxt, wmin, wamax, werr = oracle.greedy_accept(logits, draft)
    assert np.array_equal(amax, wamax)
    assert np.array_equal(n, wn) and np.array_equal(nxt, wnxt) and nmin == wmin
    assert (e in werr) if werr else e == 0
    return n


def test_accept_whisper_verify_trials_bit_exact():
    """10^4 seeded trials at the speculative-verify shape (k = 5, vocab 51865), in
    batches of 500 rows, bit-exact against the oracle; the mean accepted length matches
    the closed form sum_{i=1..5} 0.75^i."""
    ns = []
    for seed in range(20):
        logits, draft = gen_accept_inputs(make_rng(300 + seed), 500, 5, 51865)
        ns.append(_check_against_oracle(logits, draft))
    n = np.concatenate(ns)
    assert n.size == 10_000
    e_n = sum(0.75 ** i for i in range(1, 6))
    assert abs(n.mean() - e_n) < 4 * n.std() / np.sqrt(n.size)


def test_accept_batch_past_the_counter_region():
    """A batch whose per-row argmax words do not fit in the workspace's counter region
    (1400 rows x 6 x 8 bytes) takes the two-pass reduction; same results."""
    logits, draft = gen_accept_inputs(make_rng(350), 1400, 5, 3000, p_match=0.9)
    logits[3, 2, [10, 2999]] = 40.0  # a tie across segments
    _check_against_oracle(logits, draft)


def test_accept_batch_one_rounds():
    for seed in range(20):
        logits, draft = gen_accept_inputs(make_rng(400 + seed), 1, 5, 51865)
        _check_against_oracle(logits, draft)


def test_accept_worked_example():
    fx = json.load(open(os.path.join(GOLDEN, "sock_fox.json")))
    ids = {w: i for i, w in enumerate(fx["vocab"])}
    logits = np.zeros((1, 6, len(ids)), np.float32)
    for i, w in enumerate(fx["main_top"]):
        logits[0, i, ids[w]] = 5.0
    draft = np.array([[ids[w] for w in fx["draft"]]], np.int32)
    n, nxt, _, _, e = run_accept(logits, draft)
    assert e == 0 and int(n[0]) == 3 and fx["vocab"][int(nxt[0])] == "fox"


@pytest.mark.parametrize("k,V", [(1, 1), (1, 7), (16, 2049), (3, 51865), (5, 100_003),
                                 (5, 524288)])
def test_accept_shapes(k, V):
    logits, draft = gen_accept_inputs(make_rng(500 + k), 7, k, V, p_match=0.9) if V > 1 else (
        np.zeros((7, k + 1, 1), np.float32), np.zeros((7, k), np.int32))
    _check_against_oracle(logits, draft)


def test_accept_ties_nan_inf_and_bad_drafts():
    rng = make_rng(600)
    V = 5000
    logits = rng.standard_normal((4, 5, V)).astype(np.float32)
    logits[0, 0, [17, 2500, 4999]] = 50.0          # ties across segments: lowest wins
    logits[0, 1, :] = -np.inf                       # all -inf: index 0
    logits[1, 2, [3000, 12]] = np.nan               # NaN ranks first, lowest NaN wins
    logits[2, :, :] = 1.0                           # all equal: index 0
    logits[3, 3, :] = -1.0                          # -0 and +0 tie: the lower index wins
    logits[3, 3, [7, 4000]] = [-0.0, 0.0]
    logits[3, 4, :] = -2.0
    logits[3, 4, [9, 4001]] = [0.0, -0.0]
    draft = np.array([[17, 0, 5, 5], [1, 1, 1, 1], [0, 0, 0, 0], [V, -3, 2, 2]], np.int32)
    draft[1, :2] = np.argmax(logits[1, :2], axis=-1)
    _check_against_oracle(logits, draft)


# ----------------------------------------------------------------------------- beam -----

def run_beam(layers_np, parent, beam, *, lens=None, fixed_len=0, dtype="f16"):
    kvd = _kvd()
    devs = [(dev16(k, dtype), dev16(v, dtype)) for k, v in layers_np]
    caches = [kvd.make_cache(k, v) for k, v in devs]
    e = new_err()
    R = len(parent)
    kvd.kvd_beam_reorder_kv(caches, R, beam, dev_i32(parent),
                            lens=None if lens is None else dev_i32(lens), fixed_len=fixed_len,
                            dtype=torch.float16 if dtype == "f16" else torch.bfloat16, dev_err=e)
    torch.cuda.synchronize()
    return [(host16(k), host16(v)) for k, v in devs], e.item()


@pytest.mark.parametrize("L", [32, 224, 440])
def test_beam_whisper_shape_bit_exact(L):
    """8 windows x beam 5 = 40 rows, 20 heads, capacity 448, 4 layers in one call."""
    rng = make_rng(700 + L)
    layers = [gen_cache(rng, 40, 20, 448, D, "f16", 0.125, lens=[L] * 40) for _ in range(4)]
    parent = gen_parents(rng, 8, 5)
    got, e = run_beam(layers, parent, 5, fixed_len=L)
    assert e == 0
    for (gk, gv), (k, v) in zip(got, layers):
        wk, _ = oracle.beam_reorder(k, parent, 5, L, "f16")
        wv, _ = oracle.beam_reorder(v, parent, 5, L, "f16")
        assert np.array_equal(gk, wk) and np.array_equal(gv, wv)


def test_beam_every_parent_map_beam3():
    rng = make_rng(710)
    base = gen_cache(rng, 3, 2, 70, D, "bf16", 1.0)
    for parent in itertools.product(range(3), repeat=3):
        parent = np.array(parent, np.int32)
        for L in (0, 65):
            got, e = run_beam([base], parent, 3, fixed_len=L, dtype="bf16")
            wk, _ = oracle.beam_reorder(base[0], parent, 3, L, "bf16")
            wv, _ = oracle.beam_reorder(base[1], parent, 3, L, "bf16")
            assert e == 0
            assert np.array_equal(got[0][0], wk) and np.array_equal(got[0][1], wv)


def test_beam_bad_parent_and_per_row_lengths():
    rng = make_rng(720)
    layer = gen_cache(rng, 6, 2, 100, D, "f16", 1.0)
    parent = np.array([2, 0, 1, 3, 0, 3], np.int32)  # row 4 points outside its window
    lens = np.array([100, 5, 64, 9, 9, 77], np.int32)
    got, e = run_beam([layer], parent, 3, lens=lens)
    assert e == 17
    for kv in range(2):
        src = layer[kv]
        want = src.copy()
        for r in range(6):
            p = parent[r] if r != 4 else r
            want[r, :, : lens[r]] = src[p, :, : lens[r]]
        assert np.array_equal(got[0][kv], want)


def test_beam_cycle_in_place():
    """A 5-cycle of parents in one window: every row moves, sources are overwritten."""
    rng = make_rng(730)
    layer = gen_cache(rng, 5, 3, 130, D, "f16", 1.0)
    parent = np.array([1, 2, 3, 4, 0], np.int32)
    got, e = run_beam([layer], parent, 5, fixed_len=130)
    assert e == 0
    assert np.array_equal(got[0][0], layer[0][parent])
    assert np.array_equal(got[0][1], layer[1][parent])


def test_beam_padded_rows_take_the_per_thread_path():
    """Positions padded to 72 elements (144-byte rows) are not contiguous 128-byte rows,
    so the reorder runs its per-thread path instead of bulk copies; same result."""
    kvd = _kvd()
    rng = make_rng(740)
    layer = gen_cache(rng, 10, 3, 200, D, "f16", 1.0)
    parent = np.array([1, 1, 0, 4, 2, 9, 5, 5, 7, 6], np.int32)
    lens = np.array([200, 7, 64, 129, 1, 0, 63, 65, 200, 128], np.int32)
    devs = []
    for kv in range(2):
        big = torch.zeros(10, 3, 200, 72, dtype=torch.float16, device="cuda")
        big[..., :D] = dev16(layer[kv], "f16")
        devs.append(big[..., :D])
    cache = kvd.make_cache(devs[0], devs[1])
    assert cache.stride_t == 72
    e = new_err()
    kvd.kvd_beam_reorder_kv([cache], 10, 5, dev_i32(parent), lens=dev_i32(lens), dev_err=e)
    torch.cuda.synchronize()
    assert e.item() == 0
    for kv in range(2):
        want = layer[kv].copy()
        for r in range(10):
            want[r, :, : lens[r]] = layer[kv][parent[r], :, : lens[r]]
        assert np.array_equal(host16(devs[kv].contiguous()), want)


def test_binding_refuses_mistyped_and_strided_tensors():
    import kv_cached_decode_gb300 as kvd

    dev = "cuda"
    logits = torch.zeros(2, 4, 64, dtype=torch.float32, device=dev)
    draft = torch.zeros(2, 3, dtype=torch.int32, device=dev)
    n = torch.zeros(2, dtype=torch.int32, device=dev)
    nxt = torch.zeros(2, dtype=torch.int32, device=dev)
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_GREEDY_ACCEPT, 2, qlen=3,
                                                  vocab=64), device=dev)
    with pytest.raises(TypeError, match="logits must be torch.float32"):
        kvd.kvd_greedy_accept(logits.half(), draft, n, nxt, ws)
    with pytest.raises(TypeError, match="draft must be torch.int32"):
        kvd.kvd_greedy_accept(logits, draft.long(), n, nxt, ws)
    with pytest.raises(ValueError, match="draft must be contiguous"):
        kvd.kvd_greedy_accept(logits, torch.zeros(3, 2, dtype=torch.int32, device=dev).t(),
                              n, nxt, ws)
    kvd.kvd_greedy_accept(logits, draft, n, nxt, ws)  # the same call, well formed
    torch.cuda.synchronize()


def test_beam_step_chain_with_early_self_calls_matches_plain_launches():
    # The beam step as bench.py times it: the reorder, then per layer a self decode with
    # the new token appended and a cross decode shared per window. Launched with PDL,
    # the first self call after the reorder waits before touching its cache; every
    # later self call and every cross call stages its K/V before its dependency wait.
    # The same chain with plain launches must give the same bits (outputs, caches,
    # lengths), repeated over several replays of the launch sequence.
    import kv_cached_decode_gb300 as kvd

    W, beam, NL, H, cap, F, L = 4, 3, 6, 4, 256, 640, 150
    R = W * beam
    rng = make_rng(8801)
    parent = gen_parents(rng, W, beam)
    base_self = [gen_cache(rng, R, H, cap, D, "f16", 0.125) for _ in range(NL)]
    base_cross = [gen_cache(rng, W, H, F, D, "f16", 0.125) for _ in range(NL)]
    q = dev16(gen_new_kv(rng, R, H, 1, D, "f16", 0.125)[0], "f16")
    kn, vn = (dev16(a, "f16") for a in gen_new_kv(rng, R, H, 1, D, "f16", 0.125))
    pd = dev_i32(parent)
    cross_t = [tuple(dev16(a, "f16") for a in kv) for kv in base_cross]
    c_cross = [kvd.make_cache(*kv) for kv in cross_t]
    P, E = kvd.KVD_FLAG_PDL, kvd.KVD_FLAG_PDL | kvd.KVD_FLAG_EARLY_KV

    def run(pdl):
        selfs = [tuple(dev16(a, "f16") for a in kv) for kv in base_self]
        c_self = [kvd.make_cache(*kv) for kv in selfs]
        outs = [torch.empty_like(q) for _ in range(2 * NL)]
        ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, R, H, H, beam, 1, F))
        lens_in = dev_i32(np.full(R, L, np.int32))
        lens = dev_i32(np.zeros(R, np.int32))
        err = new_err()
        kvd.kvd_beam_reorder_kv(c_self, R, beam, pd, lens=lens_in, flags=P if pdl else 0,
                                dev_err=err)
        for l in range(NL):
            sf = (P if l == 0 else E) if pdl else 0
            kvd.kvd_decode_attn(q, c_self[l], outs[2 * l], ws, lens=lens_in, flags=sf,
                                append=(kn, vn, lens), dev_err=err)
            kvd.kvd_decode_attn(q, c_cross[l], outs[2 * l + 1], ws, fixed_len=F,
                                rows_per_kv=beam, flags=E if pdl else 0, dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        return ([host16(o) for o in outs], [(host16(k), host16(v)) for k, v in selfs],
                lens.cpu().numpy())

    want = run(False)
    for _ in range(3):
        got = run(True)
        for a, b in zip(got[0], want[0]):
            assert np.array_equal(a, b)
        for (ka, va), (kb, vb) in zip(got[1], want[1]):
            assert np.array_equal(ka, kb) and np.array_equal(va, vb)
        assert np.array_equal(got[2], want[2]) and np.all(got[2] == L + 1)
