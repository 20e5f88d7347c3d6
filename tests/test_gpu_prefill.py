"""Prefill on the GPU (kvd_prefill_attn) against the fp64 oracle.

The prompt's K/V must land in the cache bit-exactly at lens_in + j; each prompt row j
must match the oracle's causal attention at position lens_in + j (the oracle takes the
prompt as a causal query block of plens[b] tokens over the appended cache); rows past a
row's prompt length are zeros. Tolerance: max-abs 1e-2, rel-Frobenius 5e-3.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attn_close, dev16, dev_i32, host16, new_err, require_gpu
from gpu_util import f64
from workloads import (gen_cache, gen_lens_uniform, gen_new_kv, gen_queries, make_rng,
                       round_half_bits)

pytestmark = pytest.mark.gpu
D = 64


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_prefill(dtype, B, Hq, Hkv, cap, max_len, plens, lens_in=None, *, seed, flags=0,
                q_std=0.125, kv_std=0.125, key_growth=None):
    import kv_cached_decode_gb300 as kvd

    rng = make_rng(seed)
    plens = np.asarray(plens, np.int32)
    start = np.zeros(B, np.int32) if lens_in is None else np.asarray(lens_in, np.int32)
    # cached prefix (NaN past it), the prompt's K/V and queries
    K, V = gen_cache(rng, B, Hkv, cap, D, dtype, kv_std, lens=start)
    kn, vn = gen_new_kv(rng, B, Hkv, max_len, D, dtype, kv_std)
    q = gen_queries(rng, B, Hq, max_len, D, dtype, q_std)
    if key_growth is not None:
        # prompt key j scaled by 1 + j / key_growth: later keys score ever higher, so a
        # row's running maximum keeps growing across key tiles
        grow = 1.0 + np.arange(max_len) / key_growth
        kn = round_half_bits(f64(kn, dtype) * grow[None, None, :, None], dtype)
    # expected cache and outputs
    Kw, Vw = K.copy(), V.copy()
    want = np.zeros((B, Hq, max_len, D))
    ok = (start >= 0) & (plens >= 0) & (plens <= max_len) & (start + plens <= cap)
    for b in range(B):
        if not ok[b]:
            continue
        Kw[b, :, start[b]:start[b] + plens[b]] = kn[b, :, :plens[b]]
        Vw[b, :, start[b]:start[b] + plens[b]] = vn[b, :, :plens[b]]
        if plens[b] > 0:
            w, err = oracle.attention(q[b:b + 1, :, :plens[b]], Kw[b:b + 1], Vw[b:b + 1], dtype,
                                      lens=np.array([start[b] + plens[b]], np.int32),
                                      causal=True)
            assert not err
            want[b, :, :plens[b]] = w[0]
    Kd, Vd = dev16(K, dtype), dev16(V, dtype)
    qd = dev16(q, dtype)
    out = torch.full_like(qd, 3.0)
    lens_out = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    e = new_err()
    kvd.kvd_prefill_attn(qd, kvd.make_cache(Kd, Vd), dev16(kn, dtype), dev16(vn, dtype),
                         dev_i32(plens), out, lens_in=None if lens_in is None else dev_i32(start),
                         lens_out=lens_out, flags=flags, dev_err=e)
    torch.cuda.synchronize()
    want_lens = np.where(ok, start + plens, start)
    return (host16(out), want, host16(Kd), host16(Vd), Kw, Vw, lens_out.cpu().numpy(),
            want_lens, e.item(), ok)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_gqa_ragged(dtype):
    # prompt lengths across 64-row tiles: full, one token, empty, a ragged tail
    got, want, Kg, Vg, Kw, Vw, lo, wlo, e, ok = run_prefill(
        dtype, 4, 9, 3, 256, 200, [200, 1, 0, 130], seed=800)
    assert e == 0
    assert np.array_equal(Kg, Kw) and np.array_equal(Vg, Vw) and np.array_equal(lo, wlo)
    assert_attn_close(got, want, dtype, "prefill GQA")
    assert np.all(got[2] == 0) and np.all(got[1][:, 1:] == 0) and np.all(got[3][:, 130:] == 0)


@pytest.mark.parametrize("flags", [0, 1])
def test_prefill_after_cached_prefix(flags):
    # chunked prefill: prompts continue cached prefixes of 0, 50 and 100 positions
    got, want, Kg, Vg, Kw, Vw, lo, wlo, e, ok = run_prefill(
        "f16", 3, 4, 4, 192, 65, [64, 65, 37], [0, 50, 100], seed=801, flags=flags)
    assert e == 0
    assert np.array_equal(Kg, Kw) and np.array_equal(Vg, Vw) and np.array_equal(lo, wlo)
    assert_attn_close(got, want, "f16", "prefill after a prefix")


def test_prefill_whisper_initial_tokens():
    # the first pass over the initial tokens of a Whisper-shaped decoder layer
    got, want, Kg, Vg, Kw, Vw, lo, wlo, e, ok = run_prefill(
        "f16", 1, 20, 20, 448, 4, [4], seed=802)
    assert e == 0 and np.array_equal(Kg, Kw) and np.array_equal(lo, wlo)
    assert_attn_close(got, want, "f16", "Whisper initial tokens")


def test_prefill_long_prompts():
    # prompts of 300..640 tokens over GQA heads: up to 10 query tiles per head
    rng = make_rng(803)
    plens = gen_lens_uniform(rng, 3, 300, 640)
    got, want, Kg, Vg, Kw, Vw, lo, wlo, e, ok = run_prefill(
        "bf16", 3, 6, 2, 704, 640, plens, seed=804)
    assert e == 0 and np.array_equal(Kg, Kw) and np.array_equal(lo, wlo)
    assert_attn_close(got, want, "bf16", "long prompts")


def test_prefill_rejected_row_is_untouched():
    # row 0 would run past the capacity: flagged, cache and length kept, output zeros
    got, want, Kg, Vg, Kw, Vw, lo, wlo, e, ok = run_prefill(
        "f16", 2, 2, 2, 128, 50, [50, 20], [100, 10], seed=805)
    assert e == 16 and not ok[0] and ok[1]
    assert np.array_equal(Kg, Kw) and np.array_equal(Vg, Vw) and np.array_equal(lo, wlo)
    assert np.all(got[0] == 0)
    assert_attn_close(got[1:], want[1:], "f16", "good row")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_growing_maximum(dtype):
    # Peaked scores whose maximum grows by many units (log2) from tile to tile: every
    # change of a row's softmax reference (and the rescaling of the accumulated output
    # it brings) is exercised, against the oracle's exact softmax.
    got, want, Kg, Vg, Kw, Vw, lo, wlo, e, ok = run_prefill(
        dtype, 2, 4, 2, 320, 300, [300, 257], seed=806, q_std=1.0, kv_std=0.5,
        key_growth=16.0)
    assert e == 0 and np.array_equal(Kg, Kw) and np.array_equal(lo, wlo)
    assert_attn_close(got, want, dtype, "growing maximum")


def test_prefill_cache_smaller_than_a_tile():
    # a 40-position cache: the K/V copies are boxes of 40 rows, the tile's other rows
    # stay unwritten and must not reach the output
    got, want, Kg, Vg, Kw, Vw, lo, wlo, e, ok = run_prefill(
        "f16", 3, 2, 1, 40, 33, [33, 7, 1], [0, 30, 39], seed=807)
    assert e == 0 and np.array_equal(Kg, Kw) and np.array_equal(lo, wlo)
    assert_attn_close(got, want, "f16", "small cache")


def test_prefill_prompts_on_tile_boundaries():
    # prompt ends exactly at 64- and 128-position boundaries (no partial key tile)
    got, want, Kg, Vg, Kw, Vw, lo, wlo, e, ok = run_prefill(
        "bf16", 4, 3, 1, 512, 384, [128, 256, 64, 384], [0, 0, 64, 128], seed=808)
    assert e == 0 and np.array_equal(Kg, Kw) and np.array_equal(lo, wlo)
    assert_attn_close(got, want, "bf16", "tile boundaries")


def test_prefill_wait_that_runs_out_is_reported():
    # The test-only stall flag withholds the first K copy: every wait on it runs out
    # after about a second. The call must report KVD_ERR_TIMEOUT, leave the outputs
    # unwritten and free its tensor memory; the same stream then serves a normal call.
    import kv_cached_decode_gb300 as kvd

    dtype, B, H, cap, max_len = "f16", 1, 1, 128, 100
    rng = make_rng(809)
    K, V = gen_cache(rng, B, H, cap, D, dtype, 0.125, lens=[0])
    kn, vn = gen_new_kv(rng, B, H, max_len, D, dtype, 0.125)
    q = gen_queries(rng, B, H, max_len, D, dtype, 0.125)
    plens = np.array([max_len], np.int32)
    Kd, Vd = dev16(K, dtype), dev16(V, dtype)
    qd = dev16(q, dtype)
    out = torch.full_like(qd, 3.0)
    e = new_err()
    kvd.kvd_prefill_attn(qd, kvd.make_cache(Kd, Vd), dev16(kn, dtype), dev16(vn, dtype),
                         dev_i32(plens), out, flags=kvd.KVD_FLAG_TEST_STALL, dev_err=e)
    torch.cuda.synchronize()
    assert e.item() == 20  # KVD_ERR_TIMEOUT
    assert torch.all(out == 3.0)
    # the context and stream are usable: a normal call on fresh buffers matches the oracle
    got, want, Kg, Vg, Kw, Vw, lo, wlo, e2, ok = run_prefill(
        dtype, 2, 4, 2, 256, 150, [150, 77], seed=810)
    assert e2 == 0 and np.array_equal(Kg, Kw) and np.array_equal(lo, wlo)
    assert_attn_close(got, want, dtype, "after a timeout")


def test_prefill_bench_shape_sampled():
    # The prefill at the size bench.py times (16 rows, 9 query heads on 3 KV heads, bf16,
    # prompt lengths uniform in [256, 2048] from the bench's seed, PDL), checked on 48
    # sampled (row, head, position) outputs, each against the oracle's attention of that
    # one query over its visible keys; every cached K/V row bit-exact.
    import kv_cached_decode_gb300 as kvd
    from workloads import WORKLOADS, seed_for

    w = WORKLOADS["gqa_lm_step"]
    B, Hq, Hkv, cap, dtype = w["batch"], w["n_q_heads"], w["n_kv_heads"], w["capacity"], "bf16"
    plens = gen_lens_uniform(make_rng(seed_for("gqa_lm_step", 0, 7)), B, w["len_lo"], w["len_hi"])
    T = int(plens.max())
    rng = make_rng(811)
    K, V = gen_cache(rng, B, Hkv, cap, D, dtype, w["qkv_std"], lens=np.zeros(B, np.int32))
    kn, vn = gen_new_kv(rng, B, Hkv, T, D, dtype, w["qkv_std"])
    q = gen_queries(rng, B, Hq, T, D, dtype, w["qkv_std"])
    Kd, Vd = dev16(K, dtype), dev16(V, dtype)
    out = torch.full_like(dev16(q, dtype), 3.0)
    lens_out = torch.zeros(B, dtype=torch.int32, device="cuda")
    e = new_err()
    kvd.kvd_prefill_attn(dev16(q, dtype), kvd.make_cache(Kd, Vd), dev16(kn, dtype),
                         dev16(vn, dtype), dev_i32(plens), out, lens_out=lens_out,
                         scale=w["scale"], flags=kvd.KVD_FLAG_PDL, dev_err=e)
    torch.cuda.synchronize()
    assert e.item() == 0 and np.array_equal(lens_out.cpu().numpy(), plens)
    Kw, Vw = K.copy(), V.copy()
    for b in range(B):
        Kw[b, :, : plens[b]] = kn[b, :, : plens[b]]
        Vw[b, :, : plens[b]] = vn[b, :, : plens[b]]
    assert np.array_equal(host16(Kd), Kw) and np.array_equal(host16(Vd), Vw)
    got = host16(out)
    pick = make_rng(812)
    for _ in range(48):
        b = int(pick.integers(B))
        h = int(pick.integers(Hq))
        j = int(pick.integers(plens[b]))
        if _ % 4 == 0:
            j = int(plens[b]) - 1  # the last prompt row sees every key
        hk = h // (Hq // Hkv)
        want, err = oracle.attention(q[b:b + 1, h:h + 1, j:j + 1], Kw[b:b + 1, hk:hk + 1],
                                     Vw[b:b + 1, hk:hk + 1], dtype,
                                     lens=np.array([j + 1], np.int32))
        assert not err
        assert_attn_close(got[b:b + 1, h:h + 1, j:j + 1], want, dtype, f"row {b} head {h} pos {j}")
    # rows past each prompt are zeros
    for b in range(B):
        assert np.all(got[b, :, plens[b]:] == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_long_prompt_sampled(dtype):
    # one 8000-token prompt after a 150-token cached prefix (8192-position cache): the
    # last query blocks stream 128 key tiles; 24 sampled positions against the oracle,
    # the cache bit-exact
    import kv_cached_decode_gb300 as kvd

    B, Hq, Hkv, cap, plen, s0 = 1, 2, 1, 8192, 8000, 150
    rng = make_rng(813)
    K, V = gen_cache(rng, B, Hkv, cap, D, dtype, 0.125, lens=[s0])
    kn, vn = gen_new_kv(rng, B, Hkv, plen, D, dtype, 0.125)
    q = gen_queries(rng, B, Hq, plen, D, dtype, 0.5)  # sharper rows than N(0, 1/64)
    Kd, Vd = dev16(K, dtype), dev16(V, dtype)
    out = torch.full_like(dev16(q, dtype), 3.0)
    lens_out = torch.zeros(B, dtype=torch.int32, device="cuda")
    e = new_err()
    kvd.kvd_prefill_attn(dev16(q, dtype), kvd.make_cache(Kd, Vd), dev16(kn, dtype),
                         dev16(vn, dtype), dev_i32([plen]), out, lens_in=dev_i32([s0]),
                         lens_out=lens_out, dev_err=e)
    torch.cuda.synchronize()
    assert e.item() == 0 and lens_out.item() == s0 + plen
    Kw, Vw = K.copy(), V.copy()
    Kw[0, :, s0:s0 + plen] = kn[0]
    Vw[0, :, s0:s0 + plen] = vn[0]
    assert np.array_equal(host16(Kd), Kw) and np.array_equal(host16(Vd), Vw)
    got = host16(out)
    pick = make_rng(814)
    js = sorted(set([0, 127, 128, plen - 1] + [int(x) for x in pick.integers(0, plen, 20)]))
    for j in js:
        for h in range(Hq):
            want, err = oracle.attention(q[:, h:h + 1, j:j + 1], Kw[:, :1], Vw[:, :1], dtype,
                                         lens=np.array([s0 + j + 1], np.int32))
            assert not err
            assert_attn_close(got[:, h:h + 1, j:j + 1], want, dtype, f"head {h} pos {j}")
