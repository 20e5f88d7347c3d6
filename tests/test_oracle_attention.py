"""Oracle pins: attention over the cache (decode, cross, causal verify block). CPU only.

The oracle is a two-pass fp64 loop in C. It is pinned here by
* torch's CPU ``scaled_dot_product_attention`` in float64 (an independent library),
* closed forms (one position, identical keys, a dominant key, score shift),
* the structural identities of the method (GQA == replicated MHA, beam rows sharing a
  window == per-row copies, verify row i == decode at length L+i+1).
"""

import numpy as np
import pytest
import torch

from workloads import gen_cache, gen_queries, make_rng


def _f64(bits, dtype):
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _sdpa_reference(q, K, V, lens, rows_per_kv, causal, scale):
    """torch CPU float64 sdpa, one (row, head) at a time, with explicit masks."""
    B, Hq, nq, D = q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    out = np.zeros((B, Hq, nq, D))
    for r in range(B):
        bk = r // rows_per_kv
        L = int(lens[bk])
        for hq in range(Hq):
            h = hq // g
            qq = torch.from_numpy(q[r, hq][None, None])
            kk = torch.from_numpy(np.ascontiguousarray(K[bk, h, :L])[None, None])
            vv = torch.from_numpy(np.ascontiguousarray(V[bk, h, :L])[None, None])
            mask = torch.ones(nq, L, dtype=torch.bool)
            if causal:
                for i in range(nq):
                    mask[i, L - nq + i + 1:] = False
            o = torch.nn.functional.scaled_dot_product_attention(
                qq, kk, vv, attn_mask=mask[None, None], scale=scale)
            out[r, hq] = o[0, 0].numpy()
    return out


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("Hq,Hkv,nq,causal,rpk", [
    (4, 4, 1, False, 1),   # decode, MHA
    (6, 2, 1, False, 1),   # decode, GQA g=3
    (4, 4, 5, True, 1),    # verify block, causal
    (4, 1, 6, True, 1),    # verify block over GQA
    (2, 2, 1, False, 3),   # beam rows sharing a cross buffer
    (2, 2, 3, False, 2),   # non-causal block (cross verify) with shared rows
])
def test_matches_torch_sdpa(oracle_mod, dtype, Hq, Hkv, nq, causal, rpk):
    rng = make_rng(100 + Hq * 7 + nq)
    B = 2 * rpk
    Bkv, cap, D = B // rpk, 40, 16
    lens = np.array([37, 9][:Bkv], np.int32)
    K, V = gen_cache(rng, Bkv, Hkv, cap, D, dtype, 1.0, lens=lens)
    q = gen_queries(rng, B, Hq, nq, D, dtype, 1.0)
    got, err = oracle_mod.attention(q, K, V, dtype, lens=lens, rows_per_kv=rpk,
                                    causal=causal, scale=0.25)
    assert not err
    want = _sdpa_reference(_f64(q, dtype), _f64(K, dtype), _f64(V, dtype), lens, rpk,
                           causal, 0.25)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_single_position_returns_that_value_exactly(oracle_mod):
    rng = make_rng(5)
    K, V = gen_cache(rng, 1, 3, 4, 8, "f16", 1.0, lens=[1])
    q = gen_queries(rng, 1, 3, 1, 8, "f16", 4.0)
    out, _ = oracle_mod.attention(q, K, V, "f16", lens=np.array([1], np.int32))
    assert np.array_equal(out[0, :, 0], _f64(V[0, :, 0], "f16"))


def test_identical_keys_give_the_mean_of_values(oracle_mod):
    rng = make_rng(6)
    L, D = 17, 8
    K = np.repeat(rng.standard_normal((1, 2, 1, D)), L, axis=2)
    V = rng.standard_normal((1, 2, L, D))
    q = rng.standard_normal((1, 2, 1, D))
    out, _ = oracle_mod.attention(q, K, V, "f64", fixed_len=L)
    np.testing.assert_allclose(out[0, :, 0], V[0].mean(axis=1), rtol=0, atol=1e-15)


@pytest.mark.parametrize("pos", [0, 31, 63, 64, 99])
def test_dominant_key_selects_its_value(oracle_mod, pos):
    rng = make_rng(pos)
    L, D = 100, 8
    K = rng.standard_normal((1, 1, L, D)) * 0.01
    V = rng.standard_normal((1, 1, L, D))
    q = np.zeros((1, 1, 1, D))
    q[..., 0] = 1.0
    K[0, 0, pos, 0] = 60.0  # score 60 above the rest
    out, _ = oracle_mod.attention(q, K, V, "f64", fixed_len=L, scale=1.0)
    np.testing.assert_allclose(out[0, 0, 0], V[0, 0, pos], rtol=0, atol=1e-20 + 1e-22 * L)
    assert np.max(np.abs(out[0, 0, 0] - V[0, 0, pos])) < 1e-20


def test_score_shift_leaves_output_unchanged(oracle_mod):
    """Adding u to every key with q.u = c shifts all scores by c: softmax is unchanged."""
    rng = make_rng(8)
    L, D = 23, 8
    K = rng.standard_normal((1, 1, L, D))
    V = rng.standard_normal((1, 1, L, D))
    q = rng.standard_normal((1, 1, 1, D))
    u = q[0, 0, 0] / np.dot(q[0, 0, 0], q[0, 0, 0]) * 7.5
    a, _ = oracle_mod.attention(q, K, V, "f64", fixed_len=L)
    b, _ = oracle_mod.attention(q, K + u, V, "f64", fixed_len=L)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_gqa_equals_mha_with_replicated_kv_heads(oracle_mod):
    rng = make_rng(9)
    B, Hq, Hkv, cap, D = 2, 6, 2, 30, 16
    lens = np.array([30, 11], np.int32)
    K, V = gen_cache(rng, B, Hkv, cap, D, "bf16", 1.0, lens=lens)
    q = gen_queries(rng, B, Hq, 1, D, "bf16", 1.0)
    a, _ = oracle_mod.attention(q, K, V, "bf16", lens=lens)
    Kr = np.ascontiguousarray(np.repeat(K, Hq // Hkv, axis=1))
    Vr = np.ascontiguousarray(np.repeat(V, Hq // Hkv, axis=1))
    b, _ = oracle_mod.attention(q, Kr, Vr, "bf16", lens=lens)
    assert np.array_equal(a, b)


def test_shared_window_rows_equal_replicated_buffers(oracle_mod):
    rng = make_rng(10)
    W, beam, H, F, D = 2, 3, 2, 25, 8
    K, V = gen_cache(rng, W, H, F, D, "f16", 1.0)
    q = gen_queries(rng, W * beam, H, 1, D, "f16", 1.0)
    a, _ = oracle_mod.attention(q, K, V, "f16", fixed_len=F, rows_per_kv=beam)
    Kr = np.ascontiguousarray(np.repeat(K, beam, axis=0))
    Vr = np.ascontiguousarray(np.repeat(V, beam, axis=0))
    b, _ = oracle_mod.attention(q, Kr, Vr, "f16", fixed_len=F)
    assert np.array_equal(a, b)


def test_verify_row_equals_decode_at_its_length(oracle_mod):
    rng = make_rng(12)
    B, H, cap, D, nq = 2, 2, 20, 8, 5
    lens = np.array([20, 7], np.int32)
    K, V = gen_cache(rng, B, H, cap, D, "f16", 1.0, lens=lens)
    q = gen_queries(rng, B, H, nq, D, "f16", 1.0)
    blk, _ = oracle_mod.attention(q, K, V, "f16", lens=lens, causal=True)
    for i in range(nq):
        one, _ = oracle_mod.attention(np.ascontiguousarray(q[:, :, i:i + 1]), K, V, "f16",
                                      lens=lens - nq + i + 1)
        assert np.array_equal(blk[:, :, i:i + 1], one)


def test_empty_cache_gives_zeros_and_poison_is_never_read(oracle_mod):
    rng = make_rng(13)
    K, V = gen_cache(rng, 2, 2, 16, 8, "f16", 1.0, lens=[0, 5])
    q = gen_queries(rng, 2, 2, 1, 8, "f16", 1.0)
    out, err = oracle_mod.attention(q, K, V, "f16", lens=np.array([0, 5], np.int32))
    assert not err
    assert np.all(out[0] == 0.0)
    assert np.all(np.isfinite(out[1]))


def test_length_beyond_capacity_is_flagged(oracle_mod):
    rng = make_rng(14)
    K, V = gen_cache(rng, 1, 1, 8, 8, "f16", 1.0)
    q = gen_queries(rng, 1, 1, 1, 8, "f16", 1.0)
    out, err = oracle_mod.attention(q, K, V, "f16", lens=np.array([9], np.int32))
    assert err == {16}
    assert np.all(out == 0.0)
