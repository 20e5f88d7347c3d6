"""Oracle pins: number-format decoding and the cache append (CPU only)."""

import numpy as np
import pytest

from workloads import POISON, gen_cache, gen_new_kv, make_rng


def test_f16_decode_all_bit_patterns(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_decode_all_bit_patterns(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode(bits, "bf16")
    want = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("q", [1, 5])
@pytest.mark.parametrize("batch", [1, 2])
def test_append_equals_concatenation_every_start(oracle_mod, dtype, q, batch):
    """Brute force over every start length: the cache prefix after the append equals the
    concatenation of the old prefix and the new tokens along the sequence axis, and every
    position past it keeps its old bytes."""
    H, cap, D = 2, 12, 8
    rng = make_rng(7 + q + 10 * batch)
    for start in range(0, cap - q + 1):
        lens = np.full(batch, start, np.int32)
        if batch == 2:
            lens[1] = (start * 5 + 3) % (cap - q + 1)
        K, V = gen_cache(rng, batch, H, cap, D, dtype, 0.5, lens=lens)
        kn, vn = gen_new_kv(rng, batch, H, q, D, dtype, 0.5)
        K0, V0 = K.copy(), V.copy()
        lens_out, err = oracle_mod.kv_append(K, V, kn, vn, lens, dtype)
        assert not err
        assert np.array_equal(lens_out, lens + q)
        for b in range(batch):
            L = int(lens[b])
            cat_k = np.concatenate([K0[b, :, :L], kn[b]], axis=1)
            cat_v = np.concatenate([V0[b, :, :L], vn[b]], axis=1)
            assert np.array_equal(K[b, :, : L + q], cat_k)
            assert np.array_equal(V[b, :, : L + q], cat_v)
            assert np.array_equal(K[b, :, L + q:], K0[b, :, L + q:])
            assert np.array_equal(V[b, :, L + q:], V0[b, :, L + q:])


def test_append_overflow_flags_and_skips_row(oracle_mod):
    rng = make_rng(3)
    K, V = gen_cache(rng, 2, 2, 8, 8, "f16", 0.5, lens=[6, 2])
    kn, vn = gen_new_kv(rng, 2, 2, 3, 8, "f16", 0.5)
    K0 = K.copy()
    lens_out, err = oracle_mod.kv_append(K, V, kn, vn, np.array([6, 2], np.int32), "f16")
    assert err == {16}
    assert list(lens_out) == [6, 5]
    assert np.array_equal(K[0], K0[0])
    assert np.array_equal(K[1, :, 2:5], kn[1])
    assert np.all(K[0, :, 6:] == POISON["f16"])


def test_append_f64_and_strided_cache(oracle_mod):
    """A cache whose capacity axis is padded (stride over positions > head_dim is not
    allowed, but batch/head strides larger than dense are) gives the same result."""
    rng = make_rng(11)
    big = rng.standard_normal((2, 3, 10, 4))
    K = big[:, :, :, :]
    Kp = np.zeros((2, 3, 16, 4))  # capacity 16 storage, use first 10 positions
    Kp[:, :, :10] = K
    Vp = Kp.copy()
    kn = rng.standard_normal((2, 3, 2, 4))
    lens = np.array([4, 7], np.int32)
    Kd, Vd = K.copy(), K.copy()
    lo1, e1 = oracle_mod.kv_append(Kd, Vd, kn, kn, lens, "f64")
    lo2, e2 = oracle_mod.kv_append(Kp, Vp, kn, kn, lens, "f64")
    assert not e1 and not e2
    assert np.array_equal(lo1, lo2)
    assert np.array_equal(Kd, Kp[:, :, :10])
